"""Indexer-selected sparse MLA for one GB300: thin Python binding of libsmla.so.

Every step of the layer (indexer, causal top-k, sparse MLA) runs in the CUDA
kernels of ``csrc/`` behind the C ABI declared in ``include/smla.h``. This
module only marshals torch tensors (device memory, the current stream) into
that ABI. There is no CPU fallback: if the library is not built, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(os.path.dirname(_HERE), "include")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libsmla.so")
SOURCES = ["api.cu", "indexer.cu", "mla.cu", "noalloc.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC"]

SMLA_BF16, SMLA_FP8_E4M3, SMLA_FP8_DS_MLA = 0, 1, 2
STATUS = {0: "SMLA_OK", 1: "SMLA_ERR_INVALID_ARG", 2: "SMLA_ERR_UNSUPPORTED", 3: "SMLA_ERR_WORKSPACE",
          4: "SMLA_ERR_CUDA", 5: "SMLA_ERR_DEVICE_BOUNDS", 6: "SMLA_ERR_TIMEOUT"}
D_QK, D_V, PAGE = 576, 512, 64
STATUS_BYTES = 256  # the status word heads every workspace

_lock = threading.Lock()
_lib = None


class SmlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC)] + [os.path.join(_INCLUDE, "smla.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a into _build/libsmla.so (in-tree)."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    nvcc = _nvcc()
    objs = [os.path.join(_BUILD, s.replace(".cu", ".o")) for s in SOURCES]

    def compile_one(i):
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(_CSRC, SOURCES[i]), "-o", objs[i]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {SOURCES[i]}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout, r.stderr)

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        list(ex.map(compile_one, range(len(SOURCES))))
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class PagedCache(ctypes.Structure):
    _fields_ = [("kv", ctypes.c_void_p), ("kv_scale", ctypes.c_void_p), ("k_idx", ctypes.c_void_p),
                ("k_idx_scale", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("idx_dtype", ctypes.c_int32), ("d_idx", ctypes.c_int32)]


_vp, _i32, _sz, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "smla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "smla_version": (ctypes.c_int, []),
    "smla_indexer_topk_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "smla_indexer_topk": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp,
                                          _vp, _vp, _sz, _vp]),
    "smla_sparse_mla_fwd_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "smla_sparse_mla_fwd": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _vp, _i32, _f32,
                                            _vp, _vp, _vp, _sz, _vp]),
    "smla_sparse_mla_prefill_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "smla_sparse_mla_prefill": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _i32, _i32, _f32,
                                                _vp, _vp, _vp, _vp, _sz, _vp]),
    "smla_sparse_mla_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "smla_sparse_mla_decode": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _i32,
                                               _i32, _f32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "smla_sparse_mla_prefill_noalloc": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp, _i32, _i32,
                                                        _f32, _vp, _vp, _vp]),
    "smla_noalloc_read_status": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "smla_read_status": (ctypes.c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]),
}


def lib(build_if_missing: bool = False):
    """The loaded libsmla.so. Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                build()
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libsmla.so is not built ({LIB_PATH}); run "
                                   "indexer_top_sparse_score_gb300.build() first")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check(rc: int, what: str):
    if rc != 0:
        raise SmlaError(rc, what)


def _dtype_code(name: str) -> int:
    return {"bf16": SMLA_BF16, "fp8": SMLA_FP8_E4M3, "fp8_ds_mla": SMLA_FP8_DS_MLA}[name]


def make_cache(cache) -> PagedCache:
    """C view of a paged cache object with kv / kv_scale / k_idx / k_idx_scale
    tensors and kv_dtype / idx_dtype names ("bf16" or "fp8")."""
    return PagedCache(kv=_p(cache.kv), kv_scale=_p(cache.kv_scale), k_idx=_p(cache.k_idx),
                      k_idx_scale=_p(cache.k_idx_scale), num_pages=cache.kv.shape[0],
                      page_size=cache.kv.shape[1], kv_dtype=_dtype_code(cache.kv_dtype),
                      idx_dtype=_dtype_code(cache.idx_dtype), d_idx=cache.k_idx.shape[-1])


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------- entry points
def indexer_topk(cache, page_tables, seq_lens, max_seq_len, q_per_seq, q_idx, w, topk, out_idx=None,
                 out_scores=None, ws=None, stream=None, want_scores=False):
    """Steps 1-2 for n_seqs sequences of q_per_seq query rows (see smla_indexer_topk)."""
    L = lib()
    pt = page_tables if page_tables.dim() == 2 else page_tables[None]
    n_seqs, max_pages = pt.shape
    rows = n_seqs * q_per_seq
    h_idx = q_idx.shape[1]
    if out_idx is None:
        out_idx = torch.empty((rows, topk), dtype=torch.int32, device=q_idx.device)
    if want_scores and out_scores is None:
        out_scores = torch.empty((rows, topk), dtype=torch.float32, device=q_idx.device)
    need = L.smla_indexer_topk_workspace_size(n_seqs, max_seq_len, q_per_seq, h_idx, topk)
    if ws is None:
        ws = workspace(need, q_idx.device)
    c = make_cache(cache)
    rc = L.smla_indexer_topk(ctypes.byref(c), _p(pt), max_pages, n_seqs, _p(seq_lens), max_seq_len,
                             q_per_seq, _p(q_idx), _p(w), h_idx, topk, _p(out_idx), _p(out_scores),
                             _p(ws), ws.numel(), _stream(stream))
    _check(rc, "smla_indexer_topk")
    return (out_idx, out_scores, ws) if want_scores else (out_idx, ws)


def sparse_mla_fwd(cache, page_tables, q, idx, sm_scale, *, prefix_len=0, seq_lens=None, q_per_seq=None,
                   out=None, lse=None, ws=None, stream=None):
    """Step 3 over given index lists (see smla_sparse_mla_fwd)."""
    L = lib()
    pt = page_tables if page_tables.dim() == 2 else page_tables[None]
    n_seqs, max_pages = pt.shape
    rows, H, _ = q.shape
    topk = idx.shape[1]
    if q_per_seq is None:
        q_per_seq = rows // n_seqs
    if out is None:
        out = torch.empty((rows, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((rows, H), dtype=torch.float32, device=q.device)
    if ws is None:
        max_keys = prefix_len + q_per_seq if seq_lens is None else 0
        ws = workspace(L.smla_sparse_mla_fwd_workspace_size(max_keys, rows, H, topk, _dtype_code(cache.kv_dtype)),
                       q.device)
    c = make_cache(cache)
    rc = L.smla_sparse_mla_fwd(ctypes.byref(c), _p(pt), max_pages, n_seqs, _p(seq_lens), prefix_len,
                               q_per_seq, _p(q), H, _p(idx), topk, float(sm_scale), _p(out), _p(lse),
                               _p(ws), ws.numel(), _stream(stream))
    _check(rc, "smla_sparse_mla_fwd")
    return out, lse, ws


def prefill_workspace_bytes(prefix_len, n_tokens, n_heads, h_idx, topk, kv_dtype="bf16") -> int:
    return lib().smla_sparse_mla_prefill_workspace_size(prefix_len, n_tokens, n_heads, h_idx, topk,
                                                        _dtype_code(kv_dtype))


def sparse_mla_prefill(cache, page_table, prefix_len, q, q_idx, w, topk, sm_scale, *, out=None, lse=None,
                       out_idx=None, ws=None, stream=None):
    """Steps 1-3 for the new tokens of one sequence (see smla_sparse_mla_prefill)."""
    L = lib()
    T, H, _ = q.shape
    h_idx = q_idx.shape[1]
    if out is None:
        out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(prefill_workspace_bytes(prefix_len, T, H, h_idx, topk, cache.kv_dtype), q.device)
    c = make_cache(cache)
    rc = L.smla_sparse_mla_prefill(ctypes.byref(c), _p(page_table), prefix_len, T, _p(q), H, _p(q_idx), _p(w),
                                   h_idx, topk, float(sm_scale), _p(out), _p(lse), _p(out_idx), _p(ws),
                                   ws.numel(), _stream(stream))
    _check(rc, "smla_sparse_mla_prefill")
    return out, lse, out_idx, ws


def chunk_bounds(n_tokens: int, chunk) -> list:
    """[(start, end)] of the query-token chunks of HostPrefill: `chunk` is a size
    (the last chunk takes the rest) or a list of sizes that sum to n_tokens."""
    if isinstance(chunk, int):
        if chunk <= 0:
            raise ValueError("chunk size must be positive")
        return [(a, min(n_tokens, a + chunk)) for a in range(0, n_tokens, chunk)]
    sizes = [int(c) for c in chunk]
    if any(c <= 0 for c in sizes) or sum(sizes) != n_tokens:
        raise ValueError("chunk sizes must be positive and sum to n_tokens")
    bounds = [0]
    for c in sizes:
        bounds.append(bounds[-1] + c)
    return list(zip(bounds[:-1], bounds[1:]))


class HostPrefill:
    """Prefill from pinned HOST buffers: q, q_idx and w are copied in and out /
    lse copied back chunk by chunk, on two copy streams, so the copies of one
    chunk overlap the kernels of its neighbours. The kernels run on a stream
    of the object's own, joined to the caller's stream by one event at each
    end: work on the legacy default stream waits for every other blocking
    stream, so running the kernels there would hold each chunk's copies back
    until the kernels before them end. Each chunk of query tokens is
    one smla_sparse_mla_prefill call with the earlier tokens as its prefix (the
    cache already holds every token's rows), which gives the same rows the
    single call would. `chunk` is a chunk size, or a list of chunk sizes that
    sum to n_tokens (small first and last chunks shorten the copy-in before
    the first kernel and the copy-out after the last). Device buffers,
    workspace, streams and events are made once here; run() may be called
    repeatedly (each call waits for the previous call's use of a chunk's
    device buffers before reusing them).

    Chunk c is given the workspace from byte 256 * c on, so its status word
    (the first 256 bytes of what it is given) is its own: the scratch of chunk c
    covers only the status words of later chunks, which clear theirs when they
    start, so after run() every chunk's word is intact and read_status() reports
    the device errors of all of them.
    """

    def __init__(self, cache, page_table, prefix_len, n_tokens, n_heads, h_idx, d_idx, idx_dtype, topk,
                 sm_scale, chunk=2048, device="cuda"):
        self.cache, self.page_table, self.prefix_len = cache, page_table, prefix_len
        self.T, self.topk, self.sm_scale = n_tokens, topk, sm_scale
        self.chunks = chunk_bounds(n_tokens, chunk)
        idx_t = torch.bfloat16 if idx_dtype == "bf16" else torch.uint8
        self.q = torch.empty((n_tokens, n_heads, D_QK), dtype=torch.bfloat16, device=device)
        self.q_idx = torch.empty((n_tokens, h_idx, d_idx), dtype=idx_t, device=device)
        self.w = torch.empty((n_tokens, h_idx), dtype=torch.float32, device=device)
        self.out = torch.empty((n_tokens, n_heads, D_V), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((n_tokens, n_heads), dtype=torch.float32, device=device)
        need = max(prefill_workspace_bytes(prefix_len + a, b - a, n_heads, h_idx, topk, cache.kv_dtype)
                   for a, b in self.chunks)
        self.ws = workspace(need + STATUS_BYTES * len(self.chunks), device)
        self.s_in, self.s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        self.s_comp = torch.cuda.Stream(device)
        n = len(self.chunks)
        self.ev_in = [torch.cuda.Event() for _ in range(n)]
        self.ev_comp = [torch.cuda.Event() for _ in range(n)]
        self.ev_out = [torch.cuda.Event() for _ in range(n)]

    def run(self, q_h, q_idx_h, w_h, out_h, lse_h, stream=None):
        caller = torch.cuda.current_stream() if stream is None else stream
        comp = self.s_comp
        start = torch.cuda.Event()
        start.record(caller)
        comp.wait_event(start)
        self.s_in.wait_event(start)
        self.s_out.wait_event(start)
        for c, (a, b) in enumerate(self.chunks):
            with torch.cuda.stream(self.s_in):
                self.s_in.wait_event(self.ev_comp[c])  # the previous run's kernels read these inputs
                self.q[a:b].copy_(q_h[a:b], non_blocking=True)
                self.q_idx[a:b].copy_(q_idx_h[a:b], non_blocking=True)
                self.w[a:b].copy_(w_h[a:b], non_blocking=True)
                self.ev_in[c].record(self.s_in)
            comp.wait_event(self.ev_in[c])
            comp.wait_event(self.ev_out[c])  # the previous run's copy-out of these outputs
            sparse_mla_prefill(self.cache, self.page_table, self.prefix_len + a, self.q[a:b], self.q_idx[a:b],
                               self.w[a:b], self.topk, self.sm_scale, out=self.out[a:b], lse=self.lse[a:b],
                               ws=self.ws[STATUS_BYTES * c:], stream=comp)
            self.ev_comp[c].record(comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(self.ev_comp[c])
                out_h[a:b].copy_(self.out[a:b], non_blocking=True)
                lse_h[a:b].copy_(self.lse[a:b], non_blocking=True)
                self.ev_out[c].record(self.s_out)
        for c in range(len(self.chunks)):
            caller.wait_event(self.ev_out[c])  # the call ends on `stream` once every result is on the host
        done = torch.cuda.Event()
        done.record(comp)
        caller.wait_event(done)

    def read_status(self, stream=None):
        """(status code, raw bits) over every chunk of the last run() (waits on
        the stream)."""
        return read_status_chunks(self.ws, len(self.chunks), stream)


# precedence of the device status codes (as smla_read_status orders them)
_STATUS_RANK = {0: 0, 2: 1, 5: 2, 6: 3}


def read_status_chunks(ws: torch.Tensor, n_chunks: int, stream=None):
    """Status of n_chunks calls whose workspaces start at ws + 256 * c: the most
    severe code and the union of the raw bits."""
    code, bits = 0, 0
    for c in range(n_chunks):
        rc, b = read_status(ws[STATUS_BYTES * c:], stream)
        bits |= b
        if _STATUS_RANK.get(rc, 4) > _STATUS_RANK.get(code, 4):
            code = rc
    return code, bits


def decode_workspace_bytes(n_seqs, max_seq_len, q_per_seq, n_heads, h_idx, topk) -> int:
    return lib().smla_sparse_mla_decode_workspace_size(n_seqs, max_seq_len, q_per_seq, n_heads, h_idx, topk)


def sparse_mla_decode(cache, page_tables, seq_lens, max_seq_len, q_per_seq, q, q_idx, w, topk, sm_scale, *,
                      out=None, lse=None, out_idx=None, ws=None, stream=None):
    """Steps 1-3 for a decode batch (see smla_sparse_mla_decode)."""
    L = lib()
    n_seqs, max_pages = page_tables.shape
    rows, H, _ = q.shape
    h_idx = q_idx.shape[1]
    if out is None:
        out = torch.empty((rows, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((rows, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(decode_workspace_bytes(n_seqs, max_seq_len, q_per_seq, H, h_idx, topk), q.device)
    c = make_cache(cache)
    rc = L.smla_sparse_mla_decode(ctypes.byref(c), _p(page_tables), max_pages, n_seqs, _p(seq_lens),
                                  max_seq_len, q_per_seq, _p(q), H, _p(q_idx), _p(w), h_idx, topk,
                                  float(sm_scale), _p(out), _p(lse), _p(out_idx), _p(ws), ws.numel(),
                                  _stream(stream))
    _check(rc, "smla_sparse_mla_decode")
    return out, lse, out_idx, ws


def read_status(ws: torch.Tensor, stream=None):
    """(status code, raw bits) of the device status word in `ws` (waits on the stream)."""
    bits = ctypes.c_uint32(0)
    rc = lib().smla_read_status(_p(ws), _stream(stream), ctypes.byref(bits))
    return rc, bits.value
