"""CPU oracle for the indexer -> causal top-k -> sparse MLA step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline /
reference legs may import this package. The product path never does: it runs
the CUDA library or fails.

The arithmetic lives in ``oracle.c`` (plain C, fp32 indexer, full sort,
fp64 softmax attention); this module compiles it with gcc and marshals
arguments. Every function cites the passage it follows in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, FP8, FP8_DS_MLA = 0, 1, 2
D_QK, D_V = 576, 512


class _Problem(ctypes.Structure):
    _fields_ = [
        ("kv", ctypes.c_void_p), ("kv_scale", ctypes.c_void_p),
        ("k_idx", ctypes.c_void_p), ("k_idx_scale", ctypes.c_void_p),
        ("kv_dtype", ctypes.c_int32), ("idx_dtype", ctypes.c_int32),
        ("d_idx", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
        ("n_heads", ctypes.c_int32), ("h_idx", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
        ("is_decode", ctypes.c_int32), ("prefix_len", ctypes.c_int64),
        ("seq_lens", ctypes.c_void_p), ("q_per_seq", ctypes.c_int32),
        ("page_tables", ctypes.c_void_p), ("max_pages", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_e4m3_to_float.restype = ctypes.c_float
            L.oracle_e4m3_to_float.argtypes = [ctypes.c_uint8]
            L.oracle_bf16_to_float.restype = ctypes.c_float
            L.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
            P = ctypes.POINTER(_Problem)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
            L.oracle_scores.restype = ctypes.c_int
            L.oracle_scores.argtypes = [P, i64, vp]
            L.oracle_select_topk.restype = None
            L.oracle_select_topk.argtypes = [vp, i64, i32, vp, vp]
            L.oracle_attend.restype = ctypes.c_int
            L.oracle_attend.argtypes = [P, i64, vp, i32, vp, vp, vp]
            L.oracle_row.restype = ctypes.c_int
            L.oracle_row.argtypes = [P, i64, vp, vp, vp, vp]
            L.oracle_rows.restype = ctypes.c_int
            L.oracle_rows.argtypes = [P, vp, i64, vp, vp, vp, vp, ctypes.c_int, vp]
            L.oracle_attend_rows.restype = ctypes.c_int
            L.oracle_attend_rows.argtypes = [P, vp, i64, vp, i32, vp, vp, ctypes.c_int]
            _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return t.data_ptr()


class Oracle:
    """Binds a host-resident workloads.Problem (all tensors on the CPU).

    Keeps references to the tensors so the raw pointers stay valid.
    """

    def __init__(self, prob, topk: Optional[int] = None, sm_scale: Optional[float] = None):
        spec = prob.spec
        self.prob = prob
        c = prob.cache
        self._keep = [c.kv, c.kv_scale, c.k_idx, c.k_idx_scale, prob.q, prob.q_idx, prob.w]
        pt = prob.page_table
        if pt.dim() == 1:
            pt = pt[None, :]
        pt = pt.to(torch.int32).contiguous()
        seq_lens = None if prob.seq_lens is None else prob.seq_lens.to(torch.int32).contiguous()
        self._keep += [pt, seq_lens]
        for t in self._keep:
            if t is not None:
                assert t.device.type == "cpu" and t.is_contiguous()
        self.topk = int(topk if topk is not None else spec.topk)
        self.n_heads = spec.n_heads
        self.c = _Problem(
            kv=_ptr(c.kv), kv_scale=_ptr(c.kv_scale), k_idx=_ptr(c.k_idx),
            k_idx_scale=_ptr(c.k_idx_scale),
            kv_dtype={"bf16": BF16, "fp8": FP8, "fp8_ds_mla": FP8_DS_MLA}[c.kv_dtype],
            idx_dtype=BF16 if c.idx_dtype == "bf16" else FP8,
            d_idx=spec.d_idx, page_size=c.kv.shape[1], num_pages=c.kv.shape[0],
            q=_ptr(prob.q), q_idx=_ptr(prob.q_idx), w=_ptr(prob.w),
            n_heads=spec.n_heads, h_idx=spec.h_idx, topk=self.topk,
            sm_scale=float(sm_scale if sm_scale is not None else spec.sm_scale),
            is_decode=1 if spec.kind == "decode" else 0,
            prefix_len=prob.prefix_len,
            seq_lens=_ptr(seq_lens), q_per_seq=max(1, spec.q_per_seq),
            page_tables=_ptr(pt), max_pages=pt.shape[1])

    # -- positions (the causal placement of each row) --------------------------
    def position(self, row: int) -> int:
        if self.c.is_decode:
            b, j = divmod(row, self.c.q_per_seq)
            return int(self.prob.seq_lens[b]) - self.c.q_per_seq + j
        return self.c.prefix_len + row

    # -- steps ------------------------------------------------------------------
    def scores(self, row: int) -> np.ndarray:
        n = self.position(row) + 1
        out = np.empty(n, dtype=np.float32)
        lib().oracle_scores(ctypes.byref(self.c), row, out.ctypes.data)
        return out

    def rows(self, rows: Sequence[int], attend: bool = True, n_threads: int = 0):
        """Full step for `rows`: (idx [n,k] int32, scores [n,k] f32, out [n,H,512] f64, lse [n,H] f64, threads)."""
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows.shape[0]
        idx = np.empty((n, self.topk), dtype=np.int32)
        sc = np.empty((n, self.topk), dtype=np.float32)
        out = np.empty((n, self.n_heads, D_V), dtype=np.float64) if attend else None
        lse = np.empty((n, self.n_heads), dtype=np.float64) if attend else None
        bad = np.zeros(n, dtype=np.int32)
        used = lib().oracle_rows(ctypes.byref(self.c), rows.ctypes.data, n, idx.ctypes.data,
                                 sc.ctypes.data, None if out is None else out.ctypes.data,
                                 None if lse is None else lse.ctypes.data, n_threads,
                                 bad.ctypes.data)
        return idx, sc, out, lse, used, bad

    def attend(self, row: int, idx: np.ndarray, probs: bool = False):
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        out = np.empty((self.n_heads, D_V), dtype=np.float64)
        lse = np.empty((self.n_heads,), dtype=np.float64)
        pr = np.empty((self.n_heads, idx.shape[0]), dtype=np.float64) if probs else None
        bad = lib().oracle_attend(ctypes.byref(self.c), row, idx.ctypes.data, idx.shape[0],
                                  out.ctypes.data, lse.ctypes.data,
                                  None if pr is None else pr.ctypes.data)
        return (out, lse, pr, bad) if probs else (out, lse, bad)

    def attend_rows(self, rows: Sequence[int], idx: np.ndarray, n_threads: int = 0):
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        n = rows.shape[0]
        out = np.empty((n, self.n_heads, D_V), dtype=np.float64)
        lse = np.empty((n, self.n_heads), dtype=np.float64)
        lib().oracle_attend_rows(ctypes.byref(self.c), rows.ctypes.data, n, idx.ctypes.data,
                                 idx.shape[1], out.ctypes.data, lse.ctypes.data, n_threads)
        return out, lse


def prefill_rows(prob, rows, cache_host=None, n_threads: int = 0, sm_scale: Optional[float] = None):
    """Full step for chosen rows of a prefill Problem whose tensors may live on a GPU.

    Each chosen row becomes a one-token sequence of length pos+1 that shares the
    prefill's page table, so only the chosen q / q_I / w rows are copied to the
    host. Returns (idx, scores, out, lse, threads used, bad flags)."""
    from indexer_top_sparse_score_gb300 import workloads as wl
    spec = prob.spec
    rows = np.asarray(rows, dtype=np.int64)
    cache = cache_host if cache_host is not None else prob.cache.to("cpu")
    n = len(rows)
    pos = prob.prefix_len + rows
    pt = prob.page_table.cpu().to(torch.int32)
    pts = pt[None, :].expand(n, -1).contiguous()
    r = torch.as_tensor(rows).to(prob.q.device)
    sub = wl.Problem(wl.scaled(spec, kind="decode", n_seqs=n, q_per_seq=1), cache, pts,
                     prob.q[r].cpu().contiguous(), prob.q_idx[r].cpu().contiguous(),
                     prob.w[r].cpu().contiguous(), torch.as_tensor(pos + 1, dtype=torch.int32), 0, 0)
    return Oracle(sub, sm_scale=sm_scale).rows(np.arange(n), n_threads=n_threads)


def select_topk(scores: np.ndarray, k: int):
    """Causal top-k of one score row (ascending indices, -1 padded)."""
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    idx = np.empty(k, dtype=np.int32)
    sc = np.empty(k, dtype=np.float32)
    lib().oracle_select_topk(scores.ctypes.data, scores.shape[0], k, idx.ctypes.data, sc.ctypes.data)
    return idx, sc


def e4m3_to_float(code: int) -> float:
    return lib().oracle_e4m3_to_float(code)


def bf16_to_float(bits: int) -> float:
    return lib().oracle_bf16_to_float(bits)
