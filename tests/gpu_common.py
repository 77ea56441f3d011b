"""Helpers for the GPU parity tests: run the CUDA path, run the oracle on the
same seeded inputs, and compare (index sets exactly, outputs within tolerance)."""
import numpy as np
import torch

import indexer_top_sparse_score_gb300 as smla
import oracle

# Tolerances fixed for this layer step: BF16 KV rel-L2 <= 2e-3 and max-abs <= 1e-2,
# FP8 KV rel-L2 <= 2e-2 (the oracle sees the dequantised FP8 values, so only the
# kernel's arithmetic is measured). Those are bars over all compared values; on
# top of them every (row, head) output vector must be within `rel_l2_row_head`
# (so one wrong head, row or decode part cannot hide in the aggregate), every
# value within `max_abs`, and every lse within `lse` x max(1, |lse|). The
# kernels' own error is far below these: q and the cache rows widen exactly to
# f16 operands, the products accumulate in fp32, P is rounded to f16 (11
# significant bits) and the output to bf16 (8), about 1.2e-3 relative per
# vector; lse stays in fp32 throughout (about 1e-6).
TOL = {"bf16": dict(rel_l2=2e-3, max_abs=1e-2, rel_l2_row_head=1e-2, lse=1e-3),
       "fp8": dict(rel_l2=2e-2, max_abs=1e-2, rel_l2_row_head=2e-2, lse=1e-3),
       "fp8_ds_mla": dict(rel_l2=2e-2, max_abs=1e-2, rel_l2_row_head=2e-2, lse=1e-3)}


def run_prefill(dev, chunk=0, want_idx=True, sm_scale=None):
    """CUDA prefill of all new tokens of `dev` (a device Problem); chunked like a
    long prefill against the growing cache when chunk > 0. Returns device tensors."""
    spec = dev.spec
    scale = spec.sm_scale if sm_scale is None else sm_scale
    T, H = dev.q.shape[0], spec.n_heads
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, spec.topk), dtype=torch.int32, device="cuda") if want_idx else None
    step = chunk if chunk > 0 else T
    ws = None
    for c0 in range(0, T, step):
        c1 = min(T, c0 + step)
        P = dev.prefix_len + c0
        need = smla.prefill_workspace_bytes(P, c1 - c0, H, spec.h_idx, spec.topk, spec.kv_dtype)
        if ws is None or ws.numel() < need:
            ws = smla.workspace(need)
        smla.sparse_mla_prefill(dev.cache, dev.page_table, P, dev.q[c0:c1], dev.q_idx[c0:c1], dev.w[c0:c1],
                                spec.topk, scale, out=out[c0:c1], lse=lse[c0:c1],
                                out_idx=None if idx is None else idx[c0:c1], ws=ws)
        rc, bits = smla.read_status(ws)
        assert rc == 0, (rc, bits)
    return idx, out, lse


def indexer_ws(n_rows: int, kind: str, device="cuda"):
    """A workspace for smla_indexer_topk at 32 indexer heads that picks the
    selection mode of rows longer than 16,384 keys: "cand" holds the per-row
    candidate buffers (4 query rows per work item share 16,384 entries: 4,096
    (key, index) pairs per row, plus a count per row) but no score-array block,
    so the streaming mode defers the final selection; "min" is the status word
    alone, so the streaming mode selects inside the scoring kernel."""
    if kind == "cand":
        n = 256 + n_rows * 4096 * 8 + (n_rows * 4 + 255) // 256 * 256
    elif kind == "min":
        n = 256
    else:
        raise ValueError(kind)
    return smla.workspace(n, device)


def compare_idx(gidx: np.ndarray, ridx: np.ndarray):
    """Index sets must match exactly (order inside a row is unspecified)."""
    g = np.sort(gidx, axis=1)
    r = np.sort(ridx, axis=1)
    bad = np.nonzero((g != r).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5].tolist()}"


def compare_out(gout: np.ndarray, rout: np.ndarray, glse: np.ndarray, rlse: np.ndarray, kv_dtype: str):
    """Outputs [rows, H, 512] and lse [rows, H] against the oracle: the aggregate
    rel-L2 bar, then every (row, head) vector, every value and every lse. A
    (row, head) with no usable key must give out = 0 and lse = -inf on both sides."""
    tol = TOL[kv_dtype]
    g = gout.astype(np.float64)
    glse = glse.astype(np.float64)
    empty = np.isneginf(rlse)
    assert np.array_equal(np.isneginf(glse), empty), "rows without keys differ"
    assert (g[empty] == 0).all()
    rel = np.linalg.norm(g - rout) / np.linalg.norm(rout)
    mx = np.abs(g - rout).max()
    assert rel <= tol["rel_l2"], f"rel-L2 {rel:.3e} > {tol['rel_l2']}"
    assert mx <= tol["max_abs"], f"max-abs {mx:.3e} > {tol['max_abs']}"
    num = np.linalg.norm(g - rout, axis=-1)
    den = np.linalg.norm(rout, axis=-1)
    rh = np.where(empty, 0.0, num / np.where(den > 0, den, 1.0))
    worst = np.unravel_index(int(np.argmax(rh)), rh.shape)
    assert rh.max() <= tol["rel_l2_row_head"], f"(row, head) {worst}: rel-L2 {rh.max():.3e}"
    lerr = np.where(empty, 0.0, np.abs(glse - np.where(empty, 0.0, rlse)) / np.maximum(1.0, np.abs(
        np.where(empty, 0.0, rlse))))
    wl_ = np.unravel_index(int(np.argmax(lerr)), lerr.shape)
    assert lerr.max() <= tol["lse"], f"lse (row, head) {wl_}: error {lerr.max():.3e}"
    return rel, mx, float(lerr.max()), float(rh.max())


def stratified_rows(positions_first: int, n_rows: int, topk: int, extra=(), n_random=24, seed=0):
    """Rows covering t < k, t = k-1, k, k+1, first/last rows, given extras and random rows."""
    rng = np.random.default_rng(seed)
    P = positions_first
    cand = {0, 1, n_rows - 1, n_rows - 2, n_rows // 2}
    for pos in (topk - 2, topk - 1, topk, topk + 1):
        r = pos - P
        if 0 <= r < n_rows:
            cand.add(r)
    cand.update(r for r in extra if 0 <= r < n_rows)
    cand.update(rng.integers(0, n_rows, n_random).tolist())
    return np.array(sorted(cand), dtype=np.int64)


class Guarded:
    """A tensor with canary regions before and after it: `view` is the usable
    middle (16-byte aligned); check() asserts that the canaries are unchanged
    (nothing was written outside the view)."""

    PAD = 4096  # bytes of canary on each side

    def __init__(self, shape, dtype, fill_bits: int):
        self.shape, self.dtype = tuple(shape), dtype
        n = 1
        for d in self.shape:
            n *= d
        es = torch.empty((), dtype=dtype).element_size()
        pad = self.PAD // es
        itype = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[es]
        self.raw = torch.full((n + 2 * pad,), fill_bits, dtype=itype, device="cuda")
        self.pad, self.n = pad, n
        self.view = self.raw[pad:pad + n].view(dtype).view(self.shape)
        self.fill = fill_bits

    def check(self):
        torch.cuda.synchronize()
        lo, hi = self.raw[:self.pad], self.raw[self.pad + self.n:]
        assert bool((lo == self.fill).all()) and bool((hi == self.fill).all()), "write outside the output buffer"


def host_cache(dev):
    return dev.cache.to("cpu")


def sampled_oracle(dev, rows, cache_host=None, n_threads=0, sm_scale=None):
    idx, sc, out, lse, used, bad = oracle.prefill_rows(dev, rows, cache_host, n_threads, sm_scale=sm_scale)
    assert not bad.any()
    return idx, sc, out, lse, used
