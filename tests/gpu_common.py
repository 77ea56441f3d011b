"""Helpers for the GPU parity tests: run the CUDA path, run the oracle on the
same seeded inputs, and compare (index sets exactly, outputs within tolerance)."""
import numpy as np
import torch

import indexer_top_sparse_score_gb300 as smla
import oracle

# Tolerances fixed for this layer step: BF16 KV rel-L2 <= 2e-3 and max-abs <= 1e-2,
# FP8 KV rel-L2 <= 2e-2 (the oracle sees the dequantised FP8 values, so only the
# kernel's arithmetic is measured).
TOL = {"bf16": dict(rel_l2=2e-3, max_abs=1e-2), "fp8": dict(rel_l2=2e-2, max_abs=None),
       "fp8_ds_mla": dict(rel_l2=2e-2, max_abs=None)}


def run_prefill(dev, chunk=0, want_idx=True):
    """CUDA prefill of all new tokens of `dev` (a device Problem); chunked like a
    long prefill against the growing cache when chunk > 0. Returns device tensors."""
    spec = dev.spec
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
                                spec.topk, spec.sm_scale, out=out[c0:c1], lse=lse[c0:c1],
                                out_idx=None if idx is None else idx[c0:c1], ws=ws)
        rc, bits = smla.read_status(ws)
        assert rc == 0, (rc, bits)
    return idx, out, lse


def compare_idx(gidx: np.ndarray, ridx: np.ndarray):
    """Index sets must match exactly (order inside a row is unspecified)."""
    g = np.sort(gidx, axis=1)
    r = np.sort(ridx, axis=1)
    bad = np.nonzero((g != r).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5].tolist()}"


def compare_out(gout: np.ndarray, rout: np.ndarray, glse: np.ndarray, rlse: np.ndarray, kv_dtype: str):
    tol = TOL[kv_dtype]
    g = gout.astype(np.float64)
    rel = np.linalg.norm(g - rout) / np.linalg.norm(rout)
    mx = np.abs(g - rout).max()
    assert rel <= tol["rel_l2"], f"rel-L2 {rel:.3e} > {tol['rel_l2']}"
    if tol["max_abs"] is not None:
        assert mx <= tol["max_abs"], f"max-abs {mx:.3e} > {tol['max_abs']}"
    lerr = np.abs(glse.astype(np.float64) - rlse).max()
    assert lerr <= (2e-3 if kv_dtype == "bf16" else 2e-2) * max(1.0, np.abs(rlse).max()), f"lse err {lerr:.3e}"
    return rel, mx, lerr


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


def host_cache(dev):
    return dev.cache.to("cpu")


def sampled_oracle(dev, rows, cache_host=None, n_threads=0):
    idx, sc, out, lse, used, bad = oracle.prefill_rows(dev, rows, cache_host, n_threads)
    assert not bad.any()
    return idx, sc, out, lse, used
