"""The workspace-free prefill entry point, for callers that cannot allocate
device memory (a plugin handed only input/output pointers, an engine whose
memory belongs to a pool outside code may not use). Its scratch is a fixed
array inside the library; it must give the same results as the regular entry
point, call after call (the array keeps the previous call's contents)."""
import ctypes

import numpy as np
import pytest
import torch

import indexer_top_sparse_score_gb300 as smla
from indexer_top_sparse_score_gb300 import workloads as wl
from tests.gpu_common import TOL

pytestmark = pytest.mark.gpu


def _noalloc(L, dev, spec, out, lse):
    c = smla.make_cache(dev.cache)
    return L.smla_sparse_mla_prefill_noalloc(
        ctypes.byref(c), dev.page_table.data_ptr(), spec.prefix_len, spec.n_tokens, dev.q.data_ptr(),
        spec.n_heads, dev.q_idx.data_ptr(), dev.w.data_ptr(), spec.h_idx, spec.topk, float(spec.sm_scale),
        out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,T,P", [("prefill16k", 1500, 700), ("tiny", 1024, 0)])
def test_noalloc_prefill_matches_workspace_entry_on_two_calls(name, T, P):
    smla.build()
    L = smla.lib()
    spec = wl.scaled(wl.SPECS[name], n_tokens=T, prefix_len=P, shuffled=True)
    dev = wl.make(spec, "cuda")
    ref_out, ref_lse, _, ws = smla.sparse_mla_prefill(dev.cache, dev.page_table, P, dev.q, dev.q_idx, dev.w,
                                                      spec.topk, spec.sm_scale)
    assert smla.read_status(ws)[0] == 0
    ro = ref_out.float().cpu().numpy().astype(np.float64)
    rl = ref_lse.cpu().numpy()
    tol = TOL[spec.kv_dtype]
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _noalloc(L, dev, spec, out, lse) == 0
        torch.cuda.synchronize()
        g = out.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        rel = np.linalg.norm(g - ro) / np.linalg.norm(ro)
        assert rel <= tol["rel_l2"], rel
        assert np.abs(g - ro).max() <= tol["max_abs"]
        assert np.allclose(lse.cpu().numpy(), rl, atol=1e-3)


def test_noalloc_prefill_rejects_oversize_call():
    smla.build()
    L = smla.lib()
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=2048, prefix_len=0)   # 2048 * 2048 * 4 + 256 > 16 MiB
    dev = wl.make(spec, "cuda")
    out = torch.empty((spec.n_tokens, spec.n_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((spec.n_tokens, spec.n_heads), dtype=torch.float32, device="cuda")
    assert _noalloc(L, dev, spec, out, lse) == 3  # SMLA_ERR_WORKSPACE, nothing enqueued
