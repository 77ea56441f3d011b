"""The workspace-free prefill entry point, for callers that cannot allocate
device memory: a plugin that is handed only input and output pointers by its
host framework, or an engine whose device memory all belongs to a pool that
outside code may not draw from. Its scratch is a fixed array inside the
library that keeps the previous call's contents, so every case runs the entry
more than once. It runs the same kernels on the same bytes as the regular
entry point, so where both take the same path (rows of at most 16,384 keys)
the outputs must be bit-identical; sampled rows are also checked against the
oracle. This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import indexer_top_sparse_score_gb300 as smla
import oracle
from indexer_top_sparse_score_gb300 import workloads as wl
from tests.gpu_common import compare_out, sampled_oracle

pytestmark = pytest.mark.gpu

BOUNDS = 5


@pytest.fixture(scope="module")
def L():
    smla.build()
    oracle.build()
    return smla.lib()


def _noalloc(L, dev, spec, out, lse, page_table=None):
    c = smla.make_cache(dev.cache)
    pt = dev.page_table if page_table is None else page_table
    return L.smla_sparse_mla_prefill_noalloc(
        ctypes.byref(c), pt.data_ptr(), spec.prefix_len, spec.n_tokens, dev.q.data_ptr(),
        spec.n_heads, dev.q_idx.data_ptr(), dev.w.data_ptr(), spec.h_idx, spec.topk, float(spec.sm_scale),
        out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _noalloc_status(L):
    bits = ctypes.c_uint32(0)
    rc = L.smla_noalloc_read_status(torch.cuda.current_stream().cuda_stream, ctypes.byref(bits))
    return rc, bits.value


def _reference(dev, spec):
    out, lse, _, ws = smla.sparse_mla_prefill(dev.cache, dev.page_table, spec.prefix_len, dev.q, dev.q_idx, dev.w,
                                              spec.topk, spec.sm_scale)
    assert smla.read_status(ws)[0] == 0
    return out, lse


def _run_and_compare(L, spec, dev, ref_out, ref_lse, exact=True):
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    assert _noalloc(L, dev, spec, out, lse) == 0
    assert _noalloc_status(L) == (0, 0)
    if exact:
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)
    else:
        compare_out(out.float().cpu().numpy(), ref_out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy(),
                    ref_lse.cpu().numpy().astype(np.float64), spec.kv_dtype)
    return out, lse


CASES = {
    # BF16 cache, the f16 copy of the rows fits in the array
    "bf16-shadow": ("prefill16k", 1500, 700, "bf16"),
    # the tiny workload in full (16 heads, 4x64 BF16 indexer, top-256)
    "tiny": ("tiny", 1024, 0, "bf16"),
    # BF16 cache whose f16 copy does not fit beside the index list: rows widened in the kernel
    "bf16-no-shadow": ("prefill16k", 1900, 14000, "bf16"),
    # FP8 cache with per-token scales
    "fp8": ("prefill16k", 2000, 5000, "fp8"),
    # 656-byte tile-scaled FP8 rows (512 e4m3 values, a scale per 128, 64 bf16 rope values)
    "fp8_ds_mla": ("prefill16k", 1200, 2500, wl.FP8_DS_MLA),
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_bit_identical_to_workspace_entry_and_matches_oracle(L, case):
    name, T, P, kv = CASES[case]
    spec = wl.scaled(wl.SPECS[name], n_tokens=T, prefix_len=P, shuffled=True, kv_dtype=kv)
    dev = wl.make(spec, "cuda")
    ref_out, ref_lse = _reference(dev, spec)
    for _ in range(2):
        out, lse = _run_and_compare(L, spec, dev, ref_out, ref_lse)
    rows = np.array(sorted({0, 1, T // 3, T - 2, T - 1}), dtype=np.int64)
    _, _, rout, rlse, _ = sampled_oracle(dev, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_out(out[r].float().cpu().numpy(), rout, lse[r].cpu().numpy(), rlse, kv)


def test_noalloc_large_call_then_small_then_large(L):
    """A call leaves its index list and f16 copy in the array; a smaller call
    after a larger one, and a larger one after that, still equal the regular
    entry point bit for bit."""
    specs = [wl.scaled(wl.SPECS["prefill16k"], n_tokens=T, prefix_len=P, shuffled=True, seed=1002 + i)
             for i, (T, P) in enumerate([(2000, 3000), (300, 500), (1700, 9000)])]
    devs = [wl.make(s, "cuda") for s in specs]
    refs = [_reference(d, s) for d, s in zip(devs, specs)]
    for s, d, (ro, rl) in zip(specs, devs, refs):
        _run_and_compare(L, s, d, ro, rl)
    s, d = specs[1], devs[1]
    out, lse = _run_and_compare(L, s, d, *refs[1])
    rows = np.array([0, 150, 299], dtype=np.int64)
    _, _, rout, rlse, _ = sampled_oracle(d, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_out(out[r].float().cpu().numpy(), rout, lse[r].cpu().numpy(), rlse, "bf16")


def test_noalloc_rows_longer_than_the_dense_mode(L):
    """Rows of more than 16,384 keys: the regular entry point defers their final
    selection to a separate kernel, this one selects inside the scoring kernel
    (the array has no room for the candidate buffers). Same index sets, so the
    outputs agree within the tolerances, and sampled rows match the oracle."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=1000, prefix_len=20000, shuffled=True, kv_dtype="fp8")
    dev = wl.make(spec, "cuda")
    ref_out, ref_lse = _reference(dev, spec)
    for _ in range(2):
        out, lse = _run_and_compare(L, spec, dev, ref_out, ref_lse, exact=False)
    rows = np.array([0, 500, 998, 999], dtype=np.int64)
    _, _, rout, rlse, _ = sampled_oracle(dev, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_out(out[r].float().cpu().numpy(), rout, lse[r].cpu().numpy(), rlse, "fp8")


def test_noalloc_reports_device_errors(L):
    """A page id outside the pool is skipped on the device and reported through
    smla_noalloc_read_status; the next good call clears the report."""
    spec = wl.scaled(wl.SPECS["tiny"], n_tokens=200, prefix_len=300)
    dev = wl.make(spec, "cuda")
    pt = dev.page_table.clone()
    pt[2] = dev.cache.num_pages + 5
    out = torch.empty((spec.n_tokens, spec.n_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((spec.n_tokens, spec.n_heads), dtype=torch.float32, device="cuda")
    assert _noalloc(L, dev, spec, out, lse, page_table=pt) == 0
    rc, bits = _noalloc_status(L)
    assert rc == BOUNDS and bits & 1
    assert _noalloc(L, dev, spec, out, lse) == 0
    assert _noalloc_status(L) == (0, 0)


def test_noalloc_prefill_rejects_oversize_call(L):
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=2048, prefix_len=0)   # 2048 * 2048 * 4 + 256 > 16 MiB
    dev = wl.make(spec, "cuda")
    out = torch.empty((spec.n_tokens, spec.n_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((spec.n_tokens, spec.n_heads), dtype=torch.float32, device="cuda")
    assert _noalloc(L, dev, spec, out, lse) == 3  # SMLA_ERR_WORKSPACE, nothing enqueued
