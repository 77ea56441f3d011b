"""Host-side logic that needs no GPU: the chunk schedule of the host-buffer
prefill and the e2e schedule the bench uses."""
import sys

import pytest

import indexer_top_sparse_score_gb300 as smla


def test_chunk_bounds_even_and_ragged():
    assert smla.chunk_bounds(3000, 1024) == [(0, 1024), (1024, 2048), (2048, 3000)]
    assert smla.chunk_bounds(2048, 2048) == [(0, 2048)]
    assert smla.chunk_bounds(5, 8) == [(0, 5)]


def test_chunk_bounds_explicit_sizes():
    assert smla.chunk_bounds(3000, [200, 800, 1000, 1000]) == [(0, 200), (200, 1000), (1000, 2000),
                                                                (2000, 3000)]
    with pytest.raises(ValueError):
        smla.chunk_bounds(3000, [1000, 1000])          # does not cover the tokens
    with pytest.raises(ValueError):
        smla.chunk_bounds(3000, [3000, 0])             # empty chunk
    with pytest.raises(ValueError):
        smla.chunk_bounds(3000, 0)


def test_bench_chunk_schedule_covers_workloads():
    """The long prefill is timed as 16 calls of 8,192 query tokens against the
    growing cache; the other prefills as one call after their prefix."""
    sys.argv = ["bench.py"]
    import bench
    from indexer_top_sparse_score_gb300 import workloads as wl
    c = bench.chunk_list(wl.SPECS["prefill128k"])
    assert c == [(8192 * i, 8192) for i in range(16)]
    assert bench.chunk_list(wl.SPECS["prefix1m"]) == [(1 << 20, 8192)]
    assert bench.chunk_list(wl.SPECS["prefill16k"]) == [(0, 16384)]
    assert bench.chunk_list(wl.scaled(wl.SPECS["prefill128k"], n_tokens=20000)) == [(0, 8192), (8192, 8192),
                                                                                       (16384, 3616)]


def test_bench_stage_counts_match_the_workload_sizing():
    """The per-kernel FLOP counts of a bench step reproduce the sizing of the
    workloads: ~70.4 TFLOP of indexer and ~37.1 TFLOP of attention for the
    131,072-token prefill, ~70.6 and ~2.34 TFLOP for the 1M-token prefix."""
    sys.argv = ["bench.py"]
    import bench
    from indexer_top_sparse_score_gb300 import workloads as wl
    pk = dict(hbm=1.0, bf16=1.0, bf16_sust=1.0, src="test")
    cnt, _ = bench.stage_report(wl.SPECS["prefill128k"], 1.0, 1.0, pk)
    assert round(cnt["idx_flops"] / 1e12, 1) == 70.4 and round(cnt["mla_flops"] / 1e12, 1) == 37.1
    cnt, _ = bench.stage_report(wl.SPECS["prefix1m"], 1.0, 1.0, pk)
    assert round(cnt["idx_flops"] / 1e12, 1) == 70.6 and round(cnt["mla_flops"] / 1e12, 2) == 2.34
    cnt, _ = bench.stage_report(wl.SPECS["prefill16k"], 1.0, 1.0, pk)
    assert round(cnt["idx_flops"] / 1e12, 2) == 1.10 and round(cnt["mla_flops"] / 1e12, 2) == 4.38


def test_bench_launch_count_matches_the_measured_launch_lists(monkeypatch):
    """The bench's `gpu_launches` comes from PrefillStep.launches(), which
    mirrors the library's score-array block rule. On a 152-SM GB300 it must give
    the launch counts of the committed ncu launch lists: 62 per 131,072-token
    step (16 indexers, 14 selections, 16 f16 copies, 16 attentions), 8 for the
    1M-token prefix (three row blocks: 3 indexers, 3 selections, the copy, the
    attention) and 3 for the 16K prefill (rows within the dense mode)."""
    import types

    import torch
    sys.argv = ["bench.py"]
    import bench
    from indexer_top_sparse_score_gb300 import workloads as wl
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda i: types.SimpleNamespace(multi_processor_count=152))

    def launches(spec):
        step = object.__new__(bench.PrefillStep)  # no device buffers: only the schedule is read
        step.spec, step.chunks = spec, bench.chunk_list(spec)
        return step.launches()

    assert launches(wl.SPECS["prefill128k"]) == 62
    assert launches(wl.SPECS["prefix1m"]) == 8
    assert launches(wl.SPECS["prefill16k"]) == 3


def test_output_checker_catches_one_wrong_head_and_one_wrong_lse():
    """The GPU parity checker (per-(row, head) bound on top of the aggregate bar):
    outputs rounded like the kernel's pass; one (row, head) among 128 x 64 that is
    5% off fails although the aggregate rel-L2 and the max-abs bars pass; one
    wrong lse fails."""
    import numpy as np
    import torch
    from tests.gpu_common import compare_out
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((128, 64, 512)) * 0.04
    lse = 8.0 + rng.standard_normal((128, 64))
    got = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()  # bf16 output rounding
    for kv in ("bf16", "fp8"):
        compare_out(got, ref, lse.astype(np.float32), lse, kv)
        bad = got.copy()
        bad[77, 5] *= 1.05
        with pytest.raises(AssertionError, match="row, head"):
            compare_out(bad, ref, lse.astype(np.float32), lse, kv)
        bl = lse.copy()
        bl[3, 60] += 0.1
        with pytest.raises(AssertionError, match="lse"):
            compare_out(got, ref, bl.astype(np.float32), lse, kv)
    # a row with no usable key: out = 0 and lse = -inf on both sides
    ref2, lse2, got2 = ref.copy(), lse.copy(), got.copy()
    ref2[9], got2[9], lse2[9] = 0.0, 0.0, -np.inf
    compare_out(got2, ref2, lse2.astype(np.float32), lse2, "bf16")
    lse3 = lse2.copy()
    lse3[9, 0] = 1.0
    with pytest.raises(AssertionError):
        compare_out(got2, ref2, lse3.astype(np.float32), lse2, "bf16")
