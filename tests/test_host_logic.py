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


def test_bench_e2e_schedule_tapers_and_covers():
    sys.argv = ["bench.py"]
    import bench
    c = bench.e2e_chunks(16384)
    assert sum(c) == 16384 and c[:3] == [256, 768, 1024] and c[-3:] == [1024, 768, 256]
    assert set(c[3:-3]) == {bench.E2E_CHUNK}
    b = smla.chunk_bounds(16384, c)
    assert b[0][0] == 0 and b[-1][1] == 16384 and all(x[1] == y[0] for x, y in zip(b, b[1:]))
    assert bench.e2e_chunks(4096) == bench.E2E_CHUNK   # too short to taper: even chunks
