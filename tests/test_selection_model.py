"""A CPU model of the selection steps of select_sampled_kernel (the exact
top-k of one score row), checked against brute force on many rows.

The kernel finds each row's top-k (score descending, position ascending) in
one read of the row: a sample of runs of 128 keys gives a threshold t_lo; every
key >= t_lo is staged; when k..6,144 keys were staged, a 4,096-bin histogram of
the staged keys over [t_lo, the sample's largest key] (larger keys counted in
the top bin) gives the bin of the k-th staged key, and when that bin holds at
most 32 keys they are ranked by (key descending, position ascending) to give
the threshold (key, position). Otherwise the kernel falls back to digit rounds
over the staged keys or to an exact selection over the whole row; both are
plain definitions of the top-k, modelled here as such.

The model follows the kernel's integer arithmetic (bins, clamping, the
top-down scan, the rank inside the bin) so that a wrong bin edge, a missed
clamp, a reversed tie rule or an off-by-one in the rank makes it disagree
with brute force on some row. Keys are the kernel's order-preserving 32-bit
images of fp32 scores."""
import math

import numpy as np
import pytest

CAND = 6144          # staged candidates
BINS = 4096          # 12-bit digits
MIN_RUNS, MAX_RUNS = 32, 96
LIST = 32            # keys of the k-th key's bin ranked by one warp


def score_keys(scores: np.ndarray) -> np.ndarray:
    """Order-preserving uint32 image of fp32 scores (-0 folded into +0 by
    adding +0; negative: all bits flipped; non-negative: sign bit set)."""
    b = (np.asarray(scores, dtype=np.float32) + np.float32(0.0)).view(np.uint32)
    neg = (b >> 31) == 1
    return np.where(neg, ~b, b | np.uint32(0x80000000)).astype(np.uint32)


def shift_for(lo: int, hi: int) -> int:
    rng = hi - lo
    return (rng.bit_length() - 12) if rng >= BINS else 0


def scan_top(hist: np.ndarray, r: int):
    """The bin holding the r-th largest counted key (1-based r) and the number
    of keys in higher bins."""
    above = 0
    for b in range(BINS - 1, -1, -1):
        if above + int(hist[b]) >= r:
            return b, above
        above += int(hist[b])
    raise AssertionError("fewer than r keys counted")


def brute_topk(keys: np.ndarray, k: int) -> np.ndarray:
    order = np.lexsort((np.arange(keys.size), -keys.astype(np.int64)))
    return np.sort(order[:k])


def model_select(keys: np.ndarray, k: int, plant=None):
    """The selected positions (ascending) and the path the kernel takes.
    `plant` puts a mistake into the model (for the test that shows the
    comparison catches it): "tie_rule" (highest position wins a tie),
    "rank" (the entry after the needed rank), "clamp" (keys above the sample's
    largest not counted in the top bin)."""
    n = keys.size
    if n <= k:
        return np.arange(n), "all"
    t_lo, h_shift = 0, -1
    if n > CAND:
        runs = min(MAX_RUNS, max(MIN_RUNS, n // 2048))
        n_sample = runs * 128
        starts = [((n - 128) * run // (runs - 1)) & ~3 for run in range(runs)]
        sample = np.concatenate([keys[s:s + 128] for s in starts]).astype(np.int64)
        lo, hi = int(sample.min()), int(sample.max())
        expect = np.float32(k) * np.float32(n_sample) / np.float32(n)
        r = int(math.ceil(np.float32(1.1) * expect + np.float32(3.0) * np.sqrt(expect) + np.float32(3.0)))
        if r < n_sample:
            sh = shift_for(lo, hi)
            hist = np.bincount((sample - lo) >> sh, minlength=BINS)
            assert hist.size == BINS, "a sample key outside [lo, hi]"
            b, _ = scan_top(hist, r)
            t_lo = lo + (b << sh)
            h_shift = shift_for(t_lo, hi)
    staged = np.nonzero(keys >= t_lo)[0]
    nc = staged.size
    if not (k <= nc <= CAND):
        return brute_topk(keys, k), "whole_row"
    if nc == k:
        return staged, "all_staged"
    if h_shift < 0:
        return brute_topk(keys, k), "digits"
    sk = keys[staged].astype(np.int64)
    bins = (sk - t_lo) >> h_shift
    bins = bins if plant == "clamp" else np.minimum(bins, BINS - 1)
    hist = np.bincount(bins, minlength=BINS)[:BINS]
    if hist.sum() < k:
        return np.nonzero(bins >= 0)[0][:0], "lost_keys"
    b, above = scan_top(hist, k)
    r, m = k - above, int(hist[b])
    assert 1 <= r <= m
    if m > LIST:
        return brute_topk(keys, k), "digits"
    in_bin = staged[bins == b]
    assert in_bin.size == m
    # lane j ranks entry j: entries before it by (key desc, position asc)
    kb = keys[in_bin].astype(np.int64)
    before = (lambda a, b: a > b) if plant == "tie_rule" else (lambda a, b: a < b)
    rank = np.array([int(((kb > kb[j]) | ((kb == kb[j]) & before(in_bin, in_bin[j]))).sum()) for j in range(m)])
    want = min(r, m - 1) if plant == "rank" else r - 1
    j = int(np.nonzero(rank == want)[0][0])
    tk, ti = int(kb[j]), int(in_bin[j])
    pos = np.arange(n)
    sel = (keys.astype(np.int64) > tk) | ((keys.astype(np.int64) == tk) & (pos <= ti))
    return np.nonzero(sel)[0], "bin_rank"


def _rows(rng):
    """(name, keys, k) cases: the workloads' row lengths and k, small k,
    few distinct scores, tie groups, a crowded top, negative scores."""
    for n in (6000, 6145, 17001, 40000, 131072):
        for k in (1, 7, 100, 2048):
            yield f"normal-n{n}-k{k}", score_keys(rng.standard_normal(n)), k
    for n in (20000, 70000):
        yield f"relu-sum-n{n}", score_keys(np.maximum(rng.standard_normal((n, 8)), 0) @ rng.random(8)), 2048
        yield f"few-values-n{n}", score_keys(rng.integers(0, 50, n).astype(np.float32)), 2048
        v = rng.standard_normal(n).astype(np.float32)
        src = rng.integers(0, n, n // 4)
        v[rng.integers(0, n, n // 4)] = v[src]  # tie groups
        yield f"tie-groups-n{n}", score_keys(v), 2048
        v = rng.standard_normal(n).astype(np.float32)
        v[rng.choice(n, 3000, replace=False)] = 9.0  # 3000 equal keys above the rest
        yield f"crowded-top-n{n}", score_keys(v), 2048
        yield f"constant-n{n}", score_keys(np.full(n, 0.5, dtype=np.float32)), 2048
        yield f"signed-n{n}", score_keys(rng.standard_normal(n) * 1e3), 512


def test_score_keys_preserve_order():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000),
                        [0.0, -0.0, 1e-45, -1e-45, 3.4e38, -3.4e38]]).astype(np.float32)
    order_f = np.argsort(v, kind="stable")
    kv = score_keys(v)
    assert (np.diff(kv[order_f].astype(np.int64)) >= 0).all()


def test_model_selection_equals_brute_force():
    rng = np.random.default_rng(7)
    paths = {}
    for name, keys, k in _rows(rng):
        got, path = model_select(keys, k)
        want = brute_topk(keys, k)
        assert np.array_equal(got, want), f"{name}: {path} selects another set"
        paths.setdefault(path, []).append(name)
    # the cases reach every path of the kernel
    assert {"bin_rank", "digits", "whole_row"} <= set(paths), paths.keys()
    # random rows of the workloads' sizes take the one-bin ranking
    assert all(f"normal-n{n}-k2048" in paths["bin_rank"] for n in (17001, 40000, 131072))


@pytest.mark.parametrize("k", [1, 7])
def test_small_k_lands_in_the_clamped_top_bin(k):
    """With k far below n / n_sample the k-th key lies above the sample's
    largest key: it is counted in the top bin, which the scan must reach."""
    rng = np.random.default_rng(11 + k)
    hits = 0
    for _ in range(20):
        keys = score_keys(rng.standard_normal(131072))
        got, path = model_select(keys, k)
        assert np.array_equal(got, brute_topk(keys, k))
        n = keys.size
        runs = min(MAX_RUNS, max(MIN_RUNS, n // 2048))
        starts = [((n - 128) * run // (runs - 1)) & ~3 for run in range(runs)]
        s_max = max(int(keys[s:s + 128].max()) for s in starts)
        hits += int(np.sort(keys)[-k]) > s_max
    assert hits > 0


@pytest.mark.parametrize("plant", ["tie_rule", "rank", "clamp"])
def test_planted_mistakes_are_caught(plant):
    """A reversed tie rule inside the bin, an off-by-one rank, or keys above the
    sample's largest dropped from the count: each makes the model disagree with
    brute force on some row of the same suite."""
    rng = np.random.default_rng(7)
    wrong = []
    for name, keys, k in _rows(rng):
        got, path = model_select(keys, k, plant=plant)
        if not np.array_equal(got, brute_topk(keys, k)):
            wrong.append(name)
    assert wrong, f"planted {plant} went unnoticed"
