"""CUDA path vs the CPU oracle on seeded inputs (needs a GB300).

Index sets must match bit for bit (integer-valued indexer inputs make every
score exact); attention outputs must match within the tolerances fixed for
the layer step. Small workloads are compared row by row in full; the large
ones at their full sizes on stratified samples of rows.
"""
import numpy as np
import pytest
import torch

import indexer_top_sparse_score_gb300 as smla
import oracle
from indexer_top_sparse_score_gb300 import workloads as wl
from tests.gpu_common import (compare_idx, compare_out, host_cache, indexer_ws, run_prefill, sampled_oracle,
                              stratified_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    smla.build()
    oracle.build()
    smla.lib()


def _host(t):
    return t.cpu().numpy()


def test_tiny_prefill_full():
    """Workload 1 (T=1024, 16 heads, 4x64 BF16 indexer, top-256) in full."""
    spec = wl.SPECS["tiny"]
    prob = wl.make(spec, "cpu")
    dev = prob.to("cuda")
    idx, out, lse = run_prefill(dev)
    ridx, _, rout, rlse, _, bad = oracle.Oracle(prob).rows(np.arange(spec.n_tokens))
    assert not bad.any()
    compare_idx(_host(idx), ridx)
    compare_out(_host(out.float()), rout, _host(lse), rlse, spec.kv_dtype)


def test_indexer_scores_and_sets_group_mode():
    spec = wl.scaled(wl.SPECS["tiny"], n_tokens=777, prefix_len=333, shuffled=True)
    prob = wl.make(spec, "cpu")
    dev = prob.to("cuda")
    L = spec.prefix_len + spec.n_tokens
    seq_lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    gidx, gsc, ws = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, L, spec.n_tokens, dev.q_idx,
                                      dev.w, spec.topk, want_scores=True)
    assert smla.read_status(ws)[0] == 0
    o = oracle.Oracle(prob)
    ridx, rsc, *_ = o.rows(np.arange(spec.n_tokens), attend=False)
    compare_idx(_host(gidx), ridx)
    g_i, g_s = _host(gidx), _host(gsc)
    for r in range(0, spec.n_tokens, 37):
        full = o.scores(r)
        ok = g_i[r] >= 0
        assert np.array_equal(g_s[r][ok], full[g_i[r][ok]])


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_prefill_ragged_prefix_shuffled(kv_dtype):
    """64 heads, 32x128 FP8 indexer, top-2048; T not a multiple of the CTA's
    token group, a cached prefix, shuffled pages; rows sampled around t = k."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=3001, prefix_len=1500, shuffled=True,
                     kv_dtype=kv_dtype)
    dev = wl.make(spec, "cuda")
    idx, out, lse = run_prefill(dev)
    rows = stratified_rows(spec.prefix_len, spec.n_tokens, spec.topk, n_random=20)
    ridx, _, rout, rlse, _ = sampled_oracle(dev, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_idx(_host(idx[r]), ridx)
    compare_out(_host(out[r].float()), rout, _host(lse[r]), rlse, kv_dtype)


def test_prefill16k_full_size_sampled():
    """Workload 2 at its full size (the benchmarked configuration), sampled rows."""
    spec = wl.SPECS["prefill16k"]
    dev = wl.make(spec, "cuda")
    idx, out, lse = run_prefill(dev)
    rows = stratified_rows(0, spec.n_tokens, spec.topk, extra=(4095, 4096, 8191, 8192, 12287), n_random=480)
    ridx, _, rout, rlse, _ = sampled_oracle(dev, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_idx(_host(idx[r]), ridx)
    compare_out(_host(out[r].float()), rout, _host(lse[r]), rlse, spec.kv_dtype)
    # every row: valid entries first, unique, causal
    ih = _host(idx)
    for t in range(0, spec.n_tokens, 997):
        n = min(spec.topk, t + 1)
        v = ih[t, :n]
        assert (v >= 0).all() and (v <= t).all() and len(np.unique(v)) == n
        assert (ih[t, n:] == -1).all()


def test_prefill128k_chunked_sampled():
    """Workload 3: 131072 tokens, FP8 KV, in 8192-token chunks against the growing cache."""
    spec = wl.SPECS["prefill128k"]
    dev = wl.make(spec, "cuda")
    idx, out, lse = run_prefill(dev, chunk=spec.chunk)
    # every 8,192-token chunk edge, rows around t = k, and random rows (~530 in all)
    edges = [c * spec.chunk + d for c in range(1, 16) for d in (-1, 0, 1)]
    rows = stratified_rows(0, spec.n_tokens, spec.topk, extra=edges, n_random=480)
    ridx, _, rout, rlse, _ = sampled_oracle(dev, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_idx(_host(idx[r]), ridx)
    compare_out(_host(out[r].float()), rout, _host(lse[r]), rlse, spec.kv_dtype)


def test_prefix1m_sampled():
    """Workload 5: 8192 new tokens after a 1,048,576-token prefix, paged and shuffled."""
    spec = wl.SPECS["prefix1m"]
    dev = wl.make(spec, "cuda")
    idx, out, lse = run_prefill(dev)
    # first and last rows, rows at page boundaries of the new tokens (position
    # P + t with (P + t) % 64 in {0, 63}) and random rows: 64 in all
    rng = np.random.default_rng(5)
    fixed = {0, 1, 2, 63, 64, 127, 128, 4095, 4096, 8127, 8128, 8190, 8191}
    rnd = set(rng.choice(spec.n_tokens, 64, replace=False).tolist()) - fixed
    rows = np.array(sorted(fixed | set(sorted(rnd)[:64 - len(fixed)])), dtype=np.int64)
    assert len(rows) == 64
    ridx, _, rout, rlse, _ = sampled_oracle(dev, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_idx(_host(idx[r]), ridx)
    compare_out(_host(out[r].float()), rout, _host(lse[r]), rlse, spec.kv_dtype)


def test_decode_mtp_full():
    """Workload 4: 64 requests x 2 MTP tokens, contexts 8K-128K, shuffled paged pool; every row."""
    spec = wl.SPECS["decode"]
    dev = wl.make(spec, "cuda")
    rows = spec.n_seqs * spec.q_per_seq
    max_len = int(dev.seq_lens.max())
    idx = torch.empty((rows, spec.topk), dtype=torch.int32, device="cuda")
    out, lse, _, ws = smla.sparse_mla_decode(dev.cache, dev.page_table, dev.seq_lens, max_len, spec.q_per_seq,
                                             dev.q, dev.q_idx, dev.w, spec.topk, spec.sm_scale, out_idx=idx)
    assert smla.read_status(ws)[0] == 0
    prob = dev.to("cpu")
    ridx, _, rout, rlse, _, bad = oracle.Oracle(prob).rows(np.arange(rows))
    assert not bad.any()
    compare_idx(_host(idx), ridx)
    compare_out(_host(out.float()), rout, _host(lse), rlse, spec.kv_dtype)


def test_decode_small_batch_single_token():
    """Plain decode (one query per request), BF16 cache, short contexts below k."""
    spec = wl.scaled(wl.SPECS["decode"], n_seqs=5, q_per_seq=1, len_min=100, len_max=9000, kv_dtype="bf16",
                     seed=77)
    dev = wl.make(spec, "cuda")
    max_len = int(dev.seq_lens.max())
    idx = torch.empty((spec.n_seqs, spec.topk), dtype=torch.int32, device="cuda")
    out, lse, _, ws = smla.sparse_mla_decode(dev.cache, dev.page_table, dev.seq_lens, max_len, 1, dev.q,
                                             dev.q_idx, dev.w, spec.topk, spec.sm_scale, out_idx=idx)
    assert smla.read_status(ws)[0] == 0
    prob = dev.to("cpu")
    ridx, _, rout, rlse, _, bad = oracle.Oracle(prob).rows(np.arange(spec.n_seqs))
    compare_idx(_host(idx), ridx)
    compare_out(_host(out.float()), rout, _host(lse), rlse, "bf16")


def test_sparse_mla_given_indices_with_holes():
    """Caller-given index lists with -1 holes, duplicates-free random keys, FP8 cache."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=300, prefix_len=5000, kv_dtype="fp8", topk=512,
                     shuffled=True)
    dev = wl.make(spec, "cuda")
    g = torch.Generator().manual_seed(5)
    T, k = spec.n_tokens, spec.topk
    idx = torch.empty((T, k), dtype=torch.int32)
    for t in range(T):
        pos = spec.prefix_len + t
        perm = torch.randperm(pos + 1, generator=g)[:k].to(torch.int32)
        holes = torch.rand(k, generator=g) < 0.1
        perm[holes] = -1
        idx[t] = perm
    out, lse, ws = smla.sparse_mla_fwd(dev.cache, dev.page_table, dev.q, idx.cuda(), spec.sm_scale,
                                       prefix_len=spec.prefix_len)
    assert smla.read_status(ws)[0] == 0
    prob = dev.to("cpu")
    o = oracle.Oracle(prob)
    rows = np.arange(0, T, 7)
    rout, rlse = o.attend_rows(rows, idx.numpy()[rows])
    compare_out(_host(out.float())[rows], rout, _host(lse)[rows], rlse, "fp8")


def test_out_of_range_page_is_reported_not_faulted():
    """A page id outside the pool is skipped on the device and reported by read_status."""
    spec = wl.scaled(wl.SPECS["tiny"], n_tokens=200, prefix_len=300)
    dev = wl.make(spec, "cuda")
    pt = dev.page_table.clone()
    pt[2] = dev.cache.num_pages + 5
    out, lse, _, ws = smla.sparse_mla_prefill(dev.cache, pt, spec.prefix_len, dev.q, dev.q_idx, dev.w,
                                              spec.topk, spec.sm_scale)
    rc, bits = smla.read_status(ws)
    assert rc == 5 and bits & 1
    # the same call with the good table is clean again (the status word is reset per call)
    smla.sparse_mla_prefill(dev.cache, dev.page_table, spec.prefix_len, dev.q, dev.q_idx, dev.w, spec.topk,
                            spec.sm_scale, ws=ws)
    assert smla.read_status(ws)[0] == 0


def test_repeat_calls_same_sets():
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=2500, prefix_len=0)
    dev = wl.make(spec, "cuda")
    a, oa, la = run_prefill(dev)
    b, ob, lb = run_prefill(dev)
    assert torch.equal(torch.sort(a, dim=1).values, torch.sort(b, dim=1).values)
    assert (oa.float() - ob.float()).abs().max().item() < 1e-2


@pytest.mark.parametrize("sel", ["dense", "scores", "streaming", "in_kernel"])
@pytest.mark.parametrize("mode", ["constant", "binary"])
def test_indexer_heavy_ties(mode, sel):
    """Ties everywhere: constant keys (all scores equal -> the lowest k indices) and
    keys in {0,1} (few distinct scores); the lower index must win every tie. Rows
    of at most 16,384 keys take the dense group mode (every score in shared
    memory); longer rows the score array with the full workspace, the streaming
    candidate buffers with a workspace too small for the score array, and the
    selection inside the scoring kernel with the status word alone."""
    prefix = 6000 if sel == "dense" else 17000
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=700, prefix_len=prefix, shuffled=True)
    prob = wl.make(spec, "cpu")
    k = prob.cache.k_idx
    if mode == "constant":
        row = k.view(-1, spec.d_idx)[0].clone()
        k.view(-1, spec.d_idx)[:] = row
    else:
        g = torch.Generator().manual_seed(3)
        v = torch.randint(0, 2, k.shape, generator=g).to(torch.float32)
        k.copy_(v.to(torch.float8_e4m3fn).view(torch.uint8))
    dev = prob.to("cuda")
    L = spec.prefix_len + spec.n_tokens
    seq_lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    ws = indexer_ws(spec.n_tokens, {"streaming": "cand", "in_kernel": "min"}[sel]) \
        if sel in ("streaming", "in_kernel") else None
    gidx, ws = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, L, spec.n_tokens, dev.q_idx, dev.w,
                                 spec.topk, ws=ws)
    assert smla.read_status(ws)[0] == 0
    rows = np.arange(0, spec.n_tokens, 23)
    ridx, *_ = oracle.Oracle(prob).rows(rows, attend=False)
    compare_idx(_host(gidx)[rows], ridx)
    if mode == "constant":
        assert (np.sort(_host(gidx)[rows], axis=1) == np.arange(spec.topk)[None, :]).all()


@pytest.mark.parametrize("case", ["one_seq", "two_seqs"])
def test_indexer_score_array_row_blocks(case):
    """The score-array mode in several row blocks (a workspace holding one
    block of 700 rows, or 608 rows of each of two sequences; blocks smaller
    than a wave of work items are made equal): the rows of every block match
    the oracle, the rows at block boundaries included, and the index sets
    equal those of a call with the full workspace (one block)."""
    if case == "one_seq":
        spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=2000, prefix_len=18000, shuffled=True)
        prob = wl.make(spec, "cpu")
        dev = prob.to("cuda")
        n_seqs, qps, block = 1, spec.n_tokens, 700
        max_len = spec.prefix_len + spec.n_tokens
        seq_lens = torch.tensor([max_len], dtype=torch.int32, device="cuda")
        # room for 700 rows: three equal blocks of 668, 668 and 664 rows
        rows = sorted({0, 1, 667, 668, 669, 1335, 1336, 1999} | set(range(3, 2000, 97)))
    else:
        spec = wl.scaled(wl.SPECS["decode"], n_seqs=2, q_per_seq=900, len_min=18000, len_max=26000, seed=7)
        prob = wl.make(spec, "cpu")
        dev = prob.to("cuda")
        n_seqs, qps, block = 2, 900, 608
        seq_lens = dev.seq_lens
        max_len = int(seq_lens.max())
        # room for 608 rows of each sequence: two equal blocks of 452 and 448 rows
        rows = sorted({0, 451, 452, 899, 900, 1351, 1352, 1799} | set(range(5, 1800, 89)))
    stride = (max_len + 31) // 32 * 32
    ws = smla.workspace(256 + n_seqs * block * stride * 4, "cuda")
    gidx, ws = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, max_len, qps, dev.q_idx, dev.w, spec.topk,
                                 ws=ws)
    assert smla.read_status(ws)[0] == 0
    full, ws2 = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, max_len, qps, dev.q_idx, dev.w, spec.topk)
    assert smla.read_status(ws2)[0] == 0
    assert torch.equal(torch.sort(gidx, dim=1).values, torch.sort(full, dim=1).values)
    ridx, *_ = oracle.Oracle(prob).rows(np.array(rows), attend=False)
    compare_idx(_host(gidx)[rows], ridx)


@pytest.mark.parametrize("keys", ["random", "constant"])
def test_indexer_rows_beyond_the_bitmap(keys):
    """Rows of more than 262,144 keys in the score-array mode: the selection
    kernel collects the k positions in shared memory and sorts them instead of
    marking a bitmap of the row. Random keys take the sampled path, all-equal
    keys (every score tied) the exact fallback over the whole row; index sets
    exact against the oracle, returned in ascending order."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=400, prefix_len=270000, shuffled=True)
    prob = wl.make(spec, "cpu")
    if keys == "constant":
        k = prob.cache.k_idx
        row = k.view(-1, spec.d_idx)[0].clone()
        k.view(-1, spec.d_idx)[:] = row
    dev = prob.to("cuda")
    L = spec.prefix_len + spec.n_tokens
    seq_lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    gidx, gsc, ws = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, L, spec.n_tokens, dev.q_idx, dev.w,
                                      spec.topk, want_scores=True)
    assert smla.read_status(ws)[0] == 0
    g = _host(gidx)
    assert (np.diff(g, axis=1) > 0).all(), "indices not ascending"
    rows = np.array([0, 1, 133, 398, 399], dtype=np.int64)
    o = oracle.Oracle(prob)
    ridx, rsc, *_ = o.rows(rows, attend=False)
    compare_idx(g[rows], ridx)
    if keys == "constant":
        assert (g == np.arange(spec.topk)[None, :]).all()
    gs = _host(gsc)
    for r in range(len(rows)):
        full = o.scores(int(rows[r]))
        assert np.array_equal(gs[rows[r]], full[g[rows[r]]])


@pytest.mark.parametrize("case", ["k1", "k7", "k100", "tie_groups"])
def test_indexer_selection_small_k_and_tie_groups(case):
    """Score-array rows of 17,001-17,700 keys through the sampled selection.
    With k = 1 or 7 the k-th key lies above the sample's largest key, in the
    top bin of the staged keys' histogram (where every larger key is counted);
    with k = 100 a few bins below it. tie_groups copies 3,000 key rows to 8
    other positions each (groups of 9 keys with equal scores in every row), so
    the bin of the k-th key often holds equal keys and the lowest positions
    must win inside it. Index sets and returned scores exact."""
    topk = {"k1": 1, "k7": 7, "k100": 100, "tie_groups": 2048}[case]
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=700, prefix_len=17000, shuffled=True, topk=topk)
    prob = wl.make(spec, "cpu")
    if case == "tie_groups":
        g = torch.Generator().manual_seed(41)
        kr = prob.cache.k_idx.view(-1, spec.d_idx)
        ks = prob.cache.k_idx_scale.view(-1) if prob.cache.k_idx_scale is not None else None
        n = kr.shape[0]
        for s in torch.randint(0, n, (3000,), generator=g).tolist():
            dst = torch.randint(0, n, (8,), generator=g)
            kr[dst] = kr[s].clone()
            if ks is not None:
                ks[dst] = ks[s].clone()
    dev = prob.to("cuda")
    L = spec.prefix_len + spec.n_tokens
    seq_lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    gidx, gsc, ws = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, L, spec.n_tokens, dev.q_idx, dev.w,
                                      topk, want_scores=True)
    assert smla.read_status(ws)[0] == 0
    g_idx, g_sc = _host(gidx), _host(gsc)
    assert (np.diff(g_idx, axis=1) > 0).all(), "indices not ascending"
    rows = np.arange(0, spec.n_tokens, 7)
    o = oracle.Oracle(prob)
    ridx, *_ = o.rows(rows, attend=False)
    compare_idx(g_idx[rows], ridx)
    for r in rows:
        full = o.scores(int(r))
        assert np.array_equal(g_sc[r], full[g_idx[r]])


def test_decode_rows_beyond_the_bitmap():
    """Decode sequences of 270K-300K keys (split mode, the selection's sorted
    output): every row's index set and the attention match the oracle."""
    spec = wl.scaled(wl.SPECS["decode"], n_seqs=2, len_min=270000, len_max=300000, seed=29)
    prob = wl.make(spec, "cpu")
    dev = prob.to("cuda")
    max_len = int(dev.seq_lens.max())
    out, lse, gidx, ws = smla.sparse_mla_decode(dev.cache, dev.page_table, dev.seq_lens, max_len, spec.q_per_seq,
                                                dev.q, dev.q_idx, dev.w, spec.topk, spec.sm_scale,
                                                out_idx=torch.empty((spec.n_seqs * spec.q_per_seq, spec.topk),
                                                                    dtype=torch.int32, device="cuda"))
    assert smla.read_status(ws)[0] == 0
    rows = np.arange(spec.n_seqs * spec.q_per_seq)
    ridx, _, rout, rlse, _, bad = oracle.Oracle(prob).rows(rows)
    assert not bad.any()
    compare_idx(_host(gidx), ridx)
    compare_out(_host(out.float()), rout, _host(lse), rlse, spec.kv_dtype)


@pytest.mark.parametrize("mode", ["constant", "binary"])
def test_decode_indexer_heavy_ties(mode):
    """Decode shape (split mode) with ties everywhere, rows from 2.5K to 20K keys:
    the dense per-row selection must keep the lowest indices among equal scores
    whether the threshold bin is staged in shared memory or not."""
    spec = wl.scaled(wl.SPECS["decode"], n_seqs=5, len_min=2500, len_max=20000, seed=91)
    prob = wl.make(spec, "cpu")
    k = prob.cache.k_idx
    if mode == "constant":
        row = k.view(-1, spec.d_idx)[0].clone()
        k.view(-1, spec.d_idx)[:] = row
    else:
        g = torch.Generator().manual_seed(5)
        v = torch.randint(0, 2, k.shape, generator=g).to(torch.float32)
        k.copy_(v.to(torch.float8_e4m3fn).view(torch.uint8))
    dev = prob.to("cuda")
    max_len = int(dev.seq_lens.max())
    gidx, ws = smla.indexer_topk(dev.cache, dev.page_table, dev.seq_lens, max_len, spec.q_per_seq, dev.q_idx,
                                 dev.w, spec.topk)
    assert smla.read_status(ws)[0] == 0
    rows = np.arange(spec.n_seqs * spec.q_per_seq)
    ridx, *_ = oracle.Oracle(prob).rows(rows, attend=False)
    compare_idx(_host(gidx), ridx)
    if mode == "constant":
        assert (np.sort(_host(gidx), axis=1) == np.arange(spec.topk)[None, :]).all()


@pytest.mark.parametrize("chunk", [1024, [200, 800, 1000, 1000]], ids=["even", "tapered"])
def test_host_prefill_chunks_match_single_call(chunk):
    """The host-buffer prefill (chunks of query tokens, each one prefill call with
    the earlier tokens as its prefix, the copies overlapped on two streams) returns
    exactly what one device call returns, on two runs in a row (the second reuses
    every device buffer), and its rows match the oracle."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=3000, prefix_len=500, shuffled=True)
    dev = wl.make(spec, "cuda")
    _, out, lse = run_prefill(dev, want_idx=False)
    hp = smla.HostPrefill(dev.cache, dev.page_table, spec.prefix_len, spec.n_tokens, spec.n_heads, spec.h_idx,
                          spec.d_idx, spec.idx_dtype, spec.topk, spec.sm_scale, chunk=chunk)
    q_h, qi_h, w_h = dev.q.cpu().pin_memory(), dev.q_idx.cpu().pin_memory(), dev.w.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    for _ in range(2):
        out_h.fill_(float("nan"))
        lse_h.fill_(float("nan"))
        hp.run(q_h, qi_h, w_h, out_h, lse_h)
        torch.cuda.synchronize()
        assert smla.read_status(hp.ws)[0] == 0
        assert torch.equal(out_h.view(torch.int16), out.cpu().view(torch.int16))
        assert torch.equal(lse_h, lse.cpu())
    rows = stratified_rows(spec.prefix_len, spec.n_tokens, spec.topk, extra=(1023, 1024, 2047, 2048), n_random=6)
    _, _, rout, rlse, _ = sampled_oracle(dev, rows)
    compare_out(out_h.float().numpy()[rows], rout, lse_h.numpy()[rows], rlse, spec.kv_dtype)


def test_decode_host_resident_kv():
    """Decode with the latent cache (rows and FP8 scales) in page-locked host memory:
    the attention gathers the selected rows over the host link and returns exactly
    what the device-resident cache gives; sampled rows also match the oracle."""
    spec = wl.scaled(wl.SPECS["decode"], n_seqs=8, len_min=3000, len_max=20000, seed=77)
    prob = wl.make(spec, "cpu")
    dev = prob.to("cuda")
    lens = dev.seq_lens
    max_len = int(lens.max().item())
    args = (dev.page_table, lens, max_len, spec.q_per_seq, dev.q, dev.q_idx, dev.w, spec.topk, spec.sm_scale)
    ref_out, ref_lse, *_ = smla.sparse_mla_decode(dev.cache, *args)
    host_cache = wl.Cache(prob.cache.kv.pin_memory(), prob.cache.kv_scale.pin_memory(), dev.cache.k_idx,
                          dev.cache.k_idx_scale, spec.kv_dtype, spec.idx_dtype)
    for _ in range(2):
        out, lse, _, ws = smla.sparse_mla_decode(host_cache, *args)
        assert smla.read_status(ws)[0] == 0
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)
    rows = np.arange(0, spec.n_seqs * spec.q_per_seq, 3)
    ridx, _, rout, rlse, _, bad = oracle.Oracle(prob).rows(rows)
    assert not bad.any()
    compare_out(_host(out[torch.as_tensor(rows, device="cuda")].float()), rout,
                _host(lse[torch.as_tensor(rows, device="cuda")]), rlse, spec.kv_dtype)


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_fp8_ds_mla_rows(kind):
    """The 656-byte tile-scaled FP8 latent rows (512 e4m3 values with one fp32
    scale per 128, 64 bf16 rope values): a ragged prefill after a prefix and a
    decode batch in shuffled pools; index sets exact, outputs within the FP8
    tolerance of the oracle, which dequantises the same bytes."""
    if kind == "prefill":
        spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=1200, prefix_len=2500, shuffled=True,
                         kv_dtype=wl.FP8_DS_MLA)
        dev = wl.make(spec, "cuda")
        idx, out, lse = run_prefill(dev)
        rows = stratified_rows(spec.prefix_len, spec.n_tokens, spec.topk, n_random=10)
        ridx, _, rout, rlse, _ = sampled_oracle(dev, rows)
        r = torch.as_tensor(rows, device="cuda")
        compare_idx(_host(idx[r]), ridx)
        compare_out(_host(out[r].float()), rout, _host(lse[r]), rlse, spec.kv_dtype)
    else:
        spec = wl.scaled(wl.SPECS["decode"], n_seqs=10, len_min=1500, len_max=30000, seed=55,
                         kv_dtype=wl.FP8_DS_MLA)
        prob = wl.make(spec, "cpu")
        dev = prob.to("cuda")
        rows = spec.n_seqs * spec.q_per_seq
        max_len = int(dev.seq_lens.max())
        idx = torch.empty((rows, spec.topk), dtype=torch.int32, device="cuda")
        out, lse, _, ws = smla.sparse_mla_decode(dev.cache, dev.page_table, dev.seq_lens, max_len, spec.q_per_seq,
                                                 dev.q, dev.q_idx, dev.w, spec.topk, spec.sm_scale, out_idx=idx)
        assert smla.read_status(ws)[0] == 0
        ridx, _, rout, rlse, _, bad = oracle.Oracle(prob).rows(np.arange(rows))
        assert not bad.any()
        compare_idx(_host(idx), ridx)
        compare_out(_host(out.float()), rout, _host(lse), rlse, spec.kv_dtype)


@pytest.mark.parametrize("prefix", [500, 17000], ids=["dense", "streaming"])
@pytest.mark.parametrize("h_idx", [8, 16, 64])
def test_indexer_head_counts(h_idx, prefix):
    """Indexer heads other than the workloads' 4 and 32 (FP8 keys of 128 values):
    rows of at most 16,384 keys take the dense group mode (at 64 heads always its
    radix fallback: no staging room beside a 128-row query tile), longer rows the
    streaming candidate buffers; index sets exact against the oracle."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=300, prefix_len=prefix, shuffled=True, h_idx=h_idx,
                     topk=512)
    prob = wl.make(spec, "cpu")
    dev = prob.to("cuda")
    L = spec.prefix_len + spec.n_tokens
    seq_lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    gidx, gsc, ws = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, L, spec.n_tokens, dev.q_idx, dev.w,
                                      spec.topk, want_scores=True)
    assert smla.read_status(ws)[0] == 0
    rows = np.arange(0, spec.n_tokens, 7)
    ridx, rsc, *_ = oracle.Oracle(prob).rows(rows, attend=False)
    compare_idx(_host(gidx)[rows], ridx)
    g_i, g_s = _host(gidx)[rows], _host(gsc)[rows]
    for r in range(len(rows)):
        ok = g_i[r] >= 0
        full = oracle.Oracle(prob).scores(int(rows[r]))
        assert np.array_equal(g_s[r][ok], full[g_i[r][ok]])


def test_host_prefill_reports_errors_of_every_chunk():
    """Each chunk of the host-buffer prefill keeps its own status word: a query
    value outside the f16 range in a row of the FIRST chunk is still reported
    after run() (later chunks start with clean words of their own), and a run
    on clean inputs reports nothing."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=3000, prefix_len=500, shuffled=True)
    dev = wl.make(spec, "cuda")
    hp = smla.HostPrefill(dev.cache, dev.page_table, spec.prefix_len, spec.n_tokens, spec.n_heads, spec.h_idx,
                          spec.d_idx, spec.idx_dtype, spec.topk, spec.sm_scale, chunk=1024)
    q_bad = dev.q.cpu()
    q_bad[5, 3, 10] = 70000.0  # beyond f16's 65504
    q_bad = q_bad.pin_memory()
    qi_h, w_h = dev.q_idx.cpu().pin_memory(), dev.w.cpu().pin_memory()
    out_h = torch.empty((spec.n_tokens, spec.n_heads, 512), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((spec.n_tokens, spec.n_heads), dtype=torch.float32).pin_memory()
    hp.run(q_bad, qi_h, w_h, out_h, lse_h)
    rc, bits = hp.read_status()
    assert rc == 2 and bits & 4, (rc, bits)  # SMLA_ERR_UNSUPPORTED, the overflow bit
    hp.run(dev.q.cpu().pin_memory(), qi_h, w_h, out_h, lse_h)
    assert hp.read_status() == (0, 0)
