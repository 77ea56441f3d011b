"""CUDA path vs the CPU oracle on inputs the workloads leave at their defaults
(needs a GB300): a per-key indexer scale, another softmax scale, BF16
caller-given index lists, and output buffers guarded by canaries so that a
write past the last row (or a row left unwritten) is seen."""
import numpy as np
import pytest
import torch

import indexer_top_sparse_score_gb300 as smla
import oracle
from indexer_top_sparse_score_gb300 import workloads as wl
from tests.gpu_common import (Guarded, compare_idx, compare_out, indexer_ws, run_prefill, sampled_oracle,
                              stratified_rows)

pytestmark = pytest.mark.gpu

BF16_CANARY = 0x7FC1        # a bf16 NaN pattern no kernel writes
F32_CANARY = 0x7FC00001     # an fp32 NaN pattern
IDX_CANARY = 0x5A5A5A5A     # not a key index, not -1


@pytest.fixture(scope="module", autouse=True)
def _built():
    smla.build()
    oracle.build()
    smla.lib()


def _host(t):
    return t.cpu().numpy()


def _with_key_scale(prob, seed=13):
    """The same problem with a positive per-key indexer scale in [0.5, 2) (the
    4-byte scale of the 132-byte indexer key row); any positive fp32 value keeps
    the integer-valued score sums exact, and both sides multiply once."""
    g = torch.Generator().manual_seed(seed)
    c = prob.cache
    ks = (0.5 + 1.5 * torch.rand(c.k_idx.shape[:2], generator=g)).to(torch.float32).contiguous()
    cache = wl.Cache(c.kv, c.kv_scale, c.k_idx, ks, c.kv_dtype, c.idx_dtype)
    return wl.Problem(prob.spec, cache, prob.page_table, prob.q, prob.q_idx, prob.w, prob.seq_lens,
                      prob.prefix_len, prob.n_tokens)


@pytest.mark.parametrize("mode", ["dense", "scores", "streaming", "decode"])
def test_indexer_key_scale(mode):
    """A non-NULL per-key indexer scale: index sets and returned scores exact in
    the dense (rows <= 16,384 keys), score-array and streaming (a workspace too
    small for the score array) group modes and the decode (split) mode;
    attention outputs within tolerance."""
    if mode == "decode":
        spec = wl.scaled(wl.SPECS["decode"], n_seqs=6, len_min=3000, len_max=40000, seed=61)
    else:
        spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=600, prefix_len=4000 if mode == "dense" else 20000,
                         shuffled=True, kv_dtype="fp8")
    prob = _with_key_scale(wl.make(spec, "cpu"))
    dev = prob.to("cuda")
    o = oracle.Oracle(prob)
    if mode == "decode":
        rows = np.arange(spec.n_seqs * spec.q_per_seq)
        max_len = int(dev.seq_lens.max())
        gidx, gsc, ws = smla.indexer_topk(dev.cache, dev.page_table, dev.seq_lens, max_len, spec.q_per_seq,
                                          dev.q_idx, dev.w, spec.topk, want_scores=True)
        assert smla.read_status(ws)[0] == 0
        out, lse, _, ws = smla.sparse_mla_decode(dev.cache, dev.page_table, dev.seq_lens, max_len, spec.q_per_seq,
                                                 dev.q, dev.q_idx, dev.w, spec.topk, spec.sm_scale)
        assert smla.read_status(ws)[0] == 0
    else:
        rows = np.arange(0, spec.n_tokens, 11)
        L = spec.prefix_len + spec.n_tokens
        seq_lens = torch.tensor([L], dtype=torch.int32, device="cuda")
        ws = indexer_ws(spec.n_tokens, "cand") if mode == "streaming" else None
        gidx, gsc, ws = smla.indexer_topk(dev.cache, dev.page_table, seq_lens, L, spec.n_tokens, dev.q_idx, dev.w,
                                          spec.topk, want_scores=True, ws=ws)
        assert smla.read_status(ws)[0] == 0
        _, out, lse = run_prefill(dev, want_idx=False)
    ridx, rsc, rout, rlse, _, bad = o.rows(rows)
    assert not bad.any()
    gi, gs = _host(gidx)[rows], _host(gsc)[rows]
    compare_idx(gi, ridx)
    for r in range(len(rows)):
        ok = gi[r] >= 0
        full = o.scores(int(rows[r]))
        assert np.array_equal(gs[r][ok], full[gi[r][ok]])
    compare_out(_host(out.float())[rows], rout, _host(lse)[rows], rlse, spec.kv_dtype)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_second_softmax_scale(kv_dtype):
    """sm_scale is an argument: a prefill with 0.11 (not 1/sqrt(576)) matches the
    oracle run with the same scale; a wrong scale would move every output."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=900, prefix_len=2600, shuffled=True, kv_dtype=kv_dtype)
    dev = wl.make(spec, "cuda")
    idx, out, lse = run_prefill(dev, sm_scale=0.11)
    rows = stratified_rows(spec.prefix_len, spec.n_tokens, spec.topk, n_random=12)
    ridx, _, rout, rlse, _ = sampled_oracle(dev, rows, sm_scale=0.11)
    r = torch.as_tensor(rows, device="cuda")
    compare_idx(_host(idx[r]), ridx)
    compare_out(_host(out[r].float()), rout, _host(lse[r]), rlse, kv_dtype)


@pytest.mark.parametrize("shadow", [True, False], ids=["f16-shadow", "in-kernel-widening"])
def test_sparse_mla_given_indices_bf16(shadow):
    """Caller-given index lists with -1 holes over a BF16 cache, with the
    workspace large enough for the f16 copy of the rows and with only the
    256-byte status word (rows widened in the attention kernel)."""
    spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=300, prefix_len=5000, kv_dtype="bf16", topk=512,
                     shuffled=True)
    dev = wl.make(spec, "cuda")
    g = torch.Generator().manual_seed(15)
    T, k = spec.n_tokens, spec.topk
    idx = torch.empty((T, k), dtype=torch.int32)
    for t in range(T):
        perm = torch.randperm(spec.prefix_len + t + 1, generator=g)[:k].to(torch.int32)
        perm[torch.rand(k, generator=g) < 0.1] = -1
        idx[t] = perm
    ws = None if shadow else smla.workspace(256)
    out, lse, ws = smla.sparse_mla_fwd(dev.cache, dev.page_table, dev.q, idx.cuda(), spec.sm_scale,
                                       prefix_len=spec.prefix_len, ws=ws)
    assert smla.read_status(ws)[0] == 0
    o = oracle.Oracle(dev.to("cpu"))
    rows = np.arange(0, T, 7)
    rout, rlse = o.attend_rows(rows, idx.numpy()[rows])
    compare_out(_host(out.float())[rows], rout, _host(lse)[rows], rlse, "bf16")


def _guarded_outputs(rows, H, k):
    out = Guarded((rows, H, 512), torch.bfloat16, BF16_CANARY)
    lse = Guarded((rows, H), torch.float32, F32_CANARY)
    idx = Guarded((rows, k), torch.int32, IDX_CANARY)
    return out, lse, idx


def _check_guarded(out, lse, idx):
    for b in (out, lse, idx):
        b.check()
    # every element of the views was written
    assert not bool((out.view.view(torch.int16) == BF16_CANARY).any()), "output left unwritten"
    assert not bool((lse.view.view(torch.int32) == F32_CANARY).any()), "lse left unwritten"
    assert not bool((idx.view == IDX_CANARY).any()), "index entry left unwritten"


@pytest.mark.parametrize("case", ["dense", "scores", "streaming", "tiny"])
def test_prefill_writes_only_its_outputs(case):
    """Prefill through the product entry into outputs framed by canaries: nothing
    is written before or after out, lse and out_idx, every element inside them is
    written, and sampled rows (including the last) match the oracle. Rows of
    more than 16,384 keys take the score array with the full workspace, and the
    streaming candidate buffers with a workspace that holds those buffers but no
    score-array block."""
    if case == "tiny":
        spec = wl.scaled(wl.SPECS["tiny"], n_tokens=333, prefix_len=100, shuffled=True)
    else:
        spec = wl.scaled(wl.SPECS["prefill16k"], n_tokens=1001, prefix_len=3000 if case == "dense" else 17000,
                         shuffled=True, kv_dtype="fp8")
    dev = wl.make(spec, "cuda")
    T, H, k = spec.n_tokens, spec.n_heads, spec.topk
    ws = None
    if case == "streaming":
        # status | index list | f16 copy of the FP8 rows and their scales | candidate buffers
        r256 = lambda b: (b + 255) // 256 * 256
        n_keys = spec.prefix_len + T
        ws = smla.workspace(256 + r256(T * k * 4) + r256(n_keys * 1152) + r256(n_keys * 4)
                            + T * 4096 * 8 + r256(T * 4))
    out, lse, idx = _guarded_outputs(T, H, k)
    _, _, _, ws = smla.sparse_mla_prefill(dev.cache, dev.page_table, spec.prefix_len, dev.q, dev.q_idx, dev.w, k,
                                          spec.sm_scale, out=out.view, lse=lse.view, out_idx=idx.view, ws=ws)
    assert smla.read_status(ws)[0] == 0
    _check_guarded(out, lse, idx)
    rows = np.array(sorted({0, T // 2, T - 2, T - 1}), dtype=np.int64)
    ridx, _, rout, rlse, _ = sampled_oracle(dev, rows)
    r = torch.as_tensor(rows, device="cuda")
    compare_idx(_host(idx.view[r]), ridx)
    compare_out(_host(out.view[r].float()), rout, _host(lse.view[r]), rlse, spec.kv_dtype)


@pytest.mark.parametrize("q_per_seq", [1, 2])
def test_decode_writes_only_its_outputs(q_per_seq):
    """Decode (with rows split into parts merged by log-sum-exp) into outputs
    framed by canaries: nothing outside them is written, everything inside is,
    and every row matches the oracle."""
    spec = wl.scaled(wl.SPECS["decode"], n_seqs=7, q_per_seq=q_per_seq, len_min=1000, len_max=30000, seed=83)
    prob = wl.make(spec, "cpu")
    dev = prob.to("cuda")
    rows = spec.n_seqs * q_per_seq
    H, k = spec.n_heads, spec.topk
    out, lse, idx = _guarded_outputs(rows, H, k)
    max_len = int(dev.seq_lens.max())
    _, _, _, ws = smla.sparse_mla_decode(dev.cache, dev.page_table, dev.seq_lens, max_len, q_per_seq, dev.q,
                                         dev.q_idx, dev.w, k, spec.sm_scale, out=out.view, lse=lse.view,
                                         out_idx=idx.view)
    assert smla.read_status(ws)[0] == 0
    _check_guarded(out, lse, idx)
    ridx, _, rout, rlse, _, bad = oracle.Oracle(prob).rows(np.arange(rows))
    assert not bad.any()
    compare_idx(_host(idx.view), ridx)
    compare_out(_host(out.view.float()), rout, _host(lse.view), rlse, spec.kv_dtype)
