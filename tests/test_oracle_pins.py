"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against a hand-worked example, a closed form, an
invariant, a library routine on a special case, or brute force on tiny inputs,
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from indexer_top_sparse_score_gb300 import workloads as wl
from tests.cases import custom_prefill, fp8_codes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decoders ----
def test_e4m3_decode_matches_library_for_all_codes():
    """Every e4m3 code decodes like torch's float8_e4m3fn (a library routine)."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_to_float(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_bf16_decode_matches_library():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 1 << 16, (4096,), generator=g, dtype=torch.int32)
    bits = torch.cat([bits, torch.tensor([0, 0x8000, 0x3F80, 0xBF80, 0x7F7F, 0x0001])])
    ref = bits.to(torch.int16).view(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle.bf16_to_float(int(b) & 0xFFFF) for b in bits], dtype=np.float32)
    m = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[m], got[m])


# ---------------------------------------------------------------- indexer ----
def _golden_problem(idx_dtype="bf16"):
    g = json.load(open(os.path.join(GOLDEN, "indexer_worked_example.json")))
    prob = custom_prefill([g["q_idx"]], [g["w"]], g["k_idx"], idx_dtype=idx_dtype, topk=2)
    return g, prob


@pytest.mark.parametrize("idx_dtype", ["bf16", "fp8"])
def test_indexer_hand_worked_example(idx_dtype):
    g, prob = _golden_problem(idx_dtype)
    o = oracle.Oracle(prob)
    assert o.position(0) == 3
    assert o.scores(0).tolist() == g["scores"]
    for k in (2, 3):
        idx, _ = oracle.select_topk(np.array(g["scores"], np.float32), k)
        assert idx.tolist() == g[f"top{k}"]


def _random_int_problem(T=6, N=70, H_I=3, D_I=8, seed=0, **kw):
    gen = torch.Generator().manual_seed(seed)
    q_idx = torch.randint(-4, 5, (T, H_I, D_I), generator=gen).float()
    w = torch.randint(1, 5, (T, H_I), generator=gen).float()
    k_idx = torch.randint(-4, 5, (N, D_I), generator=gen).float()
    return q_idx, w, k_idx


def test_indexer_relu_identity_reduces_to_matmul():
    """relu(x) - relu(-x) = x: score(q) - score(-q) = sum_h w_h (k . q_h), a plain matmul."""
    q_idx, w, k_idx = _random_int_problem()
    a = oracle.Oracle(custom_prefill(q_idx, w, k_idx))
    b = oracle.Oracle(custom_prefill(-q_idx, w, k_idx))
    T = q_idx.shape[0]
    for t in range(T):
        n = a.position(t) + 1
        lin = (k_idx[:n].double() @ q_idx[t].double().T) @ w[t].double()
        diff = a.scores(t).astype(np.float64) - b.scores(t).astype(np.float64)
        assert np.array_equal(diff, lin.numpy())


def test_indexer_single_head_nonnegative_is_matmul():
    """H_I = 1, w = 1, non-negative operands: the score is k_I @ q_I (library matmul)."""
    gen = torch.Generator().manual_seed(5)
    q_idx = torch.randint(0, 5, (3, 1, 16), generator=gen).float()
    k_idx = torch.randint(0, 5, (40, 16), generator=gen).float()
    o = oracle.Oracle(custom_prefill(q_idx, torch.ones(3, 1), k_idx))
    for t in range(3):
        n = o.position(t) + 1
        assert np.array_equal(o.scores(t), (k_idx[:n] @ q_idx[t, 0]).numpy())


def test_indexer_linear_in_w_and_key_scale():
    q_idx, w, k_idx = _random_int_problem(seed=1)
    base = oracle.Oracle(custom_prefill(q_idx, w, k_idx))
    dbl = oracle.Oracle(custom_prefill(q_idx, 2 * w, k_idx))
    ks = torch.arange(k_idx.shape[0], dtype=torch.float32) % 3 + 1
    scl = oracle.Oracle(custom_prefill(q_idx, w, k_idx, k_idx_scale=ks))
    for t in range(q_idx.shape[0]):
        s = base.scores(t)
        assert np.array_equal(dbl.scores(t), 2 * s)
        assert np.array_equal(scl.scores(t), s * ks[:s.shape[0]].numpy())


def test_indexer_per_head_weights_not_transposed():
    """Only head 1 is non-zero: the score must use w[:,1], not w[:,0] or w[1,:]."""
    q = torch.zeros(2, 2, 4)
    q[:, 1, 2] = 1.0
    w = torch.tensor([[5.0, 2.0], [7.0, 3.0]])
    k = torch.zeros(5, 4)
    k[:, 2] = torch.tensor([1.0, 2.0, -1.0, 4.0, 3.0])
    o = oracle.Oracle(custom_prefill(q, w, k))
    assert o.scores(0).tolist() == [2.0, 4.0, 0.0, 8.0]
    assert o.scores(1).tolist() == [3.0, 6.0, 0.0, 12.0, 9.0]


def test_indexer_page_permutation_invariant():
    """Moving pages around the pool (and the table with them) changes nothing."""
    q_idx, w, k_idx = _random_int_problem(T=4, N=300, seed=2)
    a = oracle.Oracle(custom_prefill(q_idx, w, k_idx))
    perm = [3, 0, 4, 2, 1]
    b = oracle.Oracle(custom_prefill(q_idx, w, k_idx, page_perm=perm))
    for t in range(4):
        assert np.array_equal(a.scores(t), b.scores(t))


def test_indexer_causal_range():
    q_idx, w, k_idx = _random_int_problem(T=5, N=90, seed=4)
    o = oracle.Oracle(custom_prefill(q_idx, w, k_idx, prefix_len=60))
    for t in range(5):
        assert o.scores(t).shape[0] == 60 + t + 1


# ------------------------------------------------------------------ top-k ----
def _brute_topk(scores, k):
    """Independent O(n k) selector: repeatedly take the best remaining (lowest index on ties)."""
    taken = np.zeros(len(scores), bool)
    out = []
    for _ in range(min(k, len(scores))):
        best = -1
        for s in range(len(scores)):
            if taken[s]:
                continue
            if best < 0 or scores[s] > scores[best]:
                best = s
        taken[best] = True
        out.append(best)
    return sorted(out)


@pytest.mark.parametrize("seed", range(20))
def test_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 64))
    k = int(rng.choice([1, 3, 8, 17]))
    scores = rng.integers(0, 6, n).astype(np.float32)  # heavy ties
    idx, sc = oracle.select_topk(scores, k)
    keep = min(n, k)
    assert idx[:keep].tolist() == _brute_topk(scores, k)
    assert (idx[keep:] == -1).all()
    assert np.array_equal(sc[:keep], scores[idx[:keep]])


def test_topk_special_cases():
    n, k = 100, 8
    idx, _ = oracle.select_topk(np.full(n, 3.0, np.float32), k)
    assert idx.tolist() == list(range(k))                      # all equal -> lowest indices
    idx, _ = oracle.select_topk(np.arange(n, dtype=np.float32), k)
    assert idx.tolist() == list(range(n - k, n))               # increasing -> last k
    idx, _ = oracle.select_topk(-np.arange(n, dtype=np.float32), k)
    assert idx.tolist() == list(range(k))                      # decreasing -> first k
    idx, _ = oracle.select_topk(np.ones(5, np.float32), k)
    assert idx.tolist() == [0, 1, 2, 3, 4, -1, -1, -1]         # fewer keys than k


def test_topk_constant_keys_select_prefix():
    """k_I identical for every key: all scores tie, so the set is {0..k-1}."""
    gen = torch.Generator().manual_seed(9)
    q_idx = torch.randint(-4, 5, (3, 2, 8), generator=gen).float()
    w = torch.randint(1, 5, (3, 2), generator=gen).float()
    k_idx = torch.randint(-4, 5, (1, 8), generator=gen).float().repeat(50, 1)
    o = oracle.Oracle(custom_prefill(q_idx, w, k_idx, topk=16))
    idx, *_ = o.rows([0, 1, 2], attend=False)
    for r in range(3):
        assert idx[r].tolist() == list(range(16))


# -------------------------------------------------------------- attention ----
def _dense_causal_mla(q, kv, scale):
    """Textbook dense causal attention with a shared latent row (torch, fp64)."""
    q = q.double()
    K = kv.double()
    V = K[:, :wl.D_V]
    T, H, _ = q.shape
    N = K.shape[0]
    P = N - T
    logits = torch.einsum("thd,nd->thn", q, K) * scale
    pos = torch.arange(T)[:, None] + P
    mask = torch.arange(N)[None, :] > pos
    logits = logits.masked_fill(mask[:, None, :], float("-inf"))
    out = torch.einsum("thn,nd->thd", torch.softmax(logits, dim=-1), V)
    return out, torch.logsumexp(logits, dim=-1)


def test_attention_short_prompt_equals_dense_causal():
    """T <= k: every earlier key is selected, so sparse MLA is dense causal MLA."""
    T, N, H = 24, 40, 3
    q_idx, w, k_idx = _random_int_problem(T=T, N=N, seed=11)
    gen = torch.Generator().manual_seed(12)
    q = torch.randn(T, H, wl.D_QK, generator=gen).to(torch.bfloat16)
    kv = torch.randn(N, wl.D_QK, generator=gen).to(torch.bfloat16)
    prob = custom_prefill(q_idx, w, k_idx, n_heads=H, q=q, kv=kv, topk=64)
    scale = 0.07
    o = oracle.Oracle(prob, sm_scale=scale)
    idx, _, out, lse, _, bad = o.rows(range(T))
    assert not bad.any()
    ref_out, ref_lse = _dense_causal_mla(q.float(), kv.float(), scale)
    assert np.allclose(out, ref_out.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)
    for t in range(T):
        assert idx[t, :N - T + t + 1].tolist() == list(range(N - T + t + 1))


def _attn_problem(N=80, H=4, kv_dtype="bf16", seed=21, q=None, kv=None, kv_scale=None):
    q_idx, w, k_idx = _random_int_problem(T=1, N=N, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1)
    if q is None:
        q = torch.randn(1, H, wl.D_QK, generator=gen)
    if kv is None:
        kv = torch.randn(N, wl.D_QK, generator=gen)
    return custom_prefill(q_idx, w, k_idx, n_heads=H, q=q, kv=kv, kv_dtype=kv_dtype,
                          kv_scale=kv_scale, topk=N)


def test_attention_weights_sum_to_one():
    o = oracle.Oracle(_attn_problem())
    idx = np.arange(0, 80, 3, dtype=np.int32)
    out, lse, probs, bad = o.attend(0, idx, probs=True)
    assert bad == 0
    assert np.allclose(probs.sum(axis=1), 1.0, atol=1e-12)
    assert (probs >= 0).all()


def test_attention_zero_query_is_mean_of_values():
    """q = 0: all logits 0, uniform weights; out = mean V, lse = ln n."""
    N = 80
    gen = torch.Generator().manual_seed(2)
    kv = torch.randn(N, wl.D_QK, generator=gen).to(torch.bfloat16)
    prob = _attn_problem(N=N, q=torch.zeros(1, 4, wl.D_QK), kv=kv)
    o = oracle.Oracle(prob)
    idx = np.array([5, 9, 17, 40, 79, -1, 3], dtype=np.int32)
    out, lse, bad = o.attend(0, idx)
    sel = idx[idx >= 0]
    mean_v = kv.double()[sel, :wl.D_V].mean(dim=0).numpy()
    assert np.allclose(out, mean_v[None, :], rtol=0, atol=1e-13)
    assert np.allclose(lse, math.log(len(sel)), atol=1e-13)


def test_attention_single_key_returns_its_value():
    """One selected key: weight 1, out = V of that row, lse = its logit."""
    prob = _attn_problem()
    o = oracle.Oracle(prob, sm_scale=0.5)
    out, lse, _ = o.attend(0, np.array([13], np.int32))
    kv = prob.cache.kv.view(-1, wl.D_QK)[13].double()
    q = prob.q[0].double()
    assert np.allclose(out, kv[:wl.D_V].numpy()[None, :].repeat(4, 0), atol=0)
    assert np.allclose(lse, (0.5 * q @ kv).numpy(), rtol=1e-13)


def test_attention_equal_keys_give_uniform_weights():
    N = 64
    row = torch.randn(1, wl.D_QK, generator=torch.Generator().manual_seed(4))
    o = oracle.Oracle(_attn_problem(N=N, kv=row.repeat(N, 1)))
    _, _, probs, _ = o.attend(0, np.arange(0, N, 2, dtype=np.int32), probs=True)
    assert np.allclose(probs, 1.0 / 32, atol=1e-15)


def test_attention_lse_merge_of_partials_equals_whole():
    """Partial attentions over disjoint key sets merge exactly through their
    log-sum-exp ("Optimisations de GLM-5.3, partie 2", section DCP)."""
    o = oracle.Oracle(_attn_problem(N=120, seed=31), sm_scale=0.3)
    full = np.arange(0, 120, dtype=np.int32)
    a, b = full[::2].copy(), full[1::2].copy()
    of, lf, _ = o.attend(0, full)
    oa, la, _ = o.attend(0, a)
    ob, lb, _ = o.attend(0, b)
    lm = np.logaddexp(la, lb)
    om = oa * np.exp(la - lm)[:, None] + ob * np.exp(lb - lm)[:, None]
    assert np.allclose(lm, lf, rtol=1e-13)
    assert np.allclose(om, of, rtol=1e-10, atol=1e-12)


def test_attention_fp8_dequantises_with_per_token_scale():
    """FP8 rows: K = float(e4m3) * scale; equals the BF16 path fed the dequantised values."""
    N = 64
    gen = torch.Generator().manual_seed(6)
    codes = fp8_codes(torch.randint(-8, 9, (N, wl.D_QK), generator=gen).float() / 4)
    scale = torch.tensor([2.0 ** (i % 5 - 2) for i in range(N)])
    deq = codes.view(torch.float8_e4m3fn).float() * scale[:, None]  # exact in bf16 here
    gq = torch.randn(1, 4, wl.D_QK, generator=gen)
    p8 = _attn_problem(N=N, q=gq, kv=codes, kv_dtype="fp8", kv_scale=scale)
    pb = _attn_problem(N=N, q=gq, kv=deq)
    idx = np.arange(0, N, dtype=np.int32)
    o8, l8, _ = oracle.Oracle(p8).attend(0, idx)
    ob, lb, _ = oracle.Oracle(pb).attend(0, idx)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_attention_fp8_ds_mla_rows_dequantise_per_tile():
    """656-byte rows (512 e4m3 latent values, four fp32 scales each for one
    128-value tile, 64 bf16 rope values): K[d] = float(code[d]) * scale[d // 128]
    for d < 512 and K[512 + r] = bf16 rope value r. Equals the BF16 path fed the
    dequantised values (chosen exact in bf16); scales differ per row and per
    tile, so a wrong tile index, scale offset or rope offset changes the result."""
    N = 64
    gen = torch.Generator().manual_seed(16)
    lat = torch.randint(-8, 9, (N, wl.D_V), generator=gen).float() / 4
    codes = fp8_codes(lat)
    scales = torch.tensor([[2.0 ** ((r + 3 * t) % 5 - 2) for t in range(4)] for r in range(N)])
    rope = (torch.randint(-64, 65, (N, wl.D_QK - wl.D_V), generator=gen).float() / 16).to(torch.bfloat16)
    rows = torch.cat([codes, scales.contiguous().view(torch.uint8), rope.contiguous().view(torch.uint8)], dim=1)
    assert rows.shape == (N, wl.DS_MLA_ROW_BYTES)
    deq = torch.cat([codes.view(torch.float8_e4m3fn).float() * scales.repeat_interleave(128, dim=1),
                     rope.float()], dim=1)  # exact in bf16 here
    gq = torch.randn(1, 4, wl.D_QK, generator=gen)
    pd = _attn_problem(N=N, q=gq, kv=rows, kv_dtype=wl.FP8_DS_MLA)
    pb = _attn_problem(N=N, q=gq, kv=deq)
    idx = np.arange(0, N, dtype=np.int32)
    od, ld, _ = oracle.Oracle(pd).attend(0, idx)
    ob, lb, _ = oracle.Oracle(pb).attend(0, idx)
    assert np.array_equal(od, ob) and np.array_equal(ld, lb)


def test_attention_rejects_future_and_missing_keys():
    o = oracle.Oracle(_attn_problem(N=70))
    _, _, bad = o.attend(0, np.array([1, 2, 500], np.int32))
    assert bad == 1


# ------------------------------------------------------- generated workloads ----
def test_generated_workload_shapes_and_value_sets():
    spec = wl.scaled(wl.SPECS["prefix1m"], n_tokens=16, prefix_len=1000)
    p = wl.make(spec)
    assert p.cache.kv.shape == (-(-1016 // 64), 64, 576) and p.cache.kv.dtype == torch.uint8
    vals = p.q_idx.view(torch.float8_e4m3fn).float()
    assert set(vals.unique().tolist()) <= set(range(-4, 5))
    assert set(p.w.unique().tolist()) <= {1.0, 2.0, 3.0, 4.0}
    assert sorted(p.page_table.tolist()) == list(range(p.cache.num_pages))
    deq = p.cache.kv.view(torch.float8_e4m3fn).float().abs().amax(dim=-1)
    assert torch.allclose(deq, torch.full_like(deq, 448.0))
    d = wl.make(wl.scaled(wl.SPECS["decode"], n_seqs=4, len_min=100, len_max=300))
    lens = d.seq_lens.tolist()
    assert all(100 <= L <= 300 for L in lens)
    used = [int(x) for b, L in enumerate(lens) for x in d.page_table[b, :-(-L // 64)].tolist()]
    assert sorted(used) == list(range(d.cache.num_pages))


# --------------------------------------------------------------- decode rows ----
def _decode_problem(lens, pts, topk, H=3, H_I=2, D_I=16, seed=41, winner=False):
    """Two requests over one shared pool of 6 pages (bf16 latent rows, bf16
    indexer keys), q_per_seq = 2. Page table row b maps request b's logical
    pages to pool pages. With `winner`, the last token of every request gets a
    key that out-scores every other key for every query."""
    gen = torch.Generator().manual_seed(seed)
    pages, B, qps = 6, len(lens), 2
    rows = pages * wl.PAGE
    kv = torch.randn(rows, wl.D_QK, generator=gen).to(torch.bfloat16)
    k_idx = torch.randint(-1, 2, (rows, D_I), generator=gen).float()
    q_idx = torch.randint(-4, 5, (B * qps, H_I, D_I), generator=gen).float()
    if winner:
        q_idx = torch.ones(B * qps, H_I, D_I)
        for b, L in enumerate(lens):
            pr = pts[b][(L - 1) // wl.PAGE] * wl.PAGE + (L - 1) % wl.PAGE
            k_idx[pr] = 4.0
    w = torch.randint(1, 5, (B * qps, H_I), generator=gen).float()
    q = torch.randn(B * qps, H, wl.D_QK, generator=gen).to(torch.bfloat16)
    pt = torch.full((B, max(len(p) for p in pts)), -1, dtype=torch.int32)
    for b, p in enumerate(pts):
        pt[b, :len(p)] = torch.tensor(p, dtype=torch.int32)
    cache = wl.Cache(kv.view(pages, wl.PAGE, wl.D_QK).contiguous(), None,
                     k_idx.to(torch.bfloat16).view(pages, wl.PAGE, D_I).contiguous(), None, "bf16", "bf16")
    spec = wl.Spec("custom-decode", "decode", n_heads=H, h_idx=H_I, d_idx=D_I, idx_dtype="bf16",
                   kv_dtype="bf16", topk=topk, seed=0, n_seqs=B, q_per_seq=qps)
    return wl.Problem(spec, cache, pt, q.contiguous(), q_idx.to(torch.bfloat16).contiguous(), w.contiguous(),
                      torch.tensor(lens, dtype=torch.int32), 0, 0)


def test_decode_rows_sit_at_the_end_of_each_request():
    """Decode with two query tokens per request (the MTP shape): query j of a
    request of L keys sits at position L - 2 + j and sees keys 0..that position,
    so the first token does not see the second. With L <= k every visible key is
    selected and each row equals dense causal attention over the request's own
    rows (gathered through its page table), computed with torch in fp64."""
    lens, pts = [37, 100], [[2], [3, 1]]
    prob = _decode_problem(lens, pts, topk=128)
    scale = 0.05
    o = oracle.Oracle(prob, sm_scale=scale)
    idx, _, out, lse, _, bad = o.rows(range(4))
    assert not bad.any()
    kv = prob.cache.kv.view(-1, wl.D_QK).double()
    for b, L in enumerate(lens):
        logical = torch.tensor([pts[b][s // wl.PAGE] * wl.PAGE + s % wl.PAGE for s in range(L)])
        K = kv[logical]
        for j in range(2):
            r = 2 * b + j
            pos = L - 2 + j
            assert o.position(r) == pos
            assert idx[r, :pos + 1].tolist() == list(range(pos + 1)) and (idx[r, pos + 1:] == -1).all()
            logits = scale * (prob.q[r].double() @ K[:pos + 1].T)
            ref = torch.softmax(logits, dim=-1) @ K[:pos + 1, :wl.D_V]
            assert np.allclose(out[r], ref.numpy(), rtol=1e-12, atol=1e-12)
            assert np.allclose(lse[r], torch.logsumexp(logits, dim=-1).numpy(), rtol=1e-12)


def test_decode_first_mtp_token_cannot_select_the_second():
    """A key that beats every other is placed at the last token of each request:
    the request's last query row selects it, the row before cannot see it."""
    lens, pts = [120, 200], [[0, 2], [3, 1, 5, 4]]
    prob = _decode_problem(lens, pts, topk=8, winner=True)
    idx, *_ = oracle.Oracle(prob).rows(range(4), attend=False)
    for b, L in enumerate(lens):
        assert (L - 1) in idx[2 * b + 1].tolist()
        assert (L - 1) not in idx[2 * b].tolist()
        assert idx[2 * b].max() <= L - 2


def test_decode_rows_equal_prefill_rows_at_the_same_positions():
    """Each decode row equals the prefill row at the same absolute position of
    the same sequence (same cache, same page table), with longer requests than k."""
    lens, pts = [150, 230], [[1, 3, 0], [2, 0, 3, 1]]
    prob = _decode_problem(lens, pts, topk=16, seed=43)
    idx, sc, out, lse, _, _ = oracle.Oracle(prob).rows(range(4))
    for b, L in enumerate(lens):
        sub = wl.Problem(wl.scaled(prob.spec, kind="prefill", n_tokens=2, prefix_len=L - 2), prob.cache,
                         prob.page_table[b].clone(), prob.q[2 * b:2 * b + 2].contiguous(),
                         prob.q_idx[2 * b:2 * b + 2].contiguous(), prob.w[2 * b:2 * b + 2].contiguous(),
                         None, L - 2, 2)
        pi, ps, po, pl, _, _ = oracle.Oracle(sub).rows(range(2))
        assert np.array_equal(pi, idx[2 * b:2 * b + 2]) and np.array_equal(ps, sc[2 * b:2 * b + 2])
        assert np.array_equal(po, out[2 * b:2 * b + 2]) and np.array_equal(pl, lse[2 * b:2 * b + 2])
