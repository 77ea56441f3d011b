"""The roofline's counting rules reproduce the arithmetic printed on the pages."""
from indexer_top_sparse_score_gb300 import counting as c


def test_footnote1_intensities():
    # "Optimisations de GLM-5.3, partie 2", footnote 1: ~26 FLOP/B at 8 heads, ~191 at 64.
    assert round(c.mla_intensity(8), 2) == 26.04
    assert round(c.mla_intensity(64), 2) == 191.30
    assert round(8 * 2048 * c.MLA_FLOP_PER_ROW_HEAD / 1e6, 1) == 35.7
    assert round(64 * 2048 * c.MLA_FLOP_PER_ROW_HEAD / 1e6) == 285


def test_kv_bytes_per_token():
    # "Lower latency and higher throughput with multi-node DeepSeek deployment":
    # 61 layers of a 576-value BF16 latent row = 70,272 bytes per token.
    assert c.kv_bytes_per_token(61, c.kv_row_bytes("bf16")) == 70272
    # footnote 3 of the GLM page: 78 x 656 + 21 x 132 + 788 = 54,728 B; x 2^20 tokens = 53.4 GiB.
    per_tok = c.kv_bytes_per_token(78, 656) + c.kv_bytes_per_token(21, 132) + 788
    assert per_tok == 54728
    assert round(per_tok * 1048576 / 2 ** 30, 1) == 53.4


def test_selected_row_count_closed_form():
    for P, T, k in [(0, 100, 16), (0, 5000, 2048), (3000, 5000, 2048), (10, 3, 2048), (0, 1, 1)]:
        assert c._sum_selected(P, T, k) == sum(min(k, P + t + 1) for t in range(T))


def test_prefill_counts_small():
    r = c.prefill_counts(0, 4, n_heads=2, h_idx=1, d_idx=8, topk=2, kv_dtype="bf16", idx_bytes=2)
    assert r["pairs"] == 1 + 2 + 3 + 4
    assert r["selected_rows"] == 1 + 2 + 2 + 2
    assert r["mla_flops"] == 2176 * 2 * 7
    assert r["idx_flops"] == 16 * 10
