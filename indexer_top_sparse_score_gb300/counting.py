"""Algorithmic work and traffic of the layer step (roofline numerators).

Counting rules, from "Optimisations de GLM-5.3, partie 2" (spke.com):
  * footnote 1: sparse MLA performs 2,176 FLOPs per (query, selected row,
    head): QK over 576 dims (2*576) plus PV over 512 dims (2*512); each head
    moves its BF16 query (576 values) and output (512 values), 2,176 bytes;
    each selected row is read once for all heads;
  * the indexer performs 2*H_I*D_I FLOPs per (query, key) pair it scores
    (one dot product of length D_I per indexer head), over keys 0..pos.
Only work the method must do is counted: no dense T x T attention.
"""
from __future__ import annotations

D_QK, D_V = 576, 512
MLA_FLOP_PER_ROW_HEAD = 2 * D_QK + 2 * D_V          # 2176
BF16_Q_OUT_BYTES_PER_HEAD = 2 * D_QK + 2 * D_V      # 2176


def mla_intensity(heads: int, rows: int = 2048, row_bytes: int = 660) -> float:
    """FLOPs per byte of one query's sparse MLA (footnote 1's arithmetic)."""
    flops = heads * rows * MLA_FLOP_PER_ROW_HEAD
    bytes_ = rows * row_bytes + heads * BF16_Q_OUT_BYTES_PER_HEAD
    return flops / bytes_


def kv_row_bytes(kv_dtype: str) -> int:
    """Bytes of one latent KV row as the library stores it (FP8 adds its fp32 scale;
    the tile-scaled FP8 row of the GLM page's footnote 1 is 656 bytes)."""
    if kv_dtype == "fp8_ds_mla":
        return 656
    return D_QK * 2 if kv_dtype == "bf16" else D_QK + 4


def n_selected(pos: int, topk: int) -> int:
    """Rows a query at absolute position `pos` attends to (keys 0..pos, at most k)."""
    return min(topk, pos + 1)


def prefill_counts(prefix_len: int, n_tokens: int, n_heads: int, h_idx: int, d_idx: int,
                   topk: int, kv_dtype: str, idx_bytes: int) -> dict:
    """FLOPs and algorithmic HBM/L2 bytes of one prefill call."""
    P, T = prefix_len, n_tokens
    pairs = T * P + T * (T + 1) // 2                       # sum_t (P + t + 1)
    sel = sum(n_selected(P + t, topk) for t in range(T)) if T < 4096 else \
        _sum_selected(P, T, topk)
    rb = kv_row_bytes(kv_dtype)
    per_query = T * n_heads * (2 * D_QK + 2 * D_V + 4) + T * topk * 4  # q, out, lse, index list
    return dict(
        idx_flops=2 * h_idx * d_idx * pairs,
        mla_flops=MLA_FLOP_PER_ROW_HEAD * n_heads * sel,
        pairs=pairs, selected_rows=sel,
        # sparse-MLA kernel, HBM: every cache row at most once (P + T rows), q, out,
        # lse and the index list
        mla_bytes=(P + T) * rb + per_query,
        # the same with every selected-row gather counted (L2-level traffic: the
        # rows a query selects are mostly shared with its neighbours)
        mla_gather_bytes=sel * rb + per_query,
        # indexer kernel: every key row once, q_I, w, and the index list it writes
        idx_bytes=(P + T) * d_idx * idx_bytes + T * h_idx * (d_idx * idx_bytes + 4) + T * topk * 4,
    )


def _sum_selected(P: int, T: int, k: int) -> int:
    """Closed form of sum_{t<T} min(k, P+t+1)."""
    # positions p = P+t+1 run over P+1 .. P+T; min(k, p)
    lo, hi = P + 1, P + T
    if hi <= k:
        return (lo + hi) * T // 2
    if lo > k:
        return k * T
    below = (lo + k) * (k - lo + 1) // 2
    return below + k * (hi - k)


def decode_counts(seq_lens, q_per_seq: int, n_heads: int, h_idx: int, d_idx: int, topk: int,
                  kv_dtype: str, idx_bytes: int) -> dict:
    pairs = 0
    sel = 0
    keys = 0
    for L in seq_lens:
        keys += L
        for j in range(q_per_seq):
            pos = L - q_per_seq + j
            pairs += pos + 1
            sel += n_selected(pos, topk)
    rows = len(seq_lens) * q_per_seq
    rb = kv_row_bytes(kv_dtype)
    return dict(
        idx_flops=2 * h_idx * d_idx * pairs,
        mla_flops=MLA_FLOP_PER_ROW_HEAD * n_heads * sel,
        pairs=pairs, selected_rows=sel,
        mla_bytes=sel * rb + rows * n_heads * (2 * D_QK + 2 * D_V + 4) + rows * topk * 4,
        idx_bytes=keys * d_idx * idx_bytes + rows * h_idx * (d_idx * idx_bytes + 4) + rows * topk * 4,
    )


def kv_bytes_per_token(layers: int, row_bytes: int) -> int:
    return layers * row_bytes
