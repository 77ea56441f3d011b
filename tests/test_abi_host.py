"""The C ABI without a GPU: every symbol declared in include/smla.h is exported,
and argument checks return the documented status codes before anything is
enqueued (the fake device pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

import indexer_top_sparse_score_gb300 as smla

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "smla.h")
OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
FAKE = 0x10000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def L():
    smla.build()
    return smla.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\**\s*(smla_\w+)\s*\(", text, re.M)))


def test_header_symbols_exported(L):
    names = declared_functions()
    assert len(names) == 13
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(smla._SIGS), "binding signatures and header disagree"


def test_status_strings(L):
    for code in range(7):
        assert L.smla_status_string(code).decode().startswith("SMLA_")
    assert L.smla_status_string(99) == b"SMLA_ERR_UNKNOWN"


def _cache(**kw):
    c = dict(kv=FAKE, kv_scale=FAKE, k_idx=FAKE, k_idx_scale=None, num_pages=300, page_size=64,
             kv_dtype=smla.SMLA_FP8_E4M3, idx_dtype=smla.SMLA_FP8_E4M3, d_idx=128)
    c.update(kw)
    return smla.PagedCache(**c)


def _prefill(L, cache, *, prefix=1000, T=4096, H=64, h_idx=32, topk=2048, ws_bytes=None, q=FAKE, out=FAKE,
             pt=FAKE, sm=0.04):
    need = L.smla_sparse_mla_prefill_workspace_size(prefix, T, H, h_idx, topk, cache.kv_dtype)
    ws = need if ws_bytes is None else ws_bytes
    return L.smla_sparse_mla_prefill(ctypes.byref(cache), pt, prefix, T, q, H, FAKE, FAKE, h_idx, topk, sm,
                                     out, FAKE, None, FAKE, ws, None)


def test_prefill_argument_checks(L):
    assert _prefill(L, _cache(), q=None) == INVALID
    assert _prefill(L, _cache(), out=FAKE + 8) == INVALID          # misaligned
    assert _prefill(L, _cache(), pt=None) == INVALID
    assert _prefill(L, _cache(), T=0) == INVALID
    assert _prefill(L, _cache(), prefix=-1) == INVALID
    assert _prefill(L, _cache(page_size=32)) == UNSUPPORTED
    assert _prefill(L, _cache(num_pages=(1 << 25) + 1)) == UNSUPPORTED   # pool rows are int32
    assert _prefill(L, _cache(d_idx=64)) == UNSUPPORTED             # e4m3 x 64 = 64-byte rows
    assert _prefill(L, _cache(kv_scale=None)) == INVALID            # FP8 needs scales
    assert _prefill(L, _cache(kv_dtype=7)) == INVALID
    # the 656-byte tile-scaled FP8 rows carry their scales: no scale array needed,
    # and the format is for the latent cache only (not the indexer keys)
    assert _prefill(L, _cache(kv_dtype=smla.SMLA_FP8_DS_MLA, kv_scale=None), H=32) == UNSUPPORTED  # cache ok
    assert _prefill(L, _cache(kv_dtype=smla.SMLA_FP8_DS_MLA, idx_dtype=smla.SMLA_FP8_DS_MLA)) == INVALID
    assert _prefill(L, _cache(), H=32) == UNSUPPORTED
    assert _prefill(L, _cache(), h_idx=12) == UNSUPPORTED
    assert _prefill(L, _cache(), topk=4096) == UNSUPPORTED
    assert _prefill(L, _cache(), topk=0) == INVALID
    assert _prefill(L, _cache(), sm=float("nan")) == INVALID
    assert _prefill(L, _cache(), ws_bytes=100) == WORKSPACE


def test_decode_and_indexer_argument_checks(L):
    c = _cache()
    need = L.smla_sparse_mla_decode_workspace_size(64, 131072, 2, 64, 32, 2048)
    call = lambda **kw: L.smla_sparse_mla_decode(
        ctypes.byref(c), kw.get("pt", FAKE), kw.get("max_pages", 2048), 64, kw.get("lens", FAKE),
        kw.get("max_len", 131072), kw.get("qps", 2), FAKE, 64, FAKE, FAKE, 32, 2048, 0.04, FAKE, FAKE, None,
        FAKE, kw.get("ws", need), None)
    assert call(lens=None) == INVALID
    assert call(max_pages=10) == INVALID        # table shorter than max_seq_len
    assert call(qps=9) == UNSUPPORTED
    assert call(ws=need - 1) == WORKSPACE
    n = L.smla_indexer_topk(ctypes.byref(c), FAKE, 2048, 64, FAKE, 131072, 2, FAKE, FAKE, 32, 2048, None,
                            None, FAKE, 1 << 30, None)
    assert n == INVALID                          # out_idx required


def test_workspace_sizes(L):
    # prefill keeps the index list (status word + T x topk int32); rows of at most
    # 16384 keys are selected from full score rows in shared memory, so nothing
    # more for the indexer. A BF16 cache adds an f16 copy of the sequence's rows
    # (576 values x 2 bytes per key), a per-token FP8 cache the same copy and its
    # scales in the same order (4 bytes per key, rounded to 256), the 656-byte
    # tile-scaled FP8 rows nothing
    def r256(b):
        return (b + 255) // 256 * 256
    assert L.smla_sparse_mla_prefill_workspace_size(0, 16384, 64, 32, 2048, 0) == \
        256 + 16384 * 2048 * 4 + 16384 * 576 * 2
    assert L.smla_sparse_mla_prefill_workspace_size(0, 16384, 64, 32, 2048, 1) == \
        256 + 16384 * 2048 * 4 + 16384 * 576 * 2 + r256(16384 * 4)
    assert L.smla_sparse_mla_prefill_workspace_size(0, 16384, 64, 32, 2048, 2) == 256 + 16384 * 2048 * 4
    # longer rows at 32 indexer heads: a score array, 4 bytes per key up to
    # max_seq_len rounded up to 32, for a block of rows of every sequence: all
    # rows while the array stays within 16 GiB
    T, P = 8192, 20000
    stride = (P + T + 31) // 32 * 32
    scores = T * stride * 4
    assert L.smla_sparse_mla_prefill_workspace_size(P, T, 64, 32, 2048, 2) == 256 + T * 2048 * 4 + scores
    assert L.smla_sparse_mla_prefill_workspace_size(P, T, 64, 32, 2048, 1) == \
        256 + T * 2048 * 4 + r256((P + T) * 1152) + r256((P + T) * 4) + scores
    # one call over 131072 new tokens: blocks of 32768 rows x 131072 keys (16 GiB)
    assert L.smla_sparse_mla_prefill_workspace_size(0, 131072, 64, 32, 2048, 2) == \
        256 + 131072 * 2048 * 4 + 32768 * 131072 * 4
    # 8192 tokens after a 1M prefix: 4260 rows of 1,056,768 keys fit in 16 GiB
    stride1m = (1048576 + 8192 + 31) // 32 * 32
    assert L.smla_sparse_mla_prefill_workspace_size(1048576, 8192, 64, 32, 2048, 2) == \
        256 + 8192 * 2048 * 4 + ((16 << 30) // (stride1m * 4) // 4 * 4) * stride1m * 4
    # the indexer alone: status word + the score array (two sequences: the same
    # rows of both in one block)
    assert L.smla_indexer_topk_workspace_size(1, 16384, 16384, 32, 2048) == 256
    assert L.smla_indexer_topk_workspace_size(1, P + T, T, 32, 2048) == 256 + scores
    assert L.smla_indexer_topk_workspace_size(2, 30000, 4096, 32, 2048) == 256 + 2 * 4096 * 30016 * 4
    # other head counts: candidate buffers of rows whose final selection is
    # deferred: 4 query rows per work item (at 16 heads) share 16384 entries, so
    # 4096 (key, index) pairs per row, plus one count per row
    cand = T * 4096 * 8 + T * 4
    assert L.smla_indexer_topk_workspace_size(1, P + T, T, 16, 2048) == 256 + cand
    stride3 = (300000 + T + 31) // 32 * 32
    assert L.smla_indexer_topk_workspace_size(1, 300000 + T, T, 32, 2048) == 256 + T * stride3 * 4
    # decode: a score per (row, key) up to max_seq_len, the index list, then
    # room for the fp32 partial outputs (and lse) of rows split into up to 4 parts
    rows, k = 128, 2048
    dec = L.smla_sparse_mla_decode_workspace_size(64, 131072, 2, 64, 32, 2048)
    assert dec == 256 + rows * 131072 * 4 + rows * k * 4 + rows * 4 * 64 * 512 * 4 + rows * 4 * 64 * 4
    assert L.smla_sparse_mla_fwd_workspace_size(0, 100, 64, 2048, 0) == 256
    assert L.smla_sparse_mla_fwd_workspace_size(1000, 100, 64, 2048, 2) == 256
    assert L.smla_sparse_mla_fwd_workspace_size(1000, 100, 64, 2048, 1) == 256 + 1000 * 1152 + r256(4000)
    assert L.smla_sparse_mla_fwd_workspace_size(1000, 100, 64, 2048, 0) == 256 + 1000 * 1152
