"""Seeded synthetic inputs for the indexer -> top-k -> sparse MLA layer step.

This module only draws random numbers and lays them out in the memory format
the library consumes (paged latent KV pool, paged indexer-key pool, page
tables, queries). It holds none of the method's arithmetic: no scores, no
selection, no attention. Both the CUDA path and the CPU oracle are fed from the
tensors built here.

Shapes follow the workloads described in "Optimisations de GLM-5.3, partie 2"
(spke.com): 64 query heads sharing one 576-value latent row per token (512
latent + 64 rope), an indexer that scores every earlier token, a causal
top-2048, FP8 KV with a per-token scale, 64-token pages, and contexts from 64K
up to 1M tokens. The pages' own benchmark traces are not available; these
synthetic tensors stand in for them.

Value recipe (one seed per workload):
  * latent q and BF16 KV: N(0,1) drawn in fp32, rounded to bf16 (RNE);
  * FP8 KV: N(0,1) per token, scale = amax/448, e4m3 with RNE (torch cast);
  * fp8_ds_mla KV (the 656-byte row size of the pages' footnote 1): N(0,1)
    per token; the 512 latent values quantised to e4m3 in four tiles of 128,
    each with scale = tile amax/448; the 64 rope values rounded to bf16;
  * indexer q_I / k_I: integers uniform in [-4, 4] (exact in e4m3 and bf16);
  * head weights w: integers uniform in [1, 4] stored as fp32;
  * decode context lengths uniform in [8192, 131072]; pages of every
    request drawn from one seeded random permutation of a global pool.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

D_QK = 576  # latent (512) + rope (64) values per KV row
D_V = 512   # the first 512 values of a row serve as V
PAGE = 64   # tokens per page

BF16 = "bf16"
FP8 = "fp8"
FP8_DS_MLA = "fp8_ds_mla"  # 656-byte rows: 512 e4m3 latent | 4 fp32 tile scales | 64 bf16 rope
DS_MLA_ROW_BYTES = 656


@dataclasses.dataclass
class Spec:
    name: str
    kind: str              # "prefill" or "decode"
    n_heads: int           # query heads of the sparse MLA
    h_idx: int             # indexer heads
    d_idx: int             # indexer head dim
    idx_dtype: str         # dtype of q_I / k_I
    kv_dtype: str          # dtype of the latent KV cache
    topk: int
    seed: int
    # prefill
    n_tokens: int = 0      # new query tokens
    prefix_len: int = 0    # cached tokens before them
    chunk: int = 0         # >0: process the new tokens in chunks of this size
    shuffled: bool = False  # pages drawn from a shuffled pool
    # decode
    n_seqs: int = 0
    q_per_seq: int = 0
    len_min: int = 0
    len_max: int = 0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(D_QK)


# The five workloads. Sizes are the configurations quoted for this layer step.
SPECS = {
    "tiny": Spec("tiny", "prefill", n_heads=16, h_idx=4, d_idx=64, idx_dtype=BF16,
                 kv_dtype=BF16, topk=256, seed=1001, n_tokens=1024),
    "prefill16k": Spec("prefill16k", "prefill", n_heads=64, h_idx=32, d_idx=128,
                       idx_dtype=FP8, kv_dtype=BF16, topk=2048, seed=1002,
                       n_tokens=16384),
    "prefill128k": Spec("prefill128k", "prefill", n_heads=64, h_idx=32, d_idx=128,
                        idx_dtype=FP8, kv_dtype=FP8, topk=2048, seed=1003,
                        n_tokens=131072, chunk=8192),
    "decode": Spec("decode", "decode", n_heads=64, h_idx=32, d_idx=128,
                   idx_dtype=FP8, kv_dtype=FP8, topk=2048, seed=1004,
                   n_seqs=64, q_per_seq=2, len_min=8192, len_max=131072,
                   shuffled=True),
    "prefix1m": Spec("prefix1m", "prefill", n_heads=64, h_idx=32, d_idx=128,
                     idx_dtype=FP8, kv_dtype=FP8, topk=2048, seed=1005,
                     n_tokens=8192, prefix_len=1 << 20, shuffled=True),
}


def scaled(spec: Spec, **overrides) -> Spec:
    """A copy of `spec` with some fields replaced (smaller test cases)."""
    return dataclasses.replace(spec, **overrides)


@dataclasses.dataclass
class Cache:
    """Paged latent KV pool + paged indexer-key pool (one layer)."""
    kv: torch.Tensor                  # [pages, 64, 576] bf16 or uint8 (e4m3 bits); fp8_ds_mla [pages, 64, 656] uint8
    kv_scale: Optional[torch.Tensor]  # [pages, 64] fp32 (FP8 only)
    k_idx: torch.Tensor               # [pages, 64, d_idx] bf16, or uint8 (e4m3 bits)
    k_idx_scale: Optional[torch.Tensor]
    kv_dtype: str
    idx_dtype: str

    @property
    def num_pages(self) -> int:
        return self.kv.shape[0]

    def to(self, device) -> "Cache":
        f = lambda t: None if t is None else t.to(device)
        return Cache(f(self.kv), f(self.kv_scale), f(self.k_idx), f(self.k_idx_scale),
                     self.kv_dtype, self.idx_dtype)


@dataclasses.dataclass
class Problem:
    spec: Spec
    cache: Cache
    page_table: torch.Tensor   # prefill: [pages_needed] int32; decode: [B, max_pages]
    q: torch.Tensor            # [rows, H, 576] bf16
    q_idx: torch.Tensor        # [rows, h_idx, d_idx] bf16 or uint8 (e4m3 bits)
    w: torch.Tensor            # [rows, h_idx] fp32
    seq_lens: Optional[torch.Tensor] = None  # decode: [B] int32 (keys incl. new tokens)
    prefix_len: int = 0
    n_tokens: int = 0

    @property
    def n_rows(self) -> int:
        return self.q.shape[0]

    def to(self, device) -> "Problem":
        f = lambda t: None if t is None else t.to(device)
        return Problem(self.spec, self.cache.to(device), f(self.page_table), f(self.q),
                       f(self.q_idx), f(self.w), f(self.seq_lens), self.prefix_len,
                       self.n_tokens)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, g, device, chunk_elems=1 << 26) -> torch.Tensor:
    """N(0,1) in fp32, rounded to bf16, drawn in chunks to bound peak memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def _fp8_rows(n_rows: int, width: int, g, device, chunk_rows=1 << 17):
    """Per-row FP8 quantisation of N(0,1) rows: scale = amax/448, e4m3 RNE."""
    codes = torch.empty((n_rows, width), dtype=torch.uint8, device=device)
    scales = torch.empty((n_rows,), dtype=torch.float32, device=device)
    for s in range(0, n_rows, chunk_rows):
        e = min(n_rows, s + chunk_rows)
        x = torch.randn((e - s, width), generator=g, device=device, dtype=torch.float32)
        amax = x.abs().amax(dim=1).clamp_min(1e-12)
        sc = amax / 448.0
        q8 = (x / sc[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        codes[s:e] = q8.view(torch.uint8)
        scales[s:e] = sc
    return codes, scales


def _int_uniform(shape, lo, hi, g, device, dtype):
    """Integers uniform in [lo, hi], encoded as bf16 or e4m3 bits (both exact)."""
    x = torch.randint(lo, hi + 1, shape, generator=g, device=device, dtype=torch.int32)
    if dtype == BF16:
        return x.to(torch.bfloat16)
    if dtype == FP8:
        return x.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)
    if dtype == "f32":
        return x.to(torch.float32)
    raise ValueError(dtype)


def _ds_mla_rows(n_rows: int, g, device, chunk_rows=1 << 16) -> torch.Tensor:
    """656-byte rows: bytes 0..511 the e4m3 codes of the 512 latent values,
    512..527 four fp32 scales (one per 128-value tile, amax/448), 528..655 the 64
    rope values in bf16; all drawn N(0,1)."""
    out = torch.empty((n_rows, DS_MLA_ROW_BYTES), dtype=torch.uint8, device=device)
    for s in range(0, n_rows, chunk_rows):
        e = min(n_rows, s + chunk_rows)
        x = torch.randn((e - s, D_QK), generator=g, device=device, dtype=torch.float32)
        lat = x[:, :D_V].reshape(e - s, 4, 128)
        sc = (lat.abs().amax(dim=2).clamp_min(1e-12) / 448.0)
        codes = (lat / sc[:, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        out[s:e, :D_V] = codes.reshape(e - s, D_V)
        out[s:e, D_V:D_V + 16] = sc.contiguous().view(torch.uint8)
        out[s:e, D_V + 16:] = x[:, D_V:].to(torch.bfloat16).contiguous().view(torch.uint8)
    return out


def make_cache(spec: Spec, n_tokens_total: int, g, device, pool_pages: Optional[int] = None) -> Cache:
    pages = pool_pages if pool_pages is not None else -(-n_tokens_total // PAGE)
    rows = pages * PAGE
    if spec.kv_dtype == BF16:
        kv = _normal_bf16((pages, PAGE, D_QK), g, device)
        kv_scale = None
    elif spec.kv_dtype == FP8_DS_MLA:
        kv = _ds_mla_rows(rows, g, device).view(pages, PAGE, DS_MLA_ROW_BYTES)
        kv_scale = None
    else:
        codes, sc = _fp8_rows(rows, D_QK, g, device)
        kv = codes.view(pages, PAGE, D_QK)
        kv_scale = sc.view(pages, PAGE)
    k_idx = _int_uniform((pages, PAGE, spec.d_idx), -4, 4, g, device, spec.idx_dtype)
    return Cache(kv, kv_scale, k_idx, None, spec.kv_dtype, spec.idx_dtype)


def make_prefill(spec: Spec, device="cpu") -> Problem:
    """One prefill call: `n_tokens` new queries after `prefix_len` cached tokens.

    The page table maps logical page i of the sequence to a pool page. With
    `spec.shuffled` the pool pages are a seeded permutation, else identity.
    """
    assert spec.kind == "prefill"
    g = _gen(spec.seed, device)
    total = spec.prefix_len + spec.n_tokens
    n_pages = -(-total // PAGE)
    cache = make_cache(spec, total, g, device)
    if spec.shuffled:
        pt = torch.randperm(n_pages, generator=g, device=device).to(torch.int32)
    else:
        pt = torch.arange(n_pages, device=device, dtype=torch.int32)
    T = spec.n_tokens
    q = _normal_bf16((T, spec.n_heads, D_QK), g, device)
    q_idx = _int_uniform((T, spec.h_idx, spec.d_idx), -4, 4, g, device, spec.idx_dtype)
    w = _int_uniform((T, spec.h_idx), 1, 4, g, device, "f32")
    return Problem(spec, cache, pt, q, q_idx, w, None, spec.prefix_len, T)


def make_decode(spec: Spec, device="cpu") -> Problem:
    """Decode: `n_seqs` requests with `q_per_seq` new tokens each (already in the cache).

    seq_lens[b] counts every key of request b including its new tokens; query j of
    request b sits at position seq_lens[b] - q_per_seq + j.
    """
    assert spec.kind == "decode"
    g = _gen(spec.seed, device)
    B = spec.n_seqs
    lens = torch.randint(spec.len_min, spec.len_max + 1, (B,), generator=g, device=device,
                         dtype=torch.int32)
    pages_per = [-(-int(L) // PAGE) for L in lens.tolist()]
    total_pages = sum(pages_per)
    max_pages = max(pages_per)
    cache = make_cache(spec, total_pages * PAGE, g, device, pool_pages=total_pages)
    perm = torch.randperm(total_pages, generator=g, device=device).to(torch.int32)
    pt = torch.full((B, max_pages), -1, dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(pages_per):
        pt[b, :n] = perm[off:off + n]
        off += n
    rows = B * spec.q_per_seq
    q = _normal_bf16((rows, spec.n_heads, D_QK), g, device)
    q_idx = _int_uniform((rows, spec.h_idx, spec.d_idx), -4, 4, g, device, spec.idx_dtype)
    w = _int_uniform((rows, spec.h_idx), 1, 4, g, device, "f32")
    return Problem(spec, cache, pt, q, q_idx, w, lens, 0, 0)


def make(spec: Spec, device="cpu") -> Problem:
    return make_decode(spec, device) if spec.kind == "decode" else make_prefill(spec, device)
