"""Small hand-built problems for the oracle pins (host tensors only)."""
import torch

from indexer_top_sparse_score_gb300 import workloads as wl


def fp8_codes(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def custom_prefill(q_idx, w, k_idx, *, n_heads=2, q=None, kv=None, kv_dtype="bf16",
                   kv_scale=None, idx_dtype="bf16", topk=2, prefix_len=None, page_perm=None,
                   k_idx_scale=None):
    """One prefill sequence built from explicit tensors.

    q_idx [T,H_I,D_I], w [T,H_I], k_idx [N,D_I] (float values); kv [N,576] float
    values (bf16 path) or e4m3 codes (fp8 path); N keys are padded to whole pages.
    The query rows sit at prefix_len .. prefix_len+T-1 (default: the last T keys).
    """
    q_idx = torch.as_tensor(q_idx, dtype=torch.float32)
    w = torch.as_tensor(w, dtype=torch.float32)
    k_idx = torch.as_tensor(k_idx, dtype=torch.float32)
    T, H_I, D_I = q_idx.shape
    N = k_idx.shape[0]
    P = N - T if prefix_len is None else prefix_len
    pages = -(-N // wl.PAGE)
    rows = pages * wl.PAGE
    kpad = torch.zeros(rows, D_I)
    kpad[:N] = k_idx
    if kv is None:
        g = torch.Generator().manual_seed(7)
        kv = torch.randn(N, wl.D_QK, generator=g)
    if q is None:
        g = torch.Generator().manual_seed(8)
        q = torch.randn(T, n_heads, wl.D_QK, generator=g)
    if kv_dtype == "bf16":
        kvp = torch.zeros(rows, wl.D_QK, dtype=torch.bfloat16)
        kvp[:N] = torch.as_tensor(kv).to(torch.bfloat16)
        kvs = None
    elif kv_dtype == wl.FP8_DS_MLA:  # kv: packed 656-byte rows
        kvp = torch.zeros(rows, wl.DS_MLA_ROW_BYTES, dtype=torch.uint8)
        kvp[:N] = torch.as_tensor(kv, dtype=torch.uint8)
        kvs = None
    else:
        kvp = torch.zeros(rows, wl.D_QK, dtype=torch.uint8)
        kvp[:N] = torch.as_tensor(kv, dtype=torch.uint8)
        kvs = torch.ones(rows, dtype=torch.float32)
        if kv_scale is not None:
            kvs[:N] = torch.as_tensor(kv_scale, dtype=torch.float32)
    if idx_dtype == "bf16":
        kidx = kpad.to(torch.bfloat16)
        qidx = q_idx.to(torch.bfloat16)
    else:
        kidx = fp8_codes(kpad)
        qidx = fp8_codes(q_idx)
    kis = None
    if k_idx_scale is not None:
        kis = torch.ones(rows, dtype=torch.float32)
        kis[:N] = torch.as_tensor(k_idx_scale, dtype=torch.float32)
        kis = kis.view(pages, wl.PAGE)
    pt = torch.arange(pages, dtype=torch.int32)
    kvp = kvp.view(pages, wl.PAGE, kvp.shape[-1])
    kidx = kidx.view(pages, wl.PAGE, D_I)
    if kvs is not None:
        kvs = kvs.view(pages, wl.PAGE)
    if page_perm is not None:
        # logical page i lives at pool page perm[i]
        perm = torch.as_tensor(page_perm, dtype=torch.long)
        kvp2 = torch.empty_like(kvp)
        kvp2[perm] = kvp
        kidx2 = torch.empty_like(kidx)
        kidx2[perm] = kidx
        if kvs is not None:
            kvs2 = torch.empty_like(kvs)
            kvs2[perm] = kvs
            kvs = kvs2
        if kis is not None:
            kis2 = torch.empty_like(kis)
            kis2[perm] = kis
            kis = kis2
        kvp, kidx = kvp2, kidx2
        pt = perm.to(torch.int32)
    spec = wl.Spec("custom", "prefill", n_heads=n_heads, h_idx=H_I, d_idx=D_I,
                   idx_dtype=idx_dtype, kv_dtype=kv_dtype, topk=topk, seed=0,
                   n_tokens=T, prefix_len=P)
    cache = wl.Cache(kvp.contiguous(), None if kvs is None else kvs.contiguous(),
                     kidx.contiguous(), None if kis is None else kis.contiguous(),
                     kv_dtype, idx_dtype)
    prob = wl.Problem(spec, cache, pt.contiguous(),
                      torch.as_tensor(q).to(torch.bfloat16).contiguous(),
                      qidx.contiguous(), w.contiguous(), None, P, T)
    return prob
