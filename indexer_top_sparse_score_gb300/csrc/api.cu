// extern "C" entry points of libsmla.so: argument checks, workspace layout,
// and the launch sequence of each call. No allocation, no synchronisation
// (smla_read_status excepted).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace smla {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cache(const smla_paged_cache* c, bool need_kv, bool need_idx) {
  if (!c) return SMLA_ERR_INVALID_ARG;
  if (c->page_size != kPage || c->num_pages <= 0) return c->page_size != kPage && c->page_size > 0
                                                               ? SMLA_ERR_UNSUPPORTED
                                                               : SMLA_ERR_INVALID_ARG;
  if (c->num_pages > (1 << 25)) return SMLA_ERR_UNSUPPORTED;  // pool rows must fit int32
  if (need_kv) {
    if (!c->kv || !aligned16(c->kv)) return SMLA_ERR_INVALID_ARG;
    if (c->kv_dtype != SMLA_BF16 && c->kv_dtype != SMLA_FP8_E4M3 && c->kv_dtype != SMLA_FP8_DS_MLA)
      return SMLA_ERR_INVALID_ARG;
    if (c->kv_dtype == SMLA_FP8_E4M3 && !c->kv_scale) return SMLA_ERR_INVALID_ARG;
  }
  if (need_idx) {
    if (!c->k_idx || !aligned16(c->k_idx)) return SMLA_ERR_INVALID_ARG;
    if (c->idx_dtype != SMLA_BF16 && c->idx_dtype != SMLA_FP8_E4M3) return SMLA_ERR_INVALID_ARG;
    const int esz = c->idx_dtype == SMLA_BF16 ? 2 : 1;
    if (c->d_idx <= 0) return SMLA_ERR_INVALID_ARG;
    if (c->d_idx * esz != kIdxRowBytes) return SMLA_ERR_UNSUPPORTED;
  }
  return SMLA_OK;
}

bool valid_h_idx(int h) { return h == 4 || h == 8 || h == 16 || h == 32 || h == 64; }

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

int reset_status(void* ws, cudaStream_t st) {
  return cudaMemsetAsync(ws, 0, 4, st) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner_elems,
               uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner_elems, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t prefill_min_workspace(int32_t n_tokens, int32_t topk) {
  if (n_tokens <= 0 || topk <= 0) return kStatusBytes;
  return kStatusBytes + (static_cast<size_t>(n_tokens) * topk * 4 + 255) / 256 * 256;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

}  // namespace smla

using namespace smla;

extern "C" {

const char* smla_status_string(int status) {
  switch (status) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_INVALID_ARG: return "SMLA_ERR_INVALID_ARG: invalid argument";
    case SMLA_ERR_UNSUPPORTED: return "SMLA_ERR_UNSUPPORTED: valid but unsupported shape or type";
    case SMLA_ERR_WORKSPACE: return "SMLA_ERR_WORKSPACE: workspace missing or too small";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA: a CUDA runtime call failed";
    case SMLA_ERR_DEVICE_BOUNDS: return "SMLA_ERR_DEVICE_BOUNDS: an out-of-range page or key was skipped";
    case SMLA_ERR_TIMEOUT: return "SMLA_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "SMLA_ERR_UNKNOWN";
  }
}

int smla_version(void) { return 100; }

// ----------------------------------------------------------------- indexer
size_t smla_indexer_topk_workspace_size(int32_t n_seqs, int32_t max_seq_len, int32_t q_per_seq,
                                        int32_t h_idx, int32_t topk) {
  if (n_seqs <= 0 || max_seq_len <= 0 || q_per_seq <= 0 || topk <= 0) return kStatusBytes;
  return round256(indexer_workspace_bytes(n_seqs, max_seq_len, q_per_seq, h_idx, topk)) +
         indexer_group_cand_bytes(n_seqs * q_per_seq, q_per_seq, h_idx, topk, max_seq_len);
}

static int indexer_checks(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                          int32_t n_seqs, int32_t max_seq_len, int32_t q_per_seq, const void* q_idx,
                          const float* w, int32_t h_idx, int32_t topk) {
  int rc = check_cache(cache, false, true);
  if (rc) return rc;
  if (!page_tables || !q_idx || !w) return SMLA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(page_tables)) return SMLA_ERR_INVALID_ARG;
  if (n_seqs <= 0 || q_per_seq <= 0 || max_seq_len < q_per_seq || max_pages <= 0) return SMLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_pages) * kPage < max_seq_len) return SMLA_ERR_INVALID_ARG;
  if (topk <= 0) return SMLA_ERR_INVALID_ARG;
  if (topk > 2048) return SMLA_ERR_UNSUPPORTED;
  if (!valid_h_idx(h_idx)) return SMLA_ERR_UNSUPPORTED;
  return SMLA_OK;
}

int smla_indexer_topk(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                      int32_t n_seqs, const int32_t* seq_lens, int32_t max_seq_len, int32_t q_per_seq,
                      const void* q_idx, const float* w, int32_t h_idx, int32_t topk, int32_t* out_idx,
                      float* out_scores, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = indexer_checks(cache, page_tables, max_pages, n_seqs, max_seq_len, q_per_seq, q_idx, w, h_idx, topk);
  if (rc) return rc;
  if (!seq_lens || !out_idx) return SMLA_ERR_INVALID_ARG;
  const bool split = indexer_split_mode(q_per_seq, h_idx);
  if (indexer_tokens_per_cta(h_idx, topk, split, q_per_seq) <= 0) return SMLA_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace)) return SMLA_ERR_WORKSPACE;
  // required: status word (+ split-mode lists); the group-mode score array
  // or candidate buffers behind it are used when they fit
  const size_t ws_min = round256(indexer_workspace_bytes(n_seqs, max_seq_len, q_per_seq, h_idx, topk));
  if (workspace_bytes < ws_min) return SMLA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = reset_status(workspace, st))) return rc;
  IndexerLaunch L{cache, page_tables, max_pages, n_seqs, q_per_seq, seq_lens, 0, max_seq_len, q_idx, w,
                  h_idx, topk, out_idx, out_scores, workspace, ws_min, st};
  L.cand = static_cast<uint8_t*>(workspace) + ws_min;
  L.cand_bytes = workspace_bytes - ws_min;
  return launch_indexer(L);
}

// ----------------------------------------------------------------- sparse MLA (given indices)
size_t smla_sparse_mla_fwd_workspace_size(int32_t max_keys, int32_t, int32_t, int32_t, int32_t kv_dtype) {
  return kStatusBytes + mla_shadow_bytes(max_keys, kv_dtype);
}

static int mla_checks(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                      int32_t n_seqs, int32_t q_per_seq, const void* q, int32_t n_heads, int32_t topk,
                      const void* out, const float* lse) {
  int rc = check_cache(cache, true, false);
  if (rc) return rc;
  if (!page_tables || !q || !out) return SMLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return SMLA_ERR_INVALID_ARG;
  if (n_seqs <= 0 || q_per_seq <= 0 || max_pages <= 0) return SMLA_ERR_INVALID_ARG;
  if (topk <= 0) return SMLA_ERR_INVALID_ARG;
  if (topk > 2048) return SMLA_ERR_UNSUPPORTED;
  if (n_heads != 16 && n_heads != 64) return SMLA_ERR_UNSUPPORTED;
  return SMLA_OK;
}

int smla_sparse_mla_fwd(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                        int32_t n_seqs, const int32_t* seq_lens, int32_t prefix_len, int32_t q_per_seq,
                        const void* q, int32_t n_heads, const int32_t* idx, int32_t topk, float sm_scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = mla_checks(cache, page_tables, max_pages, n_seqs, q_per_seq, q, n_heads, topk, out, lse);
  if (rc) return rc;
  if (!idx) return SMLA_ERR_INVALID_ARG;
  if (!seq_lens && (n_seqs != 1 || prefix_len < 0)) return SMLA_ERR_INVALID_ARG;
  if (!seq_lens && static_cast<int64_t>(max_pages) * kPage < static_cast<int64_t>(prefix_len) + q_per_seq)
    return SMLA_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return SMLA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return SMLA_ERR_WORKSPACE;
  if (workspace_bytes < kStatusBytes) return SMLA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = reset_status(workspace, st))) return rc;
  MlaLaunch L{cache, page_tables, max_pages, n_seqs, q_per_seq, seq_lens, prefix_len, q, n_heads, idx, topk,
              sm_scale, out, lse, static_cast<uint32_t*>(workspace), st};
  // one sequence and room in the workspace: widen its rows once, gather f16
  const int32_t n_keys = prefix_len + q_per_seq;
  const size_t shadow_bytes = mla_shadow_bytes(n_keys, cache->kv_dtype);
  if (!seq_lens && shadow_bytes > 0 && workspace_bytes >= kStatusBytes + shadow_bytes) {
    L.shadow = static_cast<uint8_t*>(workspace) + kStatusBytes;
    L.shadow_rows = n_keys;
    if ((rc = launch_shadow_convert(L))) return rc;
  }
  return launch_mla(L);
}

// ----------------------------------------------------------------- prefill
size_t smla_sparse_mla_prefill_workspace_size(int32_t prefix_len, int32_t n_tokens, int32_t, int32_t h_idx,
                                              int32_t topk, int32_t kv_dtype) {
  if (prefix_len < 0 || n_tokens <= 0 || topk <= 0) return kStatusBytes;
  return prefill_min_workspace(n_tokens, topk) +
         mla_shadow_bytes(prefix_len + n_tokens, kv_dtype) +
         indexer_group_cand_bytes(n_tokens, n_tokens, h_idx, topk,
                                  static_cast<int32_t>(std::min<int64_t>(INT32_MAX, int64_t(prefix_len) + n_tokens)));
}

int smla_sparse_mla_prefill(const smla_paged_cache* cache, const int32_t* page_table, int32_t prefix_len,
                            int32_t n_tokens, const void* q, int32_t n_heads, const void* q_idx,
                            const float* w, int32_t h_idx, int32_t topk, float sm_scale, void* out,
                            float* lse, int32_t* out_idx, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (prefix_len < 0 || n_tokens <= 0) return SMLA_ERR_INVALID_ARG;
  const int64_t total = static_cast<int64_t>(prefix_len) + n_tokens;
  if (total > INT32_MAX - 2 * kPage) return SMLA_ERR_INVALID_ARG;
  const int32_t pages = static_cast<int32_t>((total + kPage - 1) / kPage);
  int rc = check_cache(cache, true, true);
  if (rc) return rc;
  if (!q_idx || !w || !page_table || !aligned16(q_idx) || !aligned16(page_table)) return SMLA_ERR_INVALID_ARG;
  if (!valid_h_idx(h_idx)) return SMLA_ERR_UNSUPPORTED;
  rc = mla_checks(cache, page_table, pages, 1, n_tokens, q, n_heads, topk, out, lse);
  if (rc) return rc;
  if (!(sm_scale == sm_scale)) return SMLA_ERR_INVALID_ARG;
  if (indexer_tokens_per_cta(h_idx, topk, false, n_tokens) <= 0) return SMLA_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace)) return SMLA_ERR_WORKSPACE;
  const size_t ws_min = prefill_min_workspace(n_tokens, topk);
  if (workspace_bytes < ws_min) return SMLA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = reset_status(workspace, st))) return rc;
  int32_t* idx = out_idx ? out_idx : reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
  IndexerLaunch IL{cache, page_table, pages, 1, n_tokens, nullptr, prefix_len, static_cast<int32_t>(total), q_idx,
                   w, h_idx, topk, idx, nullptr, workspace, workspace_bytes, st};
  // layout: status | index list | f16 copy of the rows (BF16 and per-token FP8 caches) |
  // the indexer's score array or deferred candidate buffers
  const size_t shadow_bytes = mla_shadow_bytes(static_cast<int32_t>(total), cache->kv_dtype);
  const size_t cand_off = ws_min + shadow_bytes;
  if (workspace_bytes > cand_off) {
    IL.cand = static_cast<uint8_t*>(workspace) + cand_off;
    IL.cand_bytes = workspace_bytes - cand_off;
  }
  if ((rc = launch_indexer(IL))) return rc;
  MlaLaunch ML{cache, page_table, pages, 1, n_tokens, nullptr, prefix_len, q, n_heads, idx, topk, sm_scale, out,
               lse, static_cast<uint32_t*>(workspace), st};
  // room in the workspace: widen the sequence's rows once, gather f16
  if (shadow_bytes > 0 && workspace_bytes >= ws_min + shadow_bytes) {
    ML.shadow = static_cast<uint8_t*>(workspace) + ws_min;
    ML.shadow_rows = static_cast<int32_t>(total);
    if ((rc = launch_shadow_convert(ML))) return rc;
  }
  return launch_mla(ML);
}

// ----------------------------------------------------------------- decode
size_t smla_sparse_mla_decode_workspace_size(int32_t n_seqs, int32_t max_seq_len, int32_t q_per_seq,
                                             int32_t n_heads, int32_t h_idx, int32_t topk) {
  if (n_seqs <= 0 || max_seq_len <= 0 || q_per_seq <= 0 || topk <= 0) return kStatusBytes;
  return round256(indexer_workspace_bytes(n_seqs, max_seq_len, q_per_seq, h_idx, topk)) +
         round256(static_cast<size_t>(n_seqs) * q_per_seq * topk * 4) +
         (n_heads > 0 ? mla_partial_bytes(n_seqs * q_per_seq, n_heads) : 0);
}

int smla_sparse_mla_decode(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                           int32_t n_seqs, const int32_t* seq_lens, int32_t max_seq_len,
                           int32_t q_per_seq, const void* q, int32_t n_heads, const void* q_idx,
                           const float* w, int32_t h_idx, int32_t topk, float sm_scale, void* out,
                           float* lse, int32_t* out_idx, void* workspace, size_t workspace_bytes,
                           void* stream) {
  int rc = indexer_checks(cache, page_tables, max_pages, n_seqs, max_seq_len, q_per_seq, q_idx, w, h_idx, topk);
  if (rc) return rc;
  if (!seq_lens) return SMLA_ERR_INVALID_ARG;
  if (q_per_seq > 8) return SMLA_ERR_UNSUPPORTED;
  rc = mla_checks(cache, page_tables, max_pages, n_seqs, q_per_seq, q, n_heads, topk, out, lse);
  if (rc) return rc;
  if (!(sm_scale == sm_scale)) return SMLA_ERR_INVALID_ARG;
  const bool split = indexer_split_mode(q_per_seq, h_idx);
  if (indexer_tokens_per_cta(h_idx, topk, split, q_per_seq) <= 0) return SMLA_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace)) return SMLA_ERR_WORKSPACE;
  if (workspace_bytes < smla_sparse_mla_decode_workspace_size(n_seqs, max_seq_len, q_per_seq, n_heads, h_idx, topk))
    return SMLA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = reset_status(workspace, st))) return rc;
  const size_t idx_ws = round256(indexer_workspace_bytes(n_seqs, max_seq_len, q_per_seq, h_idx, topk));
  int32_t* idx = out_idx ? out_idx : reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + idx_ws);
  IndexerLaunch IL{cache, page_tables, max_pages, n_seqs, q_per_seq, seq_lens, 0, max_seq_len, q_idx, w, h_idx,
                   topk, idx, nullptr, workspace, idx_ws, st};
  if ((rc = launch_indexer(IL))) return rc;
  MlaLaunch ML{cache, page_tables, max_pages, n_seqs, q_per_seq, seq_lens, 0, q, n_heads, idx, topk, sm_scale, out,
               lse, static_cast<uint32_t*>(workspace), st};
  // layout: indexer part | index list | partial outputs of split rows (if it fits)
  const size_t part_off = idx_ws + round256(static_cast<size_t>(n_seqs) * q_per_seq * topk * 4);
  if (workspace_bytes > part_off) {
    ML.partials = static_cast<uint8_t*>(workspace) + part_off;
    ML.partial_bytes = workspace_bytes - part_off;
  }
  return launch_mla(ML);
}

// ----------------------------------------------------------------- status
int smla_read_status(const void* workspace, void* stream, uint32_t* bits) {
  if (!workspace) return SMLA_ERR_INVALID_ARG;
  uint32_t v = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return SMLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SMLA_ERR_CUDA;
  if (bits) *bits = v;
  if (v & (kStatusTimeout | kStatusSetup)) return SMLA_ERR_TIMEOUT;
  if (v & kStatusBounds) return SMLA_ERR_DEVICE_BOUNDS;
  if (v & kStatusOverflow) return SMLA_ERR_UNSUPPORTED;
  return SMLA_OK;
}

}  // extern "C"
