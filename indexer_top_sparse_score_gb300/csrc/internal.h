// Host-side declarations shared by the launchers and the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/smla.h"

namespace smla {

constexpr int kPage = 64;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr size_t kStatusBytes = 256;
constexpr int kIdxRowBytes = 128;     // indexer key / query row bytes supported
constexpr int kKeyBlock = 8192;       // keys per work item in split (decode) mode
constexpr int kBufEntries = 16384;    // top-k candidate entries per indexer CTA

// Geometry of one indexer launch.
struct IndexerLaunch {
  const smla_paged_cache* cache;
  const int32_t* page_tables;
  int32_t max_pages;
  int32_t n_seqs, q_per_seq;
  const int32_t* seq_lens;  // device, or null: one sequence at prefix_len
  int32_t prefix_len;
  int32_t max_seq_len;      // host bound on keys of any sequence
  const void* q_idx;
  const float* w;
  int32_t h_idx, topk;
  int32_t* out_idx;
  float* out_scores;
  void* workspace;          // status word + candidate lists (split mode)
  size_t workspace_bytes;
  cudaStream_t stream;
  // group mode, rows longer than the dense mode takes: room for the score array
  // of a block of rows (score-array mode), else for the per-row candidate buffers
  // whose final selection is deferred to finish_kernel (null or too small for
  // either: the selection stays in the scoring kernel)
  void* cand = nullptr;
  size_t cand_bytes = 0;
};

struct MlaLaunch {
  const smla_paged_cache* cache;
  const int32_t* page_tables;
  int32_t max_pages;
  int32_t n_seqs, q_per_seq;
  const int32_t* seq_lens;
  int32_t prefix_len;
  const void* q;
  int32_t n_heads;
  const int32_t* idx;
  int32_t topk;
  float sm_scale;
  void* out;
  float* lse;
  uint32_t* status;
  cudaStream_t stream;
  // f16 copy of the sequence's cache rows in logical token order (BF16 or
  // per-token FP8 caches of a single sequence), or null to gather and widen the
  // pool rows in-kernel
  void* shadow = nullptr;
  int32_t shadow_rows = 0;
  // room for the partial outputs of split rows (few rows: each row's
  // selection is cut into parts spread over SMs and merged by lse), or null
  void* partials = nullptr;
  size_t partial_bytes = 0;
};

// Parts a row is split into when there are few rows (at most kMaxParts).
constexpr int kMaxParts = 4;
int mla_parts(int32_t n_rows, int32_t topk);
// Workspace bytes for the partial outputs of n_rows split rows.
size_t mla_partial_bytes(int32_t n_rows, int32_t n_heads);

// Workspace of a prefill without the optional f16 shadow (status + index list).
size_t prefill_min_workspace(int32_t n_tokens, int32_t topk);
// Bytes of the f16 shadow of n_keys cache rows (BF16 and per-token FP8
// caches; the FP8 shadow also holds the scales), 0 for other formats.
size_t mla_shadow_bytes(int32_t n_keys, int32_t kv_dtype);
// Fills the shadow from the pool through the page table (one sequence).
int launch_shadow_convert(const MlaLaunch& L);

// Whether the indexer runs token groups over the full key range (prefill) or
// splits each sequence's keys into blocks merged afterwards (decode).
bool indexer_split_mode(int32_t q_per_seq, int32_t h_idx);
int indexer_tokens_per_cta(int32_t h_idx, int32_t topk, bool split, int32_t q_per_seq);
// Rows per work item of dense group mode (every row's scores held in shared
// memory), or 0 when the rows are too long for it.
int indexer_dense_tokens(int32_t h_idx, int32_t topk, int32_t max_seq_len);
size_t indexer_workspace_bytes(int32_t n_seqs, int32_t max_seq_len, int32_t q_per_seq, int32_t h_idx,
                               int32_t topk);
// Group mode: bytes of the score array (one block of rows) or of the deferred
// per-row candidate buffers, whichever the rows use (0 if split or dense mode).
size_t indexer_group_cand_bytes(int32_t n_rows, int32_t q_per_seq, int32_t h_idx, int32_t topk,
                                int32_t max_seq_len);

int launch_indexer(const IndexerLaunch& L);   // returns smla_status
int launch_mla(const MlaLaunch& L);           // returns smla_status

// TMA tensor-map encoding through the driver entry point (no -lcuda).
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner_elems,
               uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swizzle);

int num_sms();

}  // namespace smla
