/*
 * smla — indexer-selected sparse latent attention (MLA) for one GB300 (sm_103a).
 *
 * C ABI of the library built from indexer_top_sparse_score_gb300/csrc
 * (libsmla.so). One layer step of long-context sparse attention, per query
 * token, as described in "Optimisations de GLM-5.3, partie 2 : PCP, DCP et
 * Hybrid HiSparse sur 16 H200" (spke.com):
 *
 *   1. the indexer scores every earlier token (section "Pourquoi pas TP ou
 *      DP ?"), with the score fixed for this library as
 *        score(t, s) = sum_h w[t,h] * ReLU(q_I[t,h,:] . k_I[s,:]) * kscale[s];
 *   2. a causal top-k (k = 2048 on the page) keeps the best keys s <= pos(t),
 *      ties going to the lower index;
 *   3. sparse MLA in MQA form: every head attends over the selected rows of one
 *      shared latent cache; QK over 576 values, PV over the first 512 (footnote
 *      1), softmax with log-sum-exp output (section "DCP").
 *
 * Conventions for every entry point
 *   - All tensor arguments are DEVICE pointers into the caller's memory unless
 *     stated otherwise; the library never allocates, frees or synchronises
 *     (except smla_read_status, which waits on the stream). The caller owns
 *     every buffer. All work is enqueued on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and returns before it completes.
 *   - Layouts are dense, row-major, C order. Pointers must be 16-byte aligned.
 *   - Return values are smla_status codes. Argument checks happen on the host
 *     before anything is enqueued; on error nothing is enqueued. Errors found
 *     on the device (a page id outside the pool, a key index outside the
 *     cache, a bounded wait that gave up) are recorded as bits in a status word
 *     at the start of the workspace and read back with smla_read_status. The
 *     kernels never trap: an out-of-range entry is skipped.
 *   - The workspace is caller-owned device memory of at least the size the
 *     matching *_workspace_size function returns; its first 256 bytes hold the
 *     status word. Calls that share a workspace must be stream-ordered.
 *   - The library keeps no state between calls apart from one-time kernel
 *     attribute setup and the driver entry point used to encode TMA tensor
 *     maps.
 */
#ifndef SMLA_H_
#define SMLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum smla_status {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, inconsistent shapes */
  SMLA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head count, dims, topk) */
  SMLA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  SMLA_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute, no device) */
  SMLA_ERR_DEVICE_BOUNDS = 5,/* (smla_read_status) an out-of-range page or key was skipped */
  SMLA_ERR_TIMEOUT = 6       /* (smla_read_status) a bounded device wait gave up */
} smla_status;

typedef enum smla_dtype {
  SMLA_BF16 = 0,      /* bfloat16 */
  SMLA_FP8_E4M3 = 1,  /* OCP FP8 E4M3 (e4m3fn), one byte per value */
  SMLA_FP8_DS_MLA = 2 /* latent cache only: 656-byte tile-scaled FP8 rows (below) */
} smla_dtype;

/* Paged cache of one layer. Token s of a sequence lives in pool page
 * page_table[s / page_size] at slot s % page_size.
 *   kv          [num_pages][page_size][576]  kv_dtype. The latent row: values
 *               0..511 are the latent (also V), 512..575 the rope part.
 *               For SMLA_FP8_DS_MLA each row is 656 bytes (the row size that
 *               footnote 1 of "Optimisations de GLM-5.3, partie 2" gives for
 *               fp8_ds_mla; the split is this library's reading): bytes 0..511
 *               the e4m3 codes of latent values 0..511, bytes 512..527 four
 *               little-endian fp32 scales (scale t for values 128t..128t+127,
 *               value = e4m3 * scale), bytes 528..655 the 64 rope values in
 *               bf16. kv_scale is not used.
 *   kv_scale    [num_pages][page_size] fp32, SMLA_FP8_E4M3 only: value = e4m3
 *               * scale.
 *   k_idx       [num_pages][page_size][d_idx] idx_dtype: indexer keys.
 *   k_idx_scale [num_pages][page_size] fp32 positive per-key indexer scale, or
 *               NULL for 1 (footnote 3's 132-byte key = 128 FP8 + 4-byte scale).
 * page_size must be 64 and num_pages at most 2^25 (pool rows are indexed
 * with 32-bit integers; more is SMLA_ERR_UNSUPPORTED). An indexer row must be
 * 128 bytes: d_idx = 128 for e4m3 keys, d_idx = 64 for bf16 keys.
 * Host-resident latent cache ("Hybrid HiSparse": the KV of contexts too long
 * for HBM kept in host memory): kv and kv_scale may point to page-locked host
 * memory allocated or registered with CUDA (device-accessible through unified
 * addressing). The attention then reads only the selected rows, over the
 * host link, with the same results; k_idx, k_idx_scale, the page tables and
 * every other buffer must be device memory (the indexer streams its keys with
 * the tensor-memory accelerator). */
typedef struct smla_paged_cache {
  const void* kv;
  const float* kv_scale;
  const void* k_idx;
  const float* k_idx_scale;
  int32_t num_pages;
  int32_t page_size;
  int32_t kv_dtype;   /* smla_dtype */
  int32_t idx_dtype;  /* smla_dtype */
  int32_t d_idx;
} smla_paged_cache;

/* Human-readable name of a status code (static string, never NULL). */
const char* smla_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int smla_version(void);

/* ---------------------------------------------------------------------------
 * smla_indexer_topk — steps 1 and 2 for a batch of sequences.
 *
 *   page_tables [n_seqs][max_pages] int32 pool page ids.
 *   seq_lens    [n_seqs] int32 (device): keys of each sequence INCLUDING its
 *               q_per_seq new tokens; query j of sequence b sits at position
 *               seq_lens[b] - q_per_seq + j and sees keys 0..that position.
 *               Every seq_lens[b] must be >= q_per_seq and <= max_seq_len.
 *   max_seq_len host-side upper bound of seq_lens (sizes the launch).
 *   q_idx       [n_seqs*q_per_seq][h_idx][d_idx] idx_dtype.
 *   w           [n_seqs*q_per_seq][h_idx] fp32 head weights.
 *   out_idx     [n_seqs*q_per_seq][topk] int32: the selected key positions of
 *               every query row, min(topk, pos+1) valid entries first in no
 *               particular order (deterministic for given inputs), then -1.
 *   out_scores  [n_seqs*q_per_seq][topk] fp32 scores of out_idx, or NULL.
 * Supported: h_idx in {4, 8, 16, 32, 64}; 1 <= topk <= 2048. Integer-valued
 * inputs make the selection bit-identical to the exact fp32 definition.
 * Workspace: the returned size. When several query rows share the key stream
 * (long per-sequence batches), 256 bytes already suffice. With max_seq_len at
 * most 16384 (8192 at h_idx = 4) every row's scores fit in shared memory and
 * the exact top-k is taken there. Longer sequences at h_idx = 32: the rest of
 * the workspace holds a score array (4 bytes per key up to max_seq_len rounded
 * up to 32, per query row) that the scoring kernel fills and a per-row kernel
 * selects from; rows are processed in equal blocks (the same rows of every
 * sequence) of which the returned size holds one of up to 16 GiB, or at least
 * 608 rows per sequence; a smaller workspace gives smaller blocks. Other head
 * counts, or a workspace too small for a 608-row block: per-row candidate
 * buffers (up to
 * 16384 / rows-per-work-item (key, index) pairs of 8 bytes, plus a count per
 * row) whose final exact selection then runs in a separate light kernel
 * instead of stalling the scoring pipeline; with less room still the
 * selection stays in the scoring kernel. All modes select the same index sets.
 * Decode-shaped
 * calls (few rows per sequence, whose keys are split across SMs) require a
 * score array per query row (4 bytes per key up to max_seq_len): the scoring
 * kernel writes every score and a per-row kernel then selects the exact top-k.
 * ------------------------------------------------------------------------- */
size_t smla_indexer_topk_workspace_size(int32_t n_seqs, int32_t max_seq_len, int32_t q_per_seq,
                                        int32_t h_idx, int32_t topk);
int smla_indexer_topk(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                      int32_t n_seqs, const int32_t* seq_lens, int32_t max_seq_len, int32_t q_per_seq,
                      const void* q_idx, const float* w, int32_t h_idx, int32_t topk, int32_t* out_idx,
                      float* out_scores, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * smla_sparse_mla_fwd — step 3 alone over caller-given index lists.
 *
 * Rows are laid out as in smla_indexer_topk: n_seqs sequences of q_per_seq
 * rows. Positions: if seq_lens is NULL there is one sequence (n_seqs must be
 * 1) and row i sits at prefix_len + i; otherwise row j of sequence b sits at
 * seq_lens[b] - q_per_seq + j.
 *   q     [rows][n_heads][576] bf16 (the absorbed query, latent + rope).
 *   idx   [rows][topk] int32 key positions. Row r reads entries
 *         [0, min(topk, pos_r + 1)); entries < 0 or > pos_r are skipped.
 *   out   [rows][n_heads][512] bf16 attention output (normalised).
 *   lse   [rows][n_heads] fp32 natural-log sum of exp(sm_scale * q.K), or NULL.
 *         A row with no usable entry gets out = 0 and lse = -inf.
 * The attention MMAs run on f16 operands (q, the cache rows and the softmax
 * probabilities are widened to f16; e4m3 widens exactly, bf16 exactly inside
 * the f16 range), so |q| and |cache values| must stay below 65504; a query
 * value beyond it is reported by smla_read_status as SMLA_ERR_UNSUPPORTED.
 * Supported: n_heads in {16, 64} (16 and 64 query heads of the configurations),
 * topk <= 2048.
 * Workspace: 256 bytes suffice. For a BF16 or SMLA_FP8_E4M3 cache of one
 * sequence (seq_lens NULL) a larger workspace, as returned for max_keys =
 * prefix_len + q_per_seq, lets the call first widen the sequence's rows to f16
 * once (576 * 2 bytes per key, plus 4 bytes per key for the FP8 scales kept in
 * the same order) so the attention gathers them without per-row conversion.
 * Both widenings are exact, so the result does not depend on the workspace.
 * ------------------------------------------------------------------------- */
size_t smla_sparse_mla_fwd_workspace_size(int32_t max_keys, int32_t rows, int32_t n_heads, int32_t topk,
                                          int32_t kv_dtype);
int smla_sparse_mla_fwd(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                        int32_t n_seqs, const int32_t* seq_lens, int32_t prefix_len, int32_t q_per_seq,
                        const void* q, int32_t n_heads, const int32_t* idx, int32_t topk, float sm_scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * smla_sparse_mla_prefill — steps 1-3 for n_tokens new query tokens of ONE
 * sequence placed after prefix_len cached tokens (query i at prefix_len + i).
 * The caller has already written the KV and indexer-key rows of all
 * prefix_len + n_tokens tokens into the cache.
 *   page_table [ceil((prefix_len + n_tokens) / 64)] int32.
 *   q, q_idx, w, out, lse as above with rows = n_tokens.
 *   out_idx    [n_tokens][topk] int32 selected indices, or NULL to keep them
 *              in the workspace only.
 * Workspace: at least 256 + n_tokens * topk * 4 bytes (rounded to 256). The
 * returned size lays out, in order: the status word, the index list, for
 * kv_dtype = SMLA_BF16 or SMLA_FP8_E4M3 an f16 copy of the sequence's
 * prefix_len + n_tokens cache rows (widened exactly, written once per call and
 * gathered by the attention without per-row conversion; for FP8 followed by
 * the rows' scales in the same order), and the indexer's score array or
 * deferred candidate buffers (see smla_indexer_topk). Each optional part is
 * used only when the workspace reaches its end.
 * ------------------------------------------------------------------------- */
size_t smla_sparse_mla_prefill_workspace_size(int32_t prefix_len, int32_t n_tokens, int32_t n_heads,
                                              int32_t h_idx, int32_t topk, int32_t kv_dtype);
int smla_sparse_mla_prefill(const smla_paged_cache* cache, const int32_t* page_table, int32_t prefix_len,
                            int32_t n_tokens, const void* q, int32_t n_heads, const void* q_idx,
                            const float* w, int32_t h_idx, int32_t topk, float sm_scale, void* out,
                            float* lse, int32_t* out_idx, void* workspace, size_t workspace_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------
 * smla_sparse_mla_decode — steps 1-3 for a decode batch: n_seqs requests with
 * q_per_seq new tokens each (1 for plain decode, 2 for one MTP draft), over a
 * paged cache with one page table per request. Arguments as in
 * smla_indexer_topk and smla_sparse_mla_fwd. q_per_seq must be in [1, 8].
 * Workspace: the returned size holds, in order, the indexer's part (see
 * smla_indexer_topk), the index list, and room for fp32 partial outputs: with
 * fewer query rows than SMs each row's selection is cut into up to 4 parts
 * attended on different SMs and merged by their log-sum-exp (used only when
 * the workspace reaches its end).
 * ------------------------------------------------------------------------- */
size_t smla_sparse_mla_decode_workspace_size(int32_t n_seqs, int32_t max_seq_len, int32_t q_per_seq,
                                             int32_t n_heads, int32_t h_idx, int32_t topk);
int smla_sparse_mla_decode(const smla_paged_cache* cache, const int32_t* page_tables, int32_t max_pages,
                           int32_t n_seqs, const int32_t* seq_lens, int32_t max_seq_len,
                           int32_t q_per_seq, const void* q, int32_t n_heads, const void* q_idx,
                           const float* w, int32_t h_idx, int32_t topk, float sm_scale, void* out,
                           float* lse, int32_t* out_idx, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ---------------------------------------------------------------------------
 * smla_sparse_mla_prefill_noalloc — the same step as smla_sparse_mla_prefill
 * for callers that cannot allocate device memory and so cannot provide a
 * workspace: for example a plugin that is handed only input and output
 * pointers by its host framework, or an engine whose device memory is all
 * owned by a pool that outside code may not draw from. (This entry point has
 * no counterpart in the pages; it only changes where the scratch lives.)
 *
 * It allocates nothing. Its scratch (status word + the selected-index list)
 * is a fixed 16 MiB array inside the library, held by every GPU that loads
 * the library until the process exits. Limit: n_tokens * topk * 4 + 256
 * bytes must fit in 16 MiB (e.g. 2047 tokens at topk = 2048); larger calls
 * return SMLA_ERR_WORKSPACE and enqueue nothing. The f16 copy of the cache rows
 * (see smla_sparse_mla_prefill) is made only if it fits in the rest, and the
 * indexer's score array and deferred candidate buffers for rows longer than
 * 16,384 keys only for small calls: otherwise such rows take their exact
 * top-k inside the scoring kernel (same index sets). The
 * selected indices are not returned. Device-side errors (an out-of-range page,
 * a bounded wait that gave up) go to the array's status word: read them with
 * smla_noalloc_read_status after the call. The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture. The address is kept per
 * device for the process: it belongs to the runtime's primary context of the
 * device, so calls from another context (made current through the driver API)
 * and calls after cudaDeviceReset are not supported. Every call on a device
 * shares the one array and leaves its contents behind (each call clears the
 * status word and rewrites the index list): calls whose work overlaps on the
 * GPU, on different streams or threads, race and give wrong results.
 * Arguments otherwise as smla_sparse_mla_prefill.
 * ------------------------------------------------------------------------- */
int smla_sparse_mla_prefill_noalloc(const smla_paged_cache* cache, const int32_t* page_table,
                                    int32_t prefix_len, int32_t n_tokens, const void* q, int32_t n_heads,
                                    const void* q_idx, const float* w, int32_t h_idx, int32_t topk,
                                    float sm_scale, void* out, float* lse, void* stream);

/* smla_noalloc_read_status — smla_read_status for the status word of
 * smla_sparse_mla_prefill_noalloc (the first word of the library's scratch
 * array on the current device): waits for `stream`, then returns the status of
 * the calls since the last one began, with the raw bits in *bits if non-NULL.
 * Allocates nothing. (No counterpart in the pages either.) */
int smla_noalloc_read_status(void* stream, uint32_t* bits);

/* ---------------------------------------------------------------------------
 * smla_read_status — waits for `stream`, then reads the device status word of
 * `workspace` written by the calls that used it: SMLA_OK, SMLA_ERR_DEVICE_BOUNDS
 * or SMLA_ERR_TIMEOUT (the latter wins); the raw bit mask goes to *bits if
 * non-NULL; SMLA_ERR_UNSUPPORTED if a value was outside the supported range.
 * Each entry point clears the word when it starts.
 * ------------------------------------------------------------------------- */
int smla_read_status(const void* workspace, void* stream, uint32_t* bits);

#ifdef __cplusplus
}
#endif
#endif /* SMLA_H_ */
