// Fused indexer + exact causal top-k (steps 1 and 2 of the layer step).
//
// "Optimisations de GLM-5.3, partie 2" (section "Pourquoi pas TP ou DP ?"):
// the indexer scores every earlier token and sparse MLA reads the best 2,048.
// Here the score is
//     score(t, s) = sum_h w[t,h] * ReLU(q_I[t,h,:] . k_I[s,:]) * kscale[s]
// and the selection keeps, per query row, the top-k keys s <= pos(t) ordered
// by (score descending, index ascending).
//
// One CTA per SM (persistent). A work item is TQ query rows against a key
// range, streamed in tiles of 128 keys:
//   warps 0, 3  TMA producers, taking the tiles in turn: k_I tiles (two
//               64-row pages each, page table resolved here) into a ring of
//               stages; warp 0 also loads the q_I tile once per item;
//   warps 1-2   MMA issuers, taking the tiles in turn: D[128 keys x (TQ*H_I)]
//               = k_I_tile . q_I^T with tcgen05 (kind::f8f6f4 for e4m3,
//               kind::f16 for bf16), fp32 accumulators in a ring of up to
//               four TMEM buffers (warp 2 also allocates TMEM);
//   warps 4..   the epilogue: each thread owns one key (TMEM lane) and
//               computes the ReLU + head-weighted sum of its query rows in
//               registers (fp32, packed FMAs).
// Work items: prefill ("group mode") takes TQ consecutive rows of one
// sequence against all their keys; items are handed out in head/tail pairs
// (the i-th cheapest with the i-th most expensive, the "V" pairing of the
// page's PCP section applied across SMs) so every CTA gets the same mix of
// short and long causal rows. How a row's top-k is taken depends on its
// length:
//   dense      rows of at most 16,384 keys (two rows per item): every score
//              goes to the row's array in shared memory at its key's
//              position; the exact top-k is taken there at the end of the
//              item. The score matrix never leaves the SM.
//   score      32 indexer heads, longer rows (four rows per item, sixteen
//   array      epilogue warps, one row per warpgroup): every
//              score goes to a per-row array in global memory with coalesced
//              stores, nothing shared between warps; select_sampled_kernel
//              then takes each row's exact top-k with one read of the row.
//              Rows go in blocks whose array fits the workspace.
//   streaming  other head counts, or a workspace too small for a score-array
//              block: scores that beat the row's threshold go to a candidate
//              buffer in shared memory; a full buffer is cut to a superset
//              of the row's top-k by a radix pass, which raises the
//              threshold (at 32 heads the two warpgroups take the tiles in
//              turn and the eight warps share the four rows' buffers). The
//              final exact selection runs in finish_kernel, or here when the
//              workspace has no room for the buffers.
// Decode ("split mode") takes all rows of one sequence against one block of
// key tiles and writes every score to the row's score array; the selection
// kernel then takes each row's exact top-k.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace smla {

namespace {

constexpr int kStages = 4;         // key-tile ring in group mode (the candidate / score buffers need the rest)
constexpr int kSplitStages = 10;   // split mode keeps no candidates: 6 more stages and a second
                                   // query tile in their space
constexpr int kTileKeys = 128;
constexpr int kStageBytes = kTileKeys * kIdxRowBytes;  // 16 KB
constexpr int kMaxN = 128;                             // TQ * H_I
constexpr int kEpiThreads = 256;
constexpr int kThreads = 384;
constexpr int kStoreThreads = 640;  // score-array mode: 16 epilogue warps, one query row per warpgroup
// Streaming prefill with 32 indexer heads (see the epilogue): the eight
// epilogue warps meet on one mbarrier of the kTokBars slots.
constexpr int kTokBars = 4;
constexpr int kHistWords = 3 * 256 * 4;  // selection histograms (room for every mode's layout)
constexpr int kMaxAcc = 4;                            // TMEM accumulator buffers at most
constexpr int kIssuers = 2;                           // MMA issuer warps
static_assert(kStages % kIssuers == 0 && kSplitStages % kIssuers == 0 && kMaxAcc % kIssuers == 0,
              "each ring barrier belongs to one issuer");
static_assert(kStages % 2 == 0 && kSplitStages % 2 == 0, "each stage belongs to one of the two producers");

struct IdxParams {
  const float* k_scale;  // [pool rows] or null
  const int32_t* page_tables;
  int32_t max_pages, num_pages;
  int32_t n_seqs, q_per_seq, n_rows;
  const int32_t* seq_lens;  // device or null
  int32_t prefix_len;
  const float* w;
  int32_t topk;
  int32_t tq, cap;
  int32_t is_bf16;
  int32_t split;
  int32_t n_groups;   // group mode: groups per sequence (of the launch's row block)
  int32_t row_base, block_rows;  // group mode: rows [row_base, row_base + block_rows) of every sequence
  int32_t n_kblocks;  // split mode: key blocks per sequence
  int32_t n_items;    // group mode: n_seqs * n_groups; split: n_seqs * n_kblocks
  int32_t tmem_cols;
  int32_t acc_shift;  // log2 of the TMEM accumulator buffers (1, 2 or 4 buffers)
  int32_t* out_idx;
  float* out_scores;
  uint32_t* cand_key;  // group mode: per-row deferred candidate buffers
  uint32_t* cand_idx;
  int32_t* cand_cnt;
  int32_t defer;       // group mode: hand rows with more than topk candidates to finish_kernel
  int32_t rot_span;    // group mode: tiles over which the CTAs' start tiles are spread (0: the whole range)
  uint32_t* scores;    // split and score-array modes: score keys [rows][score_stride], keys 0..pos
  int64_t score_stride;
  uint32_t* status;
};

struct Item {
  int seq, row0, nrows, pos0;
  int srow;  // the item's first row in the launch's score array
  int key_lo, key_hi;
  int t0, t1;
  int rot;  // tiles are streamed from t0 + rot, wrapping: CTAs start at different tiles
  int kb;
  bool trivial;
};

// Tile streamed at step tt (0 <= tt < t1 - t0) of an item. The top-k does not
// depend on the key order; rotating it per CTA keeps the CTAs from all reading
// the same key tile (and the same L2 slices) at the same time.
__device__ __forceinline__ int tile_at(const Item& it, int tt) {
  const int nt = it.t1 - it.t0;
  int u = tt + it.rot;
  if (u >= nt) u -= nt;
  return it.t0 + u;
}

// The k-th item of this CTA. Returns -1 when the CTA has no more items, 0 for
// an empty slot (skip), 1 for a real item. Every role calls this with the
// same k sequence, so all roles agree on the schedule.
// Split mode, for up to kMaxPrefixSeqs sequences: the sequences' key tiles are
// laid end to end (a per-CTA prefix sum of the tile counts, held in the
// otherwise unused histogram scratch) and CTA b takes the b-th of gridDim.x
// equal contiguous ranges; its k-th item is the k-th sequence piece of that
// range. More sequences fall back to fixed blocks of kKeyBlock keys.
constexpr int kMaxPrefixSeqs = 1535;

__device__ __forceinline__ int split_len(const IdxParams& p, int seq) {
  return min(p.seq_lens[seq], static_cast<int>(p.score_stride));  // keys with a score slot
}

__device__ __forceinline__ int next_item(const IdxParams& p, int k, Item& it, const uint32_t* pref) {
  if (!p.split) {
    const int G = p.n_items;
    const int P = (G + 1) / 2;
    const int pair = blockIdx.x + (k >> 1) * gridDim.x;
    if (pair >= P) return -1;
    int g = (k & 1) ? (G - 1 - pair) : pair;
    if ((k & 1) && g == pair) return 0;
    const int seq = g / p.n_groups;
    const int gi = g - seq * p.n_groups;
    const int rin = p.row_base + gi * p.tq;
    it.seq = seq;
    it.row0 = seq * p.q_per_seq + rin;
    it.nrows = min(p.tq, p.row_base + p.block_rows - rin);
    it.srow = seq * p.block_rows + gi * p.tq;
    const int L = p.seq_lens ? p.seq_lens[seq] : p.prefix_len + p.q_per_seq;
    it.pos0 = L - p.q_per_seq + rin;
    it.key_lo = 0;
    it.key_hi = it.pos0 + it.nrows;
    it.kb = 0;
    it.trivial = it.key_hi <= p.topk && p.out_scores == nullptr;
  } else {
    int seq;
    if (pref) {
      const uint32_t total = pref[p.n_seqs];
      const uint32_t lo = static_cast<uint32_t>(static_cast<uint64_t>(total) * blockIdx.x / gridDim.x);
      const uint32_t hi = static_cast<uint32_t>(static_cast<uint64_t>(total) * (blockIdx.x + 1) / gridDim.x);
      if (lo >= hi) return -1;
      int a = 0, b = p.n_seqs - 1;  // the last sequence starting at or before tile lo
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (pref[mid] <= lo) a = mid;
        else b = mid - 1;
      }
      seq = a + k;
      if (seq >= p.n_seqs || pref[seq] >= hi) return -1;
      const uint32_t s0 = max(lo, pref[seq]), s1 = min(hi, pref[seq + 1]);
      if (s1 <= s0) return 0;
      it.key_lo = static_cast<int>(s0 - pref[seq]) * kTileKeys;
      it.key_hi = min(split_len(p, seq), static_cast<int>(s1 - pref[seq]) * kTileKeys);
      it.kb = 0;
    } else {
      const int i = blockIdx.x + k * gridDim.x;
      if (i >= p.n_items) return -1;
      seq = i / p.n_kblocks;
      const int kb = i - seq * p.n_kblocks;
      const int L = split_len(p, seq);
      if (kb * kKeyBlock >= L) return 0;
      it.key_lo = kb * kKeyBlock;
      it.key_hi = min(L, it.key_lo + kKeyBlock);
      it.kb = kb;
    }
    it.seq = seq;
    it.row0 = seq * p.q_per_seq;
    it.srow = it.row0;
    it.nrows = p.q_per_seq;
    it.pos0 = p.seq_lens[seq] - p.q_per_seq;
    it.trivial = false;
  }
  if (it.key_hi <= it.key_lo) return 0;
  it.t0 = it.key_lo / kTileKeys;
  it.t1 = (it.key_hi + kTileKeys - 1) / kTileKeys;
  const int span = (!p.split && p.rot_span > 0) ? min(p.rot_span, it.t1 - it.t0) : it.t1 - it.t0;
  it.rot = static_cast<int>((blockIdx.x * 97u + static_cast<unsigned>(k) * 31u) % static_cast<unsigned>(span));
  return 1;
}

__device__ __forceinline__ int page_of(const IdxParams& p, const int32_t* pt, int lp) {
  if (lp >= p.max_pages) {
    set_status(p.status, kStatusBounds);
    return 0;
  }
  const int pg = __ldg(pt + lp);
  if (pg < 0 || pg >= p.num_pages) {
    set_status(p.status, kStatusBounds);
    return 0;
  }
  return pg;
}

template <int HI>
__device__ __forceinline__ void tmem_ld_heads(uint32_t taddr, uint32_t* r) {
  if constexpr (HI == 4) tmem_ld_32x32b_x4(taddr, r);
  else if constexpr (HI == 8) tmem_ld_32x32b_x8(taddr, r);
  else if constexpr (HI == 16) tmem_ld_32x32b_x16(taddr, r);
  else if constexpr (HI == 32) tmem_ld_32x32b_x32(taddr, r);
  else {
    tmem_ld_32x32b_x32(taddr, r);
    tmem_ld_32x32b_x32(taddr + 32, r + 32);
  }
}

// (d0, d1) += (a0, a1) * (b0, b1), both lanes rounded as fmaf (one packed FMA)
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rd, {%0, %1};\n\tfma.rn.f32x2 rd, ra, rb, rd;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// shared-memory counter increment whose old value is not needed
__device__ __forceinline__ void smem_inc(uint32_t* p) {
  asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(smem_u32(p)) : "memory");
}

// SPLIT: decode shape (compile-time, so the decode kernel carries none of the
// candidate-selection code). DENSE: prefill rows short enough that every
// score of a work item fits in shared memory (see the epilogue). TOK: the
// streaming prefill at 32 heads (four rows per item, the two warpgroups
// taking the tiles in turn, candidate buffers shared by the eight warps).
// STORE: prefill at 32 heads writing every score to a score array in global
// memory (select_sampled_kernel takes the exact top-k afterwards).
template <int HI, bool SPLIT, bool DENSE, bool TOK, bool STORE>
__global__ void __launch_bounds__(STORE ? kStoreThreads : kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_q,
                   const IdxParams p) {
  static_assert(!TOK || (HI == 32 && !SPLIT && !DENSE), "the streaming 32-head mode is a prefill mode");
  static_assert(!STORE || (HI == 32 && !SPLIT && !DENSE && !TOK), "the score-array mode is a 32-head prefill mode");
  constexpr int TPW_MAX = 64 / HI;  // tokens per epilogue warpgroup held in registers
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* a_tiles = smem;
  uint8_t* b_tile = smem + kStages * kStageBytes;
  uint32_t* ckey = reinterpret_cast<uint32_t*>(b_tile + kMaxN * kIdxRowBytes);
  uint32_t* cidx = ckey + kBufEntries;
  float* wbuf = reinterpret_cast<float*>(cidx + kBufEntries);
  uint32_t* hist = reinterpret_cast<uint32_t*>(wbuf + kMaxN);  // [2][3][256]; dense [2][4][256]; 32-head streaming [3][256]
  uint32_t* scratch = hist + kHistWords;                        // [2][16]; 32-head streaming [2][16]
  int32_t* cnt = reinterpret_cast<int32_t*>(scratch + 64);      // [2 tile parities][128 tokens]
  uint32_t* theta = reinterpret_cast<uint32_t*>(cnt + 256);     // [128]
  uint32_t* wsum = theta + 128;                                 // [2][2][4]
  uint32_t* wcnt = wsum + 16;                                   // [2 wg][2 parities][16 tokens][4 warps]
  uint64_t* bars = reinterpret_cast<uint64_t*>(wcnt + 256);
  // ring barriers of stages 0-3, accumulators, query tile, then the ring
  // barriers of the split-mode stages 4-11
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + kMaxAcc;
  uint64_t* b_full = acc_empty + kMaxAcc;
  uint64_t* b_empty = b_full + 1;
  uint64_t* ring_x = b_empty + 1;  // [2][kSplitStages - kStages]
  auto full_bar = [&](int st) { return st < kStages ? bars + st : ring_x + (st - kStages); };
  auto empty_bar = [&](int st) {
    return st < kStages ? bars + kStages + st : ring_x + (kSplitStages - kStages) + (st - kStages);
  };
  // query-tile barriers: buffer 0 as above, buffer 1 (split mode) after the ring
  uint64_t* qb_x = ring_x + 2 * (kSplitStages - kStages);  // [full, empty] of query buffer 1
  auto q_full = [&](int qb) { return qb == 0 ? b_full : qb_x; };
  auto q_empty = [&](int qb) { return qb == 0 ? b_empty : qb_x + 1; };
  uint64_t* wg_bar = qb_x + 2;  // TOK: wg_bar[0] is the epilogue warps' meeting barrier
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wg_bar + kTokBars);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {  // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, kStatusSetup);
    return;
  }
  const int N = HI * p.tq;
  // key-tile ring: stages 0-3 ahead of the query tile; split mode adds stages
  // 4-11 in the (unused) candidate-buffer space
  const int nst = SPLIT ? kSplitStages : kStages;
  auto stage_off = [](int st) -> uint32_t {
    return st < kStages ? static_cast<uint32_t>(st * kStageBytes)
                        : static_cast<uint32_t>(kStages * kStageBytes + kMaxN * kIdxRowBytes +
                                                (st - kStages) * kStageBytes);
  };
  static_assert((kSplitStages - kStages + 1) * kStageBytes <= 2 * kBufEntries * 4, "split stages and query tile fit");
  static_assert(kMaxN * kIdxRowBytes <= kStageBytes, "a query tile fits a stage slot");
  // query tile buffers: split mode alternates two (the next item's tile loads
  // while the current one is in use), group mode uses the first
  auto q_tile = [&](int qb) { return qb == 0 ? b_tile : smem + stage_off(kSplitStages); };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSplitStages; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      // one warpgroup per buffer; the score-array mode: every epilogue warp
      mbar_init(&acc_empty[i], STORE ? (kStoreThreads - 128) / 32 : (SPLIT || DENSE || TOK) ? 4 : kEpiThreads / 32);
    }
    for (int i = 0; i < kTokBars; ++i) mbar_init(&wg_bar[i], 8);
    for (int i = 0; i < 16; ++i) wcnt[i] = 0;  // TOK: per-row counters
    mbar_init(b_full, 1);
    mbar_init(b_empty, kIssuers);
    mbar_init(q_full(1), 1);
    mbar_init(q_empty(1), kIssuers);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  // split mode: prefix sums of the sequences' key-block counts (hist is unused there)
  const uint32_t* pref = nullptr;
  if constexpr (SPLIT) {
    if (p.n_seqs <= kMaxPrefixSeqs) {
      if (threadIdx.x == 0) {
        uint32_t acc = 0;
        for (int b = 0; b < p.n_seqs; ++b) {
          hist[b] = acc;
          const int L = split_len(p, b);
          acc += static_cast<uint32_t>(max(0, (L + kTileKeys - 1) / kTileKeys));
        }
        hist[p.n_seqs] = acc;
      }
      pref = hist;
    }
    if (threadIdx.x == 0)
      for (int b = 0; b < p.n_seqs; ++b)
        if (p.seq_lens[b] > p.score_stride) set_status(p.status, kStatusBounds);  // keys past the score row skipped
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort_v = abort_flag;

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    // Two producer warps take the key tiles in turn (tile counter parity);
    // the stage counts are even, so each stage's barriers belong to one
    // producer, which waits on their phases in order. Warp 0 also loads the
    // query tile of every item. In each warp every lane fetches one page id
    // of the warp's next 16 tiles (32 pages), so page-table latency is paid
    // once per 16 tiles, and lane 0 issues the copies.
    const int pw = warp == 0 ? 0 : 1;
    if (lane == 0) {
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_q);
    }
    uint32_t sc = 0, bi = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Item it;
      const int r = next_item(p, k, it, pref);
      if (r < 0) break;
      if (r == 0 || it.trivial) continue;
      if (pw == 0) {
        if (lane == 0) {
          const int qb = SPLIT ? static_cast<int>(bi & 1) : 0;
          const uint32_t use = SPLIT ? bi >> 1 : bi;  // earlier uses of this buffer
          ok = mbar_wait(q_empty(qb), (use & 1) ^ 1, abort_v, p.status);
          if (ok) {
            mbar_arrive_expect_tx(q_full(qb), N * kIdxRowBytes);
            tma_load_2d(q_tile(qb), &map_q, q_full(qb), 0, it.row0 * HI);
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        ++bi;
      }
      const int32_t* pt = p.page_tables + static_cast<size_t>(it.seq) * p.max_pages;
      const int nt = it.t1 - it.t0;
      const uint32_t sc0 = sc;
      for (int tw = (pw - static_cast<int>(sc0 & 1u) + 2) & 1; tw < nt && ok; tw += 32) {
        // lane l resolves page l & 1 of the tile streamed at step tw + 2 * (l / 2)
        int pg = 0;
        if (tw + 2 * (lane >> 1) < nt) {
          const int lp = 2 * tile_at(it, tw + 2 * (lane >> 1)) + (lane & 1);
          pg = lp * kPage < it.key_hi ? page_of(p, pt, lp) : 0;
        }
        const int tend = min(tw + 32, nt);
        for (int tt = tw; tt < tend; tt += 2) {
          const int pg0 = __shfl_sync(0xFFFFFFFFu, pg, tt - tw);
          const int pg1 = __shfl_sync(0xFFFFFFFFu, pg, tt - tw + 1);
          if (lane == 0) {
            const uint32_t g = sc0 + tt;
            const int t = tile_at(it, tt);
            const int s = g % nst;
            ok = mbar_wait(empty_bar(s), ((g / nst) & 1) ^ 1, abort_v, p.status);
            if (ok) {
              const bool has1 = (2 * t + 1) * kPage < it.key_hi;
              mbar_arrive_expect_tx(full_bar(s), has1 ? kStageBytes : kStageBytes / 2);
              tma_load_2d(a_tiles + stage_off(s), &map_k, full_bar(s), 0, pg0 * kPage);
              if (has1)
                tma_load_2d(a_tiles + stage_off(s) + kStageBytes / 2, &map_k, full_bar(s), 0, pg1 * kPage);
            }
          }
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
        }
      }
      sc = sc0 + nt;
    }
  } else if (warp >= 1 && warp <= kIssuers) {
    // ------------------------------------------------------------ MMA issuers
    // The tiles go round-robin (CTA tile counter modulo kIssuers) to the
    // issuer warps. One thread's chain of waits, MMAs and commits pays a long
    // issue latency per operation; several chains overlap it. All of a tile's
    // MMAs and commits come from one warp (a commit tracks its own thread's
    // MMAs), and every issuer releases the query tile once per item.
    // kIssuers divides the stage count and the accumulator count, so each
    // stage and accumulator barrier has a single issuer that waits on its
    // phases in order (a parity wait cannot tell phase n from phase n - 2).
    const int iw = warp - 1;
    const uint32_t idesc = p.is_bf16 ? instr_desc(128, N, kFmtBF16, kFmtBF16, false, false)
                                     : instr_desc(128, N, kFmtE4M3, kFmtE4M3, false, false);
    // Operands broadcast from lane 0 are warp-uniform to the compiler, which
    // can then keep the MMA descriptors in uniform registers instead of
    // re-checking per MMA that every lane holds the same value.
    uint32_t sc = 0, bi = 0;
    const uint32_t tmem_u = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    const uint32_t a_base = __shfl_sync(0xFFFFFFFFu, smem_u32(a_tiles), 0);
    const uint32_t q_base0 = __shfl_sync(0xFFFFFFFFu, smem_u32(q_tile(0)), 0);
    const uint32_t q_base1 = __shfl_sync(0xFFFFFFFFu, smem_u32(q_tile(1)), 0);
    for (int k = 0;; ++k) {
      Item it;
      const int r = next_item(p, k, it, pref);
      if (r < 0) break;
      if (r == 0 || it.trivial) continue;
      const int qb = SPLIT ? static_cast<int>(bi & 1) : 0;
      const uint32_t use = SPLIT ? bi >> 1 : bi;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(q_full(qb), use & 1, abort_v, p.status))) break;
      ++bi;
      const uint64_t b_desc0 = smem_desc(qb == 0 ? q_base0 : q_base1, 16, 1024);
      tc_fence_after();
      bool ok = true;
      const uint32_t sc0 = sc;
      const int nt = it.t1 - it.t0;
      for (int tt = (iw - static_cast<int>(sc0 % kIssuers) + kIssuers) % kIssuers; tt < nt; tt += kIssuers) {
        // CTA tile counter: stage ring and accumulator ring position
        const uint32_t g = __shfl_sync(0xFFFFFFFFu, sc0 + tt, 0);
        const int s = g % nst;
        const int buf = g & ((1u << p.acc_shift) - 1);
        // a free accumulator can take long (the epilogue is the slower side):
        // wait suspended so the spin does not take issue slots from the
        // epilogue warps on this SM sub-partition
        ok = mbar_wait_spin(full_bar(s), (g / nst) & 1, abort_v, p.status) &&
             mbar_wait(&acc_empty[buf], ((g >> p.acc_shift) & 1) ^ 1, abort_v, p.status);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = smem_desc(a_base + stage_off(s), 16, 1024);
        const uint32_t d = tmem_u + buf * N;
#pragma unroll
        for (int kk = 0; kk < kIdxRowBytes / 32; ++kk) {
          const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
          if (p.is_bf16) mma_f16_warp(d, ad + off, b_desc0 + off, idesc, kk > 0);
          else mma_f8_warp(d, ad + off, b_desc0 + off, idesc, kk > 0);
        }
        mma_commit_warp(empty_bar(s));
        mma_commit_warp(&acc_full[buf]);
      }
      if (!ok) break;
      sc = sc0 + nt;
      mma_commit_warp(q_empty(qb));
    }
  } else if (warp >= 4) {
    if constexpr (STORE) {
      // ---------------------------------------------------------- epilogue (32 heads, score array)
      // Sixteen epilogue warps: warpgroup r takes row r of every item (its 32
      // head weights in registers) and warp (r, q) the 32 keys of TMEM lane
      // quadrant q of every tile. A warp loads its row's 32 columns, releases
      // the accumulator (all sixteen warps release each one) and writes its 32
      // score keys to the row's score array: 128 contiguous bytes, nothing
      // shared between warps.
      const int ew = warp - 4;  // 0..15
      const int rr = ew >> 2;   // row of the item
      const int q = warp & 3;   // TMEM lane quadrant
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(rr * HI);
      uint32_t ac = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Item it;
        const int r = next_item(p, k, it, pref);
        if (r < 0) break;
        if (r == 0) continue;
        if (it.trivial) {
          // every key of the row is selected: 0..pos, then -1
          if (rr < it.nrows) {
            const int n = it.pos0 + rr + 1;
            int32_t* o = p.out_idx + static_cast<size_t>(it.row0 + rr) * p.topk;
            for (int e = (ew & 3) * 32 + lane; e < p.topk; e += 128) o[e] = e < n ? e : -1;
          }
          continue;
        }
        const bool active = rr < it.nrows;  // the last item of a sequence may have fewer rows
        float wr[HI];
#pragma unroll
        for (int h = 0; h < HI; ++h) wr[h] = active ? __ldg(p.w + static_cast<size_t>(it.row0 + rr) * HI + h) : 0.0f;
        uint32_t* out_row = p.scores + static_cast<int64_t>(it.srow + rr) * p.score_stride;
        const int pos = it.pos0 + rr;  // the row sees keys 0..pos
        const int32_t* pt = p.page_tables + static_cast<size_t>(it.seq) * p.max_pages;
        const uint32_t ac0 = ac;
        const int nt = it.t1 - it.t0;
        for (int tt = 0; tt < nt; ++tt) {
          const uint32_t gt = ac0 + tt;
          const int buf = gt & 3;
          if (__any_sync(0xFFFFFFFFu, !mbar_wait(&acc_full[buf], (gt >> 2) & 1u, abort_v, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t raw[32];
          tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(buf * kMaxN), raw);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
          if (!active) continue;
          const int t = tile_at(it, tt);
          const int s = t * kTileKeys + q * 32 + lane;
          float ks = 1.0f;
          if (p.k_scale && s <= pos) ks = __ldg(p.k_scale + page_of(p, pt, s / kPage) * kPage + (s % kPage));
          float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int h = 0; h < HI; h += 8) {
            fma2(a[0], a[1], wr[h + 0], wr[h + 1], fmaxf(__uint_as_float(raw[h + 0]), 0.0f),
                 fmaxf(__uint_as_float(raw[h + 1]), 0.0f));
            fma2(a[2], a[3], wr[h + 2], wr[h + 3], fmaxf(__uint_as_float(raw[h + 2]), 0.0f),
                 fmaxf(__uint_as_float(raw[h + 3]), 0.0f));
            fma2(a[4], a[5], wr[h + 4], wr[h + 5], fmaxf(__uint_as_float(raw[h + 4]), 0.0f),
                 fmaxf(__uint_as_float(raw[h + 5]), 0.0f));
            fma2(a[6], a[7], wr[h + 6], wr[h + 7], fmaxf(__uint_as_float(raw[h + 6]), 0.0f),
                 fmaxf(__uint_as_float(raw[h + 7]), 0.0f));
          }
          if (s <= pos)
            out_row[s] = score_key((((a[0] + a[4]) + (a[1] + a[5])) + ((a[2] + a[6]) + (a[3] + a[7]))) * ks);
        }
        ac = ac0 + nt;
      }
    } else if constexpr (TOK) {
      // ---------------------------------------------------------- epilogue (32 heads, streaming prefill)
      // The two warpgroups take the key tiles in turn (warpgroup g the tiles of
      // CTA tile-counter parity g: accumulator buffers 0 and 2 belong to
      // warpgroup 0, 1 and 3 to warpgroup 1), so the two halves of the
      // accumulator ring run independently. A warp loads the four rows' 32
      // columns of its TMEM lane quadrant (32 keys) at once, releases the
      // accumulator and computes the four rows' scores as independent chains.
      // A key whose score reaches its row's threshold is appended to the row's
      // candidate buffer (shared by the eight warps: one atomic per warp, row
      // and tile, no barrier per tile). A reservation that runs past the
      // buffer's end is kept in registers and requests a cut of that row; the
      // eight epilogue warps then meet on an mbarrier (each entering from
      // wherever it is: waiting for its next accumulator, or at the end of the
      // item), cut every requested buffer to a superset of its row's top-k,
      // raise those rows' thresholds and append the held entries. At the end of
      // an item a row with more than topk candidates goes to the workspace for
      // finish_kernel (or is selected here when there is no room), and every
      // row's index list ends in ascending index order.
      constexpr int kRows = 4;          // rows per item (N = 128 at 32 heads)
      constexpr int kE = 256;           // epilogue threads
      const int ew = warp - 4;          // 0..7
      const int wg = ew >> 2;
      const int q = warp & 3;           // TMEM lane quadrant
      const int tid_e = ew * 32 + lane;
      const int cap = p.cap;
      const int topk = p.topk;
      // [0..3] entries per row, [4..7] row thresholds, [8] cut requests (a bit
      // per row), [9] warps done with the tiles of their items
      uint32_t* stw = wcnt;
      volatile uint32_t* vst = stw;
      const uint32_t lanemask_lt = (1u << lane) - 1u;
      uint32_t bar_phase = 0;  // phases of the group barrier this warp has completed
      bool ok = true;
      uint32_t hold = 0;       // bit j: this lane keeps an entry of row j that did not fit
      uint32_t hkey[kRows] = {0, 0, 0, 0}, hidx[kRows] = {0, 0, 0, 0};
      uint32_t thr[kRows] = {0, 0, 0, 0};  // copies of the row thresholds (they change only in a cut)

      // The eight epilogue warps meet (bounded; false once the kernel gives up).
      auto meet = [&]() -> bool {
        __syncwarp();
        bool r = true;
        if (lane == 0) {
          mbar_arrive(&wg_bar[0]);
          r = mbar_wait_spin(&wg_bar[0], bar_phase & 1u, abort_v, p.status);
        }
        ++bar_phase;
        r = __shfl_sync(0xFFFFFFFFu, r, 0);
        __syncwarp();
        if (!r) ok = false;
        return r;
      };
      auto sync = [&]() { meet(); };
      // Keep the entries of row j's buffer [0, n) that pass `take`, in place and
      // in a fixed order (rounds of 2048 entries, 8 per thread). Returns the
      // count, or -1 when a meeting failed.
      auto compact = [&](uint32_t* kb, uint32_t* ib, int n, auto take) -> int {
        int base = 0;
        for (int r0 = 0, rnd = 0; r0 < n; r0 += 2048, ++rnd) {
          uint32_t kk[8], ii[8];
          uint32_t tmask = 0;
          int c = 0;
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const int e0 = r0 + 4 * tid_e + 1024 * v;
            uint4 kv = make_uint4(0, 0, 0, 0), iv = make_uint4(0, 0, 0, 0);
            if (e0 < n) {
              kv = *reinterpret_cast<const uint4*>(kb + e0);
              iv = *reinterpret_cast<const uint4*>(ib + e0);
            }
            kk[4 * v + 0] = kv.x; kk[4 * v + 1] = kv.y; kk[4 * v + 2] = kv.z; kk[4 * v + 3] = kv.w;
            ii[4 * v + 0] = iv.x; ii[4 * v + 1] = iv.y; ii[4 * v + 2] = iv.z; ii[4 * v + 3] = iv.w;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const bool t2 = e0 + u < n && take(kk[4 * v + u], ii[4 * v + u]);
              tmask |= (t2 ? 1u : 0u) << (4 * v + u);
              c += t2;
            }
          }
          int incl = c;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t2;
          }
          uint32_t* ws = scratch + 16 + 8 * (rnd & 1);
          if (lane == 31) ws[ew] = static_cast<uint32_t>(incl);
          if (!meet()) return -1;
          int off = base, total = 0;
#pragma unroll
          for (int w2 = 0; w2 < 8; ++w2) {
            const int v = static_cast<int>(ws[w2]);
            if (w2 < ew) off += v;
            total += v;
          }
          off += incl - c;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (!((tmask >> u) & 1u)) continue;
            if (off < cap) {
              kb[off] = kk[u];
              ib[off] = ii[u];
            }
            ++off;
          }
          base += total;
        }
        return base;
      };
      // Cut every requested row buffer to a superset of its row's top-k and raise
      // the row's threshold; then append the held entries. All eight warps call
      // it (each from wherever it noticed the request).
      auto cut = [&]() -> bool {
        if (!meet()) return false;  // every warp's reservations and writes are done
        const uint32_t mask = vst[8];
        for (int j = 0; j < kRows; ++j) {
          if (!((mask >> j) & 1u)) continue;
          uint32_t* kb = ckey + j * cap;
          uint32_t* ib = cidx + j * cap;
          const int n = min(static_cast<int>(vst[j]), cap);
          // 1. the range of the buffer's keys (the histogram is cleared meanwhile)
          uint32_t lo = 0xFFFFFFFFu, hi = 0;
          for (int e0 = 4 * tid_e; e0 < n; e0 += 4 * kE) {
            const uint4 kv = *reinterpret_cast<const uint4*>(kb + e0);
            const uint32_t v4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (e0 + u < n) {
                lo = min(lo, v4[u]);
                hi = max(hi, v4[u]);
              }
          }
          lo = __reduce_min_sync(0xFFFFFFFFu, lo);
          hi = __reduce_max_sync(0xFFFFFFFFu, hi);
          if (lane == 0) {
            scratch[ew] = lo;
            scratch[8 + ew] = hi;
          }
          hist[tid_e] = 0;
          if (!meet()) return false;
          lo = 0xFFFFFFFFu;
          hi = 0;
#pragma unroll
          for (int w2 = 0; w2 < 8; ++w2) {
            lo = min(lo, scratch[w2]);
            hi = max(hi, scratch[8 + w2]);
          }
          const uint32_t range = hi - lo;
          const int shift = range >= 256u ? (32 - __clz(range)) - 8 : 0;
          // 2. histogram of the keys over 256 bins of [lo, hi]
          for (int e0 = 4 * tid_e; e0 < n; e0 += 4 * kE) {
            const uint4 kv = *reinterpret_cast<const uint4*>(kb + e0);
            const uint32_t v4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (e0 + u < n && v4[u] >= lo && v4[u] <= hi) smem_inc(&hist[(v4[u] - lo) >> shift]);
          }
          if (!meet()) return false;
          // 3. every warp: the bin holding the topk-th best key and the entries
          //    from that bin up (lane l owns bins 255-8l down to 248-8l)
          uint32_t c8[8], sum = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            c8[i] = hist[255 - 8 * lane - i];
            sum += c8[i];
          }
          uint32_t incl = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t2;
          }
          const uint32_t excl = incl - sum;
          uint32_t mine = 0, kept = 0;
          if (excl < static_cast<uint32_t>(topk) && incl >= static_cast<uint32_t>(topk)) {
            uint32_t run = excl;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (run + c8[i] >= static_cast<uint32_t>(topk)) {
                mine = 0x80000000u | (255u - 8u * lane - i);
                kept = run + c8[i];
                break;
              }
              run += c8[i];
            }
          }
          const int src = __ffs(__ballot_sync(0xFFFFFFFFu, mine != 0)) - 1;
          uint32_t tk = 0, ti = 0xFFFFFFFFu;
          bool exact = false;
          if (src >= 0) {  // more than topk entries (always: a cut is requested when the buffer overflows)
            const uint32_t bin = __shfl_sync(0xFFFFFFFFu, mine, src) & 0xFFu;
            kept = __shfl_sync(0xFFFFFFFFu, kept, src);
            tk = lo + (bin << shift);
            // a bin too full (heavy ties) would free too little room: exact selection
            exact = static_cast<int>(kept) > cap - 512;
          }
          if (!meet()) return false;  // the histogram is read; the exact selection reuses it
          if (exact && n > topk) {
            dense_select<kE>(kb, ib, n, topk, tid_e, hist, scratch, sync, tk, ti);
            if (!ok) return false;
          }
          const uint32_t ctk = tk, cti = ti;
          const int m = exact ? compact(kb, ib, n, [&](uint32_t k2, uint32_t i2) { return selected(k2, i2, ctk, cti); })
                              : compact(kb, ib, n, [&](uint32_t k2, uint32_t) { return k2 >= ctk; });
          if (m < 0 || !meet()) return false;
          // later keys from the cut value up are admitted: keys arrive in no
          // particular order, so one equal to it may still win on its index
          if (tid_e == 0) {
            stw[j] = static_cast<uint32_t>(m);
            stw[4 + j] = tk;
          }
        }
        if (tid_e == 0) stw[8] = 0;
        if (!meet()) return false;
#pragma unroll
        for (int j = 0; j < kRows; ++j) thr[j] = vst[4 + j];
        // 4. the held entries (at most one per lane and row) that still qualify
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const bool re = ((hold >> j) & 1u) && hkey[j] >= thr[j];
          const uint32_t mm = __ballot_sync(0xFFFFFFFFu, re);
          if (mm) {
            uint32_t old = 0;
            if (lane == 0) old = atomicAdd(&stw[j], static_cast<uint32_t>(__popc(mm)));
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            const uint32_t pos = old + __popc(mm & lanemask_lt);
            if (re) {
              if (pos < static_cast<uint32_t>(cap)) {
                ckey[j * cap + pos] = hkey[j];
                cidx[j * cap + pos] = hidx[j];
              } else {
                set_status(p.status, kStatusTimeout);  // cannot happen: a cut frees >= 512 slots
              }
            }
          }
        }
        hold = 0;
        return meet();
      };
      // Ascending index order of the first m entries of a buffer (bitonic
      // network over the next power of two, padded with the largest index).
      auto sort_by_index = [&](uint32_t* kb, uint32_t* ib, int m) -> bool {
        int P = 1;
        while (P < m) P <<= 1;
        for (int e = m + tid_e; e < P; e += kE) {
          ib[e] = 0xFFFFFFFFu;
          kb[e] = 0;
        }
        if (!meet()) return false;
        for (int size = 2; size <= P; size <<= 1)
          for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid_e; i < P / 2; i += kE) {
              const int a = 2 * i - (i & (stride - 1));
              const int b = a + stride;
              const bool up = (a & size) == 0;
              const uint32_t ia = ib[a], ibb = ib[b];
              if ((ia > ibb) == up) {
                const uint32_t ka = kb[a];
                ib[a] = ibb;
                ib[b] = ia;
                kb[a] = kb[b];
                kb[b] = ka;
              }
            }
            if (!meet()) return false;
          }
        return true;
      };
      // Lane 0 polls until `ready()` or a cut request (served first: a warp
      // that holds an entry has requested one); bounded over the whole wait.
      auto wait_until = [&](auto ready) -> bool {
        const long long t0 = clock64();
        for (uint32_t itw = 0;; ++itw) {
          uint32_t st2 = 0;
          if (lane == 0) {
            st2 = ready() ? 1u : 0u;
            __threadfence_block();
            if (vst[8]) st2 = 2u;  // a request is served before the wait ends
            if (st2 != 1u && (itw & 15u) == 15u) {
              if (*abort_v) {
                st2 = 4u;
              } else if (clock64() - t0 > kWaitLimitCycles) {
                set_status(p.status, kStatusTimeout);
                *abort_v = 1;
                st2 = 4u;
              }
            }
          }
          st2 = __shfl_sync(0xFFFFFFFFu, st2, 0);
          if (st2 & 4u) {
            ok = false;
            return false;
          }
          if (st2 & 2u) {
            if (!cut()) return false;
            continue;
          }
          if (st2 & 1u) return true;
        }
      };

      uint32_t ac = 0, items_done = 0;
      for (int k = 0; ok; ++k) {
        Item it;
        const int r = next_item(p, k, it, pref);
        if (r < 0) break;
        if (r == 0) continue;
        if (it.trivial) {
          // every key of every row is selected: 0..pos, then -1
          for (int j = 0; j < it.nrows; ++j) {
            const int n = it.pos0 + j + 1;
            int32_t* o = p.out_idx + static_cast<size_t>(it.row0 + j) * topk;
            for (int e = tid_e; e < topk; e += kE) o[e] = e < n ? e : -1;
            if (p.defer && tid_e == 0) p.cand_cnt[it.row0 + j] = -1;
          }
          continue;
        }
        // the rows' head weights (read back as float4 broadcasts); the rows'
        // state starts empty (reset here, not at the end of the previous item:
        // every warp reads the final counts there before the last meeting)
        if (tid_e < kRows * HI) {
          const int j = tid_e / HI;
          wbuf[tid_e] = j < it.nrows ? __ldg(p.w + static_cast<size_t>(it.row0 + j) * HI + (tid_e % HI)) : 0.0f;
        }
        if (tid_e < 2 * kRows) stw[tid_e] = 0;
        if (!meet()) break;
#pragma unroll
        for (int j = 0; j < kRows; ++j) thr[j] = 0;
        const float4* wv4 = reinterpret_cast<const float4*>(wbuf);
        const int32_t* pt = p.page_tables + static_cast<size_t>(it.seq) * p.max_pages;
        const uint32_t ac0 = ac;
        const int nt = it.t1 - it.t0;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        for (int tt = (wg - static_cast<int>(ac0 & 1u) + 2) & 1; tt < nt && ok; tt += 2) {
          const uint32_t gt = ac0 + tt;
          const int buf = gt & 3;
          const uint32_t par = (gt >> 2) & 1u;
          if (!wait_until([&]() { return mbar_test_wait(&acc_full[buf], par); })) break;
          tc_fence_after();
          uint32_t raw[kRows][32];
#pragma unroll
          for (int j = 0; j < kRows; ++j)
            tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(buf * kMaxN + j * HI), raw[j]);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
          const int t = tile_at(it, tt);
          const int s = t * kTileKeys + q * 32 + lane;
          float ks = 1.0f;
          if (p.k_scale && s < it.key_hi) ks = __ldg(p.k_scale + page_of(p, pt, s / kPage) * kPage + (s % kPage));
          uint32_t key[kRows];
#pragma unroll
          for (int j = 0; j < kRows; ++j) {
            float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int h = 0; h < HI; h += 8) {
              const float4 wa = wv4[(j * HI + h) / 4], wb = wv4[(j * HI + h) / 4 + 1];
              fma2(a[0], a[1], wa.x, wa.y, fmaxf(__uint_as_float(raw[j][h + 0]), 0.0f),
                   fmaxf(__uint_as_float(raw[j][h + 1]), 0.0f));
              fma2(a[2], a[3], wa.z, wa.w, fmaxf(__uint_as_float(raw[j][h + 2]), 0.0f),
                   fmaxf(__uint_as_float(raw[j][h + 3]), 0.0f));
              fma2(a[4], a[5], wb.x, wb.y, fmaxf(__uint_as_float(raw[j][h + 4]), 0.0f),
                   fmaxf(__uint_as_float(raw[j][h + 5]), 0.0f));
              fma2(a[6], a[7], wb.z, wb.w, fmaxf(__uint_as_float(raw[j][h + 6]), 0.0f),
                   fmaxf(__uint_as_float(raw[j][h + 7]), 0.0f));
            }
            key[j] = score_key((((a[0] + a[4]) + (a[1] + a[5])) + ((a[2] + a[6]) + (a[3] + a[7]))) * ks);
          }
          // a warp that holds an entry requested a cut when it did not fit, and
          // serves it before appending again (its hold slot for that row is taken)
          if (__any_sync(0xFFFFFFFFu, hold != 0)) {
            if (!cut()) break;
          }
#pragma unroll
          for (int j = 0; j < kRows; ++j) {
            const bool adm = j < it.nrows && s < it.key_hi && s <= it.pos0 + j && key[j] >= thr[j];
            const uint32_t m = __ballot_sync(0xFFFFFFFFu, adm);
            if (!m) continue;
            uint32_t old = 0;
            if (lane == 0) old = atomicAdd(&stw[j], static_cast<uint32_t>(__popc(m)));
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            const uint32_t pos = old + __popc(m & lanemask_lt);
            if (adm) {
              if (pos < static_cast<uint32_t>(cap)) {
                ckey[j * cap + pos] = key[j];
                cidx[j * cap + pos] = static_cast<uint32_t>(s);
              } else {
                hold |= 1u << j;
                hkey[j] = key[j];
                hidx[j] = static_cast<uint32_t>(s);
              }
            }
            if (lane == 0 && old + __popc(m) > static_cast<uint32_t>(cap)) atomicOr(&stw[8], 1u << j);
          }
        }
        ac = ac0 + nt;
        if (!ok) break;
        // this warp is done with the item's tiles: wait for the other seven,
        // serving cut requests meanwhile. The count is read before the request:
        // a warp's request precedes its count (fenced), so a full count read
        // first cannot miss a request read after it.
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          atomicAdd(&stw[9], 1u);
        }
        ++items_done;
        if (!wait_until([&]() { return static_cast<int>(vst[9] - 8u * items_done) >= 0; })) break;
        if (!meet()) break;  // every append and cut of the item is done
        // the rows' results: to the workspace for finish_kernel, or selected here
        for (int j = 0; j < it.nrows; ++j) {
          uint32_t* kb = ckey + j * cap;
          uint32_t* ib = cidx + j * cap;
          const int n = min(static_cast<int>(vst[j]), cap);
          const int row = it.row0 + j;
          int32_t* o = p.out_idx + static_cast<size_t>(row) * topk;
          float* os = p.out_scores ? p.out_scores + static_cast<size_t>(row) * topk : nullptr;
          if (n > topk && p.defer) {
            uint4* dk = reinterpret_cast<uint4*>(p.cand_key + static_cast<size_t>(row) * cap);
            uint4* di = reinterpret_cast<uint4*>(p.cand_idx + static_cast<size_t>(row) * cap);
            for (int e = 4 * tid_e; e < n; e += 4 * kE) {
              dk[e >> 2] = *reinterpret_cast<const uint4*>(kb + e);
              di[e >> 2] = *reinterpret_cast<const uint4*>(ib + e);
            }
            if (tid_e == 0) p.cand_cnt[row] = n;
          } else {
            int m = n;
            if (n > topk) {
              uint32_t tk = 0, ti = 0xFFFFFFFFu;
              dense_select<kE>(kb, ib, n, topk, tid_e, hist, scratch, sync, tk, ti);
              if (!ok) break;
              m = compact(kb, ib, n, [&](uint32_t k2, uint32_t i2) { return selected(k2, i2, tk, ti); });
              if (m < 0 || !meet()) break;
            }
            if (!sort_by_index(kb, ib, m)) break;
            for (int e = tid_e; e < topk; e += kE) {
              o[e] = e < m ? static_cast<int32_t>(ib[e]) : -1;
              if (os) os[e] = e < m ? key_score(kb[e]) : 0.0f;
            }
            if (p.defer && tid_e == 0) p.cand_cnt[row] = -1;
          }
        }
        if (!ok || !meet()) break;  // the buffers are free for the next item
      }
    } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 4;
    const int wg = ew >> 2;
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int tid_wg = (ew & 3) * 32 + lane;
    const uint32_t bar_wg = 1 + wg;
    uint32_t* hist_wg = hist + 768 * wg;
    uint32_t* scr_wg = scratch + 16 * wg;
    uint32_t* wsum_wg = wsum + 8 * wg;
    auto wg_sync = [&]() { named_bar_sync(bar_wg, 128); };
    const int tpw = (p.tq + 1) / 2;
    const int j0 = wg * tpw, j1 = min(p.tq, j0 + tpw);
    const int cap = p.cap;
    const int topk = p.topk;
    const uint32_t lanemask_lt = (1u << lane) - 1u;
    uint32_t ac = 0;

    // Select the best `keep` of token j's buffer. If `to_output`, write the
    // selection to the output row (or the split-mode candidate slot); else
    // compact the buffer in place (stable) and raise the token's threshold.
    auto select_token = [&](int j, int n, int keep, bool to_output, const Item& it) -> int {
      uint32_t* kb = ckey + j * cap;
      uint32_t* ib = cidx + j * cap;
      if (to_output && p.defer && n > keep) {
        // hand the buffer to finish_kernel: copy it to the row's slot
        const int row = it.row0 + j;
        uint4* dk = reinterpret_cast<uint4*>(p.cand_key + static_cast<size_t>(row) * cap);
        uint4* di = reinterpret_cast<uint4*>(p.cand_idx + static_cast<size_t>(row) * cap);
        for (int e = 4 * tid_wg; e < n; e += 512) {
          dk[e >> 2] = *reinterpret_cast<const uint4*>(kb + e);
          di[e >> 2] = *reinterpret_cast<const uint4*>(ib + e);
        }
        if (tid_wg == 0) p.cand_cnt[row] = n;
        wg_sync();
        return n;
      }
      uint32_t tk = 0, ti = 0xFFFFFFFFu;
      const bool all = n <= keep;
      bool cut = false;  // mid-stream: keep key >= tk (a superset of the top-k)
      if (!all) {
        if (!to_output) {
          tk = wg_cut(kb, n, keep, tid_wg, hist_wg, scr_wg, wg_sync);
          // the cut bin may hold many ties; fall back to the exact selection
          // when the cut would not free a full tile of room
          uint32_t kept = 0;
          for (int e = tid_wg; e < n; e += 128) kept += kb[e] >= tk;
          kept = __reduce_add_sync(0xFFFFFFFFu, kept);
          if ((tid_wg & 31) == 0) scr_wg[12 + (tid_wg >> 5)] = kept;
          wg_sync();
          kept = scr_wg[12] + scr_wg[13] + scr_wg[14] + scr_wg[15];
          cut = static_cast<int>(kept) <= cap - 2 * kTileKeys;
          wg_sync();
        }
        if (!cut) wg_select(kb, ib, n, keep, tid_wg, hist_wg, scr_wg, wg_sync, tk, ti);
      }
      const int row = it.row0 + j;
      int base = 0;
      // rounds of 2048 entries: thread t owns e = r0 + 4t + 512v + q (v, q < 4);
      // every write lands below the round's end, after all of its reads
      for (int r0 = 0, rnd = 0; r0 < n; r0 += 2048, ++rnd) {
        uint32_t kk[16], ii[16];
        bool take[16];
        int c = 0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int e0 = r0 + 4 * tid_wg + 512 * v;
          uint4 kv = make_uint4(0, 0, 0, 0), iv = make_uint4(0, 0, 0, 0);
          if (e0 < n) {
            kv = *reinterpret_cast<const uint4*>(kb + e0);
            iv = *reinterpret_cast<const uint4*>(ib + e0);
          }
          kk[4 * v + 0] = kv.x; kk[4 * v + 1] = kv.y; kk[4 * v + 2] = kv.z; kk[4 * v + 3] = kv.w;
          ii[4 * v + 0] = iv.x; ii[4 * v + 1] = iv.y; ii[4 * v + 2] = iv.z; ii[4 * v + 3] = iv.w;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            take[4 * v + q4] = e0 + q4 < n && (all || (cut ? kk[4 * v + q4] >= tk
                                                            : selected(kk[4 * v + q4], ii[4 * v + q4], tk, ti)));
            c += take[4 * v + q4];
          }
        }
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += t2;
        }
        uint32_t* ws = wsum_wg + 4 * (rnd & 1);
        if (lane == 31) ws[ew & 3] = incl;
        wg_sync();
        int off = base, total = 0;
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) {
          const int v = static_cast<int>(ws[w2]);
          if (w2 < (ew & 3)) off += v;
          total += v;
        }
        off += incl - c;
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          if (!take[q4]) continue;
          if (!to_output) {
            kb[off] = kk[q4];
            ib[off] = ii[q4];
          } else {
            p.out_idx[static_cast<size_t>(row) * topk + off] = static_cast<int32_t>(ii[q4]);
            if (p.out_scores) p.out_scores[static_cast<size_t>(row) * topk + off] = key_score(kk[q4]);
          }
          ++off;
        }
        base += total;
      }
      if (to_output) {
        for (int e = base + tid_wg; e < topk; e += 128) {
          p.out_idx[static_cast<size_t>(row) * topk + e] = -1;
          if (p.out_scores) p.out_scores[static_cast<size_t>(row) * topk + e] = 0.0f;
        }
        if (p.defer && tid_wg == 0) p.cand_cnt[row] = -1;  // row complete
      }
      wg_sync();
      if (!to_output && tid_wg == 0) {
        // admit later keys from the cut (or the k-th key) up: keys stream in
        // a rotated order, so a later key equal to it may have a smaller
        // index and win the tie
        theta[j] = tk > 0 ? tk - 1 : 0;
      }
      wg_sync();
      return base;
    };

    // Dense mode: the exact top-k of token j from its full score array
    // (position = key index, keys 0..pos). Warp w of the warpgroup owns a
    // contiguous quarter of the row (a multiple of 512 entries).
    //  1. Each warp histograms its quarter into its own 256 bins of the score
    //     VALUE over the row's [min, max] (found while the tiles streamed):
    //     value bins spread a row far better than the float's top bits, so
    //     the shared-memory counters rarely collide.
    //  2. Every warp sums the four histograms and finds the bin b holding the
    //     k-th best, how many of it are needed (r) and each warp's count of
    //     entries above b.
    //  3. One pass (16 entries per lane and step, one scan of packed counts)
    //     writes each warp's entries above b at its offset, in a fixed order,
    //     and stages the warp's entries of b (key, index) in its quarter of
    //     the query tile's unused rows.
    //  4. The staged entries are ranked exactly (key descending, index
    //     ascending); the best r follow the others, in rank order.
    // A bin too full to stage (heavy ties) falls back to the range-adaptive
    // radix selection over the whole row and an ordered count-and-write. The
    // order of a row's indices is deterministic but not ascending.
    const int stage_cap = ((kMaxN - N) * kIdxRowBytes / 16) & ~15;  // staged (key, index) pairs per warpgroup
    uint32_t* stg = reinterpret_cast<uint32_t*>(b_tile + N * kIdxRowBytes) + wg * 2 * stage_cap;
    uint32_t* dsv = wcnt + 64 + 32 * wg;  // [0] staged, [1,2] threshold, [4..7] per-warp counts above b
    auto dense_token = [&](int j, const Item& it) {
      int n = it.pos0 + j + 1;
      if (n > cap) {  // a sequence longer than the host's bound: keys past the score slots are skipped
        if (tid_wg == 0) set_status(p.status, kStatusBounds);
        n = cap;
      }
      const uint32_t* kb = ckey + j * cap;
      const int row = it.row0 + j;
      int32_t* o = p.out_idx + static_cast<size_t>(row) * topk;
      float* os = p.out_scores ? p.out_scores + static_cast<size_t>(row) * topk : nullptr;
      if (n <= topk) {  // every key is kept
        for (int e = tid_wg; e < topk; e += 128) {
          o[e] = e < n ? e : -1;
          if (os) os[e] = e < n ? key_score(kb[e]) : 0.0f;
        }
        return;
      }
      const int w4 = tid_wg >> 5;
      const int cw = (n + 2047) / 2048 * 512;  // entries per warp
      const int b0 = w4 * cw, b1 = min(n, b0 + cw);
      uint32_t* dh = hist + 1024 * wg;          // [4 warps][256 bins]
      uint32_t* hw = dh + 256 * w4;
      const float vlo = key_score(wcnt[j]), vhi = key_score(wcnt[4 + j]);
      float vinv = vhi > vlo ? 256.0f / (vhi - vlo) : 0.0f;
      if (!(vinv <= 1.0e30f)) vinv = 0.0f;  // a degenerate range: one bin
      auto bin_of = [&](uint32_t key) -> int { return min(255, static_cast<int>((key_score(key) - vlo) * vinv)); };
#pragma unroll
      for (int i = 0; i < 8; ++i) hw[lane + 32 * i] = 0;
      if (tid_wg == 0) dsv[0] = 0;
      __syncwarp();
      for (int b = b0; b < b1; b += 512) {
        const bool full = b + 512 <= n;
        uint4 kv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) kv[u] = *reinterpret_cast<const uint4*>(kb + b + 128 * u + 4 * lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e0 = b + 128 * u + 4 * lane;
          const uint32_t k4[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            if (full || e0 + q4 < n) smem_inc(&hw[bin_of(k4[q4])]);
        }
      }
      wg_sync();
      // lane l owns bins 255-8l down to 248-8l: totals over the four warps
      uint32_t c[8], mine[8];
      {
        const uint4* h4 = reinterpret_cast<const uint4*>(dh + 248 - 8 * lane);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = 0;
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) {
          const uint4 lo4 = h4[64 * w2], hi4 = h4[64 * w2 + 1];  // bins 248-8l .. 255-8l of warp w2
          const uint32_t v8[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            c[i] += v8[i];
            if (w2 == w4) mine[i] = v8[i];
          }
        }
      }
      uint32_t sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += c[i];
      uint32_t incl = sum;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
        if (lane >= o2) incl += t2;
      }
      const uint32_t excl = incl - sum;
      uint32_t found = 0, r_in = 0, m_in = 0;
      if (excl < static_cast<uint32_t>(topk) && incl >= static_cast<uint32_t>(topk)) {
        uint32_t run = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (found == 0 && run + c[i] >= static_cast<uint32_t>(topk)) {
            found = 0x80000000u | static_cast<uint32_t>(255 - 8 * lane - i);
            r_in = static_cast<uint32_t>(topk) - run;
            m_in = c[i];
          }
          run += c[i];
        }
      }
      const int src = __ffs(__ballot_sync(0xFFFFFFFFu, found != 0)) - 1;
      const int bstar = static_cast<int>(__shfl_sync(0xFFFFFFFFu, found, src) & 0xFFu);
      const int r = static_cast<int>(__shfl_sync(0xFFFFFFFFu, r_in, src));
      const int m = static_cast<int>(__shfl_sync(0xFFFFFFFFu, m_in, src));
      // each warp's entries in the bin (staged in its own quarter of the room)
      const int wcap = stage_cap / 4;
      const uint32_t m0 = dh[bstar], m1 = dh[256 + bstar], m2 = dh[512 + bstar], m3 = dh[768 + bstar];
      if (max(max(m0, m1), max(m2, m3)) <= static_cast<uint32_t>(wcap)) {
        // this warp's entries above the bin, and the warps' before it
        uint32_t above = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (255 - 8 * lane - i > bstar) above += mine[i];
        above = __reduce_add_sync(0xFFFFFFFFu, above);
        if (lane == 0) dsv[4 + w4] = above;
        wg_sync();
        int base = 0;
        for (int w2 = 0; w2 < w4; ++w2) base += static_cast<int>(dsv[4 + w2]);
        const int n_above = static_cast<int>(dsv[4] + dsv[5] + dsv[6] + dsv[7]);
        uint32_t* sk = stg + w4 * wcap;              // this warp's staged keys
        uint32_t* si = stg + stage_cap + w4 * wcap;  // and their indices
        int sbase = 0;
        // 16 entries per lane and step (lane l: 4 consecutive entries in each
        // 128-entry quarter); one scan of the packed (above, in-bin) counts
        for (int b = b0; b < b1; b += 512) {
          const bool full = b + 512 <= n;
          uint4 kv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) kv[u] = *reinterpret_cast<const uint4*>(kb + b + 128 * u + 4 * lane);
          int bb[16];
          int cnt2 = 0;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t k4[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int e = b + 128 * u + 4 * lane + q4;
              bb[4 * u + q4] = (full || e < n) ? bin_of(k4[q4]) : -1;
              cnt2 += bb[4 * u + q4] > bstar ? 1 : (bb[4 * u + q4] == bstar ? 0x10000 : 0);
            }
          }
          int incl2 = cnt2;
#pragma unroll
          for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl2, o2);
            if (lane >= o2) incl2 += v;
          }
          const int ex = incl2 - cnt2;
          int off = base + (ex & 0xFFFF), soff = sbase + (ex >> 16);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t k4[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int e = b + 128 * u + 4 * lane + q4;
              if (bb[4 * u + q4] > bstar) {
                if (off < topk) {
                  o[off] = e;
                  if (os) os[off] = key_score(k4[q4]);
                }
                ++off;
              } else if (bb[4 * u + q4] == bstar) {
                if (soff < wcap) {
                  sk[soff] = k4[q4];
                  si[soff] = static_cast<uint32_t>(e);
                }
                ++soff;
              }
            }
          }
          const int tot = __shfl_sync(0xFFFFFFFFu, incl2, 31);
          base += tot & 0xFFFF;
          sbase += tot >> 16;
        }
        wg_sync();
        // the r best staged entries (key descending, index ascending) follow
        // the others, in that order
        const int mw[4] = {static_cast<int>(m0), static_cast<int>(m1), static_cast<int>(m2), static_cast<int>(m3)};
        for (int a = tid_wg; a < m; a += 128) {
          int wa = 0, ia = a;
#pragma unroll
          for (int w2 = 0; w2 < 3; ++w2)
            if (wa == w2 && ia >= mw[w2]) {
              ia -= mw[w2];
              wa = w2 + 1;
            }
          const uint32_t ka = stg[wa * wcap + ia], xa = stg[stage_cap + wa * wcap + ia];
          int rank = 0;
#pragma unroll
          for (int w2 = 0; w2 < 4; ++w2) {
            const uint32_t* fk = stg + w2 * wcap;
            const uint32_t* fi = stg + stage_cap + w2 * wcap;
            const int mf = mw[w2];
            int f = 0;
            for (; f + 4 <= mf; f += 4) {
              const uint4 k4 = *reinterpret_cast<const uint4*>(fk + f);
              const uint4 i4 = *reinterpret_cast<const uint4*>(fi + f);
              rank += (k4.x > ka || (k4.x == ka && i4.x < xa)) + (k4.y > ka || (k4.y == ka && i4.y < xa)) +
                      (k4.z > ka || (k4.z == ka && i4.z < xa)) + (k4.w > ka || (k4.w == ka && i4.w < xa));
            }
            for (; f < mf; ++f) rank += fk[f] > ka || (fk[f] == ka && fi[f] < xa);
          }
          if (rank < r && n_above + rank < topk) {
            o[n_above + rank] = static_cast<int32_t>(xa);
            if (os) os[n_above + rank] = key_score(ka);
          }
        }
      } else {
        uint32_t tk = 0, ti = 0xFFFFFFFFu;
        wg_sync();  // every warp has read the histograms
        dense_select<128>(kb, nullptr, n, topk, tid_wg, dh, scr_wg, wg_sync, tk, ti);
        int cnt_w = 0;
        for (int b = b0; b < b1; b += 128) {
          const int e0 = b + 4 * lane;
          const uint4 kv = *reinterpret_cast<const uint4*>(kb + e0);
          const uint32_t k4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            cnt_w += e0 + q4 < n && selected(k4[q4], static_cast<uint32_t>(e0 + q4), tk, ti);
        }
        cnt_w = __reduce_add_sync(0xFFFFFFFFu, cnt_w);
        if (lane == 0) dsv[4 + w4] = static_cast<uint32_t>(cnt_w);
        wg_sync();
        int base = 0;
        for (int w2 = 0; w2 < w4; ++w2) base += static_cast<int>(dsv[4 + w2]);
        for (int b = b0; b < b1; b += 128) {
          const int e0 = b + 4 * lane;
          const uint4 kv = *reinterpret_cast<const uint4*>(kb + e0);
          const uint32_t k4[4] = {kv.x, kv.y, kv.z, kv.w};
          bool t[4];
          int cl = 0;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            t[q4] = e0 + q4 < n && selected(k4[q4], static_cast<uint32_t>(e0 + q4), tk, ti);
            cl += t[q4];
          }
          int incl2 = cl;
#pragma unroll
          for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl2, o2);
            if (lane >= o2) incl2 += v;
          }
          int off = base + incl2 - cl;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            if (!t[q4]) continue;
            if (off < topk) {
              o[off] = e0 + q4;
              if (os) os[off] = key_score(k4[q4]);
            }
            ++off;
          }
          base += __shfl_sync(0xFFFFFFFFu, incl2, 31);
        }
      }
      wg_sync();  // histograms, counts and staging are reused by the next row
    };

    // A warp whose bounded wait gives up does not leave the item loop on its
    // own: the epilogue warps meet at named barriers, which have no time
    // limit. It carries on to its group's next barrier, where a vote tells
    // every warp of the group to leave together (the item's first barrier
    // for all epilogue warps, the per-tile barrier of a warpgroup in the
    // streaming mode).
    bool item_ok = true;
    for (int k = 0;; ++k) {
      Item it;
      const int r = next_item(p, k, it, pref);
      if (r < 0) break;
      if (r == 0) continue;
      if (named_bar_or(3, kEpiThreads, !item_ok)) break;
      for (int i = threadIdx.x - 128; i < N; i += kEpiThreads) {
        const int gi = it.row0 * HI + i;
        wbuf[i] = gi < p.n_rows * HI ? __ldg(p.w + gi) : 0.0f;
      }
      for (int j = threadIdx.x - 128; j < p.tq; j += kEpiThreads) {
        cnt[(ac & 1u) * 128 + j] = 0;
        theta[j] = 0;
        if constexpr (DENSE) {
          wcnt[j] = 0xFFFFFFFFu;  // the row's smallest and largest score key
          wcnt[4 + j] = 0;
        }
      }
      named_bar_sync(3, kEpiThreads);
      if (it.trivial) {
        // every key of every row is selected: write 0..pos, then -1
        for (int j = j0; j < j1 && j < it.nrows; ++j) {
          const int n = it.pos0 + j + 1;
          int32_t* o = p.out_idx + static_cast<size_t>(it.row0 + j) * topk;
          for (int e = tid_wg; e < topk; e += 128) o[e] = e < n ? e : -1;
          if (p.defer && tid_wg == 0) p.cand_cnt[it.row0 + j] = -1;  // row complete
        }
        continue;
      }
      const int32_t* pt = p.page_tables + static_cast<size_t>(it.seq) * p.max_pages;
      bool ok = true;
      if constexpr (SPLIT) {
        // decode: the two warpgroups take the tiles in turn (each accumulator
        // buffer belongs to one warpgroup) and each covers every query row of
        // its tile, TPW_MAX rows per pass; every score goes to the row's
        // score array, and select_sampled_kernel takes the exact top-k afterwards
        const uint32_t ac0 = ac;
        const int nt = it.t1 - it.t0;
        for (int tt = (wg - static_cast<int>(ac0 & 1u) + 2) & 1; tt < nt; tt += 2) {
          const uint32_t g = ac0 + tt;
          const int t = tile_at(it, tt);
          const int buf = g & ((1u << p.acc_shift) - 1);
          if (__any_sync(0xFFFFFFFFu, !mbar_wait_backoff(&acc_full[buf], (g >> p.acc_shift) & 1, abort_v, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int s = t * kTileKeys + q * 32 + lane;
          float ks = 1.0f;
          if (p.k_scale && s < it.key_hi) ks = __ldg(p.k_scale + page_of(p, pt, s / kPage) * kPage + (s % kPage));
          for (int jb = 0; jb < p.tq; jb += TPW_MAX) {
            uint32_t raw[TPW_MAX * HI];
#pragma unroll
            for (int jj = 0; jj < TPW_MAX; ++jj)
              if (jb + jj < p.tq)
                tmem_ld_heads<HI>(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * N + (jb + jj) * HI,
                                  raw + jj * HI);
            tmem_wait_ld();
            if (jb + TPW_MAX >= p.tq) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
#pragma unroll
            for (int jj = 0; jj < TPW_MAX; ++jj) {
              const int j = jb + jj;
              if (j < it.nrows && s < it.key_hi && s <= it.pos0 + j) {
                const float4* w4 = reinterpret_cast<const float4*>(wbuf + j * HI);
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
                for (int h = 0; h < HI; h += 4) {
                  const float4 wv = w4[h >> 2];
                  a0 = fmaf(wv.x, fmaxf(__uint_as_float(raw[jj * HI + h + 0]), 0.0f), a0);
                  a1 = fmaf(wv.y, fmaxf(__uint_as_float(raw[jj * HI + h + 1]), 0.0f), a1);
                  a2 = fmaf(wv.z, fmaxf(__uint_as_float(raw[jj * HI + h + 2]), 0.0f), a2);
                  a3 = fmaf(wv.w, fmaxf(__uint_as_float(raw[jj * HI + h + 3]), 0.0f), a3);
                }
                p.scores[static_cast<int64_t>(it.row0 + j) * p.score_stride + s] =
                    score_key(((a0 + a1) + (a2 + a3)) * ks);
              }
            }
          }
        }
        ac = ac0 + nt;
        item_ok = ok;  // a failure is voted on at the next item's first barrier
      } else if constexpr (DENSE) {
        // prefill, rows of at most `cap` keys: every score goes to the token's
        // array in shared memory at its key's position, so a tile needs no
        // coordination between warps; the two warpgroups take the tiles in
        // turn (each accumulator buffer belongs to one warpgroup), each
        // covering every row of its tile. Once the item's tiles are all in,
        // each warpgroup selects its rows' exact top-k.
        const uint32_t ac0 = ac;
        const int nt = it.t1 - it.t0;
        // each row's smallest and largest score key, kept per thread over the
        // item's tiles (rows jb + jj of a single pass) and merged at its end
        constexpr bool kOnePass = TPW_MAX >= 2;  // every row's scores in one pass of TPW_MAX rows
        uint32_t rmin[TPW_MAX], rmax[TPW_MAX];
#pragma unroll
        for (int jj = 0; jj < TPW_MAX; ++jj) {
          rmin[jj] = 0xFFFFFFFFu;
          rmax[jj] = 0;
        }
        for (int tt = (wg - static_cast<int>(ac0 & 1u) + 2) & 1; tt < nt; tt += 2) {
          const uint32_t g = ac0 + tt;
          const int t = tile_at(it, tt);
          const int buf = g & ((1u << p.acc_shift) - 1);
          if (__any_sync(0xFFFFFFFFu, !mbar_wait_backoff(&acc_full[buf], (g >> p.acc_shift) & 1, abort_v, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int s = t * kTileKeys + q * 32 + lane;
          float ks = 1.0f;
          if (p.k_scale && s < it.key_hi) ks = __ldg(p.k_scale + page_of(p, pt, s / kPage) * kPage + (s % kPage));
          if constexpr (kOnePass) {
            // one row's accumulator loads while the previous row is summed
            uint32_t raw[TPW_MAX * HI];
            const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * N;
            tmem_ld_heads<HI>(ta, raw);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < TPW_MAX; ++jj) {
              if (jj >= p.tq) break;
              const bool more = jj + 1 < TPW_MAX && jj + 1 < p.tq;
              if (more) tmem_ld_heads<HI>(ta + (jj + 1) * HI, raw + (jj + 1) * HI);
              if (jj < it.nrows && s < it.key_hi && s <= it.pos0 + jj && s < cap) {
                const float4* w4 = reinterpret_cast<const float4*>(wbuf + jj * HI);
                float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int h = 0; h < HI; h += 4) {
                  const float4 wv = w4[h >> 2];
                  const int o = (h >> 2) & 1 ? 4 : 0;
                  fma2(a[o + 0], a[o + 1], wv.x, wv.y, fmaxf(__uint_as_float(raw[jj * HI + h + 0]), 0.0f),
                       fmaxf(__uint_as_float(raw[jj * HI + h + 1]), 0.0f));
                  fma2(a[o + 2], a[o + 3], wv.z, wv.w, fmaxf(__uint_as_float(raw[jj * HI + h + 2]), 0.0f),
                       fmaxf(__uint_as_float(raw[jj * HI + h + 3]), 0.0f));
                }
                const uint32_t key =
                    score_key((((a[0] + a[4]) + (a[1] + a[5])) + ((a[2] + a[6]) + (a[3] + a[7]))) * ks);
                ckey[jj * cap + s] = key;
                rmin[jj] = min(rmin[jj], key);
                rmax[jj] = max(rmax[jj], key);
              }
              if (more) tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
          } else {
          for (int jb = 0; jb < p.tq; jb += TPW_MAX) {
            uint32_t raw[TPW_MAX * HI];
#pragma unroll
            for (int jj = 0; jj < TPW_MAX; ++jj)
              if (jb + jj < p.tq)
                tmem_ld_heads<HI>(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * N + (jb + jj) * HI,
                                  raw + jj * HI);
            tmem_wait_ld();
            if (jb + TPW_MAX >= p.tq) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
#pragma unroll
            for (int jj = 0; jj < TPW_MAX; ++jj) {
              const int j = jb + jj;
              if (j >= p.tq) break;
              uint32_t key = 0, kmin = 0xFFFFFFFFu, kmax = 0;
              if (j < it.nrows && s < it.key_hi && s <= it.pos0 + j && s < cap) {
                const float4* w4 = reinterpret_cast<const float4*>(wbuf + j * HI);
                float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int h = 0; h < HI; h += 4) {
                  const float4 wv = w4[h >> 2];
                  const int o = (h >> 2) & 1 ? 4 : 0;
                  a[o + 0] = fmaf(wv.x, fmaxf(__uint_as_float(raw[jj * HI + h + 0]), 0.0f), a[o + 0]);
                  a[o + 1] = fmaf(wv.y, fmaxf(__uint_as_float(raw[jj * HI + h + 1]), 0.0f), a[o + 1]);
                  a[o + 2] = fmaf(wv.z, fmaxf(__uint_as_float(raw[jj * HI + h + 2]), 0.0f), a[o + 2]);
                  a[o + 3] = fmaf(wv.w, fmaxf(__uint_as_float(raw[jj * HI + h + 3]), 0.0f), a[o + 3]);
                }
                key = score_key((((a[0] + a[4]) + (a[1] + a[5])) + ((a[2] + a[6]) + (a[3] + a[7]))) * ks);
                ckey[j * cap + s] = key;
                kmin = key;
                kmax = key;
              }
              kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
              kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
              if (lane == 0 && j < it.nrows) {
                atomicMin(&wcnt[j], kmin);
                atomicMax(&wcnt[4 + j], kmax);
              }
            }
          }
          }
        }
        if constexpr (kOnePass) {
#pragma unroll
          for (int jj = 0; jj < TPW_MAX; ++jj) {
            if (jj >= p.tq) break;
            const uint32_t kmin = __reduce_min_sync(0xFFFFFFFFu, rmin[jj]);
            const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, rmax[jj]);
            if (lane == 0 && jj < it.nrows) {
              atomicMin(&wcnt[jj], kmin);
              atomicMax(&wcnt[4 + jj], kmax);
            }
          }
        }
        ac = ac0 + nt;
        // every score of the item is in shared memory (or some warp gave up a wait)
        if (named_bar_or(3, kEpiThreads, !ok)) {
          item_ok = false;
          break;
        }
        for (int j = wg; j < it.nrows; j += 2) dense_token(j, it);
      } else {
        // prefill: both warpgroups take every tile, each for its own query rows
        for (int tt = 0; tt < it.t1 - it.t0; ++tt, ++ac) {
          const int t = tile_at(it, tt);
          const int buf = ac & ((1 << p.acc_shift) - 1);
          if (__any_sync(0xFFFFFFFFu, !mbar_wait_backoff(&acc_full[buf], (ac >> p.acc_shift) & 1, abort_v, p.status))) {
            ok = false;
            named_bar_or(bar_wg, 128, true);  // the warpgroup's vote of this tile
            break;
          }
          tc_fence_after();
          uint32_t raw[TPW_MAX * HI];
#pragma unroll
          for (int jj = 0; jj < TPW_MAX; ++jj)
            if (j0 + jj < j1)
              tmem_ld_heads<HI>(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * N + (j0 + jj) * HI,
                                raw + jj * HI);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);

          const int s = t * kTileKeys + q * 32 + lane;
          float ks = 1.0f;
          if (p.k_scale && s < it.key_hi) ks = __ldg(p.k_scale + page_of(p, pt, s / kPage) * kPage + (s % kPage));
          // ReLU + head-weighted sum with eight independent partial sums per
          // token (weights read as float4 broadcasts), then the admission test
          uint32_t key[TPW_MAX], m[TPW_MAX];
          bool adm[TPW_MAX];
#pragma unroll
          for (int jj = 0; jj < TPW_MAX; ++jj) {
            const int j = j0 + jj;
            adm[jj] = false;
            key[jj] = 0;
            if (j < j1) {
              const float4* w4 = reinterpret_cast<const float4*>(wbuf + j * HI);
              float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
              for (int h = 0; h < HI; h += 4) {
                const float4 wv = w4[h >> 2];
                const int o = (h >> 2) & 1 ? 4 : 0;
                a[o + 0] = fmaf(wv.x, fmaxf(__uint_as_float(raw[jj * HI + h + 0]), 0.0f), a[o + 0]);
                a[o + 1] = fmaf(wv.y, fmaxf(__uint_as_float(raw[jj * HI + h + 1]), 0.0f), a[o + 1]);
                a[o + 2] = fmaf(wv.z, fmaxf(__uint_as_float(raw[jj * HI + h + 2]), 0.0f), a[o + 2]);
                a[o + 3] = fmaf(wv.w, fmaxf(__uint_as_float(raw[jj * HI + h + 3]), 0.0f), a[o + 3]);
              }
              key[jj] = score_key((((a[0] + a[4]) + (a[1] + a[5])) + ((a[2] + a[6]) + (a[3] + a[7]))) * ks);
              const bool valid = j < it.nrows && s >= it.key_lo && s < it.key_hi && s <= it.pos0 + j;
              adm[jj] = valid && key[jj] > theta[j];
            }
            m[jj] = __ballot_sync(0xFFFFFFFFu, adm[jj]);
          }
          // The warps post their admitted counts and meet once: every warp
          // then knows each token's count before the tile (double-buffered by
          // tile parity, so the update below cannot race a slower warp's
          // read), the tile's total and its own offset, and all take the
          // same decision to compact a buffer the tile would overflow.
          const int par = static_cast<int>(ac & 1u);
          uint32_t* wc = wcnt + (wg * 2 + par) * 64;
          if (lane == 0) {
#pragma unroll
            for (int jj = 0; jj < TPW_MAX; ++jj) wc[jj * 4 + (ew & 3)] = static_cast<uint32_t>(__popc(m[jj]));
          }
          if (named_bar_or(bar_wg, 128, false)) {  // a warp of the warpgroup gave up its wait
            ok = false;
            break;
          }
#pragma unroll
          for (int jj = 0; jj < TPW_MAX; ++jj) {
            const int j = j0 + jj;
            if (j >= j1) continue;
            int pre = 0, tot = 0;
#pragma unroll
            for (int w2 = 0; w2 < 4; ++w2) {
              const int v = static_cast<int>(wc[jj * 4 + w2]);
              if (w2 < (ew & 3)) pre += v;
              tot += v;
            }
            int cb = cnt[par * 128 + j];
            if (cb + tot > cap) cb = select_token(j, cb, topk, false, it);
            if (adm[jj]) {
              const int pos = cb + pre + __popc(m[jj] & lanemask_lt);
              ckey[j * cap + pos] = key[jj];
              cidx[j * cap + pos] = static_cast<uint32_t>(s);
            }
            if (tid_wg == 0) cnt[(par ^ 1) * 128 + j] = cb + tot;
          }
        }
        item_ok = ok;  // a failure is voted on at the next item's first barrier
        if (ok) {
          wg_sync();
          for (int j = j0; j < j1 && j < it.nrows; ++j) select_token(j, cnt[(ac & 1u) * 128 + j], topk, true, it);
        }
      }
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, p.tmem_cols);
}

// ---------------------------------------------------------------------------
// Parameters of select_sampled_kernel (split and score-array modes, step 2). Score
// row i belongs to sequence i / block_rows, query row row_base + i % block_rows
// of that sequence.
struct SelectParams {
  const uint32_t* scores;
  int64_t score_stride;
  const int32_t* seq_lens;  // device, or null: one sequence of prefix_len + q_per_seq keys
  int32_t prefix_len;
  int32_t q_per_seq, topk;
  int32_t row_base, block_rows;
  int32_t* out_idx;
  float* out_scores;
};

// rows up to this many keys mark their selection in a bitmap (longer rows sort it)
constexpr int kSelBmBits = 1 << 18;

// ---------------------------------------------------------------------------
// Step 2 of the split and score-array modes: each row's exact top-k with one
// full read of the row.
//  1. a sample (32 to 96 runs of 128 keys spread over the row, more for longer
//     rows) gives a key t_lo that about e + 3 sqrt(e) of the sampled keys
//     reach, e being the number expected among the row's top k (one 4096-bin
//     histogram of the sample's key range);
//  2. one pass stages every key >= t_lo (and its position) in shared memory,
//     one atomic per warp and 1024 keys;
//  3. when between k and kSsCand keys were staged, they hold the row's top-k.
//     A 4096-bin histogram of the staged keys over [t_lo, the sample's largest
//     key] (larger keys in the top bin) gives the bin of the k-th staged key;
//     when that bin holds
//     at most 32 keys (nearly always: ~1.4 k keys over 4096 bins), one warp
//     ranks them by (key descending, position ascending) and the entry of the
//     needed rank is the threshold. Otherwise the k-th key follows from 12-bit
//     digits over the staged keys' range, and among keys equal to it the
//     lowest positions win (ranked by counting when few). When fewer than k or
//     more than kSsCand keys were staged (the sample misjudged the row) the
//     exact radix selection runs over the whole row in global memory;
//  4. the selected positions are marked in a bitmap of the row, gathered in
//     ascending order in shared memory and written out coalesced (rows longer
//     than the bitmap: the k positions are collected and sorted).
// 512 threads and ~96 KB of shared memory: two rows per SM at a time, so one
// row's pass over HBM overlaps the other's selection.
constexpr int kSsThreads = 512;
constexpr int kSsWarps = kSsThreads / 32;
constexpr int kSsCand = 6144;       // staged candidates
constexpr int kSsMinRuns = 32, kSsMaxRuns = 96;  // sampled runs of 128 keys
constexpr int kSsSampleMax = kSsMaxRuns * 128;   // held in the two candidate arrays
constexpr int kSsBins = 4096;       // 12-bit digits
constexpr int kSsPass = 8 * kSsThreads * 4;  // keys per iteration of the staging pass
constexpr int kSsPrefetchAhead = 2;          // iterations of the row prefetched into L2 ahead of the pass
static_assert(kSsSampleMax <= 2 * kSsCand, "the sample is held in the candidate space");

struct SsSmem {
  uint32_t bm[kSelBmBits / 32];  // selected positions of the row
  uint32_t cand_key[kSsCand], cand_idx[kSsCand];
  uint32_t hist[kSsBins];        // digit histogram; tie list; dense_select's 3 x 256 words
  uint32_t red[2 * kSsWarps];
  uint32_t wsum[kSsWarps];
  uint32_t lst_key[32], lst_idx[32];  // the staged keys of the k-th key's bin
  uint32_t n_cand, bin, above, thr_key, thr_idx, n_sel, n_lst;
};

// Block-wide minimum and maximum of v over all threads (every thread gets them).
// Also a barrier for what each thread wrote before it; S.red is read after
// it, so the next writer of S.red must follow another barrier.
__device__ __forceinline__ void ss_minmax(SsSmem& S, uint32_t& lo, uint32_t& hi, int tid) {
  const int lane = tid & 31, w = tid >> 5;
  lo = __reduce_min_sync(0xFFFFFFFFu, lo);
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
  if (lane == 0) {
    S.red[w] = lo;
    S.red[kSsWarps + w] = hi;
  }
  __syncthreads();
  lo = 0xFFFFFFFFu;
  hi = 0;
#pragma unroll
  for (int i = 0; i < kSsWarps; ++i) {
    lo = min(lo, S.red[i]);
    hi = max(hi, S.red[kSsWarps + i]);
  }
}

// The top-down scan of the counted histogram S.hist: the bin holding the r-th
// largest key and the number of keys in higher bins (S.bin, S.above).
__device__ __forceinline__ void ss_scan(SsSmem& S, uint32_t r, int tid) {
  const int lane = tid & 31, w = tid >> 5;
  constexpr int kPer = kSsBins / kSsThreads;  // bins per thread, from the top
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    c[i] = S.hist[kSsBins - 1 - (kPer * tid + i)];
    sum += c[i];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) S.wsum[w] = incl;
  __syncthreads();
  uint32_t run = incl - sum;
  for (int w2 = 0; w2 < w; ++w2) run += S.wsum[w2];
  if (run < r && run + sum >= r) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (run + c[i] >= r) {
        S.bin = static_cast<uint32_t>(kSsBins - 1 - (kPer * tid + i));
        S.above = run;
        break;
      }
      run += c[i];
    }
  }
  __syncthreads();
}

// Histogram of (key - lo) >> shift over kSsBins bins for the keys in [lo, hi]
// of keys[0, n) (shared memory), then ss_scan.
__device__ __forceinline__ void ss_digit(SsSmem& S, const uint32_t* keys, int n, uint32_t lo, uint32_t hi,
                                         int shift, uint32_t r, int tid) {
  for (int b = tid; b < kSsBins; b += kSsThreads) S.hist[b] = 0;
  __syncthreads();
  for (int e = tid; e < n; e += kSsThreads) {
    const uint32_t v = keys[e];
    if (v >= lo && v <= hi) atomicAdd(&S.hist[(v - lo) >> shift], 1u);
  }
  __syncthreads();
  ss_scan(S, r, tid);
}

__device__ __forceinline__ int ss_shift(uint32_t lo, uint32_t hi) {
  const uint32_t range = hi - lo;
  return range >= static_cast<uint32_t>(kSsBins) ? (32 - __clz(range)) - 12 : 0;
}

__global__ void __launch_bounds__(kSsThreads, 2) select_sampled_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint8_t ss_raw[];
  SsSmem& S = *reinterpret_cast<SsSmem*>(ss_raw);
  const int srow = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int seq = srow / p.block_rows;
  const int r_in = p.row_base + (srow - seq * p.block_rows);
  const int row = seq * p.q_per_seq + r_in;
  const int len = p.seq_lens ? p.seq_lens[seq] : p.prefix_len + p.q_per_seq;
  const int pos = len - p.q_per_seq + r_in;
  const int n = min(pos + 1, static_cast<int>(p.score_stride));  // keys 0..pos (with a score slot)
  const uint32_t* keys = p.scores + static_cast<int64_t>(srow) * p.score_stride;
  int32_t* o = p.out_idx + static_cast<size_t>(row) * p.topk;
  float* os = p.out_scores ? p.out_scores + static_cast<size_t>(row) * p.topk : nullptr;
  const int k = p.topk;
  if (n <= k) {
    for (int e = tid; e < k; e += kSsThreads) {
      o[e] = e < n ? e : -1;
      if (os) os[e] = e < n ? key_score(keys[e]) : 0.0f;
    }
    return;
  }
  auto sync = []() { __syncthreads(); };
  // the staging pass reads the whole row once: its next iterations are
  // prefetched into L2 ahead of it (one bulk prefetch per iteration), the first
  // ones while the sample is processed
  const uint32_t row_bytes = static_cast<uint32_t>(n) * 4u;
  auto prefetch_pass = [&](int it) {
    const uint32_t off = static_cast<uint32_t>(it) * kSsPass * 4u;
    if (tid == 0 && off < row_bytes) {
      const uint32_t len = min(static_cast<uint32_t>(kSsPass) * 4u, (row_bytes - off + 15u) & ~15u);
      prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(keys) + off, len);
    }
  };
  const bool use_bm = n <= kSelBmBits;  // else the selected positions are sorted in shared memory
  const int nw = (n + 31) / 32;
  // 1. a key that about 1.1 e + 3 sqrt(e) + 3 of the sampled keys reach; the
  //    sample's loads are issued first, the shared state is cleared while they
  //    are in flight
  const bool sampled = n > kSsCand;
  const int runs = min(kSsMaxRuns, max(kSsMinRuns, n / 2048));
  const int n_sample = runs * 128;
  constexpr int kSp = kSsSampleMax / 4 / kSsThreads;  // 16-byte sample loads per thread
  uint4 sv[kSp];
  if (sampled) {
#pragma unroll
    for (int j = 0; j < kSp; ++j) {
      const int e = tid + j * kSsThreads;
      if (e < n_sample / 4) {
        const int run = e >> 5, u = e & 31;
        const int start = static_cast<int>(static_cast<int64_t>(n - 128) * run / (runs - 1)) & ~3;
        sv[j] = *reinterpret_cast<const uint4*>(keys + start + 4 * u);
      }
    }
  }
  // the pass's first iterations, behind the sample's loads
#pragma unroll
  for (int it = 0; it < kSsPrefetchAhead; ++it) prefetch_pass(it);
  if (use_bm)
    for (int b = tid; b < ((nw + 3) & ~3); b += kSsThreads) S.bm[b] = 0;
  if (tid == 0) {
    S.n_cand = 0;
    S.n_sel = 0;
    S.n_lst = 0;
  }
  for (int b = tid; b < kSsBins; b += kSsThreads) S.hist[b] = 0;  // the sample's count
  uint32_t t_lo = 0;
  int h_shift = -1;  // >= 0: the staged keys are counted in bins of 2^h_shift from t_lo
  if (sampled) {
    uint32_t* sample = S.cand_key;  // cand_key and cand_idx, one after the other
    uint32_t lo = 0xFFFFFFFFu, hi = 0;
#pragma unroll
    for (int j = 0; j < kSp; ++j) {
      const int e = tid + j * kSsThreads;
      if (e < n_sample / 4) {
        const uint4 v = sv[j];
        *reinterpret_cast<uint4*>(&sample[4 * e]) = v;
        lo = min(min(lo, min(v.x, v.y)), min(v.z, v.w));
        hi = max(max(hi, max(v.x, v.y)), max(v.z, v.w));
      }
    }
    ss_minmax(S, lo, hi, tid);  // also orders the sample's stores and the cleared bins before the count
    const float expect = static_cast<float>(k) * static_cast<float>(n_sample) / static_cast<float>(n);
    const int r = static_cast<int>(ceilf(1.1f * expect + 3.0f * sqrtf(expect) + 3.0f));
    if (r < n_sample) {
      const int shift = ss_shift(lo, hi);
      for (int e = tid; e < n_sample; e += kSsThreads) atomicAdd(&S.hist[(sample[e] - lo) >> shift], 1u);
      __syncthreads();
      ss_scan(S, static_cast<uint32_t>(r), tid);
      t_lo = lo + (S.bin << shift);  // the r-th largest sampled key's bin, from its lower edge
      h_shift = ss_shift(t_lo, hi);
      // cleared for the staged keys' count (the scan read the bins before its last barrier)
      for (int b = tid; b < kSsBins; b += kSsThreads) S.hist[b] = 0;
    }
  }
  __syncthreads();  // the bitmap, bins and counts are cleared; the sample's space takes the candidates
  // 2. every key >= t_lo to the staging space. A lane takes 32 keys per
  //    iteration (eight 16-byte loads, each coalesced over the warp) and the
  //    warp appends its lanes' hits with one prefix sum and one shared atomic:
  //    about k / n of the keys pass, so nearly every 128-key segment holds one,
  //    and a per-segment append would set the pass's instruction count
  {
    constexpr int U = 8;
    constexpr int kStride = kSsThreads * 4;  // keys between a lane's loads
    static_assert(U * kStride == kSsPass, "one pass iteration");
    for (int b0 = 0, it = 0; b0 < n; b0 += kSsPass, ++it) {
      prefetch_pass(it + kSsPrefetchAhead);
      const int s0 = b0 + w * 128 + 4 * lane;  // load u covers keys s0 + u * kStride + 0..3
      const bool full = b0 + kSsPass <= n;
      uint4 kv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e0 = s0 + u * kStride;
        kv[u] = (full || e0 < n) ? *reinterpret_cast<const uint4*>(keys + e0) : make_uint4(0, 0, 0, 0);
      }
      uint32_t take = 0;  // bit 4u + q: key s0 + u * kStride + q passes
      static_assert(4 * U <= 32, "one bit per key of the iteration");
      if (full) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          take |= (kv[u].x >= t_lo ? 1u : 0u) << (4 * u);
          take |= (kv[u].y >= t_lo ? 2u : 0u) << (4 * u);
          take |= (kv[u].z >= t_lo ? 4u : 0u) << (4 * u);
          take |= (kv[u].w >= t_lo ? 8u : 0u) << (4 * u);
        }
      } else {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e0 = s0 + u * kStride;
          const uint32_t kk[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) take |= (e0 + q < n && kk[q] >= t_lo ? 1u : 0u) << (4 * u + q);
        }
      }
      if (!__any_sync(0xFFFFFFFFu, take != 0)) continue;
      const uint32_t c = __popc(take);
      uint32_t incl = c;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
        if (lane >= o2) incl += t2;
      }
      uint32_t base = 0;
      if (lane == 31) base = atomicAdd(&S.n_cand, incl);
      base = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - c;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        uint32_t t = (take >> (4 * u)) & 0xFu;
        while (t) {
          const int q = __ffs(t) - 1;
          t &= t - 1;
          const uint32_t key = q & 2 ? (q & 1 ? kv[u].w : kv[u].z) : (q & 1 ? kv[u].y : kv[u].x);
          if (base < static_cast<uint32_t>(kSsCand)) {
            S.cand_key[base] = key;
            S.cand_idx[base] = static_cast<uint32_t>(s0 + u * kStride + q);
          }
          ++base;
        }
      }
    }
  }
  __syncthreads();  // every thread's stores and appends precede what follows
  const int nc = static_cast<int>(S.n_cand);
  uint32_t tk = 0, ti = 0xFFFFFFFFu;
  bool exact_row = true;  // false: selected over the staged keys
  if (nc >= k && nc <= kSsCand) {
    exact_row = false;
    bool found = nc == k;  // all staged keys
    if (!found && h_shift >= 0) {
      // 3. the k-th staged key's bin: the staged keys counted in bins of
      //    2^h_shift from t_lo (larger keys than the sample's in the top bin)
      auto bin_of = [&](uint32_t key) { return min((key - t_lo) >> h_shift, static_cast<uint32_t>(kSsBins - 1)); };
      for (int e = tid; e < nc; e += kSsThreads) atomicAdd(&S.hist[bin_of(S.cand_key[e])], 1u);
      __syncthreads();
      ss_scan(S, static_cast<uint32_t>(k), tid);
      const uint32_t b = S.bin;
      const uint32_t r = static_cast<uint32_t>(k) - S.above;  // entries needed from bin b, 1..m
      const uint32_t m = S.hist[b];
      if (m <= 32u) {
        // the bin's m entries to a list; lane j of warp 0 ranks entry j by
        // (key descending, position ascending): rank r - 1 is the threshold
        for (int e = tid; e < nc; e += kSsThreads) {
          const uint32_t key = S.cand_key[e];
          if (bin_of(key) == b) {
            const uint32_t at = atomicAdd(&S.n_lst, 1u);
            if (at < 32u) {
              S.lst_key[at] = key;
              S.lst_idx[at] = S.cand_idx[e];
            }
          }
        }
        __syncthreads();
        if (w == 0 && static_cast<uint32_t>(lane) < m) {
          const uint32_t mk = S.lst_key[lane], mi = S.lst_idx[lane];
          uint32_t rank = 0;
          for (uint32_t j = 0; j < m; ++j) {
            const uint32_t kj = S.lst_key[j], ij = S.lst_idx[j];
            rank += (kj > mk || (kj == mk && ij < mi)) ? 1u : 0u;
          }
          if (rank == r - 1u) {
            S.thr_key = mk;
            S.thr_idx = mi;
          }
        }
        __syncthreads();
        tk = S.thr_key;
        ti = S.thr_idx;
        found = true;
      } else {
        __syncthreads();  // the bins are read before the digits below clear them
      }
    }
    if (!found) {
      // 3'. the k-th key: 12-bit digits over the staged keys' range
      uint32_t c_lo = t_lo, c_hi = 0;
      for (int e = tid; e < nc; e += kSsThreads) c_hi = max(c_hi, S.cand_key[e]);
      ss_minmax(S, c_lo, c_hi, tid);
      uint32_t lo = t_lo, hi = c_hi, r = static_cast<uint32_t>(k), m = 0;
      while (true) {
        const int shift = ss_shift(lo, hi);
        ss_digit(S, S.cand_key, nc, lo, hi, shift, r, tid);
        const uint32_t b = S.bin;
        r -= S.above;
        m = S.hist[b];
        const uint64_t nlo = static_cast<uint64_t>(lo) + (static_cast<uint64_t>(b) << shift);
        const uint64_t nhi = nlo + ((1ull << shift) - 1ull);
        lo = static_cast<uint32_t>(nlo);
        hi = static_cast<uint32_t>(nhi < hi ? nhi : hi);
        __syncthreads();  // S.bin, S.above and the histogram are read
        if (shift == 0) break;
      }
      tk = lo;
      if (r < m) {
        // m staged keys equal tk, the r lowest positions win
        if (m <= static_cast<uint32_t>(kSsBins) && m <= 1024u) {
          if (tid == 0) S.n_cand = 0;
          __syncthreads();
          for (int e = tid; e < nc; e += kSsThreads)
            if (S.cand_key[e] == tk) S.hist[atomicAdd(&S.n_cand, 1u)] = S.cand_idx[e];
          __syncthreads();
          for (int t = tid; t < static_cast<int>(m); t += kSsThreads) {
            const uint32_t mine = S.hist[t];
            uint32_t below = 0;
            for (uint32_t j = 0; j < m; ++j) below += S.hist[j] < mine;
            if (below == r - 1) S.thr_idx = mine;
          }
          __syncthreads();
          ti = S.thr_idx;
        } else {
          __syncthreads();  // S.red (read by ss_minmax) is rewritten by the selection
          dense_select<kSsThreads>(S.cand_key, S.cand_idx, nc, k, tid, S.hist, S.red, sync, tk, ti);
        }
      }
    }
    __syncthreads();  // the selection's scratch (S.hist) is free
    for (int e = tid; e < nc; e += kSsThreads) {
      const uint32_t i = S.cand_idx[e];
      if (!selected(S.cand_key[e], i, tk, ti)) continue;
      if (use_bm) {
        atomicOr(&S.bm[i >> 5], 1u << (i & 31));
      } else {
        const uint32_t at = atomicAdd(&S.n_sel, 1u);
        if (at < static_cast<uint32_t>(kSsBins)) S.hist[at] = i;
      }
    }
  }
  if (exact_row) {
    // 3''. the whole row from global memory; bitmap word = 8 lanes x 4 keys
    __syncthreads();  // S.red (read by ss_minmax) is rewritten by the selection
    dense_select<kSsThreads>(keys, nullptr, n, k, tid, S.hist, S.red, sync, tk, ti);
    __syncthreads();  // the selection's scratch (S.hist) is free
    for (int s0 = w * 128; s0 < n; s0 += kSsThreads * 4) {
      const int e0 = s0 + 4 * lane;
      const uint4 k4 = e0 < n ? *reinterpret_cast<const uint4*>(keys + e0) : make_uint4(0, 0, 0, 0);
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
      uint32_t take = 0;  // bit q: entry e0 + q is selected
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (e0 + q < n && selected(kk[q], static_cast<uint32_t>(e0 + q), tk, ti)) take |= 1u << q;
      if (use_bm) {
        uint32_t bits = take << (e0 & 31);  // bitmap word = 8 lanes x 4 keys
        bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
        bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 2);
        bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 4);
        if ((lane & 7) == 0 && e0 < n) S.bm[e0 >> 5] = bits;
      } else {
        const uint32_t c = __popc(take);
        uint32_t incl = c;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
          if (lane >= o2) incl += t2;
        }
        uint32_t base = 0;
        if (lane == 31 && incl) base = atomicAdd(&S.n_sel, incl);
        base = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - c;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if ((take >> q) & 1u) {
            if (base < static_cast<uint32_t>(kSsBins)) S.hist[base] = static_cast<uint32_t>(e0 + q);
            ++base;
          }
      }
    }
  }
  __syncthreads();
  if (!use_bm) {
    // 4'. ascending positions: bitonic sort of the k collected positions
    // (padded with the largest value to a power of two)
    const int m = min(static_cast<int>(S.n_sel), kSsBins);
    int P2 = 1;
    while (P2 < m) P2 <<= 1;
    for (int e = m + tid; e < P2; e += kSsThreads) S.hist[e] = 0xFFFFFFFFu;
    __syncthreads();
    for (int size = 2; size <= P2; size <<= 1)
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < P2 / 2; i += kSsThreads) {
          const int a = 2 * i - (i & (stride - 1));
          const int b2 = a + stride;
          const bool up = (a & size) == 0;
          const uint32_t va = S.hist[a], vb = S.hist[b2];
          if ((va > vb) == up) {
            S.hist[a] = vb;
            S.hist[b2] = va;
          }
        }
        __syncthreads();
      }
    for (int e = tid; e < k; e += kSsThreads) {
      o[e] = e < m ? static_cast<int32_t>(S.hist[e]) : -1;
      if (os) os[e] = e < m ? key_score(keys[S.hist[e]]) : 0.0f;
    }
    return;
  }
  // 4. ascending positions: thread t owns a run of bitmap words and places its
  //    positions in shared memory (the candidate space, free now), from where
  //    the row's k entries are written out coalesced
  //    (runs of 4 words or more are a multiple of 4 words, read 16 bytes at a
  //    time; the bitmap's words past nw are zero: cleared up to a multiple of 4)
  const int per1 = (nw + kSsThreads - 1) / kSsThreads;
  const bool vec = per1 >= 4;
  const int step = vec ? 4 : 1;
  const int per = vec ? (per1 + 3) & ~3 : per1;
  const int w0 = tid * per, w1 = min(vec ? (nw + 3) & ~3 : nw, w0 + per);
  auto words = [&](int i) {
    return vec ? *reinterpret_cast<const uint4*>(&S.bm[i]) : make_uint4(S.bm[i], 0u, 0u, 0u);
  };
  uint32_t cnt = 0;
  for (int i = w0; i < w1; i += step) {
    const uint4 b4 = words(i);
    cnt += __popc(b4.x) + __popc(b4.y) + __popc(b4.z) + __popc(b4.w);
  }
  uint32_t incl = cnt;
#pragma unroll
  for (int o2 = 1; o2 < 32; o2 <<= 1) {
    const uint32_t t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
    if (lane >= o2) incl += t2;
  }
  if (lane == 31) S.wsum[w] = incl;
  __syncthreads();
  uint32_t at = incl - cnt, total = 0;
#pragma unroll
  for (int w2 = 0; w2 < kSsWarps; ++w2) {
    const uint32_t v = S.wsum[w2];
    if (w2 < w) at += v;
    total += v;
  }
  uint32_t* out_pos = S.cand_key;
  static_assert(kSsCand >= 2048, "the candidate space holds the k <= 2048 positions");
  for (int i = w0; i < w1; i += step) {
    const uint4 b4 = words(i);
    const uint32_t wb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t bits = wb[j];
      while (bits) {
        const uint32_t e = static_cast<uint32_t>(i + j) * 32u + static_cast<uint32_t>(__ffs(bits) - 1);
        bits &= bits - 1;
        if (at < static_cast<uint32_t>(k)) out_pos[at] = e;
        ++at;
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < k; e += kSsThreads) {
    const bool has = static_cast<uint32_t>(e) < total;
    const uint32_t v = has ? out_pos[e] : 0u;
    o[e] = has ? static_cast<int32_t>(v) : -1;
    if (os) os[e] = has ? key_score(keys[v]) : 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Group mode, deferred rows: the exact top-k of one row's candidate buffer
// (copied out by the indexer when it held more than topk entries). One
// 128-thread CTA per row; the buffer is staged in shared memory and selected
// with the same exact radix selection the indexer uses in-kernel.
struct FinishParams {
  const uint32_t* cand_key;
  const uint32_t* cand_idx;
  const int32_t* cand_cnt;  // > 0: entries to select from; -1: row written by the indexer
  int32_t cap, topk;
  int32_t* out_idx;
  float* out_scores;
};

constexpr int kFinishThreads = 128;

size_t finish_smem_bytes(int cap) { return (2 * static_cast<size_t>(cap) + 768 + 16 + 4) * 4; }

__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const FinishParams p) {
  extern __shared__ __align__(16) uint32_t fsm[];
  uint32_t* keys = fsm;
  uint32_t* idxs = fsm + p.cap;
  uint32_t* hist = idxs + p.cap;  // 3 x 256
  uint32_t* red = hist + 768;     // 16
  uint32_t* wsum = red + 16;      // 4
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int n = p.cand_cnt[row];
  if (n <= 0) return;
  const uint4* sk = reinterpret_cast<const uint4*>(p.cand_key + static_cast<size_t>(row) * p.cap);
  const uint4* si = reinterpret_cast<const uint4*>(p.cand_idx + static_cast<size_t>(row) * p.cap);
  for (int e = 4 * tid; e < n; e += 4 * kFinishThreads) {
    *reinterpret_cast<uint4*>(keys + e) = __ldg(sk + (e >> 2));
    *reinterpret_cast<uint4*>(idxs + e) = __ldg(si + (e >> 2));
  }
  __syncthreads();
  auto sync = []() { __syncthreads(); };
  uint32_t tk = 0, ti = 0xFFFFFFFFu;
  const bool all = n <= p.topk;
  if (!all) wg_select(keys, idxs, n, p.topk, tid, hist, red, sync, tk, ti);
  int32_t* o = p.out_idx + static_cast<size_t>(row) * p.topk;
  float* os = p.out_scores ? p.out_scores + static_cast<size_t>(row) * p.topk : nullptr;
  const uint32_t lanemask_lt = (1u << lane) - 1u;
  // the selected entries to the front, in place (a round's reads all precede its writes)
  int base = 0;
  for (int e0 = 0; e0 < n; e0 += kFinishThreads) {
    const int e = e0 + tid;
    uint32_t kk = 0, ii = 0;
    bool take = false;
    if (e < n) {
      kk = keys[e];
      ii = idxs[e];
      take = all || selected(kk, ii, tk, ti);
    }
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, take);
    if (lane == 0) wsum[w] = __popc(m);
    __syncthreads();
    int off = base, tot = 0;
#pragma unroll
    for (int w2 = 0; w2 < kFinishThreads / 32; ++w2) {
      const int v = static_cast<int>(wsum[w2]);
      if (w2 < w) off += v;
      tot += v;
    }
    __syncthreads();
    if (take) {
      const int pos = off + __popc(m & lanemask_lt);
      keys[pos] = kk;
      idxs[pos] = ii;
    }
    base += tot;
  }
  // ascending index order (bitonic network over the next power of two, padded
  // with the largest index), so a row's list does not depend on the order in
  // which its candidates were gathered
  int P = 1;
  while (P < base) P <<= 1;
  for (int e = base + tid; e < P; e += kFinishThreads) {
    idxs[e] = 0xFFFFFFFFu;
    keys[e] = 0;
  }
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P / 2; i += kFinishThreads) {
        const int a = 2 * i - (i & (stride - 1));
        const int b = a + stride;
        const bool up = (a & size) == 0;
        const uint32_t ia = idxs[a], ib2 = idxs[b];
        if ((ia > ib2) == up) {
          const uint32_t ka = keys[a];
          idxs[a] = ib2;
          idxs[b] = ia;
          keys[a] = keys[b];
          keys[b] = ka;
        }
      }
      __syncthreads();
    }
  for (int e = tid; e < p.topk; e += kFinishThreads) {
    o[e] = e < base ? static_cast<int32_t>(idxs[e]) : -1;
    if (os) os[e] = e < base ? key_score(keys[e]) : 0.0f;
  }
}

bool set_select_attr() {
  static bool done = false;
  if (!done) {
    if (cudaFuncSetAttribute(select_sampled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(SsSmem))) != cudaSuccess)
      return false;
    done = true;
  }
  return true;
}

// step 2 of the split and score-array modes over n_rows score rows
int launch_select(const SelectParams& sp, int n_rows, cudaStream_t stream) {
  if (!set_select_attr()) return SMLA_ERR_CUDA;
  select_sampled_kernel<<<n_rows, kSsThreads, sizeof(SsSmem), stream>>>(sp);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

template <int HI, bool SPLIT, bool DENSE, bool TOK = false, bool STORE = false>
int launch_indexer_t(const IndexerLaunch& L, const IdxParams& prm) {
  CUtensorMap map_k, map_q;
  const CUtensorMapDataType dt = prm.is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t esz = prm.is_bf16 ? 2 : 1;
  const uint32_t inner = kIdxRowBytes / esz;
  const int N = HI * prm.tq;
  if (!encode_2d(&map_k, dt, L.cache->k_idx, inner, static_cast<uint64_t>(L.cache->num_pages) * kPage,
                 kIdxRowBytes, inner, kPage, CU_TENSOR_MAP_SWIZZLE_128B))
    return SMLA_ERR_CUDA;
  if (!encode_2d(&map_q, dt, L.q_idx, inner, static_cast<uint64_t>(prm.n_rows) * HI, kIdxRowBytes, inner, N,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return SMLA_ERR_CUDA;
  const size_t smem = kStages * kStageBytes + kMaxN * kIdxRowBytes + 2 * kBufEntries * 4 + kMaxN * 4 +
                      kHistWords * 4 + 64 * 4 + 256 * 4 + 128 * 4 + 16 * 4 + 256 * 4 +
                      (2 * kSplitStages + 2 * kMaxAcc + 4 + kTokBars) * 8 + 16;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(indexer_kernel<HI, SPLIT, DENSE, TOK, STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SMLA_ERR_CUDA;
    attr_done = true;
  }
  // split mode with the balanced tile ranges: up to one CTA per key tile
  const int64_t split_tiles = static_cast<int64_t>(prm.n_seqs) * ((prm.score_stride + kTileKeys - 1) / kTileKeys);
  const int grid_items = !prm.split ? (prm.n_items + 1) / 2
                         : prm.n_seqs <= kMaxPrefixSeqs ? static_cast<int>(std::min<int64_t>(split_tiles, 1 << 30))
                                                        : prm.n_items;
  const int grid = std::max(1, std::min(num_sms(), grid_items));
  indexer_kernel<HI, SPLIT, DENSE, TOK, STORE><<<grid, STORE ? kStoreThreads : kThreads, smem, L.stream>>>(map_k, map_q,
                                                                                                   prm);
  if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
  return SMLA_OK;
}

}  // namespace

bool indexer_split_mode(int32_t q_per_seq, int32_t h_idx) {
  // few query rows per sequence: split the keys so every SM streams some of them
  return q_per_seq * h_idx <= kMaxN && q_per_seq <= 8;
}

int indexer_tokens_per_cta(int32_t h_idx, int32_t topk, bool split, int32_t q_per_seq) {
  const int max_tq = kMaxN / h_idx;
  if (split) {
    int tq = 1;
    while (tq < q_per_seq) tq <<= 1;
    if (tq * h_idx < 16) tq = 16 / h_idx;
    return (tq <= max_tq && kBufEntries / tq - 2 * kTileKeys >= topk) ? tq : 0;
  }
  int tq = max_tq;
  while (tq > 1 && kBufEntries / tq - 2 * kTileKeys < topk) tq >>= 1;
  if (tq * h_idx < 16) return 0;
  return kBufEntries / tq - 2 * kTileKeys >= topk ? tq : 0;
}

int indexer_dense_tokens(int32_t h_idx, int32_t topk, int32_t max_seq_len) {
  // two query rows per work item (four at 4 heads, so the MMA has N >= 16):
  // each row's scores of keys 0..pos fill half of the candidate space
  const int tq = h_idx >= 8 ? 2 : 16 / h_idx;
  if (tq * h_idx > kMaxN) return 0;
  const int cap = 2 * kBufEntries / tq;
  return (max_seq_len <= cap && topk <= cap) ? tq : 0;
}

// Score-array mode: prefill rows at 32 indexer heads longer than the dense
// mode takes. The rows go in blocks (the same rows of every sequence) whose
// score array fits the space given, each a whole number of waves of work
// items over the SMs when it can be; the workspace size asks for blocks of up
// to kScoreArrayBudget bytes.
constexpr size_t kScoreArrayBudget = size_t(16) << 30;
constexpr int kMinStoreRows = 608;  // rows per block (per sequence) below which the streaming mode is used

bool indexer_store_mode(int32_t q_per_seq, int32_t h_idx, int32_t topk, int32_t max_seq_len) {
  return h_idx == 32 && !indexer_split_mode(q_per_seq, h_idx) && indexer_dense_tokens(h_idx, topk, max_seq_len) == 0;
}

int64_t store_stride(int32_t max_seq_len) { return (static_cast<int64_t>(max_seq_len) + 31) / 32 * 32; }

// rows per sequence of a block whose score array fits in `bytes` (a multiple of 4, at most q_per_seq)
int32_t store_block_rows(int32_t n_seqs, int32_t q_per_seq, int32_t max_seq_len, size_t bytes) {
  const size_t per_row = static_cast<size_t>(n_seqs) * static_cast<size_t>(store_stride(max_seq_len)) * 4;
  const size_t r = bytes / per_row / 4 * 4;
  return static_cast<int32_t>(std::min<size_t>(r, static_cast<size_t>(q_per_seq)));
}

size_t indexer_group_cand_bytes(int32_t n_rows, int32_t q_per_seq, int32_t h_idx, int32_t topk,
                                int32_t max_seq_len) {
  if (indexer_split_mode(q_per_seq, h_idx) || n_rows <= 0) return 0;
  if (indexer_dense_tokens(h_idx, topk, max_seq_len) > 0) return 0;  // dense mode keeps no candidate lists
  if (indexer_store_mode(q_per_seq, h_idx, topk, max_seq_len)) {
    const int32_t n_seqs = n_rows / q_per_seq;
    const int32_t rows = std::max(std::min(q_per_seq, kMinStoreRows),
                                  store_block_rows(n_seqs, q_per_seq, max_seq_len, kScoreArrayBudget));
    return static_cast<size_t>(n_seqs) * rows * static_cast<size_t>(store_stride(max_seq_len)) * 4;
  }
  const int tq = indexer_tokens_per_cta(h_idx, topk, false, q_per_seq);
  if (tq <= 0) return 0;
  const size_t cap = kBufEntries / tq;
  return static_cast<size_t>(n_rows) * cap * 8 + (static_cast<size_t>(n_rows) * 4 + 255) / 256 * 256;
}

size_t indexer_workspace_bytes(int32_t n_seqs, int32_t max_seq_len, int32_t q_per_seq, int32_t h_idx,
                               int32_t topk) {
  size_t bytes = kStatusBytes;
  if (indexer_split_mode(q_per_seq, h_idx)) {
    // one score key per (row, key): rows x max_seq_len rounded up to 4
    const size_t rows = static_cast<size_t>(n_seqs) * q_per_seq;
    bytes += rows * ((static_cast<size_t>(max_seq_len) + 3) / 4 * 4) * 4;
  }
  return bytes;
}

int launch_indexer(const IndexerLaunch& L) {
  const bool split = indexer_split_mode(L.q_per_seq, L.h_idx);
  const int dense_tq = split ? 0 : indexer_dense_tokens(L.h_idx, L.topk, L.max_seq_len);
  const bool dense = dense_tq > 0;
  const int tq = dense ? dense_tq : indexer_tokens_per_cta(L.h_idx, L.topk, split, L.q_per_seq);
  if (tq <= 0) return SMLA_ERR_UNSUPPORTED;
  IdxParams prm{};
  prm.k_scale = L.cache->k_idx_scale;
  prm.page_tables = L.page_tables;
  prm.max_pages = L.max_pages;
  prm.num_pages = L.cache->num_pages;
  prm.n_seqs = L.n_seqs;
  prm.q_per_seq = L.q_per_seq;
  prm.n_rows = L.n_seqs * L.q_per_seq;
  prm.seq_lens = L.seq_lens;
  prm.prefix_len = L.prefix_len;
  prm.w = L.w;
  prm.topk = L.topk;
  prm.tq = tq;
  prm.cap = (dense ? 2 * kBufEntries : kBufEntries) / tq;  // dense: score slots per row
  prm.is_bf16 = L.cache->idx_dtype == SMLA_BF16;
  prm.split = split;
  const int N = L.h_idx * tq;
  // as many accumulator buffers as fit in TMEM's 512 columns (at most 4)
  prm.acc_shift = 0;
  while (prm.acc_shift < 2 && (N << (prm.acc_shift + 1)) <= 512) ++prm.acc_shift;
  if ((1 << prm.acc_shift) % kIssuers != 0) return SMLA_ERR_UNSUPPORTED;  // N <= 128 always gives 4 buffers
  int cols = 32;
  while (cols < (N << prm.acc_shift)) cols <<= 1;
  prm.tmem_cols = cols;
  prm.out_idx = L.out_idx;
  prm.out_scores = L.out_scores;
  prm.row_base = 0;
  prm.block_rows = L.q_per_seq;
  uint8_t* ws = static_cast<uint8_t*>(L.workspace);
  prm.status = reinterpret_cast<uint32_t*>(ws);
  const size_t rows = static_cast<size_t>(prm.n_rows);
  if (split) {
    prm.n_kblocks = (L.max_seq_len + kKeyBlock - 1) / kKeyBlock;
    prm.n_items = L.n_seqs * prm.n_kblocks;
    prm.scores = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
    prm.score_stride = (static_cast<int64_t>(L.max_seq_len) + 3) / 4 * 4;
  } else {
    prm.n_groups = (L.q_per_seq + tq - 1) / tq;
    prm.n_items = L.n_seqs * prm.n_groups;
    // streaming prefill with 32 heads: the CTAs read the key tiles in nearly the
    // same order (start tiles spread over 8 tiles), so a key range larger than
    // L2 is read from HBM about once per wave of items instead of once per CTA
    if (!dense && L.h_idx == 32) prm.rot_span = 8;
    // score-array mode when the space given holds a large enough row block
    if (!dense && indexer_store_mode(L.q_per_seq, L.h_idx, L.topk, L.max_seq_len) && L.cand &&
        (reinterpret_cast<uintptr_t>(L.cand) & 15u) == 0) {
      int32_t block = store_block_rows(L.n_seqs, L.q_per_seq, L.max_seq_len, L.cand_bytes);
      if (block > 0 && block >= std::min(L.q_per_seq, kMinStoreRows)) {
        if (block < L.q_per_seq) {
          // several blocks: each a whole number of waves (two items of 4 rows
          // per SM) when that fits, else equal blocks of a multiple of 4 rows
          const int32_t wave = 8 * num_sms();
          if (block >= wave) {
            block = block / wave * wave;
          } else {
            const int32_t n_blocks = (L.q_per_seq + block - 1) / block;
            block = std::min(block, ((L.q_per_seq + n_blocks - 1) / n_blocks + 3) / 4 * 4);
          }
        }
        prm.scores = static_cast<uint32_t*>(L.cand);
        prm.score_stride = store_stride(L.max_seq_len);
        SelectParams sp{prm.scores, prm.score_stride, L.seq_lens, L.prefix_len, L.q_per_seq, L.topk,
                        0, 0, L.out_idx, L.out_scores};
        for (int32_t r0 = 0; r0 < L.q_per_seq; r0 += block) {
          prm.row_base = r0;
          prm.block_rows = std::min(block, L.q_per_seq - r0);
          prm.n_groups = (prm.block_rows + tq - 1) / tq;
          prm.n_items = L.n_seqs * prm.n_groups;
          const int rc = launch_indexer_t<32, false, false, false, true>(L, prm);
          if (rc != SMLA_OK) return rc;
          sp.row_base = r0;
          sp.block_rows = prm.block_rows;
          const int rs = launch_select(sp, L.n_seqs * prm.block_rows, L.stream);
          if (rs != SMLA_OK) return rs;
        }
        return SMLA_OK;
      }
    }
    const size_t cand = indexer_group_cand_bytes(prm.n_rows, L.q_per_seq, L.h_idx, L.topk, L.max_seq_len);
    if (L.cand && cand > 0 && L.cand_bytes >= cand && (reinterpret_cast<uintptr_t>(L.cand) & 15u) == 0) {
      prm.defer = 1;
      prm.cand_key = static_cast<uint32_t*>(L.cand);
      prm.cand_idx = prm.cand_key + rows * prm.cap;
      prm.cand_cnt = reinterpret_cast<int32_t*>(prm.cand_idx + rows * prm.cap);
    }
  }
  int rc;
  switch (L.h_idx) {
    case 4:
      rc = dense ? launch_indexer_t<4, false, true>(L, prm)
           : split ? launch_indexer_t<4, true, false>(L, prm) : launch_indexer_t<4, false, false>(L, prm);
      break;
    case 8:
      rc = dense ? launch_indexer_t<8, false, true>(L, prm)
           : split ? launch_indexer_t<8, true, false>(L, prm) : launch_indexer_t<8, false, false>(L, prm);
      break;
    case 16:
      rc = dense ? launch_indexer_t<16, false, true>(L, prm)
           : split ? launch_indexer_t<16, true, false>(L, prm) : launch_indexer_t<16, false, false>(L, prm);
      break;
    case 32:
      // the streaming prefill runs one epilogue warpgroup per token
      rc = dense ? launch_indexer_t<32, false, true>(L, prm)
           : split ? launch_indexer_t<32, true, false>(L, prm) : launch_indexer_t<32, false, false, true>(L, prm);
      break;
    case 64:
      rc = dense ? launch_indexer_t<64, false, true>(L, prm)
           : split ? launch_indexer_t<64, true, false>(L, prm) : launch_indexer_t<64, false, false>(L, prm);
      break;
    default: return SMLA_ERR_UNSUPPORTED;
  }
  if (rc != SMLA_OK) return rc;
  if (!split) {
    if (!prm.defer) return SMLA_OK;
    FinishParams fp{prm.cand_key, prm.cand_idx, prm.cand_cnt, prm.cap, L.topk, L.out_idx, L.out_scores};
    const size_t fsmem = finish_smem_bytes(prm.cap);
    static size_t attr_bytes = 0;
    if (fsmem > attr_bytes) {
      if (cudaFuncSetAttribute(finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(fsmem)) != cudaSuccess)
        return SMLA_ERR_CUDA;
      attr_bytes = fsmem;
    }
    finish_kernel<<<prm.n_rows, kFinishThreads, fsmem, L.stream>>>(fp);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
  }
  SelectParams sp{prm.scores, prm.score_stride, L.seq_lens, 0, L.q_per_seq, L.topk, 0, L.q_per_seq,
                  L.out_idx, L.out_scores};
  return launch_select(sp, prm.n_rows, L.stream);
}

}  // namespace smla
