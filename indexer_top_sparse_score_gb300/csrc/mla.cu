// Sparse MLA over selected latent rows (step 3 of the layer step).
//
// "Optimisations de GLM-5.3, partie 2", section "PCP" and footnote 1: each
// selected latent row (576 values) is read once and serves all query heads;
// QK uses all 576 values, PV the first 512. Per query row t:
//     l_j  = sm_scale * q[h,:] . K[s_j,:]          (s_j = selected keys)
//     out  = softmax_j(l) . K[s_j, 0:512],   lse = log sum_j exp(l_j)
//
// One CTA per SM (persistent); query rows are handed out in head/tail pairs
// (cheap causal rows with expensive ones). For each query row the selected
// rows stream through in blocks of 128, and every product is computed with
// the block's rows on the 128 TMEM lanes, so both MMAs run at M = 128:
//   S^T[128 rows x H]   = K_blk . Q^T            (K = 576)
//   O^T[512 x H]       += V_blk^T . P^T           (four M = 128 slices, K = 128)
// The block's rows live in one 144 KB shared tile of nine 64-value chunks,
// filled in five groups ({0,1} {2,3} {4,5} {6,7} {8}). PV slice d frees
// group d, so the next block's chunks load while PV is still running; the
// rope chunk (8) holds P^T once QK has read it.
//   warp 0      MMA issuer (one thread);
//   warps 4-11  softmax, one thread per selected row and half of the heads
//               (two warps per TMEM lane quadrant): logits of its heads for
//               its row, online softmax in the log2 domain against a per-head
//               reference max that is only raised (and O, l rescaled) when a
//               logit exceeds it by more than 2^8, P^T row to shared memory,
//               per-row partial sums of P in TMEM; at the end of a query row
//               the partial sums are reduced across rows and O^T is
//               normalised and written out;
//   warps 12-15 gather producers: key -> page -> pool row, row pieces into the
//               swizzled tile (cp.async from an f16 copy of the rows, or load +
//               widen bf16/e4m3 -> f16), per-row logit/probability scales; they
//               also widen the query to f16 once per query row.
// All MMA operands are f16: e4m3 -> f16 is exact and bf16 -> f16 is exact in
// the f16 normal range, and f16 gives the probabilities 11 significant bits
// (bf16 would give 8, which alone costs ~1e-3 relative output error). For
// FP8 caches the per-token scale multiplies the logit of its row and its
// probability before PV.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace smla {

namespace {

constexpr int kBlk = 128;                          // selected rows per block (MMA M)
constexpr int kChunks = kDqk / 64;                 // 9 chunks of 64 values
constexpr int kChunkBytes = kBlk * 128;            // 16 KB: 128 rows x 64 f16
constexpr int kStageBytes = kChunks * kChunkBytes;  // 144 KB
constexpr int kQChunkBytes = 64 * 128;             // 8 KB: up to 64 heads x 64 f16
constexpr int kQBytes = kChunks * kQChunkBytes;    // 72 KB
constexpr int kGroups = 5;                         // chunk groups {0,1} {2,3} {4,5} {6,7} {8}
constexpr int kPChunk = kChunks - 1;               // rope chunk, reused for P^T after QK
constexpr int kThreads = 512;
constexpr int kProducers = 128;                    // warps 12-15
constexpr uint32_t kColO = 0, kColS = 256, kColL = 320, kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
// latent cache formats: bf16 rows, e4m3 rows with one fp32 scale per token
// (separate array), 656-byte rows of e4m3 with four fp32 tile scales + bf16 rope
constexpr int kFmtBf16 = 0, kFmtTokenFp8 = 1, kFmtTileFp8 = 2;
constexpr int kTileRowBytes = 656, kTileScaleOff = 512, kTileRopeOff = 528;

struct MlaParams {
  const uint8_t* kv;
  const float* kv_scale;
  const int32_t* page_tables;
  int32_t max_pages, num_pages;
  int32_t n_seqs, q_per_seq, n_rows;
  const int32_t* seq_lens;
  int32_t prefix_len;
  const uint16_t* q;
  const int32_t* idx;
  int32_t topk;
  float scale_log2;  // sm_scale * log2(e)
  uint16_t* out;
  float* lse;
  int32_t fmt;  // latent cache format: kFmtBf16, kFmtTokenFp8 or kFmtTileFp8
  uint32_t* status;
  const uint16_t* shadow;  // f16 rows by logical position, or null
  const float* shadow_scale;  // per-token FP8 scales by logical position (FP8 cache with a shadow)
  int32_t shadow_rows;
  int32_t shadow_prefetch;  // the f16 copy is larger than half of L2: prefetch each next block's rows
  // split rows: each row's blocks are cut into n_parts items of part_blocks
  // blocks; each item writes a normalised fp32 partial output and its lse
  int32_t n_parts, part_blocks;
  float* part_o;    // [rows * n_parts][H][512]
  float* part_lse;  // [rows * n_parts][H]
};

struct SmemMeta {
  // per selected row of a block (two blocks in flight): {logit multiplier,
  // probability multiplier, valid, -}
  float4 row[2][kBlk];
  float m[64];        // reference max per head (log2 domain)
  float alpha[64];    // rescale factor per head
  float red[4][64];   // cross-warp reduction
  float linv[64];
  uint64_t q_full, q_empty, full[kGroups], empty[4], s_full, p_full, o_empty;
  uint64_t gather_meet;  // the four gather warps meet here once per query row
  uint32_t tmem_slot;
  int abort_flag;
};

constexpr size_t kSmemBytes = kQBytes + kStageBytes + sizeof(SmemMeta);
static_assert(kSmemBytes <= 232448, "shared memory budget");

// k-th work item of this CTA (a query row, or one part of a split row):
// head/tail pairs over the items. -1 done, 0 skip, 1 item.
__device__ __forceinline__ int next_row(int n_items, int k, int& item) {
  const int P = (n_items + 1) / 2;
  const int pair = blockIdx.x + (k >> 1) * gridDim.x;
  if (pair >= P) return -1;
  item = (k & 1) ? (n_items - 1 - pair) : pair;
  if ((k & 1) && item == pair) return 0;
  return 1;
}

struct RowInfo {
  int row, seq, pos, nvalid;
  int b0, nb;  // the item's blocks: b0 .. b0 + nb - 1 of the row's selection
};

__device__ __forceinline__ RowInfo row_info(const MlaParams& p, int item) {
  RowInfo r;
  r.row = item / p.n_parts;
  const int part = item - r.row * p.n_parts;
  r.seq = r.row / p.q_per_seq;
  const int j = r.row - r.seq * p.q_per_seq;
  const int L = p.seq_lens ? p.seq_lens[r.seq] : p.prefix_len + p.q_per_seq;
  r.pos = L - p.q_per_seq + j;
  r.nvalid = max(0, min(p.topk, r.pos + 1));
  const int nb_row = (r.nvalid + kBlk - 1) / kBlk;
  r.b0 = part * p.part_blocks;
  r.nb = max(0, min(nb_row - r.b0, p.part_blocks));
  return r;
}

// 2^x with the hardware approximation (relative error ~2^-22); 2^-inf = 0
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
// bf16 pair -> f16 pair (exact for values inside the f16 normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ bool bf16x2_over_f16(uint32_t w) {
  return ((w & 0x7FFFu) > 0x477Fu) || ((w & 0x7FFF0000u) > 0x477F0000u);
}
// 16-byte global load that bypasses L1 (each row is read once per block)
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  static_assert(NC == 8 || NC == 16 || NC == 32, "columns");
  if constexpr (NC == 8) tmem_ld_32x32b_x8(taddr, r);
  else if constexpr (NC == 16) tmem_ld_32x32b_x16(taddr, r);
  else tmem_ld_32x32b_x32(taddr, r);
}
template <int NC>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
  static_assert(NC == 8 || NC == 16 || NC == 32, "columns");
  if constexpr (NC == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
  } else if constexpr (NC == 16) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
  } else {
    tmem_st_32x32b_x32(taddr, r);
  }
}

// Warp reduce-scatter of NV values per lane (NV = 8, 16 or 32): afterwards
// lane L holds op over all lanes of value L / (32 / NV).
template <int NV, typename Op>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NV], int lane, Op op) {
  static_assert(NV == 8 || NV == 16 || NV == 32, "values per lane");
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int off = 16 >> s;
    const int n = NV >> s;  // values still held before this step
    if (n > 1) {
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < n / 2) {
          const float send = up ? v[i] : v[i + n / 2];
          const float keep = up ? v[i + n / 2] : v[i];
          v[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, off));
        }
      }
    } else {
      v[0] = op(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], off));
    }
  }
  return v[0];
}

struct MaxOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct AddOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

// Byte offset of 16-byte piece j of row r in a 128B-swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw_off(int r, int j) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

// TILE: 656-byte tile-scaled FP8 rows (a separate instance, so the bf16 and
// per-token FP8 gathers compile as without it)
template <int H, bool TILE>
__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const MlaParams p) {
  static_assert(H == 16 || H == 64, "heads");
  constexpr int kHalf = H < 32 ? H : 32;  // heads per softmax pass
  constexpr int kHalves = H / kHalf;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* q_tile = smem;
  uint8_t* stage = smem + kQBytes;
  SmemMeta& M = *reinterpret_cast<SmemMeta*>(smem + kQBytes + kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(p.status, kStatusSetup);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&M.q_full, 1);
    mbar_init(&M.q_empty, 1);
    for (int i = 0; i < kGroups; ++i) mbar_init(&M.full[i], kProducers);
    for (int i = 0; i < 4; ++i) mbar_init(&M.empty[i], 1);
    mbar_init(&M.s_full, 1);
    mbar_init(&M.p_full, 8);
    mbar_init(&M.o_empty, 8);
    mbar_init(&M.gather_meet, kProducers / 32);
    M.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&M.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = M.tmem_slot;
  volatile int* abort_v = &M.abort_flag;
  const uint32_t fmt = kFmtF16;  // every operand is widened to f16 (exact for e4m3 and in-range bf16)

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA
    // Per block: QK^T chunk group by chunk group as the groups arrive, then
    // (after the softmax) PV slice by slice, each slice's commit freeing the
    // chunks it read. The tensor pipe runs them in issue order. The whole warp
    // runs the loop with warp-uniform operands (broadcast from lane 0) and one
    // elected lane issues each MMA and commit.
    const uint32_t idesc_qk = instr_desc(128, H, fmt, fmt, false, false);
    const uint32_t idesc_pv = instr_desc(128, H, fmt, fmt, true, true);
    const uint32_t q0 = __shfl_sync(0xFFFFFFFFu, smem_u32(q_tile), 0);
    const uint32_t st0 = __shfl_sync(0xFFFFFFFFu, smem_u32(stage), 0);
    const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    // K-major operands (rows of 128 bytes, 8-row groups 1024 bytes apart):
    // the gathered rows (A of QK) and the query (B of QK). MN-major operands:
    // the same rows read as V^T (A of PV; the two 64-value chunks of a
    // 128-value slice are one chunk apart) and P^T (B of PV).
    const uint64_t k_desc = smem_desc(st0, 16, 1024);
    const uint64_t q_desc = smem_desc(q0, 16, 1024);
    const uint64_t vt_desc = smem_desc(st0, kChunkBytes, 1024);
    const uint64_t p_desc = smem_desc(st0 + kPChunk * kChunkBytes, kChunkBytes, 1024);
    uint32_t g = 0, tok = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int row;
      const int r = next_row(p.n_rows * p.n_parts, k, row);
      if (r < 0) break;
      if (r == 0) continue;
      const RowInfo ri = row_info(p, row);
      const int nb = __shfl_sync(0xFFFFFFFFu, ri.nb, 0);
      if (nb == 0) continue;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&M.q_full, tok & 1, abort_v, p.status))) break;
      for (int b = 0; b < nb; ++b, ++g) {
        const uint32_t ph = g & 1;
#pragma unroll 1
        for (int grp = 0; grp < kGroups; ++grp) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&M.full[grp], ph, abort_v, p.status))) { ok = false; break; }
          tc_fence_after();
          const int c1 = grp < 4 ? 2 * grp + 2 : kChunks;
#pragma unroll 1
          for (int c = 2 * grp; c < c1; ++c) {
            const uint64_t ka = k_desc + static_cast<uint64_t>((c * kChunkBytes) >> 4);
            const uint64_t qb = q_desc + static_cast<uint64_t>((c * kQChunkBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_warp(tm + kColS, ka + static_cast<uint64_t>(kk * 2), qb + static_cast<uint64_t>(kk * 2),
                           idesc_qk, (c | kk) != 0);
          }
        }
        if (!ok) break;
        mma_commit_warp(&M.s_full);
        if (b == nb - 1) mma_commit_warp(&M.q_empty);  // Q may be replaced once these finish
        const bool w_ok = mbar_wait(&M.p_full, ph, abort_v, p.status) &&
                          (b != 0 || mbar_wait(&M.o_empty, (tok & 1) ^ 1, abort_v, p.status));
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int dt = 0; dt < 4; ++dt) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_warp(tm + kColO + dt * 64,
                         vt_desc + static_cast<uint64_t>((dt * 2 * kChunkBytes + kk * 2048) >> 4),
                         p_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, (b | kk) != 0);
          mma_commit_warp(&M.empty[dt]);
        }
      }
      ++tok;
    }
  } else if (warp >= 12) {
    // ---------------------------------------------------------------- gather producers
    // Warp pw owns rows 32pw..32pw+31 of every block: lane l resolves the key
    // of row 32pw+l (keys two blocks ahead, page ids one block ahead), and a
    // chunk is copied in 8 passes of 4 rows x 8 pieces of 16 bytes, so every
    // warp instruction touches 4 full 128-byte lines.
    const int pw = warp - 12;
    const int tid = threadIdx.x - 384;
    const int psub = lane >> 3, pj = lane & 7;  // pass row offset, 16-byte piece
    const uint32_t st0 = smem_u32(stage);
    uint32_t g = 0, tok = 0, meet_phase = 0;
    bool ok = true;
    bool over = false;
    for (int k = 0; ok; ++k) {
      int row;
      const int r = next_row(p.n_rows * p.n_parts, k, row);
      if (r < 0) break;
      if (r == 0) continue;
      const RowInfo ri = row_info(p, row);
      if (ri.nb == 0) continue;
      row = ri.row;
      const int32_t* pt = p.page_tables + static_cast<size_t>(ri.seq) * p.max_pages;
      const int32_t* ir = p.idx + static_cast<size_t>(row) * p.topk;
      auto fetch_key = [&](int b) -> int {
        const int e = (ri.b0 + b) * kBlk + 32 * pw + lane;
        return (b < ri.nb && e < ri.nvalid) ? __ldg(ir + e) : -1;
      };
      auto fetch_page = [&](int key) -> int {
        if (p.shadow || key < 0 || key > ri.pos) return 0;
        const int lp = key >> 6;
        return lp < p.max_pages ? __ldg(pt + lp) : -1;
      };
      // pool (or shadow) row of a key, -1 when it is masked or out of range
      auto locate = [&](int key, int pg) -> int {
        if (key < 0 || key > ri.pos) return -1;
        if (p.shadow) return key < p.shadow_rows ? key : -1;
        if (pg < 0 || pg >= p.num_pages) {
          set_status(p.status, kStatusBounds);
          return -1;
        }
        return pg * kPage + (key & 63);
      };
      // the next item's query into L2 while this one runs (H * 1152 bytes,
      // split evenly over the gather threads)
      {
        int nrow;
        if (next_row(p.n_rows * p.n_parts, k + 1, nrow) > 0) {
          constexpr uint32_t kQSlice = H * kDqk * 2 / kProducers;
          const uint8_t* nq = reinterpret_cast<const uint8_t*>(p.q + static_cast<size_t>(nrow / p.n_parts) * H * kDqk);
          prefetch_l2_lines(nq + tid * kQSlice, kQSlice);
        }
      }
      // the BF16 query: its 16-byte pieces are copied asynchronously straight
      // into the swizzled Q tile, then each thread widens the pieces it copied
      // to f16 in place
      {
        const uint16_t* qr = p.q + static_cast<size_t>(row) * H * kDqk;
        constexpr int kQPieces = (H * 72 + kProducers - 1) / kProducers;
        if (!mbar_wait(&M.q_empty, (tok & 1) ^ 1, abort_v, p.status)) {
          ok = false;
          break;
        }
        const uint32_t q_u32 = smem_u32(q_tile);
#pragma unroll 4
        for (int u = 0; u < kQPieces; ++u) {
          const int pc = tid + u * kProducers;
          if (pc >= H * 72) break;
          const int h = pc / 72, pp = pc - h * 72;
          cp_async_16(q_u32 + (pp >> 3) * kQChunkBytes + sw_off(h, pp & 7), qr + h * kDqk + pp * 8, 16u);
        }
        cp_async_commit();
        cp_async_wait<0>();
#pragma unroll 4
        for (int u = 0; u < kQPieces; ++u) {
          const int pc = tid + u * kProducers;
          if (pc >= H * 72) break;
          const int h = pc / 72, pp = pc - h * 72;
          uint4* qp = reinterpret_cast<uint4*>(q_tile + (pp >> 3) * kQChunkBytes + sw_off(h, pp & 7));
          const uint4 v = *qp;
          const uint32_t in[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            over |= bf16x2_over_f16(in[t]);
            o[t] = bf16x2_to_f16x2(in[t]);
          }
          *qp = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        // the four gather warps meet (a bounded wait on an mbarrier rather than a
        // named barrier: a warp that gave up an earlier wait has left the loop,
        // and the others must be able to give up too instead of waiting for it)
        __syncwarp();
        bool met = true;
        if (lane == 0) {
          mbar_arrive(&M.gather_meet);
          met = mbar_wait_spin(&M.gather_meet, meet_phase & 1u, abort_v, p.status);
        }
        ++meet_phase;
        if (!__shfl_sync(0xFFFFFFFFu, met, 0)) {
          ok = false;
          break;
        }
        if (tid == 0) mbar_arrive(&M.q_full);
      }
      // keys three blocks ahead and page ids two ahead (each consumed a block
      // after it was requested); the rows of the next block (pool or f16
      // copy) are prefetched into L2 while this block is copied
      const int key0 = fetch_key(0);
      int key1 = fetch_key(1), key2 = fetch_key(2);
      int loc = locate(key0, fetch_page(key0));
      int pg1 = fetch_page(key1);
      const uint32_t row_bytes = TILE ? kTileRowBytes : p.fmt == kFmtTokenFp8 ? kDqk : 2 * kDqk;
      for (int b = 0; b < ri.nb && ok; ++b, ++g) {
        float ks = 1.0f;
        if (!TILE && p.fmt == kFmtTokenFp8 && loc >= 0) ks = __ldg((p.shadow ? p.shadow_scale : p.kv_scale) + loc);
        const int key3 = fetch_key(b + 3);
        const int loc1 = locate(key1, pg1);
        if (loc1 >= 0) {
          if (p.shadow) {
            if (p.shadow_prefetch) prefetch_l2_lines(p.shadow + static_cast<int64_t>(loc1) * kDqk, 2 * kDqk);
          } else {
            prefetch_l2_lines(p.kv + static_cast<int64_t>(loc1) * row_bytes, row_bytes);
          }
        }
        const int pg2 = fetch_page(key2);
        const uint32_t ph_e = (g & 1) ^ 1;  // slot of block g free: PV of block g-1 done
        auto meta = [&]() {
          M.row[g & 1][32 * pw + lane] =
              loc >= 0 ? make_float4(ks * p.scale_log2, ks, 1.0f, 0.0f) : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        if constexpr (TILE) {
          // 656-byte rows. Units 0-7: latent chunk u, lane l takes 16 bytes
          // (q = l & 3) of row 32pw + (l >> 2) + 8i in pass i (as the per-token
          // path) with the scale of the chunk's 128-value tile, and widens them
          // times that scale; units 8 and 9: the bf16 rope of rows 32pw + 16h +
          // (l >> 3) + 4i, lane piece l & 7 (as the bf16 path). Unit u+1 is in
          // flight while unit u is stored.
          const int rs8 = lane >> 2, q4 = lane & 3;
          int rl8[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) rl8[i] = __shfl_sync(0xFFFFFFFFu, loc, rs8 + 8 * i);
          uint4 stt[2][4];
          float scl[2][4];
          auto loadt = [&](int u, int slot) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = u < 8 ? rl8[i] : __shfl_sync(0xFFFFFFFFu, loc, 16 * (u - 8) + psub + 4 * i);
              const uint8_t* row = p.kv + static_cast<int64_t>(r < 0 ? 0 : r) * kTileRowBytes;
              stt[slot][i] = r < 0 ? make_uint4(0, 0, 0, 0) : ldg_stream(row + (u < 8 ? u * 64 + q4 * 16 : kTileRopeOff + pj * 16));
              if (u < 8) scl[slot][i] = r < 0 ? 0.0f : __ldg(reinterpret_cast<const float*>(row + kTileScaleOff) + (u >> 1));
            }
          };
          auto widen = [&](uint16_t v, float sc) -> uint32_t {
            const uint32_t hv = e4m3x2_to_f16x2(v);  // exact
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hv));
            const float a = f.x * sc, b = f.y * sc;
            over |= fabsf(a) > 65504.0f || fabsf(b) > 65504.0f;
            return pack_f16(a, b);
          };
          loadt(0, 0);
#pragma unroll
          for (int u = 0; u < 10; ++u) {
            const int c = u < 8 ? u : 8;
            const int grp = c < 8 ? c >> 1 : 4;
            if (u + 1 < 10) loadt(u + 1, (u + 1) & 1);
            if (((u < 8 && (u & 1) == 0) || u == 8) &&
                !mbar_wait(&M.empty[grp < 4 ? grp : 3], ph_e, abort_v, p.status)) {
              ok = false;
              break;
            }
            uint8_t* cp = stage + c * kChunkBytes;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 w = stt[u & 1][i];
              if (u < 8) {
                const float sc = scl[u & 1][i];
                const int rw = 32 * pw + rs8 + 8 * i;
                *reinterpret_cast<uint4*>(cp + sw_off(rw, 2 * q4)) =
                    make_uint4(widen(static_cast<uint16_t>(w.x & 0xFFFFu), sc), widen(static_cast<uint16_t>(w.x >> 16), sc),
                               widen(static_cast<uint16_t>(w.y & 0xFFFFu), sc), widen(static_cast<uint16_t>(w.y >> 16), sc));
                *reinterpret_cast<uint4*>(cp + sw_off(rw, 2 * q4 + 1)) =
                    make_uint4(widen(static_cast<uint16_t>(w.z & 0xFFFFu), sc), widen(static_cast<uint16_t>(w.z >> 16), sc),
                               widen(static_cast<uint16_t>(w.w & 0xFFFFu), sc), widen(static_cast<uint16_t>(w.w >> 16), sc));
              } else {
                over |= bf16x2_over_f16(w.x) | bf16x2_over_f16(w.y) | bf16x2_over_f16(w.z) | bf16x2_over_f16(w.w);
                *reinterpret_cast<uint4*>(cp + sw_off(32 * pw + 16 * (u - 8) + psub + 4 * i, pj)) =
                    make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
              }
            }
            if ((u < 8 && (u & 1) == 1) || u == 9) {
              if (u == 9) meta();
              fence_proxy_async_smem();
              mbar_arrive(&M.full[grp]);
            }
          }
        } else if (p.shadow) {
          int rl[8];  // pool rows of this lane's copy passes
#pragma unroll
          for (int i = 0; i < 8; ++i) rl[i] = __shfl_sync(0xFFFFFFFFu, loc, psub + 4 * i);
#pragma unroll
          for (int grp = 0; grp < kGroups; ++grp) {
            if (!mbar_wait(&M.empty[grp < 4 ? grp : 3], ph_e, abort_v, p.status)) { ok = false; break; }
#pragma unroll
            for (int c = 2 * grp; c < (grp < 4 ? 2 * grp + 2 : kChunks); ++c)
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int rw = 32 * pw + psub + 4 * i;
                cp_async_16(st0 + c * kChunkBytes + sw_off(rw, pj),
                            p.shadow + static_cast<int64_t>(rl[i] >= 0 ? rl[i] : 0) * kDqk + c * 64 + pj * 8,
                            rl[i] >= 0 ? 16u : 0u);
              }
            cp_async_commit();
            if (grp > 0) {
              cp_async_wait<1>();
              fence_proxy_async_smem();
              mbar_arrive(&M.full[grp - 1]);
            }
          }
          if (!ok) break;
          cp_async_wait<0>();
          meta();
          fence_proxy_async_smem();
          mbar_arrive(&M.full[kGroups - 1]);
        } else if (p.fmt == kFmtTokenFp8) {
          // e4m3 rows: one chunk (64 values = 64 bytes per row) per unit; lane l
          // takes 16 bytes (q = l & 3) of row 32pw + (l >> 2) + 8i in pass i and
          // widens them into f16 pieces 2q and 2q+1; units u+1 and u+2 are in
          // flight while unit u is stored
          const int rs8 = lane >> 2, q4 = lane & 3;
          int rl8[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) rl8[i] = __shfl_sync(0xFFFFFFFFu, loc, rs8 + 8 * i);
          uint4 st8[3][4];
          auto load8 = [&](int c, uint4* dst) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = rl8[i] < 0 ? make_uint4(0, 0, 0, 0)
                                  : ldg_stream(p.kv + static_cast<int64_t>(rl8[i]) * kDqk + c * 64 + q4 * 16);
          };
          load8(0, st8[0]);
          load8(1, st8[1]);
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            const int grp = c < 8 ? c >> 1 : 4;
            if (c + 2 < kChunks) load8(c + 2, st8[(c + 2) % 3]);
            if ((c & 1) == 0 && !mbar_wait(&M.empty[grp < 4 ? grp : 3], ph_e, abort_v, p.status)) {
              ok = false;
              break;
            }
            uint8_t* cp = stage + c * kChunkBytes;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 w = st8[c % 3][i];
              const int rw = 32 * pw + rs8 + 8 * i;
              *reinterpret_cast<uint4*>(cp + sw_off(rw, 2 * q4)) =
                  make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w.x & 0xFFFFu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w.x >> 16)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w.y & 0xFFFFu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w.y >> 16)));
              *reinterpret_cast<uint4*>(cp + sw_off(rw, 2 * q4 + 1)) =
                  make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w.z & 0xFFFFu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w.z >> 16)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w.w & 0xFFFFu)),
                             e4m3x2_to_f16x2(static_cast<uint16_t>(w.w >> 16)));
            }
            if ((c & 1) == 1 || c == kChunks - 1) {
              if (c == kChunks - 1) meta();
              fence_proxy_async_smem();
              mbar_arrive(&M.full[grp]);
            }
          }
        } else {
          // bf16 rows: load + widen in units of half a chunk (4 of the 8
          // passes); unit u+1 is loaded before unit u is stored
          int rl[8];  // pool rows of this lane's copy passes
#pragma unroll
          for (int i = 0; i < 8; ++i) rl[i] = __shfl_sync(0xFFFFFFFFu, loc, psub + 4 * i);
          constexpr int kUnits = 2 * kChunks;
          uint4 st[2][4];
          auto load = [&](int u, uint4* dst) {
            const int c = u >> 1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rw = rl[4 * (u & 1) + i];
              dst[i] = rw < 0 ? make_uint4(0, 0, 0, 0)
                              : ldg_stream(reinterpret_cast<const uint16_t*>(p.kv) + static_cast<int64_t>(rw) * kDqk +
                                           c * 64 + pj * 8);
            }
          };
          load(0, st[0]);
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            const int c = u >> 1;
            const int grp = c < 8 ? c >> 1 : 4;
            if (u + 1 < kUnits) load(u + 1, st[(u + 1) & 1]);
            if ((u & 3) == 0 && !mbar_wait(&M.empty[grp < 4 ? grp : 3], ph_e, abort_v, p.status)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 w = st[u & 1][i];
              over |= bf16x2_over_f16(w.x) | bf16x2_over_f16(w.y) | bf16x2_over_f16(w.z) | bf16x2_over_f16(w.w);
              *reinterpret_cast<uint4*>(stage + c * kChunkBytes + sw_off(32 * pw + psub + 4 * (4 * (u & 1) + i), pj)) =
                  make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
            }
            if ((u & 3) == 3 || u == kUnits - 1) {
              if (u == kUnits - 1) meta();
              fence_proxy_async_smem();
              mbar_arrive(&M.full[grp]);
            }
          }
        }
        loc = loc1;
        key1 = key2;
        key2 = key3;
        pg1 = pg2;
      }
      ++tok;
    }
    cp_async_wait<0>();
    if (over) set_status(p.status, kStatusOverflow);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    // Warps 4-7 take heads [0, H/2) and warps 8-11 heads [H/2, H) of the rows
    // on their TMEM lane quadrant.
    constexpr int HW = H / 2;
    const int qd = warp & 3;
    const int hq = (warp - 4) >> 2;
    const int h0 = hq * HW;
    const int tid = threadIdx.x - 128;  // 0..255
    const int rrow = qd * 32 + lane;     // selected row of the block = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t p_row = smem_u32(stage + kPChunk * kChunkBytes);
    uint32_t g = 0;
    for (int k = 0;; ++k) {
      int row;
      const int r = next_row(p.n_rows * p.n_parts, k, row);
      if (r < 0) break;
      if (r == 0) continue;
      const RowInfo ri = row_info(p, row);
      const int item = row;
      row = ri.row;
      uint16_t* orow = p.out + static_cast<size_t>(row) * H * kDv;
      if (ri.nb == 0) {
        if (p.n_parts > 1) {
          if (tid < H) p.part_lse[static_cast<size_t>(item) * H + tid] = -INFINITY;
        } else {
          for (int i = tid; i < H * kDv / 8; i += 256) reinterpret_cast<uint4*>(orow)[i] = make_uint4(0, 0, 0, 0);
          if (p.lse && tid < H) p.lse[static_cast<size_t>(row) * H + tid] = -INFINITY;
        }
        continue;
      }
      // A warp whose bounded wait gives up does not leave on its own: the eight
      // softmax warps meet at named barriers, so it carries on (touching no
      // accumulator) to the block's first barrier, which it makes take the
      // branch whose next barrier is a vote on `failed`; all eight leave there
      // together. The same vote ends a query row's epilogue.
      bool ok = true;
      for (int b = 0; b < ri.nb; ++b) {
        const uint32_t gb = g + b, ph = gb & 1;
        const bool failed = __any_sync(0xFFFFFFFFu, !mbar_wait(&M.s_full, ph, abort_v, p.status) ||
                                                        !mbar_wait(&M.full[kGroups - 1], ph, abort_v, p.status));
        tc_fence_after();
        const float4 mt = M.row[ph][rrow];
        const bool valid = !failed && mt.z != 0.0f;
        // (tcgen05.ld and its wait are warp-collective: every lane executes them,
        // `valid` only gates the arithmetic)
        uint32_t raw[HW];
        if (!failed) {
          tmem_ld_cols<HW>(tmem + lane_base + kColS + h0, raw);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < HW; ++i) raw[i] = 0;
        }
        // this thread's heads' reference maxima (16-byte broadcast loads)
        float mh[HW];
        auto load_m = [&]() {
#pragma unroll
          for (int i = 0; i < HW; i += 4) {
            const float4 v = *reinterpret_cast<const float4*>(&M.m[h0 + i]);
            mh[i] = v.x;
            mh[i + 1] = v.y;
            mh[i + 2] = v.z;
            mh[i + 3] = v.w;
          }
        };
        load_m();
        // does any logit exceed its head's reference max by more than 2^8?
        bool flag = b == 0 || failed;
        if (!flag && valid) {
          float tmax = -INFINITY;
#pragma unroll
          for (int i = 0; i < HW; ++i) tmax = fmaxf(tmax, fmaf(__uint_as_float(raw[i]), mt.x, -mh[i]));
          flag = tmax > kRescaleLog2;
        }
        if (named_bar_or(1, 256, flag)) {
          // exact per-head maximum of this block's logits
          {
            float x[HW];
#pragma unroll
            for (int i = 0; i < HW; ++i) x[i] = valid ? __uint_as_float(raw[i]) * mt.x : -INFINITY;
            const float mx = warp_reduce_scatter<HW>(x, lane, MaxOp());
            if ((lane & (32 / HW - 1)) == 0) M.red[qd][h0 + lane / (32 / HW)] = mx;
          }
          if (named_bar_or(1, 256, failed)) {  // some warp gave up a wait: all leave
            ok = false;
            break;
          }
          bool resc = false;
          if (tid < H) {
            const float bm = fmaxf(fmaxf(M.red[0][tid], M.red[1][tid]), fmaxf(M.red[2][tid], M.red[3][tid]));
            const float mu = b == 0 ? -INFINITY : M.m[tid];
            float a = 1.0f;
            if (bm > mu + kRescaleLog2 || (mu == -INFINITY && bm > -INFINITY)) {
              a = mu == -INFINITY ? 0.0f : fast_exp2(mu - bm);
              M.m[tid] = bm;
              resc = b > 0;
            } else if (b == 0) {
              M.m[tid] = -INFINITY;
            }
            M.alpha[tid] = a;
          }
          if (named_bar_or(1, 256, resc)) {
            // this thread's heads of O^T (its lane of every slice) and of its
            // row's partial sums; slot 4 is the partial sums
#pragma unroll 1
            for (int dt = 0; dt < 5; ++dt) {
              uint32_t o[HW];
              const uint32_t ta = tmem + lane_base + (dt < 4 ? kColO + dt * 64 : kColL) + h0;
              tmem_ld_cols<HW>(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < HW; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * M.alpha[h0 + i]);
              tmem_st_cols<HW>(ta, o);
            }
            tmem_wait_st();
          }
          load_m();  // the maxima may have been raised
        }
        // probabilities, partial sums, P^T row
        {
          uint32_t lp[HW];
          if (b > 0) {
            tmem_ld_cols<HW>(tmem + lane_base + kColL + h0, lp);
            tmem_wait_ld();
          }
          uint32_t pk[HW / 2];
#pragma unroll
          for (int i = 0; i < HW; i += 2) {
            float p0 = 0.0f, p1 = 0.0f;
            if (valid) {
              p0 = fast_exp2(fmaf(__uint_as_float(raw[i]), mt.x, -mh[i]));
              p1 = fast_exp2(fmaf(__uint_as_float(raw[i + 1]), mt.x, -mh[i + 1]));
            }
            lp[i] = __float_as_uint(b > 0 ? __uint_as_float(lp[i]) + p0 : p0);
            lp[i + 1] = __float_as_uint(b > 0 ? __uint_as_float(lp[i + 1]) + p1 : p1);
            pk[i >> 1] = pack_f16(p0 * mt.y, p1 * mt.y);
          }
          tmem_st_cols<HW>(tmem + lane_base + kColL + h0, lp);
#pragma unroll
          for (int u = 0; u < HW / 8; ++u)
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(p_row + sw_off(rrow, h0 / 8 + u)),
                         "r"(pk[4 * u]), "r"(pk[4 * u + 1]), "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                         : "memory");
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.p_full);
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      // the last PV of this query row has finished (a warp that gives up the
      // wait carries on to the vote below, as in the block loop)
      const bool failed = __any_sync(0xFFFFFFFFu, !mbar_wait(&M.empty[3], (g + ri.nb - 1) & 1, abort_v, p.status));
      tc_fence_after();
      {
        uint32_t raw[HW];
        if (!failed) {
          tmem_ld_cols<HW>(tmem + lane_base + kColL + h0, raw);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < HW; ++i) raw[i] = 0;
        }
        float x[HW];
#pragma unroll
        for (int i = 0; i < HW; ++i) x[i] = __uint_as_float(raw[i]);
        const float sm = warp_reduce_scatter<HW>(x, lane, AddOp());
        if ((lane & (32 / HW - 1)) == 0) M.red[qd][h0 + lane / (32 / HW)] = sm;
      }
      if (named_bar_or(1, 256, failed)) break;
      if (tid < H) {
        const float lt = (M.red[0][tid] + M.red[1][tid]) + (M.red[2][tid] + M.red[3][tid]);
        M.linv[tid] = lt > 0.0f ? 1.0f / lt : 0.0f;
        const float lse = lt > 0.0f ? (M.m[tid] + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
        if (p.n_parts > 1) p.part_lse[static_cast<size_t>(item) * H + tid] = lse;
        else if (p.lse) p.lse[static_cast<size_t>(row) * H + tid] = lse;
      }
      named_bar_sync(1, 256);
      const bool odd = lane & 1;
      float li[HW];  // this thread's heads' 1 / l
#pragma unroll
      for (int i = 0; i < HW; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(&M.linv[h0 + i]);
        li[i] = v.x;
        li[i + 1] = v.y;
        li[i + 2] = v.z;
        li[i + 3] = v.w;
      }
      if (p.n_parts > 1) {
        // normalised fp32 partial output of this part: [H][512]
        float* po = p.part_o + static_cast<size_t>(item) * H * kDv;
#pragma unroll 1
        for (int dt = 0; dt < 4; ++dt) {
          const int d = dt * 128 + qd * 32 + lane;
          uint32_t o[HW];
          tmem_ld_cols<HW>(tmem + lane_base + kColO + dt * 64 + h0, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < HW; ++c) po[static_cast<size_t>(h0 + c) * kDv + d] = __uint_as_float(o[c]) * li[c];
        }
      }
#pragma unroll 1
      for (int dt = 0; dt < (p.n_parts > 1 ? 0 : 4); ++dt) {
        const int d = dt * 128 + qd * 32 + lane;
        const int d_even = d & ~1;
        uint32_t o[HW];
        tmem_ld_cols<HW>(tmem + lane_base + kColO + dt * 64 + h0, o);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < HW; c += 2) {
          const float v0 = __uint_as_float(o[c]) * li[c];
          const float v1 = __uint_as_float(o[c + 1]) * li[c + 1];
          const float x2 = __shfl_xor_sync(0xFFFFFFFFu, odd ? v0 : v1, 1);
          const uint32_t word = odd ? pack_bf16(x2, v1) : pack_bf16(v0, x2);
          const int hh = h0 + (odd ? c + 1 : c);
          *reinterpret_cast<uint32_t*>(orow + static_cast<size_t>(hh) * kDv + d_even) = word;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.o_empty);
      g += ri.nb;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

// Merge of split rows: out = sum_s w_s * o_s with w_s = exp(lse_s - lse) and
// lse = log sum_s exp(lse_s) (the partial attentions of disjoint key sets,
// each normalised over its own keys). One CTA per (row, group of 8 heads);
// each thread combines 4 consecutive values of one head with 16-byte loads.
constexpr int kMergeHeads = 8;

__global__ void __launch_bounds__(256) part_merge_kernel(const float* __restrict__ part_o,
                                                         const float* __restrict__ part_lse, int n_parts,
                                                         int n_heads, uint16_t* __restrict__ out, float* lse) {
  __shared__ float wgt[kMaxParts][kMergeHeads];
  const int row = blockIdx.x, h0 = blockIdx.y * kMergeHeads, tid = threadIdx.x;
  const size_t item0 = static_cast<size_t>(row) * n_parts;
  if (tid < kMergeHeads && h0 + tid < n_heads) {
    const int h = h0 + tid;
    float m = -INFINITY;
    for (int s = 0; s < n_parts; ++s) m = fmaxf(m, part_lse[(item0 + s) * n_heads + h]);
    float sum = 0.0f;
    float e[kMaxParts];
    for (int s = 0; s < n_parts; ++s) {
      const float l = part_lse[(item0 + s) * n_heads + h];
      e[s] = (m == -INFINITY || l == -INFINITY) ? 0.0f : __expf(l - m);
      sum += e[s];
    }
    for (int s = 0; s < n_parts; ++s) wgt[s][tid] = sum > 0.0f ? e[s] / sum : 0.0f;
    if (lse) lse[static_cast<size_t>(row) * n_heads + h] = sum > 0.0f ? m + __logf(sum) : -INFINITY;
  }
  __syncthreads();
  // 8 heads x 512 values = 1024 float4 per CTA: 4 per thread
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = tid + u * 256;
    const int hl = i >> 7, d = (i & 127) * 4;
    const int h = h0 + hl;
    if (h >= n_heads) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_parts; ++s) {
      const float ws = wgt[s][hl];
      if (ws == 0.0f) continue;  // empty part: its output was never written
      const float4 o = __ldg(reinterpret_cast<const float4*>(part_o + ((item0 + s) * n_heads + h) * kDv + d));
      acc.x = fmaf(ws, o.x, acc.x);
      acc.y = fmaf(ws, o.y, acc.y);
      acc.z = fmaf(ws, o.z, acc.z);
      acc.w = fmaf(ws, o.w, acc.w);
    }
    *reinterpret_cast<uint2*>(out + (static_cast<size_t>(row) * n_heads + h) * kDv + d) =
        make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  }
}

template <int H, bool TILE>
int launch_t(const MlaLaunch& L, const MlaParams& prm) {
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(mla_kernel<H, TILE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return SMLA_ERR_CUDA;
    attr_done = true;
  }
  const int grid = std::max(1, std::min(num_sms(), (prm.n_rows * prm.n_parts + 1) / 2));
  mla_kernel<H, TILE><<<grid, kThreads, kSmemBytes, L.stream>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
  if (prm.n_parts > 1) {
    part_merge_kernel<<<dim3(prm.n_rows, (H + kMergeHeads - 1) / kMergeHeads), 256, 0, L.stream>>>(
        prm.part_o, prm.part_lse, prm.n_parts, H, prm.out, prm.lse);
    if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
  }
  return SMLA_OK;
}

// Widen the rows of one sequence (logical positions 0..n_rows-1, through its
// page table) to f16, stored contiguously by position: bf16 rows (exact in the
// f16 range), or e4m3 rows (always exact; their per-token scales are copied to
// shadow_scale in the same order and applied by the attention as before).
__global__ void __launch_bounds__(256) shadow_convert_kernel(const uint8_t* __restrict__ kv,
                                                             const float* __restrict__ kv_scale, int32_t fp8,
                                                             const int32_t* __restrict__ pt, int32_t max_pages,
                                                             int32_t num_pages, int32_t n_rows,
                                                             uint16_t* __restrict__ shadow,
                                                             float* __restrict__ shadow_scale, uint32_t* status) {
  const int64_t pieces = static_cast<int64_t>(n_rows) * 72;  // 8 values each
  bool over = false, bad = false;
  for (int64_t pc = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; pc < pieces;
       pc += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(pc / 72), c = static_cast<int>(pc % 72);
    const int lp = r >> 6;
    const int pg = lp < max_pages ? __ldg(pt + lp) : -1;
    uint4 o = make_uint4(0, 0, 0, 0);
    if (pg >= 0 && pg < num_pages) {
      const int64_t prow = static_cast<int64_t>(pg) * kPage + (r & 63);
      if (fp8) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(kv + prow * kDqk + c * 8));
        o = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(v.x & 0xFFFFu)),
                       e4m3x2_to_f16x2(static_cast<uint16_t>(v.x >> 16)),
                       e4m3x2_to_f16x2(static_cast<uint16_t>(v.y & 0xFFFFu)),
                       e4m3x2_to_f16x2(static_cast<uint16_t>(v.y >> 16)));
        if (c == 0) shadow_scale[r] = __ldg(kv_scale + prow);
      } else {
        const uint4 v = ldg_stream(reinterpret_cast<const uint16_t*>(kv) + prow * kDqk + c * 8);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          over |= ((in[t] & 0x7FFFu) > 0x477Fu) || ((in[t] & 0x7FFF0000u) > 0x477F0000u);
          w[t] = bf16x2_to_f16x2(in[t]);
        }
        o = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      bad = true;
      if (fp8 && c == 0) shadow_scale[r] = 0.0f;
    }
    *reinterpret_cast<uint4*>(shadow + static_cast<int64_t>(r) * kDqk + c * 8) = o;
  }
  if (over) set_status(status, kStatusOverflow);
  if (bad) set_status(status, kStatusBounds);
}

}  // namespace

int mla_parts(int32_t n_rows, int32_t topk) {
  const int nb_row = (topk + kBlk - 1) / kBlk;
  const int sms = num_sms();
  if (n_rows <= 0 || n_rows >= sms || nb_row < 2) return 1;
  // power-of-two parts (even splits of a row's blocks) while the work items
  // stay within two per SM: each item pays a query load and an epilogue, so
  // more, shorter items lose more than the finer balance gains (128 rows of
  // 16 blocks on 152 SMs: 2 parts 268 us per decode step, 3 parts 321, 4 parts 293)
  int parts = 1;
  while (2 * parts <= std::min(kMaxParts, nb_row) && n_rows * 2 * parts <= 2 * sms) parts *= 2;
  return parts;
}

size_t mla_partial_bytes(int32_t n_rows, int32_t n_heads) {
  const size_t items = static_cast<size_t>(n_rows) * kMaxParts;
  return items * n_heads * kDv * 4 + (items * n_heads * 4 + 255) / 256 * 256;
}

size_t mla_shadow_bytes(int32_t n_keys, int32_t kv_dtype) {
  if (n_keys <= 0 || (kv_dtype != SMLA_BF16 && kv_dtype != SMLA_FP8_E4M3)) return 0;
  const size_t rows = (static_cast<size_t>(n_keys) * kDqk * 2 + 255) / 256 * 256;
  return kv_dtype == SMLA_BF16 ? rows : rows + (static_cast<size_t>(n_keys) * 4 + 255) / 256 * 256;
}

namespace {
// the per-token scales of an FP8 shadow follow its rows
float* shadow_scales(void* shadow, int32_t n_keys) {
  return reinterpret_cast<float*>(static_cast<uint8_t*>(shadow) +
                                  (static_cast<size_t>(n_keys) * kDqk * 2 + 255) / 256 * 256);
}
}  // namespace

int launch_shadow_convert(const MlaLaunch& L) {
  const int64_t pieces = static_cast<int64_t>(L.shadow_rows) * 72;
  const int64_t want = (pieces + 255) / 256;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 8LL * num_sms())));
  const bool fp8 = L.cache->kv_dtype == SMLA_FP8_E4M3;
  shadow_convert_kernel<<<grid, 256, 0, L.stream>>>(
      static_cast<const uint8_t*>(L.cache->kv), L.cache->kv_scale, fp8 ? 1 : 0, L.page_tables, L.max_pages,
      L.cache->num_pages, L.shadow_rows, static_cast<uint16_t*>(L.shadow),
      fp8 ? shadow_scales(L.shadow, L.shadow_rows) : nullptr, L.status);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

int launch_mla(const MlaLaunch& L) {
  MlaParams prm{};
  prm.kv = static_cast<const uint8_t*>(L.cache->kv);
  prm.kv_scale = L.cache->kv_scale;
  prm.page_tables = L.page_tables;
  prm.max_pages = L.max_pages;
  prm.num_pages = L.cache->num_pages;
  prm.n_seqs = L.n_seqs;
  prm.q_per_seq = L.q_per_seq;
  prm.n_rows = L.n_seqs * L.q_per_seq;
  prm.seq_lens = L.seq_lens;
  prm.prefix_len = L.prefix_len;
  prm.q = static_cast<const uint16_t*>(L.q);
  prm.idx = L.idx;
  prm.topk = L.topk;
  prm.scale_log2 = L.sm_scale * 1.4426950408889634f;
  prm.out = static_cast<uint16_t*>(L.out);
  prm.lse = L.lse;
  prm.fmt = L.cache->kv_dtype == SMLA_FP8_E4M3 ? kFmtTokenFp8 : L.cache->kv_dtype == SMLA_FP8_DS_MLA ? kFmtTileFp8 : kFmtBf16;
  prm.status = L.status;
  prm.shadow = static_cast<const uint16_t*>(L.shadow);
  prm.shadow_rows = L.shadow_rows;
  // a copy that fits in half of L2 stays there; a larger one is prefetched a block ahead
  prm.shadow_prefetch = static_cast<size_t>(L.shadow_rows) * kDqk * 2 > (size_t(64) << 20);
  if (L.shadow && prm.fmt == kFmtTokenFp8) prm.shadow_scale = shadow_scales(L.shadow, L.shadow_rows);
  prm.n_parts = 1;
  prm.part_blocks = (L.topk + kBlk - 1) / kBlk;
  if (prm.n_rows == 0) return SMLA_OK;
  const int parts = mla_parts(prm.n_rows, L.topk);
  if (parts > 1 && L.partials && L.partial_bytes >= mla_partial_bytes(prm.n_rows, L.n_heads) &&
      (reinterpret_cast<uintptr_t>(L.partials) & 15u) == 0) {
    const int nb_row = (L.topk + kBlk - 1) / kBlk;
    prm.part_blocks = (nb_row + parts - 1) / parts;
    prm.n_parts = (nb_row + prm.part_blocks - 1) / prm.part_blocks;
    prm.part_o = static_cast<float*>(L.partials);
    prm.part_lse = prm.part_o + static_cast<size_t>(prm.n_rows) * kMaxParts * L.n_heads * kDv;
  }
  switch (L.n_heads) {
    case 16: return prm.fmt == kFmtTileFp8 ? launch_t<16, true>(L, prm) : launch_t<16, false>(L, prm);
    case 64: return prm.fmt == kFmtTileFp8 ? launch_t<64, true>(L, prm) : launch_t<64, false>(L, prm);
    default: return SMLA_ERR_UNSUPPORTED;
  }
}

}  // namespace smla
