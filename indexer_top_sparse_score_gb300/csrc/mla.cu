// Sparse MLA over selected latent rows (step 3 of the layer step).
//
// "Optimisations de GLM-5.3, partie 2", section "PCP" and footnote 1: each
// selected latent row (576 values) is read once and serves all query heads;
// QK uses all 576 values, PV the first 512. Per query row t:
//     l_j  = sm_scale * q[h,:] . K[s_j,:]          (s_j = selected keys)
//     out  = softmax_j(l) . K[s_j, 0:512],   lse = log sum_j exp(l_j)
//
// One CTA per SM (persistent); query rows are handed out in head/tail pairs
// (cheap causal rows with expensive ones). For each row the 2048 selected
// rows stream through in blocks of 64:
//   warps 8-15  gather producers: resolve key -> page -> pool row, load the
//               row, widen it to f16 (bf16 -> f16 or e4m3 -> f16) and store it
//               into a 128B-swizzled shared tile, 2 stages; they also widen
//               the query to f16 once per query row;
//   warp 0      MMA issuer:  S[64 heads x 64 rows] = Q . K^T   (tcgen05,
//               M=64, K=576) into one of two TMEM S buffers, and
//               O^T[512 x H] += V^T . P^T  (M=128 per 128-dim slice of V, the
//               same shared tile read MN-major, P^T from shared memory);
//   warps 4-7   softmax: S from TMEM (two threads per head), online softmax
//               in the log2 domain with a lazy rescale (O is only rescaled
//               when a head's running max grows by more than 2^8), P to
//               shared memory; finally O^T from TMEM, normalised, to HBM.
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

constexpr int kBlk = 64;                     // selected rows per block
constexpr int kChunks = kDqk / 64;           // 9 chunks of 64 values
constexpr int kChunkBytes = kBlk * 128;      // 8 KB
constexpr int kTileBytes = kChunks * kChunkBytes;  // 72 KB per stage / for Q
// P^T (64 head rows x 64 selected rows, f16) of block b is written into the
// rope chunk (chunk 8) of block b's own stage: QK(b) has finished reading it
// once S(b) is ready, and the stage is not refilled before PV(b) completes.
// Every block therefore has its own P buffer, and the softmax of block b+1
// never waits for PV(b) unless it has to rescale O.
constexpr int kPChunk = kChunks - 1;
constexpr int kThreads = 512;
constexpr int kProducers = 256;          // warps 8-15
constexpr uint32_t kColO = 0, kColS = 256, kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;

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
  int32_t fp8;
  uint32_t* status;
  const uint16_t* shadow;  // f16 rows by logical position, or null
  int32_t shadow_rows;
};

// Per selected row j of a stage: {logit multiplier, bias (0, or -inf for a
// skipped row)} and the probability multiplier (FP8 token scale). Rows 32..63
// sit one slot further so the two halves of a softmax warp hit different banks.
__host__ __device__ constexpr int meta_slot(int j) { return j + (j >= 32 ? 1 : 0); }

struct SmemMeta {
  float2 col[2][kBlk + 1];
  float pscale[2][kBlk + 1];
  float linv[64];
  float alpha[64];
  uint64_t q_full, q_empty, kv_full[2], kv_empty[2], s_full[2], s_empty[2], p_full[2], o_empty;
  uint32_t tmem_slot;
  int abort_flag;
};

constexpr size_t kSmemBytes = 2 * kTileBytes + kTileBytes + sizeof(SmemMeta);

// k-th row of this CTA: head/tail pairs. -1 done, 0 skip, 1 row.
__device__ __forceinline__ int next_row(int n_rows, int k, int& row) {
  const int P = (n_rows + 1) / 2;
  const int pair = blockIdx.x + (k >> 1) * gridDim.x;
  if (pair >= P) return -1;
  row = (k & 1) ? (n_rows - 1 - pair) : pair;
  if ((k & 1) && row == pair) return 0;
  return 1;
}

struct RowInfo {
  int seq, pos, nvalid, nb;
};

__device__ __forceinline__ RowInfo row_info(const MlaParams& p, int row) {
  RowInfo r;
  r.seq = row / p.q_per_seq;
  const int j = row - r.seq * p.q_per_seq;
  const int L = p.seq_lens ? p.seq_lens[r.seq] : p.prefix_len + p.q_per_seq;
  r.pos = L - p.q_per_seq + j;
  r.nvalid = max(0, min(p.topk, r.pos + 1));
  r.nb = (r.nvalid + kBlk - 1) / kBlk;
  return r;
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
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
  if constexpr (NC == 16) tmem_ld_32x32b_x16(taddr, r);
  else tmem_ld_32x32b_x32(taddr, r);
}
template <int NC>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
  if constexpr (NC == 16) {
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

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const MlaParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* q_tile = smem;
  uint8_t* stage = smem + kTileBytes;  // 2 stages
  SmemMeta& M = *reinterpret_cast<SmemMeta*>(smem + 3 * kTileBytes);

  constexpr int kColChunk = H < 32 ? H : 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(p.status, kStatusSetup);
    return;
  }
  // Q rows H..63 stay zero (the QK MMA always has M = 64)
  if (H < 64) {
    for (int i = threadIdx.x; i < kTileBytes / 16; i += kThreads) {
      const int rowb = (i * 16 % kChunkBytes) / 128;
      if (rowb >= H) reinterpret_cast<uint4*>(q_tile)[i] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    mbar_init(&M.q_full, 1);
    mbar_init(&M.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&M.kv_full[i], kProducers);
      mbar_init(&M.kv_empty[i], 1);
      mbar_init(&M.s_full[i], 1);
      mbar_init(&M.s_empty[i], 4);
      // per stage: the softmax may finish P(b+1) before PV(b) is issued, so one
      // barrier for all blocks could run two phases ahead of the MMA thread
      mbar_init(&M.p_full[i], 4);
    }
    mbar_init(&M.o_empty, 4);
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
    // One thread issues QK^T and PV for the CTA's rows in whatever order their
    // inputs become ready: QK(b) needs the gathered tile and a free S buffer,
    // PV(b) needs P(b) (and, for a row's first block, the previous row's O
    // read out). Polling both keeps PV(b) from waiting behind QK(b+1)'s gather.
    if (lane == 0) {
      const uint32_t idesc_qk = instr_desc(64, 64, fmt, fmt, false, false);
      const uint32_t idesc_pv = instr_desc(128, H, fmt, fmt, true, false);
      const uint32_t q0 = smem_u32(q_tile), st0 = smem_u32(stage);
      // K-major 128B-swizzled operands: SBO = 1024 (8-row groups); the gathered
      // tile read MN-major as V^T: LBO = one 64-value chunk of all rows.
      const uint64_t q_desc = smem_desc(q0, 16, 1024);
      const uint64_t st_desc0 = smem_desc(st0, 16, 1024), st_desc1 = smem_desc(st0 + kTileBytes, 16, 1024);
      const uint64_t vt_desc0 = smem_desc(st0, kChunkBytes, 1024);
      const uint64_t vt_desc1 = smem_desc(st0 + kTileBytes, kChunkBytes, 1024);
      const uint64_t p_desc0 = smem_desc(st0 + kPChunk * kChunkBytes, 16, 1024);
      const uint64_t p_desc1 = smem_desc(st0 + kTileBytes + kPChunk * kChunkBytes, 16, 1024);
      struct Cursor {
        int k, b, nb;
        uint32_t g, tok;
        bool done;
      };
      auto seek = [&](Cursor& c) {
        while (true) {
          int row;
          const int r = next_row(p.n_rows, c.k, row);
          if (r < 0) { c.done = true; return; }
          if (r == 0) { ++c.k; continue; }
          c.nb = row_info(p, row).nb;
          c.b = 0;
          if (c.nb > 0) return;
          ++c.k;
        }
      };
      Cursor qc{0, 0, 0, 0, 0, false}, pc{0, 0, 0, 0, 0, false};
      seek(qc);
      seek(pc);
      long long t_last = clock64();
      while (!pc.done) {
        bool prog = false;
        if (!qc.done) {
          const uint32_t gq = qc.g;
          const int s = gq & 1;
          if ((qc.b != 0 || mbar_test(&M.q_full, qc.tok & 1)) && mbar_test(&M.kv_full[s], (gq >> 1) & 1) &&
              mbar_test(&M.s_empty[s], ((gq >> 1) & 1) ^ 1)) {
            tc_fence_after();
            // descriptors advance by (byte offset >> 4) in their start-address field
            const uint64_t bd0 = s ? st_desc1 : st_desc0;
            const uint32_t dS = tmem + kColS + s * 64;
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t off = static_cast<uint64_t>((c * kChunkBytes + kk * 32) >> 4);
                mma_f16(dS, q_desc + off, bd0 + off, idesc_qk, (c | kk) != 0);
              }
            mma_commit(&M.s_full[s]);
            ++qc.g;
            if (++qc.b == qc.nb) {
              mma_commit(&M.q_empty);  // all QK of this row issued: Q may be replaced once they finish
              ++qc.tok;
              ++qc.k;
              seek(qc);
            }
            prog = true;
          }
        }
        if (pc.g < qc.g || (qc.done && !pc.done)) {
          const uint32_t gp = pc.g;
          if (mbar_test(&M.p_full[gp & 1], (gp >> 1) & 1) && (pc.b != 0 || mbar_test(&M.o_empty, (pc.tok & 1) ^ 1))) {
            tc_fence_after();
            const uint64_t ad0 = (gp & 1) ? vt_desc1 : vt_desc0;
            const uint64_t p_desc = (gp & 1) ? p_desc1 : p_desc0;
#pragma unroll
            for (int dt = 0; dt < 4; ++dt)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16(tmem + kColO + dt * 64, ad0 + static_cast<uint64_t>((dt * 2 * kChunkBytes + kk * 2048) >> 4),
                        p_desc + static_cast<uint64_t>((kk * 32) >> 4), idesc_pv, (pc.b | kk) != 0);
            mma_commit(&M.kv_empty[gp & 1]);
            ++pc.g;
            if (++pc.b == pc.nb) {
              ++pc.tok;
              ++pc.k;
              seek(pc);
            }
            prog = true;
          }
        }
        if (prog) {
          t_last = clock64();
        } else {
          if (*abort_v) break;
          if (clock64() - t_last > kWaitLimitCycles) {
            set_status(p.status, kStatusTimeout);
            *abort_v = 1;
            break;
          }
        }
      }
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------------- gather producers
    // Eight threads per selected row read consecutive 16-byte pieces (one
    // 128-byte line per row per load), 32 rows per pass, two passes per
    // 64-row block. The loads of block b+1 are issued right after block b is
    // stored (registers act as a third stage) and the key -> page lookups of
    // the next block run while the current block's data is in flight.
    const int tid = threadIdx.x - 256;
    const int rr = tid >> 3, part = tid & 7;  // row within a pass, piece lane
    constexpr int kPB = 9;                    // BF16: 72 pieces per row / 8 threads
    constexpr int kP8 = 5;                    // FP8: 36 pieces per row / 8 threads (rounded up)
    uint32_t g = 0, tok = 0;
    uint4 v[2][kPB];
    auto lookup = [&](const RowInfo& ri, const int32_t* ir, const int32_t* pt, int b, int jrow) -> int64_t {
      const int e = b * kBlk + jrow;
      if (e >= ri.nvalid) return -1;
      const int key = __ldg(ir + e);
      if (key < 0 || key > ri.pos) return -1;
      if (p.shadow) return key < p.shadow_rows ? key : -1;  // shadow rows are logical positions
      const int lp = key >> 6;
      const int pg = lp < p.max_pages ? __ldg(pt + lp) : -1;
      if (pg < 0 || pg >= p.num_pages) {
        set_status(p.status, kStatusBounds);
        return -1;
      }
      return static_cast<int64_t>(pg) * kPage + (key & 63);
    };
    auto load_block = [&](const int64_t* prow) {
      if (p.shadow) return;  // shadow rows are copied with cp.async once the stage is free
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        if (!p.fp8) {
          const uint16_t* src = reinterpret_cast<const uint16_t*>(p.kv) + (prow[h2] >= 0 ? prow[h2] : 0) * kDqk;
#pragma unroll
          for (int u = 0; u < kPB; ++u)
            v[h2][u] = prow[h2] >= 0 ? ldg_stream(src + (part + 8 * u) * 8) : make_uint4(0, 0, 0, 0);
        } else {
          const uint8_t* src = p.kv + (prow[h2] >= 0 ? prow[h2] : 0) * kDqk;
#pragma unroll
          for (int u = 0; u < kP8; ++u) {
            const int pc = part + 8 * u;
            v[h2][u] = (prow[h2] >= 0 && pc < 36) ? ldg_stream(src + pc * 16) : make_uint4(0, 0, 0, 0);
          }
        }
      }
    };
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int row;
      const int r = next_row(p.n_rows, k, row);
      if (r < 0) break;
      if (r == 0) continue;
      const RowInfo ri = row_info(p, row);
      if (ri.nb == 0) continue;
      const int32_t* pt = p.page_tables + static_cast<size_t>(ri.seq) * p.max_pages;
      const int32_t* ir = p.idx + static_cast<size_t>(row) * p.topk;
      // widen the BF16 query to f16 into the swizzled Q tile
      {
        const uint16_t* qr = p.q + static_cast<size_t>(row) * H * kDqk;
        constexpr int kQPieces = (H * 72 + kProducers - 1) / kProducers;
        uint4* vq = &v[0][0];
#pragma unroll
        for (int u = 0; u < kQPieces; ++u) {
          const int pc = tid + u * kProducers;
          const int h = pc / 72, pp = pc - h * 72;
          if (pc < H * 72) vq[u] = ldg_stream(qr + h * kDqk + pp * 8);
        }
        int64_t prow[2] = {lookup(ri, ir, pt, 0, rr), lookup(ri, ir, pt, 0, rr + 32)};
        if (!mbar_wait(&M.q_empty, (tok & 1) ^ 1, abort_v, p.status)) break;
        bool over = false;
#pragma unroll
        for (int u = 0; u < kQPieces; ++u) {
          const int pc = tid + u * kProducers;
          if (pc >= H * 72) break;
          const int h = pc / 72, pp = pc - h * 72;
          const uint32_t in[4] = {vq[u].x, vq[u].y, vq[u].z, vq[u].w};
          uint32_t o[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            over |= ((in[t] & 0x7FFFu) > 0x477Fu) || ((in[t] & 0x7FFF0000u) > 0x477F0000u);
            o[t] = bf16x2_to_f16x2(in[t]);
          }
          const int c = pp >> 3, qq = pp & 7;
          *reinterpret_cast<uint4*>(q_tile + c * kChunkBytes + h * 128 + ((qq ^ (h & 7)) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (over) set_status(p.status, kStatusOverflow);
        fence_proxy_async_smem();
        named_bar_sync(2, kProducers);
        if (tid == 0) mbar_arrive(&M.q_full);
        load_block(prow);
        for (int b = 0; b < ri.nb; ++b, ++g) {
          const int s = g & 1;
          int64_t prow_next[2] = {-1, -1};
          if (b + 1 < ri.nb) {
            prow_next[0] = lookup(ri, ir, pt, b + 1, rr);
            prow_next[1] = lookup(ri, ir, pt, b + 1, rr + 32);
          }
          float ks[2] = {1.0f, 1.0f};
          if (p.fp8 && part == 0) {
            if (prow[0] >= 0) ks[0] = __ldg(p.kv_scale + prow[0]);
            if (prow[1] >= 0) ks[1] = __ldg(p.kv_scale + prow[1]);
          }
          if (!mbar_wait(&M.kv_empty[s], ((g >> 1) & 1) ^ 1, abort_v, p.status)) { ok = false; break; }
#pragma unroll
          for (int h2 = 0; h2 < 2 && !p.shadow; ++h2) {
            const int j = rr + 32 * h2;
            uint8_t* rowp = stage + s * kTileBytes + j * 128;
            if (part == 0) {
              M.col[s][meta_slot(j)] = prow[h2] >= 0 ? make_float2(ks[h2] * p.scale_log2, 0.0f)
                                                     : make_float2(0.0f, -INFINITY);
              M.pscale[s][meta_slot(j)] = ks[h2];
            }
            if (!p.fp8) {
#pragma unroll
              for (int u = 0; u < kPB; ++u) {
                // piece part + 8u: chunk u, 16-byte slot `part`
                *reinterpret_cast<uint4*>(rowp + u * kChunkBytes + ((part ^ (j & 7)) << 4)) =
                    make_uint4(bf16x2_to_f16x2(v[h2][u].x), bf16x2_to_f16x2(v[h2][u].y),
                               bf16x2_to_f16x2(v[h2][u].z), bf16x2_to_f16x2(v[h2][u].w));
              }
            } else {
#pragma unroll
              for (int u = 0; u < kP8; ++u) {
                const int p8 = part + 8 * u;  // 16 e4m3 values = 32 bytes of f16
                if (p8 >= 36) break;
                const int c = p8 >> 2, qq = (p8 & 3) * 2;
                const uint32_t w[4] = {v[h2][u].x, v[h2][u].y, v[h2][u].z, v[h2][u].w};
                uint32_t o[8];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  o[2 * t] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[t] & 0xFFFFu));
                  o[2 * t + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[t] >> 16));
                }
                uint8_t* cp = rowp + c * kChunkBytes;
                *reinterpret_cast<uint4*>(cp + ((qq ^ (j & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(cp + (((qq + 1) ^ (j & 7)) << 4)) =
                    make_uint4(o[4], o[5], o[6], o[7]);
              }
            }
          }
          if (p.shadow) {
            // f16 rows already widened: 9 x 16-byte async copies per row and thread
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int j = rr + 32 * h2;
              const uint32_t rowp = smem_u32(stage + s * kTileBytes + j * 128);
              if (part == 0) {
                M.col[s][meta_slot(j)] = prow[h2] >= 0 ? make_float2(p.scale_log2, 0.0f) : make_float2(0.0f, -INFINITY);
                M.pscale[s][meta_slot(j)] = 1.0f;
              }
              const uint16_t* src = p.shadow + (prow[h2] >= 0 ? prow[h2] : 0) * kDqk;
              const uint32_t nb = prow[h2] >= 0 ? 16u : 0u;
#pragma unroll
              for (int u = 0; u < kPB; ++u)
                cp_async_16(rowp + u * kChunkBytes + ((part ^ (j & 7)) << 4), src + (part + 8 * u) * 8, nb);
            }
            cp_async_commit();
            cp_async_wait<0>();
          }
          fence_proxy_async_smem();
          mbar_arrive(&M.kv_full[s]);
          if (b + 1 < ri.nb) load_block(prow_next);
          prow[0] = prow_next[0];
          prow[1] = prow_next[1];
        }
      }
      ++tok;
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int qd = warp & 3;
    const int half = lane >> 4;
    const int h = 16 * qd + (lane & 15);
    const bool real = h < H;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    uint32_t g = 0, tok = 0;
    for (int k = 0;; ++k) {
      int row;
      const int r = next_row(p.n_rows, k, row);
      if (r < 0) break;
      if (r == 0) continue;
      const RowInfo ri = row_info(p, row);
      float m_used = -INFINITY, l = 0.0f;
      bool ok = true;
      for (int b = 0; b < ri.nb; ++b) {
        const uint32_t gb = g + b;
        const int s = gb & 1;
        if (!mbar_wait(&M.s_full[s], (gb >> 1) & 1, abort_v, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t raw[32];
        tmem_ld_16x32bx2_x32<32>(tmem + lane_base + kColS + s * 64, raw);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.s_empty[s]);
        if (!mbar_wait(&M.kv_full[s], (gb >> 1) & 1, abort_v, p.status)) { ok = false; break; }
        float x[32];
        float mx = -INFINITY;
        const float2* meta = &M.col[s][meta_slot(half * 32)];
        const float* pmeta = &M.pscale[s][meta_slot(half * 32)];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 m2 = meta[i];  // same address across the half: broadcast
          x[i] = fmaf(__uint_as_float(raw[i]), m2.x, m2.y);
          mx = fmaxf(mx, x[i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
        const float m_new = fmaxf(m_used, mx);
        const bool resc = real && b > 0 && m_new > m_used + kRescaleLog2;
        if (b == 0) m_used = m_new;
        // probabilities against the running max (unchanged unless this head rescales),
        // computed before waiting for the previous PV so they overlap it
        float sum = 0.0f;
        uint32_t pk[16];
        auto make_p = [&]() {
          const float mref = m_used == -INFINITY ? 0.0f : m_used;
          sum = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float p0 = fast_exp2(x[i] - mref), p1 = fast_exp2(x[i + 1] - mref);
            sum += p0 + p1;
            pk[i >> 1] = p.fp8 ? pack_f16(p0 * pmeta[i], p1 * pmeta[i + 1]) : pack_f16(p0, p1);
          }
        };
        if (!resc) make_p();
        const bool any = named_bar_or(1, 128, resc);
        if (any) {
          // O must hold exactly PV(0..b-1) while it is rescaled. kv_empty[stage]
          // completes when the PV of that stage's block finishes; for block b-1
          // it is at most one phase away from this wait (its stage was refilled
          // for b-1 only after PV(b-3) completed), so the parity is unambiguous.
          const uint32_t gp = gb - 1;
          if (!mbar_wait(&M.kv_empty[gp & 1], (gp >> 1) & 1, abort_v, p.status)) { ok = false; break; }
          const float a = resc ? fast_exp2(m_used - m_new) : 1.0f;
          if (resc) {
            m_used = m_new;
            l *= a;
            make_p();
          }
          if (half == 0) M.alpha[h] = a;
          named_bar_sync(1, 128);
          tc_fence_after();
#pragma unroll 1
          for (int dt = 0; dt < 4; ++dt) {
#pragma unroll 1
            for (int c0 = 0; c0 < H; c0 += kColChunk) {
              uint32_t o[kColChunk];
              const uint32_t ta = tmem + lane_base + kColO + dt * 64 + c0;
              tmem_ld_cols<kColChunk>(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < kColChunk; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * M.alpha[c0 + c]);
              tmem_st_cols<kColChunk>(ta, o);
            }
          }
          tmem_wait_st();
          tc_fence_before();
        }
        l += sum;
        uint8_t* prow = stage + s * kTileBytes + kPChunk * kChunkBytes + h * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int qq = half * 4 + u;
          *reinterpret_cast<uint4*>(prow + ((qq ^ (h & 7)) << 4)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.p_full[s]);
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      {
        // last PV of this row done (same reasoning as for the rescale wait)
        const uint32_t gl = g + ri.nb - 1;
        if (!mbar_wait(&M.kv_empty[gl & 1], (gl >> 1) & 1, abort_v, p.status)) break;
      }
      tc_fence_after();
      const float lt = l + __shfl_xor_sync(0xFFFFFFFFu, l, 16);
      if (half == 0 && real) {
        M.linv[h] = lt > 0.0f ? 1.0f / lt : 0.0f;
        if (p.lse)
          p.lse[static_cast<size_t>(row) * H + h] =
              lt > 0.0f ? (m_used + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
      }
      named_bar_sync(1, 128);
      uint16_t* orow = p.out + static_cast<size_t>(row) * H * kDv;
      const bool odd = lane & 1;
#pragma unroll 1
      for (int dt = 0; dt < 4; ++dt) {
        const int d = dt * 128 + qd * 32 + lane;
        const int d_even = d & ~1;
#pragma unroll 1
        for (int c0 = 0; c0 < H; c0 += kColChunk) {
          uint32_t o[kColChunk];
          tmem_ld_cols<kColChunk>(tmem + lane_base + kColO + dt * 64 + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < kColChunk; c += 2) {
            const float v0 = __uint_as_float(o[c]) * M.linv[c0 + c];
            const float v1 = __uint_as_float(o[c + 1]) * M.linv[c0 + c + 1];
            const float x2 = __shfl_xor_sync(0xFFFFFFFFu, odd ? v0 : v1, 1);
            const uint32_t word = odd ? pack_bf16(x2, v1) : pack_bf16(v0, x2);
            const int hh = c0 + (odd ? c + 1 : c);
            *reinterpret_cast<uint32_t*>(orow + static_cast<size_t>(hh) * kDv + d_even) = word;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.o_empty);
      g += ri.nb;
      ++tok;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

template <int H>
int launch_t(const MlaLaunch& L, const MlaParams& prm) {
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(mla_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return SMLA_ERR_CUDA;
    attr_done = true;
  }
  const int grid = std::max(1, std::min(num_sms(), (prm.n_rows + 1) / 2));
  mla_kernel<H><<<grid, kThreads, kSmemBytes, L.stream>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
  return SMLA_OK;
}

// Widen the BF16 rows of one sequence (logical positions 0..n_rows-1, through
// its page table) to f16, stored contiguously by position.
__global__ void __launch_bounds__(256) shadow_convert_kernel(const uint16_t* __restrict__ kv,
                                                             const int32_t* __restrict__ pt, int32_t max_pages,
                                                             int32_t num_pages, int32_t n_rows,
                                                             uint16_t* __restrict__ shadow, uint32_t* status) {
  const int64_t pieces = static_cast<int64_t>(n_rows) * 72;  // 8 values each
  bool over = false, bad = false;
  for (int64_t pc = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; pc < pieces;
       pc += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(pc / 72), c = static_cast<int>(pc % 72);
    const int lp = r >> 6;
    const int pg = lp < max_pages ? __ldg(pt + lp) : -1;
    uint4 o = make_uint4(0, 0, 0, 0);
    if (pg >= 0 && pg < num_pages) {
      const uint4 v = ldg_stream(kv + (static_cast<int64_t>(pg) * kPage + (r & 63)) * kDqk + c * 8);
      const uint32_t in[4] = {v.x, v.y, v.z, v.w};
      uint32_t w[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        over |= ((in[t] & 0x7FFFu) > 0x477Fu) || ((in[t] & 0x7FFF0000u) > 0x477F0000u);
        w[t] = bf16x2_to_f16x2(in[t]);
      }
      o = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      bad = true;
    }
    *reinterpret_cast<uint4*>(shadow + static_cast<int64_t>(r) * kDqk + c * 8) = o;
  }
  if (over) set_status(status, kStatusOverflow);
  if (bad) set_status(status, kStatusBounds);
}

}  // namespace

size_t mla_shadow_bytes(int32_t n_keys) {
  return n_keys > 0 ? (static_cast<size_t>(n_keys) * kDqk * 2 + 255) / 256 * 256 : 0;
}

int launch_shadow_convert(const MlaLaunch& L) {
  const int64_t pieces = static_cast<int64_t>(L.shadow_rows) * 72;
  const int64_t want = (pieces + 255) / 256;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 8LL * num_sms())));
  shadow_convert_kernel<<<grid, 256, 0, L.stream>>>(static_cast<const uint16_t*>(L.cache->kv), L.page_tables,
                                                   L.max_pages, L.cache->num_pages, L.shadow_rows,
                                                   static_cast<uint16_t*>(L.shadow), L.status);
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
  prm.fp8 = L.cache->kv_dtype == SMLA_FP8_E4M3;
  prm.status = L.status;
  prm.shadow = static_cast<const uint16_t*>(L.shadow);
  prm.shadow_rows = L.shadow_rows;
  if (prm.n_rows == 0) return SMLA_OK;
  switch (L.n_heads) {
    case 16: return launch_t<16>(L, prm);
    case 64: return launch_t<64>(L, prm);
    default: return SMLA_ERR_UNSUPPORTED;
  }
}

}  // namespace smla
