// Device helpers shared by the kernels: status reporting, order-preserving
// score keys, and an exact block-cooperative top-k selection.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace smla {

// Status word at the head of every workspace (first 256 bytes).
struct DeviceStatus {
  uint32_t bits;
  uint32_t pad[63];
};

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// fp32 -> uint32 key whose unsigned order is the float order (larger float,
// larger key). -0 is folded onto +0 so equal scores get equal keys.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// ---------------------------------------------------------------------------
// Exact selection of the `k` best (key descending, index ascending) among `n`
// entries. Cooperative over NT threads that share `hist` (256 uint32) and
// `scratch` (4 uint32) in shared memory and synchronise with `sync()`.
// `each(f)` calls f(key, idx) for every entry owned by the calling thread
// (each entry is owned by exactly one thread); the result is the pair
// (thr_key, thr_idx): an entry is selected iff key > thr_key, or key ==
// thr_key and idx <= thr_idx. Requires more than k entries and k >= 1.
//
// Method: MSB-first radix select on the 32-bit key (4 passes of 8 bits) finds
// the key value of the k-th entry and how many entries equal to it are
// needed; if not all of them, a second radix select on the index (ascending)
// finds the largest index still taken.
template <int NT, typename Each, typename Sync>
__device__ __forceinline__ void radix_select(int k, int tid, uint32_t* hist, uint32_t* scratch, Each each,
                                             Sync sync, uint32_t& thr_key, uint32_t& thr_idx) {
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  uint32_t eq_count = 0;
  // pass over key bytes, most significant first; larger keys first
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += NT) hist[b] = 0;
    sync();
    each([&](uint32_t key, uint32_t) {
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    });
    sync();
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      const int lane = tid;
      uint32_t c[8];
      uint32_t s = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
        s += c[i];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - s;
      const bool here = excl < (uint32_t)remaining && incl >= (uint32_t)remaining;
      if (here) {
        uint32_t run = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (run + c[i] >= (uint32_t)remaining) {
            scratch[0] = 255u - 8u * lane - i;       // bin
            scratch[1] = (uint32_t)remaining - run;  // still needed inside the bin
            scratch[2] = c[i];                       // entries in the bin
            break;
          }
          run += c[i];
        }
      }
    }
    sync();
    const uint32_t bin = scratch[0];
    remaining = (int)scratch[1];
    eq_count = scratch[2];
    prefix |= bin << shift;
    mask |= 0xFFu << shift;
    sync();
  }
  thr_key = prefix;
  if ((uint32_t)remaining == eq_count) {
    thr_idx = 0xFFFFFFFFu;
    return;
  }
  // among entries with key == prefix, take the `remaining` smallest indices
  uint32_t iprefix = 0, imask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += NT) hist[b] = 0;
    sync();
    each([&](uint32_t key, uint32_t idx) {
      if (key == prefix && (idx & imask) == iprefix) atomicAdd(&hist[(idx >> shift) & 255u], 1u);
    });
    sync();
    if (tid < 32) {
      // ascending: lane l owns bins 8l .. 8l+7
      const int lane = tid;
      uint32_t c[8];
      uint32_t s = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[8 * lane + i];
        s += c[i];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - s;
      if (excl < (uint32_t)remaining && incl >= (uint32_t)remaining) {
        uint32_t run = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (run + c[i] >= (uint32_t)remaining) {
            scratch[0] = 8u * lane + i;
            scratch[1] = (uint32_t)remaining - run;
            break;
          }
          run += c[i];
        }
      }
    }
    sync();
    const uint32_t bin = scratch[0];
    remaining = (int)scratch[1];
    iprefix |= bin << shift;
    imask |= 0xFFu << shift;
    sync();
  }
  thr_idx = iprefix;
}

__device__ __forceinline__ bool selected(uint32_t key, uint32_t idx, uint32_t thr_key, uint32_t thr_idx) {
  return key > thr_key || (key == thr_key && idx <= thr_idx);
}

}  // namespace smla
