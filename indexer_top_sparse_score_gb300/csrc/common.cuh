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

__device__ __forceinline__ void hist_add(uint32_t* hist, bool in, uint32_t bin) {
  if (in) atomicAdd(&hist[bin], 1u);
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
      const bool in = (key & mask) == prefix;
      hist_add(hist, in, (key >> shift) & 255u);
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
      const bool in = key == prefix && (idx & imask) == iprefix;
      hist_add(hist, in, (idx >> shift) & 255u);
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

// ---------------------------------------------------------------------------
// Exact top-k threshold over entries held in shared memory: keys[0..n),
// idxs[0..n) (n > k >= 1), 128 cooperating threads synchronised by `sync()`,
// `hist` = 3 x 256 words and `red` = 16 words of shared scratch. Returns
// (thr_key, thr_idx): entry e is among the best k (key descending, index
// ascending) iff key > thr_key, or key == thr_key and idx <= thr_idx.
//
// Method: a radix select whose bins span only the live key range [lo, hi]
// (found by a min/max pass) and shrink it by 8 bits per pass, so values that
// share a float exponent still spread over the bins; then, if the k-th key is
// tied and not all ties are needed, the same on the indices of the ties
// (ascending). Key passes read keys only, 4 per 16-byte load. Each pass costs
// one barrier: histograms rotate over three buffers (the one a pass fills was
// last read two passes ago and is cleared one pass ahead), and every warp
// scans the finished histogram itself instead of waiting for a broadcast.
template <typename Sync>
__device__ __forceinline__ void wg_select(const uint32_t* keys, const uint32_t* idxs, int n, int k, int tid,
                                          uint32_t* hist, uint32_t* red, Sync sync, uint32_t& thr_key,
                                          uint32_t& thr_idx) {
  const int lane = tid & 31, w = tid >> 5;
  int hb = 0;  // histogram buffer of the next pass
  auto each4 = [&](bool with_idx, auto f) {
    for (int e0 = tid * 4; e0 < n; e0 += 512) {
      const uint4 kv = *reinterpret_cast<const uint4*>(keys + e0);
      uint4 iv = make_uint4(0, 0, 0, 0);
      if (with_idx) iv = *reinterpret_cast<const uint4*>(idxs + e0);
      f(kv.x, iv.x, e0 + 0 < n);
      f(kv.y, iv.y, e0 + 1 < n);
      f(kv.z, iv.z, e0 + 2 < n);
      f(kv.w, iv.w, e0 + 3 < n);
    }
  };
  // min / max of a (filtered) value; also clears the first histogram buffer
  auto minmax = [&](bool ties, uint32_t tk, uint32_t& lo, uint32_t& hi, int slot) {
    for (int b = tid; b < 256; b += 128) hist[256 * hb + b] = 0;
    uint32_t a = 0xFFFFFFFFu, bmax = 0;
    each4(ties, [&](uint32_t kk, uint32_t ii, bool ok) {
      if (!ok || (ties && kk != tk)) return;
      const uint32_t v = ties ? ii : kk;
      a = min(a, v);
      bmax = max(bmax, v);
    });
    a = __reduce_min_sync(0xFFFFFFFFu, a);
    bmax = __reduce_max_sync(0xFFFFFFFFu, bmax);
    if (lane == 0) {
      red[slot + w] = a;
      red[slot + 4 + w] = bmax;
    }
    sync();
    lo = min(min(red[slot], red[slot + 1]), min(red[slot + 2], red[slot + 3]));
    hi = max(max(red[slot + 4], red[slot + 5]), max(red[slot + 6], red[slot + 7]));
  };
  // narrow [lo, hi] to the bin holding the r-th value (descending for keys,
  // ascending for tie indices) until it is a single value
  auto refine = [&](bool ties, uint32_t tk, uint32_t lo, uint32_t hi, int& r, uint32_t& value, uint32_t& count) {
    while (true) {
      const uint32_t range = hi - lo;
      const int shift = range >= 256u ? (32 - __clz(range)) - 8 : 0;
      uint32_t* h = hist + 256 * hb;
      uint32_t* hn = hist + 256 * ((hb + 1) % 3);
      for (int b = tid; b < 256; b += 128) hn[b] = 0;  // next pass's buffer (read two passes ago)
      each4(ties, [&](uint32_t kk, uint32_t ii, bool ok) {
        if (!ok) return;
        const uint32_t v = ties ? ii : kk;
        if ((ties && kk != tk) || v < lo || v > hi) return;
        atomicAdd(&h[(v - lo) >> shift], 1u);
      });
      sync();
      hb = (hb + 1) % 3;
      // every warp finds the bin holding the r-th value; lane l owns 8 consecutive bins
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int bin = ties ? 8 * lane + i : 255 - 8 * lane - i;
        c[i] = h[bin];
        sum += c[i];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t excl = incl - sum;
      uint32_t mine = 0;
      if (excl < static_cast<uint32_t>(r) && incl >= static_cast<uint32_t>(r)) {
        uint32_t run = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (run + c[i] >= static_cast<uint32_t>(r)) {
            const uint32_t bin = ties ? 8 * lane + i : 255 - 8 * lane - i;
            mine = 0x80000000u | (bin << 16) | (static_cast<uint32_t>(r) - run);  // r <= k <= 2048: 16 bits
            count = c[i];
            break;
          }
          run += c[i];
        }
      }
      const uint32_t found = __reduce_or_sync(0xFFFFFFFFu, mine);
      const int src = __ffs(__ballot_sync(0xFFFFFFFFu, mine != 0)) - 1;
      count = __shfl_sync(0xFFFFFFFFu, count, src);
      const uint32_t bin = (found >> 16) & 0xFFu;
      r = static_cast<int>(found & 0xFFFFu);
      const uint64_t nlo = static_cast<uint64_t>(lo) + (static_cast<uint64_t>(bin) << shift);
      const uint64_t nhi = nlo + ((1ull << shift) - 1ull);
      lo = static_cast<uint32_t>(nlo);
      hi = static_cast<uint32_t>(nhi < hi ? nhi : hi);
      if (shift == 0) {
        value = lo;
        return;
      }
    }
  };
  uint32_t lo, hi, cnt = 0;
  int r = k;
  minmax(false, 0, lo, hi, 0);
  refine(false, 0, lo, hi, r, thr_key, cnt);
  if (static_cast<uint32_t>(r) == cnt) {
    thr_idx = 0xFFFFFFFFu;
    return;
  }
  minmax(true, thr_key, lo, hi, 8);  // other red[] slot: the first may still be read
  refine(true, thr_key, lo, hi, r, thr_idx, cnt);
}

// ---------------------------------------------------------------------------
// Exact top-k threshold over an array of entries: entry e has key keys[e] and
// index idxs[e] (or e when idxs is null), for e in [0, n) (n > k >= 1). NT
// cooperating threads (a multiple of 128) synchronised by `sync()`; `hist` =
// 3 x 256 words and `red` = 2 * NT / 32 words of shared scratch; keys (and
// idxs) must be 16-byte aligned. Returns (thr_key, thr_idx) with the meaning
// of wg_select. Same method as wg_select (range-adaptive radix passes over the
// keys, then over the tied indices), reading the entries straight from
// (global or shared) memory, four per 16-byte load.
template <int NT, typename Sync>
__device__ __forceinline__ void dense_select(const uint32_t* keys, const uint32_t* idxs, int n, int k, int tid,
                                             uint32_t* hist, uint32_t* red, Sync sync, uint32_t& thr_key,
                                             uint32_t& thr_idx) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, w = tid >> 5;
  int hb = 0;
  // f(key, index, valid) for every entry of this thread (4 consecutive per
  // load, four loads in flight per thread); the index is idxs[e] when idxs is
  // given, else the position e
  auto each4 = [&](auto f) {
    constexpr int U = 4;
    for (int b0 = tid * 4; b0 < n; b0 += 4 * NT * U) {
      uint4 kv[U], iv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e0 = b0 + u * 4 * NT;
        kv[u] = e0 < n ? *reinterpret_cast<const uint4*>(keys + e0) : make_uint4(0, 0, 0, 0);
        iv[u] = make_uint4(e0, e0 + 1, e0 + 2, e0 + 3);
        if (idxs && e0 < n) iv[u] = *reinterpret_cast<const uint4*>(idxs + e0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e0 = b0 + u * 4 * NT;
        f(kv[u].x, iv[u].x, e0 + 0 < n);
        f(kv[u].y, iv[u].y, e0 + 1 < n);
        f(kv[u].z, iv[u].z, e0 + 2 < n);
        f(kv[u].w, iv[u].w, e0 + 3 < n);
      }
    }
  };
  auto minmax = [&](bool ties, uint32_t tk, uint32_t& lo, uint32_t& hi) {
    for (int b = tid; b < 256; b += NT) hist[256 * hb + b] = 0;
    uint32_t a = 0xFFFFFFFFu, bmax = 0;
    each4([&](uint32_t kk, uint32_t e, bool ok) {
      if (!ok || (ties && kk != tk)) return;
      const uint32_t v = ties ? e : kk;
      a = min(a, v);
      bmax = max(bmax, v);
    });
    a = __reduce_min_sync(0xFFFFFFFFu, a);
    bmax = __reduce_max_sync(0xFFFFFFFFu, bmax);
    if (lane == 0) {
      red[w] = a;
      red[NW + w] = bmax;
    }
    sync();
    lo = 0xFFFFFFFFu;
    hi = 0;
    for (int i = 0; i < NW; ++i) {
      lo = min(lo, red[i]);
      hi = max(hi, red[NW + i]);
    }
    sync();  // red is reused by the next min/max
  };
  auto refine = [&](bool ties, uint32_t tk, uint32_t lo, uint32_t hi, int& r, uint32_t& value, uint32_t& count) {
    while (true) {
      const uint32_t range = hi - lo;
      const int shift = range >= 256u ? (32 - __clz(range)) - 8 : 0;
      uint32_t* h = hist + 256 * hb;
      uint32_t* hn = hist + 256 * ((hb + 1) % 3);
      for (int b = tid; b < 256; b += NT) hn[b] = 0;
      each4([&](uint32_t kk, uint32_t e, bool ok) {
        if (!ok) return;
        const uint32_t v = ties ? e : kk;
        if ((ties && kk != tk) || v < lo || v > hi) return;
        atomicAdd(&h[(v - lo) >> shift], 1u);
      });
      sync();
      hb = (hb + 1) % 3;
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int bin = ties ? 8 * lane + i : 255 - 8 * lane - i;
        c[i] = h[bin];
        sum += c[i];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t excl = incl - sum;
      uint32_t bin_found = 0, r_in = 0, cnt = 0;
      bool mine = false;
      if (excl < static_cast<uint32_t>(r) && incl >= static_cast<uint32_t>(r)) {
        uint32_t run = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (run + c[i] >= static_cast<uint32_t>(r)) {
            bin_found = ties ? 8 * lane + i : 255 - 8 * lane - i;
            r_in = static_cast<uint32_t>(r) - run;
            cnt = c[i];
            mine = true;
            break;
          }
          run += c[i];
        }
      }
      const int src = __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1;
      bin_found = __shfl_sync(0xFFFFFFFFu, bin_found, src);
      r = static_cast<int>(__shfl_sync(0xFFFFFFFFu, r_in, src));
      count = __shfl_sync(0xFFFFFFFFu, cnt, src);
      const uint64_t nlo = static_cast<uint64_t>(lo) + (static_cast<uint64_t>(bin_found) << shift);
      const uint64_t nhi = nlo + ((1ull << shift) - 1ull);
      lo = static_cast<uint32_t>(nlo);
      hi = static_cast<uint32_t>(nhi < hi ? nhi : hi);
      if (shift == 0) {
        value = lo;
        return;
      }
    }
  };
  uint32_t lo, hi, cnt = 0;
  int r = k;
  minmax(false, 0, lo, hi);
  refine(false, 0, lo, hi, r, thr_key, cnt);
  if (static_cast<uint32_t>(r) == cnt) {
    thr_idx = 0xFFFFFFFFu;
    return;
  }
  minmax(true, thr_key, lo, hi);
  refine(true, thr_key, lo, hi, r, thr_idx, cnt);
}

// ---------------------------------------------------------------------------
// Conservative cut for a buffer that only needs shrinking (not the exact top-k):
// returns the largest L such that at least k entries have key >= L, to bin
// resolution: one min/max pass and one histogram pass over the live range.
// Every entry with key < L is beaten by k entries of the buffer and so by k
// earlier keys. Same cooperation contract and scratch as wg_select.
template <typename Sync>
__device__ __forceinline__ uint32_t wg_cut(const uint32_t* keys, int n, int k, int tid, uint32_t* hist,
                                           uint32_t* red, Sync sync) {
  const int lane = tid & 31, w = tid >> 5;
  for (int b = tid; b < 256; b += 128) hist[b] = 0;
  uint32_t a = 0xFFFFFFFFu, bmax = 0;
  for (int e0 = tid * 4; e0 < n; e0 += 512) {
    const uint4 kv = *reinterpret_cast<const uint4*>(keys + e0);
    const uint32_t v4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (e0 + q < n) {
        a = min(a, v4[q]);
        bmax = max(bmax, v4[q]);
      }
  }
  a = __reduce_min_sync(0xFFFFFFFFu, a);
  bmax = __reduce_max_sync(0xFFFFFFFFu, bmax);
  if (lane == 0) {
    red[w] = a;
    red[4 + w] = bmax;
  }
  sync();
  const uint32_t lo = min(min(red[0], red[1]), min(red[2], red[3]));
  const uint32_t hi = max(max(red[4], red[5]), max(red[6], red[7]));
  const uint32_t range = hi - lo;
  const int shift = range >= 256u ? (32 - __clz(range)) - 8 : 0;
  for (int e0 = tid * 4; e0 < n; e0 += 512) {
    const uint4 kv = *reinterpret_cast<const uint4*>(keys + e0);
    const uint32_t v4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (e0 + q < n) atomicAdd(&hist[(v4[q] - lo) >> shift], 1u);
  }
  sync();
  uint32_t c[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = hist[255 - 8 * lane - i];
    sum += c[i];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  const uint32_t excl = incl - sum;
  uint32_t mine = 0;
  if (excl < static_cast<uint32_t>(k) && incl >= static_cast<uint32_t>(k)) {
    uint32_t run = excl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (run + c[i] >= static_cast<uint32_t>(k)) {
        mine = 0x80000000u | (255u - 8u * lane - i);
        break;
      }
      run += c[i];
    }
  }
  const uint32_t bin = __reduce_or_sync(0xFFFFFFFFu, mine) & 0xFFu;
  return lo + (bin << shift);
}

}  // namespace smla
