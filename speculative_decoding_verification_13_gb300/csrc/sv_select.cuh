// Block-level selection and sorting on 64-bit composite keys, used for top-k
// (rows) and for ordering kept tokens by index (final draw).
//   block_select_kth: exact k-th largest of n keys by MSB-first radix select
//                     over 8-bit digits, with warp-aggregated shared-memory
//                     histograms; stops early once the remaining prefix group
//                     is selected whole.
//   block_sort_desc:  bitonic sort of up to NT keys (one per thread), warp
//                     shuffles for partner distances < 32, double-buffered
//                     shared memory above.
// Every thread of the group must call these with identical arguments.
#pragma once

#include "sv_internal.cuh"

namespace sv {

struct SelShared {
  int digit;
  int above;
  int cnt;
  int pad;
  unsigned long long minv;
};

// Digit positions (shift / 8) that hold the same byte in every key can be
// skipped: bit s of `skip` skips the digit at shift 8 * s.  For keys built
// from bfloat16 values the low 16 bits of the value word are constant, and for
// indices below 2^24 the top byte of ~index is constant.
constexpr uint32_t kSkipBf16 = (1u << 5) | (1u << 4) | (1u << 3);
constexpr uint32_t kSkipF32 = (1u << 3);

template <int NT, class Sync>
__device__ uint64_t block_select_kth(const uint64_t* keys, int n, int k, int tid, int* hist,
                                     SelShared* sh, Sync sync, uint32_t skip = 0) {
  const int lane = tid & 31, warp = tid >> 5;
  uint64_t prefix = 0, mask = 0;
  int need = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    if ((skip >> (shift / 8)) & 1u) continue;
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    if (tid == 0) sh->minv = ~0ull;
    sync();
    for (int base = warp * 32; base < n; base += NT) {
      const int e = base + lane;
      bool valid = false;
      uint32_t d = 0;
      if (e < n) {
        const uint64_t key = keys[e];
        if ((key & mask) == prefix) {
          valid = true;
          d = static_cast<uint32_t>(key >> shift) & 255u;
        }
      }
      const uint32_t vm = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t peers = __match_any_sync(vm, d);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
      }
    }
    sync();
    if (warp == 0) {
      int cnt[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = hist[lane * 8 + j];
        loc += cnt[j];
      }
      int suf = loc;  // inclusive suffix sum over lanes lane..31
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
      }
      int acc = suf - loc;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (acc < need && acc + cnt[j] >= need) {
          sh->digit = lane * 8 + j;
          sh->above = acc;
          sh->cnt = cnt[j];
        }
        acc += cnt[j];
      }
    }
    sync();
    const int d = sh->digit;
    need -= sh->above;
    const int grp = sh->cnt;
    prefix |= static_cast<uint64_t>(d) << shift;
    mask |= 255ull << shift;
    if (grp == need) {
      uint64_t mn = ~0ull;
      for (int e = tid; e < n; e += NT) {
        const uint64_t key = keys[e];
        if ((key & mask) == prefix && key < mn) mn = key;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t y = shfl_xor_u64(mn, o);
        mn = y < mn ? y : mn;
      }
      if (lane == 0) atomicMin(&sh->minv, static_cast<unsigned long long>(mn));
      sync();
      const uint64_t r = sh->minv;
      sync();
      return r;
    }
    sync();
  }
  return prefix;
}

// Sorts the values held one per thread (threads 0..P-1; P a power of two,
// P <= NT) into descending order: thread i ends with the i-th largest.
// Threads >= P carry padding and take part harmlessly.  xchg: 2 * NT slots.
template <int NT, class Sync>
__device__ uint64_t block_sort_desc(uint64_t v, int tid, int P, uint64_t* xchg, Sync sync) {
  int buf = 0;
  for (int size = 2; size <= P; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      uint64_t o;
      if (j >= 32) {
        xchg[buf * NT + tid] = v;
        sync();
        o = xchg[buf * NT + (tid ^ j)];
        buf ^= 1;
      } else {
        o = shfl_xor_u64(v, j);
      }
      const bool desc = (tid & size) == 0;
      const bool lower = (tid & j) == 0;
      v = (desc == lower) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Warp-level: the m-th largest of the nonzero keys the lanes hold (NV per
// lane, 0 = empty slot, keys unique), by m rounds of warp max with removal.
// Returns 0 when the warp holds fewer than m keys.  Warp-uniform result.
template <int NV>
__device__ __forceinline__ uint64_t warp_mth_largest(uint64_t (&k)[NV], int m) {
  uint64_t res = 0ull;
  for (int r = 0; r < m; ++r) {
    uint64_t lm = k[0];
    int li = 0;
#pragma unroll
    for (int j = 1; j < NV; ++j)
      if (k[j] > lm) {
        lm = k[j];
        li = j;
      }
    uint64_t wm = lm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t y = shfl_xor_u64(wm, o);
      wm = y > wm ? y : wm;
    }
    res = wm;
    if (wm == 0ull) break;
    if (lm == wm) {
#pragma unroll
      for (int j = 0; j < NV; ++j)
        if (j == li) k[j] = 0ull;
    }
  }
  return res;
}

__host__ __device__ __forceinline__ int next_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

}  // namespace sv
