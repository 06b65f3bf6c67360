// Filter / decide kernel: what follows the row pass for every request except
// the unfiltered sampled draws (the draw pass).
//
// Persistent warps over the job list of the setup kernel (one job per
// filtered row, one decide job per other request):
//   filtered row  (one warp) exact top k of the row pass's survivors
//                 (composite order: logit descending, index ascending), the
//                 temperature softmax over them, the top-p cut (keep j while
//                 the mass before j is below top_p) and the renormalisation,
//                 applied alike to target and draft rows ("Speculative decoding
//                 and multi-token prediction", "Why the output is identical").
//                 The warp that finishes a request's last row decides the
//                 request and draws its final token from the kept sets.
//   decide job    (one warp) greedy: accept while x_i equals the target argmax
//                 (lowest index on ties) and emit the argmax at the first
//                 disagreement or as the bonus ("DFlash" §4 step 5;
//                 "Speculative decoding…", "Draft and verify", step Three).
//                 Sampling: accept while u_i < p_i(x_i) / q_i(x_i), stop at the
//                 first rejection ("FlashMap…" §4, steps 1-2), then queue the
//                 final draw for the draw pass.
//
// Completion counting ("the last one to finish does the rest"): a warp
// publishes its row's results, fences, and bumps the request's counter; the
// warp that sees the final count fences again and reads the other warps'
// results through L2.  Nothing waits on another warp.
#include <math.h>

#include "sv_select.cuh"

namespace sv {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr double kFix = 36028797018963968.0;    // 2^55: unit of the kept-set fixed-point sums
                                                // (<= 256 weights <= 1 stay below 2^63)

__device__ __forceinline__ double nan64() { return __longlong_as_double(0x7ff8000000000000LL); }

// ------------------------------------------------------------- scratch
// Drawing from kept sets (one warp).
struct DrawScratch {
  int idx[kTopkMax];        // draft kept tokens
  double v[kTopkMax];       // their q, then the residual weight by target slot
  uint64_t keys[kTopkMax];  // ~(index << 32 | slot) of the target kept tokens
};

// ------------------------------------------------------------ selection
// Exact k-th largest of the n (> k) unique keys at keys[] (any memory), by
// MSB-first radix selection over 8-bit digits with a warp-private histogram;
// stops once the remaining prefix group is selected whole.  One warp.
// hist: 256 ints of shared memory; sel: 3 ints (digit, count above, count in it).
__device__ __noinline__ uint64_t warp_select_kth(const uint64_t* keys, int n, int k, int* hist, int* sel,
                                    uint32_t skip) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0ull, mask = 0ull;
  int need = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    if ((skip >> (shift / 8)) & 1u) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0;
    __syncwarp();
    for (int base = 0; base < n; base += 32) {
      const int e = base + lane;
      bool valid = false;
      uint32_t d = 0;
      if (e < n) {
        const uint64_t key = keys[e];
        if ((key & mask) == prefix) {
          valid = true;
          d = uint32_t(key >> shift) & 255u;
        }
      }
      const uint32_t vm = __ballot_sync(kFull, valid);
      if (valid) {
        const uint32_t peers = __match_any_sync(vm, d);
        if (lane == __ffs(peers) - 1) hist[d] += __popc(peers);  // distinct digits per step
      }
      __syncwarp();
    }
    int cnt[8], loc = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cnt[j] = hist[lane * 8 + j];
      loc += cnt[j];
    }
    int suf = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(kFull, suf, o);
      if (lane + o < 32) suf += y;
    }
    int acc = suf - loc;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (acc < need && acc + cnt[j] >= need) {
        sel[0] = lane * 8 + j;
        sel[1] = acc;
        sel[2] = cnt[j];
      }
      acc += cnt[j];
    }
    __syncwarp();
    const int d = sel[0];
    need -= sel[1];
    const int grp = sel[2];
    __syncwarp();
    prefix |= uint64_t(d) << shift;
    mask |= 255ull << shift;
    if (grp == need) {
      uint64_t mn = ~0ull;
      for (int e = lane; e < n; e += 32) {
        const uint64_t key = keys[e];
        if ((key & mask) == prefix && key < mn) mn = key;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t y = shfl_xor_u64(mn, o);
        mn = y < mn ? y : mn;
      }
      return mn;
    }
  }
  return prefix;
}

// Bitonic sort, descending, of the 32 * NV keys a warp holds in registers
// (lane holds position r * 32 + lane in v[r]).  Partners closer than 32 are
// exchanged with shuffles, farther ones inside the lane.
template <int NV>
__device__ __forceinline__ void warp_sort_desc_regs(uint64_t (&v)[NV]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32 * NV; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int r = 0; r < NV; ++r) {
        const bool desc = ((r * 32 + lane) & size) == 0;
        if (j >= 32) {
          const int rp = r ^ (j >> 5);
          if (rp > r) {
            const uint64_t a = v[r], b = v[rp];
            const bool sw = desc ? (a < b) : (a > b);
            v[r] = sw ? b : a;
            v[rp] = sw ? a : b;
          }
        } else {
          const uint64_t o = shfl_xor_u64(v[r], j);
          const bool lower = (lane & j) == 0;
          v[r] = (desc == lower) ? (v[r] > o ? v[r] : o) : (v[r] < o ? v[r] : o);
        }
      }
    }
  }
}

template <int NV>
__device__ __noinline__ void sort_smem_desc(uint64_t* a) {
  const int lane = threadIdx.x & 31;
  uint64_t v[NV];
#pragma unroll
  for (int r = 0; r < NV; ++r) v[r] = a[r * 32 + lane];
  warp_sort_desc_regs<NV>(v);
  __syncwarp();
#pragma unroll
  for (int r = 0; r < NV; ++r) a[r * 32 + lane] = v[r];
  __syncwarp();
}

// Sorts a[0 .. max(32, P)) descending in place, one warp (P a power of two
// <= 256; entries past the live ones must hold 0 so that they sort last).
__device__ void sort_desc(uint64_t* a, int P) {
  if (P <= 32)
    sort_smem_desc<1>(a);
  else if (P <= 64)
    sort_smem_desc<2>(a);
  else if (P <= 128)
    sort_smem_desc<4>(a);
  else
    sort_smem_desc<8>(a);
}

// ------------------------------------------------------- warp scans
template <class T>
__device__ __forceinline__ T warp_incl_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// ------------------------------------------------- kept-set weights
// 2^((v - v0) * c) for v <= v0, returned as f * 2^n with f near [1, 2).  The
// difference v - v0 is carried exactly (two-sum) and c = chi + clo, with the
// rounding error of the product kept, so the result is good to ex2.approx's
// own few-ulp error whatever the size of the exponent.
__device__ __forceinline__ float weight_split(float v, float v0, float chi, float clo, int* n) {
  const float dh = v - v0;
  const float bv = dh - v;
  const float dl = (v - (dh - bv)) + (-v0 - bv);
  const float ah = dh * chi;
  const float al = fmaf(dh, chi, -ah) + fmaf(dh, clo, dl * chi);
  const float fl = floorf(ah);
  *n = fl > -2048.f ? int(fl) : -2048;
  return ex2_approx(ah - fl) * fmaf(al, 0.6931471805599453f, 1.0f);
}

// f * 2^n (f a positive normal float, n <= 0) as a multiple of 2^-55, truncated.
__device__ __forceinline__ unsigned long long fix55(float f, int n) {
  const uint32_t b = __float_as_uint(f);
  const unsigned long long m = (b & 0x7fffffu) | 0x800000u;
  const int sh = int(b >> 23) - 127 - 23 + n + 55;
  return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> -sh) : 0ull);
}

// x * 2^n for n >= -1022 (0 below).
__device__ __forceinline__ double scale2(double x, int n) {
  return n < -1022 ? 0.0 : x * __longlong_as_double(static_cast<long long>(n + 1023) << 52);
}

// ------------------------------------------------------ filtered rows
constexpr int kRegKeys = 16;  // survivors a lane holds (512 per warp); more go the slow way

// Per-warp scratch of one filtered row.
struct WarpSel {
  uint64_t list[kTopkMax];  // the top k, unordered, then sorted descending
  union {
    int hist[256];                        // survivors per value bin
    unsigned long long before[kTopkMax];  // fixed-point mass before j
  };
  union {
    uint64_t grp[kTopkMax];   // during selection: the keys of the boundary bin
    struct {                  // weights in sorted order, wf[j] * 2^we[j]
      float wf[kTopkMax];
      int we[kTopkMax];
    };
    double wd[kTopkMax];      // weights in double (close top-p calls)
  };
  int digit, above, cnt;
  int pad;
  unsigned long long th;
};

union WarpScratch {
  WarpSel sel;
  DrawScratch draw;
};

// A row's survivor keys for the selection passes: held in registers (lane
// holds keys r * 32 + lane), or read from memory 512 at a time with every
// lane's loads issued together.  each(f) calls f(key) on every slot, in step
// across the warp (key 0 marks an empty slot).
struct RegKeys {
  const uint64_t (&key)[kRegKeys];
  int nslot;  // slots past it hold no key (warp-uniform)
  template <class F>
  __device__ __forceinline__ void each(F f) const {
#pragma unroll
    for (int r = 0; r < kRegKeys; ++r) {
      if (r >= nslot) break;
      f(key[r]);
    }
  }
};

struct MemKeys {
  const uint64_t* raw;
  int n;
  template <class F>
  __device__ __forceinline__ void each(F f) const {
    const int lane = threadIdx.x & 31;
    for (int c0 = 0; c0 < n; c0 += 32 * kRegKeys) {
      uint64_t key[kRegKeys];
#pragma unroll
      for (int r = 0; r < kRegKeys; ++r) {
        const int e = c0 + r * 32 + lane;
        key[r] = e < n ? __ldcg(raw + e) : 0ull;
      }
#pragma unroll
      for (int r = 0; r < kRegKeys; ++r) f(key[r]);
    }
  }
};

// The K-th largest of n > K unique survivor keys, exactly.  One pass bins the
// keys into 256 ordered bins, linear in the logit over [min, max] (a monotone
// map); the bin holding the K-th largest is then resolved among its own keys.
// Warp-uniform result.
template <class Src>
__device__ uint64_t select_kth(const Src& src, int K, WarpSel& ws, const uint64_t* raw, int n,
                               uint32_t skip) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t lo = ~0u, hi = 0u;
  src.each([&](uint64_t k) {
    if (k) {
      const uint32_t h = uint32_t(k >> 32);
      lo = min(lo, h);
      hi = max(hi, h);
    }
  });
  lo = __reduce_min_sync(kFull, lo);
  hi = __reduce_max_sync(kFull, hi);
  // bins linear in the logit value (the order-preserving integer image is
  // logarithmic in it and would crowd the boundary bin); an unbounded range
  // (-inf survivors) bins the integer image instead
  const float vlo = composite_value(uint64_t(lo) << 32), vhi = composite_value(uint64_t(hi) << 32);
  const bool by_value = vhi - vlo < INFINITY;
  const float scale = by_value ? (vhi > vlo ? 255.5f / (vhi - vlo) : 0.f)
                               : (hi > lo ? 255.5f / float(hi - lo) : 0.f);
  auto bin = [&](uint64_t k) {
    const float x = by_value ? (composite_value(k) - vlo) : float(uint32_t(k >> 32) - lo);
    return min(255, int(x * scale));
  };
#pragma unroll
  for (int j = 0; j < 8; ++j) ws.hist[lane * 8 + j] = 0;
  __syncwarp();
  src.each([&](uint64_t k) {
    if (k) atomicAdd(&ws.hist[bin(k)], 1);
  });
  __syncwarp();
  // the bin holding the K-th largest, the count above it and its own count
  int cnt[8], loc = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    cnt[j] = ws.hist[lane * 8 + j];
    loc += cnt[j];
  }
  int suf = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(kFull, suf, o);
    if (lane + o < 32) suf += y;
  }
  int acc = suf - loc;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (acc < K && acc + cnt[j] >= K) {
      ws.digit = lane * 8 + j;
      ws.above = acc;
      ws.cnt = cnt[j];
    }
    acc += cnt[j];
  }
  __syncwarp();
  const int bstar = ws.digit, need = K - ws.above, gcnt = ws.cnt;
  if (gcnt == need) {
    // the whole bin is kept: the threshold is its smallest key
    uint64_t mn = ~0ull;
    src.each([&](uint64_t k) {
      if (k && bin(k) == bstar && k < mn) mn = k;
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t y = shfl_xor_u64(mn, o);
      mn = y < mn ? y : mn;
    }
    return mn;
  }
  if (gcnt > kTopkMax) return warp_select_kth(raw, n, K, ws.hist, &ws.digit, skip);
  int g = 0;
  src.each([&](uint64_t k) {
    const bool in = k && bin(k) == bstar;
    const uint32_t bal = __ballot_sync(kFull, in);
    if (in) ws.grp[g + __popc(bal & lt)] = k;
    g += __popc(bal);
  });
  __syncwarp();
  if (gcnt <= 32) {
    uint64_t v[1] = {lane < gcnt ? ws.grp[lane] : 0ull};
    warp_sort_desc_regs<1>(v);
    return __shfl_sync(kFull, static_cast<unsigned long long>(v[0]), need - 1);
  }
  // rank the bin's keys: the need-th largest is the threshold
  for (int i = lane; i < gcnt; i += 32) {
    const uint64_t ki = ws.grp[i];
    int rk = 0;
    for (int j = 0; j < gcnt; ++j) rk += ws.grp[j] > ki;
    if (rk == need - 1) ws.th = ki;
  }
  __syncwarp();
  return ws.th;
}

// One filtered row, by one warp: the exact top k of the row pass's survivors
// (composite order: logit descending, index ascending), the temperature
// softmax over them, the top-p cut and the renormalisation; writes the kept
// list, the kept size and p(x) of the row's draft token.  Weights are
// float-accurate (relative error a few 1e-7) with exact fixed-point prefix
// sums; a top-p cut within 2^-17 of the threshold is redone in double
// precision, so the kept set is the double-precision one.
template <bool BF16>
__device__ __noinline__ void warp_filter_row(const Problem& P, int64_t row, int K, float T, float tp, int gx,
                                WarpSel& ws) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const uint64_t* raw = w.cand_raw + size_t(row) * kRawCap;
  // the first half of the key slots is fetched together with the survivor
  // count (the row's kRawCap slots are all addressable)
  uint64_t key[kRegKeys];
#pragma unroll
  for (int r = 0; r < kRegKeys / 2; ++r) key[r] = __ldcg(raw + r * 32 + lane);
  const int n = min(max(w.stats[row].kept, 0), kRawCap);
  const uint32_t skip = BF16 ? kSkipBf16 : kSkipF32;
  int cnt = 0;
  auto keep_top = [&](const auto& src, uint64_t th) {
    src.each([&](uint64_t k) {
      const bool keep = k && k >= th;
      const uint32_t bal = __ballot_sync(kFull, keep);
      if (keep) {
        const int sl = cnt + __popc(bal & lt);
        if (sl < kTopkMax) ws.list[sl] = k;
      }
      cnt += __popc(bal);
    });
  };
  if (n <= 32 * kRegKeys) {
#pragma unroll
    for (int r = 0; r < kRegKeys; ++r) {
      const int e = r * 32 + lane;
      if (r >= kRegKeys / 2) key[r] = e < n ? __ldcg(raw + e) : 0ull;
      else if (e >= n) key[r] = 0ull;  // keys are never 0
    }
    const RegKeys src{key, (n + 31) >> 5};
    keep_top(src, n > K ? select_kth(src, K, ws, raw, n, skip) : 0ull);
  } else {
    const MemKeys src{raw, n};
    keep_top(src, n > K ? select_kth(src, K, ws, raw, n, skip) : 0ull);
  }
  const int nsel = min(cnt, K);
  const int Psz = max(32, next_pow2(nsel > 0 ? nsel : 1));
  for (int j = nsel + lane; j < Psz; j += 32) ws.list[j] = 0ull;
  __syncwarp();
  sort_desc(ws.list, Psz);

  const float v0 = composite_value(ws.list[0]);
  // log2(e) / T split into two floats, formed once per row (the FP64 pipe is
  // narrow: per-lane double work would queue on it)
  float chi = 0.f, clo = 0.f;
  if (lane == 0) {
    const double cd = 1.4426950408889634 / double(T);
    chi = float(cd);
    clo = float(cd - double(chi));
  }
  chi = __shfl_sync(kFull, chi, 0);
  clo = __shfl_sync(kFull, clo, 0);
  // weights and the fixed-point mass before each j (integer work; the FP64
  // pipe, scarce on this part, is kept for a few operations per row)
  unsigned long long W = 0ull;
  for (int j0 = 0; j0 < nsel; j0 += 32) {
    const int j = j0 + lane;
    unsigned long long fx = 0ull;
    if (j < nsel) {
      const float v = composite_value(ws.list[j]);
      float f = 0.f;
      int e2 = 0;
      if (v > -INFINITY) {
        f = weight_split(v, v0, chi, clo, &e2);
        fx = fix55(f, e2);
      }
      ws.wf[j] = f;
      ws.we[j] = e2;
    }
    const unsigned long long incl = warp_incl_scan(fx);
    if (j < nsel) ws.before[j] = W + incl - fx;
    W += __shfl_sync(kFull, incl, 31);
  }
  __syncwarp();
  // top-p: keep j while the mass before j is below top_p of the total; the
  // masses increase with j, so the kept size is the count of such j.  A cut
  // whose fixed-point margin is under 2^-17 of the total is redone in double.
  int kp = nsel;
  bool exact = false;
  if (tp < 1.0f) {
    for (int pass = 0; pass < 2; ++pass) {
      unsigned long long lim = 0ull;
      if (lane == 0) lim = static_cast<unsigned long long>(ceil(double(tp) * double(W)));
      lim = __shfl_sync(kFull, lim, 0);
      int c = 0;
      for (int j0 = 0; j0 < nsel; j0 += 32) {
        const int j = j0 + lane;
        c += __popc(__ballot_sync(kFull, j < nsel && ws.before[j] < lim));
      }
      kp = c;
      if (pass == 1) break;
      const unsigned long long below = kp > 0 ? lim - ws.before[kp - 1] : ~0ull;
      const unsigned long long over = kp < nsel ? ws.before[kp] - lim : ~0ull;
      if (min(below, over) >= (W >> 17)) break;
      // close call: weights and masses in double precision
      exact = true;
      W = 0ull;
      for (int j0 = 0; j0 < nsel; j0 += 32) {
        const int j = j0 + lane;
        unsigned long long fx = 0ull;
        double wd = 0.0;
        if (j < nsel) {
          wd = exp((double(composite_value(ws.list[j])) - double(v0)) / double(T));
          fx = __double2ull_rn(wd * kFix);
        }
        __syncwarp();
        if (j < nsel) ws.wd[j] = wd;
        const unsigned long long incl = warp_incl_scan(fx);
        if (j < nsel) ws.before[j] = W + incl - fx;
        W += __shfl_sync(kFull, incl, 31);
      }
      __syncwarp();
    }
  }
  const unsigned long long Wp_fx = kp < nsel ? ws.before[kp] : W;
  double Wp = 0.0, invd = 0.0;
  if (lane == 0) {
    Wp = double(Wp_fx) / kFix;
    invd = 1.0 / Wp;
  }
  invd = __shfl_sync(kFull, invd, 0);
  const float invf = float(invd);
  const size_t cbase = size_t(row) * kTopkMax;
  float pgv = 0.f;
  bool hit = false;
  for (int j = lane; j < kp; j += 32) {
    const int idx = composite_index(ws.list[j]);
    float pj;
    if (exact)
      pj = float(ws.wd[j] * invd);
    else if (ws.we[j] > -100)
      pj = ws.wf[j] * invf * __int_as_float((ws.we[j] + 127) << 23);
    else
      pj = float(scale2(double(ws.wf[j]), ws.we[j]) * invd);  // far below 2^-100: in double
    w.cand_idx[cbase + j] = idx;
    w.cand_p[cbase + j] = pj;
    if (idx == gx) {
      hit = true;
      pgv = pj;
    }
  }
  const uint32_t hb = __ballot_sync(kFull, hit);
  if (hb) pgv = __shfl_sync(kFull, pgv, __ffs(hb) - 1);
  if (lane == 0) {
    RowStat st;
    st.s = Wp;
    st.pg = gx >= 0 ? pgv : nan64();
    st.m = v0;
    st.arg = -1;
    st.kept = kp;
    st.mode = kTopk;
    w.stats[row] = st;
  }
  __syncwarp();
}

// ------------------------------------------------------------- decisions
// Accept length of request b (warp-uniform), with every output except the
// final token written.  Lane i < k owns draft i.  Row results are read through
// L2: in the filtered case other warps of this kernel wrote them.
__device__ int decide(const Problem& P, int b, int k, int t0, int d0, bool greedy) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  bool acc = false;
  int x = -1;
  if (lane < k) {
    x = P.draft_tokens[d0 + lane];
    if (greedy) {
      acc = x == __ldcg(&w.stats[t0 + lane].arg);
      if (P.out_pq) {
        P.out_pq[2 * int64_t(d0 + lane)] = nan64();
        P.out_pq[2 * int64_t(d0 + lane) + 1] = nan64();
      }
    } else {
      const double p = __ldcg(&w.stats[t0 + lane].pg);
      const double q = __ldcg(&w.stats[P.Rt + d0 + lane].pg);
      acc = double(P.uniforms[t0 + lane]) * q < p;  // u < p / q without a divide
      if (P.out_pq) {
        P.out_pq[2 * int64_t(d0 + lane)] = p;
        P.out_pq[2 * int64_t(d0 + lane) + 1] = q;
      }
    }
  }
  const uint32_t rej = __ballot_sync(kFull, lane < k && !acc);
  const int L = rej ? __ffs(rej) - 1 : k;
  if (lane < k && lane != L) P.out_tokens[t0 + lane] = lane < L ? x : -1;
  if (lane == 0) {
    if (L < k) P.out_tokens[t0 + k] = -1;
    P.out_accept_len[b] = L;
  }
  return L;
}

// A request with a data error: every output -1 (NaN for (p, q)).
__device__ void fail_request(const Problem& P, int b, int k, int t0, int d0) {
  const int lane = threadIdx.x & 31;
  for (int i = lane; i <= k; i += 32) P.out_tokens[t0 + i] = -1;
  if (P.out_pq)
    for (int i = lane; i < 2 * k; i += 32) P.out_pq[2 * int64_t(d0) + i] = nan64();
  if (lane == 0) P.out_accept_len[b] = -1;
}

// Decide job of a request that is not filtered (or has a data error).
__device__ __noinline__ void decide_request(const Problem& P, int b) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  const int k = P.k_per_req[b];
  const int t0 = w.t_off[b], d0 = t0 - b;
  if (w.req_flag[b]) {
    fail_request(P, b, k, t0, d0);
    return;
  }
  const float T = P.temperature[b];
  const bool greedy = T == 0.0f;
  const int L = decide(P, b, k, t0, d0, greedy);
  if (lane != 0) return;
  if (greedy) {
    P.out_tokens[t0 + L] = w.stats[t0 + L].arg;
    return;
  }
  DrawDesc d;
  const RowStat st = w.stats[t0 + L];
  d.tr = t0 + L;
  d.dr = P.Rt + d0 + L;
  d.mt = st.m;
  d.ist = float(1.0 / st.s);
  d.md = 0.f;
  d.isd = 0.f;
  if (L < k) {
    const RowStat sd = w.stats[d.dr];
    d.md = sd.m;
    d.isd = float(1.0 / sd.s);
  }
  d.c2 = __fdiv_rn(1.4426950408889634f, T);
  d.kind = L < k ? 1 : 0;
  d.u = double(P.uniforms[t0 + k]);
  d.t0 = t0;
  d.L = L;
  w.draw[atomicAdd(&w.hdr->n_draw, 1)] = d;
}

// Final draw of a filtered request from the kept sets, by inverse CDF in
// vocabulary-index order (double precision): the residual max(0, p - q) over
// the target's kept tokens of row tr after a rejection (a token outside the
// draft row dr's kept set has q = 0), else p itself.  One warp; returns the
// token (warp-uniform).
__device__ __noinline__ int draw_kept(const Problem& P, int64_t tr, int64_t dr, bool residual,
                                      double u, DrawScratch& ds) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  // the first 64 entries of both kept lists are fetched with the kept sizes
  // (every list slot is addressable; entries past the size are ignored)
  const int* tidx = w.cand_idx + size_t(tr) * kTopkMax;
  const float* tpp = w.cand_p + size_t(tr) * kTopkMax;
  const int* didx = w.cand_idx + size_t(dr) * kTopkMax;
  const float* dpp = w.cand_p + size_t(dr) * kTopkMax;
  int tix[2], dix[2] = {0, 0};
  float tpv[2], dqv[2] = {0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    tix[h] = __ldcg(tidx + h * 32 + lane);
    tpv[h] = __ldcg(tpp + h * 32 + lane);
    if (residual) {
      dix[h] = __ldcg(didx + h * 32 + lane);
      dqv[h] = __ldcg(dpp + h * 32 + lane);
    }
  }
  const int Kt = min(max(__ldcg(&w.stats[tr].kept), 0), kTopkMax);
  const int Kd = residual ? min(max(__ldcg(&w.stats[dr].kept), 0), kTopkMax) : 0;
  for (int i = lane; i < Kd; i += 32) {
    ds.idx[i] = i < 32 ? dix[0] : (i < 64 ? dix[1] : __ldcg(didx + i));
    ds.v[i] = i < 32 ? dqv[0] : (i < 64 ? dqv[1] : __ldcg(dpp + i));
  }
  const int Psz = max(32, next_pow2(Kt > 0 ? Kt : 1));
  __syncwarp();
  double r[kTopkMax / 32];
#pragma unroll
  for (int s = 0; s < kTopkMax / 32; ++s) {
    const int j = s * 32 + lane;
    r[s] = 0.0;
    if (j < Kt) {
      const int idx = s == 0 ? tix[0] : (s == 1 ? tix[1] : __ldcg(tidx + j));
      const double p = s == 0 ? tpv[0] : (s == 1 ? tpv[1] : __ldcg(tpp + j));
      double q = 0.0;
      for (int i = 0; i < Kd; ++i)
        if (ds.idx[i] == idx) q = ds.v[i];
      r[s] = residual ? fmax(0.0, p - q) : p;
      ds.keys[j] = ~((uint64_t(uint32_t(idx)) << 32) | uint32_t(j));
    } else if (j < Psz) {
      ds.keys[j] = 0ull;  // sorts last
    }
  }
  __syncwarp();
#pragma unroll
  for (int s = 0; s < kTopkMax / 32; ++s)
    if (s * 32 + lane < Kt) ds.v[s * 32 + lane] = r[s];
  __syncwarp();
  sort_desc(ds.keys, Psz);  // ascending vocabulary index
  for (int attempt = 0; attempt < 2; ++attempt) {
    double S = 0.0;
    int last = -1;
    for (int j0 = 0; j0 < Kt; j0 += 32) {
      const int j = j0 + lane;
      const double rv = j < Kt ? ds.v[uint32_t(~ds.keys[j])] : 0.0;
      const double incl = warp_incl_scan(rv) + S;
      const uint32_t pos = __ballot_sync(kFull, rv > 0.0);
      if (pos) last = int((~ds.keys[j0 + 31 - __clz(pos)]) >> 32);
      S = __shfl_sync(kFull, incl, 31);
    }
    if (!(S > 0.0) && attempt == 0) {
      // residual mass vanished through rounding: draw from p_L
      for (int j = lane; j < Kt; j += 32) ds.v[j] = __ldcg(&w.cand_p[size_t(tr) * kTopkMax + j]);
      __syncwarp();
      continue;
    }
    const double t = u * S;
    double C = 0.0;
    int y = -1;
    for (int j0 = 0; j0 < Kt; j0 += 32) {
      const int j = j0 + lane;
      const double rv = j < Kt ? ds.v[uint32_t(~ds.keys[j])] : 0.0;
      const double incl = warp_incl_scan(rv) + C;
      const uint32_t hit = __ballot_sync(kFull, j < Kt && incl > t);
      if (hit) {
        y = int((~ds.keys[j0 + __ffs(hit) - 1]) >> 32);
        break;
      }
      C = __shfl_sync(kFull, incl, 31);
    }
    return y >= 0 ? y : last;
  }
  return -1;  // not reached: the second attempt always returns
}

constexpr int kPostThreads = 512;
constexpr int kWarps = kPostThreads / 32;
constexpr int kWave = kWarps / 2;  // positions per wave: a target and a draft row each

struct PostShared {
  int L;
};

// A filtered request, by one CTA, in waves of kWave positions: warps 2j and
// 2j + 1 filter the target and draft rows of position w0 + j, the first spare
// warp of the wave that reaches position k - 1 filters the bonus row k (when
// that wave fills every warp, k a multiple of kWave, warp 0 of one more wave
// does), then warp 0 decides the wave's positions in order.  Verification stops at the
// first rejection, so rows past it are never filtered.  (p, q) are reported
// for the positions up to the stop, NaN after it.
template <bool BF16>
__device__ void filtered_request(const Problem& P, int b, int t0, int k, WarpScratch* scr,
                                 PostShared& sh) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d0 = t0 - b;
  const int K = P.top_k[b];
  const float T = P.temperature[b];
  const float tp = P.top_p ? P.top_p[b] : 1.0f;
  for (int w0 = 0;; w0 += kWave) {
    const int pos = w0 + (warp >> 1);
    if (pos < k) {
      const int64_t row = (warp & 1) ? P.Rt + d0 + pos : int64_t(t0) + pos;
      warp_filter_row<BF16>(P, row, K, T, tp, P.draft_tokens[d0 + pos], scr[warp].sel);
    } else if (warp == 2 * max(k - w0, 0)) {
      warp_filter_row<BF16>(P, t0 + k, K, T, tp, -1, scr[warp].sel);
    }
    __syncthreads();
    if (warp == 0) {
      int L = k;  // k == 0: only the bonus row
      if (w0 < k) {
        const int n = min(kWave, k - w0);
        bool acc = true;
        double p = 0.0, q = 0.0;
        if (lane < n) {
          p = w.stats[t0 + w0 + lane].pg;
          q = w.stats[P.Rt + d0 + w0 + lane].pg;
          acc = double(P.uniforms[t0 + w0 + lane]) * q < p;  // u < p / q
        }
        const uint32_t rej = __ballot_sync(kFull, lane < n && !acc);
        // every position accepted: L = k only if this wave also filtered the
        // bonus row (a spare warp was left); otherwise the next wave does
        L = rej ? w0 + __ffs(rej) - 1 : (w0 + n == k && 2 * n < kWarps ? k : -1);
        if (P.out_pq && lane < n && (L < 0 || w0 + lane <= L)) {
          P.out_pq[2 * int64_t(d0 + w0 + lane)] = p;
          P.out_pq[2 * int64_t(d0 + w0 + lane) + 1] = q;
        }
      }
      if (lane == 0) sh.L = L;
    }
    __syncthreads();
    if (sh.L >= 0) break;
  }
  const int L = sh.L;
  if (warp == 0) {
    const int y = draw_kept(P, t0 + L, P.Rt + d0 + L, L < k, double(P.uniforms[t0 + k]),
                            scr[0].draw);
    for (int i = lane; i <= k; i += 32)
      P.out_tokens[t0 + i] = i < L ? P.draft_tokens[d0 + i] : (i == L ? y : -1);
    if (P.out_pq)
      for (int i = L + 1 + lane; i < k; i += 32) {
        P.out_pq[2 * int64_t(d0 + i)] = nan64();
        P.out_pq[2 * int64_t(d0 + i) + 1] = nan64();
      }
    if (lane == 0) P.out_accept_len[b] = L;
  }
}

// Persistent CTAs over the job lists: a filtered request takes a whole CTA;
// the other requests are decided kWarps at a time, one warp each.
template <bool BF16>
__global__ void __launch_bounds__(kPostThreads, 2) filter_decide_kernel(const Problem P) {
  extern __shared__ __align__(16) unsigned char post_smem[];
  WarpScratch* scr = reinterpret_cast<WarpScratch*>(post_smem);
  __shared__ PostShared sh;
  const Ws& w = P.ws;
  const int warp = threadIdx.x >> 5;
  if (w.hdr->global_err) {
    // batch-level data error: every output is -1 (NaN for the probabilities)
    const int64_t stride = int64_t(gridDim.x) * kPostThreads;
    const int64_t i0 = int64_t(blockIdx.x) * kPostThreads + threadIdx.x;
    for (int64_t r = i0; r < P.B; r += stride) P.out_accept_len[r] = -1;
    for (int64_t r = i0; r < P.Rt; r += stride) P.out_tokens[r] = -1;
    if (P.out_pq)
      for (int64_t r = i0; r < 2 * P.Rd; r += stride) P.out_pq[r] = nan64();
    return;
  }
  const int nf = w.hdr->n_filtered, nd = w.hdr->n_decide;
  const int units = nf + (nd + kWarps - 1) / kWarps;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    if (u < nf) {
      const int4 job = w.job[u];
      if (w.req_flag[job.x]) {  // a logit error found by the row pass
        if (warp == 0) fail_request(P, job.x, job.w, job.z, job.z - job.x);
      } else {
        filtered_request<BF16>(P, job.x, job.z, job.w, scr, sh);
      }
      __syncthreads();  // the scratch is reused by the next unit
    } else {
      const int j = (u - nf) * kWarps + warp;
      if (j < nd) decide_request(P, w.job[P.B + j].x);
    }
  }
}

}  // namespace

size_t filter_smem_bytes() { return sizeof(WarpScratch) * kWarps; }

cudaError_t launch_filter_decide(const Problem& P, bool bf16, int grid, cudaStream_t s) {
  const size_t smem = filter_smem_bytes();
  if (bf16)
    filter_decide_kernel<true><<<grid, kPostThreads, smem, s>>>(P);
  else
    filter_decide_kernel<false><<<grid, kPostThreads, smem, s>>>(P);
  return cudaGetLastError();
}

// Shared-memory limit and resident CTAs per SM of the filter / decide kernel
// (host queries; nothing is allocated).
cudaError_t filter_occupancy(int* occ) {
  const int smem = int(filter_smem_bytes());
  cudaError_t e = cudaFuncSetAttribute(filter_decide_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(filter_decide_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int a = 0, b = 0;
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, filter_decide_kernel<true>,
                                                      kPostThreads, smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, filter_decide_kernel<false>,
                                                      kPostThreads, smem);
  if (e != cudaSuccess) return e;
  *occ = max(1, min(a, b));
  return cudaSuccess;
}

}  // namespace sv
