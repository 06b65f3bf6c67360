// Filter / decide kernel: what follows the row pass for every request except
// the unfiltered sampled draws (the draw pass).
//
// Persistent CTAs over the job lists of the setup kernel:
//   filtered request  (one CTA) in waves of positions: a warp per target and
//                 draft row takes the exact top k of the row pass's survivors
//                 (composite order: logit descending, index ascending), the
//                 temperature softmax over them, the top-p cut (keep j while
//                 the mass before j is below top_p) and the renormalisation,
//                 applied alike to target and draft rows ("Speculative
//                 decoding and multi-token prediction", "Why the output is
//                 identical"); one warp then accepts while u_i < p_i(x_i) /
//                 q_i(x_i) ("FlashMap…" §4, steps 1-2) and, at the first
//                 rejection or after the last draft, draws the final token
//                 from the kept sets (§4 step 3).  Rows after the first
//                 rejection are never filtered.
//   decide job    (one warp per request) greedy: accept while x_i equals the
//                 target argmax (lowest index on ties) and emit the argmax at
//                 the first disagreement or as the bonus ("DFlash" §4 step 5;
//                 "Speculative decoding…", "Draft and verify", step Three).
//                 Unfiltered sampling: accept while u_i < p_i(x_i) / q_i(x_i),
//                 stop at the first rejection, then queue the final draw for
//                 the draw pass (vocabularies up to kInlineDrawV: draw it in
//                 the warp, and the draw pass is not launched).
#include <math.h>

#include "sv_select.cuh"
#include "sv_weights.cuh"

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
constexpr int kKeyCopy = 512;  // survivors copied to shared memory (more are read from L2)
constexpr int kBinSort = 8;    // whole bins up to this size are ordered by insertion sort
constexpr int kFastDraw = 64;  // kept sets up to this size are drawn from shared memory
constexpr int kRankMax = 64;   // boundary bins up to this size are ordered by ranks
constexpr int kRankAll = 128;  // candidate sets up to this size are ordered by ranks

// Per-warp scratch of one filtered row.  After the row it still holds the
// row's kept set (sorted keys and probabilities) and p(x) of its token, which
// the request's decision and final draw read.
//
// The per-row code runs once per row, so its instruction footprint, not its
// arithmetic, sets its speed: the passes below are short loops over a
// shared-memory copy of the survivors rather than unrolled register code.
struct WarpSel {
  uint64_t keys[kKeyCopy];  // the row's survivors
  uint64_t list[kTopkMax];  // the top k, sorted descending (composite order)
  union {
    uint64_t grp[kTopkMax];               // selection: keys of the boundary bin
    unsigned long long before[kTopkMax];  // fixed-point mass before j
  };
  union {
    struct {
      float pk[kTopkMax];  // weight j as pk[j] * 2^hw[j]; then kept probability j
      int hw[kTopkMax];    // selection: keys per value bin, then bin ends; weight exponents
    };
    double wd[kTopkMax];   // weights in double (close top-p calls)
  };
  double pg;   // p(x) of the row's token, NaN without one
  int kp;      // kept size
  int fast;    // pk[0 .. kp) holds the kept probabilities and kp <= kFastDraw
  int gcount;  // keys collected from the boundary bin
  int pad[3];
};

union WarpScratch {
  WarpSel sel;
  DrawScratch draw;
};
static_assert(sizeof(WarpScratch) % 16 == 0, "keys of every warp's scratch are 16-byte aligned");

// The min(n, K) largest of the n unique survivor keys at keys[] (shared or
// global memory), sorted descending into ws.list; returns their count.  One
// pass bins the keys into 256 ordered bins linear in the logit over [min,
// max] (a monotone map, so a higher bin holds only larger keys) and finds the
// bin holding the K-th largest.  When few keys lie in that bin or above, each
// takes its rank among them as its slot; otherwise bins wholly inside the top
// K go straight to their final slots (a counting sort over bins) and are then
// ordered within the bin, and the boundary bin contributes its largest keys
// after them.  ws.keys may be overwritten.
__device__ __noinline__ int select_sorted(const uint64_t* keys, int n, int K, WarpSel& ws,
                                          const uint64_t* raw, uint32_t skip, uint32_t lo,
                                          uint32_t hi) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  // lo / hi: this lane's smallest and largest high key words over the keys
  // e = lane (mod 32) when the caller has seen them all; ~0u / 0u asks for the
  // pass below (which also yields ~0u / 0u for a lane that has no key)
  if (lo == ~0u && hi == 0u) {
#pragma unroll 4
    for (int e = lane; e < n; e += 32) {
      const uint32_t h = uint32_t(keys[e] >> 32);
      lo = min(lo, h);
      hi = max(hi, h);
    }
  }
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
  for (int j = 0; j < 8; ++j) ws.hw[lane * 8 + j] = 0;
  if (lane == 0) ws.gcount = 0;
  __syncwarp();
  // each key's bin is kept (one byte, in ws.grp) for the compaction below
  uint8_t* kbin = reinterpret_cast<uint8_t*>(ws.grp);
#pragma unroll 4
  for (int e = lane; e < n; e += 32) {
    const int bk = bin(keys[e]);
    kbin[e] = uint8_t(bk);
    atomicAdd(&ws.hw[bk], 1);
  }
  __syncwarp();
  // lane holds bins 8 lane .. 8 lane + 7; off[j]: keys in the bins above
  int cnt[8], off[8], loc = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    cnt[j] = ws.hw[lane * 8 + j];
    loc += cnt[j];
  }
  int suf = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(kFull, suf, o);
    if (lane + o < 32) suf += y;
  }
  int acc = suf - loc, mine = -1;
  bool big = false;  // a whole bin too large for insertion sort
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    off[j] = acc;
    if (acc < K && acc + cnt[j] >= K) mine = j;  // the bin holding the K-th largest
    acc += cnt[j];
  }
  const uint32_t bm = __ballot_sync(kFull, mine >= 0);
  int bstar = -1, above = n, gcnt = 0;  // n < K: every bin is kept whole
  if (bm) {
    const int bl = __ffs(bm) - 1;
    int o = 0, c = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j == mine) {
        o = off[j];
        c = cnt[j];
      }
    bstar = bl * 8 + __shfl_sync(kFull, mine, bl);
    above = __shfl_sync(kFull, o, bl);
    gcnt = __shfl_sync(kFull, c, bl);
  }
  const int nsel = bm ? K : n;
  const int P2 = max(32, next_pow2(nsel > 0 ? nsel : 1));
  if (gcnt > kTopkMax) {
    // a crowded boundary bin (many equal or nearly equal logits): the exact
    // K-th largest by radix selection, then the keys reaching it, sorted
    __syncwarp();
    const uint64_t th = warp_select_kth(raw, n, K, ws.hw, &ws.kp, skip);
    int c = 0;
    for (int e0 = 0; e0 < n; e0 += 32) {
      const int e = e0 + lane;
      const uint64_t k = e < n ? keys[e] : 0ull;
      const bool keep = k != 0ull && k >= th;
      const uint32_t bal = __ballot_sync(kFull, keep);
      if (keep) {
        const int sl = c + __popc(bal & lt);
        if (sl < kTopkMax) ws.list[sl] = k;
      }
      c += __popc(bal);
    }
    for (int j = nsel + lane; j < P2; j += 32) ws.list[j] = 0ull;
    __syncwarp();
    sort_desc(ws.list, P2);
    return nsel;
  }
  const int ns = bm ? above + gcnt : n;  // keys in the boundary bin or above
  if (ns <= kRankAll) {
    // Few candidates (the usual case for a small k): compact the keys of the
    // bins at or above the boundary into ws.keys (in place when they are
    // there: a key only moves down), then each key's slot is its rank among
    // them, the number of larger keys (keys are unique).
    int c = 0;
    for (int e0 = 0; e0 < n; e0 += 64) {
      const int ea = e0 + lane, eb = ea + 32;
      const uint64_t ka = ea < n ? keys[ea] : 0ull, kb = eb < n ? keys[eb] : 0ull;
      const bool ia = ea < n && int(kbin[ea]) >= bstar, ib = eb < n && int(kbin[eb]) >= bstar;
      const uint32_t ba = __ballot_sync(kFull, ia), bb = __ballot_sync(kFull, ib);
      __syncwarp();  // every lane has read its keys before any lane writes
      if (ia) ws.keys[c + __popc(ba & lt)] = ka;
      if (ib) ws.keys[c + __popc(ba) + __popc(bb & lt)] = kb;
      c += __popc(ba) + __popc(bb);
    }
    __syncwarp();
    for (int e0 = 0; e0 < ns; e0 += 64) {
      const int ea = e0 + lane, eb = ea + 32;
      const uint64_t a = ea < ns ? ws.keys[ea] : ~0ull;
      const uint64_t b = eb < ns ? ws.keys[eb] : ~0ull;
      int ra = 0, rb = 0;
#pragma unroll 8
      for (int t = 0; t < ns; ++t) {
        const uint64_t x = ws.keys[t];
        ra += x > a;
        rb += x > b;
      }
      if (ea < ns && ra < nsel) ws.list[ra] = a;
      if (eb < ns && rb < nsel) ws.list[rb] = b;
    }
    __syncwarp();
    return nsel;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ws.hw[lane * 8 + j] = off[j];  // cursor: the bin's first slot
    if (lane * 8 + j > bstar && cnt[j] > kBinSort) big = true;
  }
  big = __any_sync(kFull, big);
  __syncwarp();
#pragma unroll 4
  for (int e = lane; e < n; e += 32) {
    const uint64_t k = keys[e];
    const int bk = bin(k);
    if (bk > bstar) ws.list[atomicAdd(&ws.hw[bk], 1)] = k;
    else if (bk == bstar) ws.grp[atomicAdd(&ws.gcount, 1)] = k;
  }
  __syncwarp();
  if (bstar >= 0) {
    // the boundary bin's largest K - above keys, in order: a key's rank among
    // the bin's keys is its slot
    const int need = K - above;
    if (gcnt <= kRankMax) {
      for (int e = lane; e < gcnt; e += 32) {
        const uint64_t k = ws.grp[e];
        int rk = 0;
        for (int i = 0; i < gcnt; ++i) rk += ws.grp[i] > k;
        if (rk < need) ws.list[above + rk] = k;
      }
    } else {
      const int G = next_pow2(gcnt);
      for (int j = gcnt + lane; j < G; j += 32) ws.grp[j] = 0ull;
      __syncwarp();
      sort_desc(ws.grp, G);
      for (int j = lane; j < need; j += 32) ws.list[above + j] = ws.grp[j];
    }
  }
  if (big) {
    for (int j = nsel + lane; j < P2; j += 32) ws.list[j] = 0ull;
    __syncwarp();
    sort_desc(ws.list, P2);
  } else {
    // order inside each whole bin (bins above the boundary), by the lane that
    // owns the bin; after the scatter hw[b] is the end of bin b, and bin b
    // starts where bin b + 1 ends
    for (int j = 0; j < 8; ++j) {
      const int b = lane * 8 + j;
      if (b <= bstar) continue;
      const int o = b == 255 ? 0 : ws.hw[b + 1], e = ws.hw[b];
      for (int a = o + 1; a < e; ++a) {
        const uint64_t x = ws.list[a];
        int c = a - 1;
        while (c >= o && ws.list[c] < x) {
          ws.list[c + 1] = ws.list[c];
          --c;
        }
        ws.list[c + 1] = x;
      }
    }
    __syncwarp();
  }
  return nsel;
}

// One filtered row, by one warp: the exact top k of the row pass's survivors
// (composite order: logit descending, index ascending), the temperature
// softmax over them, the top-p cut and the renormalisation; writes the kept
// list, the kept size and p(x) of the row's draft token, and leaves the kept
// set in ws.  Weights are float-accurate (relative error a few 1e-7) with
// exact fixed-point prefix sums; a top-p cut within 2^-17 of the threshold is
// redone in double precision, so the kept set is the double-precision one.
// log2(e) / T as the unevaluated sum chi + clo of two floats, formed in double
// by lane 0 (the FP64 pipe is narrow: per-lane double work would queue on it)
// and broadcast to the warp.
__device__ __forceinline__ void log2e_over_t(float T, float* chi, float* clo) {
  float h = 0.f, l = 0.f;
  if ((threadIdx.x & 31) == 0) {
    const double cd = 1.4426950408889634 / double(T);
    h = float(cd);
    l = float(cd - double(h));
  }
  *chi = __shfl_sync(kFull, h, 0);
  *clo = __shfl_sync(kFull, l, 0);
}

// n_pre >= 0: the first kKeyCopy survivor slots are already in ws.keys
// (copied ahead, see filtered_request) and n_pre is the survivor count.
template <bool BF16>
__device__ __noinline__ void warp_filter_row(const Problem& P, int64_t row, int K, float T, float chi,
                                             float clo, float tp, int gx, WarpSel& ws,
                                             int n_pre = -1) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  const uint64_t* raw = w.cand_raw + size_t(row) * kRawCap;
  int n;
  uint32_t lo = ~0u, hi = 0u;  // the range of the keys, seen as they are copied
  if (n_pre >= 0) {
    n = min(n_pre, kRawCap);  // the range is taken by select_sorted
  } else {
  // the first 256 key slots are fetched together with the survivor count
  // (the row's kRawCap slots are all addressable)
  uint64_t pre[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) pre[r] = __ldcg(raw + r * 32 + lane);
  n = min(max(w.stats[row].kept, 0), kRawCap);
  const int nc = min(n, kKeyCopy);
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (r * 32 + lane < nc) {
      ws.keys[r * 32 + lane] = pre[r];
      lo = min(lo, uint32_t(pre[r] >> 32));
      hi = max(hi, uint32_t(pre[r] >> 32));
    }
#pragma unroll 4
  for (int e = 256 + lane; e < nc; e += 32) {
    const uint64_t k = __ldcg(raw + e);
    ws.keys[e] = k;
    lo = min(lo, uint32_t(k >> 32));
    hi = max(hi, uint32_t(k >> 32));
  }
  __syncwarp();
  if (n > kKeyCopy) lo = ~0u, hi = 0u;  // keys past the copy: select reads them all
  }
  const int nsel = select_sorted(n <= kKeyCopy ? ws.keys : raw, n, K, ws, raw,
                                 BF16 ? kSkipBf16 : kSkipF32, lo, hi);

  const float v0 = composite_value(ws.list[0]);
  // weights and the fixed-point mass before each j (integer work; the FP64
  // pipe, scarce on this part, is kept for a few operations per row)
  // two consecutive entries per lane, one scan of the pair sums per 64
  unsigned long long W = 0ull;
  for (int j0 = 0; j0 < nsel; j0 += 64) {
    const int j = j0 + 2 * lane;
    unsigned long long fx[2] = {0ull, 0ull};
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (j + h < nsel) {
        const float v = composite_value(ws.list[j + h]);
        float f = 0.f;
        int e2 = 0;
        if (v > -INFINITY) {
          f = weight_split(v, v0, chi, clo, &e2);
          fx[h] = fix55(f, e2);
        }
        ws.pk[j + h] = f;
        ws.hw[j + h] = e2;
      }
    const unsigned long long pair = fx[0] + fx[1];
    const unsigned long long incl = warp_incl_scan(pair);
    const unsigned long long excl = W + incl - pair;
    if (j < nsel) ws.before[j] = excl;
    if (j + 1 < nsel) ws.before[j + 1] = excl + fx[0];
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
      // ceil(top_p * W): exactly in integers the first time (top_p = m 2^-s
      // with a 24-bit m), in double on the double-precision redo
      unsigned long long lim = 0ull;
      if (pass == 0) {
        lim = ceil_mul_frac(W, tp);
      } else {
        if (lane == 0) lim = static_cast<unsigned long long>(ceil(double(tp) * double(W)));
        lim = __shfl_sync(kFull, lim, 0);
      }
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
  const bool fast = !exact && kp <= kFastDraw;
  float pgv = 0.f;
  bool hit = false;
  for (int j = lane; j < kp; j += 32) {
    const int idx = composite_index(ws.list[j]);
    float pj;
    if (exact)
      pj = float(ws.wd[j] * invd);
    else if (ws.hw[j] > -100)
      pj = ws.pk[j] * invf * __int_as_float((ws.hw[j] + 127) << 23);
    else
      pj = float(scale2(double(ws.pk[j]), ws.hw[j]) * invd);  // far below 2^-100: in double
    w.cand_idx[cbase + j] = idx;
    w.cand_p[cbase + j] = pj;
    if (fast) ws.pk[j] = pj;  // same slot, same lane
    if (idx == gx) {
      hit = true;
      pgv = pj;
    }
  }
  const uint32_t hb = __ballot_sync(kFull, hit);
  if (hb) pgv = __shfl_sync(kFull, pgv, __ffs(hb) - 1);
  if (lane == 0) {
    const double pg = gx >= 0 ? double(pgv) : nan64();
    ws.pg = pg;
    ws.kp = kp;
    ws.fast = fast;
    RowStat st;
    st.s = Wp;
    st.pg = pg;
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

// The final token of a sampled decide job drawn in the deciding warp, for
// rows of at most kInlineDrawV elements: y* = min{ y : C_y > t }, t = floor(u S),
// over the weights of the draw pass (residual max(0, p_L - q_L), or p_k; kept-
// set masks of threshold rows; the residual falls back to p_L if its mass
// vanished through rounding), each as an exact 2^-40 fixed-point integer.
// Lane l takes a contiguous run of elements (a multiple of 8 long): one pass
// forms the lane sums, their scan gives S and each lane's first prefix, and
// the lane holding t walks its run again.  Short loops, not unrolled: this
// warp's code runs once per request, so its footprint sets its speed.
// -1 if the row has no mass.
template <bool BF16>
__device__ __noinline__ int draw_in_warp(const Problem& P, const DrawDesc& d) {
  using E = Elt<BF16>;
  const int lane = threadIdx.x & 31;
  Weights W = make_weights(d);
  const unsigned char* trow =
      static_cast<const unsigned char*>(P.target) + d.tr * P.t_stride * E::kSize;
  const unsigned char* drow =
      d.kind == 1 ? static_cast<const unsigned char*>(P.draft) + (d.dr - P.Rt) * P.d_stride * E::kSize
                  : nullptr;
  const int V = P.V, fast_end = V & ~7;
  const int run = ((V + 255) / 256) * 8;  // elements per lane, a multiple of 8
  const int e0 = lane * run, e1 = min(e0 + run, V);
  // fixed-point weights of elements e .. e + 7 (16-byte loads where all 8 lie
  // below fast_end; rows start 16-byte aligned)
  auto weights8 = [&](int e, unsigned long long* wf) {
    float xt[8], xd[8];
    elems8<BF16>(trow + size_t(e) * E::kSize, trow, e, fast_end, V, xt);
    if (W.kind == 1) elems8<BF16>(drow + size_t(e) * E::kSize, drow, e, fast_end, V, xd);
#pragma unroll
    for (int k = 0; k < 8; ++k) wf[k] = fixw(W.at(xt[k], W.kind == 1 ? xd[k] : 0.f, e + k));
  };
  auto lane_sum = [&]() {
    unsigned long long ls = 0ull, wf[8];
#pragma unroll 1
    for (int e = e0; e < e1; e += 8) {
      weights8(e, wf);
#pragma unroll
      for (int k = 0; k < 8; ++k) ls += wf[k];
    }
    return ls;
  };
  unsigned long long ls = lane_sum();
  unsigned long long S = warp_sum_u64(ls);
  if (W.kind == 1 && S == 0ull) {
    W.set_kind(2);
    ls = lane_sum();
    S = warp_sum_u64(ls);
  }
  if (S == 0ull) return -1;
  const unsigned long long ufix = (unsigned long long)(d.u * 4294967296.0);  // exact
  const unsigned long long t = (__umul64hi(S, ufix) << 32) | ((S * ufix) >> 32);
  // the lane whose run holds the first prefix above t (t < S), then the element
  const unsigned long long incl = warp_incl_scan_u64(ls);
  const uint32_t hit = __ballot_sync(kFull, ls > 0ull && incl > t);
  const int owner = __ffs(hit) - 1;
  int y = -1;
  if (lane == owner) {
    unsigned long long pre = incl - ls, wf[8];
#pragma unroll 1
    for (int e = e0; e < e1 && y < 0; e += 8) {
      weights8(e, wf);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        pre += wf[k];
        if (y < 0 && wf[k] > 0ull && pre > t) y = e + k;
      }
    }
  }
  return __shfl_sync(kFull, y, owner);
}

// Decide job of a request that is not filtered (or has a data error).
// INLINE: the sampled requests' final draws are taken here (draw_in_warp);
// otherwise they are queued for the draw pass.  The two are separate kernel
// instances: the in-warp draw's code in the kernel of the long-row workloads
// measured 2-4 µs on their filter / decide kernel (instruction fetch).
template <bool BF16, bool INLINE>
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
  if (!INLINE && lane != 0) return;
  if (greedy) {
    if (lane == 0) P.out_tokens[t0 + L] = w.stats[t0 + L].arg;
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
  // rows filtered by a threshold (kBig) draw from their kept sets only
  d.kt = st.mode == kBig ? w.cand_raw[size_t(d.tr) * kRawCap] : 0ull;
  d.kd = 0ull;
  if (L < k) {
    const RowStat sd = w.stats[d.dr];
    d.md = sd.m;
    d.isd = float(1.0 / sd.s);
    d.kd = sd.mode == kBig ? w.cand_raw[size_t(d.dr) * kRawCap] : 0ull;
  }
  d.c2 = __fdiv_rn(1.4426950408889634f, T);
  d.kind = L < k ? 1 : 0;
  d.u = double(P.uniforms[t0 + k]);
  d.t0 = t0;
  d.L = L;
  if constexpr (INLINE) {
    // every lane formed the same descriptor
    const int y = draw_in_warp<BF16>(P, d);
    if (lane == 0) {
      if (y < 0) record_error(w.hdr, SV_ERR_INTERNAL, -1, d.tr);  // no mass found
      P.out_tokens[t0 + L] = y;
    }
  } else {
    w.draw[atomicAdd(&w.hdr->n_draw, 1)] = d;
  }
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

constexpr int kPostThreads = 256;
constexpr int kWarps = kPostThreads / 32;
constexpr int kWave = kWarps / 2;  // positions per wave: a target and a draft row each

struct PostShared {
  int L;
  int idx[kFastDraw];                // draw_fast: target kept tokens
  unsigned long long r[kFastDraw];   // and their residual (or p) mass
};

// A float probability in [0, 1] as a multiple of 2^-55 (exact above 2^-31;
// subnormals count as 0).
__device__ __forceinline__ unsigned long long fix_prob(float p) {
  return p >= 1.17549435e-38f ? fix55(p, 0) : 0ull;
}

// Final draw of a filtered request from kept sets held in shared memory (at
// most kFastDraw tokens each), by inverse CDF in vocabulary-index order:
// y = min{ y : C_y > u S } over the residual max(0, p - q) of the target's
// kept tokens after a rejection (q = 0 outside the draft's kept set; p itself
// when the residual mass is zero), or over p for the bonus draw.  Masses are
// summed exactly in fixed point (multiples of 2^-55), so the order of the
// additions does not matter; C_y is each token's own prefix, summed directly
// rather than after an index sort.  One warp; warp-uniform result.
// sidx / sr: kFastDraw entries of scratch (shared memory); *qy (if given)
// receives the drawn token's probability in t (the kept probability itself).
__device__ __noinline__ int draw_fast(const WarpSel& t, const WarpSel* d, double u, int* sidx,
                                      unsigned long long* sr, float* qy) {
  const int lane = threadIdx.x & 31;
  const int Kt = t.kp, Kd = d ? d->kp : 0;
  int idx[2];
  float p[2], q[2] = {0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int j = s * 32 + lane;
    idx[s] = j < Kt ? composite_index(t.list[j]) : INT_MAX;
    p[s] = j < Kt ? t.pk[j] : 0.f;
  }
#pragma unroll 4
  for (int i = 0; i < Kd; ++i) {
    const int di = composite_index(d->list[i]);
    const float dq = d->pk[i];
#pragma unroll
    for (int s = 0; s < 2; ++s)
      if (di == idx[s]) q[s] = dq;
  }
  for (int attempt = 0; attempt < 2; ++attempt) {
    const bool residual = d != nullptr && attempt == 0;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int j = s * 32 + lane;
      const unsigned long long fp = fix_prob(p[s]), fq = residual ? fix_prob(q[s]) : 0ull;
      if (j < Kt) {
        sidx[j] = idx[s];
        sr[j] = fp > fq ? fp - fq : 0ull;
      }
    }
    __syncwarp();
    unsigned long long C[2] = {0ull, 0ull}, rmine[2] = {0ull, 0ull};
#pragma unroll 4
    for (int i = 0; i < Kt; ++i) {
      const int ii = sidx[i];
      const unsigned long long ri = sr[i];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (ii <= idx[s]) C[s] += ri;
        if (ii == idx[s]) rmine[s] = ri;
      }
    }
    // S: the prefix of the largest kept index
    unsigned long long S = max(C[0], C[1]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = shfl_xor_u64(S, o);
      S = y > S ? y : S;
    }
    __syncwarp();  // sh is rewritten by a second attempt
    if (S == 0ull && attempt == 0) continue;  // residual mass vanished: draw from p
    unsigned long long th = 0ull;
    if (lane == 0) th = static_cast<unsigned long long>(u * double(S));  // floor(u S)
    th = __shfl_sync(kFull, th, 0);
    int y = INT_MAX, last = -1;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (idx[s] != INT_MAX && C[s] > th) y = min(y, idx[s]);
      if (rmine[s] > 0ull) last = max(last, idx[s]);
    }
    y = __reduce_min_sync(kFull, y);
    last = __reduce_max_sync(kFull, last);
    y = y != INT_MAX ? y : last;  // rounding left no C above u S: the last token with mass
    if (qy) {
      float pv = 0.f;
#pragma unroll
      for (int s = 0; s < 2; ++s)
        if (idx[s] == y) pv = p[s];
      const uint32_t hb = __ballot_sync(kFull, pv != 0.f);
      *qy = hb ? __shfl_sync(kFull, pv, __ffs(hb) - 1) : 0.f;
    }
    return y;
  }
  return -1;  // not reached: the second attempt always returns
}

// The row that wave slot s (a warp index: position w0 + s / 2, target row
// for even s, draft row for odd s) of a filtered request filters, or -1; the
// bonus row k goes to the first slot left after position k - 1 (slot 0 of
// one more wave when k is a multiple of kWave).  *gx: the token whose
// probability the row reports.
__device__ __forceinline__ int64_t wave_row(const Problem& P, int b, int t0, int k, int w0, int s,
                                            int* gx) {
  const int d0 = t0 - b, pos = w0 + (s >> 1);
  if (pos < k) {
    *gx = P.draft_tokens[d0 + pos];
    return (s & 1) ? P.Rt + d0 + pos : int64_t(t0) + pos;
  }
  *gx = -1;
  return s == 2 * (k - w0) ? int64_t(t0) + k : -1;
}

// Asynchronous copy of the first kKeyCopy survivor slots of a row into a
// warp's scratch (16 bytes per lane per step, through L2 only).
__device__ __forceinline__ void copy_keys_async(const uint64_t* raw, uint64_t* keys) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kKeyCopy / 64; ++i) {
    const int c = i * 32 + lane;  // 16-byte chunk: keys 2c, 2c + 1
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(keys + 2 * c)),
                 "l"(raw + 2 * c)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void copy_keys_wait() {
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncwarp();
}

// A filtered request, by one CTA, in waves of kWave positions: warps 2j and
// 2j + 1 filter the target and draft rows of position w0 + j, the first spare
// warp of the wave that reaches position k - 1 filters the bonus row k (when
// that wave fills every warp, k a multiple of kWave, warp 0 of one more wave
// does), then warp 0 decides the wave's positions in order from the p(x), q(x)
// the filtering warps left in shared memory.  Verification stops at the first
// rejection, so rows past it are never filtered.  (p, q) are reported for the
// positions up to the stop, NaN after it.  The final draw reads the kept sets
// of the stopping position from the same shared memory (or, for kept sets
// larger than kFastDraw, from the lists in global memory).  Once a warp has
// filtered its row of a wave it starts copying its row of the next wave
// (survivor keys and count) into its scratch, so that a request going on
// finds them there.
// A filtered request's inputs: its parameters, log2(e) / T as chi + clo, the
// final draw's uniform and (warp 0, lane i) drafted token i.  They depend on
// the caller's inputs alone, so a CTA reads its first request's before the
// row pass has finished.
struct ReqParams {
  int K;
  float T, tp, chi, clo, u_last;
  int x_lane;
};

__device__ __forceinline__ ReqParams request_params(const Problem& P, int b, int t0, int k) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ReqParams r;
  r.K = P.top_k[b];
  r.T = P.temperature[b];
  r.tp = P.top_p ? P.top_p[b] : 1.0f;
  log2e_over_t(r.T, &r.chi, &r.clo);
  r.u_last = warp == 0 ? P.uniforms[t0 + k] : 0.f;
  r.x_lane = warp == 0 && lane < k ? P.draft_tokens[t0 - b + lane] : -1;
  return r;
}

template <bool BF16>
__device__ void filtered_request(const Problem& P, int b, int t0, int k, const ReqParams& rp,
                                 WarpScratch* scr, PostShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d0 = t0 - b;
  const int K = rp.K;
  const float T = rp.T;
  const float tp = rp.tp;
  const float chi = rp.chi, clo = rp.clo;
  const float u_last = rp.u_last;
  const int x_lane = rp.x_lane;
  const Ws& w = P.ws;
  int w0 = 0;
  int n_next = -1;  // survivor count of this warp's row of the next wave, being copied
  for (;; w0 += kWave) {
    float u = 0.f;  // warp 0: the uniform of position w0 + lane
    if (warp == 0 && lane < kWave && w0 + lane < k) u = P.uniforms[t0 + w0 + lane];
    int gx;
    const int64_t row = wave_row(P, b, t0, k, w0, warp, &gx);
    if (row >= 0) {
      if (n_next >= 0) copy_keys_wait();
      warp_filter_row<BF16>(P, row, K, T, chi, clo, tp, gx, scr[warp].sel, n_next);
    }
    int gn;
    const int64_t nrow = wave_row(P, b, t0, k, w0 + kWave, warp, &gn);
    n_next = -1;
    if (nrow >= 0) {
      copy_keys_async(w.cand_raw + size_t(nrow) * kRawCap, scr[warp].sel.keys);
      n_next = max(__ldcg(&w.stats[nrow].kept), 0);
    }
    __syncthreads();
    if (warp == 0) {
      int L = k;  // k == 0: only the bonus row
      if (w0 < k) {
        const int n = min(kWave, k - w0);
        bool acc = true;
        double p = 0.0, q = 0.0;
        if (lane < n) {
          p = scr[2 * lane].sel.pg;
          q = scr[2 * lane + 1].sel.pg;
          acc = double(u) * q < p;  // u < p / q
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
  if (n_next >= 0) copy_keys_wait();  // copies land before the scratch is reused
  const int L = sh.L;
  if (warp == 0) {
    // the stopping position lies in the last wave: its target (or bonus) row
    // was filtered by warp 2 (L - w0), its draft row by the next warp
    const int tw = 2 * (L - w0);
    const bool residual = L < k;
    const double u = double(u_last);
    const WarpSel& ts = scr[tw].sel;
    int y;
    if (ts.fast && (!residual || scr[tw + 1].sel.fast))
      y = draw_fast(ts, residual ? &scr[tw + 1].sel : nullptr, u, sh.idx, sh.r, nullptr);
    else
      y = draw_kept(P, t0 + L, P.Rt + d0 + L, residual, u, scr[0].draw);
    if (lane <= k) P.out_tokens[t0 + lane] = lane < L ? x_lane : (lane == L ? y : -1);
    if (lane == 0 && k == 32) P.out_tokens[t0 + 32] = L == 32 ? y : -1;
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
template <bool BF16, bool INLINE>
__global__ void __launch_bounds__(kPostThreads, 2) filter_decide_kernel(const Problem P) {
  extern __shared__ __align__(16) unsigned char post_smem[];
  WarpScratch* scr = reinterpret_cast<WarpScratch*>(post_smem);
  __shared__ PostShared sh;
  const Ws& w = P.ws;
  const int warp = threadIdx.x >> 5;
  // The job lists and the header counts come from the setup kernel, which has
  // completed before the row pass let this kernel launch; with the request's
  // inputs they are read while the row pass finishes.
  const int gerr = w.hdr->global_err;
  const int nf = w.hdr->n_filtered, nd = w.hdr->n_decide;
  int4 job0 = make_int4(0, 0, 0, 0);
  ReqParams rp0{};
  if (!gerr && int(blockIdx.x) < nf) {
    job0 = w.job[blockIdx.x];
    rp0 = request_params(P, job0.x, job0.z, job0.w);
  }
  pdl_wait();     // the row pass's results
  pdl_trigger();  // the draw pass may launch; it waits for this kernel
  if (gerr) {
    // batch-level data error: every output is -1 (NaN for the probabilities)
    const int64_t stride = int64_t(gridDim.x) * kPostThreads;
    const int64_t i0 = int64_t(blockIdx.x) * kPostThreads + threadIdx.x;
    for (int64_t r = i0; r < P.B; r += stride) P.out_accept_len[r] = -1;
    for (int64_t r = i0; r < P.Rt; r += stride) P.out_tokens[r] = -1;
    if (P.out_pq)
      for (int64_t r = i0; r < 2 * P.Rd; r += stride) P.out_pq[r] = nan64();
    return;
  }
  const int units = nf + (nd + kWarps - 1) / kWarps;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    if (u < nf) {
      const int4 job = u == int(blockIdx.x) ? job0 : w.job[u];
      if (w.req_flag[job.x]) {  // a logit error found by the row pass
        if (warp == 0) fail_request(P, job.x, job.w, job.z, job.z - job.x);
      } else {
        const ReqParams rp = u == int(blockIdx.x) ? rp0 : request_params(P, job.x, job.z, job.w);
        filtered_request<BF16>(P, job.x, job.z, job.w, rp, scr, sh);
      }
      __syncthreads();  // the scratch is reused by the next unit
    } else {
      const int j = (u - nf) * kWarps + warp;
      if (j < nd) decide_request<BF16, INLINE>(P, w.job[P.B + j].x);
    }
  }
}

// Draft sampler, after the row pass: one warp per drafter row, rows handed out
// by a counter.  Greedy rows emit the argmax; filtered rows take the exact
// top k, the softmax and top-p (the verifier's row filter) and draw from the
// kept set by inverse CDF in index order with the row's uniform; the other
// sampled rows are queued for the draw pass, which streams the row again.
template <bool BF16>
__global__ void __launch_bounds__(kPostThreads, 2) sample_post_kernel(const Problem P) {
  extern __shared__ __align__(16) unsigned char post_smem[];
  WarpScratch* scr = reinterpret_cast<WarpScratch*>(post_smem);
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();     // the row pass's results
  pdl_trigger();  // the draw pass may launch; it waits for this kernel
  if (w.hdr->global_err) {
    // batch-level data error: every output is -1 (NaN for q)
    const int64_t stride = int64_t(gridDim.x) * kPostThreads;
    for (int64_t r = int64_t(blockIdx.x) * kPostThreads + threadIdx.x; r < P.Rt; r += stride) {
      P.out_tokens[r] = -1;
      if (P.out_q) P.out_q[r] = __int_as_float(0x7fc00000);
    }
    return;
  }
  // rows listed from the front (hdr->n_active), then the kBig rows listed
  // from the back (hdr->n_big)
  const int na = w.hdr->n_active, n = na + w.hdr->n_big;
  WarpScratch& ws = scr[warp];
  for (;;) {
    int j = 0;
    if (lane == 0) j = atomicAdd(&w.hdr->next_row, 1);
    j = __shfl_sync(kFull, j, 0);
    if (j >= n) break;
    const RowJob job = j < na ? w.rowlist[j] : w.rowlist[P.Rt - 1 - (j - na)];
    const int64_t row = job.row;
    const int mode = job.mode & kModeMask;
    const double u = double(P.uniforms[row]);
    int y = -1;
    float qy = __int_as_float(0x7fc00000);
    bool queued = false;
    if (w.req_flag[job.b]) {
      // a logit error found by the row pass: the request's rows fail
    } else if (mode == kArgmax) {
      y = __ldcg(&w.stats[row].arg);
    } else if (mode == kTopk) {
      const float tp = P.top_p ? P.top_p[job.b] : 1.0f;
      float chi, clo;
      log2e_over_t(job.T, &chi, &clo);
      warp_filter_row<BF16>(P, row, job.K, job.T, chi, clo, tp, -1, ws.sel);
      if (ws.sel.fast) {
        y = draw_fast(ws.sel, nullptr, u, ws.sel.hw, ws.sel.before, &qy);
      } else {
        y = draw_kept(P, row, 0, false, u, ws.draw);
        // the drawn token's kept probability, from the kept list in global memory
        const int kp = __ldcg(&w.stats[row].kept);
        float pv = 0.f;
        for (int i = lane; i < kp; i += 32)
          if (__ldcg(&w.cand_idx[size_t(row) * kTopkMax + i]) == y)
            pv = __ldcg(&w.cand_p[size_t(row) * kTopkMax + i]);
        const uint32_t hb = __ballot_sync(kFull, pv != 0.f);
        qy = hb ? __shfl_sync(kFull, pv, __ffs(hb) - 1) : 0.f;
      }
      __syncwarp();  // the scratch is rewritten by the warp's next row
    } else {
      queued = true;
      if (lane == 0) {
        const RowStat st = w.stats[row];
        DrawDesc d;
        d.tr = row;
        d.dr = 0;
        d.mt = st.m;
        d.ist = float(1.0 / st.s);
        d.md = 0.f;
        d.isd = 0.f;
        d.kt = mode == kBig ? w.cand_raw[size_t(row) * kRawCap] : 0ull;
        d.kd = 0ull;
        d.c2 = __fdiv_rn(1.4426950408889634f, job.T);
        d.kind = 0;
        d.u = u;
        d.t0 = int32_t(row);
        d.L = 0;
        w.draw[atomicAdd(&w.hdr->n_draw, 1)] = d;
      }
    }
    if (!queued && lane == 0) {
      P.out_tokens[row] = y;
      if (P.out_q) P.out_q[row] = qy;
    }
  }
}

}  // namespace

cudaError_t launch_sample_post(const Problem& P, bool bf16, int grid, cudaStream_t s) {
  const size_t smem = sizeof(WarpScratch) * kWarps;
  if (bf16) return launch_after(sample_post_kernel<true>, grid, kPostThreads, smem, s, P);
  return launch_after(sample_post_kernel<false>, grid, kPostThreads, smem, s, P);
}

size_t filter_smem_bytes() { return sizeof(WarpScratch) * kWarps; }

cudaError_t launch_filter_decide(const Problem& P, bool bf16, int grid, cudaStream_t s) {
  const size_t smem = filter_smem_bytes();
  if (P.inline_draw)
    return bf16 ? launch_after(filter_decide_kernel<true, true>, grid, kPostThreads, smem, s, P)
                : launch_after(filter_decide_kernel<false, true>, grid, kPostThreads, smem, s, P);
  return bf16 ? launch_after(filter_decide_kernel<true, false>, grid, kPostThreads, smem, s, P)
              : launch_after(filter_decide_kernel<false, false>, grid, kPostThreads, smem, s, P);
}

// Shared-memory limit and resident CTAs per SM of the filter / decide kernel
// (host queries; nothing is allocated).
cudaError_t filter_occupancy(int* occ) {
  const int smem = int(filter_smem_bytes());
  cudaError_t e = cudaFuncSetAttribute(filter_decide_kernel<true, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(filter_decide_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(filter_decide_kernel<true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(filter_decide_kernel<false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sample_post_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sample_post_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int a = 0, b = 0, c = 0, d = 0;
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, filter_decide_kernel<true, false>,
                                                      kPostThreads, smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, filter_decide_kernel<false, false>,
                                                      kPostThreads, smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, filter_decide_kernel<true, true>,
                                                      kPostThreads, smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d, filter_decide_kernel<false, true>,
                                                      kPostThreads, smem);
  if (e != cudaSuccess) return e;
  *occ = max(1, min(min(a, b), min(c, d)));
  return cudaSuccess;
}

}  // namespace sv
