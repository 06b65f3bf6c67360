// Finalize kernel: one CTA per request.
//
// 1. Decision (one warp; k <= 32 so lane i owns draft i):
//      greedy   : accept_i = (x_i == argmax of target row i)
//      sampling : accept_i = (u_i < p_i(x_i) / q_i(x_i)), in double
//    The first rejection is the lowest set bit of the ballot of rejections
//    ("FlashMap…" §4 steps 1-3: stop at the first rejection; "DFlash" §4).
// 2. Final token at L (the accept length):
//      greedy   : argmax of target row L ("Speculative decoding…", "Draft and
//                 verify", step Three: emit the target's own token);
//      sampling : inverse CDF at u_k over index order of the normalised
//                 residual max(0, p_L - q_L) if L < k, else of p_k (bonus).
//                 Filtered rows: over the kept sets (<= SV_TOPK_MAX tokens) in
//                 double precision.  Unfiltered rows: a pass over the row(s)
//                 with per-256-element tile sums, then a re-scan of the one
//                 tile that holds the draw.
#include <math.h>

#include "sv_select.cuh"

namespace sv {
namespace {

constexpr int kWarps = kFinalThreads / 32;
static_assert(kFinalThreads >= kTopkMax, "one thread per kept token in the filtered draw");
constexpr int kScanTile = 256;  // elements per warp tile (32 lanes x 8)

struct BlockSync {
  __device__ void operator()() const { __syncthreads(); }
};

template <bool BF16>
struct Row8;

template <>
struct Row8<true> {
  static constexpr int kSize = 2;
  // 8 consecutive elements starting at i (i a multiple of 8); elements past V read as -inf.
  __device__ static void load(const void* row, int i, int V, float* x) {
    const uint16_t* r = static_cast<const uint16_t*>(row);
    if (i + 8 <= V) {
      const uint4 q = *reinterpret_cast<const uint4*>(r + i);
      x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x); x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
      x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z); x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
    } else {
      for (int e = 0; e < 8; ++e)
        x[e] = i + e < V ? __uint_as_float(uint32_t(r[i + e]) << 16) : -INFINITY;
    }
  }
};

template <>
struct Row8<false> {
  static constexpr int kSize = 4;
  __device__ static void load(const void* row, int i, int V, float* x) {
    const float* r = static_cast<const float*>(row);
    if (i + 8 <= V) {
      const float4 a = *reinterpret_cast<const float4*>(r + i);
      const float4 c = *reinterpret_cast<const float4*>(r + i + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
    } else {
      for (int e = 0; e < 8; ++e) x[e] = i + e < V ? r[i + e] : -INFINITY;
    }
  }
};

struct FinalShared {
  int L;
  int ystar;
  int seg_tile;
  int fallback;
  double seg[kWarps];
  double R;
  double S;
  double t;
  int lastpos[kWarps];
  int yfound[kWarps];
  // filtered draw
  int d_idx[kTopkMax];
  double d_q[kTopkMax];
  double slot_r[kTopkMax];
  double slot_p[kTopkMax];
  int slot_idx[kTopkMax];
  double srt_r[kTopkMax];
  double srt_p[kTopkMax];
  int srt_idx[kTopkMax];
  uint64_t xchg[2 * kFinalThreads];
};

// Weight of element y for the unfiltered final draw.
//   kind 0: bonus, exp((x_t - m_t)/T)             (unnormalised p_k)
//   kind 1: residual, max(0, p_t - q_t)
//   kind 2: residual fallback, p_t
struct Weights {
  float mt, ist, md, isd, c2;
  int kind;
  __device__ __forceinline__ float operator()(float xt, float xd) const {
    const float et = ex2_approx((xt - mt) * c2);
    if (kind == 0) return et;
    if (kind == 2) return et * ist;
    const float ed = ex2_approx((xd - md) * c2);
    return fmaxf(0.f, et * ist - ed * isd);
  }
};

template <bool BF16>
__device__ void tile_weights(const void* trow, const void* drow, int base, int V, const Weights& W,
                             float* r) {
  float xt[8], xd[8];
  Row8<BF16>::load(trow, base, V, xt);
  if (W.kind == 1) Row8<BF16>::load(drow, base, V, xd);
#pragma unroll
  for (int e = 0; e < 8; ++e) r[e] = base + e < V ? W(xt[e], W.kind == 1 ? xd[e] : 0.f) : 0.f;
}

// Inverse-CDF draw over a full row: returns the token.  All threads call.
template <bool BF16>
__device__ int unfiltered_draw(const void* trow, const void* drow, int V, Weights W, double u,
                               float* tile_sum, FinalShared& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntile = (V + kScanTile - 1) / kScanTile;
  const int per_warp = (ntile + kWarps - 1) / kWarps;
  const int tw0 = warp * per_warp;
  const int tw1 = min(ntile, tw0 + per_warp);
  for (int attempt = 0; attempt < 2; ++attempt) {
    // pass A: per-tile sums (warp inclusive scan, so pass B reproduces them)
    double Rw = 0.0;
    int lastpos = -1;
    for (int tau = tw0; tau < tw1; ++tau) {
      const int base = tau * kScanTile + lane * 8;
      float r[8];
      tile_weights<BF16>(trow, drow, base, V, W, r);
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ls += r[e];
        if (r[e] > 0.f) lastpos = base + e;
      }
      float incl = ls;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const float tot = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) tile_sum[tau] = tot;
      Rw += double(tot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
    if (lane == 0) {
      S.seg[warp] = Rw;
      S.lastpos[warp] = lastpos;
    }
    __syncthreads();
    if (tid == 0) {
      double tot = 0.0;
      for (int i = 0; i < kWarps; ++i) tot += S.seg[i];
      S.S = tot;
      S.fallback = (W.kind == 1 && !(tot > 0.0)) ? 1 : 0;
    }
    __syncthreads();
    if (!S.fallback) break;
    W.kind = 2;  // residual mass vanished through rounding: draw from p_L
    __syncthreads();
  }
  if (tid == 0) {
    const double t = u * S.S;
    S.t = t;
    int last = -1;
    for (int i = 0; i < kWarps; ++i) last = max(last, S.lastpos[i]);
    double R = 0.0;
    int found = -1;
    for (int i = 0; i < kWarps && found < 0; ++i) {
      if (R + S.seg[i] > t) {
        const int a = i * per_warp, z = min(ntile, a + per_warp);
        double Ri = R;
        int lastpos_tile = -1;
        for (int tau = a; tau < z; ++tau) {
          if (tile_sum[tau] > 0.f) lastpos_tile = tau;
          if (Ri + double(tile_sum[tau]) > t) {
            found = tau;
            break;
          }
          Ri += double(tile_sum[tau]);
        }
        if (found < 0) {  // rounding at the segment end: last tile with mass
          found = lastpos_tile;
          Ri = R;
          for (int tau = a; tau < found; ++tau) Ri += double(tile_sum[tau]);
        }
        S.R = Ri;
        break;
      }
      R += S.seg[i];
    }
    S.seg_tile = found;
    S.ystar = last;  // used when t lies beyond every prefix (rounding)
  }
  __syncthreads();
  const int tau = S.seg_tile;
  if (tau >= 0 && warp == 0) {
    // pass B: the draw lies in tile tau; first y with R + C_y > t
    const int base = tau * kScanTile + lane * 8;
    float r[8];
    tile_weights<BF16>(trow, drow, base, V, W, r);
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ls += r[e];
    float incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const double R = S.R, t = S.t;
    int y = INT_MAX, lastp = -1;
    float pre = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      pre += r[e];
      if (r[e] > 0.f) lastp = base + e;
      if (y == INT_MAX && r[e] > 0.f && R + double(excl + pre) > t) y = base + e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      y = min(y, __shfl_xor_sync(0xffffffffu, y, o));
      lastp = max(lastp, __shfl_xor_sync(0xffffffffu, lastp, o));
    }
    if (lane == 0) S.ystar = (y != INT_MAX) ? y : lastp;
  }
  __syncthreads();
  return S.ystar;
}

// Per-warp scratch for selecting one filtered row's top k.
struct WarpSel {
  int hist[256];
  uint64_t list[kTopkMax];  // the row's top k, then sorted descending
  double w[kTopkMax];       // exp((x_j - x_max) / T) in sorted order
  int digit, above, cnt, pad;
};

constexpr int kRegKeys = 10;  // survivors held in registers per lane (320 per warp)

// Exact k-th largest of the n (> k) unique keys at keys[] (any memory), by
// MSB-first radix selection over 8-bit digits with a warp-private histogram;
// stops once the remaining prefix group is selected whole.
__device__ uint64_t warp_select_kth(const uint64_t* keys, int n, int k, WarpSel& ws,
                                    uint32_t skip) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0ull, mask = 0ull;
  int need = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    if ((skip >> (shift / 8)) & 1u) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) ws.hist[lane * 8 + j] = 0;
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
      const uint32_t vm = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t peers = __match_any_sync(vm, d);
        if (lane == __ffs(peers) - 1) ws.hist[d] += __popc(peers);  // distinct digits per step
      }
      __syncwarp();
    }
    int cnt[8], loc = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cnt[j] = ws.hist[lane * 8 + j];
      loc += cnt[j];
    }
    int suf = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += y;
    }
    int acc = suf - loc;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (acc < need && acc + cnt[j] >= need) {
        ws.digit = lane * 8 + j;
        ws.above = acc;
        ws.cnt = cnt[j];
      }
      acc += cnt[j];
    }
    __syncwarp();
    const int d = ws.digit;
    need -= ws.above;
    const int grp = ws.cnt;
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

// Same selection over keys held in registers (lane holds keys[j] = key
// j * 32 + lane, 0 for an empty slot).
__device__ uint64_t warp_select_kth_regs(const uint64_t (&keys)[kRegKeys], int k, WarpSel& ws,
                                         uint32_t skip) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0ull, mask = 0ull;
  int need = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    if ((skip >> (shift / 8)) & 1u) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) ws.hist[lane * 8 + j] = 0;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kRegKeys; ++r) {
      const uint64_t key = keys[r];
      const bool valid = key != 0ull && (key & mask) == prefix;
      const uint32_t d = uint32_t(key >> shift) & 255u;
      const uint32_t vm = __ballot_sync(0xffffffffu, valid);
      if (vm == 0u) continue;
      if (valid) {
        const uint32_t peers = __match_any_sync(vm, d);
        if (lane == __ffs(peers) - 1) ws.hist[d] += __popc(peers);
      }
      __syncwarp();
    }
    int cnt[8], loc = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cnt[j] = ws.hist[lane * 8 + j];
      loc += cnt[j];
    }
    int suf = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += y;
    }
    int acc = suf - loc;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (acc < need && acc + cnt[j] >= need) {
        ws.digit = lane * 8 + j;
        ws.above = acc;
        ws.cnt = cnt[j];
      }
      acc += cnt[j];
    }
    __syncwarp();
    const int d = ws.digit;
    need -= ws.above;
    const int grp = ws.cnt;
    __syncwarp();
    prefix |= uint64_t(d) << shift;
    mask |= 255ull << shift;
    if (grp == need) {
      uint64_t mn = ~0ull;
#pragma unroll
      for (int r = 0; r < kRegKeys; ++r) {
        const uint64_t key = keys[r];
        if (key != 0ull && (key & mask) == prefix && key < mn) mn = key;
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

// Bitonic sort, descending, of a[0..P) in shared memory by one warp (P a power of two).
__device__ void warp_sort_desc(uint64_t* a, int P) {
  const int lane = threadIdx.x & 31;
  for (int size = 2; size <= P; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      for (int p = lane; p < P / 2; p += 32) {
        const int i = (p / j) * 2 * j + (p % j);  // lower index of the pair
        const int q = i + j;
        const uint64_t x = a[i], y = a[q];
        const bool desc = (i & size) == 0;
        if (desc ? (x < y) : (x > y)) {
          a[i] = y;
          a[q] = x;
        }
      }
      __syncwarp();
    }
  }
}

// One filtered row: exact top k of the row pass's survivors (composite order:
// logit descending, index ascending), then the temperature softmax over them,
// the top-p cut (keep j while the probability mass before j is below top_p)
// and the renormalisation, in double precision.  Writes the kept list, the
// kept size and p(x) of the row's draft token.  One warp.
template <bool BF16>
__device__ void warp_filter_row(const Problem& P, int64_t row, int K, float T, float tp, int gx,
                                WarpSel& ws) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const int n = w.stats[row].kept;
  const uint64_t* raw = w.cand_raw + size_t(row) * kRawCap;
  const uint32_t skip = BF16 ? kSkipBf16 : kSkipF32;
  int cnt = 0;
  if (n <= 32 * kRegKeys) {
    uint64_t keys[kRegKeys];
#pragma unroll
    for (int r = 0; r < kRegKeys; ++r) {
      const int e = r * 32 + lane;
      keys[r] = e < n ? raw[e] : 0ull;
    }
    const uint64_t th = n > K ? warp_select_kth_regs(keys, K, ws, skip) : 0ull;
#pragma unroll
    for (int r = 0; r < kRegKeys; ++r) {
      const bool keep = keys[r] != 0ull && keys[r] >= th;
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const int sl = cnt + __popc(bal & lt);
        if (sl < kTopkMax) ws.list[sl] = keys[r];
      }
      cnt += __popc(bal);
    }
  } else {
    const uint64_t th = n > K ? warp_select_kth(raw, n, K, ws, skip) : 0ull;
    for (int base = 0; base < n; base += 32) {
      const int e = base + lane;
      const uint64_t key = e < n ? raw[e] : 0ull;
      const bool keep = e < n && key >= th;
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const int sl = cnt + __popc(bal & lt);
        if (sl < kTopkMax) ws.list[sl] = key;
      }
      cnt += __popc(bal);
    }
  }
  const int nsel = cnt < K ? cnt : K;
  const int Psz = next_pow2(nsel > 0 ? nsel : 1);
  for (int j = nsel + lane; j < Psz; j += 32) ws.list[j] = 0ull;
  __syncwarp();
  warp_sort_desc(ws.list, Psz);
  const double v0 = double(composite_value(ws.list[0]));
  const double invT = 1.0 / double(T);
  // Weights w_j = exp((x_j - x_max) / T) in double (w_0 = 1, all in (0, 1]).
  // Their prefix sums are taken exactly in 64-bit fixed point (unit 2^-55;
  // at most K * 2^-56 absolute rounding), which keeps FP64 work, the scarce
  // resource here, to one exponential and two multiplies per token.
  constexpr double kFix = 36028797018963968.0;  // 2^55: K <= 256 weights <= 1 sum below 2^63
  unsigned long long carry = 0ull;
  for (int j0 = 0; j0 < nsel; j0 += 32) {
    const int j = j0 + lane;
    double wv = 0.0;
    if (j < nsel) {
      wv = exp((double(composite_value(ws.list[j])) - v0) * invT);
      ws.w[j] = wv;
    }
    unsigned long long incl = (unsigned long long)__double2ull_rn(wv * kFix);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
  const unsigned long long Wfx = carry;
  // the kept prefix ends at the first j whose mass before it is not below top_p
  int kp = nsel;
  unsigned long long Wpfx = Wfx;
  if (tp < 1.0f) {
    const double lim = double(tp) * double(Wfx);
    unsigned long long c2 = 0ull;
    for (int j0 = 0; j0 < nsel && kp == nsel; j0 += 32) {
      const int j = j0 + lane;
      const unsigned long long mine =
          j < nsel ? (unsigned long long)__double2ull_rn(ws.w[j] * kFix) : 0ull;
      unsigned long long incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned long long before = c2 + incl - mine;
      const bool drop = j < nsel && !(double(before) < lim);
      const uint32_t bal = __ballot_sync(0xffffffffu, drop);
      if (bal) {
        kp = j0 + __ffs(bal) - 1;
        Wpfx = __shfl_sync(0xffffffffu, before, kp - j0);
      }
      c2 += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  const double Wp = double(Wpfx) / kFix;
  const double inv = 1.0 / Wp;
  const size_t cbase = size_t(row) * kTopkMax;
  bool hit = false;
  double pgv = 0.0;
  for (int j = lane; j < kp; j += 32) {
    const int idx = composite_index(ws.list[j]);
    const double pj = ws.w[j] * inv;
    w.cand_idx[cbase + j] = idx;
    w.cand_p[cbase + j] = pj;
    if (idx == gx) {
      hit = true;
      pgv = pj;
    }
  }
  const uint32_t hb = __ballot_sync(0xffffffffu, hit);
  if (hb) pgv = __shfl_sync(0xffffffffu, pgv, __ffs(hb) - 1);
  if (lane == 0) {
    RowStat st;
    st.s = Wp;
    st.pg = gx >= 0 ? pgv : __longlong_as_double(0x7ff8000000000000LL);
    st.m = float(v0);
    st.arg = -1;
    st.kept = kp;
    st.mode = kTopk;
    w.stats[row] = st;
  }
  __syncwarp();
}

// Inverse-CDF draw over kept sets (double, index order).  All threads call.
//   residual: target kept set of row tr against draft kept set of row dr
//   bonus   : target kept set of row tr
__device__ int filtered_draw(const Problem& P, int64_t tr, int64_t dr, bool residual, double u,
                             FinalShared& S) {
  const Ws& w = P.ws;
  const int tid = threadIdx.x;
  const int Kt = w.stats[tr].kept;
  const int Kd = residual ? w.stats[dr].kept : 0;
  for (int i = tid; i < Kd; i += kFinalThreads) {
    S.d_idx[i] = w.cand_idx[size_t(dr) * kTopkMax + i];
    S.d_q[i] = w.cand_p[size_t(dr) * kTopkMax + i];
  }
  __syncthreads();
  uint64_t key = 0ull;
  if (tid < Kt) {
    const int idx = w.cand_idx[size_t(tr) * kTopkMax + tid];
    const double p = w.cand_p[size_t(tr) * kTopkMax + tid];
    double q = 0.0;
    for (int i = 0; i < Kd; ++i)
      if (S.d_idx[i] == idx) q = S.d_q[i];
    S.slot_r[tid] = residual ? fmax(0.0, p - q) : p;
    S.slot_p[tid] = p;
    S.slot_idx[tid] = idx;
    // descending sort of the complement = ascending vocabulary index
    key = ~((uint64_t(uint32_t(idx)) << 32) | uint32_t(tid));
  }
  const int Psz = next_pow2(Kt > 0 ? Kt : 1);
  key = block_sort_desc<kFinalThreads>(key, tid, Psz, S.xchg, BlockSync());
  __syncthreads();  // slot_* written by other threads (the sort may not sync for small sizes)
  if (tid < Kt) {
    const int slot = int(uint32_t(~key));
    S.srt_r[tid] = S.slot_r[slot];
    S.srt_p[tid] = S.slot_p[slot];
    S.srt_idx[tid] = S.slot_idx[slot];
  }
  __syncthreads();
  if (tid == 0) {
    double tot = 0.0;
    for (int i = 0; i < Kt; ++i) tot += S.srt_r[i];
    const double* r = S.srt_r;
    if (!(tot > 0.0)) {  // residual mass vanished through rounding: draw from p_L
      r = S.srt_p;
      tot = 0.0;
      for (int i = 0; i < Kt; ++i) tot += r[i];
    }
    const double t = u * tot;
    double C = 0.0;
    int y = -1, last = -1;
    for (int i = 0; i < Kt; ++i) {
      if (r[i] > 0.0) last = S.srt_idx[i];
      C += r[i];
      if (C > t) {
        y = S.srt_idx[i];
        break;
      }
    }
    S.ystar = y >= 0 ? y : last;
  }
  __syncthreads();
  return S.ystar;
}

template <bool BF16>
__global__ void __launch_bounds__(kFinalThreads, 1) finalize_kernel(const Problem P) {
  extern __shared__ __align__(16) unsigned char fsmem[];
  WarpSel* wsel = reinterpret_cast<WarpSel*>(fsmem);
  float* tile_sum = reinterpret_cast<float*>(fsmem + sizeof(WarpSel) * kWarps);
  __shared__ FinalShared S;
  const Ws& w = P.ws;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const double kNaN = __longlong_as_double(0x7ff8000000000000LL);

  if (w.hdr->global_err) {
    // batch-level data error: every output is -1 (NaN for the probabilities)
    const int64_t stride = int64_t(gridDim.x) * kFinalThreads;
    if (tid == 0) P.out_accept_len[b] = -1;
    for (int64_t r = int64_t(b) * kFinalThreads + tid; r < P.Rt; r += stride) P.out_tokens[r] = -1;
    if (P.out_pq)
      for (int64_t r = int64_t(b) * kFinalThreads + tid; r < 2 * P.Rd; r += stride)
        P.out_pq[r] = kNaN;
    return;
  }
  const int k = P.k_per_req[b];
  const int t0 = w.t_off[b], d0 = t0 - b;
  if (w.req_flag[b]) {
    for (int i = tid; i <= k; i += kFinalThreads) P.out_tokens[t0 + i] = -1;
    if (P.out_pq)
      for (int i = tid; i < 2 * k; i += kFinalThreads) P.out_pq[2 * int64_t(d0) + i] = kNaN;
    if (tid == 0) P.out_accept_len[b] = -1;
    return;
  }
  const float T = P.temperature[b];
  const bool greedy = T == 0.0f;

  // Filtered requests: exact top k, softmax and top-p of every row (target
  // rows 0..k, draft rows 0..k-1), one warp per row.
  if (!greedy && w.stats[t0].mode == kTopk) {
    const int K = P.top_k[b];
    const float tp = P.top_p ? P.top_p[b] : 1.0f;
    for (int i = warp; i < 2 * k + 1; i += kWarps) {
      int64_t row;
      int gx;
      if (i <= k) {
        row = t0 + i;
        gx = i < k ? P.draft_tokens[d0 + i] : -1;
      } else {
        row = P.Rt + d0 + (i - k - 1);
        gx = P.draft_tokens[d0 + (i - k - 1)];
      }
      warp_filter_row<BF16>(P, row, K, T, tp, gx, wsel[warp]);
    }
    __syncthreads();
  }

  if (warp == 0) {
    bool acc = false;
    int x = -1;
    if (lane < k) {
      x = P.draft_tokens[d0 + lane];
      if (greedy) {
        acc = x == w.stats[t0 + lane].arg;
        if (P.out_pq) {
          P.out_pq[2 * int64_t(d0 + lane)] = kNaN;
          P.out_pq[2 * int64_t(d0 + lane) + 1] = kNaN;
        }
      } else {
        const double p = w.stats[t0 + lane].pg;
        const double q = w.stats[P.Rt + d0 + lane].pg;
        acc = double(P.uniforms[t0 + lane]) < p / q;
        if (P.out_pq) {
          P.out_pq[2 * int64_t(d0 + lane)] = p;
          P.out_pq[2 * int64_t(d0 + lane) + 1] = q;
        }
      }
    }
    const uint32_t rej = __ballot_sync(0xffffffffu, lane < k && !acc);
    const int L = rej ? __ffs(rej) - 1 : k;
    if (lane < k && lane != L) P.out_tokens[t0 + lane] = lane < L ? x : -1;
    if (lane == 0) S.L = L;
  }
  __syncthreads();
  const int L = S.L;
  int ystar;
  if (greedy) {
    ystar = w.stats[t0 + L].arg;
  } else {
    const int64_t tr = t0 + L;
    const int64_t dr = P.Rt + d0 + L;
    const bool residual = L < k;
    const double u = double(P.uniforms[t0 + k]);
    if (w.stats[tr].mode == kTopk) {
      ystar = filtered_draw(P, tr, dr, residual, u, S);
    } else {
      const RowStat st = w.stats[tr];
      Weights W;
      W.c2 = __fdiv_rn(1.4426950408889634f, T);
      W.mt = st.m;
      W.ist = float(1.0 / st.s);
      W.kind = residual ? 1 : 0;
      W.md = 0.f;
      W.isd = 0.f;
      const void* trow = static_cast<const char*>(P.target) + tr * P.t_stride * Row8<BF16>::kSize;
      const void* drow = nullptr;
      if (residual) {
        const RowStat sd = w.stats[dr];
        W.md = sd.m;
        W.isd = float(1.0 / sd.s);
        drow = static_cast<const char*>(P.draft) + (dr - P.Rt) * P.d_stride * Row8<BF16>::kSize;
      }
      ystar = unfiltered_draw<BF16>(trow, drow, P.V, W, u, tile_sum, S);
    }
  }
  if (tid == 0) {
    P.out_tokens[t0 + L] = ystar;
    if (L < k) P.out_tokens[t0 + k] = -1;
    P.out_accept_len[b] = L;
  }
}

}  // namespace

size_t finalize_smem_bytes(int V) {
  return sizeof(WarpSel) * kWarps + sizeof(float) * size_t((V + kScanTile - 1) / kScanTile);
}

cudaError_t launch_finalize(const Problem& P, bool bf16, cudaStream_t s) {
  const size_t smem = finalize_smem_bytes(P.V);
  if (bf16)
    finalize_kernel<true><<<P.B, kFinalThreads, smem, s>>>(P);
  else
    finalize_kernel<false><<<P.B, kFinalThreads, smem, s>>>(P);
  return cudaGetLastError();
}

cudaError_t finalize_configure() {
  const int smem = int(finalize_smem_bytes(SV_VOCAB_MAX));
  cudaError_t e = cudaFuncSetAttribute(finalize_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(finalize_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem);
}

}  // namespace sv
