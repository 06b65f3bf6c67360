// Weights of the final draw (inverse CDF over the residual max(0, p_L - q_L)
// or p_k, with kept-set masks), shared by the draw pass, the locate kernel and
// the in-place draw of the decide jobs: the element weight, element loads,
// the 2^-40 fixed point of the exact prefix sums and the warp scans over it.
#pragma once

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kDTile = 256;  // elements per tile (32 lanes x 8)

// Weight of element y.
//   kind 0: bonus, exp((x_t - m_t)/T)             (unnormalised p_k)
//   kind 1: residual, max(0, p_t - q_t)
//   kind 2: residual fallback, p_t
// A row filtered by a threshold (top-p alone or a large top-k) keeps y iff
// its composite key (logit descending, index ascending) is at least the
// threshold's: x > v, or x == v and y <= i for the threshold's value v and
// index i; p or q is 0 outside the kept set.
// The probabilities are formed as 2^((x - m) c2 - l), x - m exact for bf16
// logits and one FMA: l = 0 for the unnormalised bonus weights, l = log2 S
// for normalised p and q (the weights near the row maximum, which carry the
// mass, keep the accuracy of ex2.approx).
struct Weights {
  float mt, ist, md, isd, c2;
  float bt, bd;   // log2 normalisers of the target and draft weights (kind)
  float bt0, btn; // bonus (unnormalised: 0) and normalised target ones
  int kind;
  bool mask_t, mask_d;
  float vt, vd;
  uint32_t it, id;
  __device__ __forceinline__ void set_kind(int k) {
    kind = k;
    bt = k == 0 ? bt0 : btn;
  }
  __device__ __forceinline__ float operator()(float xt, float xd) const {
    const float et = ex2_approx(fmaf(xt - mt, c2, -bt));
    if (kind != 1) return et;
    const float ed = ex2_approx(fmaf(xd - md, c2, -bd));
    return fmaxf(0.f, et - ed);
  }
  // the same with the kept-set masks (y: the element's index)
  __device__ __forceinline__ float masked(float xt, float xd, uint32_t y) const {
    const bool kt = !mask_t || xt > vt || (xt == vt && y <= it);
    const float et = kt ? ex2_approx(fmaf(xt - mt, c2, -bt)) : 0.f;
    if (kind != 1) return et;
    const bool kd = !mask_d || xd > vd || (xd == vd && y <= id);
    const float ed = kd ? ex2_approx(fmaf(xd - md, c2, -bd)) : 0.f;
    return fmaxf(0.f, et - ed);
  }
  __device__ __forceinline__ float at(float xt, float xd, int y) const {
    return (mask_t || mask_d) ? masked(xt, xd, uint32_t(y)) : (*this)(xt, xd);
  }
};

template <bool BF16>
struct Elt;

template <>
struct Elt<true> {
  static constexpr int kSize = 2;
  // 8 elements from 16 aligned bytes
  __device__ static void vec8(const void* p, float* x) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x); x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
    x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z); x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
  }
  __device__ static float one(const void* p, int64_t i) {
    return __uint_as_float(uint32_t(static_cast<const uint16_t*>(p)[i]) << 16);
  }
};

template <>
struct Elt<false> {
  static constexpr int kSize = 4;
  __device__ static void vec8(const void* p, float* x) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  __device__ static float one(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
  }
};

// 8 elements starting at e (a multiple of 8): from `fast` (16-byte aligned
// memory holding element e at its start) when all 8 lie below `fast_end`,
// else one by one: below fast_end from `fast`, below V from the row in
// global memory, -inf past V.
template <bool BF16>
__device__ __forceinline__ void elems8(const unsigned char* fast, const void* row, int e,
                                       int fast_end, int V, float* x) {
  if (e + 8 <= fast_end) {
    Elt<BF16>::vec8(fast, x);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = e + q;
      x[q] = i < fast_end ? Elt<BF16>::one(fast, q)
                          : (i < V ? Elt<BF16>::one(row, i) : -INFINITY);
    }
  }
}

// A float weight (or sum of weights) as an integer multiple of 2^-40.
__device__ __forceinline__ unsigned long long fixw(float x) {
  return __float2ull_rn(x * 1099511627776.0f);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// The weights of a queued draw, from its descriptor.
__device__ __forceinline__ Weights make_weights(const DrawDesc& d) {
  Weights W;
  W.mt = d.mt;
  W.ist = d.ist;
  W.md = d.md;
  W.isd = d.isd;
  W.c2 = d.c2;
  W.bt0 = 0.f;
  W.btn = -log2f(d.ist);
  W.bd = d.kind == 1 ? -log2f(d.isd) : 0.f;
  W.set_kind(d.kind);
  W.mask_t = d.kt != 0ull;
  W.mask_d = d.kind == 1 && d.kd != 0ull;
  W.vt = W.mask_t ? composite_value(d.kt) : 0.f;
  W.vd = W.mask_d ? composite_value(d.kd) : 0.f;
  W.it = uint32_t(composite_index(d.kt));
  W.id = uint32_t(composite_index(d.kd));
  return W;
}

// The lane's 8 weights of tile tau, read from global memory.
template <bool BF16>
__device__ __forceinline__ void lane_tile_global(const Weights& Wt, const void* trow,
                                                 const void* drow, int tau, int V, float* r) {
  const int e = tau * kDTile + (threadIdx.x & 31) * 8;
  float xt[8], xd[8];
  elems8<BF16>(nullptr, trow, e, 0, V, xt);
  if (Wt.kind == 1) elems8<BF16>(nullptr, drow, e, 0, V, xd);
#pragma unroll
  for (int k = 0; k < 8; ++k) r[k] = Wt.at(xt[k], Wt.kind == 1 ? xd[k] : 0.f, e + k);
}

}  // namespace
}  // namespace sv
