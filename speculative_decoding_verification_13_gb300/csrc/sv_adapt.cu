// Per-request speculation length from measured acceptance (adaptive k), on
// the stream right after verification, without a host round trip.
//
// "Speculative decoding and multi-token prediction", section "Acceptance rate
// is the whole economics": a position beyond k is worth alpha^k tokens for a
// draft step's cost c, so speculation pays while alpha^k stays above c.  Per
// request: the accept length L of the last pass (out of k drafts) adds L
// accepted positions and, when L < k, one rejected position to counts that
// decay by d per pass; alpha = (S + 1) / (S + F + 2); the next k is the
// largest k in [k_min, k_max] with alpha^k > c (k_min if none), alpha^k taken
// as the product of k factors.  L = -1 (failed verification) keeps the
// request's counts and k.  Every double operation is rounded on its own (no
// contraction), so the result is reproducible bit for bit.
#include "sv_internal.cuh"

namespace sv {
namespace {

__global__ void adapt_k_kernel(const int32_t* accept_len, const int32_t* k_used, double* succ,
                               double* fail, double decay, double c, int k_min, int k_max,
                               int32_t* k_next, float* alpha_out, int B) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int L = accept_len[b], k = k_used[b];
  double s = succ[b], f = fail[b];
  if (L >= 0) {
    s = __dadd_rn(__dmul_rn(decay, s), double(L));
    f = __dadd_rn(__dmul_rn(decay, f), L < k ? 1.0 : 0.0);
    succ[b] = s;
    fail[b] = f;
  }
  const double a = __ddiv_rn(__dadd_rn(s, 1.0), __dadd_rn(__dadd_rn(s, f), 2.0));
  int kn = k_min;
  double p = 1.0;
  for (int j = 1; j <= k_max; ++j) {
    p = __dmul_rn(p, a);
    if (j >= k_min && p > c) kn = j;
  }
  k_next[b] = L >= 0 ? kn : k;
  if (alpha_out) alpha_out[b] = float(a);
}

}  // namespace

cudaError_t launch_adapt_k(const int32_t* accept_len, const int32_t* k_used, double* succ,
                           double* fail, double decay, double c, int k_min, int k_max,
                           int32_t* k_next, float* alpha, int B, cudaStream_t s) {
  adapt_k_kernel<<<(B + 255) / 256, 256, 0, s>>>(accept_len, k_used, succ, fail, decay, c, k_min,
                                                 k_max, k_next, alpha, B);
  return cudaGetLastError();
}

}  // namespace sv
