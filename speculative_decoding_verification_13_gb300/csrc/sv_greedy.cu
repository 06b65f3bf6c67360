// Greedy verification from the target rows' argmax alone (no logits).
//
// At temperature 0 verification reads of each target row only its argmax:
// the longest prefix of drafts equal to the target's argmax is accepted and
// the argmax at the first disagreement (or after a full acceptance, the
// bonus) is emitted ("DFlash" §4 step 5; "Speculative decoding and
// multi-token prediction", "Draft and verify", step Three).  The LM-head GEMM
// (sv_lmhead.cu) produces each row's argmax in its epilogue, so a greedy
// request chained after it never needs its logits in memory.
//
// One CTA: a first pass forms the row offsets t_off[b] = sum_{j<b} (k_j + 1)
// and checks them against the target row count (any error fails the whole
// batch before a row is read); the second pass decides each request, one
// thread per request.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kGThreads = 1024;

// Exclusive scan of v over the CTA; *total gets the sum.
__device__ int greedy_scan(int v, int* total) {
  __shared__ int s_warp[kGThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int y = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_warp[lane] = y;
  }
  __syncthreads();
  const int ex = x - v + (warp ? s_warp[warp - 1] : 0);
  *total = s_warp[kGThreads / 32 - 1];
  __syncthreads();
  return ex;
}

__global__ void __launch_bounds__(kGThreads) greedy_kernel(const int32_t* argmax,
                                                           const int32_t* draft_tokens,
                                                           const int32_t* k_per_req,
                                                           int32_t* out_accept_len,
                                                           int32_t* out_tokens, int B, int64_t Rt,
                                                           int V, WsHeader* hdr) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    hdr->err_code = 0;
    hdr->err_req = -1;
    hdr->err_row = -1;
    s_bad = 0;
  }
  __syncthreads();
  // pass 1: offsets and the batch-level checks
  int64_t carry = 0;
  for (int base = 0; base < B; base += kGThreads) {
    const int b = base + threadIdx.x;
    int k = 0;
    if (b < B) {
      k = k_per_req[b];
      if (k < 0 || k > SV_MAX_K) {
        record_error(hdr, SV_ERR_DATA_K, b, -1);
        atomicOr(&s_bad, 1);
        k = 0;
      }
    }
    int tot;
    greedy_scan(b < B ? k + 1 : 0, &tot);
    carry += tot;
  }
  if (threadIdx.x == 0 && !s_bad && carry != Rt) {
    record_error(hdr, SV_ERR_DATA_ROWS, -1, -1);
    s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    for (int b = threadIdx.x; b < B; b += kGThreads) out_accept_len[b] = -1;
    for (int64_t r = threadIdx.x; r < Rt; r += kGThreads) out_tokens[r] = -1;
    return;
  }
  // pass 2: one request per thread
  carry = 0;
  for (int base = 0; base < B; base += kGThreads) {
    const int b = base + threadIdx.x;
    const int k = b < B ? k_per_req[b] : 0;
    int tot;
    const int64_t t0 = carry + greedy_scan(b < B ? k + 1 : 0, &tot);
    carry += tot;
    if (b >= B) continue;
    const int64_t d0 = t0 - b;
    bool bad = false;
    int L = k;
    for (int i = 0; i < k; ++i) {
      const int x = draft_tokens[d0 + i];
      const int g = argmax[t0 + i];
      bad |= x < 0 || x >= V || g < 0 || g >= V;
      if (L == k && x != g) L = i;
    }
    const int gL = argmax[t0 + L];
    bad |= gL < 0 || gL >= V;
    if (bad) {
      record_error(hdr, SV_ERR_DATA_TOKEN, b, -1);
      for (int i = 0; i <= k; ++i) out_tokens[t0 + i] = -1;
      out_accept_len[b] = -1;
      continue;
    }
    for (int i = 0; i < L; ++i) out_tokens[t0 + i] = draft_tokens[d0 + i];
    out_tokens[t0 + L] = gL;
    for (int i = L + 1; i <= k; ++i) out_tokens[t0 + i] = -1;
    out_accept_len[b] = L;
  }
}

}  // namespace

cudaError_t launch_greedy_from_argmax(const int32_t* argmax, const int32_t* draft_tokens,
                                      const int32_t* k_per_req, int32_t* out_accept_len,
                                      int32_t* out_tokens, int B, int64_t Rt, int V,
                                      void* workspace, cudaStream_t s) {
  greedy_kernel<<<1, kGThreads, 0, s>>>(argmax, draft_tokens, k_per_req, out_accept_len,
                                        out_tokens, B, Rt, V,
                                        static_cast<WsHeader*>(workspace));
  return cudaGetLastError();
}

}  // namespace sv
