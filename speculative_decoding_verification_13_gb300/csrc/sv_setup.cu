// Setup kernel: one CTA per call.  Computes the ragged row offsets
// t_off[b] = sum_{j<b} (k_j + 1), validates every request's parameters and
// drafted tokens, picks each row's mode, writes the list of rows the
// streaming pass must read (ordered by request) and the list of post-pass jobs,
// and zeroes the per-request counters the post-pass kernels count with.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kSetupThreads = 1024;

// Exclusive scan over the CTA; *total receives the sum.  Two counters travel
// packed in one 64-bit word (each field's sum over a chunk stays below 2^32).
__device__ unsigned long long block_exclusive_scan(unsigned long long v, unsigned long long* total) {
  __shared__ unsigned long long s_warp[kSetupThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long y = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_warp[lane] = y;
  }
  __syncthreads();
  const unsigned long long excl = x - v + (warp ? s_warp[warp - 1] : 0ull);
  *total = s_warp[kSetupThreads / 32 - 1];
  __syncthreads();
  return excl;
}

__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

__global__ void __launch_bounds__(kSetupThreads) setup_kernel(const Problem P) {
  const Ws& w = P.ws;
  __shared__ int s_bad;
  pdl_trigger();  // the row pass may launch and set up; it waits for this kernel
  if (threadIdx.x == 0) {
    w.hdr->err_code = 0;
    w.hdr->err_req = -1;
    w.hdr->err_row = -1;
    w.hdr->n_active = 0;
    w.hdr->global_err = 0;
    w.hdr->n_filtered = 0;
    w.hdr->n_decide = 0;
    w.hdr->n_draw = 0;
    s_bad = 0;
  }
  __syncthreads();

  // Pass 1: row offsets; a k outside [0, SV_MAX_K] makes the layout undefined.
  // With a single chunk (B <= kSetupThreads) every per-request value read or
  // formed here stays in registers for pass 2.
  const bool one = P.B <= kSetupThreads;
  int k1 = 0, t01 = 0, tk1 = 0;
  float T1 = 0.f, tp1 = 1.0f;
  int carry = 0, carry_d = 0;
  for (int base = 0; base < P.B; base += kSetupThreads) {
    const int b = base + threadIdx.x;
    int k = 0;
    if (b < P.B) {
      k = P.k_per_req[b];
      if (one) {
        T1 = P.temperature[b];
        tp1 = P.top_p ? P.top_p[b] : 1.0f;
        tk1 = P.top_k ? P.top_k[b] : 0;
      }
      if (k < 0 || k > SV_MAX_K) {
        record_error(w.hdr, SV_ERR_DATA_K, b, -1);
        atomicOr(&s_bad, 1);
        k = 0;
      }
    }
    unsigned long long tot;
    const unsigned long long ex =
        block_exclusive_scan(b < P.B ? pack2(uint32_t(k + 1), uint32_t(k)) : 0ull, &tot);
    if (b < P.B) w.t_off[b] = carry + int(uint32_t(ex));
    k1 = k;
    t01 = carry + int(uint32_t(ex));
    carry += int(uint32_t(tot));
    carry_d += int(uint32_t(tot >> 32));
  }
  if (threadIdx.x == 0) {
    w.t_off[P.B] = carry;
    if (!s_bad && (carry != P.Rt || carry_d != P.Rd)) {
      record_error(w.hdr, SV_ERR_DATA_ROWS, -1, -1);
      s_bad = 1;
    }
    if (s_bad) w.hdr->global_err = 1;
  }
  __syncthreads();
  if (s_bad) return;

  // Pass 2: per-request validation, modes, the active row list and the
  // post-pass job lists (filtered requests; all others).
  int carry_a = 0, carry_f = 0, carry_o = 0;
  for (int base = 0; base < P.B; base += kSetupThreads) {
    const int b = base + threadIdx.x;
    int code = 0, active = 0, mode_t = kSkip, mode_d = kSkip, k = 0, t0 = 0, d0 = 0;
    float T = 0.f;
    int tk = 0;
    if (b < P.B) {
      k = one ? k1 : P.k_per_req[b];
      t0 = one ? t01 : w.t_off[b];
      d0 = t0 - b;
      T = one ? T1 : P.temperature[b];
      const float tp = one ? tp1 : (P.top_p ? P.top_p[b] : 1.0f);
      tk = one ? tk1 : (P.top_k ? P.top_k[b] : 0);
      const bool topk_on = tk > 0 && tk < P.V;
      const bool filtered = T > 0.0f && (topk_on || tp < 1.0f);
      if (!(T >= 0.0f) || isinf(T)) code = SV_ERR_DATA_TEMPERATURE;
      else if (!(tp > 0.0f && tp <= 1.0f)) code = SV_ERR_DATA_TOP_P;
      else if (tk < 0) code = SV_ERR_DATA_TOP_K;
      else if (filtered && (!topk_on || tk > SV_TOPK_MAX)) code = SV_ERR_DATA_TOP_K;
      else if (T > 0.0f && k > 0 && P.draft == nullptr) code = SV_ERR_DATA_NO_DRAFT;
      if (!code) {
        // no early exit: the (at most SV_MAX_K) loads are independent
        bool bad = false;
#pragma unroll 8
        for (int i = 0; i < k; ++i) {
          const int x = P.draft_tokens[d0 + i];
          bad |= x < 0 || x >= P.V;
        }
        if (bad) code = SV_ERR_DATA_TOKEN;
      }
      w.req_flag[b] = code;
      if (code) {
        record_error(w.hdr, code, b, -1);
      } else if (T == 0.0f) {
        mode_t = kArgmax;
        active = k + 1;
      } else {
        mode_t = mode_d = filtered ? kTopk : kStats;
        active = 2 * k + 1;
      }
    }
    const bool filt = !code && mode_t == kTopk;
    // active rows (low half); filtered requests and the others (high half,
    // 16 bits each: a chunk holds at most kSetupThreads requests)
    unsigned long long tot;
    const uint32_t fo = b < P.B ? (filt ? 1u : 1u << 16) : 0u;
    const unsigned long long ex = block_exclusive_scan(pack2(uint32_t(active), fo), &tot);
    const int a0 = carry_a + int(uint32_t(ex));
    const int f0 = carry_f + int((ex >> 32) & 0xffffu);
    const int o0 = carry_o + int(ex >> 48);
    carry_a += int(uint32_t(tot));
    carry_f += int((tot >> 32) & 0xffffu);
    carry_o += int(tot >> 48);
    if (b < P.B) {
      w.seg_cnt[b] = 0;
      if (filt)
        w.job[f0] = make_int4(b, 0, t0, k);
      else
        w.job[P.B + o0] = make_int4(b, 0, t0, k);
    }
    if (b < P.B && active) {
      int a = a0;
      for (int i = 0; i <= k; ++i) {
        const int gx = i < k ? P.draft_tokens[d0 + i] : -1;
        w.rowlist[a++] = RowJob{t0 + i, b, gx, (i << 2) | mode_t, T, tk, {0, 0}};
      }
      if (mode_d != kSkip)
        for (int i = 0; i < k; ++i)
          w.rowlist[a++] = RowJob{(int)P.Rt + d0 + i, b, P.draft_tokens[d0 + i],
                                  (i << 2) | mode_d, T, tk, {0, 0}};
    }
    if (b < P.B && (code || mode_d == kSkip)) {
      // Rows the streaming pass will not visit still get a defined record.
      for (int i = 0; i < k; ++i) {
        RowStat& st = w.stats[P.Rt + d0 + i];
        st.s = 0.0;
        st.pg = __longlong_as_double(0x7ff8000000000000LL);
        st.m = 0.0f;
        st.arg = -1;
        st.kept = 0;
        st.mode = kSkip;
      }
    }
  }
  if (threadIdx.x == 0) {
    w.hdr->n_active = carry_a;
    w.hdr->n_filtered = carry_f;
    w.hdr->n_decide = carry_o;
  }
}

// Setup of the draft sampler: one CTA.  Request b owns drafter rows
// d_off[b] .. d_off[b] + k_b - 1 with d_off[b] = sum_{j<b} k_j (the verifier's
// draft-row layout).  Validates each request's parameters, writes the row list
// (every row of a valid request; mode argmax at T = 0, top-k survivors when
// the request filters, softmax statistics otherwise) and gives the rows of a
// failed request their outputs (-1, NaN) here.
__global__ void __launch_bounds__(kSetupThreads) sample_setup_kernel(const Problem P) {
  const Ws& w = P.ws;
  __shared__ int s_bad;
  pdl_trigger();  // the row pass may launch and set up; it waits for this kernel
  if (threadIdx.x == 0) {
    w.hdr->err_code = 0;
    w.hdr->err_req = -1;
    w.hdr->err_row = -1;
    w.hdr->n_active = 0;
    w.hdr->global_err = 0;
    w.hdr->n_filtered = 0;
    w.hdr->n_decide = 0;
    w.hdr->n_draw = 0;
    w.hdr->next_row = 0;
    s_bad = 0;
  }
  // every row may queue a draw: their segment counters start at zero
  for (int64_t q = threadIdx.x; q < P.Rt; q += kSetupThreads) w.seg_cnt[q] = 0;
  __syncthreads();

  // Pass 1: row offsets; a k outside [0, SV_MAX_K] makes the layout undefined.
  int carry = 0;
  for (int base = 0; base < P.B; base += kSetupThreads) {
    const int b = base + threadIdx.x;
    int k = 0;
    if (b < P.B) {
      k = P.k_per_req[b];
      if (k < 0 || k > SV_MAX_K) {
        record_error(w.hdr, SV_ERR_DATA_K, b, -1);
        atomicOr(&s_bad, 1);
        k = 0;
      }
    }
    unsigned long long tot;
    const unsigned long long ex = block_exclusive_scan(b < P.B ? pack2(uint32_t(k), 0u) : 0ull, &tot);
    if (b < P.B) w.t_off[b] = carry + int(uint32_t(ex));
    carry += int(uint32_t(tot));
  }
  if (threadIdx.x == 0) {
    w.t_off[P.B] = carry;
    if (!s_bad && carry != P.Rt) {
      record_error(w.hdr, SV_ERR_DATA_ROWS, -1, -1);
      s_bad = 1;
    }
    if (s_bad) w.hdr->global_err = 1;
  }
  __syncthreads();
  if (s_bad) return;

  // Pass 2: per-request validation, modes and the row list.
  int carry_a = 0;
  for (int base = 0; base < P.B; base += kSetupThreads) {
    const int b = base + threadIdx.x;
    int code = 0, active = 0, mode = kSkip, k = 0, d0 = 0, tk = 0;
    float T = 0.f;
    if (b < P.B) {
      k = P.k_per_req[b];
      d0 = w.t_off[b];
      T = P.temperature[b];
      const float tp = P.top_p ? P.top_p[b] : 1.0f;
      tk = P.top_k ? P.top_k[b] : 0;
      const bool topk_on = tk > 0 && tk < P.V;
      const bool filtered = T > 0.0f && (topk_on || tp < 1.0f);
      if (!(T >= 0.0f) || isinf(T)) code = SV_ERR_DATA_TEMPERATURE;
      else if (!(tp > 0.0f && tp <= 1.0f)) code = SV_ERR_DATA_TOP_P;
      else if (tk < 0) code = SV_ERR_DATA_TOP_K;
      else if (filtered && (!topk_on || tk > SV_TOPK_MAX)) code = SV_ERR_DATA_TOP_K;
      w.req_flag[b] = code;
      if (code) {
        record_error(w.hdr, code, b, -1);
        for (int i = 0; i < k; ++i) {
          P.out_tokens[d0 + i] = -1;
          if (P.out_q) P.out_q[d0 + i] = __int_as_float(0x7fc00000);
        }
      } else {
        mode = T == 0.0f ? kArgmax : (filtered ? kTopk : kStats);
        active = k;
      }
    }
    unsigned long long tot;
    const int a0 = carry_a + int(uint32_t(block_exclusive_scan(uint32_t(active), &tot)));
    carry_a += int(uint32_t(tot));
    for (int i = 0; i < active; ++i)
      w.rowlist[a0 + i] = RowJob{d0 + i, b, -1, (i << 2) | mode, T, tk, {0, 0}};
  }
  if (threadIdx.x == 0) w.hdr->n_active = carry_a;
}

}  // namespace

cudaError_t launch_sample_setup(const Problem& P, cudaStream_t s) {
  sample_setup_kernel<<<1, kSetupThreads, 0, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_setup(const Problem& P, cudaStream_t s) {
  setup_kernel<<<1, kSetupThreads, 0, s>>>(P);
  return cudaGetLastError();
}

}  // namespace sv
