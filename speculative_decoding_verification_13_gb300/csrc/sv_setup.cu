// Setup kernel: one CTA per call.  Computes the ragged row offsets
// t_off[b] = sum_{j<b} (k_j + 1), validates every request's parameters and
// drafted tokens, picks each row's mode, writes the list of rows the
// streaming pass must read (ordered by request) and the list of post-pass jobs,
// and zeroes the per-request counters the post-pass kernels count with.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kSetupThreads = 1024;
constexpr int kSetupCtas = 8;  // CTAs that share the row-list writes

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

// One request of the current chunk, as the row-list fill needs it.
struct ReqRows {
  int a0;      // first entry of the request in the row list
  int t0, d0;  // first target row, first draft row (relative to R_t)
  int k;       // drafts
  int active;  // entries: k + 1 target rows, then the k draft rows when streamed
  int modes;   // target row mode | draft row mode << 8 | 1 << 16 when the
               // draft rows are not streamed (they get a defined record here)
  int tk;      // top-k
  float T;     // temperature
  int big;     // the rows are kBig rows: listed from the end of the row list
};

// Writes the row list of the chunk's requests, one warp per request, so that
// consecutive lanes write consecutive 32-byte entries (a thread walking its
// own request's entries would leave every store uncoalesced).  The requests
// are spread over the warps of every CTA of the grid: the list is a few
// hundred KB, more than one SM writes out quickly.
__device__ void fill_rows(const Problem& P, const ReqRows* rq, int base, int nb) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  constexpr int kW = kSetupThreads / 32;
  for (int r = blockIdx.x * kW + (threadIdx.x >> 5); r < nb; r += gridDim.x * kW) {
    const ReqRows q = rq[r];
    const int last = int(P.Rt + P.Rd) - 1;
    for (int e = lane; e < q.active; e += 32) {
      const bool tgt = e <= q.k;
      const int i = tgt ? e : e - q.k - 1;
      const int row = tgt ? q.t0 + i : int(P.Rt) + q.d0 + i;
      const int gx = i < q.k ? P.draft_tokens[q.d0 + i] : -1;
      const int mode = (i << kModeBits) | (tgt ? (q.modes & 0xff) : ((q.modes >> 8) & 0xff));
      int4* dst = reinterpret_cast<int4*>(w.rowlist + (q.big ? last - (q.a0 + e) : q.a0 + e));
      dst[0] = make_int4(row, base + r, gx, mode);
      dst[1] = make_int4(__float_as_int(q.T), q.tk, 0, 0);
    }
    if (q.modes >> 16)
      // Rows the streaming pass will not visit still get a defined record.
      for (int i = lane; i < q.k; i += 32) {
        RowStat st;
        st.s = 0.0;
        st.pg = __longlong_as_double(0x7ff8000000000000LL);
        st.m = 0.0f;
        st.arg = -1;
        st.kept = 0;
        st.mode = kSkip;
        w.stats[P.Rt + q.d0 + i] = st;
      }
  }
}

__global__ void __launch_bounds__(kSetupThreads) setup_kernel(const Problem P) {
  const Ws& w = P.ws;
  __shared__ int s_bad;
  __shared__ ReqRows s_req[kSetupThreads];
  // launched as a dependent of whatever the stream ran before (the previous
  // call's last kernel, or the kernel that produced the inputs): nothing is
  // read or written before that has completed
  pdl_wait();
  pdl_trigger();  // the row pass may launch and set up; it waits for this kernel
  // Every CTA forms the same offsets, modes and scans; CTA 0 alone writes the
  // header, the offsets, the flags and the job lists, and each CTA writes its
  // share of the row list.  (More than one CTA only when B <= kSetupThreads.)
  const bool lead = blockIdx.x == 0;
  if (threadIdx.x == 0) {
    if (lead) {
      w.hdr->err_code = 0;
      w.hdr->err_req = -1;
      w.hdr->err_row = -1;
      w.hdr->n_active = 0;
      w.hdr->global_err = 0;
      w.hdr->n_filtered = 0;
      w.hdr->n_decide = 0;
      w.hdr->n_draw = 0;
      w.hdr->rp_next = 0;
      w.hdr->n_big = 0;
      w.hdr->rp_next_big = 0;
      w.hdr->dp_next = 0;
    }
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
        if (lead) record_error(w.hdr, SV_ERR_DATA_K, b, -1);
        atomicOr(&s_bad, 1);
        k = 0;
      }
    }
    unsigned long long tot;
    const unsigned long long ex =
        block_exclusive_scan(b < P.B ? pack2(uint32_t(k + 1), uint32_t(k)) : 0ull, &tot);
    if (b < P.B && lead) w.t_off[b] = carry + int(uint32_t(ex));
    k1 = k;
    t01 = carry + int(uint32_t(ex));
    carry += int(uint32_t(tot));
    carry_d += int(uint32_t(tot >> 32));
  }
  if (threadIdx.x == 0) {
    if (!s_bad && (carry != P.Rt || carry_d != P.Rd)) {
      if (lead) record_error(w.hdr, SV_ERR_DATA_ROWS, -1, -1);
      s_bad = 1;
    }
    if (lead) {
      w.t_off[P.B] = carry;
      if (s_bad) w.hdr->global_err = 1;
    }
  }
  __syncthreads();
  if (s_bad) return;

  // Pass 2: per-request validation, modes, the active row list and the
  // post-pass job lists (filtered requests; all others).
  int carry_a = 0, carry_g = 0, carry_f = 0, carry_o = 0;
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
      if (lead) {
        w.req_flag[b] = code;
        if (code) record_error(w.hdr, code, b, -1);
      }
      if (code == 0 && T == 0.0f) {
        mode_t = kArgmax;
        active = k + 1;
      } else if (code == 0) {
        // a small top-k takes the candidate path; top-p alone and larger
        // top-k take the threshold path
        mode_t = mode_d = !filtered ? kStats : (topk_on && tk <= SV_TOPK_MAX ? kTopk : kBig);
        active = 2 * k + 1;
      }
    }
    const bool filt = !code && mode_t == kTopk;
    const bool big = !code && mode_t == kBig;
    // four counters in one word: other active rows (bits 0-19), kBig rows
    // (20-39), filtered requests (40-51) and the other requests (52-63); a
    // chunk holds at most kSetupThreads requests of at most 2 SV_MAX_K + 1
    // rows each
    static_assert(kSetupThreads * (2 * SV_MAX_K + 1) < (1 << 20) && kSetupThreads < (1 << 12),
                  "setup scan fields");
    unsigned long long tot;
    const unsigned long long fo =
        b < P.B ? (filt ? 1ull << 40 : 1ull << 52) : 0ull;
    const unsigned long long ex = block_exclusive_scan(
        (big ? uint64_t(active) << 20 : uint64_t(active)) | fo, &tot);
    const int a0 = big ? carry_g + int((ex >> 20) & 0xfffffu) : carry_a + int(ex & 0xfffffu);
    const int f0 = carry_f + int((ex >> 40) & 0xfffu);
    const int o0 = carry_o + int(ex >> 52);
    carry_a += int(tot & 0xfffffu);
    carry_g += int((tot >> 20) & 0xfffffu);
    carry_f += int((tot >> 40) & 0xfffu);
    carry_o += int(tot >> 52);
    if (b < P.B && lead) {
      w.seg_cnt[b] = 0;
      if (filt)
        w.job[f0] = make_int4(b, 0, t0, k);
      else
        w.job[P.B + o0] = make_int4(b, 0, t0, k);
    }
    s_req[threadIdx.x] =
        ReqRows{a0, t0, d0, k, b < P.B ? active : 0,
                mode_t | (mode_d << 8) | (b < P.B && mode_d == kSkip ? 1 << 16 : 0), tk, T,
                big ? 1 : 0};
    __syncthreads();
    fill_rows(P, s_req, base, min(kSetupThreads, P.B - base));
    __syncthreads();  // s_req is rewritten by the next chunk
  }
  if (threadIdx.x == 0 && lead) {
    w.hdr->n_active = carry_a;
    w.hdr->n_big = carry_g;
    w.hdr->n_filtered = carry_f;
    w.hdr->n_decide = carry_o;
  }
}

// The draft sampler's row list, one warp per request (coalesced entries):
// request b's drafter rows d_off[b] + i, i < k_b, all in the request's mode,
// reporting no token.
__device__ void fill_sample_rows(const Problem& P, const ReqRows* rq, int base, int nb) {
  const Ws& w = P.ws;
  const int lane = threadIdx.x & 31;
  constexpr int kW = kSetupThreads / 32;
  for (int r = blockIdx.x * kW + (threadIdx.x >> 5); r < nb; r += gridDim.x * kW) {
    const ReqRows q = rq[r];
    const int last = int(P.Rt) - 1;
    for (int i = lane; i < q.active; i += 32) {
      int4* dst = reinterpret_cast<int4*>(w.rowlist + (q.big ? last - (q.a0 + i) : q.a0 + i));
      dst[0] = make_int4(q.t0 + i, base + r, -1, (i << kModeBits) | q.modes);
      dst[1] = make_int4(__float_as_int(q.T), q.tk, 0, 0);
    }
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
  __shared__ ReqRows s_req[kSetupThreads];
  // launched as a dependent of whatever the stream ran before (the previous
  // call's last kernel, or the kernel that produced the inputs): nothing is
  // read or written before that has completed
  pdl_wait();
  pdl_trigger();  // the row pass may launch and set up; it waits for this kernel
  // As in the verifier's setup: CTA 0 writes the header, offsets, flags and
  // the outputs of failed requests; every CTA writes its share of the row
  // list and of the zeroed counters.
  const bool lead = blockIdx.x == 0;
  if (threadIdx.x == 0 && lead) {
    w.hdr->err_code = 0;
    w.hdr->err_req = -1;
    w.hdr->err_row = -1;
    w.hdr->n_active = 0;
    w.hdr->global_err = 0;
    w.hdr->n_filtered = 0;
    w.hdr->n_decide = 0;
    w.hdr->n_draw = 0;
    w.hdr->next_row = 0;
    w.hdr->rp_next = 0;
    w.hdr->n_big = 0;
    w.hdr->rp_next_big = 0;
    w.hdr->dp_next = 0;
  }
  if (threadIdx.x == 0) s_bad = 0;
  // every row may queue a draw: their segment counters start at zero
  for (int64_t q = int64_t(blockIdx.x) * kSetupThreads + threadIdx.x; q < P.Rt;
       q += int64_t(gridDim.x) * kSetupThreads)
    w.seg_cnt[q] = 0;
  __syncthreads();

  // Pass 1: row offsets; a k outside [0, SV_MAX_K] makes the layout undefined.
  // With a single chunk (B <= kSetupThreads) each offset stays in a register.
  const bool one = P.B <= kSetupThreads;
  int d01 = 0;
  int carry = 0;
  for (int base = 0; base < P.B; base += kSetupThreads) {
    const int b = base + threadIdx.x;
    int k = 0;
    if (b < P.B) {
      k = P.k_per_req[b];
      if (k < 0 || k > SV_MAX_K) {
        if (lead) record_error(w.hdr, SV_ERR_DATA_K, b, -1);
        atomicOr(&s_bad, 1);
        k = 0;
      }
    }
    unsigned long long tot;
    const unsigned long long ex = block_exclusive_scan(b < P.B ? pack2(uint32_t(k), 0u) : 0ull, &tot);
    if (b < P.B && lead) w.t_off[b] = carry + int(uint32_t(ex));
    d01 = carry + int(uint32_t(ex));
    carry += int(uint32_t(tot));
  }
  if (threadIdx.x == 0) {
    if (!s_bad && carry != P.Rt) {
      if (lead) record_error(w.hdr, SV_ERR_DATA_ROWS, -1, -1);
      s_bad = 1;
    }
    if (lead) {
      w.t_off[P.B] = carry;
      if (s_bad) w.hdr->global_err = 1;
    }
  }
  __syncthreads();
  if (s_bad) return;

  // Pass 2: per-request validation, modes and the row list.
  int carry_a = 0, carry_g = 0;
  for (int base = 0; base < P.B; base += kSetupThreads) {
    const int b = base + threadIdx.x;
    int code = 0, active = 0, mode = kSkip, k = 0, d0 = 0, tk = 0;
    float T = 0.f;
    if (b < P.B) {
      k = P.k_per_req[b];
      d0 = one ? d01 : w.t_off[b];
      T = P.temperature[b];
      const float tp = P.top_p ? P.top_p[b] : 1.0f;
      tk = P.top_k ? P.top_k[b] : 0;
      const bool topk_on = tk > 0 && tk < P.V;
      const bool filtered = T > 0.0f && (topk_on || tp < 1.0f);
      if (!(T >= 0.0f) || isinf(T)) code = SV_ERR_DATA_TEMPERATURE;
      else if (!(tp > 0.0f && tp <= 1.0f)) code = SV_ERR_DATA_TOP_P;
      else if (tk < 0) code = SV_ERR_DATA_TOP_K;
      if (code && lead) {
        w.req_flag[b] = code;
        record_error(w.hdr, code, b, -1);
        for (int i = 0; i < k; ++i) {
          P.out_tokens[d0 + i] = -1;
          if (P.out_q) P.out_q[d0 + i] = __int_as_float(0x7fc00000);
        }
      } else if (lead) {
        w.req_flag[b] = 0;
      }
      if (!code) {
        mode = T == 0.0f ? kArgmax
                         : (!filtered ? kStats : (topk_on && tk <= SV_TOPK_MAX ? kTopk : kBig));
        active = k;
      }
    }
    // other rows (low half), kBig rows (high half)
    const bool big = mode == kBig;
    unsigned long long tot;
    const unsigned long long ex =
        block_exclusive_scan(big ? pack2(0u, uint32_t(active)) : pack2(uint32_t(active), 0u), &tot);
    const int a0 = big ? carry_g + int(ex >> 32) : carry_a + int(uint32_t(ex));
    carry_a += int(uint32_t(tot));
    carry_g += int(tot >> 32);
    // fill_sample_rows reads a0, t0 (the first drafter row), active, modes, tk, T, big
    s_req[threadIdx.x] = ReqRows{a0, d0, 0, k, active, mode, tk, T, big ? 1 : 0};
    __syncthreads();
    fill_sample_rows(P, s_req, base, min(kSetupThreads, P.B - base));
    __syncthreads();  // s_req is rewritten by the next chunk
  }
  if (threadIdx.x == 0 && lead) {
    w.hdr->n_active = carry_a;
    w.hdr->n_big = carry_g;
  }
}

}  // namespace

// More than one CTA only with a single chunk of requests: the CTAs other than
// the first rely on the offsets they keep in registers.
int setup_grid(int64_t B) { return B <= kSetupThreads ? kSetupCtas : 1; }

cudaError_t launch_sample_setup(const Problem& P, cudaStream_t s) {
  return launch_after(sample_setup_kernel, setup_grid(P.B), kSetupThreads, 0, s, P);
}

cudaError_t launch_setup(const Problem& P, cudaStream_t s) {
  return launch_after(setup_kernel, setup_grid(P.B), kSetupThreads, 0, s, P);
}

}  // namespace sv
