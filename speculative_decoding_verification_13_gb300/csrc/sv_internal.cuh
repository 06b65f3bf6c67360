// Internal declarations of libspecverify: workspace layout, kernel parameter
// block and small device helpers (inline PTX for mbarriers, bulk copies and
// named barriers).  Nothing here is shared with the oracle.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/specverify.h"

namespace sv {

// ---------------------------------------------------------------- constants
constexpr int kConsumerWarps = 8;                        // warps that read tiles
constexpr int kConsumers = kConsumerWarps * 32;          // 256 threads
constexpr int kRowpassThreads = kConsumers + 32;         // + one producer warp
constexpr int kRowpassCtasPerSm = 2;                     // one CTA's epilogue overlaps
                                                         // the other's streaming
constexpr int kTileBytes = 16384;                        // one bulk copy
constexpr int kStages = 4;                               // smem ring depth per CTA
constexpr int kBufCap = 2560;                            // top-k candidate buffer
constexpr int kRegion = kBufCap / kConsumerWarps;        // per-warp region (fast path)
constexpr int kRawCap = 1024;                            // top-k survivors kept per row
constexpr int kScratch = 1024;                           // selection scratch entries
constexpr int kStage = 64;                               // staged flagged vectors per warp
constexpr int kTopkMax = SV_TOPK_MAX;
constexpr uint64_t kWaitNs = 100ull * 1000 * 1000;       // a wait gives up after 100 ms
constexpr uint32_t kWaitPolls = 1u << 28;                // ... or after this many polls
constexpr uint64_t kTestWaitNs = 1000ull * 1000;         // the expiring test wait: 1 ms
constexpr int kMaxSeg = 16;                              // draw-pass segments per row (at most)
constexpr int kDrawUnitsPerCta = 8;                      // draw-pass units per resident CTA (target)
// Vocabularies up to this size draw the final token of a decide job in the
// deciding warp: a pass for S and one for the crossing over a few tiles cost
// less than the two dependent launches of the draw pass and the locate kernel.
constexpr int kInlineDrawV = 2048;

// Row modes chosen per request by the setup kernel.  kTopk: a filtered row
// whose top-k is active and at most SV_TOPK_MAX (candidates captured in one
// pass, kept set materialised by the filter kernel); kBig: any other filtered
// row (top-p alone, or a larger top-k), whose kept set is a threshold on the
// composite key found by the row pass itself.
enum RowMode : int { kSkip = 0, kStats = 1, kArgmax = 2, kTopk = 3, kBig = 4 };
constexpr int kModeBits = 3;   // RowJob::mode = (position << kModeBits) | row mode
constexpr int kModeMask = 7;
constexpr int kBigPasses = 3;  // streams of a kBig row: max, histogram, collection

// ---------------------------------------------------------------- workspace
struct WsHeader {
  int32_t err_code;
  int32_t err_req;
  int64_t err_row;
  int32_t n_active;     // rows the row pass must stream
  int32_t global_err;   // batch-level data error (row counts)
  int32_t n_filtered;   // filtered requests listed by the setup kernel
  int32_t n_decide;     // other requests listed by the setup kernel
  int32_t n_draw;       // requests queued for the unfiltered draw
  int32_t next_row;     // draft sampler: rows handed out to warps so far
  int32_t rp_next;      // row pass: rows claimed past each CTA's first
  int32_t n_big;        // kBig rows, listed from the end of the row list
  int32_t rp_next_big;  // row pass over the kBig rows: rows claimed past each CTA's first
  int32_t dp_next;      // draw pass: units claimed past each CTA's first
  int32_t pad[2];
};

struct RowStat {
  double s;     // softmax normaliser (sampling rows; kept-set weight for filtered rows,
                // relative to the row max m for kBig rows)
  double pg;    // p(x) of the row's draft token
  float m;      // row max logit
  int32_t arg;  // greedy argmax
  int32_t kept; // filtered rows: survivors after the row pass, then the kept-set size
  int32_t mode;
};

// What the unfiltered draw of one request needs (written by its decide job).
struct DrawDesc {
  int64_t tr, dr;  // target row p_L, draft row q_L (residual only)
  float mt, ist;   // target row max and 1 / normaliser
  float md, isd;   // draft row max and 1 / normaliser
  float c2;        // log2(e) / T
  int32_t kind;    // 0 bonus p_k, 1 residual max(0, p_L - q_L), 2 residual fallback p_L
  double u;        // the final uniform u_k
  int32_t t0, L;
  // kept sets of kBig rows: the element y of a row is kept iff its composite
  // key is >= the row's threshold (0 keeps every element: unfiltered rows)
  uint64_t kt, kd;
};

// One entry of the row pass's work list, in request order (setup kernel).
// The row pass reads the first six fields as 32-bit words, in this order.
struct __align__(16) RowJob {
  int32_t row;   // target rows 0 .. R_t - 1, then draft rows R_t ..
  int32_t b;     // request
  int32_t gx;    // token whose probability the row reports, or -1
  int32_t mode;  // (position << kModeBits) | row mode
  float T;       // the request's temperature
  int32_t K;     // the request's top-k (filtered rows)
  int32_t pad[2];
};
static_assert(sizeof(RowJob) == 32, "row job layout");

struct Ws {
  WsHeader* hdr;
  int32_t* t_off;    // [B + 1]
  int32_t* req_flag; // [B]
  RowJob* rowlist;   // [R] rows the row pass streams: the hdr->n_active others
                     // from the front, the hdr->n_big kBig rows from the back
                     // (kBig row j at R - 1 - j)
  RowStat* stats;    // [R]
  int32_t* cand_idx; // [R, kTopkMax]
  float* cand_p;     // [R, kTopkMax] kept probabilities
  uint64_t* cand_raw; // [R, kRawCap] top-k survivors of the row pass (composite keys);
                      // kBig rows: slot 0 holds the kept-set threshold key
  int4* job;          // [2B] {request, 0, t_off, k}: filtered requests from 0,
                      //      the other requests from B
  DrawDesc* draw;     // [B] queued draws, in queue order
  double* seg_sum;    // [B, kMaxSeg] weight sum of each segment of a queued draw
  int32_t* seg_cnt;   // [B] segments of a queued draw finished
};

struct WsLayout {
  size_t off_t_off, off_flag, off_rowlist, off_stats, off_cidx, off_cp, off_raw, off_job,
      off_draw, off_seg, off_scnt, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t B, int64_t Rt, int64_t Rd) {
  WsLayout L;
  const int64_t R = Rt + Rd;
  size_t o = align256(sizeof(WsHeader));
  L.off_t_off = o;   o = align256(o + sizeof(int32_t) * (size_t)(B + 1));
  L.off_flag = o;    o = align256(o + sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
  L.off_rowlist = o; o = align256(o + sizeof(RowJob) * (size_t)(R > 0 ? R : 1));
  L.off_stats = o;   o = align256(o + sizeof(RowStat) * (size_t)(R > 0 ? R : 1));
  L.off_cidx = o;    o = align256(o + sizeof(int32_t) * kTopkMax * (size_t)(R > 0 ? R : 1));
  L.off_cp = o;      o = align256(o + sizeof(float) * kTopkMax * (size_t)(R > 0 ? R : 1));
  L.off_raw = o;     o = align256(o + sizeof(uint64_t) * kRawCap * (size_t)(R > 0 ? R : 1));
  const size_t B1 = (size_t)(B > 0 ? B : 1);
  L.off_job = o;     o = align256(o + sizeof(int4) * 2 * B1);
  L.off_draw = o;    o = align256(o + sizeof(DrawDesc) * B1);
  L.off_seg = o;     o = align256(o + sizeof(double) * kMaxSeg * B1);
  L.off_scnt = o;    o = align256(o + sizeof(int32_t) * B1);
  L.total = o;
  return L;
}

// Draft sampler: per-queue arrays hold one entry per row (every sampled row
// may queue a draw), per-request arrays one per request.
inline WsLayout sample_ws_layout(int64_t B, int64_t R) {
  return ws_layout(B > R ? B : R, R, 0);
}

inline Ws ws_bind(void* base, const WsLayout& L) {
  char* p = static_cast<char*>(base);
  Ws w;
  w.hdr = reinterpret_cast<WsHeader*>(p);
  w.t_off = reinterpret_cast<int32_t*>(p + L.off_t_off);
  w.req_flag = reinterpret_cast<int32_t*>(p + L.off_flag);
  w.rowlist = reinterpret_cast<RowJob*>(p + L.off_rowlist);
  w.stats = reinterpret_cast<RowStat*>(p + L.off_stats);
  w.cand_idx = reinterpret_cast<int32_t*>(p + L.off_cidx);
  w.cand_p = reinterpret_cast<float*>(p + L.off_cp);
  w.cand_raw = reinterpret_cast<uint64_t*>(p + L.off_raw);
  w.job = reinterpret_cast<int4*>(p + L.off_job);
  w.draw = reinterpret_cast<DrawDesc*>(p + L.off_draw);
  w.seg_sum = reinterpret_cast<double*>(p + L.off_seg);
  w.seg_cnt = reinterpret_cast<int32_t*>(p + L.off_scnt);
  return w;
}

// Everything a kernel needs about one call.
struct Problem {
  const void* target;
  const void* draft;
  int64_t t_stride, d_stride;   // elements
  int64_t Rt, Rd;
  int32_t V;
  int32_t B;
  int32_t n_seg;                // draw-pass segments per queued draw (1..kMaxSeg)
  int32_t test_expire;          // test only: one bounded wait of the row pass expires
  int32_t inline_draw;          // rows of at most kInlineDrawV elements: decide jobs draw
                                // their final token in place (no draw pass, no locate)
  const int32_t* draft_tokens;
  const int32_t* k_per_req;
  const float* temperature;
  const int32_t* top_k;         // may be null
  const float* top_p;           // may be null
  const float* uniforms;
  int32_t* out_accept_len;
  int32_t* out_tokens;
  double* out_pq;               // may be null
  float* out_q;                 // draft sampler: q(x) of each drawn token, may be null
  Ws ws;
};

// ------------------------------------------------------- host-side launchers
cudaError_t launch_setup(const Problem& P, cudaStream_t s);
cudaError_t launch_rowpass(const Problem& P, bool bf16, bool big, int grid, cudaStream_t s);
cudaError_t launch_filter_decide(const Problem& P, bool bf16, int grid, cudaStream_t s);
cudaError_t launch_draw(const Problem& P, bool bf16, int grid, cudaStream_t s);
cudaError_t launch_locate(const Problem& P, bool bf16, int grid, cudaStream_t s);
cudaError_t launch_sample_setup(const Problem& P, cudaStream_t s);
size_t kv_workspace_bytes(int32_t B);
size_t lmhead_workspace_bytes(int M, int V);
cudaError_t launch_adapt_k(const int32_t* accept_len, const int32_t* k_used, double* succ,
                           double* fail, double decay, double c, int k_min, int k_max,
                           int32_t* k_next, float* alpha, int B, cudaStream_t s);
int launch_lmhead_stats(const void* H, const void* W, int M, int V, int K,
                        const float* temperature, const int32_t* tokens, float* out_m,
                        double* out_s, int32_t* out_arg, float* out_xt, void* workspace,
                        int sms, cudaStream_t s);
cudaError_t launch_kv_commit(void* cache, const void* spec, int64_t num_pages, int n_layers,
                             int page_size, int64_t entry_bytes, int spec_slots,
                             const int32_t* accept_len, const int32_t* k_per_req,
                             int32_t* kv_len, const int32_t* block_table, int max_pages, int B,
                             void* workspace, int sms, cudaStream_t s);
cudaError_t launch_sample_post(const Problem& P, bool bf16, int grid, cudaStream_t s);
cudaError_t launch_greedy_from_argmax(const int32_t* argmax, const int32_t* draft_tokens,
                                      const int32_t* k_per_req, int32_t* out_accept_len,
                                      int32_t* out_tokens, int B, int64_t Rt, int V,
                                      void* workspace, cudaStream_t s);
size_t rowpass_smem_bytes();

// Launch of a kernel that may start while the previous kernel on the stream
// finishes (programmatic dependent launch): it must execute pdl_wait() before
// touching memory that the previous kernel writes or reads.
template <class Kern>
inline cudaError_t launch_after(Kern kernel, int grid, int threads, size_t smem, cudaStream_t s,
                                const Problem& P) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

// ------------------------------------------------------------ device helpers
#ifdef __CUDACC__

__device__ __forceinline__ void record_error(WsHeader* h, int code, int req, int64_t row) {
  if (atomicCAS(&h->err_code, 0, code) == 0) {
    h->err_req = req;
    h->err_row = row;
  }
}

__device__ __forceinline__ void flag_request(const Ws& w, int b, int code, int64_t row) {
  atomicCAS(&w.req_flag[b], 0, code);
  record_error(w.hdr, code, b, row);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Nanoseconds of the GPU's global timer (wall-clock time).
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: true once the phase completes; false
// after limit_ns of GPU wall-clock time without completion, after kWaitPolls
// polls, or as soon as one of the optional abort flags is set (both checked
// every 256 polls).  The caller records SV_ERR_TIMEOUT.  sleep_ns: back-off
// between polls, so that a waiting warp leaves the issue slots to the warps
// that work.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity,
                                              uint64_t limit_ns = kWaitNs,
                                              const int* f1 = nullptr, const int* f2 = nullptr,
                                              uint32_t sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1; it < kWaitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (f1 && *reinterpret_cast<const volatile int*>(f1)) return false;
      if (f2 && *reinterpret_cast<const volatile int*>(f2)) return false;
      if (global_ns() - t0 > limit_ns) return false;
    }
    if (sleep_ns) __nanosleep(sleep_ns);
  }
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  return mbar_wait_for(bar, parity);
}

// One bulk global -> shared copy completing on an mbarrier (TMA, non-tensor form).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// L2 policy for data read once and not again in this call (the logit rows):
// evicted first, so that streaming them does not push the call's small
// working set (row records, survivor lists, code) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_load with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Programmatic dependent launch: wait until the previous kernel on the stream
// has completed and its writes are visible (a no-op when the kernel was
// launched normally); let the next kernel on the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier among the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Packed pairs of floats for the f32x2 instructions (two IEEE round-to-nearest
// operations each, bit for bit those of the scalar forms): one issue for the
// arithmetic of two elements.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Total order used by top-k: (logit descending, index ascending).  The key is
// the order-preserving unsigned image of the float (with -0 folded onto +0);
// the low word holds ~index so that a smaller index compares larger.
__device__ __forceinline__ uint64_t composite_key(float v, uint32_t idx) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  const uint32_t key = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~idx);
}

__device__ __forceinline__ float composite_value(uint64_t c) {
  const uint32_t key = static_cast<uint32_t>(c >> 32);
  const uint32_t b = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(b);
}

__device__ __forceinline__ int32_t composite_index(uint64_t c) {
  return static_cast<int32_t>(~static_cast<uint32_t>(c));
}

// ceil(W * p) for 0 < p < 1 (a float), exactly: p = m 2^-s with m < 2^24 and
// s >= 24, and W * m has at most 88 bits.
__device__ __forceinline__ unsigned long long ceil_mul_frac(unsigned long long W, float p) {
  const uint32_t b = __float_as_uint(p);
  const uint32_t E = b >> 23;
  const unsigned long long m = E ? ((b & 0x7fffffu) | 0x800000u) : (b & 0x7fffffu);
  const int s = E ? 150 - int(E) : 149;
  const unsigned long long lo = W * m, hi = __umul64hi(W, m);
  unsigned long long q;
  bool rem;
  if (s < 64) {
    q = (hi << (64 - s)) | (lo >> s);
    rem = (lo & ((1ull << s) - 1ull)) != 0ull;
  } else {
    const int t = s - 64;
    q = t < 64 ? (hi >> t) : 0ull;
    rem = lo != 0ull || (t < 64 ? (hi & ((1ull << t) - 1ull)) != 0ull : hi != 0ull);
  }
  return q + (rem ? 1ull : 0ull);
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

#endif  // __CUDACC__

}  // namespace sv
