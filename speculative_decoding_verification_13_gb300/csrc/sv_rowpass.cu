// Row pass: the one kernel that streams every logit row from HBM once.
//
// Persistent, two CTAs per SM.  Warp 0 is the producer: one lane claims rows of
// the active-row list (its CTA's index first, then the next unclaimed row
// from a counter, claimed a few tiles before the current row's last copy, so
// that CTAs streaming faster take more rows and all finish together) and
// issues TMA bulk copies
// (cp.async.bulk, 16 KB each) into a 4-stage shared-memory ring, each stage
// guarded by a "full" mbarrier (transaction bytes) and an "empty" mbarrier (one
// arrival per consumer warp).  Warps 1..8 consume the tiles and reduce each row
// in one of three modes (chosen per request by the setup kernel):
//   kStats  - temperature softmax statistics of a sampled, unfiltered row: the
//             row max M and S = sum_y exp((x_y - M) / T) by an online
//             (running-max, rescaled) sum; then p(x) = exp((x_x - M) / T) / S
//             of the row's draft token in double precision.
//             ("FlashMap…" §5 draft_block step 5: logits / T, softmax.)
//   kArgmax - greedy: argmax of the raw logits, lowest index on ties.
//   kTopk   - the top-k candidates of a filtered row: a speculative threshold
//             from the first tile (the r-th largest per-vector maximum), then
//             every tile's vectors are flagged against it, the flagged
//             vectors are staged per warp and their elements at or above it
//             become candidates; the survivors (at least
//             k, at most kRawCap) are published unsorted for the filter
//             kernel, which selects the exact top k.  A failed speculation is
//             redone exactly from global memory (certified radix selection).
//             ("Speculative decoding and multi-token prediction", "Why the
//             output is identical": the same filter on both distributions.)
//   kBig    - a row filtered by top-p alone or by a top-k above SV_TOPK_MAX:
//             streamed three times (max; histogram; the crossing bins), it
//             ends with the kept set's threshold key and mass (sv_bigrow.cuh).
// Every wait is bounded; on expiry the kernel records SV_ERR_TIMEOUT, stops
// issuing copies, lets the copies it issued land, and exits.
#include <math.h>

#include "sv_select.cuh"

namespace sv {
namespace {

constexpr size_t kOffBuf = size_t(kStages) * kTileBytes;
constexpr size_t kOffScratch = kOffBuf + size_t(kBufCap) * 8;
constexpr size_t kOffXchg = kOffScratch + size_t(kScratch) * 8;
constexpr size_t kOffBars = kOffXchg + size_t(2 * kConsumers) * 8;
constexpr size_t kOffStage = kOffBars + size_t(2 * kStages) * 8;
constexpr size_t kOffStageIdx = kOffStage + size_t(kConsumerWarps) * kStage * 16;
constexpr size_t kSmemBytes = kOffStageIdx + size_t(kConsumerWarps) * kStage * 4;
static_assert(kOffStage % 16 == 0, "staged vectors are 16-byte aligned");
static_assert(kRowpassCtasPerSm * (kSmemBytes + 4096 + 1024) <= 228 * 1024,
              "shared memory budget for the resident CTAs of one SM");

#include "sv_bigrow.cuh"

// kBig rows use the candidate buffer and the selection scratch (contiguous)
// as their work area: the histogram, then the band's keys.
static_assert(kOffScratch == kOffBuf + size_t(kBufCap) * 8, "contiguous work area");
static_assert(kBigWorkBytes <= size_t(kBufCap + kScratch) * 8, "kBig work area");
static_assert(size_t(kBigCap) * 8 <= size_t(kBufCap + kScratch) * 8, "kBig band keys");

struct RowShared {
  RowJob rowq[kStages];  // the row each ring phase starts (row = -1: no more rows)
  unsigned long long test_bar_word;  // an mbarrier nothing arrives on (timeout test)
  BigShared big;
  int hist[256];
  SelShared sel;
  unsigned long long thmin[3];
  unsigned int bnd[2];
  unsigned int ins[2];
  int count;
  int tmpcount;
  int ovf;
  int cabort;
  int pabort;
  int bad;
  unsigned int nbad;
  int kp;
  int wcnt[kConsumerWarps];
  float v0;
  double wp;
  double inv_wp;
  double pg;
  float red_f[kConsumerWarps];
  int red_i[kConsumerWarps];
  float red_hi[kConsumerWarps];
  float red_lo[kConsumerWarps];
  double red_d[kConsumerWarps];
};

struct ConsumerSync {
  __device__ void operator()() const { consumer_sync(); }
};

template <bool BF16>
struct Elt;

template <>
struct Elt<true> {
  static constexpr int kPerVec = 8;
  static constexpr int kSize = 2;
  __device__ static void decode(const uint4& q, float* x) {
    x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x); x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
    x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z); x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
  }
  // Largest element; NaN if any element is NaN.
  __device__ static float vmax(const uint4& q) {
    const uint32_t m = pmax(q);
    return fmax_nan(bf16_lo(m), bf16_hi(m));
  }
  // Packed maxima (even elements, odd elements) as bf16x2; NaN propagates.
  __device__ static uint32_t pmax(const uint4& q) {
    return bmax2_nan(bmax2_nan(q.x, q.y), bmax2_nan(q.z, q.w));
  }
  __device__ static float scalar(const void* row, int64_t i) {
    return __uint_as_float(uint32_t(static_cast<const uint16_t*>(row)[i]) << 16);
  }
  // Element e (0..7) of the vector.
  __device__ static float elem(const uint4& q, int e) {
    const uint32_t w = e < 4 ? (e < 2 ? q.x : q.y) : (e < 6 ? q.z : q.w);
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
};

template <>
struct Elt<false> {
  static constexpr int kPerVec = 4;
  static constexpr int kSize = 4;
  __device__ static void decode(const uint4& q, float* x) {
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
  }
  __device__ static float vmax(const uint4& q) {
    return fmax_nan(fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                    fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
  }
  __device__ static float scalar(const void* row, int64_t i) {
    return static_cast<const float*>(row)[i];
  }
  // Element e (0..3) of the vector.
  __device__ static float elem(const uint4& q, int e) {
    return __uint_as_float(e < 2 ? (e == 0 ? q.x : q.y) : (e == 2 ? q.z : q.w));
  }
};

// Bounded wait with back-off: a waiting warp sleeps between polls so that it
// does not take issue slots from the warps that do the work.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const int* f1,
                                              const int* f2, uint32_t sleep_ns) {
  return mbar_wait_for(bar, parity, kWaitNs, f1, f2, sleep_ns);
}

// A bf16 value d below v (v itself a bf16 value), in both halves of a
// bf16x2, such that every packed element h >= v has max(h, d) != d: the next
// bf16 below v, or -(smallest normal) when v is zero or subnormal (so that the
// comparison never hinges on a subnormal, which the packed max may treat as
// zero).  Elements between d and v are flagged too; flags are only a filter,
// the exact key comparison decides.  For v = -inf, and for the NaN that the
// empty threshold (key 0) decodes to, the pattern is a NaN, so every element
// is flagged.
__device__ __forceinline__ uint32_t bf16_below2(float v) {
  if (v != v) return 0xff81ff81u;
  const uint32_t b = __float_as_uint(v) >> 16;
  const uint32_t d = (b & 0x7f80u) == 0u ? 0x8080u : ((b & 0x8000u) ? b + 1u : b - 1u);
  return d | (d << 16);
}

// Descending bitonic sort of the 32 floats a warp holds, one per lane.
__device__ __forceinline__ float warp_sort_desc_f32(float u) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, u, j);
      const bool desc = (lane & size) == 0;
      const bool lower = (lane & j) == 0;
      u = (desc == lower) ? fmaxf(u, o) : fminf(u, o);
    }
  }
  return u;
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// BIG selects the rows a launch streams: false, every row other than the kBig
// rows (hdr->n_active, from the front of the row list); true, the kBig rows
// only (hdr->n_big, from the back).  The two are separate instantiations so
// that each compiles only its own modes.
template <bool BF16, bool BIG>
__global__ void __launch_bounds__(kRowpassThreads, kRowpassCtasPerSm) rowpass_kernel(const Problem P) {
  using E = Elt<BF16>;
  constexpr int EPV = E::kPerVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ RowShared S;
  unsigned char* ring = smem;
  uint64_t* buf = reinterpret_cast<uint64_t*>(smem + kOffBuf);
  uint64_t* scratch = reinterpret_cast<uint64_t*>(smem + kOffScratch);
  uint64_t* xchg = reinterpret_cast<uint64_t*>(smem + kOffXchg);
  const uint32_t full0 = smem_addr(smem + kOffBars);
  const uint32_t empty0 = full0 + 8u * kStages;
  const uint32_t test_bar = smem_addr(&S.test_bar_word);
  const Ws& w = P.ws;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, kConsumerWarps);
    }
    mbar_init(test_bar, 1);  // never arrived on (the timeout test)
    fence_mbar_init();
    S.cabort = 0;
    S.pabort = 0;
    S.count = 0;
    S.ovf = 0;
    S.bnd[0] = S.bnd[1] = 0u;
    S.ins[0] = S.ins[1] = 0u;
    S.bad = 0;
    S.nbad = 0u;
    S.thmin[0] = S.thmin[1] = ~0ull;
    S.tmpcount = 0;
  }
  __syncthreads();
  // The previous kernel: the setup kernel (its lists and header), or for the
  // kBig rows the other row pass (which waited for the setup kernel).  The
  // first row pass lets the next kernel launch once the setup kernel is
  // done; the second one at once, so that the filter kernel can read the
  // setup kernel's lists and its requests' inputs during the first row
  // pass's tail (it waits for both row passes before it reads their results).
  if (BIG) pdl_trigger();
  pdl_wait();
  if (!BIG) pdl_trigger();

  const int n_active = BIG ? w.hdr->n_big : w.hdr->n_active;
  const int64_t last_row = P.Rt + P.Rd - 1;  // kBig row j is listed at last_row - j
  auto listed = [&](int j) -> const RowJob& {
    return BIG ? w.rowlist[last_row - j] : w.rowlist[j];
  };
  int* const claim_ctr = BIG ? &w.hdr->rp_next_big : &w.hdr->rp_next;
  const int64_t row_bytes = int64_t(P.V) * E::kSize;
  const int64_t bulk = row_bytes & ~int64_t(15);
  const int ntiles = int((bulk + kTileBytes - 1) / kTileBytes);
  const int tail_start = int(bulk / E::kSize);
  const int n_tail = P.V - tail_start;
  constexpr int kTileElems = kTileBytes / E::kSize;

  // ------------------------------------------------------------- producer
  if (warp == 0) {
    if (lane != 0) return;
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    const uint64_t stream_pol = l2_evict_first_policy();
    bool stop = false;
    // Each row's first ring phase carries its entry in S.rowq (the consumers
    // read it once the phase completes); a row without bulk tiles, and the
    // end of the list, take a phase of their own with no copy.  `issued`
    // counts phases.
    int j = blockIdx.x;
    RowJob job = listed(min(j, max(n_active - 1, 0)));
    for (uint32_t q = 0; !stop; ++q) {
      const bool end = j >= n_active;
      if (end) job.row = -1;
      const int64_t row = job.row;
      const char* src =
          row < P.Rt
              ? static_cast<const char*>(P.target) + row * P.t_stride * E::kSize
              : static_cast<const char*>(P.draft) + (row - P.Rt) * P.d_stride * E::kSize;
      // a kBig row is streamed kBigPasses times; its earlier streams keep the
      // default L2 policy so that the later ones are served from L2
      const int passes = BIG ? kBigPasses : 1;
      const int nt = end ? 0 : ntiles * passes;
      const int claim_t = nt > 4 ? nt - 4 : 0;
      int jn = n_active;
      for (int t = 0; t < (nt > 0 ? nt : 1); ++t) {
        if (!wait_or_abort(empty0 + 8u * stage, phase ^ 1u, &S.cabort, &S.pabort, 64)) {
          *reinterpret_cast<volatile int*>(&S.pabort) = 1;
          record_error(w.hdr, SV_ERR_TIMEOUT, -1, row);
          stop = true;
          break;
        }
        if (t == 0) S.rowq[q % kStages] = job;
        if (t == claim_t && !end) jn = int(gridDim.x) + atomicAdd(claim_ctr, 1);
        if (nt == 0) {
          mbar_arrive(full0 + 8u * stage);
        } else {
          const int tt = passes == 1 ? t : t % ntiles;  // tile of the row
          const int64_t rem = bulk - int64_t(tt) * kTileBytes;
          const uint32_t bytes = uint32_t(rem < kTileBytes ? rem : kTileBytes);
          mbar_arrive_expect_tx(full0 + 8u * stage, bytes);
          if (t >= nt - ntiles)  // the row's last stream: read once more, never again
            bulk_load_hint(smem_addr(ring + size_t(stage) * kTileBytes),
                           src + int64_t(tt) * kTileBytes, bytes, full0 + 8u * stage, stream_pol);
          else
            bulk_load(smem_addr(ring + size_t(stage) * kTileBytes),
                      src + int64_t(tt) * kTileBytes, bytes, full0 + 8u * stage);
        }
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (end) break;
      j = jn;
      if (j < n_active) job = listed(j);
    }
    if (stop || *reinterpret_cast<volatile int*>(&S.cabort)) {
      // Let every copy this CTA issued land before the CTA may exit.
      const long long first = issued > kStages ? issued - kStages : 0;
      for (long long g = first; g < issued; ++g) {
        const uint32_t st = uint32_t(g % kStages), ph = uint32_t((g / kStages) & 1);
        mbar_wait_for(full0 + 8u * st, ph);
      }
    }
    return;
  }

  // ------------------------------------------------------------- consumers
  const int ctid = tid - 32, cwarp = warp - 1;
  uint32_t stage = 0, phase = 0;
  unsigned bnd_seen[2] = {0u, 0u};
  unsigned ins_seen[2] = {0u, 0u};
  unsigned gtile = 0;  // tiles consumed by this CTA (parity of the tally counters)
  int tsel = 0;        // which of the two CTA-minimum slots is live

  auto acquire = [&]() -> const uint4* {
    if (!wait_or_abort(full0 + 8u * stage, phase, &S.cabort, &S.pabort, 16)) {
      *reinterpret_cast<volatile int*>(&S.cabort) = 1;
      record_error(w.hdr, SV_ERR_TIMEOUT, -1, -1);
    }
    return reinterpret_cast<const uint4*>(ring + size_t(stage) * kTileBytes);
  };
  auto release = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8u * stage);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  };
  // vectors in tile t: full tiles, then the last (possibly partial) one
  const int last_nvec = int((bulk - int64_t(ntiles - 1) * kTileBytes) / 16);
  auto tile_vectors = [&](int t) -> int {
    return t + 1 < ntiles ? kTileBytes / 16 : last_nvec;
  };
  unsigned bad_seen = 0u;  // value of S.nbad after the previous row

  for (uint32_t q = 0;; ++q) {
    // The row's first phase holds its entry.  A wait that fails sets
    // S.cabort before the first barrier, and no thread can set it again
    // before the second, so all threads take the same branch.
    acquire();
    consumer_sync();
    const int ab0 = *reinterpret_cast<volatile int*>(&S.cabort);
    consumer_sync();
    if (ab0) break;
    const RowJob ent = S.rowq[q % kStages];
    if (ent.row < 0) break;  // no more rows
    if (P.test_expire && !BIG && blockIdx.x == 0 && q == 0) {
      // Test of the timeout path: a bounded wait on a barrier nothing
      // arrives on expires as a stalled copy's would.  The row's request
      // fails with SV_ERR_TIMEOUT, this CTA stops; its producer sees the
      // abort, lets the copies it issued land and exits.
      if (!mbar_wait_for(test_bar, 0u, kTestWaitNs)) {
        *reinterpret_cast<volatile int*>(&S.cabort) = 1;
        if (ctid == 0) flag_request(w, ent.b, SV_ERR_TIMEOUT, ent.row);
      }
      consumer_sync();
      break;
    }
    if (ntiles == 0) release();  // a phase without a copy
    const int64_t row = ent.row;
    const int b = ent.b;
    const int gx = ent.gx;
    const int mode = ent.mode & kModeMask;
    const float T = ent.T;
    const int Kreq = ent.K;
    const void* rowp =
        row < P.Rt ? static_cast<const char*>(P.target) + row * P.t_stride * E::kSize
                   : static_cast<const char*>(P.draft) + (row - P.Rt) * P.d_stride * E::kSize;

    if (BIG) {
      // ---------------------------------------------- top-p alone / large top-k
      const BigRing br{ring, full0, empty0, &stage, &phase, &S.cabort, &S.pabort, w.hdr};
      big_row<E>(P, br, S.big, S.hist, &S.sel, smem + kOffBuf, ent, rowp, ntiles, last_nvec,
                 tail_start, n_tail);
    } else if (mode == kStats) {
      // ---------------------------------------------- online softmax sums
      const float c2 = __fdiv_rn(1.4426950408889634f, T);  // log2(e) / T
      float m = -INFINITY, mc2 = 0.f, s = 0.f, comp = 0.f;
      bool nan_seen = false;
      // 2^((x - m) log2(e) / T).  bf16 rows fold the shift into one FMA with
      // m log2(e) / T rounded once (a few ulp of it, common to every term
      // taken at the same m: far inside the bf16 probability tolerance); f32
      // rows keep x - m exact.
      auto term = [&](float x) -> float {
        return ex2_approx(BF16 ? fmaf(x, c2, -mc2) : (x - m) * c2);
      };
      auto raise = [&](float vm) {  // a new running maximum vm > m
        if (m != -INFINITY) {
          const float f = ex2_approx((m - vm) * c2);
          s *= f;
          comp *= f;
        }
        m = vm;
        mc2 = vm * c2;
      };
      auto add = [&](float acc) {  // Kahan-compensated running sum
        const float y = acc - comp;
        const float t2 = s + y;
        comp = (t2 - s) - y;
        s = t2;
      };
      // n elements (a partial tile, the tail); the maximum propagates NaN
      auto consume = [&](const float* x, int n) {
        float vm = x[0];
        for (int e = 1; e < n; ++e) vm = fmax_nan(vm, x[e]);
        nan_seen |= vm != vm;
        if (vm > m) raise(vm);
        if (m != -INFINITY) {
          float acc = 0.f;
          for (int e = 0; e < n; ++e) acc += term(x[e]);
          add(acc);
        }
      };
      constexpr int VPT = (kTileBytes / 16 + kConsumers - 1) / kConsumers;
      for (int t = 0; t < ntiles; ++t) {
        const uint4* tile = acquire();
        const int nvec = tile_vectors(t);
        if (nvec == kTileBytes / 16) {
          // a full tile: two vectors per step, their 2 EPV terms summed as a
          // tree (independent exponentials, short dependency chains)
#pragma unroll
          for (int i = 0; i < VPT; i += 2) {
            const uint4 qa = tile[ctid + i * kConsumers], qb = tile[ctid + (i + 1) * kConsumers];
            float x[2 * EPV];
            E::decode(qa, x);
            E::decode(qb, x + EPV);
            float vm;
            if constexpr (BF16) {
              const uint32_t pm = bmax2_nan(E::pmax(qa), E::pmax(qb));
              vm = fmax_nan(bf16_lo(pm), bf16_hi(pm));
            } else {
              vm = fmax_nan(E::vmax(qa), E::vmax(qb));
            }
            nan_seen |= vm != vm;
            if (vm > m) raise(vm);
            if (m != -INFINITY) {
              if constexpr (BF16) {
                // element pairs: one f32x2 FMA for two shifts, the 16 terms
                // summed as eight pairs by a tree of f32x2 adds, then the
                // pair's halves
                const uint64_t c2p = pk2(c2, c2), nmp = pk2(-mc2, -mc2);
                uint64_t r[EPV];
#pragma unroll
                for (int k = 0; k < EPV; ++k) {
                  float a0, a1;
                  upk2(fma2(pk2(x[2 * k], x[2 * k + 1]), c2p, nmp), a0, a1);
                  r[k] = pk2(ex2_approx(a0), ex2_approx(a1));
                }
#pragma unroll
                for (int w2 = 1; w2 < EPV; w2 <<= 1)
#pragma unroll
                  for (int k = 0; k + w2 < EPV; k += 2 * w2) r[k] = add2(r[k], r[k + w2]);
                float lo2, hi2;
                upk2(r[0], lo2, hi2);
                add(lo2 + hi2);
              } else {
                float e[2 * EPV];
#pragma unroll
                for (int k = 0; k < 2 * EPV; ++k) e[k] = term(x[k]);
#pragma unroll
                for (int w2 = 1; w2 < 2 * EPV; w2 <<= 1)
#pragma unroll
                  for (int k = 0; k + w2 < 2 * EPV; k += 2 * w2) e[k] += e[k + w2];
                add(e[0]);
              }
            }
          }
        } else {
          for (int v = ctid; v < nvec; v += kConsumers) {
            float x[EPV];
            E::decode(tile[v], x);
            consume(x, EPV);
          }
        }
        release();
      }
      if (ctid < n_tail) {
        const float x = E::scalar(rowp, tail_start + ctid);
        consume(&x, 1);
      }
      if (nan_seen) s = __int_as_float(0x7fc00000);  // a NaN logit: the row is bad
      // block max, then TwoSum-reduced sum rescaled to it
      float M = m;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      if (lane == 0) S.red_f[cwarp] = M;
      consumer_sync();
      M = S.red_f[0];
#pragma unroll
      for (int i = 1; i < kConsumerWarps; ++i) M = fmaxf(M, S.red_f[i]);
      const float sc = (m == -INFINITY || M == -INFINITY) ? 0.f : ex2_approx((m - M) * c2);
      float hi = (s - comp) * sc, lo = 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        float sum, err;
        two_sum(hi, h2, sum, err);
        hi = sum;
        lo = lo + l2 + err;
      }
      if (lane == 0) {
        S.red_hi[cwarp] = hi;
        S.red_lo[cwarp] = lo;
      }
      consumer_sync();
      if (ctid == 0) {
        double tot = 0.0;
        for (int i = 0; i < kConsumerWarps; ++i)
          tot += double(S.red_hi[i]) + double(S.red_lo[i]);
        const bool bad = !(tot == tot) || isinf(tot) || isinf(M) || M != M;
        double pg = __longlong_as_double(0x7ff8000000000000LL);
        if (bad) {
          flag_request(w, b, SV_ERR_DATA_LOGIT, row);
        } else if (gx >= 0) {
          const float xg = E::scalar(rowp, gx);
          pg = exp((double(xg) - double(M)) / double(T)) / tot;
        }
        RowStat st;
        st.s = tot;
        st.pg = pg;
        st.m = M;
        st.arg = -1;
        st.kept = 0;
        st.mode = kStats;
        w.stats[row] = st;
      }
    } else if (mode == kArgmax) {
      // ---------------------------------------------- greedy argmax
      float best = -INFINITY;
      int bidx = INT_MAX;
      bool bad = false;
      auto scan = [&](const float* x, int n, int idx0) {
        for (int e = 0; e < n; ++e) {
          const float xe = x[e];
          if (xe != xe || xe == INFINITY) bad = true;
          else if (xe > best) {
            best = xe;
            bidx = idx0 + e;
          }
        }
      };
      for (int t = 0; t < ntiles; ++t) {
        const uint4* tile = acquire();
        const int nvec = tile_vectors(t);
        for (int v = ctid; v < nvec; v += kConsumers) {
          const uint4 q = tile[v];
          if (!(E::vmax(q) <= best)) {
            float x[EPV];
            E::decode(q, x);
            scan(x, EPV, t * kTileElems + v * EPV);
          }
        }
        release();
      }
      if (ctid < n_tail) {
        const float x = E::scalar(rowp, tail_start + ctid);
        scan(&x, 1, tail_start + ctid);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (b2 > best || (b2 == best && i2 < bidx)) {
          best = b2;
          bidx = i2;
        }
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&S.bad, 1);
      if (lane == 0) {
        S.red_f[cwarp] = best;
        S.red_i[cwarp] = bidx;
      }
      consumer_sync();
      if (ctid == 0) {
        for (int i = 0; i < kConsumerWarps; ++i)
          if (S.red_f[i] > best || (S.red_f[i] == best && S.red_i[i] < bidx)) {
            best = S.red_f[i];
            bidx = S.red_i[i];
          }
        if (S.bad) flag_request(w, b, SV_ERR_DATA_LOGIT, row);
        S.bad = 0;
        RowStat st;
        st.s = 0.0;
        st.pg = __longlong_as_double(0x7ff8000000000000LL);
        st.m = best;
        st.arg = best == -INFINITY ? 0 : bidx;
        st.kept = 0;
        st.mode = kArgmax;
        w.stats[row] = st;
      }
    } else {
      // ---------------------------------------------- top-k / top-p
      // Fast path (one pass, no per-tile barrier): a speculative threshold is
      // taken from tile 0 -- a rank there that the row's top K exceed only
      // with negligible probability (tile 0 holds about lambda = K * |tile| / V
      // of them; rank lambda + 4 sqrt(lambda) + 4) -- and every element at or
      // above it is appended to a shared buffer.  At the end of the row the
      // speculation is verified: if nothing overflowed and at least K
      // elements passed, the row's top K are all in the buffer.  Otherwise
      // the row is streamed again from global memory by the certified path:
      // per tile, phase A flags the vectors whose maximum reaches the
      // threshold and tallies an upper bound of the candidates, one barrier
      // checks the buffer capacity (compacting to the exact K largest when
      // needed), and phase B inserts.
      //
      // Thresholds: each warp takes the m-th largest of the keys it holds and
      // the CTA takes the minimum, so at least 8m keys reach it.
      const int K = Kreq;
      constexpr uint32_t kSkip = BF16 ? kSkipBf16 : kSkipF32;
      constexpr int VPT = (kTileBytes / 16 + kConsumers - 1) / kConsumers;
      constexpr int GROUP = 32 / EPV;
      constexpr int UNR = 2;
      const int m = (K + kConsumerWarps - 1) / kConsumerWarps;
      uint64_t theta = 0ull;  // uniform
      int count = 0;          // exact buffer fill at the last tile boundary (uniform)
      bool bad = false;
      bool redo = false;      // the speculative pass must be redone by the certified path

      auto tally = [&](unsigned* ctr, unsigned& seen, unsigned wv) -> int {
        if (lane == 0 && wv) atomicAdd(ctr, wv);
        consumer_sync();
        const unsigned now = *reinterpret_cast<volatile unsigned*>(ctr);
        const int tot = int(now - seen);
        seen = now;
        return tot;
      };
      // CTA minimum of the per-warp values (one barrier).
      auto cta_min = [&](uint64_t wv) -> uint64_t {
        if (lane == 0) atomicMin(&S.thmin[tsel], static_cast<unsigned long long>(wv));
        consumer_sync();
        const uint64_t r = *reinterpret_cast<volatile unsigned long long*>(&S.thmin[tsel]);
        if (ctid == 0) S.thmin[tsel ^ 1] = ~0ull;
        tsel ^= 1;
        return r;
      };
      auto phase_a = [&](const uint4* tile, int nvec, float thv, uint32_t& cbits) -> unsigned {
        cbits = 0u;
        unsigned nb = 0;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = ctid + i * kConsumers;
          const bool c = v < nvec && !(E::vmax(tile[v]) < thv);
          nb += __popc(__ballot_sync(0xffffffffu, c));
          if (c) cbits |= 1u << i;
        }
        return nb * EPV;
      };
      auto element = [&](const char* tb, int v, int e) -> float {
        if (BF16)
          return __uint_as_float(
              uint32_t(*reinterpret_cast<const uint16_t*>(tb + size_t(v) * 16 + e * 2)) << 16);
        return *reinterpret_cast<const float*>(tb + size_t(v) * 16 + e * 4);
      };
      auto phase_b = [&](const uint4* tile, int t, uint32_t cbits, uint64_t th) -> unsigned {
        const int g = lane / EPV, e = lane % EPV;
        const char* tb = reinterpret_cast<const char*>(tile);
        uint64_t key[VPT][UNR];
        uint32_t pm[VPT][UNR];
        uint32_t rest[VPT];
        int tot = 0;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          uint32_t mm = __ballot_sync(0xffffffffu, (cbits >> i) & 1u);
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            key[i][u] = 0ull;
            pm[i][u] = 0u;
            if (mm) {
              uint32_t mg = mm;
              for (int j = 0; j < g; ++j) mg &= mg - 1u;  // the g-th flagged vector
              bool pass = false;
              if (mg) {
                const int v = cwarp * 32 + (__ffs(mg) - 1) + i * kConsumers;
                const float x = element(tb, v, e);
                if (x != x || x == INFINITY) {
                  bad = true;
                } else {
                  key[i][u] = composite_key(x, uint32_t(t * kTileElems + v * EPV + e));
                  pass = key[i][u] >= th;
                }
              }
              pm[i][u] = __ballot_sync(0xffffffffu, pass);
              tot += __popc(pm[i][u]);
#pragma unroll
              for (int j = 0; j < GROUP; ++j) mm &= mm - 1u;
            }
          }
          rest[i] = mm;
        }
        int base = 0;
        if (lane == 0 && tot) base = atomicAdd(&S.count, tot);
        base = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            if ((pm[i][u] >> lane) & 1u) {
              const int slot = base + __popc(pm[i][u] & lt);
              if (slot < kBufCap) buf[slot] = key[i][u];
            }
            base += __popc(pm[i][u]);
          }
        unsigned ins = unsigned(tot);
        // rare: a vector slot with more than UNR groups of flagged vectors
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          uint32_t mm = rest[i];
          while (mm) {
            uint32_t mg = mm;
            for (int j = 0; j < g; ++j) mg &= mg - 1u;
            uint64_t k1 = 0ull;
            bool pass = false;
            if (mg) {
              const int v = cwarp * 32 + (__ffs(mg) - 1) + i * kConsumers;
              const float x = element(tb, v, e);
              if (x != x || x == INFINITY) {
                bad = true;
              } else {
                k1 = composite_key(x, uint32_t(t * kTileElems + v * EPV + e));
                pass = k1 >= th;
              }
            }
            const uint32_t pb = __ballot_sync(0xffffffffu, pass);
            const int np = __popc(pb);
            int b1 = 0;
            if (lane == 0 && np) b1 = atomicAdd(&S.count, np);
            b1 = __shfl_sync(0xffffffffu, b1, 0);
            if (pass) {
              const int slot = b1 + __popc(pb & lt);
              if (slot < kBufCap) buf[slot] = k1;
            }
            ins += unsigned(np);
#pragma unroll
            for (int j = 0; j < GROUP; ++j) mm &= mm - 1u;
          }
        }
        return ins;
      };
      // Fast path: flag the tile's vectors with a packed max and copy the
      // flagged ones (with their vector index in the row) to this warp's
      // staging area; when it fills, and at the end of the row, one lane per
      // staged vector tests its elements and the passing ones are appended to
      // this warp's own buffer region.  Flagged vectors are few (about r per
      // tile for the whole CTA), so the per-tile work stays a load, a packed
      // compare and a vote.  No atomics and no barrier; a region overflow
      // marks the row for the certified redo.
      uint64_t* region = buf + cwarp * kRegion;
      uint4* stg_v = reinterpret_cast<uint4*>(smem + kOffStage) + cwarp * kStage;
      int* stg_i = reinterpret_cast<int*>(smem + kOffStageIdx) + cwarp * kStage;
      int wcnt = 0;  // fill of this warp's region (warp-uniform)
      int sn = 0;    // staged vectors of this warp (warp-uniform)
      auto drain = [&](uint64_t th) {
        const float thv = composite_value(th);
        const uint32_t lt = (1u << lane) - 1u;
        __syncwarp();
        for (int b0 = 0; b0 < sn; b0 += 32) {
          uint32_t mbits = 0u;
          uint4 q = make_uint4(0u, 0u, 0u, 0u);
          int vi = 0;
          if (b0 + lane < sn) {
            q = stg_v[b0 + lane];
            vi = stg_i[b0 + lane];
#pragma unroll
            for (int e = 0; e < EPV; ++e)  // also NaN and +inf (checked below)
              if (!(E::elem(q, e) < thv)) mbits |= 1u << e;
          }
          while (__any_sync(0xffffffffu, mbits != 0u)) {
            uint64_t key = 0ull;
            bool pass = false;
            if (mbits) {
              const int e = __ffs(mbits) - 1;
              mbits &= mbits - 1u;
              const float xe = E::elem(q, e);
              if (xe != xe || xe == INFINITY) {
                bad = true;
              } else {
                key = composite_key(xe, uint32_t(vi * EPV + e));
                pass = key >= th;
              }
            }
            const uint32_t pm = __ballot_sync(0xffffffffu, pass);
            if (pass) {
              const int sidx = wcnt + __popc(pm & lt);
              if (sidx < kRegion) region[sidx] = key;
            }
            wcnt += __popc(pm);
          }
        }
        sn = 0;
        __syncwarp();  // the staging area is rewritten next
      };
      // Stage the flagged vectors of one ballot (at most 32 of them).
      auto stage = [&](bool c, const uint4& q, int vrow, uint32_t bal, uint64_t th) {
        const int nf = __popc(bal);
        if (sn + nf > kStage) drain(th);
        if (c) {
          const int slot = sn + __popc(bal & ((1u << lane) - 1u));
          stg_v[slot] = q;
          stg_i[slot] = vrow;
        }
        sn += nf;
      };
      auto fused_pass = [&](const uint4* tile, int nvec, int t, uint64_t th, float thv,
                            [[maybe_unused]] uint32_t below2) {
        const int vt = t * (kTileBytes / 16);  // first vector of the tile in the row
        if (nvec == kTileBytes / 16) {
          // full tile: two vectors per compare, no bounds checks
#pragma unroll
          for (int i = 0; i < VPT; i += 2) {
            const int va = ctid + i * kConsumers, vb = va + kConsumers;
            const uint4 qa = tile[va], qb = tile[vb];
            bool any, ca, cb;
            if constexpr (BF16) {
              // packed: a vector is flagged when one of its elements is >= thv
              const uint32_t ma = E::pmax(qa), mb = E::pmax(qb);
              any = bmax2_nan(bmax2_nan(ma, mb), below2) != below2;
              ca = any && bmax2_nan(ma, below2) != below2;
              cb = any && bmax2_nan(mb, below2) != below2;
            } else {
              any = !(fmax_nan(E::vmax(qa), E::vmax(qb)) < thv);
              ca = any && !(E::vmax(qa) < thv);
              cb = any && !(E::vmax(qb) < thv);
            }
            if (__any_sync(0xffffffffu, any)) {
              stage(ca, qa, vt + va, __ballot_sync(0xffffffffu, ca), th);
              stage(cb, qb, vt + vb, __ballot_sync(0xffffffffu, cb), th);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < VPT; ++i) {
            const int v0 = ctid + i * kConsumers;
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (v0 < nvec) q = tile[v0];
            const bool c = v0 < nvec && !(E::vmax(q) < thv);
            stage(c, q, vt + v0, __ballot_sync(0xffffffffu, c), th);
          }
        }
      };
      // Per-vector maximum in the composite order (value, first index).
      auto vector_max_key = [&](const uint4* tile, int v, int t) -> uint64_t {
        const uint4 q = tile[v];
        const float vm = E::vmax(q);
        float x[EPV];
        E::decode(q, x);
        int first = 0;
        for (int e = EPV - 1; e >= 0; --e)
          if (x[e] == vm) first = e;
        return composite_key(vm, uint32_t(t * kTileElems + v * EPV + first));
      };
      // Tight speculative threshold from tile 0: each warp extracts the top L
      // of its vector maxima and the r-th largest of the 8L candidates is
      // taken.  A speculative threshold needs no exact tie order (the row-end
      // check decides), so it is keyed as the smallest key of its value.  With
      // 8L <= 32 candidates every warp sorts them itself after one barrier;
      // larger L take the CTA sort.
      auto bootstrap_spec = [&](const uint4* tile, int nvec, int t, int r, int L) {
        const int nu = kConsumerWarps * L;
        if (nu <= 32) {
          float* cand = reinterpret_cast<float*>(scratch);
          float mx[VPT];
#pragma unroll
          for (int i = 0; i < VPT; ++i) {
            const int v = ctid + i * kConsumers;
            const float m = v < nvec ? E::vmax(tile[v]) : -INFINITY;
            mx[i] = m == m ? m : -INFINITY;  // a NaN row is flagged by the sweep
          }
          for (int q = 0; q < L; ++q) {
            float lm = mx[0];
            int li = 0;
#pragma unroll
            for (int j = 1; j < VPT; ++j)
              if (mx[j] > lm) {
                lm = mx[j];
                li = j;
              }
            float wm = lm;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
            if (lane == 0) cand[cwarp * L + q] = wm;
            // lanes holding the maximum drop it (ties may drop several: the
            // threshold only gets looser)
            if (lm == wm) {
#pragma unroll
              for (int j = 0; j < VPT; ++j)
                if (j == li) mx[j] = -INFINITY;
            }
          }
          consumer_sync();
          const float u = warp_sort_desc_f32(lane < nu ? cand[lane] : -INFINITY);
          const float thr = __shfl_sync(0xffffffffu, u, r - 1);
          const uint64_t tb = composite_key(thr, 0xffffffffu);
          if (tb > theta) theta = tb;
          return;
        }
        uint64_t mx[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = ctid + i * kConsumers;
          mx[i] = v < nvec ? composite_key(E::vmax(tile[v]), uint32_t(t * kTileElems + v * EPV))
                           : 0ull;
        }
        for (int q = 0; q < L; ++q) {
          uint64_t lm = mx[0];
          int li = 0;
#pragma unroll
          for (int j = 1; j < VPT; ++j)
            if (mx[j] > lm) {
              lm = mx[j];
              li = j;
            }
          uint64_t wm = lm;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const uint64_t y = shfl_xor_u64(wm, o);
            wm = y > wm ? y : wm;
          }
          if (lane == 0) scratch[cwarp * L + q] = wm;
          if (wm != 0ull && lm == wm) {
#pragma unroll
            for (int j = 0; j < VPT; ++j)
              if (j == li) mx[j] = 0ull;
          }
        }
        consumer_sync();
        uint64_t u = ctid < nu ? scratch[ctid] : 0ull;
        u = block_sort_desc<kConsumers>(u, ctid, next_pow2(nu), xchg, ConsumerSync());
        if (ctid == r - 1) S.thmin[2] = u;
        consumer_sync();
        const uint64_t tb = S.thmin[2];
        if (tb > theta) theta = tb;
        consumer_sync();  // scratch and S.thmin[2] may be reused
      };
      // Threshold from one tile's vector maxima: at least 8 * mw elements of
      // the tile reach it.
      auto bootstrap = [&](const uint4* tile, int nvec, int t, int mw) {
        uint64_t mx[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = ctid + i * kConsumers;
          mx[i] = v < nvec ? vector_max_key(tile, v, t) : 0ull;
        }
        const uint64_t r = warp_mth_largest<VPT>(mx, mw);
        const uint64_t tb = cta_min(r);
        if (tb > theta) theta = tb;
      };
      // Exact variant: the K-th largest vector maximum (bounds the tile's
      // candidates by K * EPV).
      auto bootstrap_exact = [&](const uint4* tile, int nvec, int t) {
        for (int v = ctid; v < nvec; v += kConsumers) scratch[v] = vector_max_key(tile, v, t);
        consumer_sync();
        const uint64_t tb = block_select_kth<kConsumers>(scratch, nvec, K, ctid, S.hist, &S.sel,
                                                         ConsumerSync(), kSkip);
        if (tb > theta) theta = tb;
      };
      // Keep exactly the K largest of the n buffered candidates.
      auto compact = [&](int n) {
        const uint64_t th = block_select_kth<kConsumers>(buf, n, K, ctid, S.hist, &S.sel,
                                                         ConsumerSync(), kSkip);
        if (ctid == 0) S.tmpcount = 0;
        consumer_sync();
        for (int base = cwarp * 32; base < n; base += kConsumers) {
          const int e = base + lane;
          const uint64_t key = e < n ? buf[e] : 0ull;
          const bool keep = e < n && key >= th;
          const uint32_t bal = __ballot_sync(0xffffffffu, keep);
          int slot0 = 0;
          if (lane == 0 && bal) slot0 = atomicAdd(&S.tmpcount, __popc(bal));
          slot0 = __shfl_sync(0xffffffffu, slot0, 0);
          if (keep) {
            const int slot = slot0 + __popc(bal & ((1u << lane) - 1u));
            if (slot < kScratch) scratch[slot] = key;
          }
        }
        consumer_sync();
        for (int e = ctid; e < K; e += kConsumers) buf[e] = scratch[e];
        if (ctid == 0) S.count = K;
        if (th > theta) theta = th;
        consumer_sync();
      };

      // Certified handling of one tile (any address space).
      auto certified_tile = [&](const uint4* tile, int nvec, int t) {
        const int par = int(gtile & 1u);
        const int prev = par ^ 1;
        if (t == 0 && nvec >= K) bootstrap(tile, nvec, t, m);
        uint32_t cbits;
        unsigned wb = phase_a(tile, nvec, composite_value(theta), cbits);
        int bound = tally(&S.bnd[par], bnd_seen[par], wb);
        if (t > 0) {
          // insertions of the previous tile are complete once every warp passed the barrier
          const unsigned now = *reinterpret_cast<volatile unsigned*>(&S.ins[prev]);
          count += int(now - ins_seen[prev]);
          ins_seen[prev] = now;
        }
        if (count + bound > kBufCap - 8) {  // make room first
          consumer_sync();
          if (count > K) {
            compact(count);
            count = K;
          }
          wb = phase_a(tile, nvec, composite_value(theta), cbits);
          bound = tally(&S.bnd[par], bnd_seen[par], wb);
          if (count + bound > kBufCap - 8 && nvec >= K) {
            bootstrap_exact(tile, nvec, t);
            wb = phase_a(tile, nvec, composite_value(theta), cbits);
            bound = tally(&S.bnd[par], bnd_seen[par], wb);
          }
        }
        const unsigned ins = phase_b(tile, t, cbits, theta);
        if (lane == 0 && ins) atomicAdd(&S.ins[par], ins);
        ++gtile;
      };
      // Tail elements (fewer than 16 bytes), read directly from global memory.
      auto tail_insert = [&]() {
        if (ctid < n_tail) {
          const float x = E::scalar(rowp, tail_start + ctid);
          if (x != x || x == INFINITY) {
            bad = true;
          } else {
            const uint64_t key = composite_key(x, uint32_t(tail_start + ctid));
            if (key >= theta) {
              const int slot = atomicAdd(&S.count, 1);
              if (slot < kBufCap) buf[slot] = key;
              else S.ovf = 1;
            }
          }
        }
      };

      // ---- fast path: speculative threshold, one sweep
      {
        const int e0 = tail_start < kTileElems ? tail_start : kTileElems;  // elements in tile 0
        // float arithmetic: r is a safety margin, and the FP64 pipe is narrow
        const float lam = float(K) * float(e0) / float(P.V);
        const int r = int(ceilf(lam + 4.0f * sqrtf(lam) + 4.0f));
        const int L = (2 * r + kConsumerWarps - 1) / kConsumerWarps;
        float thv = 0.0f;     // the threshold's value, and for bf16 the packed
        uint32_t below2 = 0u; // flag pattern (fixed once tile 0 set theta)
        for (int t = 0; t < ntiles; ++t) {
          const uint4* tile = acquire();
          const int nvec = tile_vectors(t);
          if (t == 0) {
            if (L <= 32 && nvec >= kConsumerWarps * L) bootstrap_spec(tile, nvec, 0, r, L);
            thv = composite_value(theta);
            if constexpr (BF16) below2 = bf16_below2(thv);
          }
          fused_pass(tile, nvec, t, theta, thv, below2);
          release();
        }
        drain(theta);
        // tail elements go to warp 0's region
        const bool tp_ok = ctid < n_tail;
        uint64_t tkey = 0ull;
        bool tpass = false;
        if (tp_ok) {
          const float x = E::scalar(rowp, tail_start + ctid);
          if (x != x || x == INFINITY) {
            bad = true;
          } else {
            tkey = composite_key(x, uint32_t(tail_start + ctid));
            tpass = tkey >= theta;
          }
        }
        const uint32_t pm = __ballot_sync(0xffffffffu, tpass);
        if (cwarp == 0) {
          if (tpass) {
            const int sidx = wcnt + __popc(pm & ((1u << lane) - 1u));
            if (sidx < kRegion) region[sidx] = tkey;
          }
          wcnt += __popc(pm);
        }
        if (lane == 0) S.wcnt[cwarp] = wcnt;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicAdd(&S.nbad, 1u);
      consumer_sync();
      // S.nbad only grows, so no reset (and no extra barrier) is needed
      unsigned nb = *reinterpret_cast<volatile unsigned*>(&S.nbad);
      bool rowbad = nb != bad_seen;
      {
        int tot = 0;
        bool ovf = false;
        for (int i = 0; i < kConsumerWarps; ++i) {
          tot += S.wcnt[i];
          ovf = ovf || S.wcnt[i] > kRegion;
        }
        count = tot;
        redo = !rowbad && (ovf || count < K);
      }
      if (!redo && !rowbad && count > kRawCap) redo = true;  // too many survivors: exact path
      if (redo) {
        // ---- certified path: the speculation missed; stream the row again
        consumer_sync();
        if (ctid == 0) {
          S.count = 0;
          S.ovf = 0;
          S.tmpcount = 0;
        }
        theta = 0ull;
        count = 0;
        ins_seen[0] = *reinterpret_cast<volatile unsigned*>(&S.ins[0]);
        ins_seen[1] = *reinterpret_cast<volatile unsigned*>(&S.ins[1]);
        consumer_sync();
        const char* rowc = static_cast<const char*>(rowp);
        for (int t = 0; t < ntiles; ++t)
          certified_tile(reinterpret_cast<const uint4*>(rowc + size_t(t) * kTileBytes),
                         tile_vectors(t), t);
        tail_insert();
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicAdd(&S.nbad, 1u);
        consumer_sync();
        nb = *reinterpret_cast<volatile unsigned*>(&S.nbad);
        rowbad = nb != bad_seen;
        count = *reinterpret_cast<volatile int*>(&S.count);
        ins_seen[0] = *reinterpret_cast<volatile unsigned*>(&S.ins[0]);
        ins_seen[1] = *reinterpret_cast<volatile unsigned*>(&S.ins[1]);
        if (count > kBufCap) {  // only after a data error (the path above bounds the fill)
          if (ctid == 0 && !rowbad) flag_request(w, b, SV_ERR_INTERNAL, row);
          count = kBufCap;
        }
        if (count > K) compact(count);  // exact: the K largest in buf[0..K)
        if (count > K) count = K;
        consumer_sync();
      }

      // publish the survivors: the per-warp regions (fast path) or buf[0..K)
      // (certified path), contiguously; the finalize kernel selects the exact
      // top K from them and applies the temperature softmax and top-p.
      const size_t rbase = size_t(row) * kRawCap;
      if (!rowbad) {
        if (redo) {
          for (int j = ctid; j < count; j += kConsumers) w.cand_raw[rbase + j] = buf[j];
        } else {
          int off = 0;
          for (int i = 0; i < cwarp; ++i) off += S.wcnt[i];
          for (int j = lane; j < wcnt; j += 32) w.cand_raw[rbase + off + j] = region[j];
        }
      }
      bad_seen = nb;
      if (ctid == 0) {
        if (rowbad) flag_request(w, b, SV_ERR_DATA_LOGIT, row);
        RowStat st;
        st.s = 0.0;
        st.pg = __longlong_as_double(0x7ff8000000000000LL);
        st.m = 0.0f;
        st.arg = -1;
        st.kept = rowbad ? 0 : count;
        st.mode = kTopk;
        w.stats[row] = st;
      }
    }

    // Row boundary.  S.cabort is written only inside acquire(), and every
    // consumer thread has passed a barrier after its last acquire of this row
    // (each mode ends with one) and none acquires again before the barrier
    // below, so all threads read the same value here.
    const int ab = *reinterpret_cast<volatile int*>(&S.cabort);
    consumer_sync();
    if (ab) break;
  }
}

}  // namespace

size_t rowpass_smem_bytes() { return kSmemBytes; }

cudaError_t launch_rowpass(const Problem& P, bool bf16, bool big, int grid, cudaStream_t s) {
  if (bf16)
    return big ? launch_after(rowpass_kernel<true, true>, grid, kRowpassThreads, kSmemBytes, s, P)
               : launch_after(rowpass_kernel<true, false>, grid, kRowpassThreads, kSmemBytes, s,
                              P);
  return big ? launch_after(rowpass_kernel<false, true>, grid, kRowpassThreads, kSmemBytes, s, P)
             : launch_after(rowpass_kernel<false, false>, grid, kRowpassThreads, kSmemBytes, s, P);
}

cudaError_t rowpass_configure() {
  const int smem = int(kSmemBytes);
  cudaError_t e = cudaFuncSetAttribute(rowpass_kernel<true, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(rowpass_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(rowpass_kernel<true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(rowpass_kernel<false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

}  // namespace sv
