// Row pass: the one kernel that streams every logit row from HBM once.
//
// Persistent, one CTA per SM.  Warp 0 is the producer: it walks the CTA's
// share of the active-row list and issues TMA bulk copies (cp.async.bulk,
// 16 KB each) into an 8-stage shared-memory ring, each stage guarded by a
// "full" mbarrier (transaction bytes) and an "empty" mbarrier (one arrival per
// consumer warp).  Warps 1..16 consume the tiles and reduce each row in one of
// three modes (chosen per request by the setup kernel):
//   kStats  - temperature softmax statistics of a sampled, unfiltered row: the
//             row max M and S = sum_y exp((x_y - M) / T) by an online
//             (running-max, rescaled) sum; then p(x) = exp((x_x - M) / T) / S
//             of the row's draft token in double precision.
//             ("FlashMap…" §5 draft_block step 5: logits / T, softmax.)
//   kArgmax - greedy: argmax of the raw logits, lowest index on ties.
//   kTopk   - the top-k tokens in (logit desc, index asc) order, selected with
//             a running threshold: a tile's candidates are counted, and
//             inserted into a shared buffer only if they beat the threshold;
//             the threshold is seeded from the k-th largest per-vector maximum
//             of the first tile and tightened by exact radix selection when
//             the buffer fills.  The epilogue applies the temperature softmax
//             over the survivors, the top-p cut and the renormalisation in
//             double precision ("Speculative decoding and multi-token
//             prediction", "Why the output is identical": the same filter on
//             both distributions).
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
constexpr size_t kSmemBytes = kOffBars + size_t(2 * kStages) * 8;
static_assert(kRowpassCtasPerSm * (kSmemBytes + 4096 + 1024) <= 228 * 1024,
              "shared memory budget for the resident CTAs of one SM");

struct RowShared {
  int hist[256];
  SelShared sel;
  unsigned long long theta;
  unsigned int bnd[2];
  unsigned int ins[2];
  int count;
  int tmpcount;
  int cabort;
  int pabort;
  int bad;
  int kp;
  float v0;
  double wp;
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
    const uint32_t m = bmax2_nan(bmax2_nan(q.x, q.y), bmax2_nan(q.z, q.w));
    return fmax_nan(bf16_lo(m), bf16_hi(m));
  }
  __device__ static float scalar(const void* row, int64_t i) {
    return __uint_as_float(uint32_t(static_cast<const uint16_t*>(row)[i]) << 16);
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
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const int* f1,
                                              const int* f2) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u &&
        (*reinterpret_cast<const volatile int*>(f1) || *reinterpret_cast<const volatile int*>(f2)))
      return false;
  }
  return false;
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

template <bool BF16>
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
  const Ws& w = P.ws;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, kConsumerWarps);
    }
    fence_mbar_init();
    S.cabort = 0;
    S.pabort = 0;
    S.count = 0;
    S.bnd[0] = S.bnd[1] = 0u;
    S.ins[0] = S.ins[1] = 0u;
    S.bad = 0;
    S.theta = 0ull;
  }
  __syncthreads();

  const int n_active = w.hdr->n_active;
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
    bool stop = false;
    for (int j = blockIdx.x; j < n_active && !stop; j += gridDim.x) {
      const int4 info = w.rowlist[j];
      const int64_t row = info.x;
      const char* src =
          row < P.Rt
              ? static_cast<const char*>(P.target) + row * P.t_stride * E::kSize
              : static_cast<const char*>(P.draft) + (row - P.Rt) * P.d_stride * E::kSize;
      for (int t = 0; t < ntiles; ++t) {
        const int64_t rem = bulk - int64_t(t) * kTileBytes;
        const uint32_t bytes = uint32_t(rem < kTileBytes ? rem : kTileBytes);
        if (!wait_or_abort(empty0 + 8u * stage, phase ^ 1u, &S.cabort, &S.pabort)) {
          *reinterpret_cast<volatile int*>(&S.pabort) = 1;
          record_error(w.hdr, SV_ERR_TIMEOUT, -1, row);
          stop = true;
          break;
        }
        mbar_arrive_expect_tx(full0 + 8u * stage, bytes);
        bulk_load(smem_addr(ring + size_t(stage) * kTileBytes), src + int64_t(t) * kTileBytes,
                  bytes, full0 + 8u * stage);
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (stop || *reinterpret_cast<volatile int*>(&S.cabort)) {
      // Let every copy this CTA issued land before the CTA may exit.
      const long long first = issued > kStages ? issued - kStages : 0;
      for (long long g = first; g < issued; ++g) {
        const uint32_t st = uint32_t(g % kStages), ph = uint32_t((g / kStages) & 1);
        for (uint32_t it = 0; it < kWaitLimit; ++it)
          if (mbar_try_wait(full0 + 8u * st, ph)) break;
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

  auto acquire = [&]() -> const uint4* {
    if (!wait_or_abort(full0 + 8u * stage, phase, &S.cabort, &S.pabort)) {
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
  auto tile_vectors = [&](int t) -> int {
    const int64_t rem = bulk - int64_t(t) * kTileBytes;
    return int((rem < kTileBytes ? rem : kTileBytes) / 16);
  };

  for (int j = blockIdx.x; j < n_active; j += gridDim.x) {
    const int4 info = w.rowlist[j];
    const int64_t row = info.x;
    const int b = info.y;
    const int gx = info.z;
    const int mode = info.w & 3;
    const void* rowp =
        row < P.Rt ? static_cast<const char*>(P.target) + row * P.t_stride * E::kSize
                   : static_cast<const char*>(P.draft) + (row - P.Rt) * P.d_stride * E::kSize;
    const float T = P.temperature[b];

    if (mode == kStats) {
      // ---------------------------------------------- online softmax sums
      const float c2 = __fdiv_rn(1.4426950408889634f, T);  // log2(e) / T
      float m = -INFINITY, s = 0.f, comp = 0.f;
      auto consume = [&](const float* x, int n) {
        float vm = x[0];
        for (int e = 1; e < n; ++e) vm = fmaxf(vm, x[e]);
        if (vm > m) {
          if (m != -INFINITY) {
            const float f = ex2_approx((m - vm) * c2);
            s *= f;
            comp *= f;
          }
          m = vm;
        }
        if (m != -INFINITY) {
          float acc = 0.f;
          for (int e = 0; e < n; ++e) acc += ex2_approx((x[e] - m) * c2);
          const float y = acc - comp;  // Kahan-compensated running sum
          const float t2 = s + y;
          comp = (t2 - s) - y;
          s = t2;
        }
      };
      for (int t = 0; t < ntiles; ++t) {
        const uint4* tile = acquire();
        const int nvec = tile_vectors(t);
        for (int v = ctid; v < nvec; v += kConsumers) {
          float x[EPV];
          E::decode(tile[v], x);
          consume(x, EPV);
        }
        release();
      }
      if (ctid < n_tail) {
        const float x = E::scalar(rowp, tail_start + ctid);
        consume(&x, 1);
      }
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
      // Per tile: phase A flags the vectors whose maximum reaches the
      // threshold (packed max, no decoding) and tallies an upper bound of the
      // candidates; one barrier; phase B reads the flagged vectors back from
      // shared memory GROUP at a time (EPV lanes per vector, so a warp never
      // runs a per-lane slow path) and appends the elements that beat the
      // threshold.  Exact fill counts travel through monotone counters that
      // alternate with the tile parity, so no second barrier is needed.
      const int K = P.top_k[b];
      const float tp = P.top_p ? P.top_p[b] : 1.0f;
      constexpr uint32_t kSkip = BF16 ? kSkipBf16 : kSkipF32;
      constexpr int VPT = (kTileBytes / 16 + kConsumers - 1) / kConsumers;
      constexpr int GROUP = 32 / EPV;
      int count = 0;  // exact buffer fill at the last tile boundary (uniform)
      bool bad = false;

      auto tally = [&](unsigned* ctr, unsigned& seen, unsigned wv) -> int {
        if (lane == 0 && wv) atomicAdd(ctr, wv);
        consumer_sync();
        const unsigned now = *reinterpret_cast<volatile unsigned*>(ctr);
        const int tot = int(now - seen);
        seen = now;
        return tot;
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
      auto phase_b = [&](const uint4* tile, int t, uint32_t cbits, uint64_t th) -> unsigned {
        unsigned ins = 0;
        const int g = lane / EPV, e = lane % EPV;
        const char* tb = reinterpret_cast<const char*>(tile);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          uint32_t m = __ballot_sync(0xffffffffu, (cbits >> i) & 1u);
          while (m) {
            uint32_t mg = m;
            for (int j = 0; j < g; ++j) mg &= mg - 1u;  // drop g lowest set bits
            const bool has = mg != 0u;
            uint64_t key = 0ull;
            bool pass = false;
            if (has) {
              const int v = cwarp * 32 + (__ffs(mg) - 1) + i * kConsumers;
              float x;
              if (BF16)
                x = __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(
                                        tb + size_t(v) * 16 + e * 2)) << 16);
              else
                x = *reinterpret_cast<const float*>(tb + size_t(v) * 16 + e * 4);
              if (x != x || x == INFINITY) {
                bad = true;
              } else {
                key = composite_key(x, uint32_t(t * kTileElems + v * EPV + e));
                pass = key >= th;
              }
            }
            const uint32_t pm = __ballot_sync(0xffffffffu, pass);
            const int np = __popc(pm);
            int base = 0;
            if (lane == 0 && np) base = atomicAdd(&S.count, np);
            base = __shfl_sync(0xffffffffu, base, 0);
            if (pass) {
              const int slot = base + __popc(pm & ((1u << lane) - 1u));
              if (slot < kBufCap) buf[slot] = key;
            }
            ins += unsigned(np);
#pragma unroll
            for (int j = 0; j < GROUP; ++j) m &= m - 1u;
          }
        }
        return ins;
      };
      // Threshold from this tile: the K-th largest per-vector maximum (the
      // maximum taken in the same composite order), a lower bound of the
      // row's K-th largest element.
      auto bootstrap = [&](const uint4* tile, int nvec, int t) {
        for (int v = ctid; v < nvec; v += kConsumers) {
          const uint4 q = tile[v];
          const float vm = E::vmax(q);
          float x[EPV];
          E::decode(q, x);
          int first = 0;
          for (int e = EPV - 1; e >= 0; --e)
            if (x[e] == vm) first = e;
          scratch[v] = composite_key(vm, uint32_t(t * kTileElems + v * EPV + first));
        }
        consumer_sync();
        const uint64_t tb = block_select_kth<kConsumers>(scratch, nvec, K, ctid, S.hist, &S.sel,
                                                         ConsumerSync(), kSkip);
        if (ctid == 0 && tb > S.theta) S.theta = tb;
        consumer_sync();
      };
      // Keep exactly the K largest of the n buffered candidates; the K-th
      // becomes the threshold.
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
        if (ctid == 0) {
          S.count = K;
          if (th > S.theta) S.theta = th;
        }
        consumer_sync();
      };

      for (int t = 0; t < ntiles; ++t) {
        const uint4* tile = acquire();
        const int nvec = tile_vectors(t);
        const int par = int(gtile & 1u);
        const int prev = par ^ 1;
        if (t == 0 && nvec >= K) bootstrap(tile, nvec, t);
        uint64_t th = S.theta;
        uint32_t cbits;
        unsigned wb = phase_a(tile, nvec, composite_value(th), cbits);
        int bound = tally(&S.bnd[par], bnd_seen[par], wb);
        if (t > 0) {
          // insertions of the previous tile are complete once every warp passed the barrier
          const unsigned now = *reinterpret_cast<volatile unsigned*>(&S.ins[prev]);
          count += int(now - ins_seen[prev]);
          ins_seen[prev] = now;
        }
        if (count + bound > kBufCap - 8) {  // rare: make room first
          consumer_sync();
          if (count > K) {
            compact(count);
            count = K;
          }
          th = S.theta;
          wb = phase_a(tile, nvec, composite_value(th), cbits);
          bound = tally(&S.bnd[par], bnd_seen[par], wb);
          if (count + bound > kBufCap - 8 && nvec >= K) {
            bootstrap(tile, nvec, t);
            th = S.theta;
            wb = phase_a(tile, nvec, composite_value(th), cbits);
            bound = tally(&S.bnd[par], bnd_seen[par], wb);
          }
        }
        const unsigned ins = phase_b(tile, t, cbits, th);
        if (lane == 0 && ins) atomicAdd(&S.ins[par], ins);
        release();
        ++gtile;
      }
      // ragged tail (fewer than 16 bytes), read directly from global memory
      if (ctid < n_tail) {
        const float x = E::scalar(rowp, tail_start + ctid);
        if (x != x || x == INFINITY) {
          bad = true;
        } else {
          const uint64_t key = composite_key(x, uint32_t(tail_start + ctid));
          if (key >= S.theta) {
            const int slot = atomicAdd(&S.count, 1);
            if (slot < kBufCap) buf[slot] = key;
          }
        }
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&S.bad, 1);
      consumer_sync();
      count = *reinterpret_cast<volatile int*>(&S.count);
      ins_seen[0] = *reinterpret_cast<volatile unsigned*>(&S.ins[0]);
      ins_seen[1] = *reinterpret_cast<volatile unsigned*>(&S.ins[1]);
      if (count > kBufCap) {  // cannot happen (capacity bound); never read past the buffer
        if (ctid == 0) flag_request(w, b, SV_ERR_INTERNAL, row);
        count = kBufCap;
      }

      // final selection: exactly min(count, K) survivors, sorted descending
      const int nsel = count < K ? count : K;
      if (count > K) compact(count);  // leaves the K largest in buf[0..K)
      const int Psz = next_pow2(nsel > 0 ? nsel : 1);
      uint64_t v = (ctid < nsel) ? buf[ctid] : 0ull;
      v = block_sort_desc<kConsumers>(v, ctid, Psz, xchg, ConsumerSync());

      // temperature softmax over the survivors, top-p, renormalisation (double)
      const bool has = ctid < nsel;
      const float vi = composite_value(v);
      const int idx = composite_index(v);
      if (ctid == 0) {
        S.v0 = vi;
        S.pg = 0.0;
      }
      consumer_sync();
      const double v0 = double(S.v0);
      const bool rowbad = S.bad != 0 || nsel == 0 || !(v0 > -INFINITY);
      double wi = 0.0;
      if (has && !rowbad) wi = exp((double(vi) - v0) / double(T));
      // inclusive scan of wi over the first nsel threads (warps beyond hold 0)
      double incl = wi;
      const bool active_warp = cwarp * 32 < Psz;
      if (active_warp) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) S.red_d[cwarp] = incl;
      }
      consumer_sync();
      double woff = 0.0, W = 0.0;
      if (active_warp) {
        for (int i = 0; i < kConsumerWarps && i * 32 < Psz; ++i) {
          if (i < cwarp) woff += S.red_d[i];
          W += S.red_d[i];
        }
      }
      incl += woff;
      const double before = incl - wi;
      const bool keep = has && (tp >= 1.0f || before / W < double(tp));
      // the kept set is the prefix that ends at the first dropped survivor
      const uint32_t drop = __ballot_sync(0xffffffffu, has && !keep);
      if (lane == 0) S.red_i[cwarp] = drop ? cwarp * 32 + __ffs(drop) - 1 : INT_MAX;
      consumer_sync();
      int kp = nsel;
      for (int i = 0; i < kConsumerWarps; ++i) kp = S.red_i[i] < kp ? S.red_i[i] : kp;
      if (ctid == kp - 1) S.wp = incl;
      consumer_sync();
      const double Wp = S.wp;
      const size_t cbase = size_t(row) * kTopkMax;
      if (ctid < kp && !rowbad) {
        const double p = wi / Wp;
        w.cand_idx[cbase + ctid] = idx;
        w.cand_p[cbase + ctid] = p;
        if (idx == gx) S.pg = p;
      }
      consumer_sync();
      if (ctid == 0) {
        if (rowbad) flag_request(w, b, SV_ERR_DATA_LOGIT, row);
        RowStat st;
        st.s = Wp;
        st.pg = gx >= 0 ? S.pg : __longlong_as_double(0x7ff8000000000000LL);
        st.m = S.v0;
        st.arg = -1;
        st.kept = rowbad ? 0 : kp;
        st.mode = kTopk;
        w.stats[row] = st;
        S.count = 0;
        S.theta = 0ull;
        S.bad = 0;
      }
    }

    // row boundary: a consistent view of the abort flag
    consumer_sync();
    const int ab = *reinterpret_cast<volatile int*>(&S.cabort);
    consumer_sync();
    if (ab) break;
  }
}

}  // namespace

size_t rowpass_smem_bytes() { return kSmemBytes; }

cudaError_t launch_rowpass(const Problem& P, bool bf16, int grid, cudaStream_t s) {
  if (bf16)
    rowpass_kernel<true><<<grid, kRowpassThreads, kSmemBytes, s>>>(P);
  else
    rowpass_kernel<false><<<grid, kRowpassThreads, kSmemBytes, s>>>(P);
  return cudaGetLastError();
}

cudaError_t rowpass_configure() {
  cudaError_t e = cudaFuncSetAttribute(rowpass_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(rowpass_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(kSmemBytes));
}

}  // namespace sv
