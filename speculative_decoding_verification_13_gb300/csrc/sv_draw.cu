// Draw pass: the final token of every sampled request that is unfiltered or
// filtered by a kept-set threshold (top-p alone, large top-k), by inverse
// CDF in vocabulary-index order, y* = min{ y : C_y > u_k S }, over
//   the normalised residual max(0, p_L - q_L) after a rejection at L
//     ("FlashMap…" §4 step 3; "DFlash" §4), or
//   p_k after a full acceptance (the bonus token),
// with p and q zero outside their rows' kept sets.  (Vocabularies of at most
// kInlineDrawV elements take these draws in the deciding warps instead, and
// neither kernel here is launched.)
//
// Two kernels.  The draw pass (persistent CTAs) cuts each queued draw into
// segments of whole stages; a unit of work is one segment, and CTAs claim
// units from a counter.  As in the row pass, warp 0 is a producer that
// streams the unit's piece of the target row (and of the draft row, for a
// residual) through a 4-stage shared-memory ring with TMA bulk copies
// (cp.async.bulk, one 8 KB piece of each row per stage, completing on a
// "full" mbarrier; consumer warps release stages on an "empty" mbarrier),
// with the unit and its descriptor in a slot per stage.  The 8 consumer warps
// turn each 256-element tile into its weight sum (float; packed f32x2
// arithmetic for rows without a kept-set mask) and store the segment's tile
// sums and its total (an exact integer in units of 2^-40) to global memory.
// The locate kernel then takes each draw from those sums alone: the segment,
// the tile and the element where the prefix first exceeds t = u_k S, with
// only the crossing tile's elements read again.  Nothing in the draw pass
// waits for another CTA.
// Every wait is bounded; on expiry the kernel records SV_ERR_TIMEOUT, stops,
// and lets the copies it issued land before exiting.
#include <math.h>

#include "sv_weights.cuh"

namespace sv {
namespace {

constexpr int kDStages = 4;
constexpr int kDHalf = 8192;                  // bytes of one row per stage
constexpr int kDStageBytes = 2 * kDHalf;      // target piece, then draft piece
constexpr int kDConsumerWarps = 8;
constexpr int kDConsumers = kDConsumerWarps * 32;
constexpr int kDThreads = kDConsumers + 32;
// tile sums a row's survivor slot holds past its first 64 bytes
constexpr int kTileStore = (kRawCap * 8 - 64) / 4;
constexpr uint32_t kFull = 0xffffffffu;

struct DrawPassShared {
  int cabort;  // a consumer wait gave up
  int pabort;  // the producer's wait gave up
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const int* f1,
                                         const int* f2, uint32_t sleep_ns) {
  return mbar_wait_for(bar, parity, kWaitNs, f1, f2, sleep_ns);
}

__device__ __forceinline__ void draw_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kDConsumers) : "memory");
}

__device__ __forceinline__ float sum8(const float* r) {
  return ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
}

// Warp sums (every lane gets the total) and an inclusive warp scan.
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// bf16 elements 2j, 2j+1 of 16 bytes (one 32-bit word) as a packed pair.
__device__ __forceinline__ uint64_t bf16_pair(const uint4& q, int j) {
  const uint32_t w = j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
  return pk2(bf16_lo(w), bf16_hi(w));
}

// Weight sum of a lane's 8 consecutive elements of an unmasked row pair, the
// loop-invariant parts (m, c2, log2 normaliser) packed once per draw:
//   KIND 0: 2^((x_t - m_t) c2 - b_t)
//   KIND 1: max(0, 2^((x_t - m_t) c2 - b_t) - 2^((x_d - m_d) c2 - b_d))
// The same per-element weights as Weights::operator(); the 8 are summed as
// pairs, then the pair's halves.
struct PackedW {
  uint64_t mt, md, c2, nbt, nbd;
};

template <int KIND>
__device__ __forceinline__ float lane8_sum_bf16(const PackedW& pw, const unsigned char* tp,
                                                const unsigned char* dp) {
  const uint4 qt = *reinterpret_cast<const uint4*>(tp);
  uint4 qd = make_uint4(0u, 0u, 0u, 0u);
  if (KIND == 1) qd = *reinterpret_cast<const uint4*>(dp);
  uint64_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float a0, a1;
    upk2(fma2(sub2(bf16_pair(qt, j), pw.mt), pw.c2, pw.nbt), a0, a1);
    float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
    if (KIND == 1) {
      float b0, b1;
      upk2(fma2(sub2(bf16_pair(qd, j), pw.md), pw.c2, pw.nbd), b0, b1);
      float d0, d1;
      upk2(sub2(pk2(e0, e1), pk2(ex2_approx(b0), ex2_approx(b1))), d0, d1);
      e0 = fmaxf(0.f, d0);
      e1 = fmaxf(0.f, d1);
    }
    r[j] = pk2(e0, e1);
  }
  float lo, hi;
  upk2(add2(add2(r[0], r[1]), add2(r[2], r[3])), lo, hi);
  return lo + hi;
}

template <int KIND>
__device__ __forceinline__ float lane8_sum_f32(const PackedW& pw, const unsigned char* tp,
                                               const unsigned char* dp) {
  const uint4* t4 = reinterpret_cast<const uint4*>(tp);
  const uint4* d4 = reinterpret_cast<const uint4*>(dp);
  uint64_t r[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 qt = t4[h];
    uint4 qd = make_uint4(0u, 0u, 0u, 0u);
    if (KIND == 1) qd = d4[h];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint64_t xt = j == 0 ? (uint64_t(qt.y) << 32 | qt.x) : (uint64_t(qt.w) << 32 | qt.z);
      float a0, a1;
      upk2(fma2(sub2(xt, pw.mt), pw.c2, pw.nbt), a0, a1);
      float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
      if (KIND == 1) {
        const uint64_t xd =
            j == 0 ? (uint64_t(qd.y) << 32 | qd.x) : (uint64_t(qd.w) << 32 | qd.z);
        float b0, b1;
        upk2(fma2(sub2(xd, pw.md), pw.c2, pw.nbd), b0, b1);
        float d0, d1;
        upk2(sub2(pk2(e0, e1), pk2(ex2_approx(b0), ex2_approx(b1))), d0, d1);
        e0 = fmaxf(0.f, d0);
        e1 = fmaxf(0.f, d1);
      }
      r[2 * h + j] = pk2(e0, e1);
    }
  }
  float lo, hi;
  upk2(add2(add2(r[0], r[1]), add2(r[2], r[3])), lo, hi);
  return lo + hi;
}

template <bool BF16, int KIND>
__device__ __forceinline__ float lane8_sum(const PackedW& pw, const unsigned char* tp,
                                           const unsigned char* dp) {
  return BF16 ? lane8_sum_bf16<KIND>(pw, tp, dp) : lane8_sum_f32<KIND>(pw, tp, dp);
}

// A tile's weight sum from global memory (one warp; every lane gets it).
template <bool BF16>
__device__ __forceinline__ float tile_from_global(const Weights& Wt, const void* trow,
                                                  const void* drow, int tau, int V) {
  float r[8];
  lane_tile_global<BF16>(Wt, trow, drow, tau, V, r);
  return warp_sum_f(sum8(r));
}

// How a row of V elements is cut into stages, tiles and segments (the draw
// pass and the locate kernel must agree): nst bulk-copied stages of
// kDHalf bytes (fast_end elements), ntile tiles of kDTile, nseg segments of
// sps whole stages each, none empty (the last one also owns the tiles past
// the bulk-copied part).
struct DrawSegs {
  int nst, ntile, fast_end, sps, nseg, tps;
  int64_t bulk;
  __device__ void stages(int s, int* a, int* z) const {
    *a = min(nst, s * sps);
    *z = min(nst, (s + 1) * sps);
  }
  __device__ void tiles(int s, int* a, int* z) const {
    *a = min(ntile, s * sps * tps);
    *z = s == nseg - 1 ? ntile : min(ntile, (s + 1) * sps * tps);
  }
};

template <int kSize>
__device__ __forceinline__ DrawSegs draw_segs(int V, int n_seg) {
  DrawSegs g;
  g.ntile = (V + kDTile - 1) / kDTile;
  g.bulk = (int64_t(V) * kSize) & ~int64_t(15);
  g.nst = int((g.bulk + kDHalf - 1) / kDHalf);
  g.fast_end = int(g.bulk / kSize);
  const int nseg0 = max(1, min(n_seg, g.nst));
  g.sps = g.nst > 0 ? (g.nst + nseg0 - 1) / nseg0 : 0;
  g.nseg = g.sps > 0 ? (g.nst + g.sps - 1) / g.sps : 1;
  g.tps = kDHalf / kSize / kDTile;
  return g;
}

// Stage slot: what the producer armed a ring phase with.
struct StageSlot {
  int32_t unit;  // queued draw x segments index, or -1: no more work
  int32_t s;     // the stage of the row the phase carries, or -1: a phase with no copy
};

template <bool BF16>
__global__ void __launch_bounds__(kDThreads, 3) draw_pass_kernel(const Problem P) {
  using E = Elt<BF16>;
  constexpr int kEPS = kDHalf / E::kSize;  // elements of a row per stage
  constexpr int kTPS = kEPS / kDTile;      // tiles per stage
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ DrawPassShared S;
  __shared__ StageSlot slot[kDStages];
  __shared__ DrawDesc sdesc[kDStages];
  __shared__ DrawDesc cdesc;  // the consumers' current unit
  unsigned char* ring = smem;
  const uint32_t full0 = smem_addr(smem + size_t(kDStages) * kDStageBytes);
  const uint32_t empty0 = full0 + 8u * kDStages;
  float* ts = reinterpret_cast<float*>(smem + size_t(kDStages) * kDStageBytes + 16 * kDStages);
  const Ws& w = P.ws;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, kDConsumerWarps);
    }
    fence_mbar_init();
    S.cabort = 0;
    S.pabort = 0;
  }
  __syncthreads();
  pdl_trigger();  // the locate kernel may launch; it waits for this one
  pdl_wait();     // the filter / decide kernel's queue
  const int n_draw = w.hdr->n_draw;
  const int V = P.V;
  // Each queued draw is cut into nseg segments of whole stages; a unit is one
  // segment.  CTA i starts with unit i and claims further units from a
  // counter, so that CTAs whose units were bonus draws (one row) or finished
  // early take more.
  const DrawSegs g = draw_segs<E::kSize>(V, P.n_seg);
  const int ntile = g.ntile, nst = g.nst, nseg = g.nseg, fast_end = g.fast_end;
  const int64_t bulk = g.bulk;
  const int units = n_draw * nseg;
  auto seg_stages = [&](int s, int* a, int* z) { g.stages(s, a, z); };
  auto seg_tiles = [&](int s, int* a, int* z) { g.tiles(s, a, z); };

  // ------------------------------------------------------------- producer
  // Arms one ring phase per stage of each unit it claims (a phase with no copy
  // for a unit without bulk stages), after writing the phase's slot: the unit,
  // the stage and the draw's descriptor, which the consumers read once the
  // phase completes (the arrival releases the writes).  A last phase with unit
  // -1 tells the consumers that the work is done.
  if (warp == 0) {
    if (lane != 0) return;
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    bool stop = false;
    const uint64_t pol = l2_evict_first_policy();
    int u = blockIdx.x;
    while (!stop) {
      const bool live = u < units;
      // the next unit, claimed now: the atomic's round trip overlaps this unit's copies
      const int next = live ? int(gridDim.x) + atomicAdd(&w.hdr->dp_next, 1) : units;
      DrawDesc d{};
      int sa = 0, sz = 0;
      const char* tsrc = nullptr;
      const char* dsrc = nullptr;
      if (live) {
        const int q = u / nseg, sg = u - q * nseg;
        d = w.draw[q];
        seg_stages(sg, &sa, &sz);
        tsrc = static_cast<const char*>(P.target) + d.tr * P.t_stride * E::kSize;
        if (d.kind == 1)
          dsrc = static_cast<const char*>(P.draft) + (d.dr - P.Rt) * P.d_stride * E::kSize;
      }
      int s = sa;
      do {
        if (!wait_bar(empty0 + 8u * stage, phase ^ 1u, &S.cabort, &S.pabort, 64)) {
          *reinterpret_cast<volatile int*>(&S.pabort) = 1;
          record_error(w.hdr, SV_ERR_TIMEOUT, -1, live ? d.tr : -1);
          stop = true;
          break;
        }
        const uint32_t full = full0 + 8u * stage;
        const bool copy = live && s < sz;
        slot[stage] = StageSlot{live ? u : -1, copy ? s : -1};
        if (live) sdesc[stage] = d;
        if (copy) {
          const int64_t rem = bulk - int64_t(s) * kDHalf;
          const uint32_t bytes = uint32_t(rem < kDHalf ? rem : kDHalf);
          mbar_arrive_expect_tx(full, dsrc ? 2u * bytes : bytes);
          unsigned char* dst = ring + size_t(stage) * kDStageBytes;
          bulk_load_hint(smem_addr(dst), tsrc + int64_t(s) * kDHalf, bytes, full, pol);
          if (dsrc)
            bulk_load_hint(smem_addr(dst + kDHalf), dsrc + int64_t(s) * kDHalf, bytes, full, pol);
        } else {
          mbar_arrive(full);
        }
        ++issued;
        if (++stage == kDStages) {
          stage = 0;
          phase ^= 1u;
        }
      } while (++s < sz);
      if (!live) break;
      u = next;
    }
    if (stop || *reinterpret_cast<volatile int*>(&S.cabort)) {
      // Let every copy this CTA issued land before the CTA may exit.
      const long long first = issued > kDStages ? issued - kDStages : 0;
      for (long long g = first; g < issued; ++g) {
        const uint32_t st = uint32_t(g % kDStages), ph = uint32_t((g / kDStages) & 1);
        mbar_wait_for(full0 + 8u * st, ph);
      }
    }
    return;
  }

  // ------------------------------------------------------------- consumers
  // Prefix work is done on fixed-point copies of the float tile sums (units
  // of 2^-40 of the row's largest weight, as integers): additions in any
  // order are then exact and cheap, where double additions (the narrow FP64
  // pipe) set the pace of one warp for microseconds per draw.  A weight is at
  // most 1 and a tile holds 256, so a tile sum is below 2^48 and a row's
  // below 2^62.
  const int cwarp = warp - 1;
  uint32_t stage = 0, phase = 0;
  // sum of tiles [a, z) in fixed point, one warp
  auto tiles_total = [&](int a, int z) -> unsigned long long {
    unsigned long long tot = 0ull;
    for (int t0 = a + lane; t0 < z; t0 += 32) tot += fixw(ts[t0]);
    return warp_sum_u64(tot);
  };
  unsigned long long* seg_fix = reinterpret_cast<unsigned long long*>(w.seg_sum);
  int cur = -1;  // the unit being summed
  Weights W{};
  bool fast = true;  // no kept-set mask: the packed path
  int q = 0, sg = 0, sa = 0, sz = 0, ta = 0, tz = 0;
  const void* trow = nullptr;
  const void* drow = nullptr;
  for (;;) {
    // The phases of one unit.  Every consumer warp leaves this loop for the
    // barrier below exactly once per unit: after the unit's last phase, at the
    // end marker, or after a wait that gave up (which makes every later wait
    // give up at once), so that the named barriers below always match.
    bool end = false;
    for (;;) {
      if (!wait_bar(full0 + 8u * stage, phase, &S.cabort, &S.pabort, 16)) {
        *reinterpret_cast<volatile int*>(&S.cabort) = 1;
        record_error(w.hdr, SV_ERR_TIMEOUT, -1, -1);
        break;
      }
      const StageSlot sl = slot[stage];
      if (sl.unit < 0) {
        end = true;
        break;
      }
      if (sl.unit != cur) {
        cur = sl.unit;
        const DrawDesc d = sdesc[stage];
        if (cwarp == 0 && lane == 0) cdesc = d;  // for the unit's epilogue
        q = cur / nseg;
        sg = cur - q * nseg;
        W = make_weights(d);
        fast = !W.mask_t && !W.mask_d;
        trow = static_cast<const char*>(P.target) + d.tr * P.t_stride * E::kSize;
        drow = d.kind == 1 ? static_cast<const char*>(P.draft) +
                                 (d.dr - P.Rt) * P.d_stride * E::kSize
                           : nullptr;
        seg_stages(sg, &sa, &sz);
        seg_tiles(sg, &ta, &tz);
      }
      if (sl.s >= 0) {
        // the stage's tiles, two per warp at a time (independent sums,
        // reduced side by side)
        const int s = sl.s;
        const unsigned char* tp = ring + size_t(stage) * kDStageBytes;
        PackedW pw;
        pw.mt = pk2(W.mt, W.mt);
        pw.md = pk2(W.md, W.md);
        pw.c2 = pk2(W.c2, W.c2);
        pw.nbt = pk2(-W.bt, -W.bt);
        pw.nbd = pk2(-W.bd, -W.bd);
        auto lane_sum = [&](int i) -> float {
          const int e = (s * kTPS + i) * kDTile + lane * 8;
          const int off = (i * kDTile + lane * 8) * E::kSize;
          if (fast && e + 8 <= fast_end)
            return W.kind == 1 ? lane8_sum<BF16, 1>(pw, tp + off, tp + kDHalf + off)
                               : lane8_sum<BF16, 0>(pw, tp + off, tp + off);
          float xt[8], xd[8], r[8];
          elems8<BF16>(tp + off, trow, e, fast_end, V, xt);
          if (W.kind == 1) elems8<BF16>(tp + kDHalf + off, drow, e, fast_end, V, xd);
#pragma unroll
          for (int k = 0; k < 8; ++k) r[k] = W.at(xt[k], W.kind == 1 ? xd[k] : 0.f, e + k);
          return sum8(r);
        };
        for (int i = cwarp; i < kTPS; i += 2 * kDConsumerWarps) {
          const int i2 = i + kDConsumerWarps;
          const bool two = i2 < kTPS;
          float la = lane_sum(i);
          float lb = two ? lane_sum(i2) : 0.f;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            la += __shfl_xor_sync(kFull, la, o);
            lb += __shfl_xor_sync(kFull, lb, o);
          }
          const int tau = s * kTPS + i, tau2 = s * kTPS + i2;
          if (lane == 0) {
            if (tau < ntile) ts[tau] = la;
            if (two && tau2 < ntile) ts[tau2] = lb;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * stage);
      if (++stage == kDStages) {
        stage = 0;
        phase ^= 1u;
      }
      if (sl.s < 0 || sl.s == sz - 1) break;
    }
    const bool run = !end && !*reinterpret_cast<volatile int*>(&S.cabort);
    // tiles past the bulk-copied part of the row (last segment), from global memory
    if (run)
      for (int tau = max(ta, nst * kTPS) + cwarp; tau < tz; tau += kDConsumerWarps) {
        const float tsum = tile_from_global<BF16>(W, trow, drow, tau, V);
        if (lane == 0) ts[tau] = tsum;
      }
    draw_sync();
    if (end || *reinterpret_cast<volatile int*>(&S.cabort)) break;
    // The segment's tile sums (in the target row's survivor slot, unused by
    // rows the draw pass serves, past the 8 bytes of a kept-set threshold,
    // when the row's tiles fit there) and its sum, for the locate kernel.
    if (ntile <= kTileStore) {
      float* gts = reinterpret_cast<float*>(w.cand_raw + size_t(cdesc.tr) * kRawCap) + 16;
      for (int tau = ta + (tid - 32); tau < tz; tau += kDConsumers) gts[tau] = ts[tau];
    }
    if (cwarp == 0) {
      const unsigned long long segsum = tiles_total(ta, tz);
      if (lane == 0) seg_fix[size_t(q) * kMaxSeg + sg] = segsum;
    }
    draw_sync();  // tile sums are rewritten by the next unit
  }
}

// ------------------------------------------------------------------ locate
// The draw of each queued request from its segments' sums, after the draw
// pass: one CTA per draw (persistent over the queue).  Warp 0 reads the
// segment sums (exact integers, 2^-40 units), forms S and t = floor(u_k S)
// and finds the segment whose inclusive prefix first exceeds t; the CTA loads
// that segment's tile sums (stored by the draw pass, else recomputed from the
// rows), sums them in chunks of 32 tiles side by side, and warp 0 walks the
// chunk sums, then the chunk's tiles, then the tile's elements (recomputed
// from the rows) to the first y whose inclusive prefix exceeds t.
constexpr int kLThreads = 256;
constexpr int kLWarps = kLThreads / 32;

struct LocateShared {
  unsigned long long S, R, t;
  int sstar, fallback;
};

// Shared memory of the locate kernel: the crossing segment's tile sums (at
// most every tile of the row), then one fixed-point sum per 32 of them.
size_t locate_smem_bytes(int V) {
  const size_t nt = size_t((V + kDTile - 1) / kDTile);
  return ((sizeof(float) * nt + 15) & ~size_t(15)) + sizeof(unsigned long long) * ((nt + 31) / 32);
}

template <bool BF16>
__global__ void __launch_bounds__(kLThreads) locate_kernel(const Problem P) {
  using E = Elt<BF16>;
  extern __shared__ __align__(16) unsigned char lsm[];
  __shared__ LocateShared L;
  const Ws& w = P.ws;
  const int V = P.V;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DrawSegs g = draw_segs<E::kSize>(V, P.n_seg);
  float* lts = reinterpret_cast<float*>(lsm);
  unsigned long long* chunk = reinterpret_cast<unsigned long long*>(
      lsm + ((sizeof(float) * size_t(g.ntile) + 15) & ~size_t(15)));
  pdl_wait();  // the draw pass's sums
  const int n_draw = w.hdr->n_draw;
  // a draw pass that gave up leaves its sums incomplete: nothing is drawn
  if (w.hdr->err_code == SV_ERR_TIMEOUT) return;
  const unsigned long long* seg_fix = reinterpret_cast<const unsigned long long*>(w.seg_sum);
  for (int q = blockIdx.x; q < n_draw; q += gridDim.x) {
    const DrawDesc d = w.draw[q];
    Weights W = make_weights(d);
    const void* trow = static_cast<const char*>(P.target) + d.tr * P.t_stride * E::kSize;
    const void* drow = d.kind == 1 ? static_cast<const char*>(P.draft) +
                                         (d.dr - P.Rt) * P.d_stride * E::kSize
                                   : nullptr;
    const unsigned long long ufix = (unsigned long long)(d.u * 4294967296.0);  // exact
    // t = floor(u_k S): the draw is the first y whose inclusive prefix
    // exceeds t (for an integer prefix C, C > u S iff C > floor(u S))
    auto floor_uS = [&](unsigned long long Stot) {
      return (__umul64hi(Stot, ufix) << 32) | ((Stot * ufix) >> 32);
    };
    if (warp == 0) {
      const unsigned long long v =
          lane < g.nseg ? __ldcg(&seg_fix[size_t(q) * kMaxSeg + lane]) : 0ull;
      const unsigned long long tot = warp_sum_u64(v);
      const unsigned long long t = floor_uS(tot);
      const unsigned long long incl = warp_incl_scan_u64(v);
      const uint32_t hit = __ballot_sync(kFull, lane < g.nseg && incl > t);
      const uint32_t pos = __ballot_sync(kFull, lane < g.nseg && v > 0ull);
      const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : g.nseg - 1);
      const unsigned long long R = __shfl_sync(kFull, incl - v, l);
      if (lane == 0) {
        L.S = tot;
        L.t = t;
        L.fallback = W.kind == 1 && tot == 0ull;
        L.sstar = l;
        L.R = R;
      }
    }
    __syncthreads();
    int sa, sz;
    if (L.fallback) {
      // residual mass vanished through rounding: draw from p_L, every tile
      W.set_kind(2);
      sa = 0;
      sz = g.ntile;
      for (int tau = warp; tau < sz; tau += kLWarps) {
        const float ts = tile_from_global<BF16>(W, trow, drow, tau, V);
        if (lane == 0) lts[tau] = ts;
      }
      __syncthreads();
      if (warp == 0) {
        unsigned long long tot = 0ull;
        for (int tau = lane; tau < sz; tau += 32) tot += fixw(lts[tau]);
        tot = warp_sum_u64(tot);
        if (lane == 0) {
          L.S = tot;
          L.t = floor_uS(tot);
          L.R = 0ull;
        }
      }
    } else {
      g.tiles(L.sstar, &sa, &sz);
      if (g.ntile <= kTileStore) {
        // the segment's tile sums, as the draw pass stored them
        const float* gts = reinterpret_cast<const float*>(w.cand_raw + size_t(d.tr) * kRawCap) + 16;
        for (int tau = sa + tid; tau < sz; tau += kLThreads) lts[tau] = __ldcg(gts + tau);
      } else {
        // the segment's tile sums, recomputed from the rows
        for (int tau = sa + warp; tau < sz; tau += kLWarps) {
          const float ts = tile_from_global<BF16>(W, trow, drow, tau, V);
          if (lane == 0) lts[tau] = ts;
        }
      }
    }
    __syncthreads();
    // fixed-point sums of 32 tiles each, side by side
    const int nch = (sz - sa + 31) / 32;
    for (int c = warp; c < nch; c += kLWarps) {
      const int tau = sa + c * 32 + lane;
      const unsigned long long cs = warp_sum_u64(tau < sz ? fixw(lts[tau]) : 0ull);
      if (lane == 0) chunk[c] = cs;
    }
    __syncthreads();
    if (warp == 0) {
      const unsigned long long t = L.t;
      // the chunk where the prefix first exceeds t, else the last with mass
      unsigned long long carry = L.R, R = L.R, Rlast = L.R;
      int cstar = -1, clast = -1;
      for (int c0 = 0; c0 < nch && cstar < 0; c0 += 32) {
        const unsigned long long v = c0 + lane < nch ? chunk[c0 + lane] : 0ull;
        const unsigned long long incl = warp_incl_scan_u64(v) + carry;
        const uint32_t pos = __ballot_sync(kFull, v > 0ull);
        const uint32_t hit = __ballot_sync(kFull, c0 + lane < nch && incl > t);
        if (pos) {
          const int l = 31 - __clz(pos);
          clast = c0 + l;
          Rlast = __shfl_sync(kFull, incl - v, l);
        }
        if (hit) {
          const int l = __ffs(hit) - 1;
          cstar = c0 + l;
          R = __shfl_sync(kFull, incl - v, l);
        }
        carry = __shfl_sync(kFull, incl, 31);
      }
      const bool beyond = cstar < 0;  // t beyond every prefix (rounding)
      if (beyond) {
        cstar = clast;
        R = Rlast;
      }
      int y = -1;
      if (cstar >= 0) {
        // the tile in the chunk (the last with mass when beyond)
        const int tau0 = sa + cstar * 32;
        const unsigned long long v = tau0 + lane < sz ? fixw(lts[tau0 + lane]) : 0ull;
        const unsigned long long incl = warp_incl_scan_u64(v) + R;
        const uint32_t pos = __ballot_sync(kFull, v > 0ull);
        const uint32_t hit = __ballot_sync(kFull, tau0 + lane < sz && incl > t);
        const int l = (!beyond && hit) ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
        const int tstar = l >= 0 ? tau0 + l : -1;
        const unsigned long long Rt = __shfl_sync(kFull, incl - v, max(l, 0));
        // the tile's elements in fixed point; the first one whose inclusive
        // prefix exceeds t, else (the tile's float sum rounded above its
        // elements' fixed-point sum) the last one with mass
        const int base = max(tstar, 0) * kDTile + lane * 8;
        float r[8];
        lane_tile_global<BF16>(W, trow, drow, max(tstar, 0), V, r);
        unsigned long long wf[8], ls = 0ull;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          wf[k] = fixw(r[k]);
          ls += wf[k];
        }
        const unsigned long long ex = warp_incl_scan_u64(ls) - ls;
        int ye = INT_MAX, lastp = -1;
        unsigned long long pre = Rt + ex;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          pre += wf[k];
          if (r[k] > 0.f) lastp = base + k;
          if (ye == INT_MAX && wf[k] > 0ull && pre > t) ye = base + k;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ye = min(ye, __shfl_xor_sync(kFull, ye, o));
          lastp = max(lastp, __shfl_xor_sync(kFull, lastp, o));
        }
        y = tstar < 0 ? -1 : ye != INT_MAX ? ye : lastp;
      }
      if (lane == 0) {
        if (y < 0) record_error(w.hdr, SV_ERR_INTERNAL, -1, d.tr);  // no mass found
        P.out_tokens[d.t0 + d.L] = y;
        if (P.out_q)  // draft sampler: the drawn token's probability (a bonus-kind draw)
          P.out_q[d.t0 + d.L] =
              y >= 0 ? ex2_approx((Elt<BF16>::one(trow, y) - d.mt) * d.c2) * d.ist
                     : __int_as_float(0x7fc00000);
      }
    }
    __syncthreads();  // L, lts and the chunk sums are rewritten for the next draw
  }
}

}  // namespace

size_t draw_pass_smem_bytes(int V) {
  return size_t(kDStages) * kDStageBytes + 16 * kDStages +
         sizeof(float) * size_t((V + kDTile - 1) / kDTile);
}

cudaError_t launch_locate(const Problem& P, bool bf16, int grid, cudaStream_t s) {
  const size_t smem = locate_smem_bytes(P.V);
  if (bf16) return launch_after(locate_kernel<true>, grid, kLThreads, smem, s, P);
  return launch_after(locate_kernel<false>, grid, kLThreads, smem, s, P);
}

cudaError_t launch_draw(const Problem& P, bool bf16, int grid, cudaStream_t s) {
  const size_t smem = draw_pass_smem_bytes(P.V);
  if (bf16)
    return launch_after(draw_pass_kernel<true>, grid, kDThreads, smem, s, P);
  return launch_after(draw_pass_kernel<false>, grid, kDThreads, smem, s, P);
}

// Shared-memory limit (largest vocabulary) and resident CTAs per SM for a
// vocabulary of V (host queries; nothing is allocated).
cudaError_t draw_configure() {
  const int smem = int(draw_pass_smem_bytes(SV_VOCAB_MAX));
  cudaError_t e = cudaFuncSetAttribute(draw_pass_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(draw_pass_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem);
  if (e != cudaSuccess) return e;
  const int lsmem = int(locate_smem_bytes(SV_VOCAB_MAX));
  e = cudaFuncSetAttribute(locate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           lsmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(locate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              lsmem);
}

cudaError_t draw_occupancy(int V, int* occ, int* occ_locate) {
  int a = 0, b = 0, c = 0, d = 0;
  const size_t smem = draw_pass_smem_bytes(V), lsmem = locate_smem_bytes(V);
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, draw_pass_kernel<true>,
                                                                kDThreads, smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, draw_pass_kernel<false>, kDThreads,
                                                      smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, locate_kernel<true>, kLThreads, lsmem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d, locate_kernel<false>, kLThreads, lsmem);
  if (e != cudaSuccess) return e;
  *occ = max(1, min(a, b));
  *occ_locate = max(1, min(c, d));
  return cudaSuccess;
}

}  // namespace sv
