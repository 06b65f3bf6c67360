// Rows filtered by top-p alone, or by a top-k above SV_TOPK_MAX (row mode
// kBig), in the row pass.
//
// The kept set of a filtered row is a prefix of the row in the composite order
// (logit descending, index ascending): the top_k largest, then, on the top-k
// renormalised distribution, every token whose preceding mass is below top_p
// (the crossing token kept).  "Speculative decoding and multi-token
// prediction", "Why the output is identical", asks that the same filter act on
// target and draft; the order, the ties and the crossing token are the
// readings the oracle states.  A prefix is fixed by its last key, so such a row
// is summarised by a threshold key kappa (y is kept iff key(y) >= kappa) and
// its kept mass W; p(y) = w(y) / W for kept y.  Nothing per token is stored, so
// nuclei of thousands of tokens cost no more than small ones.
//
// The producer streams a kBig row three times (the second and third reads come
// from L2):
//   A  the row max M (NaN-propagating: NaN / +inf are data errors) and the
//      smallest finite logit;
//   B  a histogram over kBigBins bins linear in u = (M - x) log2(e) / T from 0
//      to the row's range (a monotone map: a lower bin holds only larger keys):
//      per bin the element count and the fixed-point mass of the weights
//      w(x) = 2^((x - M) log2(e) / T) (units of 2^-40, truncated; the sums are
//      exact integers, so every later comparison is exact for these weights);
//      the bin holding the K-th largest key (top-k) and the bins that can hold
//      the top-p crossing follow from the cumulative counts and masses;
//   C  the keys of those few bins (the band) are collected in shared memory,
//      sorted, and the cut is taken exactly inside them.  A band of one logit
//      value (a tie group, common on bf16 rows, where one value can hold
//      thousands of tokens) is ordered by index alone.
// A band too large for shared memory falls back to an exact radix selection
// over the band's composite keys (the digits below those all its keys share),
// with counts and masses per 8-bit digit, reading the row from global memory
// once per digit.
//
// Weights: ex2.approx of (x - M) * log2(e) / T in float (the formula the draw
// pass uses, so kept probabilities are the same function on both sides),
// good to a few 1e-7 relative; the fixed-point truncation adds at most
// V * 2^-40 to a mass (W >= 1 in these units of the largest weight).
//
// Included by sv_rowpass.cu inside its anonymous namespace; E is the row
// pass's element accessor (bf16 or f32).
#pragma once

constexpr int kBigBins = 2048;             // histogram bins of pass B
constexpr int kBigSort = 2048;             // band keys sorted in shared memory
constexpr int kBigCap = 3584;              // band keys collected
constexpr int kBandBins = 8;               // top-p band bins resolved from the counts
constexpr float kFix40 = 1099511627776.0f; // 2^40: unit of the fixed-point masses
constexpr size_t kBigWorkBytes = size_t(kBigBins) * (4 + 8);

struct BigShared {
  float wmax[kConsumerWarps];
  float wmin[kConsumerWarps];
  unsigned wc[kConsumerWarps];
  unsigned long long wm[kConsumerWarps];
  int ck, plo, phi, sk, nband, count, nkept, pk_found;
  unsigned cnt_ck_before, cnt_ck, cnt_p_before, cnt_phi_end;
  unsigned long long mass_ck_before, mass_ck, mass_p_before, total_mass;
  unsigned long long pre_sk, pre_pk1, key_k, key, W, minkey, maxkey;
  int digit, dcnt, kept, nmixed, vknown;
  float vhi, vlo, vk;
  unsigned cnt_first, rk, rp;
  // the band's bins (top-p bins plo.., then the top-k bin when it lies apart)
  unsigned bcnt[kBandBins + 1], bcb[kBandBins + 1];
  unsigned long long bmb[kBandBins + 1], bw[kBandBins + 1];
  unsigned dabove;
  unsigned long long dmass_above, dmass;
  // the cut of a band whose bins each hold one value: the value, its kept
  // occurrences (in index order) and their count, the tile holding the last
  // kept one, the rank of that one in the tile, and its index
  float fc_v;
  unsigned fc_m, fc_expect, fc_tile, fc_mr;
  int fc_idx, fc_ok;
};

struct BigSync {
  __device__ void operator()() const { consumer_sync(); }
};

// The ring as the kBig passes see it (the kernel's own stage / phase).
struct BigRing {
  const unsigned char* ring;
  uint32_t full0, empty0;
  uint32_t* stage;
  uint32_t* phase;
  int* cabort;
  int* pabort;
  WsHeader* hdr;
};

__device__ __forceinline__ const uint4* big_acquire(const BigRing& r) {
  const uint32_t bar = r.full0 + 8u * *r.stage;
  if (!mbar_wait_for(bar, *r.phase, kWaitNs, r.cabort, r.pabort, 16)) {
    *reinterpret_cast<volatile int*>(r.cabort) = 1;
    record_error(r.hdr, SV_ERR_TIMEOUT, -1, -1);
  }
  return reinterpret_cast<const uint4*>(r.ring + size_t(*r.stage) * kTileBytes);
}

__device__ __forceinline__ void big_release(const BigRing& r) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(r.empty0 + 8u * *r.stage);
  if (++*r.stage == kStages) {
    *r.stage = 0;
    *r.phase ^= 1u;
  }
}

// One stream of the row through the ring: f(x, i0, vmask) for every 16-byte
// vector (x: its E::kPerVec elements, i0: the first one's index, vmask: the
// elements that exist), with all lanes of a warp in step (f may vote); the
// elements past the bulk-copied part come from global memory, one per lane
// of warp 0 (element 0 of x).
template <class E, class F>
__device__ __forceinline__ void big_stream(const BigRing& r, int ntiles, int last_nvec,
                                           const void* rowp, int tail_start, int n_tail, F&& f) {
  constexpr int EPV = E::kPerVec;
  constexpr int kTileElems = kTileBytes / E::kSize;
  constexpr uint32_t kAll = (1u << EPV) - 1u;
  const int ctid = threadIdx.x - 32, cwarp = ctid >> 5, lane = ctid & 31;
  for (int t = 0; t < ntiles; ++t) {
    const uint4* tile = big_acquire(r);
    const int nvec = t + 1 < ntiles ? kTileBytes / 16 : last_nvec;
    for (int v0 = cwarp * 32; v0 < nvec; v0 += kConsumers) {
      const int v = v0 + lane;
      const bool valid = v < nvec;
      float x[EPV];
      E::decode(valid ? tile[v] : make_uint4(0u, 0u, 0u, 0u), x);
      f(x, t * kTileElems + v * EPV, valid ? kAll : 0u);
    }
    big_release(r);
  }
  if (cwarp == 0 && n_tail > 0) {
    const bool valid = lane < n_tail;
    float x[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) x[e] = -INFINITY;
    x[0] = valid ? E::scalar(rowp, tail_start + lane) : -INFINITY;
    f(x, tail_start + lane, valid ? 1u : 0u);
  }
}

// The same visit over the row in global memory (the exact fallback).
template <class E, class F>
__device__ __forceinline__ void big_visit_global(const void* rowp, int V, F&& f) {
  constexpr int EPV = E::kPerVec;
  const int ctid = threadIdx.x - 32;
  const int nvec = int((int64_t(V) * E::kSize) / 16);
  const uint4* vp = static_cast<const uint4*>(rowp);
  for (int v = ctid; v < nvec; v += kConsumers) {
    float x[EPV];
    E::decode(__ldcg(vp + v), x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) f(x[e], v * EPV + e);
  }
  const int tail_start = nvec * EPV;
  if (ctid < V - tail_start) f(E::scalar(rowp, tail_start + ctid), tail_start + ctid);
}

__device__ __forceinline__ unsigned long long big_wfix(float x, float M, float c2) {
  return __float2ull_rz(ex2_approx((x - M) * c2) * kFix40);
}

// Exclusive scan over the consumer threads of (count, mass); returns the
// thread's prefix and, in *tc / *tm, the totals.
__device__ __forceinline__ void big_scan(unsigned c, unsigned long long m, BigShared& S,
                                         unsigned* pc, unsigned long long* pm, unsigned* tc,
                                         unsigned long long* tm) {
  const int ctid = threadIdx.x - 32, cwarp = ctid >> 5, lane = ctid & 31;
  unsigned ci = c;
  unsigned long long mi = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned yc = __shfl_up_sync(0xffffffffu, ci, o);
    const unsigned long long ym = __shfl_up_sync(0xffffffffu, mi, o);
    if (lane >= o) {
      ci += yc;
      mi += ym;
    }
  }
  if (lane == 31) {
    S.wc[cwarp] = ci;
    S.wm[cwarp] = mi;
  }
  consumer_sync();
  unsigned oc = 0, ac = 0;
  unsigned long long om = 0, am = 0;
#pragma unroll
  for (int i = 0; i < kConsumerWarps; ++i) {
    if (i < cwarp) {
      oc += S.wc[i];
      om += S.wm[i];
    }
    ac += S.wc[i];
    am += S.wm[i];
  }
  *pc = oc + ci - c;
  *pm = om + mi - m;
  *tc = ac;
  *tm = am;
  consumer_sync();  // S.wc / S.wm may be reused
}

// Descending bitonic sort of keys[0, P) (P a power of two) by the consumer threads.
__device__ __forceinline__ void big_sort_desc(unsigned long long* keys, int P) {
  const int ctid = threadIdx.x - 32;
  for (int size = 2; size <= P; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      for (int i = ctid; i < P; i += kConsumers) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long a = keys[i], b = keys[l];
          const bool desc = (i & size) == 0;
          if (desc ? a < b : a > b) {
            keys[i] = b;
            keys[l] = a;
          }
        }
      }
      consumer_sync();
    }
  }
}

// Ascending bitonic sort of idx[0, P) (P a power of two) by the consumer threads.
__device__ __forceinline__ void big_sort_asc_u32(uint32_t* idx, int P) {
  const int ctid = threadIdx.x - 32;
  for (int size = 2; size <= P; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      for (int i = ctid; i < P; i += kConsumers) {
        const int l = i ^ j;
        if (l > i) {
          const uint32_t a = idx[i], b = idx[l];
          const bool asc = (i & size) == 0;
          if (asc ? a > b : a < b) {
            idx[i] = b;
            idx[l] = a;
          }
        }
      }
      consumer_sync();
    }
  }
}

// Exact radix selection over the band's composite keys (fallback).  One pass
// over the row per 8-bit digit, from the highest digit in which the band's
// keys differ: counts and fixed-point masses of the digit values among the
// band's keys that match the prefix so far and are >= floor.  Lanes holding
// the same digit and the same logit are combined before the shared-memory
// atomics (equal logits have equal weights).
//   by_mass == false: the need-th largest band key (top-k); *W = base mass +
//                     the mass of the band keys >= it, *kept = base count +
//                     need.
//   by_mass == true:  the last band key (in descending order) whose preceding
//                     mass (base mass + the band keys above it) is below lim
//                     (top-p); *W = the mass up to and including it, *kept =
//                     the keys >= it.
template <class E, class InBand>
__device__ unsigned long long big_radix(const void* rowp, int V, float M, float c2, bool by_mass,
                                        unsigned need, unsigned long long lim,
                                        unsigned long long floor, unsigned cnt_base,
                                        unsigned long long mass_base, unsigned long long kmin,
                                        unsigned long long kmax, InBand in_band, unsigned* hc,
                                        unsigned long long* hm, BigShared& S,
                                        unsigned long long* W, int* kept) {
  const int ctid = threadIdx.x - 32, lane = ctid & 31;
  constexpr uint32_t skip = E::kSize == 2 ? ((1u << 5) | (1u << 4) | (1u << 3)) : (1u << 3);
  const unsigned long long diff = kmin ^ kmax;
  const int top = diff ? ((63 - __clzll(diff)) & ~7) : 0;  // highest differing digit
  unsigned long long mask = top + 8 < 64 ? ~0ull << (top + 8) : 0ull;
  unsigned long long prefix = kmax & mask;
  unsigned long long mass_above = mass_base;
  unsigned cnt_above = cnt_base;
  for (int shift = top; shift >= 0; shift -= 8) {
    if ((skip >> (shift / 8)) & 1u) continue;
    for (int i = ctid; i < 256; i += kConsumers) {
      hc[i] = 0u;
      hm[i] = 0ull;
    }
    consumer_sync();
    big_visit_global<E>(rowp, V, [&](float x, int idx) {
      if (!in_band(x)) return;
      const unsigned long long key = composite_key(x, uint32_t(idx));
      if ((key & mask) == prefix && key >= floor) {
        const int d = int(key >> shift) & 255;
        atomicAdd(&hc[d], 1u);
        const unsigned long long wf = big_wfix(x, M, c2);
        if (wf) atomicAdd(&hm[d], wf);
      }
    });
    consumer_sync();
    if (ctid < 32) {
      // lane owns digits 8 lane .. 8 lane + 7; suffix sums over higher digits
      unsigned c8[8], lc = 0u;
      unsigned long long m8[8], lm = 0ull;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c8[j] = hc[lane * 8 + j];
        m8[j] = hm[lane * 8 + j];
        lc += c8[j];
        lm += m8[j];
      }
      unsigned sc = lc;
      unsigned long long sm = lm;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned yc = __shfl_down_sync(0xffffffffu, sc, o);
        const unsigned long long ym = __shfl_down_sync(0xffffffffu, sm, o);
        if (lane + o < 32) {
          sc += yc;
          sm += ym;
        }
      }
      unsigned ac = sc - lc;           // counts of the digits above this lane's
      unsigned long long am = sm - lm; // and their masses
      int best = -1;
      unsigned bc = 0u, bcnt = 0u;
      unsigned long long bm = 0ull, bmass = 0ull;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        const bool pick = by_mass ? (c8[j] > 0u && mass_above + am < lim)
                                  : (ac < need && ac + c8[j] >= need);
        if (pick) {  // by mass: keep the lowest digit that qualifies
          best = lane * 8 + j;
          bc = ac;
          bm = am;
          bcnt = c8[j];
          bmass = m8[j];
        }
        ac += c8[j];
        am += m8[j];
      }
      // by count exactly one digit qualifies; by mass the lowest one is wanted
      const int dmin = __reduce_min_sync(0xffffffffu, best >= 0 ? best : 1 << 30);
      if (best >= 0 && best == dmin) {
        S.digit = best;
        S.dabove = bc;
        S.dmass_above = bm;
        S.dcnt = int(bcnt);
        S.dmass = bmass;
      }
    }
    consumer_sync();
    const int d = S.digit;
    const unsigned above = S.dabove, grp = unsigned(S.dcnt);
    const unsigned long long mabove = S.dmass_above, gmass = S.dmass;
    consumer_sync();
    prefix |= static_cast<unsigned long long>(d) << shift;
    mask |= 255ull << shift;
    cnt_above += above;
    mass_above += mabove;
    if (!by_mass) need -= above;
    if ((!by_mass && grp == need) || (by_mass && grp == 1u) || shift == 0) {
      // the group is taken whole (by count) or is a single key (by mass): its
      // smallest key is the threshold
      if (ctid == 0) S.minkey = ~0ull;
      consumer_sync();
      unsigned long long mn = ~0ull;
      big_visit_global<E>(rowp, V, [&](float x, int idx) {
        if (!in_band(x)) return;
        const unsigned long long key = composite_key(x, uint32_t(idx));
        if ((key & mask) == prefix && key >= floor && key < mn) mn = key;
      });
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long y = shfl_xor_u64(mn, o);
        mn = y < mn ? y : mn;
      }
      if (lane == 0) atomicMin(&S.minkey, mn);
      consumer_sync();
      const unsigned long long key = S.minkey;
      consumer_sync();
      *W = mass_above + gmass;
      *kept = int(cnt_above + grp);
      return key;
    }
  }
  *W = mass_above;  // not reached: the last digit leaves a single key
  *kept = int(cnt_above);
  return prefix;
}

// One kBig row: three streams of the row, then the threshold and kept mass.
// hist / sel: the row pass's selection scratch (radix selection in the band).
template <class E>
__device__ __forceinline__ void big_row(const Problem& P, const BigRing& r, BigShared& S,
                                        int* hist, SelShared* sel, unsigned char* work,
                                        const RowJob ent, const void* rowp, int ntiles,
                                        int last_nvec, int tail_start, int n_tail) {
  const Ws& w = P.ws;
  const int ctid = threadIdx.x - 32, cwarp = ctid >> 5, lane = ctid & 31;
  const int64_t row = ent.row;
  const int b = ent.b;
  const float T = ent.T;
  const int V = P.V;
  const int K = ent.K;
  const bool topk_on = K > 0 && K < V;
  const float tp = P.top_p ? P.top_p[b] : 1.0f;
  const bool topp_on = tp < 1.0f;
  unsigned* hc = reinterpret_cast<unsigned*>(work);
  unsigned long long* hm = reinterpret_cast<unsigned long long*>(work + 4 * kBigBins);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(work);
  constexpr unsigned long long kTag = 1ull << 63;  // hm[bin]: a single value's bits

  // ---- A: max (NaN-propagating) and the smallest finite logit
  float mx = -INFINITY, mn = INFINITY;
  big_stream<E>(r, ntiles, last_nvec, rowp, tail_start, n_tail,
                [&](const float* x, int, uint32_t vm) {
    if (!vm) return;
    float a = x[0], c = x[0];
#pragma unroll
    for (int e = 1; e < E::kPerVec; ++e) {
      a = fmax_nan(a, x[e]);
      c = fminf(c, x[e]);
    }
    mx = fmax_nan(mx, a);
    if (c > -INFINITY) {
      mn = fminf(mn, c);
    } else {  // -inf among them: the smallest finite one, element by element
#pragma unroll
      for (int e = 0; e < E::kPerVec; ++e)
        if (x[e] > -INFINITY) mn = fminf(mn, x[e]);
    }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if (lane == 0) {
    S.wmax[cwarp] = mx;
    S.wmin[cwarp] = mn;
  }
  consumer_sync();
  float M = S.wmax[0], Mn = S.wmin[0];
#pragma unroll
  for (int i = 1; i < kConsumerWarps; ++i) {
    M = fmax_nan(M, S.wmax[i]);
    Mn = fminf(Mn, S.wmin[i]);
  }
  // NaN or +inf anywhere, or no finite logit: a data error of the request
  const bool bad = !(M < INFINITY) || M == -INFINITY;
  const float c2 = __fdiv_rn(1.4426950408889634f, T);  // log2(e) / T
  float U = Mn > -INFINITY ? (M - Mn) * c2 : 64.0f;    // the bins' range of u
  U = fminf(fmaxf(U, 1.0f), 128.0f);
  // finite logits fill bins 0 .. kBigBins - 2 (the last one only by
  // rounding), -inf goes to the last bin
  const float cs = float(kBigBins - 2) / U * c2;
  auto bin_of = [&](float x) -> int {
    // round((M - x) * cs) (>= 0: M is the maximum) clamped to kBigBins - 1:
    // monotone in x
    const float u = fminf((M - x) * cs, float(kBigBins - 1));
    return __float_as_int(u + 12582912.0f) - 0x4B400000;
  };
  // A bin holds a single logit value when that value's neighbours in the
  // logit format (bf16 or f32) are at least two bin widths away: the value's
  // binary exponent then reaches ethr (its smaller neighbour gap is
  // 2^(E - 8) for bf16, 2^(E - 24) for f32; the bin width is 1 / cs).
  const int ethr = int(floorf(127.0f + float(E::kSize == 2 ? 8 : 24) + 1.0f - log2f(cs) +
                              1e-3f)) + 1;
  // |x| >= thr_abs iff the exponent of x reaches ethr
  const float thr_abs = ethr <= 0 ? 0.0f : (ethr >= 255 ? INFINITY : __int_as_float(ethr << 23));

  // ---- B: counts per bin; masses per bin, in fixed point: a single-value
  // bin's mass is its count times its value's weight (the value is recovered
  // from the bin below), any other bin sums its elements' weights
  for (int i = ctid; i < kBigBins; i += kConsumers) {
    hc[i] = 0u;
    hm[i] = 0ull;
  }
  consumer_sync();
  big_stream<E>(r, ntiles, last_nvec, rowp, tail_start, n_tail,
                [&](const float* x, int, uint32_t vm) {
    if (bad) return;
    constexpr uint32_t kAllE = (1u << E::kPerVec) - 1u;
    if (vm == kAllE) {
      // a whole vector: the bins first, then the counts, then the rare masses
      int bn[E::kPerVec];
#pragma unroll
      for (int e = 0; e < E::kPerVec; ++e) bn[e] = bin_of(x[e]);
#pragma unroll
      for (int e = 0; e < E::kPerVec; ++e) atomicAdd(&hc[bn[e]], 1u);
      uint32_t mixed = 0u;
#pragma unroll
      for (int e = 0; e < E::kPerVec; ++e)
        mixed |= (bn[e] >= kBigBins - 2 || !(fabsf(x[e]) >= thr_abs)) ? 1u << e : 0u;
      if (mixed) {
#pragma unroll
        for (int e = 0; e < E::kPerVec; ++e)
          if ((mixed >> e) & 1u) {
            const unsigned long long wf = big_wfix(x[e], M, c2);
            if (wf) atomicAdd(&hm[bn[e]], wf);
          }
      }
      return;
    }
#pragma unroll
    for (int e = 0; e < E::kPerVec; ++e) {
      if (!((vm >> e) & 1u)) continue;
      const int bn = bin_of(x[e]);
      atomicAdd(&hc[bn], 1u);
      if (bn >= kBigBins - 2 || !(fabsf(x[e]) >= thr_abs)) {
        const unsigned long long wf = big_wfix(x[e], M, c2);
        if (wf) atomicAdd(&hm[bn], wf);
      }
    }
  });
  consumer_sync();

  // ---- band: the bin of the K-th largest key and the bins of the top-p cut
  constexpr int BPT = kBigBins / kConsumers;  // bins per thread
  unsigned c8[BPT];
  unsigned long long m8[BPT];
  unsigned lc = 0u, pure_mask = 0u;
  unsigned long long lm = 0ull;
  const double inv_cs = 1.0 / double(cs);  // the bin width, for the bins' centres
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int bn = ctid * BPT + j;
    c8[j] = hc[bn];
    unsigned long long h = hm[bn];
    if (c8[j] > 0u && h == 0ull && bn < kBigBins - 2) {
      // A bin whose elements reach ethr holds one value, the representable
      // value nearest the bin's centre M - bn / cs (any other lies at least
      // 1.5 bin widths from it); its elements added no mass.  Its value is
      // recorded as the bin's tag.
      const float vc = float(fma(-double(bn), inv_cs, double(M)));
      float v = vc;
      if (E::kSize == 2) {
        uint32_t u = __float_as_uint(vc);
        u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;  // to bf16, nearest even
        v = __uint_as_float(u);
      }
      if (fabsf(v) >= thr_abs && bin_of(v) == bn) {
        h = kTag | __float_as_uint(v);
        hm[bn] = h;
      }
    }
    if (h & kTag) {
      m8[j] = (unsigned long long)c8[j] * big_wfix(__uint_as_float(uint32_t(h)), M, c2);
      pure_mask |= 1u << j;
    } else {
      m8[j] = h;
      if (c8[j] <= 1u) pure_mask |= 1u << j;
    }
    lc += c8[j];
    lm += m8[j];
  }
  unsigned pc0, tc;
  unsigned long long pm0, tm;
  big_scan(lc, lm, S, &pc0, &pm0, &tc, &tm);
  // the count and mass before each of this thread's bins, formed as the bins
  // are walked (kept in no arrays: registers are scarce here)
#define BIG_WALK_BINS(BODY)                    \
  {                                            \
    unsigned cbj = pc0;                        \
    unsigned long long mbj = pm0;              \
    _Pragma("unroll") for (int j = 0; j < BPT; ++j) { \
      BODY;                                    \
      cbj += c8[j];                            \
      mbj += m8[j];                            \
    }                                          \
  }
  if (ctid == 0) {
    S.ck = -1;
    S.plo = -1;
    S.phi = -1;
    S.total_mass = tm;
    S.nmixed = 0;
  }
  consumer_sync();
  if (topk_on) {
    BIG_WALK_BINS(if (cbj < unsigned(K) && unsigned(K) <= cbj + c8[j]) {
      S.ck = ctid * BPT + j;
      S.cnt_ck_before = cbj;
      S.mass_ck_before = mbj;
      S.cnt_ck = c8[j];
      S.mass_ck = m8[j];
    })
    consumer_sync();
  }
  const int ck = S.ck;
  if (topp_on) {
    // the top-p limit ceil(top_p * W_k) lies between the limits of the two
    // bounds of the top-k mass (equal without top-k); the crossing bin of a
    // limit L is the last non-empty bin whose preceding mass is below L
    const unsigned long long Wlo = topk_on ? S.mass_ck_before : tm;
    const unsigned long long Whi = topk_on ? S.mass_ck_before + S.mass_ck : tm;
    const unsigned long long llo = ceil_mul_frac(Wlo, tp), lhi = ceil_mul_frac(Whi, tp);
    int blo = -1, bhi = -1;
    BIG_WALK_BINS({
      const int bn = ctid * BPT + j;
      if (c8[j] > 0u && (!topk_on || bn <= ck)) {
        if (mbj < llo) blo = bn;
        if (mbj < lhi) bhi = bn;
      }
    })
    if (blo >= 0) atomicMax(&S.plo, blo);
    if (bhi >= 0) atomicMax(&S.phi, bhi);
    consumer_sync();
    // bin 0 holds the maximum, whose preceding mass is 0
    const int plo = max(S.plo, 0), phi = max(S.phi, plo);
    BIG_WALK_BINS({
      const int bn = ctid * BPT + j;
      if (bn == plo) {
        S.cnt_p_before = cbj;
        S.mass_p_before = mbj;
      }
      if (bn == phi) S.cnt_phi_end = cbj + c8[j];
    })
    consumer_sync();
    if (ctid == 0) {
      S.plo = plo;
      S.phi = phi;
      unsigned n = S.cnt_phi_end - S.cnt_p_before;
      if (topk_on && ck > phi) n += S.cnt_ck;
      S.nband = int(n);
    }
  } else if (ctid == 0) {
    S.nband = int(S.cnt_ck);
  }
  if (ctid == 0) S.count = 0;
  consumer_sync();
  const int plo = S.plo, phi = S.phi;
  // a band bin holding more than one value needs the band sorted
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int bn = ctid * BPT + j;
    if (!((pure_mask >> j) & 1u) && ((bn >= plo && bn <= phi) || bn == ck))
      atomicAdd(&S.nmixed, 1);
  }
  auto in_band = [&](float x) {
    const int bn = bin_of(x);
    return (bn >= plo && bn <= phi) || bn == ck;
  };

  // ---- C: the band's keys (as many as fit), and its key range.  When every
  // band bin holds one value and the values of its end bins are known, the
  // band is the value range [v(phi), v(plo)] (plus v(ck) for a top-k bin
  // apart): x lies in a band bin iff it lies in that range.
  unsigned long long kmin = ~0ull, kmax = 0ull;
  if (ctid == 0) {
    S.minkey = ~0ull;
    S.maxkey = 0ull;
    const float qnan = __int_as_float(0x7fc00000);
    float vhi = qnan, vlo = qnan, vk = qnan;
    bool known = true;
    auto tagged = [&](int bn, float* v) {
      const unsigned long long h = hm[bn];
      if (h & kTag) *v = __uint_as_float(uint32_t(h));
      else known = false;
    };
    if (topp_on) {
      tagged(plo, &vhi);
      tagged(phi, &vlo);
    }
    if (topk_on && !(topp_on && ck >= plo && ck <= phi)) tagged(ck, &vk);
    S.vhi = vhi;
    S.vlo = vlo;
    S.vk = vk;
    S.vknown = known;
  }
  consumer_sync();
  const bool by_value = S.vknown && S.nmixed == 0;
  const float vhi = S.vhi, vlo = S.vlo, vk = S.vk;
  unsigned long long kappa = 0ull, Wk = 0ull, Wfin = 0ull;
  int kept = 0;
  if (!bad && by_value && (!topp_on || phi - plo < kBandBins)) {
    // ---- every band bin holds one value: the cut follows from the counts
    // and the value weights alone.  The cut's value v and the number m of its
    // occurrences that are kept are known from the bins; the kept key is that
    // of the m-th occurrence of v in index order, found by counting v per
    // tile in one stream and then scanning the one tile that holds it.
    BIG_WALK_BINS({
      const int bn = ctid * BPT + j;
      const bool in_p = topp_on && bn >= plo && bn <= phi;
      if (in_p) {
        const int sl = bn - plo;
        S.bcnt[sl] = c8[j];
        S.bcb[sl] = cbj;
        S.bmb[sl] = mbj;
        S.bw[sl] = c8[j] ? m8[j] / c8[j] : 0ull;  // a single value's weight
      }
    })
    consumer_sync();
    if (ctid == 0) {
      S.fc_ok = 1;
      int cut_bin = -1;
      unsigned m = 0u;
      unsigned long long W_k = S.total_mass;
      unsigned need = 0u;
      if (topk_on) {
        need = unsigned(K) - S.cnt_ck_before;
        W_k = S.mass_ck_before + (unsigned long long)need * (S.cnt_ck ? S.mass_ck / S.cnt_ck : 0ull);
        cut_bin = ck;
        m = need;
      }
      S.W = W_k;
      S.kept = topk_on ? K : V;
      if (topp_on) {
        const unsigned long long lim = ceil_mul_frac(W_k, tp);
        const int nb = min(phi - plo + 1, kBandBins);
        cut_bin = -1;
        for (int sl = 0; sl < nb; ++sl) {
          const int bn = plo + sl;
          const unsigned c = S.bcnt[sl];
          if (c == 0u) continue;
          const unsigned long long before = S.bmb[sl], wv = S.bw[sl];
          if (before >= lim) break;  // nothing of this bin is kept
          // keep occurrence j of the bin's value while before + j wv < lim
          unsigned nk = wv ? unsigned(min((unsigned long long)c, (lim - before + wv - 1) / wv)) : c;
          bool stop = nk < c;
          if (topk_on && bn == ck && nk >= need) {
            nk = need;  // the top-k cut comes first
            stop = true;
          }
          cut_bin = bn;
          m = nk;
          S.W = before + (unsigned long long)nk * wv;
          S.kept = int(S.bcb[sl] + nk);
          if (stop) break;
        }
        if (cut_bin < 0) S.kept = -1;  // a band without the crossing
      }
      const unsigned long long h = cut_bin >= 0 ? hm[cut_bin] : 0ull;
      if (cut_bin < 0 || !(h & kTag) || m == 0u) {
        S.fc_ok = 0;
      } else {
        S.fc_v = __uint_as_float(uint32_t(h));
        S.fc_m = m;
        S.fc_expect = hc[cut_bin];
      }
    }
    consumer_sync();
    const bool ok = S.fc_ok != 0;
    const float fv = S.fc_v;
    // occurrences of v per tile (the bulk tiles, then the tail as one more)
    unsigned* tcnt = hc;
    for (int i = ctid; i <= ntiles; i += kConsumers) tcnt[i] = 0u;
    consumer_sync();
    constexpr int kTE = kTileBytes / E::kSize;  // elements per tile
    big_stream<E>(r, ntiles, last_nvec, rowp, tail_start, n_tail,
                  [&](const float* x, int i0, uint32_t vm) {
      if (!ok) return;
      unsigned c = 0u;
#pragma unroll
      for (int e = 0; e < E::kPerVec; ++e) c += ((vm >> e) & 1u) && x[e] == fv ? 1u : 0u;
      c = __reduce_add_sync(0xffffffffu, c);
      // a warp's vectors lie in one tile (the tail's elements in the last one)
      if (lane == 0 && c) atomicAdd(&tcnt[min(i0 / kTE, ntiles)], c);
    });
    consumer_sync();
    if (ok && cwarp == 0) {
      // the tile holding occurrence m: the first whose inclusive count reaches m
      unsigned carry = 0u, tstar = ~0u, before = 0u;
      for (int t0 = 0; t0 <= ntiles; t0 += 32) {
        const unsigned v = t0 + lane <= ntiles ? tcnt[t0 + lane] : 0u;
        unsigned incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        incl += carry;
        const uint32_t hit = __ballot_sync(0xffffffffu, tstar == ~0u && incl >= S.fc_m);
        if (tstar == ~0u && hit) {
          const int l = __ffs(hit) - 1;
          tstar = unsigned(t0 + l);
          before = __shfl_sync(0xffffffffu, incl - v, l);
        }
        carry = __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        if (carry != S.fc_expect || tstar == ~0u) {
          S.fc_ok = 0;  // the streams disagree
        } else {
          S.fc_tile = tstar;
          S.fc_mr = S.fc_m - before;
        }
      }
    }
    consumer_sync();
    if (S.fc_ok) {
      // the tile's elements in index order, a run of consecutive ones per thread
      const int e0 = int(S.fc_tile) * kTE;
      const int e1 = min(V, e0 + kTE);
      constexpr int kRun = kTE / kConsumers;  // 64 bytes: four 16-byte vectors
      constexpr int kVec = kRun / E::kPerVec;
      static_assert(kVec == 4, "a thread's run is four vectors");
      const int a = e0 + ctid * kRun, z = min(e1, a + kRun);
      // the run's match mask (bit i: element a + i), from four vector loads
      // when the run lies whole inside the row
      uint32_t mm = 0u;
      if (z - a == kRun) {
        const uint4* vp = reinterpret_cast<const uint4*>(static_cast<const char*>(rowp) +
                                                         size_t(a) * E::kSize);
        uint4 q[kVec];
#pragma unroll
        for (int i = 0; i < kVec; ++i) q[i] = __ldcg(vp + i);
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
          float x[E::kPerVec];
          E::decode(q[i], x);
#pragma unroll
          for (int e = 0; e < E::kPerVec; ++e)
            mm |= x[e] == fv ? 1u << (i * E::kPerVec + e) : 0u;
        }
      } else {
        for (int e = a; e < z; ++e) mm |= E::scalar(rowp, e) == fv ? 1u << (e - a) : 0u;
      }
      const unsigned c = __popc(mm);
      unsigned pre, tot;
      unsigned long long pm, tm;
      big_scan(c, 0ull, S, &pre, &pm, &tot, &tm);
      const unsigned mr = S.fc_mr;
      if (pre < mr && mr <= pre + c) {
        // the (mr - pre)-th set bit of the mask
        uint32_t m2 = mm;
        for (unsigned k = pre + 1; k < mr; ++k) m2 &= m2 - 1u;
        S.fc_idx = a + __ffs(m2) - 1;
      }
      consumer_sync();
      kappa = composite_key(fv, uint32_t(S.fc_idx));
      Wfin = S.W;
      Wk = Wfin;
      kept = S.kept;
      if (kept < 0) {
        if (ctid == 0) flag_request(w, b, SV_ERR_INTERNAL, row);
        kept = 0;
      }
    } else if (ctid == 0) {
      flag_request(w, b, SV_ERR_INTERNAL, row);  // the two streams disagree
    }
  } else {
    big_stream<E>(r, ntiles, last_nvec, rowp, tail_start, n_tail,
                  [&](const float* x, int i0, uint32_t vm) {
      if (bad) return;
      uint32_t m = 0u;
  #pragma unroll
      for (int e = 0; e < E::kPerVec; ++e) {
        const bool in = by_value ? ((x[e] >= vlo && x[e] <= vhi) || x[e] == vk) : in_band(x[e]);
        m |= (in && ((vm >> e) & 1u)) ? 1u << e : 0u;
      }
      if (!__any_sync(0xffffffffu, m != 0u)) return;
      const int cnt = __popc(m);
      int incl = cnt;
  #pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int base = 0;
      if (lane == 31) base = atomicAdd(&S.count, incl);
      base = __shfl_sync(0xffffffffu, base, 31);
      int slot = base + incl - cnt;
  #pragma unroll
      for (int e = 0; e < E::kPerVec; ++e)
        if ((m >> e) & 1u) {
          const unsigned long long key = composite_key(x[e], uint32_t(i0 + e));
          if (slot < kBigCap) keys[slot] = key;
          ++slot;
          kmin = key < kmin ? key : kmin;
          kmax = key > kmax ? key : kmax;
        }
    });
  #pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long a = shfl_xor_u64(kmin, o), c = shfl_xor_u64(kmax, o);
      kmin = a < kmin ? a : kmin;
      kmax = c > kmax ? c : kmax;
    }
    if (lane == 0 && !bad) {
      atomicMin(&S.minkey, kmin);
      atomicMax(&S.maxkey, kmax);
    }
    consumer_sync();
    const unsigned long long band_min = S.minkey, band_max = S.maxkey;
    const int n = S.count;
    const bool pure = S.nmixed == 0;

    if (!bad && n != S.nband && ctid == 0)
      flag_request(w, b, SV_ERR_INTERNAL, row);  // the two streams disagree
    if (!bad && pure && n <= kBigCap && n == S.nband && (!topp_on || phi - plo < kBandBins)) {
      // ---- every band bin holds one value: the cut follows from the counts
      // and the value weights, and the kept key from one radix selection over
      // the band's keys (the r-th largest: r counted from the band's first bin)
      constexpr uint32_t kSkip = E::kSize == 2 ? kSkipBf16 : kSkipF32;
      const int first = topp_on ? plo : ck;
      if (ctid == 0) {
        // cnt_before / mass_before / value weight of the bins met below
        S.kept = 0;
      }
      consumer_sync();
      // per-bin facts of the band bins, gathered by their owner threads: slot
      // bn - plo for the top-p bins, slot kBandBins for a top-k bin apart
      // from them
      BIG_WALK_BINS({
        const int bn = ctid * BPT + j;
        if (bn == first) S.cnt_first = cbj;
        const bool in_p = topp_on && bn >= plo && bn <= phi;
        const bool apart_k = topk_on && bn == ck && !in_p;
        if (in_p || apart_k) {
          const int s = in_p ? bn - plo : kBandBins;
          S.bcnt[s] = c8[j];
          S.bcb[s] = cbj;
          S.bmb[s] = mbj;
          S.bw[s] = c8[j] ? m8[j] / c8[j] : 0ull;  // a single value's weight
        }
      })
      consumer_sync();
      unsigned r_k = 0u, r_p = 0u;  // ranks (1-based) in the band of the two cuts
      if (ctid == 0) {
        unsigned long long W_k = S.total_mass;
        unsigned need = 0u;
        int sk = -1;
        if (topk_on) {
          sk = topp_on && ck >= plo && ck <= phi ? ck - plo : kBandBins;
          need = unsigned(K) - S.cnt_ck_before;
          W_k = S.mass_ck_before + (unsigned long long)need * S.bw[sk];
          r_k = (S.cnt_ck_before - S.cnt_first) + need;
          if (topp_on && ck > phi) r_k = (S.cnt_phi_end - S.cnt_first) + need;
        }
        S.W = W_k;
        S.kept = topk_on ? K : V;
        S.rk = r_k;
        S.rp = 0u;
        if (topp_on) {
          const unsigned long long lim = ceil_mul_frac(W_k, tp);
          const int nb = min(phi - plo + 1, kBandBins);
          for (int s = 0; s < nb; ++s) {
            const int bn = plo + s;
            const unsigned c = S.bcnt[s];
            if (c == 0u) continue;
            const unsigned long long before = S.bmb[s], wv = S.bw[s];
            if (before >= lim) break;  // nothing of this bin is kept
            // keep element j of the bin while before + j wv < lim
            unsigned nk = wv ? unsigned(min((unsigned long long)c, (lim - before + wv - 1) / wv)) : c;
            bool stop = nk < c;
            if (topk_on && bn == ck && nk >= need) {
              nk = need;  // the top-k cut comes first
              stop = true;
            }
            S.rp = (S.bcb[s] - S.cnt_first) + nk;
            S.W = before + (unsigned long long)nk * wv;
            S.kept = int(S.bcb[s] + nk);
            if (stop) break;
          }
          if (S.rp == 0u) S.kept = -1;  // a band without the crossing
        }
      }
      consumer_sync();
      r_k = S.rk;
      r_p = S.rp;
      Wfin = S.W;
      kept = S.kept;
      if (topk_on) {
        kappa = block_select_kth<kConsumers>(reinterpret_cast<const uint64_t*>(keys), n, int(r_k),
                                             ctid, hist, sel, BigSync(), kSkip);
        Wk = Wfin;
      }
      if (topp_on) {
        if (kept < 0) {
          if (ctid == 0) flag_request(w, b, SV_ERR_INTERNAL, row);
          kept = 0;
        } else {
          kappa = block_select_kth<kConsumers>(reinterpret_cast<const uint64_t*>(keys), n,
                                               int(r_p), ctid, hist, sel, BigSync(), kSkip);
        }
      }
    } else if (!bad && n <= kBigSort && n == S.nband) {
      // ---- a band bin holds several values: sort the band (descending key)
      const int P2 = next_pow2(n > 1 ? n : 2);
      for (int i = n + ctid; i < P2; i += kConsumers) keys[i] = 0ull;  // sorts last
      consumer_sync();
      big_sort_desc(keys, P2);
      const int C = (n + kConsumers - 1) / kConsumers;  // positions per thread
      const int c0 = min(n, ctid * C), c1 = min(n, c0 + C);
      unsigned long long cm = 0ull;
      for (int i = c0; i < c1; ++i) cm += big_wfix(composite_value(keys[i]), M, c2);
      unsigned dummy_c, dummy_t;
      unsigned long long pre0, dummy_m;
      big_scan(0u, cm, S, &dummy_c, &pre0, &dummy_t, &dummy_m);  // mass before c0
      if (ctid == 0) {
        S.sk = n;
        S.nkept = 0;
      }
      consumer_sync();
      if (topk_on) {
        for (int i = c0; i < c1; ++i)
          if (bin_of(composite_value(keys[i])) == ck) {
            atomicMin(&S.sk, i);
            break;
          }
        consumer_sync();
        const int sk = S.sk;
        const int pk = sk + int(unsigned(K) - S.cnt_ck_before) - 1;  // the K-th largest
        unsigned long long pre = pre0;
        for (int i = c0; i < c1; ++i) {
          if (i == sk) S.pre_sk = pre;
          pre += big_wfix(composite_value(keys[i]), M, c2);
          if (i == pk) {
            S.pre_pk1 = pre;
            S.key_k = keys[i];
          }
        }
        consumer_sync();
        Wk = S.mass_ck_before + (S.pre_pk1 - S.pre_sk);
        kappa = S.key_k;
        kept = K;
      } else {
        Wk = S.total_mass;
      }
      Wfin = Wk;
      if (topp_on) {
        // keep j while the mass before it is below ceil(top_p * W_k) (and j is
        // within the top k): a prefix of the band's first bins
        const unsigned long long lim = ceil_mul_frac(Wk, tp);
        const unsigned long long kfloor = kappa;
        unsigned long long pre = pre0;
        int nk = 0;
        for (int i = c0; i < c1; ++i) {
          const unsigned long long key = keys[i];
          const float v = composite_value(key);
          if (bin_of(v) <= phi && S.mass_p_before + pre < lim && key >= kfloor) ++nk;
          pre += big_wfix(v, M, c2);
        }
        if (nk) atomicAdd(&S.nkept, nk);
        consumer_sync();
        const int istar = S.nkept - 1;
        pre = pre0;
        for (int i = c0; i < c1; ++i) {
          const unsigned long long key = keys[i];
          const unsigned long long wf = big_wfix(composite_value(key), M, c2);
          if (i == istar) {
            S.key = key;
            S.W = S.mass_p_before + pre + wf;
          }
          pre += wf;
        }
        consumer_sync();
        if (istar >= 0) {
          kappa = S.key;
          Wfin = S.W;
          kept = int(S.cnt_p_before) + istar + 1;
        } else if (ctid == 0) {
          flag_request(w, b, SV_ERR_INTERNAL, row);  // a band without the crossing
        }
      }
    } else if (!bad && n == S.nband) {
      // ---- exact radix selection over the band, from global memory
      unsigned* xc = reinterpret_cast<unsigned*>(work);
      unsigned long long* xm = reinterpret_cast<unsigned long long*>(work + 1024);
      kappa = 0ull;
      Wk = S.total_mass;
      kept = V;
      if (topk_on) {
        auto in_k = [&](float x) { return bin_of(x) == ck; };
        kappa = big_radix<E>(rowp, V, M, c2, false, unsigned(K) - S.cnt_ck_before, 0ull, 0ull,
                             S.cnt_ck_before, S.mass_ck_before, band_min, band_max, in_k, xc, xm,
                             S, &Wk, &kept);
      }
      Wfin = Wk;
      if (topp_on) {
        auto in_p = [&](float x) {
          const int bn = bin_of(x);
          return bn >= plo && bn <= phi;
        };
        kappa = big_radix<E>(rowp, V, M, c2, true, 0u, ceil_mul_frac(Wk, tp), kappa,
                             S.cnt_p_before, S.mass_p_before, band_min, band_max, in_p, xc, xm, S,
                             &Wfin, &kept);
      }
    }
  }
  if (ctid == 0) {
    double pg = __longlong_as_double(0x7ff8000000000000LL);
    const int gx = ent.gx;
    if (bad) {
      flag_request(w, b, SV_ERR_DATA_LOGIT, row);
    } else if (gx >= 0) {
      const float xg = E::scalar(rowp, gx);
      pg = composite_key(xg, uint32_t(gx)) >= kappa
               ? exp((double(xg) - double(M)) / double(T)) / (double(Wfin) / double(kFix40))
               : 0.0;
    }
    RowStat st;
    st.s = bad ? 0.0 : double(Wfin) / double(kFix40);
    st.pg = pg;
    st.m = M;
    st.arg = -1;
    st.kept = bad ? 0 : kept;
    st.mode = kBig;
    w.stats[row] = st;
    w.cand_raw[size_t(row) * kRawCap] = kappa;
  }
  consumer_sync();  // the work area and S are reused by the next row
}
#undef BIG_WALK_BINS
