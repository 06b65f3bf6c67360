// LM-head GEMM with a fused verification-statistics epilogue, on the
// fifth-generation tensor cores (tcgen05) with TMA operand loads.
//
// The target's logits are the final hidden states times the unembedding
// matrix, z = H W^T ("FlashMap: Flow Map Speculative Decoding…", section 1),
// and verification needs of each row only its softmax statistics at the row's
// temperature, its argmax and its token's logit (§5 draft_block step 5; §4).
// Computing them in the epilogue means the logits never reach memory.
//
// Persistent CTAs (one per SM), work units of one 128-row tile of H by
// nchunk 256-column tiles of W (32, 16 or 8, chosen per call).  Warp 0: TMA
// producer (one lane) filling a 4-stage ring of 128-byte-swizzled 128x64 (H)
// and 256x64 (W) bf16 tiles.
// Warp 1: TMEM allocation and the MMA issuer (one lane): 128x256x16
// tcgen05.mma (kind::f16, bf16 inputs, f32 accumulators in TMEM), four per
// 64-wide K block, into one of two 256-column accumulators.  Warps 2-5: the
// epilogue, one row per thread (tcgen05.ld of 32 columns at a time): running
// max, first-index argmax, the token's logit and the online sum of
// exp((z - max) / T).  Per-chunk partial statistics go to global memory and a
// second kernel combines them per row.  Every wait is bounded; on expiry the
// kernel records SV_ERR_TIMEOUT, lets its copies and MMAs land and frees TMEM.
#include <cuda.h>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, kLmStages = 4;
constexpr int kLmThreads = 192;                       // 6 warps
constexpr int kTileA = BM * BK * 2;                   // 16 KB
constexpr int kTileB = BN * BK * 2;                   // 32 KB
constexpr int kLmStageBytes = kTileA + kTileB;        // 48 KB
constexpr int kNChunkMin = 8;                         // fewest W tiles per work unit
constexpr uint32_t kTmemCols = 2 * BN;                // two accumulators
constexpr size_t kLmSmem = size_t(kLmStages) * kLmStageBytes + 1024;  // + alignment slack

struct LmPartial {
  float m, s, xt;
  int arg;
};

struct LmArgs {
  int M, V, K;
  int mtiles, ntiles, n_chunks, kblocks;
  int nchunk;                // W tiles per work unit
  const float* temperature;  // [M]
  const int32_t* tokens;     // [M] or null
  LmPartial* part;           // [n_chunks, M]
  WsHeader* hdr;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  return uint64_t((addr & 0x3FFFFu) >> 4)       // start address
         | (uint64_t(1) << 16)                  // leading-dimension offset (unused here)
         | (uint64_t(1024 >> 4) << 32)          // stride between 8-row groups
         | (uint64_t(1) << 46)                  // descriptor version
         | (uint64_t(2) << 61);                 // 128-byte swizzle
}

// Instruction descriptor: f32 accumulator, bf16 A and B, both K-major, M x N.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                            (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait on an mbarrier phase; false (and the CTA's abort flag set) on expiry.
__device__ __forceinline__ bool lm_wait(uint32_t bar, uint32_t parity, int* abort_flag,
                                        uint32_t sleep_ns) {
  if (mbar_wait_for(bar, parity, kWaitNs, abort_flag, nullptr, sleep_ns)) return true;
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  return false;
}

__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_stats_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB, const LmArgs A) {
  extern __shared__ unsigned char lm_smem_raw[];
  __shared__ uint64_t bars[2 * kLmStages + 4];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // 1024-byte alignment for the swizzled tiles
  const uint32_t raw = smem_addr(lm_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t full0 = smem_addr(&bars[0]), empty0 = full0 + 8u * kLmStages;
  const uint32_t afull0 = empty0 + 8u * kLmStages, aempty0 = afull0 + 16u;
  if (tid == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(afull0 + 8u * b, 1);
      mbar_init(aempty0 + 8u * b, 4);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const int n_units = A.mtiles * A.n_chunks;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    bool stop = false;
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      const int mt = u % A.mtiles, c = u / A.mtiles;
      const int nt1 = min((c + 1) * A.nchunk, A.ntiles);
      for (int nt = c * A.nchunk; nt < nt1 && !stop; ++nt)
        for (int kb = 0; kb < A.kblocks; ++kb) {
          if (!lm_wait(empty0 + 8u * stage, phase ^ 1u, &abort_flag, 32)) {
            stop = true;
            break;
          }
          const uint32_t sa = base + stage * kLmStageBytes, sb = sa + kTileA;
          mbar_arrive_expect_tx(full0 + 8u * stage, kLmStageBytes);
          tma_load_2d(sa, &mapA, kb * BK, mt * BM, full0 + 8u * stage);
          tma_load_2d(sb, &mapB, kb * BK, nt * BN, full0 + 8u * stage);
          ++issued;
          if (++stage == kLmStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
    }
    if (stop) {
      record_error(A.hdr, SV_ERR_TIMEOUT, -1, -1);
      // let the copies this CTA issued land before the CTA exits
      const long long first = issued > kLmStages ? issued - kLmStages : 0;
      for (long long g = first; g < issued; ++g) {
        const uint32_t st = uint32_t(g % kLmStages), ph = uint32_t((g / kLmStages) & 1);
        mbar_wait_for(full0 + 8u * st, ph);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t stage = 0, phase = 0, ab = 0, aphase = 0;
    bool stop = false;
    long long commits = 0;  // accumulator commits issued
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      const int c = u / A.mtiles;
      const int nt1 = min((c + 1) * A.nchunk, A.ntiles);
      for (int nt = c * A.nchunk; nt < nt1 && !stop; ++nt) {
        if (!lm_wait(aempty0 + 8u * ab, aphase ^ 1u, &abort_flag, 64)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + ab * BN;
        for (int kb = 0; kb < A.kblocks; ++kb) {
          if (!lm_wait(full0 + 8u * stage, phase, &abort_flag, 16)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * kLmStageBytes, sb = sa + kTileA;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), (kb | k) != 0);
          umma_commit(empty0 + 8u * stage);  // the stage is free once these MMAs have read it
          if (++stage == kLmStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit(afull0 + 8u * ab);  // the accumulator is complete
        ++commits;
        if (++ab == 2) {
          ab = 0;
          aphase ^= 1u;
        }
      }
    }
    if (stop) {
      record_error(A.hdr, SV_ERR_TIMEOUT, -1, -1);
      // every MMA issued must finish before TMEM is freed: commit once more and wait
      umma_commit(afull0 + 8u * ab);
      mbar_wait_for(afull0 + 8u * ab, aphase);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // the TMEM lane quarter this warp may read
    const int r_in = q * 32 + lane;
    uint32_t ab = 0, aphase = 0;
    bool stop = false;
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      const int mt = u % A.mtiles, c = u / A.mtiles;
      const int row = mt * BM + r_in;
      const bool live = row < A.M;
      const float T = live ? A.temperature[row] : 1.0f;
      const float c2 = 1.4426950408889634f / (T > 0.0f ? T : 1.0f);
      const int tok = live && A.tokens ? A.tokens[row] : -1;
      float best = -INFINITY, s = 0.f, xt = __int_as_float(0x7fc00000);
      int arg = -1;
      const int nt1 = min((c + 1) * A.nchunk, A.ntiles);
      for (int nt = c * A.nchunk; nt < nt1; ++nt) {
        if (!lm_wait(afull0 + 8u * ab, aphase, &abort_flag, 128)) {
          stop = true;
          break;
        }
        tc_fence_after();
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + (uint32_t(q * 32) << 16) + ab * BN + cc * 32, r);
          tmem_ld_wait();
          const int n0 = nt * BN + cc * 32;
          const float prev = best;  // the maximum before these 32 columns
          bool any = false;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = __uint_as_float(r[j]);
            const bool ok = n0 + j < A.V;
            any |= ok;
            if (ok && x > best) {  // columns in increasing order: the first maximum stays
              best = x;
              arg = n0 + j;
            }
            if (n0 + j == tok) xt = x;
          }
          if (any) {
            // online sum of exp((x - max) / T): the old sum is rescaled to the
            // new maximum (a factor of 1 when it did not grow, 0 times 0 at the start)
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < A.V) acc += ex2_approx((__uint_as_float(r[j]) - best) * c2);
            s = s * ex2_approx((prev - best) * c2) + acc;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aempty0 + 8u * ab);
        if (++ab == 2) {
          ab = 0;
          aphase ^= 1u;
        }
      }
      if (live && !stop) A.part[size_t(c) * A.M + row] = LmPartial{best, s, xt, arg};
    }
  }
  __syncwarp();  // lanes without a role wait for their warp's lane 0
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

// Per row: combine the chunks' partial statistics.
__global__ void lmhead_combine_kernel(const LmArgs A, float* out_m, double* out_s,
                                      int32_t* out_arg, float* out_xt) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= A.M) return;
  const float T = A.temperature[r];
  const double c = 1.0 / double(T > 0.0f ? T : 1.0f);
  float m = -INFINITY, xt = __int_as_float(0x7fc00000);
  int arg = -1;
  for (int k = 0; k < A.n_chunks; ++k) {
    const LmPartial p = A.part[size_t(k) * A.M + r];
    if (p.m > m) {  // chunks in column order: the first maximum keeps the lowest index
      m = p.m;
      arg = p.arg;
    }
    if (p.xt == p.xt) xt = p.xt;
  }
  double s = 0.0;
  for (int k = 0; k < A.n_chunks; ++k) {
    const LmPartial p = A.part[size_t(k) * A.M + r];
    if (p.m > -INFINITY) s += double(p.s) * exp((double(p.m) - double(m)) * c);
  }
  out_m[r] = m;
  out_s[r] = s;
  out_arg[r] = arg;
  out_xt[r] = xt;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// A [rows, K] bf16 row-major matrix as TMA tiles of box_rows x 64, 128-byte swizzled.
bool make_map(CUtensorMap* map, const void* data, int rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(data), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W tiles per work unit: of 32, 16 and 8, the one that leaves the busiest
// CTA the fewest tiles (units in whole rounds over the grid), the larger on a
// tie.  Longer runs on one column chunk measured faster: the CTAs that share
// a W tile (one per row tile) stay on it together (4096 x 151936 x 4096:
// 32 tiles 2-4 % faster than 8 or 16; 24, which leaves a part-filled last
// round, 7 % slower).
int lm_nchunk(int mtiles, int ntiles, int sms) {
  int best = kNChunkMin;
  int64_t best_load = INT64_MAX;
  for (int c = 32; c >= kNChunkMin; c >>= 1) {
    const int64_t units = int64_t(mtiles) * ((ntiles + c - 1) / c);
    const int64_t grid = units < sms ? units : sms;
    const int64_t load = (units + grid - 1) / grid * c;
    if (load < best_load) {
      best_load = load;
      best = c;
    }
  }
  return best;
}

}  // namespace

size_t lmhead_workspace_bytes(int M, int V) {
  const int ntiles = (V + BN - 1) / BN;
  const int n_chunks = (ntiles + kNChunkMin - 1) / kNChunkMin;  // the most chunks a call uses
  return align256(sizeof(WsHeader)) + align256(sizeof(LmPartial) * size_t(n_chunks) * size_t(M > 0 ? M : 1));
}

int launch_lmhead_stats(const void* H, const void* W, int M, int V, int K,
                        const float* temperature, const int32_t* tokens, float* out_m,
                        double* out_s, int32_t* out_arg, float* out_xt, void* workspace,
                        int sms, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(lmhead_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kLmSmem)) != cudaSuccess)
      return SV_ERR_CUDA;
    configured = true;
  }
  CUtensorMap ma, mb;
  if (!make_map(&ma, H, M, K, BM) || !make_map(&mb, W, V, K, BN)) return SV_ERR_UNSUPPORTED;
  LmArgs A;
  A.M = M;
  A.V = V;
  A.K = K;
  A.mtiles = (M + BM - 1) / BM;
  A.ntiles = (V + BN - 1) / BN;
  A.nchunk = lm_nchunk(A.mtiles, A.ntiles, sms);
  A.n_chunks = (A.ntiles + A.nchunk - 1) / A.nchunk;
  A.kblocks = (K + BK - 1) / BK;
  A.temperature = temperature;
  A.tokens = tokens;
  A.hdr = static_cast<WsHeader*>(workspace);
  A.part = reinterpret_cast<LmPartial*>(static_cast<char*>(workspace) + align256(sizeof(WsHeader)));
  if (cudaMemsetAsync(A.hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return SV_ERR_CUDA;
  const int units = A.mtiles * A.n_chunks;
  const int grid = units < sms ? units : sms;
  lmhead_stats_kernel<<<grid, kLmThreads, kLmSmem, s>>>(ma, mb, A);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  lmhead_combine_kernel<<<(M + 255) / 256, 256, 0, s>>>(A, out_m, out_s, out_arg, out_xt);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace sv
