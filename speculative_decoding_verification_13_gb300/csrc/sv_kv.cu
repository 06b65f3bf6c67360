// KV-cache commit after verification: the accepted entries of each request's
// speculative K/V buffer are appended to its paged cache, the rejected ones
// are dropped ("FlashMap…", section "Architecture": the verification stage
// updates the paged KV cache with the accepted tokens; "Speculative decoding
// and multi-token prediction", "Practical guidance": a rollback that does not
// truncate on rejection breaks the equality of outputs).
//
// Layout (chosen; the pages define none): cache [num_pages, n_layers, 2,
// page_size, E], spec [B, spec_slots, n_layers, 2, E]; position p of request
// b lives in page block_table[b][p / page_size], slot p % page_size.  With
// accept length L >= 0, spec entries 0..L (the last emitted token, then the L
// accepted drafts) go to positions kv_len .. kv_len + L, and kv_len grows by
// L + 1.
//
// Two launches: a validation CTA (accept lengths, destination pages, new
// lengths, the list of tokens to copy), then a copy kernel in which one warp
// moves one (token, layer, K or V) entry of E elements with 16-byte loads and
// stores.  The copy is HBM-bound: every byte is read once and written once.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kKvThreads = 1024;   // validation CTA
constexpr int kCopyThreads = 256;  // copy kernel

struct KvProblem {
  char* cache;
  const char* spec;
  int64_t num_pages;
  int32_t n_layers, page_size;
  int64_t entry_bytes;     // E * element size, a multiple of 16
  int32_t spec_slots;
  const int32_t* accept_len;
  const int32_t* k_per_req;
  int32_t* kv_len;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t B;
  WsHeader* hdr;
  int32_t* start;          // [B] kv_len before the commit
  int2* tokens;            // [B * (SV_MAX_K + 1)] (request, entry) to copy
};

__device__ int kv_block_scan(int v, int* total) {
  __shared__ int s_w[kKvThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int y = s_w[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_w[lane] = y;
  }
  __syncthreads();
  const int ex = x - v + (warp ? s_w[warp - 1] : 0);
  *total = s_w[kKvThreads / 32 - 1];
  __syncthreads();
  return ex;
}

__global__ void __launch_bounds__(kKvThreads) kv_validate_kernel(const KvProblem Q) {
  // launched as a dependent of whatever the stream ran before: nothing is
  // read or written before that has completed
  pdl_wait();
  pdl_trigger();  // the copy kernel may launch; it waits for this one
  if (threadIdx.x == 0) {
    Q.hdr->err_code = 0;
    Q.hdr->err_req = -1;
    Q.hdr->err_row = -1;
    Q.hdr->n_active = 0;
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < Q.B; base += kKvThreads) {
    const int b = base + threadIdx.x;
    int cnt = 0;
    if (b < Q.B) {
      const int L = Q.accept_len[b];
      const int n = Q.kv_len[b];
      int code = 0;
      if (L >= 0) {
        if (L > SV_MAX_K || L > Q.k_per_req[b] || L + 1 > Q.spec_slots) {
          code = SV_ERR_DATA_ACCEPT;
        } else if (n < 0) {
          code = SV_ERR_DATA_PAGE;
        } else {
          // every destination page must be in the block table and the pool
          const int64_t c0 = int64_t(n) / Q.page_size, c1 = (int64_t(n) + L) / Q.page_size;
          for (int64_t col = c0; col <= c1; ++col) {
            const int page = col < Q.max_pages ? Q.block_table[int64_t(b) * Q.max_pages + col] : -1;
            if (page < 0 || page >= Q.num_pages) code = SV_ERR_DATA_PAGE;
          }
        }
        if (code) record_error(Q.hdr, code, b, -1);
        else cnt = L + 1;
      }
      Q.start[b] = n;
      if (cnt) Q.kv_len[b] = n + cnt;
    }
    int tot;
    const int t0 = carry + kv_block_scan(cnt, &tot);
    for (int j = 0; j < cnt; ++j) Q.tokens[t0 + j] = make_int2(b, j);
    carry += tot;
  }
  if (threadIdx.x == 0) Q.hdr->n_active = carry;
}

// One warp per (token, layer, K/V) entry, entries taken round-robin.
__global__ void __launch_bounds__(kCopyThreads) kv_copy_kernel(const KvProblem Q) {
  pdl_wait();  // the token list, start lengths and validation
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t(blockIdx.x) * kCopyThreads + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * kCopyThreads) >> 5;
  const int64_t per_token = int64_t(Q.n_layers) * 2;
  const int64_t items = int64_t(Q.hdr->n_active) * per_token;
  const int64_t vecs = Q.entry_bytes / 16;
  for (int64_t it = wid; it < items; it += nw) {
    const int2 tk = Q.tokens[it / per_token];
    const int64_t lc = it % per_token;  // layer * 2 + (K or V)
    const int64_t pos = int64_t(Q.start[tk.x]) + tk.y;
    const int64_t page = Q.block_table[int64_t(tk.x) * Q.max_pages + pos / Q.page_size];
    const int64_t slot = pos % Q.page_size;
    const uint4* src = reinterpret_cast<const uint4*>(
        Q.spec + ((int64_t(tk.x) * Q.spec_slots + tk.y) * per_token + lc) * Q.entry_bytes);
    uint4* dst = reinterpret_cast<uint4*>(
        Q.cache + ((page * per_token + lc) * Q.page_size + slot) * Q.entry_bytes);
    // four 16-byte vectors per lane in flight, then their stores
    int64_t v = lane;
    for (; v + 96 < vecs; v += 128) {
      const uint4 a = __ldcs(src + v), b = __ldcs(src + v + 32), c = __ldcs(src + v + 64),
                  d = __ldcs(src + v + 96);
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = d;
    }
    for (; v < vecs; v += 32) dst[v] = __ldcs(src + v);
  }
}

}  // namespace

size_t kv_workspace_bytes(int32_t B) {
  size_t o = align256(sizeof(WsHeader));
  o = align256(o + sizeof(int32_t) * size_t(B > 0 ? B : 1));
  o = align256(o + sizeof(int2) * size_t(B > 0 ? B : 1) * (SV_MAX_K + 1));
  return o;
}

cudaError_t launch_kv_commit(void* cache, const void* spec, int64_t num_pages, int n_layers,
                             int page_size, int64_t entry_bytes, int spec_slots,
                             const int32_t* accept_len, const int32_t* k_per_req,
                             int32_t* kv_len, const int32_t* block_table, int max_pages, int B,
                             void* workspace, int sms, cudaStream_t s) {
  KvProblem Q;
  Q.cache = static_cast<char*>(cache);
  Q.spec = static_cast<const char*>(spec);
  Q.num_pages = num_pages;
  Q.n_layers = n_layers;
  Q.page_size = page_size;
  Q.entry_bytes = entry_bytes;
  Q.spec_slots = spec_slots;
  Q.accept_len = accept_len;
  Q.k_per_req = k_per_req;
  Q.kv_len = kv_len;
  Q.block_table = block_table;
  Q.max_pages = max_pages;
  Q.B = B;
  char* w = static_cast<char*>(workspace);
  size_t o = 0;
  Q.hdr = reinterpret_cast<WsHeader*>(w);
  o = align256(sizeof(WsHeader));
  Q.start = reinterpret_cast<int32_t*>(w + o);
  o = align256(o + sizeof(int32_t) * size_t(B > 0 ? B : 1));
  Q.tokens = reinterpret_cast<int2*>(w + o);
  cudaLaunchConfig_t vc = {};
  vc.gridDim = dim3(1);
  vc.blockDim = dim3(kKvThreads);
  vc.dynamicSmemBytes = 0;
  vc.stream = s;
  cudaLaunchAttribute va[1];
  va[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  va[0].val.programmaticStreamSerializationAllowed = 1;
  vc.attrs = va;
  vc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&vc, kv_validate_kernel, Q);
  if (e != cudaSuccess) return e;
  // enough warps for every entry of the largest commit, at most 8 CTAs per SM
  const int64_t items = int64_t(B) * (spec_slots < SV_MAX_K + 1 ? spec_slots : SV_MAX_K + 1) *
                        n_layers * 2;
  const int64_t want = (items + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int64_t cap = int64_t(sms) * 8;
  const int grid = int(want < cap ? (want > 0 ? want : 1) : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kCopyThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_copy_kernel, Q);
}

}  // namespace sv
