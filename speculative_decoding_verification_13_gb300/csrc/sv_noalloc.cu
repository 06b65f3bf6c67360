// spec_verify_noalloc: the same verification as spec_verify, with its
// workspace taken from a fixed buffer that lives inside this library (a
// file-scope __device__ array) instead of memory the caller allocates.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they verify -- a plain C host program that links only this library and owns
// no device allocator, or a serving loop whose device memory is planned once at
// start-up and which must not call an allocator inside its decode step.  The
// library's own path (spec_verify) already allocates nothing; this entry point
// removes the caller's workspace allocation as well.
//
// Limits and rules:
//   - one buffer of SV_NOALLOC_SCRATCH_BYTES per device; a batch whose
//     workspace (spec_verify_workspace_size) is larger gets SV_ERR_WORKSPACE
//     and nothing is enqueued;
//   - calls that can overlap on one device (two streams, two host threads
//     without ordering) share the buffer and race: order them on one stream or
//     with events;
//   - the buffer's address is looked up once per device with that device
//     current (cudaGetSymbolAddress); make the first call on each device before
//     any stream capture begins;
//   - nothing in the buffer has to start at zero: the first kernel of every call
//     writes every field that the later kernels read.
// No cudaMalloc / cudaFree or allocating library call is made here.
#include <cuda_runtime.h>

#include <mutex>

#include "sv_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];

// Device address of the current device's buffer, looked up on first use.
int noalloc_scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SV_OK;
}

}  // namespace

extern "C" {

int spec_verify_noalloc_scratch(void** scratch, size_t* bytes) {
  if (!scratch) return SV_ERR_ARG;
  if (int rc = noalloc_scratch_ptr(scratch)) return rc;
  if (bytes) *bytes = SV_NOALLOC_SCRATCH_BYTES;
  return SV_OK;
}

int spec_verify_noalloc(const sv_logits* target_logits, const sv_logits* draft_logits,
                        const int32_t* draft_tokens, const int32_t* k_per_req,
                        const float* temperature, const int32_t* top_k, const float* top_p,
                        const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                        void* stream, int32_t batch, const sv_options* options) {
  if (!target_logits || !draft_logits || batch < 0) return SV_ERR_ARG;
  const size_t need =
      spec_verify_workspace_size(batch, target_logits->rows, draft_logits->rows);
  if (need == 0) return SV_ERR_ARG;
  if (need > size_t(SV_NOALLOC_SCRATCH_BYTES)) return SV_ERR_WORKSPACE;
  void* ws = nullptr;
  if (int rc = noalloc_scratch_ptr(&ws)) return rc;
  return spec_verify(target_logits, draft_logits, draft_tokens, k_per_req, temperature, top_k,
                     top_p, uniforms, out_accept_len, out_tokens, stream, batch, ws,
                     SV_NOALLOC_SCRATCH_BYTES, options);
}

}  // extern "C"
