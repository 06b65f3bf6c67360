// Host side of the C ABI: argument validation, workspace layout, and the
// launches on the caller's stream: setup -> row pass over the rows not
// filtered by a kept-set threshold -> row pass over those -> filter / decide
// -> draw pass for verification; sampler setup -> the same two row passes ->
// sampler rows -> draw pass for the draft-side sampler.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>
#include <vector>

#include "sv_internal.cuh"

namespace sv {
cudaError_t rowpass_configure();
cudaError_t filter_occupancy(int* occ);
cudaError_t draw_configure();
cudaError_t draw_occupancy(int V, int* occ, int* occ_locate);
}  // namespace sv

using namespace sv;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  int sms = 0;
  int occ_filter = 1;  // resident filter / decide CTAs per SM
  int occ_draw = 1;    // resident draw CTAs per SM for vocabulary draw_v
  int occ_locate = 1;  // resident locate CTAs per SM for vocabulary draw_v
  int draw_v = -1;
  bool ready = false;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Per-device set-up: SM count, the kernels' shared-memory limits and the
// post-pass kernels' occupancy (the draw pass's depends on the vocabulary).
int prepare_device(int vocab, DeviceState* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev[dev].ready) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return SV_ERR_CUDA;
    int of = 1;
    if (rowpass_configure() != cudaSuccess || draw_configure() != cudaSuccess ||
        filter_occupancy(&of) != cudaSuccess)
      return SV_ERR_CUDA;
    g_dev[dev].sms = n;
    g_dev[dev].occ_filter = of;
    g_dev[dev].ready = true;
  }
  if (g_dev[dev].draw_v != vocab) {
    int od = 1, ol = 1;
    if (draw_occupancy(vocab, &od, &ol) != cudaSuccess) return SV_ERR_CUDA;
    g_dev[dev].occ_draw = od;
    g_dev[dev].occ_locate = ol;
    g_dev[dev].draw_v = vocab;
  }
  *out = g_dev[dev];
  return SV_OK;
}

bool misaligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

size_t elem_size(int dtype) { return dtype == SV_BF16 ? 2 : 4; }

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int32_t batch, int64_t target_rows, int64_t draft_rows) {
  if (batch < 0 || target_rows < 0 || draft_rows < 0 || target_rows + draft_rows >= INT_MAX)
    return 0;
  return ws_layout(batch, target_rows, draft_rows).total;
}

int spec_verify(const sv_logits* target_logits, const sv_logits* draft_logits,
                const int32_t* draft_tokens, const int32_t* k_per_req, const float* temperature,
                const int32_t* top_k, const float* top_p, const float* uniforms,
                int32_t* out_accept_len, int32_t* out_tokens, void* stream, int32_t batch,
                void* workspace, size_t workspace_bytes, const sv_options* options) {
  if (!target_logits || !draft_logits || batch < 0) return SV_ERR_ARG;
  const sv_logits& t = *target_logits;
  const sv_logits& d = *draft_logits;
  if (t.dtype != SV_F32 && t.dtype != SV_BF16) return SV_ERR_UNSUPPORTED;
  if (d.dtype != t.dtype) return SV_ERR_UNSUPPORTED;
  if (d.vocab != t.vocab || t.vocab < 1) return SV_ERR_ARG;
  if (t.vocab > SV_VOCAB_MAX) return SV_ERR_UNSUPPORTED;
  if (t.rows < 0 || d.rows < 0 || t.rows + d.rows >= INT_MAX) return SV_ERR_ARG;
  // sum_b (k_b + 1) = B + sum_b k_b, whatever the k_b are
  if (t.rows != int64_t(batch) + d.rows) return SV_ERR_ARG;
  const size_t es = elem_size(t.dtype);
  if (t.row_stride < t.vocab) return SV_ERR_ARG;
  if (d.data && d.rows > 0 && d.row_stride < d.vocab) return SV_ERR_ARG;
  if (batch > 0 && (!t.data || !k_per_req || !temperature || !uniforms || !out_accept_len ||
                    !out_tokens))
    return SV_ERR_ARG;
  if (d.rows > 0 && !draft_tokens) return SV_ERR_ARG;
  if (misaligned(t.data, 16) || (size_t(t.row_stride) * es) % 16 != 0) return SV_ERR_UNSUPPORTED;
  if (d.data && (misaligned(d.data, 16) || (size_t(d.row_stride) * es) % 16 != 0))
    return SV_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(batch, t.rows, d.rows);
  if (!workspace || misaligned(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;
  if (batch == 0) return SV_OK;

  DeviceState ds;
  if (int rc = prepare_device(t.vocab, &ds)) return rc;
  const int sms = ds.sms;

  Problem P{};
  P.target = t.data;
  P.draft = d.data;
  P.t_stride = t.row_stride;
  P.d_stride = d.data ? d.row_stride : 0;
  P.Rt = t.rows;
  P.Rd = d.rows;
  P.V = t.vocab;
  P.B = batch;
  P.draft_tokens = draft_tokens;
  P.k_per_req = k_per_req;
  P.temperature = temperature;
  P.top_k = top_k;
  P.top_p = top_p;
  P.uniforms = uniforms;
  P.out_accept_len = out_accept_len;
  P.out_tokens = out_tokens;
  P.out_pq = options ? options->out_pq : nullptr;
  P.out_q = nullptr;
  P.n_seg = 1;
  P.test_expire = options ? options->test_expire_wait : 0;
  P.inline_draw = t.vocab <= kInlineDrawV;
  P.ws = ws_bind(workspace, L);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_setup(P, s) != cudaSuccess) return SV_ERR_CUDA;
  const int64_t rows = t.rows + d.rows;
  const int64_t ctas = int64_t(sms) * kRowpassCtasPerSm;
  const int grid = int(rows < ctas ? rows : ctas);
  if (options && options->event_rowpass_begin &&
      cudaEventRecord(static_cast<cudaEvent_t>(options->event_rowpass_begin), s) != cudaSuccess)
    return SV_ERR_CUDA;
  // every row but those filtered by a kept-set threshold (top-p alone, large
  // top-k), then those: the second launch's CTAs become resident in the
  // first one's tail, so that it costs little when it has no rows; without
  // top_k and top_p arrays no row can need it, and it is not launched
  const bool threshold_rows = top_k != nullptr || top_p != nullptr;
  if (grid > 0 && (launch_rowpass(P, t.dtype == SV_BF16, false, grid, s) != cudaSuccess ||
                   (threshold_rows &&
                    launch_rowpass(P, t.dtype == SV_BF16, true, grid, s) != cudaSuccess)))
    return SV_ERR_CUDA;
  if (options && options->event_rowpass_end &&
      cudaEventRecord(static_cast<cudaEvent_t>(options->event_rowpass_end), s) != cudaSuccess)
    return SV_ERR_CUDA;
  const bool bf16 = t.dtype == SV_BF16;
  const int64_t fjobs = rows;  // at most one job per row
  const int64_t fmax = int64_t(sms) * ds.occ_filter;
  if (launch_filter_decide(P, bf16, int(fjobs < fmax ? fjobs : fmax), s) != cudaSuccess)
    return SV_ERR_CUDA;
  // short rows: every draw was taken by its decide job
  if (P.inline_draw) return SV_OK;
  // draw pass: a queued draw is cut into segments so that the units (draws x
  // segments) outnumber the resident CTAs about kDrawUnitsPerCta-fold and the
  // last round is short (at most one queued draw per request); then the
  // locate kernel, one CTA per queued draw
  const int64_t dmax = int64_t(sms) * ds.occ_draw;
  P.n_seg = int(std::max<int64_t>(
      1, std::min<int64_t>(kMaxSeg, (kDrawUnitsPerCta * dmax + batch - 1) / std::max(batch, 1))));
  const int64_t djobs = int64_t(batch) * P.n_seg;
  const int64_t lmax = int64_t(sms) * ds.occ_locate;
  if (launch_draw(P, bf16, int(djobs < dmax ? djobs : dmax), s) != cudaSuccess ||
      launch_locate(P, bf16, int(batch < lmax ? batch : lmax), s) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

size_t spec_draft_sample_workspace_size(int32_t batch, int64_t rows) {
  if (batch < 0 || rows < 0 || rows >= INT_MAX) return 0;
  return sample_ws_layout(batch, rows).total;
}

int spec_draft_sample(const sv_logits* draft_logits, const int32_t* k_per_req,
                      const float* temperature, const int32_t* top_k, const float* top_p,
                      const float* uniforms, int32_t* out_tokens, float* out_q, void* stream,
                      int32_t batch, void* workspace, size_t workspace_bytes,
                      const sv_options* options) {
  if (!draft_logits || batch < 0) return SV_ERR_ARG;
  const sv_logits& x = *draft_logits;
  if (x.dtype != SV_F32 && x.dtype != SV_BF16) return SV_ERR_UNSUPPORTED;
  if (x.vocab < 1) return SV_ERR_ARG;
  if (x.vocab > SV_VOCAB_MAX) return SV_ERR_UNSUPPORTED;
  if (x.rows < 0 || x.rows >= INT_MAX || x.row_stride < x.vocab) return SV_ERR_ARG;
  if (batch > 0 && (!k_per_req || !temperature)) return SV_ERR_ARG;
  if (x.rows > 0 && (!x.data || !uniforms || !out_tokens)) return SV_ERR_ARG;
  const size_t es = elem_size(x.dtype);
  if (x.data && (misaligned(x.data, 16) || (size_t(x.row_stride) * es) % 16 != 0))
    return SV_ERR_UNSUPPORTED;
  const WsLayout L = sample_ws_layout(batch, x.rows);
  if (!workspace || misaligned(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;
  if (batch == 0) return x.rows == 0 ? SV_OK : SV_ERR_ARG;

  DeviceState ds;
  if (int rc = prepare_device(x.vocab, &ds)) return rc;
  const int sms = ds.sms;

  Problem P{};
  P.target = x.data;
  P.draft = nullptr;
  P.t_stride = x.row_stride;
  P.d_stride = 0;
  P.Rt = x.rows;  // the drafter rows play the part of target rows in the row pass
  P.Rd = 0;
  P.V = x.vocab;
  P.B = batch;
  P.n_seg = 1;
  P.draft_tokens = nullptr;
  P.k_per_req = k_per_req;
  P.temperature = temperature;
  P.top_k = top_k;
  P.top_p = top_p;
  P.uniforms = uniforms;
  P.out_accept_len = nullptr;
  P.out_tokens = out_tokens;
  P.out_pq = nullptr;
  P.out_q = out_q;
  P.test_expire = 0;
  P.ws = ws_bind(workspace, L);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_sample_setup(P, s) != cudaSuccess) return SV_ERR_CUDA;
  const int64_t rows = x.rows;
  if (rows == 0) return SV_OK;
  const bool bf16 = x.dtype == SV_BF16;
  const int64_t ctas = int64_t(sms) * kRowpassCtasPerSm;
  if (options && options->event_rowpass_begin &&
      cudaEventRecord(static_cast<cudaEvent_t>(options->event_rowpass_begin), s) != cudaSuccess)
    return SV_ERR_CUDA;
  const bool threshold_rows = top_k != nullptr || top_p != nullptr;
  if (launch_rowpass(P, bf16, false, int(rows < ctas ? rows : ctas), s) != cudaSuccess ||
      (threshold_rows &&
       launch_rowpass(P, bf16, true, int(rows < ctas ? rows : ctas), s) != cudaSuccess))
    return SV_ERR_CUDA;
  if (options && options->event_rowpass_end &&
      cudaEventRecord(static_cast<cudaEvent_t>(options->event_rowpass_end), s) != cudaSuccess)
    return SV_ERR_CUDA;
  const int64_t fmax = int64_t(sms) * ds.occ_filter;
  if (launch_sample_post(P, bf16, int(rows < fmax ? rows : fmax), s) != cudaSuccess)
    return SV_ERR_CUDA;
  // every sampled unfiltered row may queue a draw
  const int64_t dmax = int64_t(sms) * ds.occ_draw;
  P.n_seg = int(std::max<int64_t>(
      1, std::min<int64_t>(kMaxSeg, (kDrawUnitsPerCta * dmax + rows - 1) / rows)));
  const int64_t djobs = rows * P.n_seg;
  const int64_t lmax = int64_t(sms) * ds.occ_locate;
  if (launch_draw(P, bf16, int(djobs < dmax ? djobs : dmax), s) != cudaSuccess ||
      launch_locate(P, bf16, int(rows < lmax ? rows : lmax), s) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

size_t spec_kv_commit_workspace_size(int32_t batch) {
  return batch < 0 ? 0 : kv_workspace_bytes(batch);
}

int spec_kv_commit(const sv_kv_cache* cache, const void* spec, int32_t spec_slots,
                   const int32_t* accept_len, const int32_t* k_per_req, int32_t* kv_len,
                   const int32_t* block_table, int32_t max_pages, void* stream, int32_t batch,
                   void* workspace, size_t workspace_bytes) {
  if (!cache || batch < 0 || spec_slots < 1 || max_pages < 0) return SV_ERR_ARG;
  const sv_kv_cache& c = *cache;
  if (c.num_pages < 0 || c.n_layers < 1 || c.page_size < 1 || c.entry_elems < 1 ||
      (c.elem_bytes != 2 && c.elem_bytes != 4))
    return SV_ERR_ARG;
  const int64_t entry_bytes = int64_t(c.entry_elems) * c.elem_bytes;
  if (entry_bytes % 16 != 0) return SV_ERR_UNSUPPORTED;
  if (!workspace || misaligned(workspace, 256) || workspace_bytes < kv_workspace_bytes(batch))
    return SV_ERR_WORKSPACE;
  if (batch == 0) return SV_OK;
  if (!c.data || !spec || !accept_len || !k_per_req || !kv_len || (max_pages > 0 && !block_table))
    return SV_ERR_ARG;
  if (misaligned(c.data, 16) || misaligned(spec, 16)) return SV_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SV_ERR_CUDA;
  if (launch_kv_commit(c.data, spec, c.num_pages, c.n_layers, c.page_size, entry_bytes,
                       spec_slots, accept_len, k_per_req, kv_len, block_table, max_pages, batch,
                       workspace, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

size_t spec_lmhead_stats_workspace_size(int32_t rows, int32_t vocab) {
  if (rows < 0 || vocab < 1) return 0;
  return lmhead_workspace_bytes(rows, vocab);
}

int spec_lmhead_stats(const void* hidden, const void* unembed, int32_t rows, int32_t vocab,
                      int32_t d, const float* temperature, const int32_t* tokens,
                      float* out_max, double* out_sum, int32_t* out_argmax, float* out_token,
                      void* stream, void* workspace, size_t workspace_bytes) {
  if (rows < 0 || vocab < 1 || d < 1) return SV_ERR_ARG;
  if (d % 8 != 0) return SV_ERR_UNSUPPORTED;
  if (!workspace || misaligned(workspace, 256) ||
      workspace_bytes < lmhead_workspace_bytes(rows, vocab))
    return SV_ERR_WORKSPACE;
  if (rows == 0) return SV_OK;
  if (!hidden || !unembed || !temperature || !out_max || !out_sum || !out_argmax || !out_token)
    return SV_ERR_ARG;
  if (misaligned(hidden, 16) || misaligned(unembed, 16)) return SV_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SV_ERR_CUDA;
  return launch_lmhead_stats(hidden, unembed, rows, vocab, d, temperature, tokens, out_max,
                             out_sum, out_argmax, out_token, workspace, sms,
                             static_cast<cudaStream_t>(stream));
}

int spec_adapt_k(const int32_t* accept_len, const int32_t* k_used, double* succ, double* fail,
                 double decay, double c, int32_t k_min, int32_t k_max, int32_t* k_next,
                 float* alpha, void* stream, int32_t batch) {
  if (batch < 0 || k_min < 0 || k_max < k_min || k_max > SV_MAX_K || !(decay >= 0.0) ||
      !(decay <= 1.0) || !(c >= 0.0))
    return SV_ERR_ARG;
  if (batch == 0) return SV_OK;
  if (!accept_len || !k_used || !succ || !fail || !k_next) return SV_ERR_ARG;
  return launch_adapt_k(accept_len, k_used, succ, fail, decay, c, k_min, k_max, k_next, alpha,
                        batch, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

size_t spec_verify_greedy_workspace_size(void) { return align256(sizeof(WsHeader)); }

int spec_verify_greedy_from_argmax(const int32_t* target_argmax, const int32_t* draft_tokens,
                                   const int32_t* k_per_req, int32_t* out_accept_len,
                                   int32_t* out_tokens, void* stream, int32_t batch,
                                   int64_t target_rows, int32_t vocab, void* workspace,
                                   size_t workspace_bytes) {
  if (batch < 0 || target_rows < 0 || vocab < 1 || target_rows >= INT_MAX) return SV_ERR_ARG;
  if (target_rows < int64_t(batch)) return SV_ERR_ARG;
  if (!workspace || misaligned(workspace, 256) || workspace_bytes < sizeof(WsHeader))
    return SV_ERR_WORKSPACE;
  if (batch == 0) return SV_OK;
  if (!target_argmax || !k_per_req || !out_accept_len || !out_tokens) return SV_ERR_ARG;
  if (target_rows > int64_t(batch) && !draft_tokens) return SV_ERR_ARG;
  return launch_greedy_from_argmax(target_argmax, draft_tokens, k_per_req, out_accept_len,
                                   out_tokens, batch, target_rows, vocab, workspace,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

int spec_verify_get_error(const void* workspace, void* stream, int32_t* code, int32_t* request,
                          int64_t* row) {
  if (!workspace || !code) return SV_ERR_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SV_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SV_ERR_CUDA;
  *code = h.err_code;
  if (request) *request = h.err_req;
  if (row) *row = h.err_row;
  return SV_OK;
}

int spec_verify_dump_rows(const void* workspace, size_t workspace_bytes, int32_t batch,
                          int64_t target_rows, int64_t draft_rows, void* stream, double* stats,
                          int32_t* kept_count, int32_t* kept_idx, double* kept_p) {
  if (!workspace || batch < 0 || target_rows < 0 || draft_rows < 0) return SV_ERR_ARG;
  const WsLayout L = ws_layout(batch, target_rows, draft_rows);
  if (workspace_bytes < L.total) return SV_ERR_WORKSPACE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SV_ERR_CUDA;
  const char* base = static_cast<const char*>(workspace);
  const size_t R = size_t(target_rows + draft_rows);
  if (R == 0) return SV_OK;
  if (stats || kept_count) {
    std::vector<RowStat> st(R);
    if (cudaMemcpy(st.data(), base + L.off_stats, R * sizeof(RowStat), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
      return SV_ERR_CUDA;
    // the kept-set thresholds of kBig rows (slot 0 of each row's survivors)
    std::vector<uint64_t> th(R, 0ull);
    for (size_t r = 0; r < R; ++r)
      if (st[r].mode == kBig &&
          cudaMemcpy(&th[r], base + L.off_raw + r * kRawCap * sizeof(uint64_t), sizeof(uint64_t),
                     cudaMemcpyDeviceToHost) != cudaSuccess)
        return SV_ERR_CUDA;
    for (size_t r = 0; r < R; ++r) {
      if (stats) {
        stats[5 * r + 0] = st[r].m;
        stats[5 * r + 1] = st[r].s;
        stats[5 * r + 2] = st[r].pg;
        stats[5 * r + 3] = st[r].arg;
        // the last kept token of a threshold-filtered row: ~ the key's low word
        stats[5 * r + 4] = st[r].mode == kBig ? double(int32_t(~uint32_t(th[r]))) : -1.0;
      }
      if (kept_count) kept_count[r] = (st[r].mode == kTopk || st[r].mode == kBig) ? st[r].kept : 0;
    }
  }
  if (kept_idx && cudaMemcpy(kept_idx, base + L.off_cidx, R * kTopkMax * sizeof(int32_t),
                             cudaMemcpyDeviceToHost) != cudaSuccess)
    return SV_ERR_CUDA;
  if (kept_p) {
    std::vector<float> kp(R * kTopkMax);
    if (cudaMemcpy(kp.data(), base + L.off_cp, R * kTopkMax * sizeof(float),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
      return SV_ERR_CUDA;
    for (size_t i = 0; i < kp.size(); ++i) kept_p[i] = kp[i];
  }
  return SV_OK;
}

const char* spec_verify_strerror(int code) {
  switch (code) {
    case SV_OK: return "ok";
    case SV_ERR_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported dtype, vocabulary size, alignment or stride";
    case SV_ERR_CUDA: return "CUDA runtime error";
    case SV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SV_ERR_DATA_K: return "k_per_req outside [0, SV_MAX_K]";
    case SV_ERR_DATA_TEMPERATURE: return "temperature negative, NaN or infinite";
    case SV_ERR_DATA_TOP_P: return "top_p outside (0, 1]";
    case SV_ERR_DATA_TOP_K: return "top_k negative";
    case SV_ERR_DATA_TOKEN: return "draft token outside [0, V)";
    case SV_ERR_DATA_ROWS: return "row counts do not match k_per_req";
    case SV_ERR_DATA_LOGIT: return "NaN or +inf logit, or a sampled row without a finite logit";
    case SV_ERR_DATA_NO_DRAFT: return "temperature > 0 without draft logits";
    case SV_ERR_TIMEOUT: return "internal bounded wait expired";
    case SV_ERR_INTERNAL: return "internal capacity invariant failed";
    case SV_ERR_DATA_ACCEPT: return "KV commit: accept length above k";
    case SV_ERR_DATA_PAGE: return "KV commit: destination page missing or negative kv_len";
    default: return "unknown status";
  }
}

int spec_verify_version(void) { return 100; }

}  // extern "C"
