// Speculative-decoding verification oracle (and the draft-side sampler that
// produces the drafted tokens it verifies).
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
// statement of what batched speculative-decoding verification computes.  It is
// single-threaded, works in IEEE double precision and shares no code, header,
// table or helper with the CUDA library under
// speculative_decoding_verification_13_gb300/.  Only tests/, the smoke check in
// __graft_entry__.py and bench.py's CPU-baseline / reference arm may load it;
// the product path never does.
//
// Sources (page title, then section):
//   [FM]  "FlashMap: Flow Map Speculative Decoding and the Mathematical
//         Elimination of Suffix Decay", §4 "The Rejection Sampling Invariant"
//         (steps 1-3 and the identity P(Y=y) = p(y)), §5 draft_block step 5
//         (logits / temperature, softmax; argmax at temperature 0).
//   [DF]  "DFlash", §4 (target yields p_1..p_{gamma+1} in one pass; greedy mode
//         accepts the longest matching prefix; sampling accepts x_k with
//         probability min(1, p_k(x_k)/q_k(x_k)) and on rejection samples the
//         normalised residual max(0, p_k - q_k)).
//   [SD]  "Speculative decoding and multi-token prediction", sections
//         "Draft and verify" (k+1 distributions; stop at the first
//         disagreement and emit the target's own token; even a full rejection
//         advances one token), "Why the output is identical" (acceptance
//         min(1, p/q); residual = positive part of p - q; top-k / top-p applied
//         identically to both distributions).
//
// Readings where the pages leave a step open:
//   R1  accept iff u < p/q (the pages write r <= min(1, p/q); the two differ on
//       a set of measure zero; with u in [0,1) this never accepts p = 0 and
//       always accepts p >= q).
//   R2  the final (residual or bonus) draw uses the extra uniform u_k, never
//       the u_L that caused the rejection.
//   R3  inverse CDF in vocabulary-index order: y* = min{ y : C_y > u * S },
//       C the inclusive prefix sum of the (unnormalised) residual weights.
//   R4  temperature first, then top-k, then top-p on the top-k-renormalised
//       distribution; the sort order is (logit descending, index ascending);
//       token j survives top-p iff the cumulative probability of the tokens
//       before it is < top_p (the crossing token is kept); top_p >= 1 and
//       top_k in {0} U [V, inf) switch the respective filter off.
//   R5  residual mass S == 0 (only possible through rounding) falls back to p.
//   R6  if rounding leaves u * S >= C_{V-1}, the last token with positive
//       weight is emitted.
//   R7  the exponent of every softmax is evaluated as (x - x_max) / T (one
//       subtraction that is exact for the input formats, one division), which
//       equals z - z_max with z = x / T in exact arithmetic.
//   R8  temperature 0 is greedy: argmax of the raw target logits, lowest index
//       on ties; draft logits are never read.
//
// Margins returned per request (used to decide which sampled outputs a
// floating-point implementation may legitimately round differently):
//   m_acc  = min over evaluated positions of |u_i - ratio_i|,
//   m_cdf  = min(C_{y*} - t, t - C_{y*-1}) / S   with t = u_k * S,
//   m_topp = min over filtered rows of |cum_before_j - top_p| over the
//            evaluated top-p decisions.
// Each is +inf where no such decision was taken.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <vector>

namespace {

enum { DT_F32 = 0, DT_BF16 = 1, DT_F64 = 2 };

enum {
  OR_OK = 0,
  OR_ERR_ARG = 1,
  OR_ERR_ROWS = 21,
};

// Per-request data errors (reported through accept_len = -1).
enum {
  REQ_OK = 0,
  REQ_BAD_K = 16,
  REQ_BAD_TEMP = 17,
  REQ_BAD_TOPP = 18,
  REQ_BAD_TOPK = 19,
  REQ_BAD_TOKEN = 20,
  REQ_BAD_LOGIT = 22,
};

const double kInf = std::numeric_limits<double>::infinity();
const int kMaxK = 32;

double load_logit(const void* base, int dtype, int64_t off) {
  if (dtype == DT_F32) return (double)static_cast<const float*>(base)[off];
  if (dtype == DT_F64) return static_cast<const double*>(base)[off];
  // bf16: the upper 16 bits of an IEEE binary32 value.
  uint32_t bits = (uint32_t)static_cast<const uint16_t*>(base)[off] << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return (double)f;
}

std::vector<double> load_row(const void* base, int dtype, int64_t row, int64_t stride, int V) {
  std::vector<double> x(V);
  for (int y = 0; y < V; ++y) x[y] = load_logit(base, dtype, row * stride + y);
  return x;
}

// NaN or +inf anywhere is a data error in every mode.
bool row_has_bad_value(const std::vector<double>& x) {
  for (double v : x)
    if (std::isnan(v) || v == kInf) return true;
  return false;
}

// Greedy token (R8, [FM] §5 step 5, [DF] §4 step 5): first index of the maximum.
int argmax_first(const std::vector<double>& x) {
  int best = 0;
  for (int y = 1; y < (int)x.size(); ++y)
    if (x[y] > x[best]) best = y;
  return best;
}

bool filter_active(int V, int top_k, double top_p) {
  return (top_k > 0 && top_k < V) || top_p < 1.0;
}

// Probability distribution of one row at temperature T > 0 with the optional
// top-k / top-p filter (reading R4, R7).  Returns false when the row has no
// finite logit (no distribution exists).  *topp_margin receives the smallest
// |cum_before - top_p| over the top-p decisions that were taken.
bool row_distribution(const std::vector<double>& x, double T, int top_k, double top_p,
                      std::vector<double>& p, double* topp_margin) {
  const int V = (int)x.size();
  p.assign(V, 0.0);
  *topp_margin = kInf;
  const int imax = argmax_first(x);
  const double xmax = x[imax];
  if (xmax == -kInf) return false;

  if (!filter_active(V, top_k, top_p)) {
    // Plain softmax of x / T, normaliser summed in index order.
    double W = 0.0;
    for (int y = 0; y < V; ++y) {
      p[y] = std::exp((x[y] - xmax) / T);
      W += p[y];
    }
    for (int y = 0; y < V; ++y) p[y] /= W;
    return true;
  }

  // Order of the vocabulary: logit descending, index ascending (equals the
  // order of x / T for T > 0).
  const int K = (top_k > 0 && top_k < V) ? top_k : V;
  std::vector<int> order(V);
  std::iota(order.begin(), order.end(), 0);
  auto before = [&](int a, int b) { return x[a] > x[b] || (x[a] == x[b] && a < b); };
  if (K < V)
    std::partial_sort(order.begin(), order.begin() + K, order.end(), before);
  else
    std::sort(order.begin(), order.end(), before);

  // Softmax over the top-k survivors; sums in that order.
  std::vector<double> w(K);
  double W = 0.0;
  for (int j = 0; j < K; ++j) {
    w[j] = std::exp((x[order[j]] - xmax) / T);
    W += w[j];
  }
  // Top-p on the top-k-renormalised distribution: keep j iff the cumulative
  // probability of the tokens before it is < top_p.
  int Kp = K;
  if (top_p < 1.0) {
    double cum = 0.0;
    Kp = 0;
    for (int j = 0; j < K; ++j) {
      *topp_margin = std::min(*topp_margin, std::fabs(cum - top_p));
      if (!(cum < top_p)) break;
      Kp = j + 1;
      cum += w[j] / W;
    }
  }
  // Renormalise over the final kept set (sum in the same order).
  double Wp = 0.0;
  for (int j = 0; j < Kp; ++j) Wp += w[j];
  for (int j = 0; j < Kp; ++j) p[order[j]] = w[j] / Wp;
  return true;
}

struct Margins {
  double acc = kInf, cdf = kInf, topp = kInf;
};

// Inverse-CDF draw over non-negative weights r in index order (R3, R6).
int inverse_cdf(const std::vector<double>& r, double u, double* margin) {
  double S = 0.0;
  for (double v : r) S += v;
  const double t = u * S;
  double C = 0.0, Cprev = 0.0;
  for (int y = 0; y < (int)r.size(); ++y) {
    Cprev = C;
    C += r[y];
    if (C > t) {
      *margin = std::min(C - t, t - Cprev) / S;
      return y;
    }
  }
  *margin = 0.0;
  int last = -1;
  for (int y = 0; y < (int)r.size(); ++y)
    if (r[y] > 0.0) last = y;
  return last;
}

// The rejection rule for one request whose distributions are known.
//   p[i], i = 0..k : target distributions after 0..k drafted tokens
//   q[i], i = 0..k-1 : draft distributions
//   x[i] : drafted tokens, u[i], i = 0..k : uniforms (u[k] drives the final draw)
// [FM] §4 steps 1-3, [DF] §4, [SD] "Draft and verify" / "Why the output is identical".
int verify_sampled(int k, const std::vector<std::vector<double>>& p,
                   const std::vector<std::vector<double>>& q, const int32_t* x,
                   const float* u, int32_t* tokens, double* pq, Margins* mg) {
  int L = k;
  for (int i = 0; i < k; ++i) {
    const double pi = p[i][x[i]], qi = q[i][x[i]];
    if (pq) {
      pq[2 * i] = pi;
      pq[2 * i + 1] = qi;
    }
    if (i > L) continue;  // the probabilities are still reported for parity checks
    const double ratio = pi / qi;  // IEEE: q = 0 < p gives +inf (accept), p = q = 0 gives NaN (reject)
    const double ui = (double)u[i];
    if (std::isfinite(ratio)) mg->acc = std::min(mg->acc, std::fabs(ui - ratio));
    if (!(ui < ratio) && L == k) L = i;
  }
  std::vector<double> r;
  if (L < k) {
    // Rejection at L: normalised positive part of p_L - q_L.
    const int V = (int)p[L].size();
    r.resize(V);
    double S = 0.0;
    for (int y = 0; y < V; ++y) {
      r[y] = std::max(0.0, p[L][y] - q[L][y]);
      S += r[y];
    }
    if (!(S > 0.0)) r = p[L];  // R5
  } else {
    // Every draft accepted: bonus token from the target's distribution after all k.
    r = p[k];
  }
  double mcdf = kInf;
  const int ystar = inverse_cdf(r, (double)u[k], &mcdf);
  mg->cdf = mcdf;
  for (int i = 0; i < L; ++i) tokens[i] = x[i];
  tokens[L] = ystar;
  for (int i = L + 1; i <= k; ++i) tokens[i] = -1;
  return L;
}

int verify_greedy(int k, const std::vector<int>& g, const int32_t* x, int32_t* tokens) {
  int L = k;
  for (int i = 0; i < k; ++i)
    if (x[i] != g[i]) {
      L = i;
      break;
    }
  for (int i = 0; i < L; ++i) tokens[i] = x[i];
  tokens[L] = g[L];
  for (int i = L + 1; i <= k; ++i) tokens[i] = -1;
  return L;
}

int check_params(int k, float T, int top_k, float top_p) {
  if (k < 0 || k > kMaxK) return REQ_BAD_K;
  if (!(T >= 0.0f) || std::isinf(T)) return REQ_BAD_TEMP;
  if (!(top_p > 0.0f && top_p <= 1.0f)) return REQ_BAD_TOPP;
  if (top_k < 0) return REQ_BAD_TOPK;
  return REQ_OK;
}

// One request, rows given as base pointers of its own block of rows.
int run_request(int V, int dtype, const void* trows, int64_t t_stride, const void* drows,
                int64_t d_stride, int k, float T, int top_k, float top_p, const int32_t* x,
                const float* u, int32_t* tokens, double* pq, Margins* mg) {
  for (int i = 0; i < k; ++i)
    if (x[i] < 0 || x[i] >= V) return -REQ_BAD_TOKEN;
  if (T == 0.0f) {
    std::vector<int> g(k + 1);
    for (int i = 0; i <= k; ++i) {
      std::vector<double> xr = load_row(trows, dtype, i, t_stride, V);
      if (row_has_bad_value(xr)) return -REQ_BAD_LOGIT;
      g[i] = argmax_first(xr);
    }
    return verify_greedy(k, g, x, tokens);
  }
  const double Td = (double)T, tp = (double)top_p;
  std::vector<std::vector<double>> p(k + 1), q(k);
  for (int i = 0; i <= k; ++i) {
    std::vector<double> xr = load_row(trows, dtype, i, t_stride, V);
    double m;
    if (row_has_bad_value(xr) || !row_distribution(xr, Td, top_k, tp, p[i], &m))
      return -REQ_BAD_LOGIT;
    mg->topp = std::min(mg->topp, m);
  }
  for (int i = 0; i < k; ++i) {
    std::vector<double> xr = load_row(drows, dtype, i, d_stride, V);
    double m;
    if (row_has_bad_value(xr) || !row_distribution(xr, Td, top_k, tp, q[i], &m))
      return -REQ_BAD_LOGIT;
    mg->topp = std::min(mg->topp, m);
  }
  return verify_sampled(k, p, q, x, u, tokens, pq, mg);
}

size_t elem_size(int dtype) { return dtype == DT_F32 ? 4 : dtype == DT_BF16 ? 2 : 8; }

}  // namespace

extern "C" {

// Whole batch.  Request b owns target rows t_off[b] .. t_off[b] + k_b with
// t_off[b] = sum_{j<b} (k_j + 1), and draft rows t_off[b] - b .. t_off[b] - b + k_b - 1.
// uniforms / out_tokens are indexed like target rows.  out_pq is [draft_rows, 2]
// (may be NULL), out_margins [batch, 3] (may be NULL).  Per-request data errors
// give accept_len = -1 and tokens = -1.  Returns 0, or a batch-level error.
int oracle_verify(int32_t batch, int32_t vocab, int32_t dtype, const void* target,
                  int64_t t_rows, int64_t t_stride, const void* draft, int64_t d_rows,
                  int64_t d_stride, const int32_t* draft_tokens, const int32_t* k_per_req,
                  const float* temperature, const int32_t* top_k, const float* top_p,
                  const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                  double* out_pq, double* out_margins) {
  if (batch < 0 || vocab < 1 || (dtype != DT_F32 && dtype != DT_BF16 && dtype != DT_F64) ||
      !target || !k_per_req || !temperature || !uniforms || !out_accept_len || !out_tokens)
    return OR_ERR_ARG;
  int64_t rt = 0, rd = 0;
  for (int b = 0; b < batch; ++b) {
    if (k_per_req[b] < 0 || k_per_req[b] > kMaxK) {
      rt = -1;
      break;
    }
    rt += k_per_req[b] + 1;
    rd += k_per_req[b];
  }
  if (rt != t_rows || rd != d_rows) {
    for (int b = 0; b < batch; ++b) out_accept_len[b] = -1;
    for (int64_t r = 0; r < t_rows; ++r) out_tokens[r] = -1;
    return OR_ERR_ROWS;
  }
  const size_t es = elem_size(dtype);
  int64_t t0 = 0;
  for (int b = 0; b < batch; ++b) {
    const int k = k_per_req[b];
    const int64_t d0 = t0 - b;
    const float T = temperature[b];
    const int tk = top_k ? top_k[b] : 0;
    const float tp = top_p ? top_p[b] : 1.0f;
    Margins mg;
    int rc = check_params(k, T, tk, tp);
    if (rc == REQ_OK && T > 0.0f && !draft && k > 0) rc = REQ_BAD_LOGIT;
    int L = -1;
    if (rc == REQ_OK) {
      const void* trows = static_cast<const char*>(target) + (size_t)(t0 * t_stride) * es;
      const void* drows =
          draft ? static_cast<const char*>(draft) + (size_t)(d0 * d_stride) * es : nullptr;
      L = run_request(vocab, dtype, trows, t_stride, drows, d_stride, k, T, tk, tp,
                      draft_tokens + d0, uniforms + t0, out_tokens + t0,
                      out_pq ? out_pq + 2 * d0 : nullptr, &mg);
    }
    if (L < 0) {
      out_accept_len[b] = -1;
      for (int i = 0; i <= k; ++i) out_tokens[t0 + i] = -1;
      if (out_pq)
        for (int i = 0; i < 2 * k; ++i) out_pq[2 * d0 + i] = std::nan("");
      if (out_margins)
        for (int j = 0; j < 3; ++j) out_margins[3 * b + j] = std::nan("");
    } else {
      out_accept_len[b] = L;
      if (out_pq && T == 0.0f)
        for (int i = 0; i < 2 * k; ++i) out_pq[2 * d0 + i] = std::nan("");
      if (out_margins) {
        out_margins[3 * b + 0] = mg.acc;
        out_margins[3 * b + 1] = mg.cdf;
        out_margins[3 * b + 2] = mg.topp;
      }
    }
    t0 += k + 1;
  }
  return OR_OK;
}

// One request's rows verified against many independent (draft tokens, uniforms)
// trials; the distributions are built once.  target: [k+1, V] contiguous,
// draft: [k, V] contiguous.  draft_tokens [n, k], uniforms [n, k+1],
// out_accept_len [n], out_tokens [n, k+1], out_margins [n, 3] (may be NULL).
int oracle_verify_trials(int32_t vocab, int32_t dtype, int32_t k, const void* target,
                         const void* draft, float temperature, int32_t top_k, float top_p,
                         int64_t n_trials, const int32_t* draft_tokens, const float* uniforms,
                         int32_t* out_accept_len, int32_t* out_tokens, double* out_margins) {
  if (vocab < 1 || !target || n_trials < 0 || !draft_tokens || !uniforms || !out_accept_len ||
      !out_tokens)
    return OR_ERR_ARG;
  int rc = check_params(k, temperature, top_k, top_p);
  if (rc != REQ_OK) return rc;
  const int V = vocab;
  const double Td = (double)temperature, tp = (double)top_p;
  std::vector<std::vector<double>> p(k + 1), q(k);
  std::vector<int> g(k + 1);
  double mtopp = kInf;
  for (int i = 0; i <= k; ++i) {
    std::vector<double> xr = load_row(target, dtype, i, V, V);
    if (row_has_bad_value(xr)) return REQ_BAD_LOGIT;
    g[i] = argmax_first(xr);
    double m;
    if (temperature > 0.0f) {
      if (!row_distribution(xr, Td, top_k, tp, p[i], &m)) return REQ_BAD_LOGIT;
      mtopp = std::min(mtopp, m);
    }
  }
  if (temperature > 0.0f) {
    if (!draft && k > 0) return OR_ERR_ARG;
    for (int i = 0; i < k; ++i) {
      std::vector<double> xr = load_row(draft, dtype, i, V, V);
      double m;
      if (row_has_bad_value(xr) || !row_distribution(xr, Td, top_k, tp, q[i], &m))
        return REQ_BAD_LOGIT;
      mtopp = std::min(mtopp, m);
    }
  }
  for (int64_t n = 0; n < n_trials; ++n) {
    const int32_t* x = draft_tokens + n * k;
    int32_t* tok = out_tokens + n * (k + 1);
    bool bad = false;
    for (int i = 0; i < k; ++i)
      if (x[i] < 0 || x[i] >= V) bad = true;
    Margins mg;
    mg.topp = mtopp;
    int L;
    if (bad) {
      L = -1;
      for (int i = 0; i <= k; ++i) tok[i] = -1;
    } else if (temperature == 0.0f) {
      L = verify_greedy(k, g, x, tok);
    } else {
      L = verify_sampled(k, p, q, x, uniforms + n * (k + 1), tok, nullptr, &mg);
    }
    out_accept_len[n] = L;
    if (out_margins) {
      out_margins[3 * n + 0] = mg.acc;
      out_margins[3 * n + 1] = mg.cdf;
      out_margins[3 * n + 2] = mg.topp;
    }
  }
  return OR_OK;
}

// Distribution of one row (length V) at temperature T with the optional filter.
// T == 0 returns the one-hot distribution of the greedy token.  Returns 0, or a
// data-error code (NaN / +inf, or no finite logit at T > 0).
int oracle_row_probs(int32_t vocab, int32_t dtype, const void* row, float temperature,
                     int32_t top_k, float top_p, double* out_p, double* out_topp_margin) {
  if (vocab < 1 || !row || !out_p) return OR_ERR_ARG;
  int rc = check_params(0, temperature, top_k, top_p);
  if (rc != REQ_OK) return rc;
  std::vector<double> x = load_row(row, dtype, 0, vocab, vocab);
  if (row_has_bad_value(x)) return REQ_BAD_LOGIT;
  std::vector<double> p;
  double m = kInf;
  if (temperature == 0.0f) {
    p.assign(vocab, 0.0);
    p[argmax_first(x)] = 1.0;
  } else if (!row_distribution(x, (double)temperature, top_k, (double)top_p, p, &m)) {
    return REQ_BAD_LOGIT;
  }
  std::copy(p.begin(), p.end(), out_p);
  if (out_topp_margin) *out_topp_margin = m;
  return OR_OK;
}

// Draft-side sampling ([FM] §5 draft_block step 5: logits / temperature,
// softmax, a multinomial draw; argmax at temperature 0), for a batch laid out
// like the verifier's draft rows: request b owns rows d_off[b] .. d_off[b] +
// k_b - 1 with d_off[b] = sum_{j<b} k_j.  Row i of request b draws
//   x_i = min{ y : C_y > u_i * S }  (reading R3; S = sum of the row's p)
// from the row's distribution at the request's temperature with its top-k /
// top-p filter (R4, R7), or takes the argmax of the raw logits, lowest index on
// ties, at temperature 0 (R8).  u_i = uniforms[d_off[b] + i].
//   out_tokens [rows]: x_i, -1 for every row of a request with a data error
//   out_q      [rows] (may be NULL): q_i(x_i), NaN for greedy and failed rows
//   out_margins [rows, 2] (may be NULL): (m_cdf, m_topp) of the row, +inf
//              where no such decision was taken, NaN for failed rows
// Returns 0, or a batch-level error (the row count does not match sum k_b;
// every token is then -1).
int oracle_draft_sample(int32_t batch, int32_t vocab, int32_t dtype, const void* logits,
                        int64_t rows, int64_t stride, const int32_t* k_per_req,
                        const float* temperature, const int32_t* top_k, const float* top_p,
                        const float* uniforms, int32_t* out_tokens, double* out_q,
                        double* out_margins) {
  if (batch < 0 || vocab < 1 || (dtype != DT_F32 && dtype != DT_BF16 && dtype != DT_F64) ||
      (rows > 0 && !logits) || !k_per_req || !temperature || (rows > 0 && !uniforms) ||
      (rows > 0 && !out_tokens))
    return OR_ERR_ARG;
  int64_t total = 0;
  for (int b = 0; b < batch; ++b) {
    if (k_per_req[b] < 0 || k_per_req[b] > kMaxK) {
      total = -1;
      break;
    }
    total += k_per_req[b];
  }
  const double nan = std::nan("");
  auto fail_rows = [&](int64_t r0, int64_t n) {
    for (int64_t r = r0; r < r0 + n; ++r) {
      out_tokens[r] = -1;
      if (out_q) out_q[r] = nan;
      if (out_margins) out_margins[2 * r] = out_margins[2 * r + 1] = nan;
    }
  };
  if (total != rows) {
    fail_rows(0, rows);
    return OR_ERR_ROWS;
  }
  int64_t d0 = 0;
  for (int b = 0; b < batch; ++b) {
    const int k = k_per_req[b];
    const float T = temperature[b];
    const int tk = top_k ? top_k[b] : 0;
    const float tp = top_p ? top_p[b] : 1.0f;
    bool ok = check_params(k, T, tk, tp) == REQ_OK;
    std::vector<int32_t> tok(k);
    std::vector<double> q(k, nan), mc(k, kInf), mt(k, kInf);
    for (int i = 0; ok && i < k; ++i) {
      std::vector<double> x = load_row(logits, dtype, d0 + i, stride, vocab);
      if (row_has_bad_value(x)) {
        ok = false;
        break;
      }
      if (T == 0.0f) {
        tok[i] = argmax_first(x);
        continue;
      }
      std::vector<double> p;
      if (!row_distribution(x, (double)T, tk, (double)tp, p, &mt[i])) {
        ok = false;
        break;
      }
      tok[i] = inverse_cdf(p, (double)uniforms[d0 + i], &mc[i]);
      q[i] = p[tok[i]];
    }
    if (!ok) {
      fail_rows(d0, k);
    } else {
      for (int i = 0; i < k; ++i) {
        out_tokens[d0 + i] = tok[i];
        if (out_q) out_q[d0 + i] = q[i];
        if (out_margins) {
          out_margins[2 * (d0 + i)] = mc[i];
          out_margins[2 * (d0 + i) + 1] = mt[i];
        }
      }
    }
    d0 += k;
  }
  return OR_OK;
}

// Greedy token of one row; -1 for a row holding NaN or +inf.
int32_t oracle_argmax(int32_t vocab, int32_t dtype, const void* row) {
  if (vocab < 1 || !row) return -1;
  std::vector<double> x = load_row(row, dtype, 0, vocab, vocab);
  if (row_has_bad_value(x)) return -1;
  return argmax_first(x);
}

}  // extern "C"
