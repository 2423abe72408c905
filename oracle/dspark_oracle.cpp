// CPU oracle for the DSpark per-step hot path -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow C++ restatement of the four stages of one DSpark speculative
// step, in float64, written to be checked against the pages by eye.  Only
// the test suite, the package smoke check and the benchmark's CPU-baseline
// leg may load it (through oracle/native.py).  The CUDA library never calls
// it and shares no code, header or table with it.
//
// Sources (page title, then section):
//  * "DeepSeek DSpark: Confidence-Scheduled Speculative Decoding 技术解析"
//    (CSDN tutorial), section 四: the draft head samples left to right,
//    feeding the previous token into the next position.
//  * "DSpark.让每一轮计算，多走几步" (explainer): the Markov-head panel (a
//    low-rank transition table biases the vocabulary scores before each
//    draw), the survival panel (a_j = c_1...c_j, E = R + sum a, rate =
//    E / T(B)) and the lossless panel (accept with min(1, p/q), resample from
//    max(p - q, 0) normalised, bonus token from the next target row).
//  * "DSpark: Confidence-Scheduled Speculative Decoding with Semi-
//    Autoregressive Generation" (news article): section 2.1 (confidence head
//    c_k = sigma(w . [h_k ; W1[x_{k-1}]]), sequential temperature scaling),
//    section 2.2 (maximise tau * SPS(B), B = sum_r (1 + l_r), greedy sort with
//    early stop) and challenge 2 (global search without early stop; the
//    verification capacity predicted from the confidences of two steps
//    earlier, the candidates still taken top-K by the current confidences).
//  * "为什么DSpark 可以加速推理？以及DSpark会不会导致降智？" (forum post),
//    lossless proof: acceptance sum_x min(p, q), failure mass
//    sum_x max(0, p - q), emitted marginal p.
//
// Readings where the pages are silent:
//  * x_0 is the anchor token (the bias applies from the first draft position);
//    an anchor of -1 switches the first-position bias off.
//  * The temperature divides logit + bias; the target uses the same
//    temperature; temperature 0 is greedy (argmax, lowest index on ties).
//  * Inverse CDF: the smallest v whose running sum (index order) exceeds
//    u times the total; if rounding leaves none, the last token with
//    non-zero weight.
//  * Confidence head: no bias term; W1 is the Markov embedding; STS divides
//    the head's logit by t_k.
//  * Scheduler: Theta_i = (R + S_i) * SPS[R + i], S_i the sum of the i
//    largest survival values in the order (a descending, request, position);
//    each a is rounded to the nearest multiple of 2^-40 and summed as an
//    integer.  Early stop adds candidate i+1 only while Theta_{i+1} >
//    Theta_i; global mode takes the first argmax; a batch cap max_B bounds i.
//  * Capacity scheduling: with a capacity K (the batch the global search
//    chose on the survival values two steps earlier) the batch is exactly the
//    first min(max(K - R, 0), R*gamma) candidates of the current order.
//  * RNN sequential head (named, no formula given): s_k = tanh(E[x_{k-1}] +
//    s_{k-1} U), s_{-1} = 0, U an r x r matrix; s_k replaces the Markov row
//    E[x_{k-1}] in the bias (bias_k = s_k W).  The confidence head keeps
//    W1[x_{k-1}].  The state is stored in the table's type (bf16 or fp32);
//    its pre-activation is accumulated in fp32 (the embedding, then the fused
//    multiply-adds s_{k-1}[i] * U[i][j], i ascending) and tanh is taken in
//    double, so the stored (quantised) state is decided in the same
//    precision as on the GPU.
//  * Verification: accept position j iff u_acc < p_j(x_j) / q_j(x_j)
//    (strict); at the first rejection draw from max(0, p - q) with the
//    request's final uniform, or from p if that mass is zero; if every
//    verified position is accepted, draw the bonus row's p.  Greedy: accept
//    iff the draft token is the target argmax; the final token is the argmax.
//
// Every sum runs in index order in double; compiled without FMA contraction
// so that x86-64 and aarch64 hosts give the same bits.  OpenMP threads split
// only independent requests; each request's arithmetic is sequential.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

constexpr int kFixShift = 40;  // survival values summed in units of 2^-40

// ------------------------------------------------ Markov head and softmax
// Explainer, Markov-head panel; news article, innovation 1 (low-rank table).

// bias[v] = sum_{i < r} e[i] * W[i][v], i ascending; zero if e is null.
void row_bias(int V, int r, const double* e, const double* W, double* bias) {
  for (int v = 0; v < V; ++v) bias[v] = 0.0;
  if (e == nullptr) return;
  for (int i = 0; i < r; ++i) {
    const double ei = e[i];
    const double* w = W + (size_t)i * V;
    for (int v = 0; v < V; ++v) bias[v] = bias[v] + ei * w[v];
  }
}

// bias[v] = sum_{i < r} E[prev][i] * W[i][v], i ascending; zero if prev < 0.
void markov_bias_row(int V, int r, const double* E, const double* W, int64_t prev, double* bias) {
  row_bias(V, r, prev >= 0 ? E + (size_t)prev * r : nullptr, W, bias);
}

// ------------------------------------------------ RNN sequential head
// News article, innovation 1 (an RNN head keeps a recurrent state);
// explainer, Markov-head panel (it accumulates the prefix inside the block).

// Nearest bf16 value to x (8 significant bits, ties to even), as a double.
double round_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  if (std::fabs(x) < std::ldexp(1.0, -126))  // subnormal bf16: multiples of 2^-133
    return std::ldexp(std::nearbyint(std::ldexp(x, 133)), -133);
  int e;
  const double m = std::frexp(x, &e);  // 0.5 <= |m| < 1
  return std::ldexp(std::nearbyint(std::ldexp(m, 8)), e - 8);
}

// dt 0: bf16, 1: fp32 (the conversion rounds to nearest, ties to even).
double round_state(double x, int dt) { return dt == 0 ? round_bf16(x) : (double)(float)x; }

// s[j] = round(tanh(pre_j)); pre_j in fp32: E[prev][j] (0 if prev < 0), then
// fmaf(s_prev[i], U[i][j], pre_j) for i = 0..r-1.
void rnn_state(int r, int dt, const double* E, const double* U, int64_t prev,
               const double* s_prev, double* s) {
  for (int j = 0; j < r; ++j) {
    float acc = prev >= 0 ? (float)E[(size_t)prev * r + j] : 0.0f;
    for (int i = 0; i < r; ++i) acc = std::fmaf((float)s_prev[i], (float)U[(size_t)i * r + j], acc);
    s[j] = round_state(std::tanh((double)acc), dt);
  }
}

// Weights exp(y - max y) into w; returns their index-order sum; *m = max y.
double softmax_weights(int V, const double* y, double* w, double* m) {
  double mx = -std::numeric_limits<double>::infinity();
  for (int v = 0; v < V; ++v) mx = y[v] > mx ? y[v] : mx;
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    w[v] = std::exp(y[v] - mx);
    S = S + w[v];
  }
  *m = mx;
  return S;
}

// Smallest v with C_v > u * C_{V-1}, C the index-order running sum of w.
int64_t inverse_cdf(int V, const double* w, double u) {
  double total = 0.0;
  for (int v = 0; v < V; ++v) total = total + w[v];
  const double thr = u * total;
  double C = 0.0;
  for (int v = 0; v < V; ++v) {
    C = C + w[v];
    if (C > thr) return v;
  }
  for (int v = V - 1; v >= 0; --v)
    if (w[v] > 0.0) return v;
  return V - 1;
}

int64_t first_argmax(int V, const double* y) {
  int64_t best = 0;
  for (int v = 1; v < V; ++v)
    if (y[v] > y[best]) best = v;
  return best;
}

// q over the vocabulary at one draft position: softmax((z_k + e W) / T),
// e the bias row (null: no bias).
void draft_distribution_row(int V, int r, double T, const double* zk, const double* e,
                            const double* W, double* q, double* tmp) {
  row_bias(V, r, e, W, tmp);
  for (int v = 0; v < V; ++v) tmp[v] = (zk[v] + tmp[v]) / T;
  double m;
  const double S = softmax_weights(V, tmp, q, &m);
  const double lse = m + std::log(S);
  for (int v = 0; v < V; ++v) q[v] = std::exp(tmp[v] - lse);
}

// q over the vocabulary at one draft position: softmax((z_k + E[prev] W) / T).
void draft_distribution(int V, int r, double T, const double* zk, const double* E, const double* W,
                        int64_t prev, double* q, double* tmp) {
  draft_distribution_row(V, r, T, zk, prev >= 0 ? E + (size_t)prev * r : nullptr, W, q, tmp);
}

// The bias row of request n's draft position j: the RNN state S[n][j] when
// S is given, else the Markov row E[x_{j-1}] (x_{-1} the anchor; null if < 0).
const double* bias_row(int G, int r, const double* E, const double* S, const int64_t* anchor,
                       const int64_t* tokens, int n, int64_t j) {
  if (S != nullptr) return S + ((size_t)n * G + j) * r;
  const int64_t prev = j == 0 ? anchor[n] : tokens[(size_t)n * G + j - 1];
  return prev >= 0 ? E + (size_t)prev * r : nullptr;
}

// p over the vocabulary of one target row: softmax(row / T); returns lse.
double target_distribution(int V, double T, const double* row, double* p, double* tmp) {
  for (int v = 0; v < V; ++v) tmp[v] = row[v] / T;
  double m;
  const double S = softmax_weights(V, tmp, p, &m);
  const double lse = m + std::log(S);
  for (int v = 0; v < V; ++v) p[v] = std::exp(tmp[v] - lse);
  return lse;
}

// ------------------------------------------------------------- scheduler
// News article, section 2.2 and challenge 2; explainer, survival panel.

int64_t to_fixed(double a) { return (int64_t)std::nearbyint(a * std::ldexp(1.0, kFixShift)); }

// Candidate order: a descending, then flat index n * gamma + j ascending
// (request, then position): a stable sort by a alone keeps the index order.
std::vector<int64_t> candidate_order(int64_t N, const double* a) {
  std::vector<int64_t> idx(N);
  std::iota(idx.begin(), idx.end(), 0);
  std::stable_sort(idx.begin(), idx.end(), [a](int64_t x, int64_t y) { return a[x] > a[y]; });
  return idx;
}

// The lengths and row offsets of the first i candidates of `order`.
void lengths_of_prefix(int R, int G, const std::vector<int64_t>& order, int64_t i, int64_t* ell,
                       int64_t* row_off) {
  for (int n = 0; n < R; ++n) ell[n] = 0;
  for (int64_t p = 0; p < i; ++p) ell[order[p] / G] += 1;
  row_off[0] = 0;
  for (int n = 0; n < R; ++n) row_off[n + 1] = row_off[n] + 1 + ell[n];
}

}  // namespace

extern "C" {

// ------------------------------------------------------------- threads

void oc_set_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
  (void)n;
#endif
}

int oc_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// ------------------------------------------------------------- helpers

void oc_markov_bias(int n, int V, int r, const double* E, const double* W, const int64_t* prev,
                    double* out) {
  for (int k = 0; k < n; ++k) markov_bias_row(V, r, E, W, prev[k], out + (size_t)k * V);
}

void oc_softmax_rows(int n, int V, const double* y, double* e, double* lse) {
  for (int k = 0; k < n; ++k) {
    double m;
    const double S = softmax_weights(V, y + (size_t)k * V, e + (size_t)k * V, &m);
    lse[k] = m + std::log(S);
  }
}

void oc_inverse_cdf(int n, int V, const double* w, const double* u, int64_t* out) {
  for (int k = 0; k < n; ++k) out[k] = inverse_cdf(V, w + (size_t)k * V, u[k]);
}

void oc_first_argmax(int n, int V, const double* y, int64_t* out) {
  for (int k = 0; k < n; ++k) out[k] = first_argmax(V, y + (size_t)k * V);
}

void oc_to_fixed(int64_t n, const double* a, int64_t* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = to_fixed(a[k]);
}

void oc_draft_distribution(int n, int V, int r, double T, const double* z, const double* E,
                           const double* W, const int64_t* prev, double* q) {
  std::vector<double> tmp(V);
  for (int k = 0; k < n; ++k)
    draft_distribution(V, r, T, z + (size_t)k * V, E, W, prev[k], q + (size_t)k * V, tmp.data());
}

// ------------------------------------------------------------- stage 1: draft
// For k = 1..gamma, left to right: y = (z_k + E[x_{k-1}] W) / T,
// q_k = softmax(y), x_k = inverse CDF of q_k at u_k; greedy when T == 0.
// q_lse: ln sum exp(y) (the maximum of z + bias when greedy);
// q_tok: q_k(x_k) (1 when greedy).
void oc_draft_sample(int R, int G, int V, int r, double T, const double* z, const double* E,
                     const double* W, const int64_t* anchor, const double* u, int64_t* tokens,
                     double* q_lse, double* q_tok) {
#pragma omp parallel
  {
    std::vector<double> y(V), w(V);
#pragma omp for schedule(dynamic, 1)
    for (int n = 0; n < R; ++n) {
      int64_t prev = anchor[n];
      for (int k = 0; k < G; ++k) {
        const size_t nk = (size_t)n * G + k;
        markov_bias_row(V, r, E, W, prev, y.data());
        const double* zk = z + nk * V;
        for (int v = 0; v < V; ++v) y[v] = zk[v] + y[v];
        int64_t x;
        if (T == 0.0) {
          x = first_argmax(V, y.data());
          q_lse[nk] = y[x];
          q_tok[nk] = 1.0;
        } else {
          for (int v = 0; v < V; ++v) y[v] = y[v] / T;
          double m;
          const double S = softmax_weights(V, y.data(), w.data(), &m);
          const double lse = m + std::log(S);
          x = inverse_cdf(V, w.data(), u[nk]);
          q_lse[nk] = lse;
          q_tok[nk] = std::exp(y[x] - lse);
        }
        tokens[nk] = x;
        prev = x;
      }
    }
  }
}

// The RNN head's draft: for k = 0..gamma-1, s_k = rnn_state(x_{k-1}, s_{k-1})
// (s_{-1} = 0, x_{-1} the anchor), y = (z_k + s_k W) / T, then as above.
// S: [R][G][r] the states.
void oc_draft_sample_rnn(int R, int G, int V, int r, int dt, double T, const double* z,
                         const double* E, const double* U, const double* W,
                         const int64_t* anchor, const double* u, int64_t* tokens, double* q_lse,
                         double* q_tok, double* S) {
#pragma omp parallel
  {
    std::vector<double> y(V), w(V), zero(r, 0.0);
#pragma omp for schedule(dynamic, 1)
    for (int n = 0; n < R; ++n) {
      int64_t prev = anchor[n];
      const double* s_prev = zero.data();
      for (int k = 0; k < G; ++k) {
        const size_t nk = (size_t)n * G + k;
        double* s = S + nk * r;
        rnn_state(r, dt, E, U, prev, s_prev, s);
        row_bias(V, r, s, W, y.data());
        const double* zk = z + nk * V;
        for (int v = 0; v < V; ++v) y[v] = zk[v] + y[v];
        int64_t x;
        if (T == 0.0) {
          x = first_argmax(V, y.data());
          q_lse[nk] = y[x];
          q_tok[nk] = 1.0;
        } else {
          for (int v = 0; v < V; ++v) y[v] = y[v] / T;
          double m;
          const double Sw = softmax_weights(V, y.data(), w.data(), &m);
          const double lse = m + std::log(Sw);
          x = inverse_cdf(V, w.data(), u[nk]);
          q_lse[nk] = lse;
          q_tok[nk] = std::exp(y[x] - lse);
        }
        tokens[nk] = x;
        prev = x;
        s_prev = s;
      }
    }
  }
}

// The RNN states of given drafts (s_k from x_{k-1} and s_{k-1}): S [R][G][r].
void oc_rnn_states(int R, int G, int r, int dt, const double* E, const double* U,
                   const int64_t* anchor, const int64_t* tokens, double* S) {
#pragma omp parallel
  {
    std::vector<double> zero(r, 0.0);
#pragma omp for schedule(static)
    for (int n = 0; n < R; ++n) {
      const double* s_prev = zero.data();
      for (int k = 0; k < G; ++k) {
        const int64_t prev = k == 0 ? anchor[n] : tokens[(size_t)n * G + k - 1];
        double* s = S + ((size_t)n * G + k) * r;
        rnn_state(r, dt, E, U, prev, s_prev, s);
        s_prev = s;
      }
    }
  }
}

void oc_round_state(int64_t n, int dt, const double* x, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = round_state(x[i], dt);
}

// ------------------------------------------------------------- stage 2: confidence
// c_{n,k} = sigmoid((w[:d] . h_{n,k} + w[d:] . E1[x_{k-1}]) / t_k); a = running
// product of c.  With c_in given the head is skipped (d, h, w, E1 unused).
void oc_confidence(int R, int G, int d, int r, const double* h, const double* w, const double* E1,
                   const int64_t* anchor, const int64_t* tokens, const double* sts,
                   const double* c_in, double* c, double* a) {
  if (c_in != nullptr) {
    for (size_t i = 0; i < (size_t)R * G; ++i) c[i] = c_in[i];
  } else {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < R; ++n) {
      for (int k = 0; k < G; ++k) {
        const size_t nk = (size_t)n * G + k;
        const int64_t prev = k == 0 ? anchor[n] : tokens[nk - 1];
        double sh = 0.0;
        for (int i = 0; i < d; ++i) sh = sh + h[nk * d + i] * w[i];
        double se = 0.0;
        if (prev >= 0)
          for (int i = 0; i < r; ++i) se = se + E1[(size_t)prev * r + i] * w[d + i];
        const double s = sh + se;
        c[nk] = 1.0 / (1.0 + std::exp(-s / sts[k]));
      }
    }
  }
  for (int n = 0; n < R; ++n) {
    double run = 1.0;
    for (int k = 0; k < G; ++k) {
      run = run * c[(size_t)n * G + k];
      a[(size_t)n * G + k] = run;
    }
  }
}

// ------------------------------------------------------------- stage 3: scheduler
// Returns 0, or -1 if the SPS table is shorter than the largest batch
// considered.  theta ([imax + 1]) and order ([R*G]) may be NULL.
int oc_schedule(int R, int G, const double* a, const double* sps, int64_t n_sps, int early_stop,
                int64_t max_B, int64_t* ell, int64_t* row_off, int64_t* B, double* E,
                int64_t* i_star, double* theta, int64_t* order) {
  const int64_t N = (int64_t)R * G;
  const std::vector<int64_t> idx = candidate_order(N, a);
  std::vector<int64_t> S(N + 1, 0);  // S[i] = sum of the first i, in 2^-40 units
  for (int64_t i = 0; i < N; ++i) S[i + 1] = S[i] + to_fixed(a[idx[i]]);
  int64_t imax = N;
  if (max_B > 0) imax = std::max<int64_t>(0, std::min<int64_t>(N, max_B - R));
  if (R + imax >= n_sps) return -1;
  const double unit = std::ldexp(1.0, -kFixShift);
  std::vector<double> th(imax + 1);
  for (int64_t i = 0; i <= imax; ++i) {
    const double e_i = (double)R + (double)S[i] * unit;
    th[i] = e_i * sps[R + i];
  }
  int64_t is = 0;
  if (early_stop) {
    is = imax;
    for (int64_t i = 0; i < imax; ++i)
      if (!(th[i + 1] > th[i])) {
        is = i;
        break;
      }
  } else {
    for (int64_t i = 1; i <= imax; ++i)
      if (th[i] > th[is]) is = i;
  }
  lengths_of_prefix(R, G, idx, is, ell, row_off);
  *B = R + is;
  *E = (double)R + (double)S[is] * unit;
  *i_star = is;
  if (theta)
    for (int64_t i = 0; i <= imax; ++i) theta[i] = th[i];
  if (order)
    for (int64_t i = 0; i < N; ++i) order[i] = idx[i];
  return 0;
}

// Capacity scheduling: the batch is exactly the first
// i = min(max(K - R, 0), R*G) candidates of the current order.
void oc_schedule_capacity(int R, int G, const double* a, int64_t K, int64_t* ell,
                          int64_t* row_off, int64_t* B, double* E, int64_t* i_star) {
  const int64_t N = (int64_t)R * G;
  const std::vector<int64_t> idx = candidate_order(N, a);
  const int64_t i = std::max<int64_t>(0, std::min<int64_t>(N, K - R));
  int64_t S = 0;
  for (int64_t p = 0; p < i; ++p) S = S + to_fixed(a[idx[p]]);
  lengths_of_prefix(R, G, idx, i, ell, row_off);
  *B = R + i;
  *E = (double)R + (double)S * std::ldexp(1.0, -kFixShift);
  *i_star = i;
}

// ------------------------------------------------------------- stage 4: verify
// Request n's verified rows are target[row_off[n] + j], j = 0..ell[n]; row j
// is the target for draft position j+1, row ell[n] the bonus row.
// Outputs: n_acc, out_tokens [R][G+1] (-1 padded), p_lse [n_rows] (NaN for
// rows no request verifies; the row maximum when greedy), final_kind
// (0 bonus, 1 residual, 2 residual mass zero so p is used), final_row.
void oc_verify(int R, int G, int V, int r, double T, const double* z, const double* E,
               const double* W, const int64_t* anchor, const int64_t* tokens, const int64_t* ell,
               const int64_t* row_off, const double* target, int64_t n_rows, const double* u_acc,
               const double* u_fin, int64_t* n_acc, int64_t* out_tokens, double* p_lse,
               int64_t* final_kind, int64_t* final_row, const double* S) {
  for (int64_t i = 0; i < n_rows; ++i) p_lse[i] = std::numeric_limits<double>::quiet_NaN();
#pragma omp parallel
  {
    std::vector<double> p(V), q(V), tmp(V);
#pragma omp for schedule(dynamic, 1)
    for (int n = 0; n < R; ++n) {
      const int64_t L = ell[n];
      for (int64_t j = 0; j <= L; ++j) {
        const double* row = target + (size_t)(row_off[n] + j) * V;
        if (T == 0.0) {
          p_lse[row_off[n] + j] = row[first_argmax(V, row)];
        } else {
          p_lse[row_off[n] + j] = target_distribution(V, T, row, p.data(), tmp.data());
        }
      }
      int64_t na = L;
      for (int64_t j = 0; j < L; ++j) {
        const double* row = target + (size_t)(row_off[n] + j) * V;
        const int64_t x = tokens[(size_t)n * G + j];
        bool acc;
        if (T == 0.0) {
          acc = first_argmax(V, row) == x;
        } else {
          target_distribution(V, T, row, p.data(), tmp.data());
          draft_distribution_row(V, r, T, z + ((size_t)n * G + j) * V,
                                 bias_row(G, r, E, S, anchor, tokens, n, j), W, q.data(),
                                 tmp.data());
          acc = u_acc[(size_t)n * G + j] < p[x] / q[x];
        }
        if (!acc) {
          na = j;
          break;
        }
      }
      n_acc[n] = na;
      int64_t* out = out_tokens + (size_t)n * (G + 1);
      for (int j = 0; j <= G; ++j) out[j] = j < na ? tokens[(size_t)n * G + j] : -1;
      const int64_t frow = row_off[n] + na;
      final_row[n] = frow;
      const bool rejected = na < L;
      const double* row = target + (size_t)frow * V;
      int64_t kind = rejected ? 1 : 0;
      int64_t tok;
      if (T == 0.0) {
        tok = first_argmax(V, row);
      } else {
        target_distribution(V, T, row, p.data(), tmp.data());
        if (rejected) {
          draft_distribution_row(V, r, T, z + ((size_t)n * G + na) * V,
                                 bias_row(G, r, E, S, anchor, tokens, n, na), W, q.data(),
                                 tmp.data());
          double mass = 0.0;
          for (int v = 0; v < V; ++v) {
            q[v] = std::max(0.0, p[v] - q[v]);  // the residual, in place of q
            mass = mass + q[v];
          }
          if (!(mass > 0.0)) {
            kind = 2;
            tok = inverse_cdf(V, p.data(), u_fin[n]);
          } else {
            tok = inverse_cdf(V, q.data(), u_fin[n]);
          }
        } else {
          tok = inverse_cdf(V, p.data(), u_fin[n]);
        }
      }
      out[na] = tok;
      final_kind[n] = kind;
    }
  }
}

// The distribution request n's final token is drawn from, given its target
// row for position j+1: the residual max(0, p - q_{j+1}) when rejected there
// (p if that mass is zero), else the bonus row's p.  z_row is z[n][j]; the
// bias row is s_row when given (the RNN state), else E[prev].
void oc_final_weights(int V, int r, double T, const double* z_row, const double* E,
                      const double* W, int64_t prev, const double* target_row, int rejected,
                      double* w, const double* s_row) {
  std::vector<double> q(V), tmp(V);
  target_distribution(V, T, target_row, w, tmp.data());
  if (!rejected) return;
  const double* e = s_row != nullptr ? s_row : (prev >= 0 ? E + (size_t)prev * r : nullptr);
  draft_distribution_row(V, r, T, z_row, e, W, q.data(), tmp.data());
  double mass = 0.0;
  for (int v = 0; v < V; ++v) {
    tmp[v] = std::max(0.0, w[v] - q[v]);
    mass = mass + tmp[v];
  }
  if (mass > 0.0)
    for (int v = 0; v < V; ++v) w[v] = tmp[v];
}

}  // extern "C"
