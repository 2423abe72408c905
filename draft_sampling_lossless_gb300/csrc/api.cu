// C ABI of libdspark: argument validation, workspace layout and launches.
// The four stage calls follow the header include/dspark.h, which cites the
// page and section each operation comes from.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "dspark.h"
#include "common.cuh"

using namespace dspark;

namespace {

thread_local char g_err[256] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(DSPARK_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  size_t status, bias, part, sub, row_part, vstate, fin_part, prev, stage, rank, skeys, hpart, vcnt,
      tkey, spre, total;
};

bool sizes_ok(int R, int gamma, int V, int r) {
  return R >= 1 && gamma >= 1 && gamma <= kMaxGamma && V >= 2 && V <= (1 << 22) && r >= 1 &&
         r <= 1024 && (long long)R * gamma <= (1 << 20);
}

Layout layout(int R, int gamma, int V, int r) {
  Layout L;
  const size_t n_chunks = (V + kChunkV - 1) / kChunkV;
  const size_t N = (size_t)R * gamma;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.bias = off;
  off += align_up((size_t)R * V * sizeof(float));
  L.part = off;
  off += align_up((size_t)R * ((V + 127) / 128) * sizeof(double));  // 128-token partials (tensor-core path) or 256
  L.sub = off;
  off += align_up((size_t)R * ((V + 127) / 128) * 8 * sizeof(float));  // their 16-token group sums
  L.row_part = off;
  off += align_up((size_t)R * (gamma + 1) * n_chunks * sizeof(double));
  L.vstate = off;
  off += align_up((size_t)R * sizeof(VerifyState));
  L.fin_part = off;
  // 128-token halves (tensor-core path) or 256-token tiles
  off += align_up((size_t)R * ((V + 127) / 128) * 2 * sizeof(long long));
  L.prev = off;
  off += align_up((size_t)R * sizeof(int32_t));
  L.stage = off;
  off += align_up((size_t)R * r * 2);
  L.rank = off;
  off += align_up(N * sizeof(int32_t));
  L.skeys = off;  // the scheduler's sort keys, two buffers
  off += align_up(N * 2 * sizeof(unsigned long long));
  L.hpart = off;  // lane partials of the confidence head when the draft runs it
  off += align_up((N < (size_t)kFuseMaxCandidates ? N : (size_t)kFuseMaxCandidates) * 32 *
                  sizeof(float));
  L.vcnt = off;  // the row pass's per-request item counters (zero between calls)
  off += align_up((size_t)R * sizeof(int));
  // the fused scheduler's Theta keys and prefixes by rank
  const size_t nf = (N < (size_t)kFuseMaxCandidates ? N : (size_t)kFuseMaxCandidates) + 1;
  L.tkey = off;
  off += align_up(nf * sizeof(unsigned long long));
  L.spre = off;
  off += align_up(nf * sizeof(long long));
  L.total = off;
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

int check_ws(void* ws, size_t ws_bytes, const Layout& L) {
  if (ws == nullptr) return fail(DSPARK_ERR_INVALID_ARG, "workspace is NULL");
  if (((uintptr_t)ws & 255) != 0) return fail(DSPARK_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (ws_bytes < L.total)
    return fail(DSPARK_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, L.total);
  return DSPARK_OK;
}

int check_common(int R, int gamma, int V, int r, int dt) {
  if (!sizes_ok(R, gamma, V, r))
    return fail(DSPARK_ERR_INVALID_ARG,
                "sizes out of range (R=%d gamma=%d V=%d r=%d; need R>=1, 1<=gamma<=%d, "
                "2<=V<=2^22, 1<=r<=1024, R*gamma<=2^20)",
                R, gamma, V, r, kMaxGamma);
  if (dt != DSPARK_BF16 && dt != DSPARK_F32) return fail(DSPARK_ERR_INVALID_ARG, "dt must be 0 (bf16) or 1 (f32)");
  if (dt == DSPARK_BF16 && V % 8 != 0) return fail(DSPARK_ERR_INVALID_ARG, "V must be a multiple of 8 for bf16");
  if (dt == DSPARK_F32 && V % 4 != 0) return fail(DSPARK_ERR_INVALID_ARG, "V must be a multiple of 4 for f32");
  return DSPARK_OK;
}

#define REQUIRE(p)                                                           \
  do {                                                                       \
    if ((p) == nullptr) return fail(DSPARK_ERR_INVALID_ARG, "%s is NULL", #p); \
  } while (0)

}  // namespace

extern "C" {

const char* dspark_status_string(int status) {
  switch (status) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_ERR_INVALID_ARG: return "DSPARK_ERR_INVALID_ARG";
    case DSPARK_ERR_CUDA: return "DSPARK_ERR_CUDA";
    case DSPARK_ERR_UNSUPPORTED: return "DSPARK_ERR_UNSUPPORTED";
    case DSPARK_ERR_WORKSPACE: return "DSPARK_ERR_WORKSPACE";
    default: return "DSPARK_ERR_UNKNOWN";
  }
}

const char* dspark_last_error(void) { return g_err; }

const char* dspark_version(void) { return "libdspark 0.1 sm_103a"; }

size_t dspark_workspace_bytes(int R, int gamma, int V, int r, int n_sps) {
  (void)n_sps;
  if (!sizes_ok(R, gamma, V, r)) return 0;
  return layout(R, gamma, V, r).total;
}

int dspark_device_status(void* ws, int clear, uint32_t* flags, void* stream) {
  REQUIRE(ws);
  REQUIRE(flags);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_device_status");
  return DSPARK_OK;
}

}  // extern "C"

namespace {

// Validates dspark_draft_sample's arguments and fills its launch arguments.
int draft_args(int R, int gamma, int V, int r, float temperature, const void* z, const void* E,
               const void* Wt, int dt, const int32_t* anchor, const float* u_draft,
               int32_t* tokens, double* q_lse, float* q_tok, void* ws, size_t ws_bytes,
               DraftArgs& a) {
  int s = check_common(R, gamma, V, r, dt);
  if (s) return s;
  if (!isfinite(temperature) || temperature < 0.0f)
    return fail(DSPARK_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  REQUIRE(z);
  REQUIRE(E);
  REQUIRE(Wt);
  REQUIRE(anchor);
  REQUIRE(tokens);
  REQUIRE(q_lse);
  REQUIRE(q_tok);
  if (temperature > 0.0f) REQUIRE(u_draft);
  const Layout L = layout(R, gamma, V, r);
  if ((s = check_ws(ws, ws_bytes, L))) return s;
  a.R = R;
  a.gamma = gamma;
  a.V = V;
  a.r = r;
  a.dt = dt;
  a.T = temperature;
  a.z = z;
  a.E = E;
  a.Wt = Wt;
  a.anchor = anchor;
  a.u = u_draft;
  a.tokens = tokens;
  a.q_lse = q_lse;
  a.q_tok = q_tok;
  a.status = at<uint32_t>(ws, L.status);
  a.bias = at<float>(ws, L.bias);
  a.part = at<double>(ws, L.part);
  a.sub = at<float>(ws, L.sub);
  a.grid_counter = at<unsigned>(ws, L.status + 64);
  a.stage = at<void>(ws, L.stage);
  return DSPARK_OK;
}

// Validates dspark_confidence's arguments and fills its launch arguments.
int conf_args(int R, int gamma, int d, int r, int V, const void* hidden, const float* w,
              const void* E1, int dt, const int32_t* anchor, const int32_t* tokens,
              const float* sts_t, const float* c_in, float* c_out, float* a_out, void* ws,
              size_t ws_bytes, ConfArgs& a) {
  if (R < 1 || gamma < 1 || gamma > kMaxGamma || (long long)R * gamma > (1 << 20))
    return fail(DSPARK_ERR_INVALID_ARG, "sizes out of range (R=%d gamma=%d)", R, gamma);
  REQUIRE(c_out);
  REQUIRE(a_out);
  if (c_in == nullptr) {
    int s = check_common(R, gamma, V, r, dt);
    if (s) return s;
    if (d < 1 || d > (1 << 20)) return fail(DSPARK_ERR_INVALID_ARG, "d out of range (%d)", d);
    REQUIRE(hidden);
    REQUIRE(w);
    REQUIRE(E1);
    REQUIRE(anchor);
    REQUIRE(tokens);
    REQUIRE(sts_t);
  }
  if (ws == nullptr) return fail(DSPARK_ERR_INVALID_ARG, "workspace is NULL");
  if (ws_bytes < 256) return fail(DSPARK_ERR_WORKSPACE, "workspace has %zu bytes, needs 256", ws_bytes);
  a.R = R;
  a.gamma = gamma;
  a.d = d;
  a.r = r;
  a.V = V;
  a.dt = dt;
  a.h = hidden;
  a.w = w;
  a.E1 = E1;
  a.anchor = anchor;
  a.tokens = tokens;
  a.sts = sts_t;
  a.c_in = c_in;
  a.c_out = c_out;
  a.a_out = a_out;
  a.status = at<uint32_t>(ws, 0);
  return DSPARK_OK;
}

// Validates dspark_schedule's arguments and fills its launch arguments.
int sched_args(int R, int gamma, const float* a, const float* sps, int n_sps, int early_stop,
               int max_B, int32_t* ell, int32_t* row_off, int32_t* B_out, double* E_out,
               void* ws, size_t ws_bytes, SchedArgs& s) {
  if (R < 1 || gamma < 1 || gamma > kMaxGamma || (long long)R * gamma > (1 << 20))
    return fail(DSPARK_ERR_INVALID_ARG, "sizes out of range (R=%d gamma=%d)", R, gamma);
  REQUIRE(a);
  REQUIRE(sps);
  REQUIRE(ell);
  REQUIRE(row_off);
  REQUIRE(B_out);
  REQUIRE(E_out);
  const int N = R * gamma;
  if (max_B < 0 || (max_B > 0 && max_B < R))
    return fail(DSPARK_ERR_INVALID_ARG, "max_B must be 0 or >= R (got %d, R=%d)", max_B, R);
  const int imax = max_B > 0 ? (max_B - R < N ? max_B - R : N) : N;
  if ((long long)n_sps <= (long long)R + imax)
    return fail(DSPARK_ERR_INVALID_ARG, "SPS table has %d entries, needs more than R + imax = %d",
                n_sps, R + imax);
  if (ws == nullptr) return fail(DSPARK_ERR_INVALID_ARG, "workspace is NULL");
  if (((uintptr_t)ws & 255) != 0) return fail(DSPARK_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  s.R = R;
  s.gamma = gamma;
  s.n_sps = n_sps;
  s.early_stop = early_stop;
  s.max_B = max_B;
  s.a = a;
  s.sps = sps;
  s.ell = ell;
  s.row_off = row_off;
  s.B_out = B_out;
  s.E_out = E_out;
  s.status = at<uint32_t>(ws, 0);
  // the scheduler's arrays follow the status word; any workspace sized by
  // dspark_workspace_bytes for these R and gamma covers them
  s.rank = at<int32_t>(ws, 256);
  s.keys = at<unsigned long long>(ws, 256 + align_up((size_t)N * sizeof(int32_t)));
  const size_t need = 256 + sched_scratch_bytes((size_t)N);
  if (ws_bytes < need) return fail(DSPARK_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  s.imax = imax;
  return DSPARK_OK;
}

}  // namespace

extern "C" {

int dspark_draft_sample(int R, int gamma, int V, int r, float temperature, const void* z,
                        const void* E, const void* Wt, int dt, const int32_t* anchor,
                        const float* u_draft, int32_t* tokens, double* q_lse, float* q_tok,
                        void* ws, size_t ws_bytes, void* stream) {
  DraftArgs a;
  int s = draft_args(R, gamma, V, r, temperature, z, E, Wt, dt, anchor, u_draft, tokens, q_lse,
                     q_tok, ws, ws_bytes, a);
  if (s) return s;
  cudaError_t e = launch_draft(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_draft_sample");
  return DSPARK_OK;
}

int dspark_draft_sample_rnn(int R, int gamma, int V, int r, float temperature, const void* z,
                            const void* E, const void* U, const void* Wt, int dt,
                            const int32_t* anchor, const float* u_draft, int32_t* tokens,
                            double* q_lse, float* q_tok, void* S, void* ws, size_t ws_bytes,
                            void* stream) {
  DraftArgs a;
  int s = draft_args(R, gamma, V, r, temperature, z, E, Wt, dt, anchor, u_draft, tokens, q_lse,
                     q_tok, ws, ws_bytes, a);
  if (s) return s;
  REQUIRE(U);
  REQUIRE(S);
  if (((uintptr_t)S & 15) != 0) return fail(DSPARK_ERR_INVALID_ARG, "S must be 16-byte aligned");
  a.U = U;
  a.S = S;
  cudaError_t e = launch_draft(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_draft_sample_rnn");
  return DSPARK_OK;
}

int dspark_confidence(int R, int gamma, int d, int r, int V, const void* hidden, const float* w,
                      const void* E1, int dt, const int32_t* anchor, const int32_t* tokens,
                      const float* sts_t, const float* c_in, float* c_out, float* a_out,
                      void* ws, size_t ws_bytes, void* stream) {
  ConfArgs a;
  int s = conf_args(R, gamma, d, r, V, hidden, w, E1, dt, anchor, tokens, sts_t, c_in, c_out,
                    a_out, ws, ws_bytes, a);
  if (s) return s;
  cudaError_t e = launch_confidence(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_confidence");
  return DSPARK_OK;
}

int dspark_schedule(int R, int gamma, const float* a, const float* sps, int n_sps, int early_stop,
                    int max_B, int32_t* ell, int32_t* row_off, int32_t* B_out, double* E_out,
                    void* ws, size_t ws_bytes, void* stream) {
  SchedArgs s{};
  int st = sched_args(R, gamma, a, sps, n_sps, early_stop, max_B, ell, row_off, B_out, E_out, ws,
                      ws_bytes, s);
  if (st) return st;
  cudaError_t e = launch_schedule(s, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_schedule");
  return DSPARK_OK;
}

int dspark_schedule_async(int R, int gamma, const float* a, const int32_t* capacity,
                          int32_t* ell, int32_t* row_off, int32_t* B_out, double* E_out,
                          void* ws, size_t ws_bytes, void* stream) {
  if (R < 1 || gamma < 1 || gamma > kMaxGamma || (long long)R * gamma > (1 << 20))
    return fail(DSPARK_ERR_INVALID_ARG, "sizes out of range (R=%d gamma=%d)", R, gamma);
  REQUIRE(a);
  REQUIRE(capacity);
  REQUIRE(ell);
  REQUIRE(row_off);
  REQUIRE(B_out);
  REQUIRE(E_out);
  if (ws == nullptr) return fail(DSPARK_ERR_INVALID_ARG, "workspace is NULL");
  if (((uintptr_t)ws & 255) != 0) return fail(DSPARK_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  const size_t N = (size_t)R * gamma;
  const size_t need = 256 + sched_scratch_bytes(N);
  if (ws_bytes < need) return fail(DSPARK_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  SchedArgs sa{};
  sa.R = R;
  sa.gamma = gamma;
  sa.a = a;
  sa.ell = ell;
  sa.row_off = row_off;
  sa.B_out = B_out;
  sa.E_out = E_out;
  sa.status = at<uint32_t>(ws, 0);
  sa.rank = at<int32_t>(ws, 256);
  sa.keys = at<unsigned long long>(ws, 256 + align_up(N * sizeof(int32_t)));
  sa.imax = (int)N;
  cudaError_t e = launch_schedule_async(sa, capacity, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_schedule_async");
  return DSPARK_OK;
}

int dspark_draft_schedule(int R, int gamma, int V, int r, float temperature, const void* z,
                          const void* E, const void* Wt, int dt, const int32_t* anchor,
                          const float* u_draft, int d, const void* hidden, const float* w,
                          const void* E1, const float* sts_t, const float* c_in,
                          const float* sps, int n_sps, int early_stop, int max_B,
                          int32_t* tokens, double* q_lse, float* q_tok, float* c_out,
                          float* a_out, int32_t* ell, int32_t* row_off, int32_t* B_out,
                          double* E_out, void* ws, size_t ws_bytes, void* stream) {
  DraftArgs da;
  ConfArgs ca;
  SchedArgs sa{};
  int s = draft_args(R, gamma, V, r, temperature, z, E, Wt, dt, anchor, u_draft, tokens, q_lse,
                     q_tok, ws, ws_bytes, da);
  if (s) return s;
  if ((s = conf_args(R, gamma, d, r, V, hidden, w, E1, dt, anchor, tokens, sts_t, c_in, c_out,
                     a_out, ws, ws_bytes, ca)))
    return s;
  if ((s = sched_args(R, gamma, a_out, sps, n_sps, early_stop, max_B, ell, row_off, B_out, E_out,
                      ws, ws_bytes, sa)))
    return s;
  const Layout L = layout(R, gamma, V, r);
  DraftFuse f;
  f.d = d;
  f.h = hidden;
  f.w = w;
  f.E1 = E1;
  f.sts = sts_t;
  f.c_in = c_in;
  f.c_out = c_out;
  f.a_out = a_out;
  f.hpart = at<float>(ws, L.hpart);
  f.early_stop = early_stop;
  f.imax = sa.imax < 0 ? 0 : sa.imax;
  f.sps = sps;
  f.rank = at<int32_t>(ws, L.rank);
  f.tkey = at<unsigned long long>(ws, L.tkey);
  f.spre = at<long long>(ws, L.spre);
  f.ell = ell;
  f.row_off = row_off;
  f.B_out = B_out;
  f.E_out = E_out;
  int fused = 0;
  da.fuse = &f;
  da.fused = &fused;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = launch_draft(da, st);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_draft_schedule (draft)");
  if (!fused) {
    e = launch_confidence(ca, st);
    if (e != cudaSuccess) return cuda_fail(e, "dspark_draft_schedule (confidence)");
    e = launch_schedule(sa, st);
    if (e != cudaSuccess) return cuda_fail(e, "dspark_draft_schedule (schedule)");
  }
  return DSPARK_OK;
}

}  // extern "C"

namespace {

// dspark_verify and dspark_verify_rnn: with rnn set, E is the states table
// [R][gamma][r] and anchor is unused (the bias row of position j is S[n][j]).
int verify_call(bool rnn, int R, int gamma, int V, int r, float temperature, const void* z,
                const void* E, const void* Wt, int dt, const int32_t* anchor,
                const int32_t* tokens, const double* q_lse, const float* q_tok,
                const int32_t* ell, const int32_t* row_off, const void* target,
                int64_t n_target_rows, const float* u_acc, const float* u_fin, int32_t* n_acc,
                int32_t* out_tokens, double* p_lse, void* ws, size_t ws_bytes, void* stream,
                const char* name) {
  int s = check_common(R, gamma, V, r, dt);
  if (s) return s;
  if (!isfinite(temperature) || temperature < 0.0f)
    return fail(DSPARK_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  REQUIRE(tokens);
  REQUIRE(ell);
  REQUIRE(row_off);
  REQUIRE(target);
  REQUIRE(n_acc);
  REQUIRE(out_tokens);
  if (((uintptr_t)target | (uintptr_t)z) & 15)
    return fail(DSPARK_ERR_INVALID_ARG, "target and z must be 16-byte aligned");
  if (n_target_rows < 1 || n_target_rows > (int64_t)1 << 31)
    return fail(DSPARK_ERR_INVALID_ARG, "n_target_rows out of range");
  if (temperature > 0.0f) {
    REQUIRE(z);
    REQUIRE(E);
    REQUIRE(Wt);
    if (!rnn) REQUIRE(anchor);
    REQUIRE(q_lse);
    REQUIRE(q_tok);
    REQUIRE(u_acc);
    REQUIRE(u_fin);
  }
  const Layout L = layout(R, gamma, V, r);
  if ((s = check_ws(ws, ws_bytes, L))) return s;
  VerifyArgs a;
  a.R = R;
  a.gamma = gamma;
  a.V = V;
  a.r = r;
  a.dt = dt;
  a.T = temperature;
  a.z = z;
  a.E = E;
  a.Wt = Wt;
  a.anchor = rnn ? nullptr : anchor;
  a.tokens = tokens;
  a.q_lse = q_lse;
  a.q_tok = q_tok;
  a.ell = ell;
  a.row_off = row_off;
  a.target = target;
  a.n_rows = n_target_rows;
  a.u_acc = u_acc;
  a.u_fin = u_fin;
  a.n_acc = n_acc;
  a.out_tokens = out_tokens;
  a.p_lse = p_lse;
  a.status = at<uint32_t>(ws, L.status);
  a.row_part = at<double>(ws, L.row_part);
  a.vstate = at<VerifyState>(ws, L.vstate);
  a.bias = at<float>(ws, L.bias);
  a.fin_part = at<long long>(ws, L.fin_part);
  a.prev = at<int32_t>(ws, L.prev);
  a.vcnt = at<int>(ws, L.vcnt);
  cudaError_t e = launch_verify(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return DSPARK_OK;
}

}  // namespace

extern "C" {

int dspark_verify(int R, int gamma, int V, int r, float temperature, const void* z, const void* E,
                  const void* Wt, int dt, const int32_t* anchor, const int32_t* tokens,
                  const double* q_lse, const float* q_tok, const int32_t* ell,
                  const int32_t* row_off, const void* target, int64_t n_target_rows,
                  const float* u_acc, const float* u_fin, int32_t* n_acc, int32_t* out_tokens,
                  double* p_lse, void* ws, size_t ws_bytes, void* stream) {
  return verify_call(false, R, gamma, V, r, temperature, z, E, Wt, dt, anchor, tokens, q_lse,
                     q_tok, ell, row_off, target, n_target_rows, u_acc, u_fin, n_acc, out_tokens,
                     p_lse, ws, ws_bytes, stream, "dspark_verify");
}

int dspark_verify_rnn(int R, int gamma, int V, int r, float temperature, const void* z,
                      const void* S, const void* Wt, int dt, const int32_t* tokens,
                      const double* q_lse, const float* q_tok, const int32_t* ell,
                      const int32_t* row_off, const void* target, int64_t n_target_rows,
                      const float* u_acc, const float* u_fin, int32_t* n_acc,
                      int32_t* out_tokens, double* p_lse, void* ws, size_t ws_bytes,
                      void* stream) {
  if (S != nullptr && ((uintptr_t)S & 15) != 0)
    return fail(DSPARK_ERR_INVALID_ARG, "S must be 16-byte aligned");
  return verify_call(true, R, gamma, V, r, temperature, z, S, Wt, dt, nullptr, tokens, q_lse,
                     q_tok, ell, row_off, target, n_target_rows, u_acc, u_fin, n_acc, out_tokens,
                     p_lse, ws, ws_bytes, stream, "dspark_verify_rnn");
}

int dspark_check_wait_timeout(int limit_us, void* ws, size_t ws_bytes, void* stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(DSPARK_ERR_INVALID_ARG, "limit_us must be in [1, 1000000] (got %d)", limit_us);
  REQUIRE(ws);
  if (((uintptr_t)ws & 255) != 0) return fail(DSPARK_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (ws_bytes < 256) return fail(DSPARK_ERR_WORKSPACE, "workspace has %zu bytes, needs 256", ws_bytes);
  cudaStream_t st = (cudaStream_t)stream;
  // the same header words the persistent draft uses: status, grid counter
  unsigned* ctr = at<unsigned>(ws, 64);
  int* out = at<int>(ws, 128);
  cudaError_t e = cudaMemsetAsync(ctr, 0, sizeof(unsigned), st);
  if (e == cudaSuccess)
    e = launch_wait_check((uint64_t)limit_us * 1000ull, ctr, at<uint32_t>(ws, 0), out, st);
  if (e != cudaSuccess) return cuda_fail(e, "dspark_check_wait_timeout");
  return DSPARK_OK;
}

}  // extern "C"

namespace dspark {
// Lets other translation units report a reason through dspark_last_error().
void set_error_text(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }
}  // namespace dspark
