/*
 * libdspark -- the per-step hot path of DSpark confidence-scheduled
 * speculative decoding on one GB300 (sm_103a).
 *
 * One speculative step over R requests, a draft block of gamma positions and
 * a vocabulary of V tokens runs as four calls, in this order, on one CUDA
 * stream:
 *
 *   dspark_draft_sample  semi-autoregressive draft with the Markov head
 *   dspark_confidence    confidence head, sequential temperature scaling,
 *                        cumulative survival
 *   dspark_schedule      hardware-aware prefix scheduler
 *   (the target model's forward pass over the scheduled rows -- not here)
 *   dspark_verify        lossless rejection-sampling (or greedy) verification
 *   dspark_draft_sample_rnn, dspark_verify_rnn
 *                        the same two stages with the RNN sequential head
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array argument is a DEVICE pointer owned by the caller, row-major,
 *   densely packed, with the layout given beside it.  The library never
 *   allocates, frees or retains the caller's memory.  Its only state that
 *   outlives a call: per-device launch set-up (shared-memory opt-ins,
 *   occupancy and SM counts, made once per device under a lock), launch
 *   counters and trace events, and the static device scratch of
 *   dspark_schedule_noalloc (shared by every call of that entry point).
 * - Scratch memory comes from the caller's workspace `ws` of `ws_bytes`
 *   bytes, at least dspark_workspace_bytes(...) for the same sizes, 256-byte
 *   aligned.  Its first 4 bytes are a device status word: kernels OR the
 *   DSPARK_DEVFLAG_* bits into it when they meet bad data they can only see
 *   on the device (a token id out of range, a non-finite value).  Zero the
 *   whole workspace once after allocating it; read the word with
 *   dspark_device_status().  Calls leave the workspace's counters at zero
 *   when they complete; after a call that set DSPARK_DEVFLAG_TIMEOUT, zero
 *   the workspace again before reusing it.
 *   Two calls in flight at the same time need two workspaces.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *   call only enqueues work on it and returns; nothing is synchronised.
 * - Every call validates its host-visible arguments before launching anything
 *   and returns DSPARK_ERR_INVALID_ARG (nothing enqueued) on a null pointer,
 *   a non-positive or too large size, or an inconsistent combination;
 *   DSPARK_ERR_WORKSPACE if ws_bytes is too small; DSPARK_ERR_CUDA if a launch
 *   fails.  dspark_last_error() gives a one-line reason for the last failure
 *   in the calling thread.  No call throws, traps or waits without bound.
 * - Logits, the Markov tables and hidden states share one element type `dt`
 *   (DSPARK_BF16 or DSPARK_F32); arithmetic is fp32 with fp64 / integer
 *   accumulation where sums decide a sampled token.
 * - Sizes: 1 <= R, 1 <= gamma <= 32, 2 <= V <= 2^22, 1 <= r <= 1024,
 *   R * gamma <= 2^20; V a multiple of 8 for bf16 and of 4 for fp32.
 *
 * Sources for each operation are given as the page title and its section.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1,
  DSPARK_ERR_CUDA = 2,
  DSPARK_ERR_UNSUPPORTED = 3,
  DSPARK_ERR_WORKSPACE = 4
} dspark_status;

typedef enum { DSPARK_BF16 = 0, DSPARK_F32 = 1 } dspark_dtype;

/* Bits of the device status word (first 4 bytes of the workspace). */
#define DSPARK_DEVFLAG_TOKEN_RANGE 0x1u /* a token id outside [0, V) (anchor: [-1, V)) */
#define DSPARK_DEVFLAG_NONFINITE 0x2u   /* a NaN / inf logit, survival or SPS value */
#define DSPARK_DEVFLAG_ROW_RANGE 0x4u   /* a target row index outside [0, n_target_rows) */
#define DSPARK_DEVFLAG_SPS_RANGE 0x8u   /* the scheduler needed SPS[B] beyond the table */
#define DSPARK_DEVFLAG_TIMEOUT 0x10u    /* a bounded on-chip wait gave up (results invalid) */

/* Human-readable name of a status code.  Never NULL. */
const char* dspark_status_string(int status);

/* One-line reason for the last non-OK status returned in this thread. */
const char* dspark_last_error(void);

/* Library version string, e.g. "libdspark 0.1 sm_103a". */
const char* dspark_version(void);

/* Workspace bytes that cover every call below for these sizes (n_sps = SPS
 * table length).  Returns 0 if the sizes are out of range. */
size_t dspark_workspace_bytes(int R, int gamma, int V, int r, int n_sps);

/* Copies the device status word to *flags (synchronises `stream`) and, if
 * clear != 0, zeroes it afterwards.  Returns DSPARK_OK or DSPARK_ERR_CUDA. */
int dspark_device_status(void* ws, int clear, uint32_t* flags, void* stream);

/*
 * dspark_draft_sample -- semi-autoregressive draft sampling.
 *
 * "DSpark.让每一轮计算，多走几步" (explainer), Markov head panel, and the news
 * article "DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation", innovation 1, second stage (sequential
 * head, low-rank Markov table); the CSDN tutorial, section 四 (left-to-right
 * sampling that feeds the previous token forward).
 *
 * For k = 1..gamma, left to right, for every request n:
 *   bias_k[v] = sum_i E[x_{k-1}][i] * W[i][v]     (x_0 = anchor[n])
 *   y_k[v]    = (z[n][k-1][v] + bias_k[v]) / T
 *   x_k       = smallest v with C(v) > u * C(V-1), C the running sum of
 *               exp(y_k) in index order, u = u_draft[n][k-1]
 * With T == 0 (greedy) x_k = argmax_v (z + bias), lowest index on ties.
 *
 *   z        [R][gamma][V] dt   base logits of the parallel backbone
 *   E        [V][r] dt          Markov embedding table
 *   Wt       [V][r] dt          Markov output table, TRANSPOSED: Wt[v][i] = W[i][v]
 *   anchor   [R] int32          x_0; -1 = no bias at the first position
 *   u_draft  [R][gamma] f32     uniforms in [0,1); may be NULL iff T == 0
 *   tokens   [R][gamma] int32   out: x_1..x_gamma
 *   q_lse    [R][gamma] f64     out: ln sum_v exp(y_k[v]) (T > 0); max_v (z+bias) (T == 0)
 *   q_tok    [R][gamma] f32     out: q_k(x_k) = exp(y_k[x_k] - q_lse) (T > 0); 1 (T == 0)
 *
 * q_lse is carried in double so that verification can renormalise the draft
 * distribution without an fp32 rounding that would shift every residual CDF
 * boundary.  temperature must be finite and >= 0.
 */
int dspark_draft_sample(int R, int gamma, int V, int r, float temperature,
                        const void* z, const void* E, const void* Wt, int dt,
                        const int32_t* anchor, const float* u_draft,
                        int32_t* tokens, double* q_lse, float* q_tok,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_draft_sample_rnn -- the semi-autoregressive draft with the RNN
 * sequential head instead of the Markov head.
 *
 * News article "DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation", innovation 1, second stage (the RNN head
 * keeps a recurrent state that captures longer dependencies); explainer
 * "DSpark.让每一轮计算，多走几步", Markov-head panel (an RNN head accumulates
 * the prefix inside the block).  The pages give no formula; this library's
 * reading is an Elman recurrence in the Markov head's shapes:
 *
 *   s_0 = 0 (before the first position), x_0 = anchor[n]
 *   s_k[j] = round(tanh(pre_k[j])), pre_k[j] = E[x_{k-1}][j] + sum_i s_{k-1}[i] U[i][j]
 *   bias_k = s_k W, then y_k, x_k, q_lse, q_tok exactly as dspark_draft_sample
 *
 * U = 0 gives the Markov head on the table round(tanh(E)).  pre_k is
 * accumulated in fp32 in a fixed order -- the E entry first, then one fused
 * multiply-add per i, i ascending (s_0 = 0 still runs the chain) -- tanh is
 * taken in double and rounded once to dt: the states are bit-reproducible.
 * An anchor of -1 (or a token outside [0, V), flagged) contributes a zero E
 * row.  Runs one state launch and one draw per position (no persistent
 * launch).
 *
 *   z, E, Wt, anchor, u_draft, tokens, q_lse, q_tok: as dspark_draft_sample
 *   U        [r][r] dt          recurrence matrix, r <= 1024
 *   S        [R][gamma][r] dt   out: the states s_1..s_gamma (S[n][k-1] = s_k,
 *                               the bias row of position k); 16-byte aligned;
 *                               dspark_verify_rnn takes it in place of E
 */
int dspark_draft_sample_rnn(int R, int gamma, int V, int r, float temperature,
                            const void* z, const void* E, const void* U, const void* Wt,
                            int dt, const int32_t* anchor, const float* u_draft,
                            int32_t* tokens, double* q_lse, float* q_tok, void* S,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_confidence -- confidence head with sequential temperature scaling
 * and cumulative survival.
 *
 * News article, section 2.1 (confidence head c_k = sigma(w . [h_k ; W1[x_{k-1}]]),
 * post-hoc sequential temperature scaling); explainer, survival panel
 * (a_j = c_1 ... c_j).
 *
 *   s[n][k] = sum_i w[i] * h[n][k][i] + sum_i w[d+i] * E1[x_{k-1}][i]
 *   c[n][k] = 1 / (1 + exp(-s[n][k] / sts_t[k]))
 *   a[n][j] = c[n][0] * ... * c[n][j]       (fp32 running product, never increases)
 *
 *   hidden  [R][gamma][d] dt   backbone hidden states; NULL iff c_in != NULL
 *   w       [d + r] f32        head weights (no bias term)
 *   E1      [V][r] dt          Markov embedding (may alias E)
 *   anchor  [R], tokens [R][gamma] int32   x_0 and x_1..x_gamma (x_{k-1} indexing)
 *   sts_t   [gamma] f32        per-position STS temperatures (> 0)
 *   c_in    [R][gamma] f32     if non-NULL: confidences given, the head is skipped
 *   c_out, a_out [R][gamma] f32   out
 * d may be 0 only when c_in != NULL.
 */
int dspark_confidence(int R, int gamma, int d, int r, int V,
                      const void* hidden, const float* w, const void* E1, int dt,
                      const int32_t* anchor, const int32_t* tokens, const float* sts_t,
                      const float* c_in, float* c_out, float* a_out,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_schedule -- hardware-aware prefix scheduler.
 *
 * News article, section 2.2 (maximise tau * SPS(B) over l_1..l_R with
 * B = sum_r (1 + l_r); sort all candidates by survival, add them greedily,
 * stop as soon as throughput stops rising; SPS profiled into a lookup table)
 * and challenge 2 (global search without early stop); explainer, survival
 * panel (E = R + sum_r sum_{j<=l_r} a_{r,j}, rate = E / T(B)).
 *
 * Candidates (n, j) are ordered by a[n][j] descending, then n, then j
 * ascending (a stable radix sort of the survival values over one cluster of
 * thread blocks).  With S_i the sum of the first i (each a rounded to a multiple
 * of 2^-40 and summed exactly as an integer):
 *   Theta_i = (R + S_i) * SPS[R + i]                       (double)
 *   early_stop != 0: i* = first i with Theta_{i+1} <= Theta_i (else the last)
 *   early_stop == 0: i* = first argmax_i Theta_i
 * for i in [0, imax], imax = R*gamma, or max_B - R when max_B > 0.
 *   l_n = number of request n's candidates among the first i*
 *
 *   a        [R][gamma] f32   survival values (finite, >= 0)
 *   sps      [n_sps] f32      steps/s for a verify batch of B rows, B = 0..n_sps-1;
 *                             n_sps > R + imax is required
 *   ell      [R] int32        out: l_n
 *   row_off  [R+1] int32      out: exclusive prefix sum of (1 + l_n)
 *   B_out    [1] int32        out: R + i*  (= row_off[R])
 *   E_out    [1] f64          out: R + S_{i*}
 */
int dspark_schedule(int R, int gamma, const float* a, const float* sps, int n_sps,
                    int early_stop, int max_B, int32_t* ell, int32_t* row_off,
                    int32_t* B_out, double* E_out, void* ws, size_t ws_bytes,
                    void* stream);

/*
 * dspark_schedule_async -- asynchronous scheduling with a capacity fixed
 * before the step.
 *
 * News article, challenge 2: zero-overhead scheduling needs the next step's
 * verification batch size before the current step finishes, and the
 * profiled SPS curve is not smooth, so the verification capacity is taken
 * from the confidences of two steps earlier while the candidates that fill it
 * are still chosen by the current confidences; because the capacity does not
 * depend on the current step's draft, a global search (no early stop) stays
 * lossless.  Explainer, survival panel (production sets the capacity from
 * earlier steps' predictions).
 *
 * With K = capacity[0], read on the device (so a capacity produced by an
 * earlier call -- e.g. the B_out of a global-search dspark_schedule on the
 * survival values of two steps earlier -- never needs a host read):
 *   i*  = min(max(K - R, 0), R * gamma)
 *   l_n = number of request n's candidates among the first i* of the order
 *         (a descending, then n, then j ascending), as in dspark_schedule
 *   B_out = R + i*,  E_out = R + S_{i*}  (S as in dspark_schedule)
 *
 *   a         [R][gamma] f32   current survival values (finite, >= 0)
 *   capacity  [1] int32        device: the batch capacity K
 *   ell, row_off, B_out, E_out as in dspark_schedule
 * Uses the scheduler's part of `ws` (a workspace sized by
 * dspark_workspace_bytes for R and gamma).
 */
int dspark_schedule_async(int R, int gamma, const float* a, const int32_t* capacity,
                          int32_t* ell, int32_t* row_off, int32_t* B_out, double* E_out,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_draft_schedule -- dspark_draft_sample, dspark_confidence and
 * dspark_schedule in one call.
 *
 * The three stages of the news article's figure 1 pipeline (draft, confidence
 * head with STS, hardware-aware scheduler; innovation 1 and sections 2.1 and
 * 2.2) with the arguments of the three calls, in that order: the draft's,
 * then the head's (d, hidden, w, E1, sts_t, c_in; r, V and dt are the
 * draft's), then the scheduler's (sps, n_sps, early_stop, max_B), then every
 * output.  The confidence head reads the tokens just drafted; the scheduler
 * reads a_out.  Results are bit-identical to the three calls in sequence.
 *
 * When the draft runs as one persistent launch and the head takes its bf16
 * one-pass form (d <= 4096 and a multiple of 8, 16-byte aligned rows and
 * weights) or c_in is given, and R * gamma <= 8192, the head and the
 * scheduler run inside that launch after the last draft position (the hidden
 * states' term at the first position, while its bias is computed); otherwise
 * the three stages are launched one after another.  Errors: those of the
 * three calls.
 */
int dspark_draft_schedule(int R, int gamma, int V, int r, float temperature,
                          const void* z, const void* E, const void* Wt, int dt,
                          const int32_t* anchor, const float* u_draft,
                          int d, const void* hidden, const float* w, const void* E1,
                          const float* sts_t, const float* c_in,
                          const float* sps, int n_sps, int early_stop, int max_B,
                          int32_t* tokens, double* q_lse, float* q_tok,
                          float* c_out, float* a_out,
                          int32_t* ell, int32_t* row_off, int32_t* B_out, double* E_out,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_verify -- lossless rejection-sampling or greedy verification.
 *
 * Forum post "为什么DSpark 可以加速推理？以及DSpark会不会导致降智？", lossless
 * proof (accept with min(1, p/q), resample from max(0, p - q) normalised,
 * marginal equals p); explainer, lossless panel (bonus token from the next
 * target distribution when the whole block is accepted); CSDN tutorial,
 * section 五 (acceptance rule, stop at the first rejection).
 *
 * Request n's verified target rows are row_off[n] + j, j = 0..ell[n]; row j
 * is the target's distribution for draft position j+1 and row ell[n] the
 * bonus row.  With p_j = softmax(target_row / T), q_j the draft distribution
 * of position j (rebuilt from z, E, Wt and q_lse):
 *   accept position j+1 iff u_acc[n][j] < p_j(x_{j+1}) / q_tok[n][j]
 *   n_acc[n] = index of the first rejected position (0-based), or ell[n]
 *   final token: rejected -> inverse CDF of max(0, p - q) (of p if that mass
 *                is zero) with u_fin[n]; all accepted -> inverse CDF of the
 *                bonus row's p with u_fin[n]
 * Greedy (T == 0): accept iff x_{j+1} == argmax(target row j) (lowest index
 * on ties); the final token is the argmax of row n_acc.
 *
 *   z, E, Wt, anchor, tokens, q_lse, q_tok   as produced / consumed by dspark_draft_sample
 *   ell [R], row_off [R+1] int32             from dspark_schedule (or any layout
 *                                            whose rows exist)
 *   target        [n_target_rows][V] dt      target logits
 *   u_acc [R][gamma], u_fin [R] f32          uniforms in [0,1); may be NULL iff T == 0
 *   n_acc     [R] int32                      out
 *   out_tokens [R][gamma+1] int32            out: the n_acc accepted tokens, then the
 *                                            correction / bonus token, then -1
 *   p_lse     [n_target_rows] f64 or NULL    out: ln sum exp(row / T) of every verified
 *                                            row (row maximum when T == 0)
 */
int dspark_verify(int R, int gamma, int V, int r, float temperature,
                  const void* z, const void* E, const void* Wt, int dt,
                  const int32_t* anchor, const int32_t* tokens, const double* q_lse,
                  const float* q_tok, const int32_t* ell, const int32_t* row_off,
                  const void* target, int64_t n_target_rows, const float* u_acc,
                  const float* u_fin, int32_t* n_acc, int32_t* out_tokens,
                  double* p_lse, void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_verify_rnn -- dspark_verify for drafts made with the RNN head
 * (dspark_draft_sample_rnn): the draft distribution of position j is rebuilt
 * with the bias row S[n][j-1] (the state that drafted it) instead of
 * E[x_{j-1}], for the accept tests and the residual max(0, p - q).  Same
 * pages and rules as dspark_verify; anchor is not needed.
 *
 *   S        [R][gamma][r] dt   the states written by dspark_draft_sample_rnn
 *   every other argument: as dspark_verify (S replaces E; no anchor)
 */
int dspark_verify_rnn(int R, int gamma, int V, int r, float temperature, const void* z,
                      const void* S, const void* Wt, int dt, const int32_t* tokens,
                      const double* q_lse, const float* q_tok, const int32_t* ell,
                      const int32_t* row_off, const void* target, int64_t n_target_rows,
                      const float* u_acc, const float* u_fin, int32_t* n_acc,
                      int32_t* out_tokens, double* p_lse, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * dspark_schedule_noalloc -- dspark_schedule for callers that cannot allocate
 * device memory.  The paper has no counterpart: this is a deployment variant.
 *
 * Some callers cannot call cudaMalloc or pass a workspace: an engine that
 * replays a fixed memory map reserved once at start-up (allocating inside the
 * decode loop would break the plan, or the CUDA graph that replays it), or a
 * plugin inside a host framework that owns the device heap.  This entry point
 * runs the same scheduler with its scratch in a static device array inside
 * the library instead of `ws`; it calls no cudaMalloc / cudaFree.
 *
 * Arguments and results are those of dspark_schedule, except:
 *   dev_status  [1] uint32 or NULL   device status word the kernels OR
 *                                    DSPARK_DEVFLAG_* bits into (caller-owned,
 *                                    zero it first); NULL = not reported
 * Limits:
 *   R * gamma <= 32768, else DSPARK_ERR_INVALID_ARG with a reason in
 *   dspark_last_error().  The static array (about 384 KiB) stays resident on
 *   every GPU that loads the library until the process exits.
 *   All calls share that array: calls that overlap on the GPU (different
 *   streams or host threads) race and must be serialised by the caller.
 *   The first call on each device resolves the array's address while that
 *   device is current (cudaGetSymbolAddress); make it before any stream
 *   capture.
 */
int dspark_schedule_noalloc(int R, int gamma, const float* a, const float* sps, int n_sps,
                            int early_stop, int max_B, int32_t* ell, int32_t* row_off,
                            int32_t* B_out, double* E_out, uint32_t* dev_status, void* stream);

/*
 * dspark_check_wait_timeout -- diagnostic of the library's bounded waits.
 * The pages have no counterpart: this exercises the failure handling.
 *
 * Every on-chip wait in the library's kernels (an mbarrier phase, the
 * persistent draft's grid barrier) gives up after a time limit, ORs
 * DSPARK_DEVFLAG_TIMEOUT into the status word and lets the kernel return, so
 * a stalled pipeline never leaves the GPU hung.  This call runs those same
 * two waits in a one-block kernel against barriers that nothing completes,
 * each with a limit of limit_us microseconds (1 .. 10^6).  Once the stream
 * reaches it, the status word has DSPARK_DEVFLAG_TIMEOUT set and the device
 * stays usable.  It uses the first 256 bytes of `ws` (at least 256 bytes,
 * 256-byte aligned): the status word at byte 0, a counter at byte 64 that it
 * leaves at zero, and at byte 128 two int32 results (1 if the mbarrier wait
 * claimed success -- it must not -- and 1 if the grid wait gave up).
 * Errors: DSPARK_ERR_INVALID_ARG (limit out of range, NULL or misaligned
 * ws), DSPARK_ERR_WORKSPACE, DSPARK_ERR_CUDA.
 */
int dspark_check_wait_timeout(int limit_us, void* ws, size_t ws_bytes, void* stream);

/*
 * Launch counting and kernel tracing (measurement support; no counterpart on
 * the pages).  Host-side only: these calls create CUDA events once and never
 * allocate device memory.
 *
 * dspark_launch_count  total kernel launches this process has issued through
 *                      the library (a stream capture counts its launches once).
 * dspark_trace_start   reset the per-kernel totals and bracket every following
 *                      launch with a pair of CUDA events on its stream (up to
 *                      8192 launches; inside a stream capture the records
 *                      become graph nodes and fire on every replay).
 * dspark_trace_stop    stop bracketing new launches (recorded pairs stay valid).
 * dspark_trace_collect wait for every recorded pair and add its elapsed time
 *                      to the totals of its kernel; returns the number of
 *                      pairs read, or -1 on a CUDA error.  Call it once after
 *                      each replay of a traced graph.
 * dspark_trace_kinds / dspark_trace_get  the kernel names and their
 *                      (launches, total milliseconds).
 */
long long dspark_launch_count(void);
int dspark_trace_start(void);
int dspark_trace_stop(void);
int dspark_trace_collect(void);
int dspark_trace_kinds(void);
int dspark_trace_get(int i, const char** name, long long* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
