// Device helpers and internal launch interfaces shared by the libdspark
// kernels.  Nothing here is part of the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

namespace dspark {

// Vocabulary tile of the draft / final-sampling partial sums, and chunk of
// the verification row pass.
constexpr int kTileV = 256;
constexpr int kChunkV = 4096;  // tokens per warp item of the verification row pass
// Fixed-point fraction bits: weights relative to a tile's power-of-two
// reference (each <= 1) are summed exactly as integers in units of 2^-kFixRel;
// normalised weights (p, residual) in units of 2^-kFixAbs.
constexpr int kFixRel = 40;
constexpr int kFixAbs = 60;
constexpr int kMaxGamma = 32;

constexpr uint32_t kFlagTokenRange = 0x1u;
constexpr uint32_t kFlagNonFinite = 0x2u;
constexpr uint32_t kFlagRowRange = 0x4u;
constexpr uint32_t kFlagSpsRange = 0x8u;
constexpr uint32_t kFlagWaitTimeout = 0x10u;  // a bounded on-chip wait gave up

// log2(e) as a double-float pair (hi = fp32 rounding, lo = remainder) so that
// y * log2(e) / T carries no shared fp32 rounding of the constant.
struct ScalePair {
  float hi, lo;
};

__host__ inline ScalePair make_scale(double c) {
  ScalePair s;
  s.hi = (float)c;
  s.lo = (float)(c - (double)s.hi);
  return s;
}

// y * (hi + lo); -inf (a masked or impossible token) stays -inf, where the
// two-term product would give inf - inf = NaN whenever lo < 0.
__device__ __forceinline__ float scaled(float y, ScalePair s) {
  return y > -INFINITY ? fmaf(y, s.hi, y * s.lo) : -INFINITY;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ float ldf(const T* p, size_t i) {
  return to_f32<T>(p[i]);
}

__device__ __forceinline__ void set_flag(uint32_t* status, uint32_t f) {
  atomicOr(status, f);
}

// ---------------------------------------------------------------- reductions

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index) arg-max with the lowest index winning ties.
struct ArgMax {
  float v;
  int i;
};

// max(a, b) that returns NaN when either operand is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax b;
    b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    a = better(a, b);
  }
  return a;
}

// Block-wide reductions for blockDim.x a multiple of 32 (<= 1024).  `sh`
// must hold 32 elements; every thread receives the result.
template <typename T>
__device__ T block_sum(T v, T* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  T t = lane < nw ? sh[lane] : T(0);
  return warp_sum(t);
}

__device__ inline float block_max(float v, float* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  float t = lane < nw ? sh[lane] : -INFINITY;
  return warp_max(t);
}

__device__ inline ArgMax block_argmax(ArgMax a, ArgMax* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  a = warp_argmax(a);
  __syncthreads();
  if (lane == 0) sh[wid] = a;
  __syncthreads();
  ArgMax t = lane < nw ? sh[lane] : ArgMax{-INFINITY, 0x7fffffff};
  return warp_argmax(t);
}

__device__ inline int block_min_int(int v, int* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = __reduce_min_sync(0xffffffffu, v);
  __syncthreads();
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  return __reduce_min_sync(0xffffffffu, lane < nw ? sh[lane] : 0x7fffffff);
}

__device__ inline int block_max_int(int v, int* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = __reduce_max_sync(0xffffffffu, v);
  __syncthreads();
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  return __reduce_max_sync(0xffffffffu, lane < nw ? sh[lane] : -0x7fffffff);
}

// Inclusive block scan (Hillis-Steele over warps); `sh` holds 32 elements.
template <typename T>
__device__ T block_inclusive_scan(T v, T* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  __syncthreads();
  if (lane == 31) sh[wid] = v;
  __syncthreads();
  if (wid == 0) {
    T s = lane < nw ? sh[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < nw) sh[lane] = s;
  }
  __syncthreads();
  if (wid > 0) v += sh[wid - 1];
  return v;
}

// ---------------------------------------------------------------- tracing
// Kernel kinds, in the order of the names in trace.cu.
enum KernelKind {
  kKindBias = 0,
  kKindDraftPartial,
  kKindDraftFinish,
  kKindConfidence,
  kKindSchedule,
  kKindVerifyRows,
  kKindVerifyDecide,
  kKindFinalPartial,
  kKindFinalPick,
  kKindDraftFusedTc,
  kKindDraftPersistent,
  kKindFinalTc,
  kKindWaitCheck,
  kKindRnnState,
  kKindCount
};

// Programmatic dependent launch: a kernel launched with launch_pdl may start
// while the previous kernel on its stream is still draining; it calls
// grid_dependency_wait() before reading anything that kernel wrote (a no-op
// when launched without the attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

void trace_begin(int kind, cudaStream_t st);
void set_error_text(const char* msg);  // the text dspark_last_error() returns
void trace_end(int kind, cudaStream_t st);

// Launch set-up that belongs to a device, not to the process (launch_state.cu).
// Each is resolved on the calling thread's current device, once per device,
// under a lock, so a process that drives several GPUs or calls from several
// host threads sets every device up itself.
int sm_count();  // multiprocessors of the current device
// Raises `func`'s dynamic shared-memory limit on the current device to at
// least `bytes` (cudaFuncSetAttribute is per device).
cudaError_t ensure_smem_attr(const void* func, int bytes);
// Resident blocks of `func` per multiprocessor of the current device at
// `threads` threads and `dyn_smem` bytes of dynamic shared memory, cached per
// (device, func, threads, dyn_smem); 0 if the query fails.
int blocks_per_sm(const void* func, int threads, size_t dyn_smem);

// Every kernel launch: counted, and bracketed by trace events when tracing.
#define DSPARK_LAUNCH(kind, st, ...)   \
  do {                                 \
    ::dspark::trace_begin((kind), (st)); \
    __VA_ARGS__;                       \
    ::dspark::trace_end((kind), (st));   \
  } while (0)

// ---------------------------------------------------------------- launchers
// (defined in the kernel translation units; all enqueue on `st`)

// The confidence head and the prefix scheduler, evaluated by the persistent
// draft kernel after its last position when the caller asks for the three
// stages in one call (dspark_draft_schedule) and the shapes allow it (see
// draft_fuse_supported).  Same arithmetic as the confidence and scheduler
// kernels, so the results are bit-identical to the separate calls.
struct DraftFuse {
  int d;
  const void* h;      // [R][gamma][d] bf16, NULL when c_in is given
  const float* w;     // [d + r]
  const void* E1;     // [V][r] bf16
  const float* sts;   // [gamma]
  const float* c_in;  // [R][gamma] or NULL
  float* c_out;       // [R][gamma]
  float* a_out;       // [R][gamma]
  float* hpart;       // [R * gamma][32] scratch: lane partials of w_h . h
  int early_stop, imax;
  const float* sps;
  int32_t* rank;      // [R * gamma] scratch
  unsigned long long* tkey;  // [R * gamma + 1] scratch: Theta_i order keys by rank
  long long* spre;           // [R * gamma + 1] scratch: exact prefixes S_i by rank
  int32_t* ell;
  int32_t* row_off;
  int32_t* B_out;
  double* E_out;
};
constexpr int kFuseMaxCandidates = 8192;

struct DraftArgs {
  int R, gamma, V, r, dt;
  float T;
  const void* z;
  const void* E;
  const void* Wt;
  const int32_t* anchor;
  const float* u;
  int32_t* tokens;
  double* q_lse;
  float* q_tok;
  uint32_t* status;
  float* bias;      // [R][V] scratch
  double* part;     // [R][n_tiles] scratch (greedy: ArgMax pairs)
  float* sub;       // [R][n_tiles][8] 16-token group sums of 128-token partials
  unsigned* grid_counter;  // grid-barrier counter of the persistent draft kernel
  void* stage;             // [R][r] bf16: E rows of the latest drafted tokens
  const DraftFuse* fuse = nullptr;  // confidence + scheduler in the same launch, if possible
  int* fused = nullptr;             // out: 1 when the launch included them
  // RNN head (when U is set): U [r][r] in the table's type, S [R][gamma][r]
  // the states; position k's bias row is S[n][k] instead of E[x_{k-1}]
  const void* U = nullptr;
  void* S = nullptr;
};
cudaError_t launch_draft(const DraftArgs& a, cudaStream_t st);
// Whether the persistent draft can also evaluate the confidence head and the
// scheduler for these arguments (host-side shape and alignment checks).
bool draft_fuse_supported(const DraftArgs& a, const DraftFuse& f);
cudaError_t launch_draft_persistent_tc(const DraftArgs& a, cudaStream_t st);

// Tensor-core path of the draft (bf16, r % 8 == 0, r <= 256, 16-byte aligned
// operands): the fused bias GEMM + partial pass for draft position k.
bool draft_tc_supported(const DraftArgs& a);
bool tc_shape_supported(int dt, int V, int r, const void* a, const void* b, const void* c);
// bias[n][v] = E[prev[n * prev_stride]] . Wt[v] on the tensor cores; rows
// prev >= prev_limit (or < -1) are flagged and zero.
cudaError_t launch_bias_tc(int R, int V, int r, const void* E, const void* Wt,
                           const int32_t* prev, int prev_stride, int prev_limit, float* bias,
                           uint32_t* status, cudaStream_t st);
cudaError_t launch_draft_partial_tc(const DraftArgs& a, int k, const int32_t* prev,
                                    int prev_stride, cudaStream_t st);

struct ConfArgs {
  int R, gamma, d, r, V, dt;
  const void* h;
  const float* w;
  const void* E1;
  const int32_t* anchor;
  const int32_t* tokens;
  const float* sts;
  const float* c_in;
  float* c_out;
  float* a_out;
  uint32_t* status;
};
cudaError_t launch_confidence(const ConfArgs& a, cudaStream_t st);

struct SchedArgs {
  int R, gamma, n_sps, early_stop, max_B;
  int imax;  // last admissible candidate count (R * gamma, or max_B - R)
  const float* a;
  const float* sps;
  int32_t* ell;
  int32_t* row_off;
  int32_t* B_out;
  double* E_out;
  uint32_t* status;
  int32_t* rank;             // [N] scratch: each candidate's position in the order
  unsigned long long* keys;  // [2N] scratch: the radix sort's ping-pong buffers
};

// Scheduler scratch for N candidates: rank (4N) then keys (16N), each rounded
// up to 256 bytes.
constexpr size_t sched_scratch_bytes(size_t N) {
  return ((N * 4 + 255) & ~(size_t)255) + ((N * 16 + 255) & ~(size_t)255);
}
cudaError_t launch_schedule(const SchedArgs& a, cudaStream_t st);
// Capacity (asynchronous) scheduling: the batch is the first
// min(max(capacity[0] - R, 0), R*gamma) candidates; capacity is device memory.
cudaError_t launch_schedule_async(const SchedArgs& a, const int32_t* capacity, cudaStream_t st);

// The bounded-wait diagnostic (draft_tc.cu): waits that nothing completes,
// each giving up after limit_ns.
cudaError_t launch_wait_check(uint64_t limit_ns, unsigned* ctr, uint32_t* status, int* out,
                              cudaStream_t st);

// 1/S for a row normaliser S, as (hi + lo) * 2^e with hi in [0.5, 1): the
// final pass scales it by a tile's power-of-two reference with exponent
// arithmetic only.  hi = lo = 0 means "no such row".
struct InvPair {
  float hi, lo;
  int e;
};

struct VerifyState {
  int n_acc;
  int mode;       // 0 bonus, 1 residual
  int final_row;  // target row of the final draw
  int prev;       // token before the rejected position (residual), -1 none
  InvPair ip;     // 1 / Sp, Sp = sum_v exp(target_row / T) of the final row
  InvPair iq;     // 1 / Sq, Sq = sum_v exp(y_draft) of the rejected position
                  // (zero when not a residual draw)
};

// Fast base-2 exponential (MUFU ex2, flush-to-zero; results below 2^-126
// are far below every fixed-point unit used here).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// y * (hi + lo) clamped to >= -3e38: -inf and NaN inputs become a finite
// "no mass" value (their exponential is 0) instead of NaN.
__device__ __forceinline__ float scaled_clamped(float y, ScalePair s) {
  return fmaxf(fmaf(y, s.hi, y * s.lo), -3.0e38f);
}

// Eight consecutive elements starting at p[v0] as fp32 (16/32-byte vector
// loads when all eight lie below V, else masked scalar loads with `fill`).
template <typename T>
__device__ __forceinline__ void load8(const T* p, int v0, int V, float (&o)[8], float fill);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, int v0, int V,
                                                     float (&o)[8], float fill) {
  if (v0 + 8 <= V) {
    const uint4 q = *reinterpret_cast<const uint4*>(p + v0);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = v0 + i < V ? __bfloat162float(p[v0 + i]) : fill;
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, int v0, int V, float (&o)[8],
                                             float fill) {
  if (v0 + 8 <= V) {
    const float4 a = *reinterpret_cast<const float4*>(p + v0);
    const float4 b = *reinterpret_cast<const float4*>(p + v0 + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = v0 + i < V ? p[v0 + i] : fill;
  }
}

// Exact warp sum of non-negative 64-bit values whose total is below 2^63:
// three 21-bit limbs, each summed by one reduction instruction.
__device__ __forceinline__ long long warp_sum_nonneg_ll(long long v) {
  const unsigned long long u = (unsigned long long)v;
  const unsigned long long a = __reduce_add_sync(0xffffffffu, (unsigned)(u >> 42));
  const unsigned long long b = __reduce_add_sync(0xffffffffu, (unsigned)(u >> 21) & 0x1fffffu);
  const unsigned long long c = __reduce_add_sync(0xffffffffu, (unsigned)u & 0x1fffffu);
  return (long long)((a << 42) + (b << 21) + c);
}

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct VerifyArgs {
  int R, gamma, V, r, dt;
  float T;
  const void* z;
  const void* E;  // Markov table [V][r]; RNN head (anchor null): the states [R][gamma][r]
  const void* Wt;
  const int32_t* anchor;
  const int32_t* tokens;
  const double* q_lse;
  const float* q_tok;
  const int32_t* ell;
  const int32_t* row_off;
  const void* target;
  long long n_rows;
  const float* u_acc;
  const float* u_fin;
  int32_t* n_acc;
  int32_t* out_tokens;
  double* p_lse;
  uint32_t* status;
  double* row_part;      // [R*(gamma+1)][n_chunks]
  VerifyState* vstate;   // [R]
  float* bias;           // [R][V]
  long long* fin_part;   // [R][n_tiles][2]
  int32_t* prev;         // [R]
  int* vcnt;             // [R] row-pass items counted per request, zero between calls
};
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t st);
// Final-draw partial sums on the tensor cores: fin_part[R][ceil(V / 128)][2]
// (residual, p) in units of 2^-60, the bias of each rejected position formed
// in TMEM (bf16, tensor-core shapes only).
cudaError_t launch_final_tc(const VerifyArgs& a, const VerifyState* vstate, long long* fin_part,
                            cudaStream_t st);

// CUDA-core Markov bias: bias[n][v] = sum_i E[prev[n]][i] * Wt[v][i] for the
// n = 0..R-1 rows whose previous token is prev_base[n * prev_stride]
// (negative = zero row; at or above prev_limit: flagged, zero row).  With
// prev_base null the row of request n is n * prev_stride (the RNN states).
cudaError_t launch_bias(int R, int V, int r, int dt, const void* E, const void* Wt,
                        const int32_t* prev_base, int prev_stride, int prev_limit, float* bias,
                        uint32_t* status, cudaStream_t st);

// RNN head, draft position k: S[n][k] = round(tanh(pre)), pre[j] in fp32 =
// E[x_{k-1}][j] (0 when x_{k-1} < 0; x_{-1} the anchor, x_{k-1} = tokens[n][k-1])
// followed by the fused multiply-adds S[n][k-1][i] * U[i][j], i ascending
// (none at k = 0); tanh in double; rounded to the table's type (dt).
cudaError_t launch_rnn_state(int R, int gamma, int r, int dt, int k, const void* E, const void* U,
                             const int32_t* anchor, const int32_t* tokens, int V, void* S,
                             uint32_t* status, cudaStream_t st);

// ------------------------------------------------- integer-built doubles
// The FP64 pipe of this part is narrow, so the hot paths build and take
// apart doubles with integer operations only.

// acc * 2^e2 as a double, for acc >= 0 (exact while acc < 2^53; wider values
// are truncated to 53 bits).  Results below the normal range are 0.
__device__ __forceinline__ double fix_to_double(long long acc, int e2) {
  if (acc <= 0) return 0.0;
  const int msb = 63 - __clzll(acc);
  const int ex = msb + e2;
  if (ex < -1022) return 0.0;
  if (ex > 1023) return __longlong_as_double(0x7ff0000000000000ll);
  unsigned long long m = (unsigned long long)acc;
  m = msb >= 52 ? (m >> (msb - 52)) : (m << (52 - msb));
  return __longlong_as_double((long long)(((unsigned long long)(ex + 1023) << 52) |
                                          (m & 0x000fffffffffffffull)));
}

// Unbiased binary exponent of a finite x > 0 (x in [2^e, 2^(e+1))); INT_MIN
// for zero, negative and subnormal x.
__device__ __forceinline__ int double_exponent(double x) {
  const long long b = __double_as_longlong(x);
  const int be = (int)((b >> 52) & 0x7ff);
  return (b <= 0 || be == 0) ? INT_MIN : be - 1023;
}

// floor(x / 2^g) for finite x >= 0; the caller keeps the result below 2^62.
__device__ __forceinline__ long long double_to_fix(double x, int g) {
  const long long b = __double_as_longlong(x);
  const int be = (int)((b >> 52) & 0x7ff);
  if (b <= 0 || be == 0) return 0;
  const long long m = (b & 0x000fffffffffffffll) | 0x0010000000000000ll;
  const int sh = be - 1075 - g;  // x = m * 2^(be - 1075)
  if (sh >= 0) return sh > 9 ? 0x3fffffffffffffffll : (m << sh);
  return -sh >= 63 ? 0 : (m >> -sh);
}

// x * 2^k for a finite fp32 x by exponent arithmetic; results below the
// normal range flush to 0.
__device__ __forceinline__ float scale_pow2(float x, int k) {
  if (x == 0.0f || k < -252) return 0.0f;
  if (k > 254) k = 254;
  // two steps so that every k in range gives a normal factor
  const int k1 = k / 2, k2 = k - k1;
  return x * __int_as_float((k1 + 127) << 23) * __int_as_float((k2 + 127) << 23);
}

// floor(u * F) exactly, for u in [0, 1) and 0 <= F < 2^62, from u's bits
// (u = m * 2^(E - 150)) and a 128-bit integer product: no conversion
// instructions (those between floats and 64-bit integers are slow here).
// u >= 1 (outside the contract) clamps to F.
__device__ __forceinline__ long long floor_mul(float u, long long F) {
  if (!(u > 0.0f)) return 0;
  if (!(u < 1.0f)) return F;
  const uint32_t b = __float_as_uint(u);
  const int E = (int)(b >> 23);  // u > 0: no sign bit
  const unsigned long long m = E ? ((b & 0x7fffffu) | 0x800000u) : (b & 0x7fffffu);
  const int sh = 150 - (E ? E : 1);  // u = m * 2^-sh, sh > 23 since u < 1
  const unsigned long long lo = m * (unsigned long long)F;
  const unsigned long long hi = __umul64hi(m, (unsigned long long)F);
  if (sh >= 128) return 0;
  if (sh >= 64) return (long long)(hi >> (sh - 64));
  return (long long)((lo >> sh) | (hi << (64 - sh)));
}

// a * b > c * d for non-negative 64-bit operands, exactly (128-bit products).
__device__ __forceinline__ bool mul_gt(unsigned long long a, unsigned long long b,
                                       unsigned long long c, unsigned long long d) {
  const unsigned long long h1 = __umul64hi(a, b), h2 = __umul64hi(c, d);
  return h1 != h2 ? h1 > h2 : a * b > c * d;
}

// ---- Without double instructions.  The FP64 pipe of this GPU is narrow: a
// dependent double division, logarithm or exponential costs on the order of
// a microsecond, so paths that feed a per-request decision use the integer
// and fp32 forms below.

// v * 2^e2 as a float, v's top 24 bits (truncated); below the normal range: 0.
__device__ __forceinline__ float fix_to_float(long long v, int e2) {
  if (v == 0) return 0.f;
  const bool neg = v < 0;
  const unsigned long long a = neg ? 0ull - (unsigned long long)v : (unsigned long long)v;
  const int msb = 63 - __clzll(a);
  const uint32_t top = msb >= 23 ? (uint32_t)(a >> (msb - 23)) : (uint32_t)(a << (23 - msb));
  const int ex = msb + e2;  // |value| = 1.top * 2^ex
  if (ex < -126) return 0.f;
  if (ex > 127) return neg ? -INFINITY : INFINITY;
  return __uint_as_float((neg ? 0x80000000u : 0u) | ((uint32_t)(ex + 127) << 23) | (top & 0x7fffffu));
}

// Natural logarithm of F * 2^g (F > 0) in fp32 arithmetic, to about 3e-7
// relative.  Away from 1 (value outside [0.5, 2), |log| > 0.69): the binary
// exponent times ln 2 (split so that the large product is exact) plus the
// logarithm of F's top 24 bits normalised to [1, 2).  Near 1: log1p of
// value - 1, formed exactly in fixed point, so a logarithm near 0 keeps
// its relative precision.
__device__ __forceinline__ float fix_log(long long F, int g) {
  const int msb = 63 - __clzll(F);
  if ((msb + g == 0 || msb + g == -1) && g <= 0 && g >= -62) {
    const long long u = F - (1ll << -g);  // (value - 1) * 2^-g, exact
    return log1pf(fix_to_float(u, g));
  }
  const uint32_t top =
      msb >= 23 ? (uint32_t)(F >> (msb - 23)) : (uint32_t)((unsigned long long)F << (23 - msb));
  const float m = __uint_as_float(0x3f800000u | (top & 0x7fffffu));  // [1, 2)
  const float A = (float)(msb + g);
  constexpr float kLn2Hi = 0.693115234375f;        // 2839 / 4096: A * kLn2Hi is exact
  constexpr float kLn2Lo = 3.1946184945309417e-05f;  // ln 2 - kLn2Hi
  return fmaf(A, kLn2Hi, fmaf(A, kLn2Lo, logf(m)));
}

// Natural logarithm of a positive finite double x (as fix_log, from its
// bits); 0 or negative: -inf.
__device__ __forceinline__ float dbl_log(double x) {
  const long long b = __double_as_longlong(x);
  const int be = (int)((b >> 52) & 0x7ff);
  if (b <= 0 || be == 0) return -INFINITY;
  return fix_log((b & 0x000fffffffffffffll) | 0x0010000000000000ll, be - 1075);
}

// 1 / (F * 2^g) as an InvPair (F > 0; else the zero pair): an fp32
// reciprocal of F's top bits, corrected by the exactly computed residual
// 1 - x * r0 (128-bit integer product), relative error about 2^-45.
__device__ __forceinline__ InvPair inv_fix(long long F, int g) {
  InvPair r{0.f, 0.f, 0};
  if (F <= 0) return r;
  const int msb = 63 - __clzll(F);
  const unsigned long long Fn = (unsigned long long)F << (63 - msb);  // x = Fn / 2^64 in [0.5, 1)
  const float xf = (float)(uint32_t)(Fn >> 40) * 5.9604644775390625e-08f;  // top 24 bits * 2^-24
  const float r0 = 1.0f / xf;                                             // (1, 2]
  const unsigned long long Mr = (unsigned long long)__float_as_uint(r0) == 0x40000000u
                                    ? (1ull << 24)
                                    : (((__float_as_uint(r0) & 0x7fffffu) | 0x800000u));  // r0 = Mr * 2^-23
  // D = 2^87 - Fn * Mr = (1 - x * r0) * 2^87, |D| < 2^66
  const unsigned long long plo = Fn * Mr, phi = __umul64hi(Fn, Mr);
  const unsigned long long dlo = 0ull - plo;
  const unsigned long long dhi = (1ull << 23) - phi - (plo != 0 ? 1ull : 0ull);
  const long long d35 = (long long)((dlo >> 35) | (dhi << 29));  // D >> 35 (arithmetic)
  const float eps = (float)(int)d35 * 2.220446049250313e-16f;    // D * 2^-87 = (D >> 35) * 2^-52
  r.hi = 0.5f * r0;
  r.lo = 0.5f * r0 * eps;
  r.e = -(msb + g);  // 1 / (F 2^g) = (r0 + r0 eps) / 2 * 2^-(msb + g)
  if (r.hi >= 1.0f) {
    r.hi *= 0.5f;
    r.lo *= 0.5f;
    r.e += 1;
  }
  return r;
}

// exp(-x) for a double x as an InvPair (hi in [0.5, 1), lo = 0, e), without
// double instructions: t = x log2(e) formed in fixed point from x's bits
// (64-bit constant, 128-bit product, 32 fraction bits), then
// 2^-t = 2^(1 - frac) / 2 * 2^-floor(t) with exp2f.  Relative error about
// 3e-7.  x = NaN, +-inf or |x log2 e| >= 2^31: the zero pair.
__device__ __forceinline__ InvPair exp_neg_pair(double x) {
  InvPair r{0.f, 0.f, 0};
  const unsigned long long xb = (unsigned long long)__double_as_longlong(x);
  const int E = (int)((xb >> 52) & 0x7ff);
  if (E == 0x7ff) return r;
  if (E == 0) {  // zero or subnormal: exp(-x) = 1 to fp32 precision
    r.hi = 0.5f;
    r.e = 1;
    return r;
  }
  const unsigned long long xm = (xb & 0x000fffffffffffffull) | 0x0010000000000000ull;
  constexpr unsigned long long kLog2E = 6653256548922161246ull;  // round(log2(e) * 2^62)
  const unsigned long long plo = xm * kLog2E, phi = __umul64hi(xm, kLog2E);
  // t * 2^32 = P * 2^(E - 1075 - 62 + 32) = P >> (1105 - E)
  const int sh = 1105 - E;
  if (sh < 33) return r;  // t >= 2^31
  unsigned long long T;
  if (sh >= 128) {
    T = 0;
  } else if (sh >= 64) {
    T = phi >> (sh - 64);
  } else {
    if ((phi >> sh) != 0) return r;  // P >> sh does not fit 64 bits: t >= 2^32
    T = (plo >> sh) | (phi << (64 - sh));
  }
  if (T >> 63) return r;  // t >= 2^31
  const long long k = (long long)(T >> 32);
  const uint32_t f = (uint32_t)T;  // fraction of t in 2^-32 units
  const bool neg = (xb >> 63) != 0;  // x < 0: exp(-x) = 2^+t
  if (!neg) {
    // 2^-t = (2^(1 - f 2^-32) / 2) * 2^-k, 2^(1 - .) in (1, 2]
    const float fp = 1.0f - (float)f * 2.3283064365386963e-10f;
    r.hi = 0.5f * exp2f(fp);
    r.e = (int)-k;
  } else {
    // 2^t = (2^(f 2^-32) / 2) * 2^(k + 1), 2^(.) in [1, 2)
    r.hi = 0.5f * exp2f((float)f * 2.3283064365386963e-10f);
    r.e = (int)k + 1;
  }
  if (r.hi >= 1.0f) {
    r.hi *= 0.5f;
    r.e += 1;
  }
  return r;
}

}  // namespace dspark
