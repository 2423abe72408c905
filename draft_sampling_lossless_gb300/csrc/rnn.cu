// RNN sequential head: the recurrent state of the draft.
//
// "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation" (news article), innovation 1, second stage: besides the Markov
// head (a low-rank table of the previous token) the sequential head can be an
// RNN that keeps a recurrent state and so sees the whole prefix of the block;
// "DSpark.让每一轮计算，多走几步" (explainer), Markov-head panel: the RNN head
// accumulates the prefix inside the block.  The pages give no formula; this
// library takes an Elman recurrence in the Markov head's shapes,
//   s_k = tanh(E[x_{k-1}] + s_{k-1} U),  s_{-1} = 0,  bias_k = s_k W,
// so that U = 0 leaves a one-token memory.
//
// The state is stored in the table's type and feeds the tensor-core bias
// GEMM like an E row.  Its rounding is a quantisation, so the arithmetic
// before it is fixed: pre[j] in fp32 starts from E[x_{k-1}][j] and adds the
// fused multiply-adds s_{k-1}[i] * U[i][j] for i ascending; tanh in double;
// one rounding from double to bf16 (or fp32).  Any implementation that keeps
// these steps stores the same state bits (up to a 1-ulp difference between
// double tanh implementations landing on a rounding boundary, about 2^-45 a
// value).
#include "common.cuh"
#include "rnn.cuh"

namespace dspark {

namespace {

constexpr int kRnnMaxR = 1024;  // largest rank

constexpr int kRnnCols = 32;  // columns of S a block computes (one per lane)
constexpr int kRnnReqs = 8;   // requests a block computes (one per warp)

size_t rnn_smem_bytes(int r, size_t esz) {
  return (size_t)r * kRnnCols * esz + (size_t)kRnnReqs * r * sizeof(float);
}

// Block (bx, by): columns j = 32 bx + lane of requests n = 8 by + warp.  The
// block's 32-column slice of U and the previous states of its 8 requests
// (zero at k = 0, where the same chain of fused multiply-adds adds zero
// products) are staged in shared memory; each thread then runs its column's
// chain: lanes read consecutive U entries of a row, the state entry is a
// broadcast.
template <typename T>
__global__ void __launch_bounds__(256) rnn_state_kernel(int R, int gamma, int r, int k, int V,
                                                        const T* __restrict__ E,
                                                        const T* __restrict__ U,
                                                        const int32_t* __restrict__ anchor,
                                                        const int32_t* __restrict__ tokens,
                                                        T* __restrict__ S, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char rnn_smem[];
  T* Us = reinterpret_cast<T*>(rnn_smem);                                  // [r][32]
  float* sp = reinterpret_cast<float*>(rnn_smem + (size_t)r * kRnnCols * sizeof(T));  // [8][r]
  const int j0 = blockIdx.x * kRnnCols, n0 = blockIdx.y * kRnnReqs;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // the U slice: 16-byte loads when the rows allow them, else element loads;
  // eight loads in flight per thread before their stores
  constexpr int kGpr = kRnnCols * (int)sizeof(T) / 16;  // 16-byte granules a slice row
  if ((r * sizeof(T)) % 16 == 0 && ((uintptr_t)U & 15) == 0 && j0 + kRnnCols <= r) {
    const int ng = r * kGpr;
    for (int base = 0; base < ng; base += 256 * 8) {
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int g = base + tid + 256 * q;
        if (g < ng) {
          const int i = g / kGpr, c = g - i * kGpr;
          v[q] = reinterpret_cast<const uint4*>(U + (size_t)i * r + j0)[c];
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int g = base + tid + 256 * q;
        if (g < ng) reinterpret_cast<uint4*>(Us)[g] = v[q];
      }
    }
  } else {
    const int ne = r * kRnnCols;
    for (int base = 0; base < ne; base += 256 * 8) {
      T v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = base + tid + 256 * q;
        const int i = e / kRnnCols, c = e - i * kRnnCols;
        v[q] = (e < ne && j0 + c < r) ? U[(size_t)i * r + j0 + c] : T(0.f);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = base + tid + 256 * q;
        if (e < ne) Us[e] = v[q];
      }
    }
  }
  {
    const int ne = kRnnReqs * r;
    for (int base = 0; base < ne; base += 256 * 8) {
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = base + tid + 256 * q;
        const int m = e / r, i = e - m * r;
        const int n = n0 + m;
        v[q] = (e < ne && k > 0 && n < R) ? to_f32<T>(S[((size_t)n * gamma + k - 1) * r + i])
                                          : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = base + tid + 256 * q;
        if (e < ne) sp[e] = v[q];
      }
    }
  }
  __syncthreads();
  const int n = n0 + w, j = j0 + lane;
  if (n >= R || j >= r) return;
  int x = k == 0 ? anchor[n] : tokens[(size_t)n * gamma + k - 1];
  if (x >= V || x < -1) {
    if (j == 0) set_flag(status, kFlagTokenRange);
    x = -1;
  }
  float acc = x >= 0 ? to_f32<T>(E[(size_t)x * r + j]) : 0.f;
  const float* s = sp + (size_t)w * r;
  // pre[j] = E[x][j], then + s[i] * U[i][j] for i ascending, one fused
  // multiply-add each
#pragma unroll 8
  for (int i = 0; i < r; ++i) acc = fmaf(s[i], to_f32<T>(Us[i * kRnnCols + lane]), acc);
  rnn::store_state(S + ((size_t)n * gamma + k) * r + j, acc);
}

}  // namespace

cudaError_t launch_rnn_state(int R, int gamma, int r, int dt, int k, const void* E, const void* U,
                             const int32_t* anchor, const int32_t* tokens, int V, void* S,
                             uint32_t* status, cudaStream_t st) {
  if (r > kRnnMaxR) return cudaErrorInvalidValue;
  const dim3 grid((r + kRnnCols - 1) / kRnnCols, (R + kRnnReqs - 1) / kRnnReqs);
  cudaError_t e;
  if (dt == 0) {
    const size_t smem = rnn_smem_bytes(r, 2);
    e = ensure_smem_attr((const void*)rnn_state_kernel<__nv_bfloat16>, (int)rnn_smem_bytes(kRnnMaxR, 2));
    if (e != cudaSuccess) return e;
    DSPARK_LAUNCH(kKindRnnState, st,
                  rnn_state_kernel<__nv_bfloat16><<<grid, 256, smem, st>>>(
                      R, gamma, r, k, V, (const __nv_bfloat16*)E, (const __nv_bfloat16*)U, anchor,
                      tokens, (__nv_bfloat16*)S, status));
  } else {
    const size_t smem = rnn_smem_bytes(r, 4);
    e = ensure_smem_attr((const void*)rnn_state_kernel<float>, (int)rnn_smem_bytes(kRnnMaxR, 4));
    if (e != cudaSuccess) return e;
    DSPARK_LAUNCH(kKindRnnState, st,
                  rnn_state_kernel<float><<<grid, 256, smem, st>>>(R, gamma, r, k, V, (const float*)E,
                                                                   (const float*)U, anchor, tokens,
                                                                   (float*)S, status));
  }
  return cudaGetLastError();
}

}  // namespace dspark
