// Semi-autoregressive draft sampling with the Markov head, CUDA-core path.
//
// "DSpark.让每一轮计算，多走几步" (explainer), Markov head panel: a low-rank
// transition table biases the vocabulary scores before every left-to-right
// draw; news article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", innovation 1, second stage.
//
// Per draft position k the step is
//   bias  = E[x_{k-1}] . W                    (launch_bias, CUDA cores)
//   part  = per (request, 256-token tile) sum of 2^(a - ref_tile), a = y*log2(e)/T,
//           summed exactly in fixed point and stored as a double
//   token = inverse CDF over the tiles, then inside the chosen tile
// The fp32 path (and the tiny workload) uses this file end to end; the bf16
// path runs the tensor-core kernels of draft_tc.cu and the shared finish.
#include "common.cuh"
#include "finish.cuh"

namespace dspark {

// ---------------------------------------------------------------- bias

template <typename T>
__global__ void __launch_bounds__(256) bias_kernel(int R, int V, int r, const T* __restrict__ E,
                                                   const T* __restrict__ Wt,
                                                   const int32_t* __restrict__ prev_base,
                                                   int prev_stride, int prev_limit,
                                                   float* __restrict__ bias, uint32_t* status) {
  // Tile: 64 vocabulary columns x 32 requests, K in chunks of 32.
  __shared__ float Es[32][33];
  __shared__ float Ws[64][33];
  __shared__ int prev_s[32];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16
  const int v0 = blockIdx.x * 64, n0 = blockIdx.y * 32;
  if (threadIdx.x < 32) {
    int n = n0 + threadIdx.x;
    int p = -1;
    if (n < R && prev_base == nullptr) {
      p = n * prev_stride;  // the RNN state of request n
    } else if (n < R) {
      p = prev_base[(size_t)n * prev_stride];
      if (p >= prev_limit || p < -1) {
        set_flag(status, kFlagTokenRange);
        p = -1;
      }
    }
    prev_s[threadIdx.x] = p;
  }
  float acc[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  __syncthreads();
  for (int k0 = 0; k0 < r; k0 += 32) {
    for (int e = threadIdx.x; e < 32 * 32; e += 256) {
      int row = e >> 5, col = e & 31;
      int p = prev_s[row];
      float val = 0.f;
      if (p >= 0 && k0 + col < r) val = ldf(E, (size_t)p * r + k0 + col);
      Es[row][col] = val;
    }
    for (int e = threadIdx.x; e < 64 * 32; e += 256) {
      int row = e >> 5, col = e & 31;
      int v = v0 + row;
      float val = 0.f;
      if (v < V && k0 + col < r) val = ldf(Wt, (size_t)v * r + k0 + col);
      Ws[row][col] = val;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float ev[2], wv[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) ev[i] = Es[ty * 2 + i][kk];
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = Ws[tx + 16 * j][kk];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ev[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    int n = n0 + ty * 2 + i;
    if (n >= R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int v = v0 + tx + 16 * j;
      if (v < V) bias[(size_t)n * V + v] = acc[i][j];
    }
  }
}

cudaError_t launch_bias(int R, int V, int r, int dt, const void* E, const void* Wt,
                        const int32_t* prev_base, int prev_stride, int prev_limit, float* bias,
                        uint32_t* status, cudaStream_t st) {
  dim3 grid((V + 63) / 64, (R + 31) / 32);
  if (dt == 0)
    DSPARK_LAUNCH(kKindBias, st, bias_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        R, V, r, (const __nv_bfloat16*)E, (const __nv_bfloat16*)Wt, prev_base, prev_stride,
        prev_limit, bias, status));
  else
    DSPARK_LAUNCH(kKindBias, st, bias_kernel<float><<<grid, 256, 0, st>>>(
        R, V, r, (const float*)E, (const float*)Wt, prev_base, prev_stride, prev_limit, bias,
        status));
  return cudaGetLastError();
}

// ---------------------------------------------------------------- partials

// One block per (tile, request): y = z + bias; stochastic: exact tile sum of
// 2^(y*log2e/T - ref) with ref = ceil(max); greedy: (max, lowest argmax).
template <typename T>
__global__ void __launch_bounds__(kTileV) draft_partial_kernel(
    int V, int gamma, int k, int n_tiles, const T* __restrict__ z, const float* __restrict__ bias,
    ScalePair sc, int greedy, double* __restrict__ part, uint32_t* status) {
  __shared__ float shf[32];
  __shared__ long long shl[32];
  __shared__ ArgMax sha[32];
  const int t = blockIdx.x, n = blockIdx.y;
  const int v = t * kTileV + threadIdx.x;
  const bool ok = v < V;
  float y = -INFINITY;
  if (ok) y = ldf(z, ((size_t)n * gamma + k) * V + v) + bias[(size_t)n * V + v];
  if (ok && (isnan(y) || y == INFINITY)) {
    set_flag(status, kFlagNonFinite);
    y = -INFINITY;
  }
  if (greedy) {
    ArgMax am = block_argmax(ArgMax{y, ok ? v : 0x7fffffff}, sha);
    if (threadIdx.x == 0) reinterpret_cast<ArgMax*>(part)[(size_t)n * n_tiles + t] = am;
    return;
  }
  const float a = scaled(y, sc);
  const float amax = block_max(a, shf);
  double S = 0.0;
  if (amax > -INFINITY) {
    const float ref = ceilf(amax);
    float w;
    long long f = (a > -INFINITY) ? rel_fix(a, ref, &w) : 0ll;
    long long tot = block_sum(f, shl);
    S = fix_to_double(tot, (int)ref - kFixRel);
  }
  if (threadIdx.x == 0) part[(size_t)n * n_tiles + t] = S;
}

// One block of 256 threads per request: the finish of draft position k.
template <typename T, int TW>
__global__ void __launch_bounds__(256) draft_finish_kernel(
    int V, int gamma, int k, int n_tiles, const T* __restrict__ z, BiasSrc bsrc, ScalePair sc,
    int greedy, const double* __restrict__ part, const float* __restrict__ u,
    int32_t* __restrict__ tokens, double* __restrict__ q_lse, float* __restrict__ q_tok,
    uint32_t* status, const float* __restrict__ sub) {
  __shared__ FinishScratch s;
  finish_request<T, TW, BlockSync, false>(s, blockIdx.x, V, gamma, k, n_tiles, z, bsrc, sc, greedy, part,
                                   u, tokens, q_lse, q_tok, status, nullptr, sub);
}

template <typename T, int TW>
cudaError_t launch_finish(const DraftArgs& a, int k, const BiasSrc& b, ScalePair sc, bool greedy,
                          cudaStream_t st) {
  const int n_tiles = (a.V + TW - 1) / TW;
  DSPARK_LAUNCH(kKindDraftFinish, st,
                draft_finish_kernel<T, TW><<<a.R, 256, 0, st>>>(
                    a.V, a.gamma, k, n_tiles, (const T*)a.z, b, sc, greedy, a.part, a.u,
                    a.tokens, a.q_lse, a.q_tok, a.status, TW == 128 ? a.sub : nullptr));
  return cudaGetLastError();
}

// RNN head: per position, the state kernel, then the bias and the draw with
// the state rows S[n][k] (row n * gamma of the table S + k * r) as the bias
// rows.
cudaError_t launch_draft_rnn(const DraftArgs& a, cudaStream_t st) {
  const int n_tiles = (a.V + kTileV - 1) / kTileV;
  const bool greedy = a.T == 0.0f;
  const ScalePair sc = make_scale(greedy ? 1.0 : 1.4426950408889634 / (double)a.T);
  const bool tc = draft_tc_supported(a);
  const size_t esz = a.dt == 0 ? 2 : 4;
  for (int k = 0; k < a.gamma; ++k) {
    cudaError_t e = launch_rnn_state(a.R, a.gamma, a.r, a.dt, k, a.E, a.U, a.anchor, a.tokens,
                                     a.V, a.S, a.status, st);
    if (e != cudaSuccess) return e;
    DraftArgs b = a;
    b.E = static_cast<const char*>(a.S) + (size_t)k * a.r * esz;  // row n * gamma: S[n][k]
    if (tc) {
      e = launch_draft_partial_tc(b, k, nullptr, a.gamma, st);
      if (e != cudaSuccess) return e;
      BiasSrc bs{nullptr, (const __nv_bfloat16*)b.E, (const __nv_bfloat16*)a.Wt, nullptr, a.gamma,
                 a.r};
      e = launch_finish<__nv_bfloat16, 128>(a, k, bs, sc, greedy, st);
      if (e != cudaSuccess) return e;
      continue;
    }
    e = launch_bias(a.R, a.V, a.r, a.dt, b.E, a.Wt, nullptr, a.gamma, 0, a.bias, a.status, st);
    if (e != cudaSuccess) return e;
    dim3 g1(n_tiles, a.R);
    BiasSrc bs{a.bias, nullptr, nullptr, nullptr, a.gamma, a.r};
    if (a.dt == 0) {
      DSPARK_LAUNCH(kKindDraftPartial, st,
                    draft_partial_kernel<__nv_bfloat16><<<g1, kTileV, 0, st>>>(
                        a.V, a.gamma, k, n_tiles, (const __nv_bfloat16*)a.z, a.bias, sc, greedy,
                        a.part, a.status));
      e = launch_finish<__nv_bfloat16, kTileV>(a, k, bs, sc, greedy, st);
    } else {
      DSPARK_LAUNCH(kKindDraftPartial, st,
                    draft_partial_kernel<float><<<g1, kTileV, 0, st>>>(
                        a.V, a.gamma, k, n_tiles, (const float*)a.z, a.bias, sc, greedy, a.part,
                        a.status));
      e = launch_finish<float, kTileV>(a, k, bs, sc, greedy, st);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_draft(const DraftArgs& a, cudaStream_t st) {
  if (a.U != nullptr) return launch_draft_rnn(a, st);
  const int n_tiles = (a.V + kTileV - 1) / kTileV;
  const bool greedy = a.T == 0.0f;
  const ScalePair sc = make_scale(greedy ? 1.0 : 1.4426950408889634 / (double)a.T);
  const bool tc = draft_tc_supported(a);
  if (tc) {
    // bf16 on the tensor cores: every draft position in one persistent
    // cooperative launch when the GPU can host it, else one fused launch
    // plus one finish launch per position
    cudaError_t e = launch_draft_persistent_tc(a, st);
    if (e != cudaErrorNotSupported) return e;
  }
  for (int k = 0; k < a.gamma; ++k) {
    const int32_t* prev = k == 0 ? a.anchor : a.tokens + (k - 1);
    const int stride = k == 0 ? 1 : a.gamma;
    cudaError_t e;
    if (tc) {
      e = launch_draft_partial_tc(a, k, prev, stride, st);
      if (e != cudaSuccess) return e;
      BiasSrc b{nullptr, (const __nv_bfloat16*)a.E, (const __nv_bfloat16*)a.Wt, prev, stride, a.r};
      e = launch_finish<__nv_bfloat16, 128>(a, k, b, sc, greedy, st);
      if (e != cudaSuccess) return e;
      continue;
    }
    e = launch_bias(a.R, a.V, a.r, a.dt, a.E, a.Wt, prev, stride, a.V, a.bias, a.status, st);
    if (e != cudaSuccess) return e;
    dim3 g1(n_tiles, a.R);
    BiasSrc b{a.bias, nullptr, nullptr, prev, stride, a.r};
    if (a.dt == 0) {
      DSPARK_LAUNCH(kKindDraftPartial, st,
                    draft_partial_kernel<__nv_bfloat16><<<g1, kTileV, 0, st>>>(
                        a.V, a.gamma, k, n_tiles, (const __nv_bfloat16*)a.z, a.bias, sc, greedy,
                        a.part, a.status));
      e = launch_finish<__nv_bfloat16, kTileV>(a, k, b, sc, greedy, st);
    } else {
      DSPARK_LAUNCH(kKindDraftPartial, st,
                    draft_partial_kernel<float><<<g1, kTileV, 0, st>>>(
                        a.V, a.gamma, k, n_tiles, (const float*)a.z, a.bias, sc, greedy, a.part,
                        a.status));
      e = launch_finish<float, kTileV>(a, k, b, sc, greedy, st);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
