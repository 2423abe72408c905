// Confidence head, sequential temperature scaling and cumulative survival.
//
// News article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 2.1: c_k = sigma(w . [h_k ; W1[x_{k-1}]])
// with a per-position temperature fitted left to right (STS); explainer
// "DSpark.让每一轮计算，多走几步", survival panel: a_j = c_1 ... c_j.
//
// One block per request, one warp per draft position: the warp reads the
// position's hidden state and the previous token's embedding row with
// coalesced loads, reduces the dot product, applies sigma(s / t_k); lane 0 of
// warp 0 then forms the running product along the block.
#include "common.cuh"

namespace dspark {

template <typename T>
__global__ void confidence_kernel(int gamma, int d, int r, int V, const T* __restrict__ h,
                                  const float* __restrict__ w, const T* __restrict__ E1,
                                  const int32_t* __restrict__ anchor,
                                  const int32_t* __restrict__ tokens,
                                  const float* __restrict__ sts, const float* __restrict__ c_in,
                                  float* __restrict__ c_out, float* __restrict__ a_out,
                                  uint32_t* status) {
  __shared__ float c_s[kMaxGamma];
  const int n = blockIdx.x;
  const int k = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (k < gamma) {
    const size_t idx = (size_t)n * gamma + k;
    float c;
    if (c_in != nullptr) {
      c = c_in[idx];
    } else {
      int prev = k == 0 ? anchor[n] : tokens[idx - 1];
      if (prev >= V || prev < -1) {
        if (lane == 0) set_flag(status, kFlagTokenRange);
        prev = -1;
      }
      float s = 0.f;
      const T* hr = h + idx * d;
      for (int i = lane; i < d; i += 32) s = fmaf(w[i], to_f32<T>(hr[i]), s);
      if (prev >= 0) {
        const T* er = E1 + (size_t)prev * r;
        for (int i = lane; i < r; i += 32) s = fmaf(w[d + i], to_f32<T>(er[i]), s);
      }
      s = warp_sum(s);
      c = 1.0f / (1.0f + expf(-s / sts[k]));
    }
    if (lane == 0) {
      if (!isfinite(c)) set_flag(status, kFlagNonFinite);
      c_s[k] = c;
      c_out[idx] = c;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float run = 1.0f;
    for (int j = 0; j < gamma; ++j) {
      run = run * c_s[j];
      a_out[(size_t)n * gamma + j] = run;
    }
  }
}

cudaError_t launch_confidence(const ConfArgs& a, cudaStream_t st) {
  const int threads = 32 * a.gamma;
  if (a.dt == 0)
    DSPARK_LAUNCH(kKindConfidence, st, confidence_kernel<__nv_bfloat16><<<a.R, threads, 0, st>>>(
        a.gamma, a.d, a.r, a.V, (const __nv_bfloat16*)a.h, a.w, (const __nv_bfloat16*)a.E1,
        a.anchor, a.tokens, a.sts, a.c_in, a.c_out, a.a_out, a.status));
  else
    DSPARK_LAUNCH(kKindConfidence, st, confidence_kernel<float><<<a.R, threads, 0, st>>>(
        a.gamma, a.d, a.r, a.V, (const float*)a.h, a.w, (const float*)a.E1, a.anchor, a.tokens,
        a.sts, a.c_in, a.c_out, a.a_out, a.status));
  return cudaGetLastError();
}

}  // namespace dspark
