// Confidence head, sequential temperature scaling and cumulative survival.
//
// News article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 2.1: c_k = sigma(w . [h_k ; W1[x_{k-1}]])
// with a per-position temperature fitted left to right (STS); explainer
// "DSpark.让每一轮计算，多走几步", survival panel: a_j = c_1 ... c_j.
//
// One block per request, one warp per draft position: the warp reads the
// position's hidden state and the previous token's embedding row with
// 16-byte loads (eight elements per lane per step), reduces the dot product,
// applies sigma(s / t_k); thread 0 then forms the running product along the
// block.  HBM-bound: R * gamma * (d + r) elements.
#include "common.cuh"
#include "confidence.cuh"

namespace dspark {

namespace {

using namespace conf;

// sum_i w[i] * x[i] over n elements, the warp's lanes taking eight at a time
// (x 16-byte aligned and n a multiple of 8 for the vector path).  The vector
// path issues four steps' loads before their multiply-adds, so a lane has up
// to four 16-byte loads in flight instead of one dependent chain.
template <typename T>
__device__ __forceinline__ float warp_dot(const float* __restrict__ w, const T* __restrict__ x,
                                          int n, bool vec) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  if (vec) {
    constexpr int kU = 4;
    int i = lane * 8;
    for (; i + (kU - 1) * 256 < n; i += kU * 256) {
      float xv[kU][8];
      float4 wv[kU][2];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        load8<T>(x, i + u * 256, n, xv[u], 0.f);
        wv[u][0] = *reinterpret_cast<const float4*>(w + i + u * 256);
        wv[u][1] = *reinterpret_cast<const float4*>(w + i + u * 256 + 4);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        s = fmaf(wv[u][0].x, xv[u][0], s);
        s = fmaf(wv[u][0].y, xv[u][1], s);
        s = fmaf(wv[u][0].z, xv[u][2], s);
        s = fmaf(wv[u][0].w, xv[u][3], s);
        s = fmaf(wv[u][1].x, xv[u][4], s);
        s = fmaf(wv[u][1].y, xv[u][5], s);
        s = fmaf(wv[u][1].z, xv[u][6], s);
        s = fmaf(wv[u][1].w, xv[u][7], s);
      }
    }
    for (; i < n; i += 256) {
      float xv[8];
      load8<T>(x, i, n, xv, 0.f);
      const float4 w0 = *reinterpret_cast<const float4*>(w + i);
      const float4 w1 = *reinterpret_cast<const float4*>(w + i + 4);
      s = fmaf(w0.x, xv[0], s);
      s = fmaf(w0.y, xv[1], s);
      s = fmaf(w0.z, xv[2], s);
      s = fmaf(w0.w, xv[3], s);
      s = fmaf(w1.x, xv[4], s);
      s = fmaf(w1.y, xv[5], s);
      s = fmaf(w1.z, xv[6], s);
      s = fmaf(w1.w, xv[7], s);
    }
  } else {
    for (int i = lane; i < n; i += 32) s = fmaf(w[i], to_f32<T>(x[i]), s);
  }
  return s;
}

template <typename T>
__global__ void confidence_kernel(int gamma, int d, int r, int V, int vec,
                                  const T* __restrict__ h, const float* __restrict__ w,
                                  const T* __restrict__ E1, const int32_t* __restrict__ anchor,
                                  const int32_t* __restrict__ tokens,
                                  const float* __restrict__ sts, const float* __restrict__ c_in,
                                  float* __restrict__ c_out, float* __restrict__ a_out,
                                  uint32_t* status) {
  __shared__ float c_s[kMaxGamma];
  const int n = blockIdx.x;
  const int k = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t idx = (size_t)n * gamma + k;
  const bool one_pass = sizeof(T) == 2 && vec && d <= kHMaxD && r <= 256;
  uint4 hq[kHLoads];
  if (one_pass && k < gamma && c_in == nullptr) {
    // h does not depend on the draft: request it before waiting for the tokens
    conf_load_h(reinterpret_cast<const __nv_bfloat16*>(h) + idx * d, d, hq);
  }
  grid_dependency_wait();  // the drafted tokens
  if (k < gamma) {
    float c;
    if (c_in != nullptr) {
      c = c_in[idx];
    } else {
      int prev = k == 0 ? anchor[n] : tokens[idx - 1];
      if (prev >= V || prev < -1) {
        if (lane == 0) set_flag(status, kFlagTokenRange);
        prev = -1;
      }
      if (one_pass) {
        const uint4 eq = conf_load_e1(reinterpret_cast<const __nv_bfloat16*>(E1), prev, r);
        c = conf_sigma(
            conf_h_lane_all(hq, reinterpret_cast<const __nv_bfloat16*>(h) + idx * d, w, d), eq,
            prev, r, w + d, sts[k]);
      } else {
        float s = warp_dot<T>(w, h + idx * d, d, vec);
        if (prev >= 0) s += warp_dot<T>(w + d, E1 + (size_t)prev * r, r, vec);
        s = warp_sum(s);
        c = 1.0f / (1.0f + expf(-s / sts[k]));
      }
    }
    if (lane == 0) {
      if (!isfinite(c)) set_flag(status, kFlagNonFinite);
      c_s[k] = c;
      c_out[idx] = c;
    }
  }
  __syncthreads();
  if (threadIdx.x < gamma) {
    // a_j = prod_{i <= j} c_i, each thread its own prefix (gamma <= 32)
    float run = 1.0f;
    for (int j = 0; j <= (int)threadIdx.x; ++j) run = run * c_s[j];
    a_out[(size_t)n * gamma + threadIdx.x] = run;
  }
}

}  // namespace

cudaError_t launch_confidence(const ConfArgs& a, cudaStream_t st) {
  const int threads = 32 * a.gamma;
  // vector loads need 16-byte aligned rows and weights, d and r multiples of 8
  const uintptr_t mis = reinterpret_cast<uintptr_t>(a.h) | reinterpret_cast<uintptr_t>(a.E1) |
                        reinterpret_cast<uintptr_t>(a.w);
  const int esz = a.dt == 0 ? 2 : 4;
  const int vec = a.c_in == nullptr && (mis & 15) == 0 && a.d % 8 == 0 && a.r % 8 == 0 &&
                  ((size_t)a.d * esz) % 16 == 0 && ((size_t)a.d * 4) % 16 == 0;
  if (a.dt == 0)
    DSPARK_LAUNCH(kKindConfidence, st,
                  launch_pdl(confidence_kernel<__nv_bfloat16>, dim3(a.R), dim3(threads), 0, st,
                             a.gamma, a.d, a.r, a.V, vec, (const __nv_bfloat16*)a.h, a.w,
                             (const __nv_bfloat16*)a.E1, a.anchor, a.tokens, a.sts, a.c_in,
                             a.c_out, a.a_out, a.status));
  else
    DSPARK_LAUNCH(kKindConfidence, st,
                  launch_pdl(confidence_kernel<float>, dim3(a.R), dim3(threads), 0, st, a.gamma,
                             a.d, a.r, a.V, vec, (const float*)a.h, a.w, (const float*)a.E1,
                             a.anchor, a.tokens, a.sts, a.c_in, a.c_out, a.a_out, a.status));
  return cudaGetLastError();
}

}  // namespace dspark
