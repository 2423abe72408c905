// Per-warp arithmetic of the confidence head, shared by the confidence kernel
// and by the persistent draft kernel (which can evaluate the head after its
// last draft position), so that both give the same bits.
//
// News article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 2.1: c_k = sigma(w . [h_k ; W1[x_{k-1}]])
// with a per-position temperature (STS).
#pragma once

#include "common.cuh"

namespace dspark {
namespace conf {

// One warp per (request, position): c = sigmoid((w_h . h + w_e . E1[prev]) / sts).
// bf16 with vector loads (the common case): the lane's share of h (up to
// kHLoads 16-byte loads at once, a second batch for d above 4096) and the
// previous token are requested together, then the E1 row once the token is
// known, so a dot product costs about two memory round trips (three with a
// second batch); w (shared by every warp) is read through L1.
constexpr int kHLoads = 16;   // 16-byte loads a lane holds at once
constexpr int kHBatches = 2;  // d <= 32 * 8 * kHLoads * kHBatches = 8192 on the one-pass path
constexpr int kHMaxD = 32 * 8 * kHLoads * kHBatches;

__device__ __forceinline__ float dot8_bf16(const uint4 q, const float* __restrict__ w) {
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(w));
  const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + 4));
  float s = 0.f;
  s = fmaf(w0.x, __uint_as_float(q.x << 16), s);
  s = fmaf(w0.y, __uint_as_float(q.x & 0xffff0000u), s);
  s = fmaf(w0.z, __uint_as_float(q.y << 16), s);
  s = fmaf(w0.w, __uint_as_float(q.y & 0xffff0000u), s);
  s = fmaf(w1.x, __uint_as_float(q.z << 16), s);
  s = fmaf(w1.y, __uint_as_float(q.z & 0xffff0000u), s);
  s = fmaf(w1.z, __uint_as_float(q.w << 16), s);
  s = fmaf(w1.w, __uint_as_float(q.w & 0xffff0000u), s);
  return s;
}

// The lane's partial of w_h . h for one (request, position) on the one-pass
// bf16 path: the lane's 16-byte loads of h (issued by conf_load_h) times w,
// accumulated in load order.
// Batch b of a lane's loads: steps i = 16 b .. 16 b + 15 (elements
// (i * 32 + lane) * 8 .. + 7); a lane's partial adds the steps in order,
// batch after batch, so the sum does not depend on how the loads are grouped.
__device__ __forceinline__ void conf_load_h(const __nv_bfloat16* __restrict__ hp, int d,
                                            uint4 (&hq)[kHLoads], int batch = 0) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kHLoads; ++i) {
    const int j = ((batch * kHLoads + i) * 32 + lane) * 8;
    hq[i] = j < d ? __ldcs(reinterpret_cast<const uint4*>(hp + j)) : make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ float conf_h_lane(const uint4 (&hq)[kHLoads],
                                             const float* __restrict__ w, int d, int batch = 0,
                                             float s = 0.f) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kHLoads; ++i) {
    const int j = ((batch * kHLoads + i) * 32 + lane) * 8;
    if (j < d) s += dot8_bf16(hq[i], w + j);
  }
  return s;
}

// The lane's whole partial of w . h: the first batch from hq (already
// loaded), the second (d > 4096) loaded and added here.
__device__ __forceinline__ float conf_h_lane_all(uint4 (&hq)[kHLoads],
                                                 const __nv_bfloat16* __restrict__ hp,
                                                 const float* __restrict__ w, int d) {
  float s = conf_h_lane(hq, w, d, 0);
  if (d > 32 * 8 * kHLoads) {
    conf_load_h(hp, d, hq, 1);
    s = conf_h_lane(hq, w, d, 1, s);
  }
  return s;
}

// The lane's eight elements of E1[prev] (zero when prev < 0 or past r).
__device__ __forceinline__ uint4 conf_load_e1(const __nv_bfloat16* __restrict__ E1, int prev,
                                              int r) {
  const int je = (threadIdx.x & 31) * 8;
  if (prev >= 0 && je < r) return *reinterpret_cast<const uint4*>(E1 + (size_t)prev * r + je);
  return make_uint4(0, 0, 0, 0);
}

// c from the lane's partial of the hidden-state term: add the embedding term,
// reduce over the warp, scale by the STS temperature, apply sigma.
__device__ __forceinline__ float conf_sigma(float s, uint4 eq, int prev, int r,
                                            const float* __restrict__ w_e, float t) {
  const int je = (threadIdx.x & 31) * 8;
  if (prev >= 0 && je < r) s += dot8_bf16(eq, w_e + je);
  s = warp_sum(s);
  return 1.0f / (1.0f + expf(-s / t));
}

}  // namespace conf
}  // namespace dspark
