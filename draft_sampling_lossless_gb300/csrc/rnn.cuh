// The RNN head's state rounding (see rnn.cu for the head): s = round(tanh(pre))
// with tanh taken in double and one rounding to the table's type.
#pragma once

#include <cuda_bf16.h>

namespace dspark {
namespace rnn {

// One rounding from double to bf16 (8 significant bits, ties to even).
__device__ __forceinline__ __nv_bfloat16 bf16_from_double(double x) {
  if (x == 0.0 || isnan(x)) return __float2bfloat16_rn((float)x);
  double y;
  if (fabs(x) < 0x1p-126) {
    y = ldexp(rint(ldexp(x, 133)), -133);  // bf16 subnormals: multiples of 2^-133
  } else {
    int e;
    const double m = frexp(x, &e);  // 0.5 <= |m| < 1
    y = ldexp(rint(ldexp(m, 8)), e - 8);
  }
  return __float2bfloat16_rn((float)y);  // y is a bf16 value: exact
}

static __device__ __noinline__ __nv_bfloat16 state_bf16_double(float x) {
  return bf16_from_double(tanh((double)x));
}

// round_bf16(tanh(x)).  The fp32 tanhf (a few ulp of fp32 from the exact
// value) already decides the bf16 rounding unless its result lies within 8
// fp32 ulps of a bf16 rounding midpoint (low 16 bits near 0x8000, about one
// value in 4000); only then is tanh taken in double (GB300's double rate is
// a small fraction of its fp32 rate), out of line and behind a warp vote so
// that no warp without such a value executes any of it.
__device__ __forceinline__ __nv_bfloat16 state_bf16(float x) {
  const float t = tanhf(x);
  const int low = (int)(__float_as_uint(t) & 0xffffu);
  const bool near = abs(low - 0x8000) <= 8;
  __nv_bfloat16 v = __float2bfloat16_rn(t);
  if (__any_sync(__activemask(), near)) {
    if (near) v = state_bf16_double(x);
  }
  return v;
}

__device__ __forceinline__ void store_state(__nv_bfloat16* p, float x) { *p = state_bf16(x); }
__device__ __forceinline__ void store_state(float* p, float x) {
  *p = __double2float_rn(tanh((double)x));
}

}  // namespace rnn
}  // namespace dspark
