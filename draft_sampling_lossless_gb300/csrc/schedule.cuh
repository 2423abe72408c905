// Device-side pieces of the prefix scheduler shared by its own kernel and by
// the persistent draft kernel, which can run the scheduler after its last
// draft position: survival-value cleaning, the exact 2^-40 fixed point, the
// integer emulation of the double roundings of Theta, E and B, and the
// one-block cut over precomputed Theta keys.
//
// News article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 2.2 (objective, greedy order,
// early stop); explainer "DSpark.让每一轮计算，多走几步", survival panel.
#pragma once

#include "common.cuh"

namespace dspark {
namespace sched {

__device__ __forceinline__ float clean_a(float a, uint32_t* status) {
  if (!(a >= 0.0f) || a == INFINITY) {  // NaN, negative or infinite
    set_flag(status, kFlagNonFinite);
    return 0.0f;
  }
  return a;
}

// Nearest multiple of 2^-40 (ties to even) of a finite a >= 0, in 2^-40
// units: the same integer as rounding the double a * 2^40.
__device__ __forceinline__ long long to_fixed(float a) {
  const uint32_t b = __float_as_uint(a);
  const int E = (int)(b >> 23) & 0xff;
  if (E == 0) return 0;  // subnormal: below 2^-126, rounds to 0
  const unsigned long long m = (b & 0x7fffffu) | 0x800000u;  // a = m * 2^(E - 150)
  const int sh = E - 110;                                     // a * 2^40 = m * 2^sh
  if (sh >= 0) return sh > 39 ? LLONG_MAX : (long long)(m << sh);
  const int k = -sh;
  if (k > 25) return 0;
  const unsigned long long q = m >> k, r = m & ((1ull << k) - 1), half = 1ull << (k - 1);
  return (long long)(q + ((r > half || (r == half && (q & 1))) ? 1 : 0));
}

// x rounded to 53 significant bits (ties to even), for x < 2^63: the value
// of the double nearest to x, as an integer.
__device__ __forceinline__ unsigned long long rne53(unsigned long long x) {
  const int msb = 63 - __clzll(x | 1);
  if (msb <= 52) return x;
  const int k = msb - 52;
  const unsigned long long q = x >> k, r = x & ((1ull << k) - 1), half = 1ull << (k - 1);
  return (q + ((r > half || (r == half && (q & 1))) ? 1 : 0)) << k;
}

// Bits of the double x * 2^e2 for an integer x < 2^63 with at most 53
// significant bits (exact), x > 0.
__device__ __forceinline__ unsigned long long dbl_bits(unsigned long long x, int e2) {
  const int msb = 63 - __clzll(x);
  const unsigned long long mant = msb <= 52 ? x << (52 - msb) : x >> (msb - 52);
  return ((unsigned long long)(msb + e2 + 1023) << 52) | (mant & 0x000fffffffffffffull);
}

// Bits of the double product d * s rounded to nearest (ties to even), d a
// positive normal double (bits), s a finite float; the result is a normal
// double for every such pair met here (d in [1, 2^23]).  Zero: +0.
__device__ __forceinline__ unsigned long long dbl_mul_float(unsigned long long d, float s) {
  const uint32_t fb = __float_as_uint(s);
  const int fe = (int)(fb >> 23) & 0xff;
  unsigned long long fm = fb & 0x7fffffu;
  if (fe == 0 && fm == 0) return 0;
  int fexp;  // s = fm * 2^fexp
  if (fe == 0) {
    fexp = -149;
  } else {
    fm |= 0x800000u;
    fexp = fe - 150;
  }
  const unsigned long long dm = (d & 0x000fffffffffffffull) | 0x0010000000000000ull;
  const int dexp = (int)((d >> 52) & 0x7ff) - 1075;  // d = dm * 2^dexp
  // exact product dm * fm (< 2^77) as hi:lo
  const unsigned long long lo = dm * fm, hi = __umul64hi(dm, fm);
  const int msb = hi ? 127 - __clzll(hi) : 63 - __clzll(lo);
  const int k = msb - 52;  // bits below the 53 kept (k >= 0: dm alone has 53)
  unsigned long long q, rlo, rhi;  // kept bits; remainder below them (hi:lo)
  if (k >= 64) {
    q = hi >> (k - 64);
    rhi = hi & ((1ull << (k - 64)) - 1);
    rlo = lo;
  } else if (k > 0) {
    q = (lo >> k) | (hi << (64 - k));
    rhi = 0;
    rlo = lo & ((1ull << k) - 1);
  } else {
    q = lo;
    rhi = 0;
    rlo = 0;
  }
  bool up = false;
  if (k > 0) {
    // compare the remainder with half = 2^(k-1)
    bool gt, eq;
    if (k - 1 >= 64) {
      const unsigned long long hh = 1ull << (k - 1 - 64);
      gt = rhi > hh || (rhi == hh && rlo > 0);
      eq = rhi == hh && rlo == 0;
    } else {
      const unsigned long long hl = 1ull << (k - 1);
      gt = rhi > 0 || rlo > hl;
      eq = rhi == 0 && rlo == hl;
    }
    up = gt || (eq && (q & 1));
  }
  q += up ? 1 : 0;
  int ex = msb + dexp + fexp;  // value = q * 2^(ex - 52)
  if (q >> 53) {
    q >>= 1;
    ++ex;
  }
  const unsigned long long sign = (unsigned long long)(fb >> 31) << 63;
  return sign | ((unsigned long long)(ex + 1023) << 52) | (q & 0x000fffffffffffffull);
}

// Unsigned key with the numeric order of the double whose bits are b (b not
// NaN; -0 compares equal to +0).
__device__ __forceinline__ unsigned long long dbl_key(unsigned long long b) {
  if ((b << 1) == 0) b = 0;
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

// Theta_i's order key from the exact prefix S_i (units of 2^-40), in the
// oracle's operation order ((double)S * 2^-40 + R) * SPS[R + i]: S rounded
// to a double, the sum rounded, the product rounded; returned as an order
// key of the double's bits.  A non-finite SPS entry counts as 0 (flagged).
__device__ __forceinline__ unsigned long long theta_key_of(int R, int i, long long S,
                                                           const float* __restrict__ sps,
                                                           uint32_t* status) {
  const unsigned long long e =
      rne53(((unsigned long long)R << 40) + rne53((unsigned long long)S));  // (R + S 2^-40) 2^40
  float sv = sps[R + i];
  if (!isfinite(sv)) {
    set_flag(status, kFlagNonFinite);
    sv = 0.0f;
  }
  return dbl_key(dbl_mul_float(dbl_bits(e, -40), sv));
}

// The block's first argmax over (key, index) pairs: the largest key, the
// lowest index among equal keys (index 0x7fffffff: no candidate).
__device__ inline int block_first_argmax(unsigned long long v, int bi, unsigned long long* shk,
                                         int* shidx, int* res) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > v || (ov == v && oi < bi)) {
      v = ov;
      bi = oi;
    }
  }
  __syncthreads();
  if (lane == 0) {
    shk[wid] = v;
    shidx[wid] = bi;
  }
  __syncthreads();
  if (wid == 0) {
    v = lane < nw ? shk[lane] : 0ull;
    bi = lane < nw ? shidx[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > v || (ov == v && oi < bi)) {
        v = ov;
        bi = oi;
      }
    }
    if (lane == 0) *res = bi;
  }
  __syncthreads();
  return *res;
}

// l_r = the number of request r's candidates ranked below i*, row_off (their
// exclusive scan of 1 + l_r), by one whole block.
__device__ inline void schedule_lengths(int R, int gamma, int istar, const int32_t* rank,
                                        int32_t* __restrict__ ell,
                                        int32_t* __restrict__ row_off, long long* shl) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int rseg = (R + nt - 1) / nt;
  const int r0 = min(R, tid * rseg), r1 = min(R, r0 + rseg);
  long long lsum = 0;
  for (int r = r0; r < r1; ++r) {
    int c = 0;
    for (int j = 0; j < gamma; ++j) c += rank[(size_t)r * gamma + j] < istar;
    ell[r] = c;
    lsum += 1 + c;
  }
  long long rincl = block_inclusive_scan(lsum, shl);
  long long run = rincl - lsum;
  for (int r = r0; r < r1; ++r) {
    row_off[r] = (int32_t)run;
    run += 1 + ell[r];
  }
  if (tid == nt - 1) row_off[R] = (int32_t)rincl;
}

// E = R + S_{i*} as the oracle's double, B = R + i*.
__device__ __forceinline__ void schedule_store_EB(int R, int istar, long long S,
                                                  int32_t* __restrict__ B_out,
                                                  double* __restrict__ E_out) {
  const unsigned long long e = rne53(((unsigned long long)R << 40) + rne53((unsigned long long)S));
  E_out[0] = __longlong_as_double((long long)dbl_bits(e, -40));
  B_out[0] = R + istar;
}

// The cut when every Theta_i key (i = 0..imax) and every prefix S_i
// (i = 0..N) is already known (the persistent draft's ranking CTAs form them
// with the ranks): the stop or the first argmax over the keys, E from
// S_{i*}, then the lengths.  The same definitions as the scheduler kernel's
// cut (schedule.cu), so the same results.  tkey and spre are read from L2 (written by other CTAs).
__device__ inline void schedule_cut_keys(int R, int gamma, int imax, int early_stop,
                                         const unsigned long long* tkey, const long long* spre,
                                         const int32_t* rank, int32_t* __restrict__ ell,
                                         int32_t* __restrict__ row_off,
                                         int32_t* __restrict__ B_out,
                                         double* __restrict__ E_out) {
  __shared__ long long shl[32];
  __shared__ int shi[32];
  __shared__ unsigned long long shk[32];
  __shared__ int shidx[32];
  __shared__ int istar_s;
  const int tid = threadIdx.x, nt = blockDim.x;
  int my_stop = 0x7fffffff;
  unsigned long long best_v = 0;
  int best_i = 0x7fffffff;
  for (int i = tid; i <= imax; i += nt) {
    const unsigned long long th = __ldcg(tkey + i);
    if (i > 0 && !(th > __ldcg(tkey + i - 1))) my_stop = min(my_stop, i - 1);
    if (best_i == 0x7fffffff || th > best_v) {  // i ascends within the thread
      best_v = th;
      best_i = i;
    }
  }
  int istar;
  if (early_stop) {
    const int st = block_min_int(my_stop, shi);
    istar = st == 0x7fffffff ? imax : st;
  } else {
    istar = block_first_argmax(best_v, best_i, shk, shidx, &istar_s);
    if (istar == 0x7fffffff) istar = 0;
  }
  if (tid == 0) schedule_store_EB(R, istar, __ldcg(spre + istar), B_out, E_out);
  schedule_lengths(R, gamma, istar, rank, ell, row_off, shl);
}

}  // namespace sched
}  // namespace dspark
