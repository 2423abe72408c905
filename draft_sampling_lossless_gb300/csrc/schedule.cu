// Hardware-aware prefix scheduler.
//
// News article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 2.2: maximise tau * SPS(B) over the
// per-request verify lengths, B = sum_r (1 + l_r); sort every candidate by its
// survival probability, add them greedily, stop as soon as throughput stops
// rising (O(gamma R log gamma R)); challenge 2: the same search without early
// stop.  Explainer "DSpark.让每一轮计算，多走几步", survival panel:
// E = R + sum a, rate = E / T(B), candidates added in sorted order.
//
// Two launches:
//   rank   -- the position of every candidate in the total order
//             (a descending, then flat index n*gamma + j ascending), counted by
//             comparisons against all others; ranks are a permutation because
//             the order is strict, so no sort network or stable radix pass is
//             needed and the result does not depend on thread timing.
//   finish -- one block: scatter to sorted order, exact integer prefix sums of
//             the 2^-40 fixed-point survival values, Theta_i rounded exactly as
//             the oracle's double arithmetic rounds it, the early-stop or
//             argmax cut, then l_r, row_off, B and E.
// No floating-point double instruction runs here: the double roundings are
// reproduced with integer arithmetic (round to nearest, ties to even), which
// gives the same bits and avoids the narrow FP64 pipe.
#include "common.cuh"

namespace dspark {

namespace {

constexpr int kRankThreads = 256;
constexpr int kRankChunk = 2048;
constexpr int kFinThreads = 1024;

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

// grid: (ceil(N / 256), n_split); block 256.  rank[] must be zero on entry.
__global__ void __launch_bounds__(kRankThreads) rank_kernel(int N, int per_split,
                                                            const float* __restrict__ a,
                                                            int32_t* __restrict__ rank,
                                                            uint32_t* status) {
  __shared__ float as[kRankChunk];
  const int e = blockIdx.x * kRankThreads + threadIdx.x;
  const float ae = e < N ? clean_a(a[e], status) : 0.0f;
  const int lo = blockIdx.y * per_split, hi = min(N, lo + per_split);
  int cnt = 0;
  for (int c0 = lo; c0 < hi; c0 += kRankChunk) {
    const int c1 = min(hi, c0 + kRankChunk);
    __syncthreads();
    for (int i = c0 + threadIdx.x; i < c1; i += kRankThreads) {
      float v = a[i];
      as[i - c0] = (!(v >= 0.0f) || v == INFINITY) ? 0.0f : v;
    }
    __syncthreads();
    if (e < N) {
      for (int i = c0; i < c1; ++i) {
        const float ai = as[i - c0];
        cnt += (ai > ae) | ((ai == ae) & (i < e));
      }
    }
  }
  if (e < N && cnt) atomicAdd(&rank[e], cnt);
}

// The cut and the per-request outputs, by one block of kFinThreads threads,
// given every candidate's rank.
// a, rank and sfix may point to shared or global memory.
__device__ __forceinline__ void schedule_finish(
    int R, int gamma, int imax, int early_stop, const float* a,
    const float* __restrict__ sps, const int32_t* rank, long long* sfix,
    int32_t* __restrict__ ell, int32_t* __restrict__ row_off, int32_t* __restrict__ B_out,
    double* __restrict__ E_out, uint32_t* status) {
  __shared__ long long shl[32];
  __shared__ int shi[32];
  __shared__ unsigned long long shk[32];
  __shared__ int shidx[32];
  __shared__ int istar_s;
  const int N = R * gamma;
  const int tid = threadIdx.x, nt = blockDim.x;
  // 1. scatter the fixed-point survival values to their sorted positions
  for (int e = tid; e < N; e += nt) {
    float v = a[e];
    v = (!(v >= 0.0f) || v == INFINITY) ? 0.0f : v;
    sfix[rank[e]] = to_fixed(v);
  }
  __syncthreads();
  // 2. Theta_i for i in [0, imax]; thread chunk [i0, i1) over i
  const int n_i = imax + 1;
  const int seg = (n_i + nt - 1) / nt;
  const int i0 = min(n_i, tid * seg), i1 = min(n_i, i0 + seg);
  long long loc = 0;
  for (int i = i0; i < i1; ++i)
    if (i < N) loc += sfix[i];
  long long incl = block_inclusive_scan(loc, shl);
  const long long S0 = incl - loc;  // exact: integers
  // Theta in the oracle's operation order, ((double)S * 2^-40 + R) * SPS:
  // S rounded to a double, the sum rounded, the product rounded; returned as
  // an order key of the double's bits.
  auto theta_key = [&](int i, long long S) -> unsigned long long {
    const unsigned long long e =
        rne53(((unsigned long long)R << 40) + rne53((unsigned long long)S));  // (R + S 2^-40) 2^40
    float s = sps[R + i];
    if (!isfinite(s)) {
      set_flag(status, kFlagNonFinite);
      s = 0.0f;
    }
    return dbl_key(dbl_mul_float(dbl_bits(e, -40), s));
  };
  int my_stop = 0x7fffffff;
  unsigned long long best_v = 0;
  int best_i = 0x7fffffff;
  {
    long long S = S0;
    unsigned long long prev_th = 0;
    for (int i = i0; i < i1; ++i) {
      const unsigned long long th = theta_key(i, S);
      if (i > i0 && !(th > prev_th) && my_stop == 0x7fffffff) my_stop = i - 1;
      if (best_i == 0x7fffffff || th > best_v) {
        best_v = th;
        best_i = i;
      }
      prev_th = th;
      if (i < N) S += sfix[i];
    }
    // the pair that straddles the chunk boundary (i1 - 1, i1)
    if (i1 > i0 && i1 < n_i && my_stop == 0x7fffffff) {
      const unsigned long long th = theta_key(i1, S);
      if (!(th > prev_th)) my_stop = i1 - 1;
    }
  }
  int istar;
  if (early_stop) {
    int s = block_min_int(my_stop, shi);
    istar = s == 0x7fffffff ? imax : s;
  } else {
    // first argmax: max value, then lowest index
    // (key 0 is below every double's key: a thread with no i never wins)
    const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
    unsigned long long v = best_v;
    int bi = best_i;
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
      if (lane == 0) istar_s = bi;
    }
    __syncthreads();
    istar = istar_s;
    if (istar == 0x7fffffff) istar = 0;
  }
  // 3. E = R + S_{i*}
  if (istar >= i0 && istar < i1) {
    long long S = S0;
    for (int i = i0; i < istar; ++i) S += sfix[i];
    const unsigned long long e =
        rne53(((unsigned long long)R << 40) + rne53((unsigned long long)S));
    E_out[0] = __longlong_as_double((long long)dbl_bits(e, -40));
    B_out[0] = R + istar;
  }
  // 4. l_r = number of request r's candidates ranked below i*, and row_off
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

__global__ void __launch_bounds__(kFinThreads) schedule_finish_kernel(
    int R, int gamma, int imax, int early_stop, const float* __restrict__ a,
    const float* __restrict__ sps, const int32_t* __restrict__ rank, long long* __restrict__ sfix,
    int32_t* __restrict__ ell, int32_t* __restrict__ row_off, int32_t* __restrict__ B_out,
    double* __restrict__ E_out, uint32_t* status) {
  schedule_finish(R, gamma, imax, early_stop, a, sps, rank, sfix, ell, row_off, B_out, E_out,
                  status);
}

// Small batches (N <= kFusedMax candidates): the ranks and the cut in one
// block, everything in shared memory.  The cleaned survival values are
// non-negative (zero as +0), so their bit patterns order like the values:
// candidate e's rank counts the i < e with bits >= its own and the i > e with
// bits > its own.  Each candidate's comparison range is split over
// blockDim / N threads that add their counts with shared-memory atomics.
constexpr int kFusedMax = 1024;

__global__ void __launch_bounds__(kFinThreads) schedule_fused_kernel(
    int R, int gamma, int imax, int early_stop, const float* __restrict__ a,
    const float* __restrict__ sps, int32_t* __restrict__ rank_out, int32_t* __restrict__ ell,
    int32_t* __restrict__ row_off, int32_t* __restrict__ B_out, double* __restrict__ E_out,
    uint32_t* status) {
  __shared__ float as[kFusedMax];
  __shared__ uint32_t ab[kFusedMax];
  __shared__ int32_t rk[kFusedMax];
  __shared__ long long sf[kFusedMax];
  grid_dependency_wait();  // the survival values
  const int N = R * gamma, nt = blockDim.x;
  for (int e = threadIdx.x; e < N; e += nt) {
    const float v = clean_a(a[e], status) + 0.0f;  // -0 -> +0
    as[e] = v;
    ab[e] = __float_as_uint(v);
    rk[e] = 0;
  }
  __syncthreads();
  const int P = max(1, nt / N);  // threads per candidate
  const int span = (N + P - 1) / P;
  for (int t = threadIdx.x; t < N * P; t += nt) {
    const int e = t % N, part = t / N;
    const int i0 = part * span, i1 = min(N, i0 + span);
    const uint32_t be = ab[e];
    int cnt = 0;
    const int im = min(max(e, i0), i1);
#pragma unroll 8
    for (int i = i0; i < im; ++i) cnt += ab[i] >= be ? 1 : 0;
#pragma unroll 8
    for (int i = max(im, e + 1); i < i1; ++i) cnt += ab[i] > be ? 1 : 0;
    if (cnt) atomicAdd(&rk[e], cnt);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += nt) rank_out[e] = rk[e];
  schedule_finish(R, gamma, imax, early_stop, as, sps, rk, sf, ell, row_off, B_out, E_out, status);
}

}  // namespace

cudaError_t launch_schedule(const SchedArgs& s, cudaStream_t st) {
  const int N = s.R * s.gamma;
  const int imax0 = s.max_B > 0 ? (s.max_B - s.R < N ? s.max_B - s.R : N) : N;
  if (N <= kFusedMax) {
    DSPARK_LAUNCH(kKindSchedFinish, st,
                  launch_pdl(schedule_fused_kernel, dim3(1), dim3(kFinThreads), 0, st, s.R,
                             s.gamma, imax0 < 0 ? 0 : imax0, s.early_stop, s.a, s.sps, s.rank,
                             s.ell, s.row_off, s.B_out, s.E_out, s.status));
    return cudaGetLastError();
  }
  cudaError_t e = cudaMemsetAsync(s.rank, 0, sizeof(int32_t) * (size_t)N, st);
  if (e != cudaSuccess) return e;
  const int bx = (N + kRankThreads - 1) / kRankThreads;
  // split the comparison range so the grid has a few waves on 152 SMs
  int n_split = 1;
  while ((long long)bx * n_split < 1024 && N / (n_split * 2) >= kRankChunk) n_split *= 2;
  const int per_split = (N + n_split - 1) / n_split;
  DSPARK_LAUNCH(kKindRank, st, rank_kernel<<<dim3(bx, n_split), kRankThreads, 0, st>>>(N, per_split, s.a, s.rank, s.status));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int imax = s.max_B > 0 ? (s.max_B - s.R < N ? s.max_B - s.R : N) : N;
  DSPARK_LAUNCH(kKindSchedFinish, st, schedule_finish_kernel<<<1, kFinThreads, 0, st>>>(s.R, s.gamma, imax < 0 ? 0 : imax,
                                                   s.early_stop, s.a, s.sps, s.rank, s.sfix,
                                                   s.ell, s.row_off, s.B_out, s.E_out, s.status));
  return cudaGetLastError();
}

}  // namespace dspark
