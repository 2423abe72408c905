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
// For R * gamma <= 1024 one block does both steps below (schedule_fused_
// kernel); larger batches take two launches:
//   rank   -- the position of every candidate in the total order
//             (a descending, then flat index n*gamma + j ascending), counted by
//             comparisons against all others; ranks are a permutation because
//             the order is strict, so no sort network or stable radix pass is
//             needed and the result does not depend on thread timing.
//   finish -- one block: scatter to sorted order, exact integer prefix sums of
//             the 2^-40 fixed-point survival values, Theta_i rounded exactly as
//             the oracle's double arithmetic rounds it, the early-stop or
//             argmax cut, then l_r, row_off, B and E.
// The persistent draft kernel can run the same steps after its last position
// (dspark_draft_schedule): its idle CTAs rank the candidates and form the
// prefixes and Theta keys, one CTA finds the cut (schedule.cuh).
// No floating-point double instruction runs here: the double roundings are
// reproduced with integer arithmetic (round to nearest, ties to even), which
// gives the same bits and avoids the narrow FP64 pipe.
#include "common.cuh"
#include "schedule.cuh"

namespace dspark {

namespace {

using namespace sched;

constexpr int kRankThreads = 256;
constexpr int kRankChunk = 2048;
constexpr int kFinThreads = 1024;

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
