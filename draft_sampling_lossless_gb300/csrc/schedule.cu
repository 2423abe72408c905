// Hardware-aware prefix scheduler: one launch of one thread-block cluster.
//
// News article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 2.2: maximise tau * SPS(B) over the
// per-request verify lengths, B = sum_r (1 + l_r); sort every candidate by its
// survival probability, add them greedily, stop as soon as throughput stops
// rising (O(gamma R log gamma R)); challenge 2: the same search without early
// stop, and asynchronous scheduling -- a capacity fixed before the step (from
// the confidences of two steps earlier) filled with the current candidates,
// still taken in the current order.  Explainer "DSpark.让每一轮计算，多走几步",
// survival panel: E = R + sum a, rate = E / T(B).
//
// The kernel (schedule_radix_kernel) runs on a cluster of C <= 8 CTAs of 512
// threads (one CTA per 1024 candidates, so a mid-size batch still has several
// CTAs' loads in flight); CTA c owns a contiguous chunk of the candidates and of the
// requests.  Candidates are 64-bit words (key << 32 | flat index n*gamma + j)
// with key = 0xffffffff - bits(a): for a >= 0 the float's bits order like its
// value, so ascending keys are descending a.
//
//   sort  -- a stable LSD radix sort of the keys, 8 bits a pass, four
//            passes.  A pass: each warp counts the digits of its contiguous
//            slice (__match_any_sync groups equal digits, the group's lowest
//            lane adds its size); the CTA's digit totals go to shared memory,
//            where every CTA of the cluster reads them (distributed shared
//            memory) after a cluster barrier; each thread then has, for its
//            digit, the number of smaller digits in the whole batch and of
//            equal digits in the CTAs before its own, and the warps scatter
//            their slices in order to a global ping-pong buffer (a warp's
//            equal digits ranked by their lane).  Stability makes the flat
//            index the tie-break, so the order is (a descending, request,
//            position).  A pass in which every candidate has the same digit
//            is the identity and is skipped.
//   scan  -- the rank of every candidate, the exact 2^-40 fixed-point
//            prefix sums S_i in sorted order (per-thread runs, a block scan,
//            the CTAs' totals through distributed shared memory), Theta_i
//            with the double roundings of the oracle's expression reproduced
//            in integer arithmetic, and the cut: the first i with
//            Theta_{i+1} <= Theta_i (early stop), the first argmax (global),
//            or i = min(max(K - R, 0), R*gamma) (capacity K read on the
//            device), reduced over the cluster;
//   lengths -- l_r = the number of request r's candidates ranked below the
//            cut, row_off = the exclusive scan of 1 + l_r over the cluster's
//            request chunks, B = R + i*, E = R + S_{i*}.
// No floating-point double instruction runs here.  The persistent draft
// kernel can run its own form of the scheduler after its last position
// (dspark_draft_schedule, schedule.cuh) with the same definitions.
#include <cooperative_groups.h>

#include "common.cuh"
#include "schedule.cuh"

namespace dspark {

namespace {

namespace cg = cooperative_groups;
using namespace sched;

constexpr int kSortThreads = 512;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kBins = 256;
constexpr int kMaxClusterCtas = 8;
constexpr int kPerCta = 1024;  // candidates a CTA owns before the cluster grows

enum { kModeEarly = 0, kModeGlobal = 1, kModeCapacity = 2 };

// The candidate word of flat index e, from its survival value (cleaned: NaN,
// negative or infinite values count as 0 and are flagged).
__device__ __forceinline__ unsigned long long candidate(const float* __restrict__ a, int e,
                                                        uint32_t* status) {
  const float v = clean_a(a[e], status) + 0.0f;  // -0 -> +0
  return ((unsigned long long)(0xffffffffu - __float_as_uint(v)) << 32) | (unsigned)e;
}

__device__ __forceinline__ float value_of(unsigned long long x) {
  return __uint_as_float(0xffffffffu - (unsigned)(x >> 32));
}

// Block-wide (largest key, lowest index) over all threads; every thread gets it.
__device__ inline void block_best(unsigned long long& v, int& i, unsigned long long* shk,
                                  int* shi) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
  __syncthreads();
  if (lane == 0) {
    shk[wid] = v;
    shi[wid] = i;
  }
  __syncthreads();
  v = lane < nw ? shk[lane] : 0ull;
  i = lane < nw ? shi[lane] : 0x7fffffff;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

__global__ void __launch_bounds__(kSortThreads) schedule_radix_kernel(
    int R, int gamma, int imax, int mode, const int32_t* __restrict__ capacity,
    const float* __restrict__ a, const float* __restrict__ sps,
    unsigned long long* __restrict__ buf0, unsigned long long* __restrict__ buf1,
    int32_t* __restrict__ rank, int32_t* __restrict__ ell, int32_t* __restrict__ row_off,
    int32_t* __restrict__ B_out, double* __restrict__ E_out, uint32_t* status) {
  __shared__ int wcnt[kSortWarps][kBins];  // a warp's digit counts, then its scatter bases
  __shared__ int hist[2][kBins];           // this CTA's digit totals (read cluster-wide)
  __shared__ int skip_s[4];  // a pass whose digit is uniform (one flag a pass)
  __shared__ long long shl[32];
  __shared__ int shi[32];
  __shared__ unsigned long long shk[32];
  __shared__ long long cta_sum;  // this CTA's fixed-point total (read cluster-wide)
  __shared__ long long cta_rows;  // this CTA's sum of 1 + l_r (read cluster-wide)
  __shared__ int cut_i;           // this CTA's stop / argmax index (read cluster-wide)
  __shared__ unsigned long long cut_v;

  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks(), c = (int)cl.block_rank();
  const int N = R * gamma;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int chunk = (N + C - 1) / C;
  const int c0 = min(N, c * chunk), c1 = min(N, c0 + chunk);
  const int wsub = (c1 - c0 + kSortWarps - 1) / kSortWarps;
  const int w0 = min(c1, c0 + wid * wsub), w1 = min(c1, w0 + wsub);
  const unsigned lt_mask = (1u << lane) - 1u;
  if (tid < 4) skip_s[tid] = 0;

  grid_dependency_wait();  // the survival values (and the capacity)

  // ------------------------------------------------------------- sort
  const unsigned long long* src = nullptr;
  unsigned long long* dst = buf0;
  int par = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int sh = 32 + 8 * pass;
    for (int i = tid; i < kSortWarps * kBins; i += kSortThreads) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    // four rounds of 32 at a time: their loads are in flight together
    for (int base = w0; base < w1; base += 128) {
      unsigned long long xs[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = base + q * 32 + lane;
        xs[q] = e < w1 ? (pass == 0 ? candidate(a, e, status) : src[e]) : 0ull;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool ok = base + q * 32 + lane < w1;
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (ok) {
          const unsigned d = (unsigned)(xs[q] >> sh) & 255u;
          const unsigned peers = __match_any_sync(m, d);
          if (lane == __ffs(peers) - 1) wcnt[wid][d] += __popc(peers);
        }
      }
    }
    __syncthreads();
    int mine = 0;  // this CTA's count of digit tid (tid < kBins)
    if (tid < kBins) {
      for (int w = 0; w < kSortWarps; ++w) {
        const int x = wcnt[w][tid];
        wcnt[w][tid] = mine;  // the warps before w
        mine += x;
      }
      hist[par][tid] = mine;
    }
    cl.sync();  // every CTA's totals of this pass are in place
    int total = 0, before = 0;
    if (tid < kBins) {
      for (int q = 0; q < C; ++q) {
        const int x = cl.map_shared_rank(&hist[par][0], q)[tid];
        total += x;
        before += q < c ? x : 0;
      }
      if (total == N) skip_s[pass] = 1;
    }
    const int incl = block_inclusive_scan(tid < kBins ? total : 0, shi);
    __syncthreads();
    const bool skip = pass > 0 && skip_s[pass] != 0;  // uniform over the cluster
    if (!skip) {
      if (tid < kBins) {
        const int base = incl - total + before;  // smaller digits + this digit in earlier CTAs
        for (int w = 0; w < kSortWarps; ++w) wcnt[w][tid] += base;
      }
      __syncthreads();
      for (int base = w0; base < w1; base += 128) {
        unsigned long long xs[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = base + q * 32 + lane;
          xs[q] = e < w1 ? (pass == 0 ? candidate(a, e, status) : src[e]) : 0ull;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // in order: the scatter is stable
          const bool ok = base + q * 32 + lane < w1;
          const unsigned m = __ballot_sync(0xffffffffu, ok);
          unsigned d = 0, peers = 0;
          int pos = 0;
          if (ok) {
            d = (unsigned)(xs[q] >> sh) & 255u;
            peers = __match_any_sync(m, d);
            pos = wcnt[wid][d] + __popc(peers & lt_mask);
          }
          __syncwarp();
          if (ok && lane == __ffs(peers) - 1) wcnt[wid][d] += __popc(peers);
          __syncwarp();
          if (ok) dst[pos] = xs[q];
        }
      }
      cl.sync();  // the pass's output is complete and visible to the cluster
      src = dst;
      dst = dst == buf0 ? buf1 : buf0;
    }
    par ^= 1;
  }
  const unsigned long long* srt = src;

  // ------------------------------------------------------------- scan
  // thread-contiguous sorted positions [t0, t1) of this CTA's chunk
  const int tseg = (c1 - c0 + kSortThreads - 1) / kSortThreads;
  const int t0 = min(c1, c0 + tid * tseg), t1 = min(c1, t0 + tseg);
  long long loc = 0;
  for (int p = t0; p < t1; ++p) {
    const unsigned long long x = srt[p];
    rank[(unsigned)x] = p;
    loc += to_fixed(value_of(x));
  }
  const long long incl = block_inclusive_scan(loc, shl);
  if (tid == kSortThreads - 1) cta_sum = incl;
  cl.sync();  // ranks written, every CTA's total published
  long long S = incl - loc;  // S_{t0}: the values before position t0
  for (int q = 0; q < c; ++q) S += *cl.map_shared_rank(&cta_sum, q);
  // Theta_i is evaluated by the thread owning position i; i = N by the
  // thread owning position N - 1
  const int t1e = t1 + (t1 == N && t0 < t1 ? 1 : 0);
  int istar;
  if (mode == kModeCapacity) {
    const long long i = (long long)__ldg(capacity) - R;
    istar = (int)(i < 0 ? 0 : (i > N ? N : i));
  } else {
    const int ia = t0, ib = min(t1e, imax + 1);
    int my_stop = 0x7fffffff;
    unsigned long long best_v = 0;
    int best_i = 0x7fffffff;
    long long Si = S;
    unsigned long long prev_th = 0;
    for (int i = ia; i < ib; ++i) {
      const unsigned long long th = theta_key_of(R, i, Si, sps, status);
      if (i > ia && !(th > prev_th) && my_stop == 0x7fffffff) my_stop = i - 1;
      if (best_i == 0x7fffffff || th > best_v) {
        best_v = th;
        best_i = i;
      }
      prev_th = th;
      if (i < N) Si += to_fixed(value_of(srt[i]));
    }
    // the pair that straddles the end of the thread's range, (ib - 1, ib)
    if (ib > ia && ib <= imax && my_stop == 0x7fffffff) {
      const unsigned long long th = theta_key_of(R, ib, Si, sps, status);
      if (!(th > prev_th)) my_stop = ib - 1;
    }
    if (mode == kModeEarly) {
      const int st = block_min_int(my_stop, shi);
      if (tid == 0) cut_i = st;
      cl.sync();
      int s = 0x7fffffff;
      for (int q = 0; q < C; ++q) s = min(s, *cl.map_shared_rank(&cut_i, q));
      istar = s == 0x7fffffff ? imax : s;
    } else {
      block_best(best_v, best_i, shk, shi);
      if (tid == 0) {
        cut_v = best_v;
        cut_i = best_i;
      }
      cl.sync();
      unsigned long long v = 0;
      int bi = 0x7fffffff;
      for (int q = 0; q < C; ++q) {
        const unsigned long long ov = *cl.map_shared_rank(&cut_v, q);
        const int oi = *cl.map_shared_rank(&cut_i, q);
        if (ov > v || (ov == v && oi < bi)) {
          v = ov;
          bi = oi;
        }
      }
      istar = bi == 0x7fffffff ? 0 : bi;
    }
  }
  // B and E by the thread whose range holds i*
  if (istar >= t0 && istar < t1e) {
    long long Sx = S;
    for (int p = t0; p < istar; ++p) Sx += to_fixed(value_of(srt[p]));
    schedule_store_EB(R, istar, Sx, B_out, E_out);
  }

  // ------------------------------------------------------------- lengths
  const int rchunk = (R + C - 1) / C;
  const int r0 = min(R, c * rchunk), r1 = min(R, r0 + rchunk);
  const int rseg = (r1 - r0 + kSortThreads - 1) / kSortThreads;
  const int q0 = min(r1, r0 + tid * rseg), q1 = min(r1, q0 + rseg);
  long long lsum = 0;
  for (int r = q0; r < q1; ++r) {
    int cnt = 0;
#pragma unroll 8
    for (int j = 0; j < gamma; ++j) cnt += __ldcg(rank + (size_t)r * gamma + j) < istar;
    ell[r] = cnt;
    lsum += 1 + cnt;
  }
  const long long rin = block_inclusive_scan(lsum, shl);
  if (tid == kSortThreads - 1) cta_rows = rin;
  cl.sync();
  long long run = rin - lsum;
  for (int q = 0; q < c; ++q) run += *cl.map_shared_rank(&cta_rows, q);
  if (r1 == R && r0 < r1 && tid == kSortThreads - 1) row_off[R] = (int32_t)(run + lsum);
  for (int r = q0; r < q1; ++r) {
    row_off[r] = (int32_t)run;
    run += 1 + ell[r];
  }
  cl.sync();  // no CTA leaves while another may still read its shared memory
}

cudaError_t launch_radix(const SchedArgs& s, int mode, const int32_t* capacity, int imax,
                         cudaStream_t st) {
  const int N = s.R * s.gamma;
  int C = (N + kPerCta - 1) / kPerCta;
  C = C < 1 ? 1 : (C > kMaxClusterCtas ? kMaxClusterCtas : C);
  unsigned long long* buf0 = s.keys;
  unsigned long long* buf1 = s.keys + N;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kSortThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 2 : 1;  // one CTA: a plain launch (an implicit cluster of one)
  cudaError_t e = cudaSuccess;
  DSPARK_LAUNCH(kKindSchedule, st,
                e = cudaLaunchKernelEx(&cfg, schedule_radix_kernel, s.R, s.gamma, imax, mode,
                                       capacity, s.a, s.sps, buf0, buf1, s.rank, s.ell,
                                       s.row_off, s.B_out, s.E_out, s.status));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_schedule(const SchedArgs& s, cudaStream_t st) {
  const int N = s.R * s.gamma;
  int imax = s.max_B > 0 ? (s.max_B - s.R < N ? s.max_B - s.R : N) : N;
  if (imax < 0) imax = 0;
  return launch_radix(s, s.early_stop ? kModeEarly : kModeGlobal, nullptr, imax, st);
}

cudaError_t launch_schedule_async(const SchedArgs& s, const int32_t* capacity, cudaStream_t st) {
  return launch_radix(s, kModeCapacity, capacity, s.R * s.gamma, st);
}

}  // namespace dspark
