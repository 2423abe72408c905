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
// The fp32 path (and the tiny workload) uses this file end to end.
#include "common.cuh"

namespace dspark {

// ---------------------------------------------------------------- bias

template <typename T>
__global__ void __launch_bounds__(256) bias_kernel(int R, int V, int r, const T* __restrict__ E,
                                                   const T* __restrict__ Wt,
                                                   const int32_t* __restrict__ prev_base,
                                                   int prev_stride, float* __restrict__ bias,
                                                   uint32_t* status) {
  // Tile: 64 vocabulary columns x 32 requests, K in chunks of 32.
  __shared__ float Es[32][33];
  __shared__ float Ws[64][33];
  __shared__ int prev_s[32];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16
  const int v0 = blockIdx.x * 64, n0 = blockIdx.y * 32;
  if (threadIdx.x < 32) {
    int n = n0 + threadIdx.x;
    int p = -1;
    if (n < R) {
      p = prev_base[(size_t)n * prev_stride];
      if (p >= V || p < -1) {
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
                        const int32_t* prev_base, int prev_stride, float* bias, uint32_t* status,
                        cudaStream_t st) {
  dim3 grid((V + 63) / 64, (R + 31) / 32);
  if (dt == 0)
    DSPARK_LAUNCH(kKindBias, st, bias_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        R, V, r, (const __nv_bfloat16*)E, (const __nv_bfloat16*)Wt, prev_base, prev_stride, bias,
        status));
  else
    DSPARK_LAUNCH(kKindBias, st, bias_kernel<float><<<grid, 256, 0, st>>>(R, V, r, (const float*)E, (const float*)Wt,
                                             prev_base, prev_stride, bias, status));
  return cudaGetLastError();
}

// ---------------------------------------------------------------- tile weights

// Weight of one token relative to the tile reference: 2^(a - ref) <= 1.
// Returns the fixed-point units (2^-kFixRel) and the fp32 weight.
__device__ __forceinline__ long long rel_fix(float a, float ref, float* w_out) {
  float w = exp2f(a - ref);
  *w_out = w;
  return __float2ll_rn(w * 1099511627776.0f);  // 2^40
}

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
    S = ldexp((double)tot, (int)ref - kFixRel);
  }
  if (threadIdx.x == 0) part[(size_t)n * n_tiles + t] = S;
}

// Where the finish kernel gets the chosen tile's bias: the CUDA-core bias
// array of the workspace (bias != nullptr), or recomputed on CUDA cores from
// E, Wt and the previous token (the fused tensor-core pass stores no bias).
struct BiasSrc {
  const float* bias;
  const __nv_bfloat16* E;
  const __nv_bfloat16* Wt;
  const int32_t* prev;
  int prev_stride, r;
};

// bias_s[c] = E[prev] . Wt[v0 + c] for the TW columns of one tile: warp w
// takes columns w*TW/8 .. +TW/8, lanes split the rank dimension (16-byte
// loads of a Wt row, r a multiple of 8, r <= 256); all of a warp's row loads
// are issued before the reductions so their L2 latencies overlap.
template <int TW>
__device__ void tile_bias_recompute(const BiasSrc& b, int n, int V, int v0, float* erow,
                                    float* bias_s, uint32_t* status) {
  // erow (the previous token's E row, fp32) was filled at kernel start
  constexpr int CPW = TW / 8;
  (void)n;
  (void)status;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane * 8;
  const bool lane_on = j < b.r;
  uint4 raw[CPW];
#pragma unroll
  for (int c = 0; c < CPW; ++c) {
    const int v = v0 + warp * CPW + c;
    raw[c] = (lane_on && v < V) ? *reinterpret_cast<const uint4*>(b.Wt + (size_t)v * b.r + j)
                                : make_uint4(0, 0, 0, 0);
  }
  float e8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e8[i] = lane_on ? erow[j + i] : 0.f;
#pragma unroll
  for (int c = 0; c < CPW; ++c) {
    const uint32_t w4[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(w4[e] << 16), e8[2 * e], acc);
      acc = fmaf(__uint_as_float(w4[e] & 0xffff0000u), e8[2 * e + 1], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) bias_s[warp * CPW + c] = acc;
  }
  __syncthreads();
}

// One block per request: choose the tile whose running sum crosses u*S, then
// the token inside it by recomputing the tile's weights.  With a recomputed
// bias the tile's weights can differ from the partial pass in the last bits,
// so the position inside the tile is taken as the same fraction of the
// recomputed tile mass.
template <typename T, int TW>
__global__ void __launch_bounds__(256) draft_finish_kernel(
    int V, int gamma, int k, int n_tiles, const T* __restrict__ z, BiasSrc bsrc, ScalePair sc,
    int greedy, const double* __restrict__ part, const float* __restrict__ u,
    int32_t* __restrict__ tokens, double* __restrict__ q_lse, float* __restrict__ q_tok,
    uint32_t* status) {
  __shared__ double shd[32];
  __shared__ double incl_s[256];
  __shared__ long long shl[32];
  __shared__ float shf[32];
  __shared__ int shi[32];
  __shared__ ArgMax sha[32];
  __shared__ double base_s;
  __shared__ float bias_s[TW];
  __shared__ float erow[1024];
  const int n = blockIdx.x, tid = threadIdx.x;
  const size_t out = (size_t)n * gamma + k;
  if (greedy) {
    const ArgMax* P = reinterpret_cast<const ArgMax*>(part) + (size_t)n * n_tiles;
    ArgMax best{-INFINITY, 0x7fffffff};
    for (int t = tid; t < n_tiles; t += blockDim.x) best = better(best, P[t]);
    best = block_argmax(best, sha);
    if (tid == 0) {
      int tok = best.i;
      if (tok < 0 || tok >= V) {
        set_flag(status, kFlagNonFinite);
        tok = 0;
      }
      tokens[out] = tok;
      q_lse[out] = (double)best.v;
      q_tok[out] = 1.0f;
    }
    return;
  }
  if (bsrc.bias == nullptr) {
    // the previous token's E row, needed once the tile is chosen: load it now
    int tok = bsrc.prev[(size_t)n * bsrc.prev_stride];
    if (tok >= V || tok < -1) {
      if (tid == 0) set_flag(status, kFlagTokenRange);
      tok = -1;
    }
    for (int i = tid; i < bsrc.r; i += blockDim.x)
      erow[i] = tok >= 0 ? __bfloat162float(bsrc.E[(size_t)tok * bsrc.r + i]) : 0.f;
  }
  const double* S = part + (size_t)n * n_tiles;
  const int seg = (n_tiles + blockDim.x - 1) / blockDim.x;
  const int t0 = min(n_tiles, tid * seg), t1 = min(n_tiles, t0 + seg);
  double loc = 0.0;
  for (int t = t0; t < t1; ++t) loc += S[t];
  double incl = block_inclusive_scan(loc, shd);
  incl_s[tid] = incl;
  __syncthreads();
  const double excl = tid > 0 ? incl_s[tid - 1] : 0.0;
  const double total = incl_s[blockDim.x - 1];
  const double thr = (double)u[out] * total;
  int cand = 0x7fffffff;
  double base = 0.0;
  {
    double run = excl;
    for (int t = t0; t < t1; ++t) {
      double nx = run + S[t];
      if (nx > thr) {
        cand = t;
        base = run;
        break;
      }
      run = nx;
    }
  }
  int tsel = block_min_int(cand, shi);
  if (tsel == 0x7fffffff) {
    // rounding left no crossing: last tile with mass
    int last = -1;
    for (int t = t0; t < t1; ++t)
      if (S[t] > 0.0) last = t;
    tsel = block_max_int(last, shi);
    if (tsel < 0) tsel = 0;
    if (tid == 0) base_s = -1.0;  // marks the fallback
  } else if (cand == tsel) {
    base_s = base;
  }
  __syncthreads();
  const bool fallback = base_s < 0.0;
  base = base_s;
  // Recompute the chosen tile.
  const int v = tsel * TW + tid;
  const bool ok = tid < TW && v < V;
  const float zv = ok ? ldf(z, out * V + v) : 0.f;  // issued before the bias loads
  float bv = 0.f;
  if (bsrc.bias != nullptr) {
    if (ok) bv = bsrc.bias[(size_t)n * V + v];
  } else {
    tile_bias_recompute<TW>(bsrc, n, V, tsel * TW, erow, bias_s, status);
    bv = tid < TW ? bias_s[tid] : 0.f;
  }
  float y = -INFINITY;
  if (ok) y = zv + bv;
  if (ok && (isnan(y) || y == INFINITY)) y = -INFINITY;
  const float a = scaled(y, sc);
  const float amax = block_max(a, shf);
  const float ref = ceilf(amax);
  float w = 0.f;
  long long f = (ok && a > -INFINITY && amax > -INFINITY) ? rel_fix(a, ref, &w) : 0ll;
  long long cum = block_inclusive_scan(f, shl);
  __syncthreads();
  if (tid == blockDim.x - 1) incl_s[0] = ldexp((double)cum, (int)ref - kFixRel);
  __syncthreads();
  const double tile_mass = incl_s[0];
  // the crossing's position inside the tile, as a fraction of the tile mass
  const double target = S[tsel] > 0.0 ? (thr - base) * (tile_mass / S[tsel]) : 0.0;
  int pick = 0x7fffffff;
  if (!fallback && f > 0 && ldexp((double)cum, (int)ref - kFixRel) > target) pick = tid;
  int isel = block_min_int(pick, shi);
  if (isel == 0x7fffffff) isel = block_max_int(f > 0 ? tid : -1, shi);
  if (isel < 0) isel = 0;
  if (tid == isel) {
    tokens[out] = tsel * TW + isel;
    if (!(total > 0.0) || !isfinite(total)) set_flag(status, kFlagNonFinite);
    q_lse[out] = log(total);
    q_tok[out] = (float)(ldexp((double)w, (int)ref) / total);
  }
}

template <typename T, int TW>
cudaError_t launch_finish(const DraftArgs& a, int k, const BiasSrc& b, ScalePair sc, bool greedy,
                          cudaStream_t st) {
  const int n_tiles = (a.V + TW - 1) / TW;
  DSPARK_LAUNCH(kKindDraftFinish, st,
                draft_finish_kernel<T, TW><<<a.R, 256, 0, st>>>(
                    a.V, a.gamma, k, n_tiles, (const T*)a.z, b, sc, greedy, a.part, a.u,
                    a.tokens, a.q_lse, a.q_tok, a.status));
  return cudaGetLastError();
}

cudaError_t launch_draft(const DraftArgs& a, cudaStream_t st) {
  const int n_tiles = (a.V + kTileV - 1) / kTileV;
  const bool greedy = a.T == 0.0f;
  const ScalePair sc = make_scale(greedy ? 1.0 : 1.4426950408889634 / (double)a.T);
  const bool tc = draft_tc_supported(a);
  for (int k = 0; k < a.gamma; ++k) {
    const int32_t* prev = k == 0 ? a.anchor : a.tokens + (k - 1);
    const int stride = k == 0 ? 1 : a.gamma;
    cudaError_t e;
    if (tc) {
      // bf16 on the tensor cores: fused bias GEMM + partial pass, then the
      // finish recomputes the chosen tile's bias
      e = launch_draft_partial_tc(a, k, prev, stride, st);
      if (e != cudaSuccess) return e;
      BiasSrc b{nullptr, (const __nv_bfloat16*)a.E, (const __nv_bfloat16*)a.Wt, prev, stride, a.r};
      e = launch_finish<__nv_bfloat16, 128>(a, k, b, sc, greedy, st);
      if (e != cudaSuccess) return e;
      continue;
    }
    e = launch_bias(a.R, a.V, a.r, a.dt, a.E, a.Wt, prev, stride, a.bias, a.status, st);
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
