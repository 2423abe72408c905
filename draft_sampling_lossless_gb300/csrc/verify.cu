// Lossless rejection-sampling and greedy verification.
//
// Forum post "为什么DSpark 可以加速推理？以及DSpark会不会导致降智？", lossless
// proof: accept the drafted token with probability min(1, p/q); on rejection
// draw from max(0, p - q) normalised; the emitted marginal is p.  Explainer
// "DSpark.让每一轮计算，多走几步", lossless panel: if the whole block passes,
// one more (bonus) token comes from the next target distribution.  CSDN
// tutorial, section 五: the first rejection ends the block.
//
// Launches (stochastic; greedy needs only the first two):
//   rows    -- every verified target row streamed once in 4096-token chunks:
//              exact chunk sums of 2^(t*log2e/T - ref) (greedy: chunk argmax)
//   decide  -- per request: row normalisers, p_lse, the sequential accept test
//              u < p(x)/q(x), n_acc, the accepted tokens and the final-draw setup
//   bias    -- Markov bias of each rejected position (CUDA cores)
//   final   -- per (request, 256-token tile): exact fixed-point sums of the
//              residual max(0, p - q) and of p, both normalised
//   pick    -- per request: inverse CDF over the tiles and inside the tile, with
//              an exact integer comparison against u * total
#include "common.cuh"

namespace dspark {

namespace {

constexpr int kRowThreads = 256;
constexpr int kPerThread = kChunkV / kRowThreads;  // 16

template <typename T>
__global__ void __launch_bounds__(kRowThreads) verify_rows_kernel(
    int gamma, int V, int n_chunks, long long n_rows, const T* __restrict__ target,
    const int32_t* __restrict__ ell, const int32_t* __restrict__ row_off, ScalePair sc,
    int greedy, double* __restrict__ row_part) {
  __shared__ float shf[32];
  __shared__ long long shl[32];
  __shared__ ArgMax sha[32];
  const int c = blockIdx.x, j = blockIdx.y, n = blockIdx.z;
  const int L = ell[n];
  if (j > L || L > gamma) return;
  const long long row = (long long)row_off[n] + j;
  if (row < 0 || row >= n_rows) return;  // reported by the decide kernel
  const T* tr = target + (size_t)row * V;
  const int base = c * kChunkV + threadIdx.x;
  double* out = row_part + ((size_t)n * (gamma + 1) + j) * n_chunks + c;
  if (greedy) {
    ArgMax am{-INFINITY, 0x7fffffff};
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int v = base + e * kRowThreads;
      if (v < V) am = better(am, ArgMax{to_f32<T>(tr[v]), v});
    }
    am = block_argmax(am, sha);
    if (threadIdx.x == 0) *reinterpret_cast<ArgMax*>(out) = am;
    return;
  }
  float a[kPerThread];
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    const int v = base + e * kRowThreads;
    float t = v < V ? to_f32<T>(tr[v]) : -INFINITY;
    if (isnan(t) || t == INFINITY) t = -INFINITY;  // flagged by the decide kernel's checks
    a[e] = scaled(t, sc);
    m = fmaxf(m, a[e]);
  }
  m = block_max(m, shf);
  double S = 0.0;
  if (m > -INFINITY) {
    const float ref = ceilf(m);
    long long f = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e)
      if (a[e] > -INFINITY) f += __float2ll_rn(exp2f(a[e] - ref) * 1099511627776.0f);
    f = block_sum(f, shl);
    S = ldexp((double)f, (int)ref - kFixRel);
  }
  if (threadIdx.x == 0) *out = S;
}

template <typename T>
__global__ void __launch_bounds__(256) verify_decide_kernel(
    int gamma, int V, int n_chunks, long long n_rows, const T* __restrict__ target,
    ScalePair sc, int greedy, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const double* __restrict__ q_lse,
    const float* __restrict__ q_tok, const int32_t* __restrict__ ell,
    const int32_t* __restrict__ row_off, const float* __restrict__ u_acc,
    const double* __restrict__ row_part, double* __restrict__ p_lse,
    int32_t* __restrict__ n_acc_out, int32_t* __restrict__ out_tokens,
    VerifyState* __restrict__ vstate, int32_t* __restrict__ prev_out, uint32_t* status) {
  __shared__ double Sp[kMaxGamma + 1];
  __shared__ ArgMax am_s[kMaxGamma + 1];
  __shared__ int bad_s;
  const int n = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int L = ell[n];
  const long long r0 = row_off[n];
  if (tid == 0) {
    bad_s = (L < 0 || L > gamma || r0 < 0 || r0 + L >= n_rows);
    if (bad_s) set_flag(status, kFlagRowRange);
  }
  __syncthreads();
  int32_t* ot = out_tokens + (size_t)n * (gamma + 1);
  if (bad_s) {
    for (int j = tid; j <= gamma; j += blockDim.x) ot[j] = -1;
    if (tid == 0) {
      n_acc_out[n] = 0;
      VerifyState st{0, -1, 0, -1, 0.0, 0.0};
      vstate[n] = st;
      prev_out[n] = -1;
    }
    return;
  }
  const double* part = row_part + (size_t)n * (gamma + 1) * n_chunks;
  for (int j = wid; j <= L; j += blockDim.x >> 5) {
    const double* pj = part + (size_t)j * n_chunks;
    if (greedy) {
      ArgMax am{-INFINITY, 0x7fffffff};
      for (int c = lane; c < n_chunks; c += 32) am = better(am, reinterpret_cast<const ArgMax*>(pj)[c]);
      am = warp_argmax(am);
      if (lane == 0) {
        am_s[j] = am;
        if (p_lse) p_lse[r0 + j] = (double)am.v;
      }
    } else {
      double s = 0.0;
      for (int c = lane; c < n_chunks; c += 32) s += pj[c];
      s = warp_sum(s);
      if (lane == 0) {
        Sp[j] = s;
        if (!(s > 0.0) || !isfinite(s)) set_flag(status, kFlagNonFinite);
        if (p_lse) p_lse[r0 + j] = log(s);
      }
    }
  }
  __syncthreads();
  if (tid != 0) return;
  int nacc = L;
  for (int j = 0; j < L; ++j) {
    const int x = tokens[(size_t)n * gamma + j];
    bool acc;
    if (x < 0 || x >= V) {
      set_flag(status, kFlagTokenRange);
      acc = false;
    } else if (greedy) {
      acc = (x == am_s[j].i);
    } else {
      const float tx = to_f32<T>(target[(size_t)(r0 + j) * V + x]);
      const double px = exp2((double)scaled(tx, sc)) / Sp[j];
      const double ratio = px / (double)q_tok[(size_t)n * gamma + j];
      acc = (double)u_acc[(size_t)n * gamma + j] < ratio;
    }
    if (!acc) {
      nacc = j;
      break;
    }
  }
  n_acc_out[n] = nacc;
  for (int j = 0; j <= gamma; ++j) {
    int v = -1;
    if (j < nacc) v = tokens[(size_t)n * gamma + j];
    else if (j == nacc && greedy) v = am_s[nacc].i;
    ot[j] = v;
  }
  VerifyState st;
  st.n_acc = nacc;
  st.mode = greedy ? -1 : (nacc == L ? 0 : 1);
  st.final_row = (int)(r0 + nacc);
  st.prev = -1;
  st.Sp = greedy ? 0.0 : Sp[nacc];
  st.Sq = 0.0;
  if (st.mode == 1) {
    st.prev = nacc == 0 ? anchor[n] : tokens[(size_t)n * gamma + nacc - 1];
    st.Sq = exp(q_lse[(size_t)n * gamma + nacc]);
  }
  vstate[n] = st;
  prev_out[n] = st.prev;
}

// Normalised weight split as (hi, lo) fp32 for k = 2^ref / S in double.
__device__ __forceinline__ ScalePair norm_pair(float ref, double S) {
  const double k = ldexp(1.0, (int)ref) / S;
  ScalePair p;
  p.hi = (float)k;
  p.lo = (float)(k - (double)p.hi);
  return p;
}

// Weights of token v of request n's final draw: p (target, normalised) and
// the residual max(0, p - q) (mode 1) -- recomputed identically by the pick
// kernel.  Returns fixed-point units of 2^-60 for both.  The tile's power-of-
// two references and the double-float scales 2^ref / S are formed once per
// block (thread 0) and shared through `shk`.
template <typename T>
__device__ void final_tile_weights(int gamma, int V, int t, const T* __restrict__ z,
                                   const float* __restrict__ bias, const T* __restrict__ target,
                                   ScalePair sc, const VerifyState& st, int n, float* shf,
                                   ScalePair* shk, long long* fr, long long* fp) {
  const int v = t * kTileV + threadIdx.x;
  const bool ok = v < V;
  float tv = ok ? to_f32<T>(target[(size_t)st.final_row * V + v]) : -INFINITY;
  if (isnan(tv) || tv == INFINITY) tv = -INFINITY;
  const float ap = scaled(tv, sc);
  float aq = -INFINITY;
  if (st.mode == 1 && ok) {
    float y = to_f32<T>(z[((size_t)n * gamma + st.n_acc) * V + v]) + bias[(size_t)n * V + v];
    if (isnan(y) || y == INFINITY) y = -INFINITY;
    aq = scaled(y, sc);
  }
  const float mp = block_max(ap, shf);
  const float mq = st.mode == 1 ? block_max(aq, shf) : -INFINITY;
  if (threadIdx.x == 0) {
    shk[0] = mp > -INFINITY ? norm_pair(ceilf(mp), st.Sp) : ScalePair{0.f, 0.f};
    shk[1] = mq > -INFINITY ? norm_pair(ceilf(mq), st.Sq) : ScalePair{0.f, 0.f};
  }
  __syncthreads();
  float p = 0.f;
  if (ap > -INFINITY) {
    const float w = exp2f(ap - ceilf(mp));
    p = fmaf(w, shk[0].hi, w * shk[0].lo);
  }
  float rho = p;
  if (st.mode == 1) {
    float q = 0.f;
    if (aq > -INFINITY) {
      const float w = exp2f(aq - ceilf(mq));
      q = fmaf(w, shk[1].hi, w * shk[1].lo);
    }
    rho = fmaxf(0.0f, p - q);
  }
  constexpr float k2_60 = 1152921504606846976.0f;  // 2^60
  *fp = __float2ll_rn(p * k2_60);
  *fr = __float2ll_rn(rho * k2_60);
}

template <typename T>
__global__ void __launch_bounds__(kTileV) final_partial_kernel(
    int gamma, int V, int n_tiles, const T* __restrict__ z, const float* __restrict__ bias,
    const T* __restrict__ target, ScalePair sc, const VerifyState* __restrict__ vstate,
    long long* __restrict__ fin_part) {
  __shared__ float shf[32];
  __shared__ long long shl[32];
  __shared__ ScalePair shk[2];
  const int t = blockIdx.x, n = blockIdx.y;
  const VerifyState st = vstate[n];
  long long* out = fin_part + ((size_t)n * n_tiles + t) * 2;
  if (st.mode < 0) {
    if (threadIdx.x == 0) out[0] = out[1] = 0;
    return;
  }
  long long fr, fp;
  final_tile_weights<T>(gamma, V, t, z, bias, target, sc, st, n, shf, shk, &fr, &fp);
  fr = block_sum(fr, shl);
  fp = block_sum(fp, shl);
  if (threadIdx.x == 0) {
    out[0] = fr;
    out[1] = fp;
  }
}

// floor(u * F) exactly, for u in [0, 1) and 0 <= F < 2^62.
__device__ __forceinline__ long long floor_mul(float u, long long F) {
  if (!(u > 0.0f)) return 0;
  int e;
  const float mf = frexpf(u, &e);  // u = mf * 2^e, mf in [0.5, 1)
  const unsigned long long m = (unsigned long long)(mf * 16777216.0f);  // u = m * 2^(e-24)
  const unsigned long long lo = m * (unsigned long long)F;
  const unsigned long long hi = __umul64hi(m, (unsigned long long)F);
  const int sh = 24 - e;
  if (sh <= 0) return F;  // u >= 1: outside the contract, clamp
  if (sh >= 128) return 0;
  if (sh >= 64) return (long long)(hi >> (sh - 64));
  return (long long)((lo >> sh) | (hi << (64 - sh)));
}

template <typename T>
__global__ void __launch_bounds__(kTileV) final_pick_kernel(
    int gamma, int V, int n_tiles, const T* __restrict__ z, const float* __restrict__ bias,
    const T* __restrict__ target, ScalePair sc, const VerifyState* __restrict__ vstate,
    const long long* __restrict__ fin_part, const float* __restrict__ u_fin,
    int32_t* __restrict__ out_tokens, uint32_t* status) {
  __shared__ float shf[32];
  __shared__ long long shl[32];
  __shared__ int shi[32];
  __shared__ long long incl_s[kTileV];
  __shared__ long long base_s;
  __shared__ ScalePair shk[2];
  const int n = blockIdx.x, tid = threadIdx.x;
  const VerifyState st = vstate[n];
  if (st.mode < 0) return;
  const long long* P = fin_part + (size_t)n * n_tiles * 2;
  const int seg = (n_tiles + blockDim.x - 1) / blockDim.x;
  const int t0 = min(n_tiles, tid * seg), t1 = min(n_tiles, t0 + seg);
  long long lr = 0, lp = 0;
  for (int t = t0; t < t1; ++t) {
    lr += P[2 * t];
    lp += P[2 * t + 1];
  }
  const long long Fr = block_sum(lr, shl);
  const int col = (st.mode == 1 && Fr > 0) ? 0 : 1;
  const long long loc = col == 0 ? lr : lp;
  const long long incl = block_inclusive_scan(loc, shl);
  incl_s[tid] = incl;
  __syncthreads();
  const long long F = incl_s[blockDim.x - 1];
  if (F <= 0) {
    if (tid == 0) {
      set_flag(status, kFlagNonFinite);
      out_tokens[(size_t)n * (gamma + 1) + st.n_acc] = 0;
    }
    return;
  }
  const long long thr = floor_mul(u_fin[n], F);  // C > u*F  <=>  C > floor(u*F)
  int cand = 0x7fffffff;
  long long base = 0;
  {
    long long run = incl - loc;
    for (int t = t0; t < t1; ++t) {
      const long long nx = run + P[2 * t + col];
      if (nx > thr) {
        cand = t;
        base = run;
        break;
      }
      run = nx;
    }
  }
  const int tsel = block_min_int(cand, shi);  // always found: the total exceeds thr
  if (cand == tsel) base_s = base;
  __syncthreads();
  base = base_s;
  long long fr, fp;
  final_tile_weights<T>(gamma, V, tsel, z, bias, target, sc, st, n, shf, shk, &fr, &fp);
  const long long f = col == 0 ? fr : fp;
  const long long cum = block_inclusive_scan(f, shl);
  int pick = (f > 0 && base + cum > thr) ? tid : 0x7fffffff;
  int isel = block_min_int(pick, shi);
  if (isel == 0x7fffffff) isel = block_max_int(f > 0 ? tid : -1, shi);
  if (isel < 0) isel = 0;
  if (tid == 0) out_tokens[(size_t)n * (gamma + 1) + st.n_acc] = tsel * kTileV + isel;
}

template <typename T>
cudaError_t run_verify(const VerifyArgs& a, cudaStream_t st) {
  const bool greedy = a.T == 0.0f;
  const ScalePair sc = make_scale(greedy ? 1.0 : 1.4426950408889634 / (double)a.T);
  const int n_chunks = (a.V + kChunkV - 1) / kChunkV;
  const int n_tiles = (a.V + kTileV - 1) / kTileV;
  const T* z = (const T*)a.z;
  const T* tg = (const T*)a.target;
  DSPARK_LAUNCH(kKindVerifyRows, st, verify_rows_kernel<T><<<dim3(n_chunks, a.gamma + 1, a.R), kRowThreads, 0, st>>>(
      a.gamma, a.V, n_chunks, a.n_rows, tg, a.ell, a.row_off, sc, greedy, a.row_part));
  DSPARK_LAUNCH(kKindVerifyDecide, st, verify_decide_kernel<T><<<a.R, 256, 0, st>>>(
      a.gamma, a.V, n_chunks, a.n_rows, tg, sc, greedy, a.anchor, a.tokens, a.q_lse, a.q_tok,
      a.ell, a.row_off, a.u_acc, a.row_part, a.p_lse, a.n_acc, a.out_tokens, a.vstate, a.prev,
      a.status));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || greedy) return e;
  e = tc_shape_supported(a.dt, a.V, a.r, a.z, a.E, a.Wt)
          ? launch_bias_tc(a.R, a.V, a.r, a.E, a.Wt, a.prev, 1, a.bias, a.status, st)
          : launch_bias(a.R, a.V, a.r, a.dt, a.E, a.Wt, a.prev, 1, a.bias, a.status, st);
  if (e != cudaSuccess) return e;
  DSPARK_LAUNCH(kKindFinalPartial, st, final_partial_kernel<T><<<dim3(n_tiles, a.R), kTileV, 0, st>>>(
      a.gamma, a.V, n_tiles, z, a.bias, tg, sc, a.vstate, a.fin_part));
  DSPARK_LAUNCH(kKindFinalPick, st, final_pick_kernel<T><<<a.R, kTileV, 0, st>>>(a.gamma, a.V, n_tiles, z, a.bias, tg, sc,
                                               a.vstate, a.fin_part, a.u_fin, a.out_tokens,
                                               a.status));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t st) {
  return a.dt == 0 ? run_verify<__nv_bfloat16>(a, st) : run_verify<float>(a, st);
}

}  // namespace dspark
