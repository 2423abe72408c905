// Per-request finish of one draft position: from the per-tile partial sums,
// choose the tile whose running sum crosses u*S, recompute that tile and
// choose the token inside it.  Shared by the standalone finish kernel (a
// 256-thread block) and the persistent draft kernel (its 256 epilogue
// threads, synchronised by a named barrier).
//
// "DSpark.让每一轮计算，多走几步" (explainer), Markov head panel: the
// left-to-right draw of each draft position from softmax((z + bias) / T).
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace dspark {

// The threads that run one finish and how they synchronise: kWarps warps,
// tid() the thread's index among them.  BlockSync: a 256-thread block;
// NamedSync: threads 0 .. kThreads-1 of a larger block, on barrier kId;
// GroupSync: the block's warps in groups of NW, group g on barrier kBase + g
// (several finishes at once, one per group).
struct BlockSync {
  static constexpr int kWarps = 8;
  __device__ __forceinline__ static void sync() { __syncthreads(); }
  __device__ __forceinline__ static int tid() { return threadIdx.x; }
};

template <int kId, int kThreads>
struct NamedSync {
  static constexpr int kWarps = kThreads / 32;
  __device__ __forceinline__ static void sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kThreads) : "memory");
  }
  __device__ __forceinline__ static int tid() { return threadIdx.x; }
};

template <int kBase, int NW>
struct GroupSync {
  static constexpr int kWarps = NW;
  __device__ __forceinline__ static void sync() {
    const int id = kBase + (int)(threadIdx.x >> 5) / NW;
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(NW * 32) : "memory");
  }
  __device__ __forceinline__ static int tid() { return (int)threadIdx.x % (NW * 32); }
};

// Where the finish gets the chosen tile's bias: the CUDA-core bias array of
// the workspace (bias != nullptr), or recomputed on CUDA cores from E, Wt and
// the previous token prev[n * prev_stride] (the fused tensor-core pass stores
// no bias); with prev null, from row n * prev_stride of E (the RNN states).
struct BiasSrc {
  const float* bias;
  const __nv_bfloat16* E;
  const __nv_bfloat16* Wt;
  const int32_t* prev;
  int prev_stride, r;
};

// Shared-memory scratch of one finish (about 8 KiB).
struct FinishScratch {
  long long shl[8];
  long long shl2[8];
  float shf[8];
  int shi[8];
  ArgMax sha[8];
  long long base;
  long long ssel;
  int fallback;
  int tok;
  int grp;      // 16-token group of the chosen tile holding the draw
  float f2;     // position of the draw inside that group, as a fraction of its mass
  float bias[256];
  float erow[1024];
};

// ---- reductions over the S::kWarps warps of a finish, every thread gets the result

// Warp maximum of floats that are never NaN (-inf allowed), as one integer
// reduction instruction on an order-preserving image of the bits (a negative
// float's magnitude bits flipped), instead of five dependent shuffles.
__device__ __forceinline__ float warp_max_nonan(float a) {
  int k = __float_as_int(a);
  k = k >= 0 ? k : (k ^ 0x7fffffff);
  k = __reduce_max_sync(0xffffffffu, k);
  return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff));
}

// Inclusive scan over the finish's threads; *total receives the sum of all.
template <class S>
__device__ __forceinline__ long long g_scan_ll(long long v, long long* sh, long long* total) {
  const int lane = S::tid() & 31, wid = S::tid() >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  S::sync();
  if (lane == 31) sh[wid] = v;
  S::sync();
  long long off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < S::kWarps; ++w) {
    const long long x = sh[w];
    if (w < wid) off += x;
    tot += x;
  }
  *total = tot;
  return v + off;
}

// Two inclusive scans at once (the same latency as one); *ta, *tb the totals.
template <class S>
__device__ __forceinline__ void g_scan_ll2(long long& a, long long& b, long long* sha,
                                           long long* shb, long long* ta, long long* tb) {
  const int lane = S::tid() & 31, wid = S::tid() >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long na = __shfl_up_sync(0xffffffffu, a, o);
    const long long nb = __shfl_up_sync(0xffffffffu, b, o);
    if (lane >= o) {
      a += na;
      b += nb;
    }
  }
  S::sync();
  if (lane == 31) {
    sha[wid] = a;
    shb[wid] = b;
  }
  S::sync();
  long long oa = 0, ob = 0, sa = 0, sb = 0;
#pragma unroll
  for (int w = 0; w < S::kWarps; ++w) {
    const long long xa = sha[w], xb = shb[w];
    if (w < wid) {
      oa += xa;
      ob += xb;
    }
    sa += xa;
    sb += xb;
  }
  a += oa;
  b += ob;
  *ta = sa;
  *tb = sb;
}

template <class S>
__device__ __forceinline__ int g_min_i(int v, int* sh) {
  const int lane = S::tid() & 31, wid = S::tid() >> 5;
  v = __reduce_min_sync(0xffffffffu, v);  // one warp-wide reduction instruction
  S::sync();
  if (lane == 0) sh[wid] = v;
  S::sync();
  int r = sh[0];
#pragma unroll
  for (int w = 1; w < S::kWarps; ++w) r = min(r, sh[w]);
  return r;
}

template <class S>
__device__ __forceinline__ int g_max_i(int v, int* sh) {
  const int lane = S::tid() & 31, wid = S::tid() >> 5;
  v = __reduce_max_sync(0xffffffffu, v);
  S::sync();
  if (lane == 0) sh[wid] = v;
  S::sync();
  int r = sh[0];
#pragma unroll
  for (int w = 1; w < S::kWarps; ++w) r = max(r, sh[w]);
  return r;
}

// (v never NaN)
template <class S>
__device__ __forceinline__ float g_max_f(float v, float* sh) {
  const int lane = S::tid() & 31, wid = S::tid() >> 5;
  v = warp_max_nonan(v);
  S::sync();
  if (lane == 0) sh[wid] = v;
  S::sync();
  float r = sh[0];
#pragma unroll
  for (int w = 1; w < S::kWarps; ++w) r = fmaxf(r, sh[w]);
  return r;
}

template <class S>
__device__ __forceinline__ ArgMax g_argmax(ArgMax a, ArgMax* sh) {
  const int lane = S::tid() & 31, wid = S::tid() >> 5;
  a = warp_argmax(a);
  S::sync();
  if (lane == 0) sh[wid] = a;
  S::sync();
  ArgMax r = sh[0];
#pragma unroll
  for (int w = 1; w < S::kWarps; ++w) r = better(r, sh[w]);
  return r;
}

// Weight of one token relative to the tile reference: 2^(a - ref) <= 1, in
// fixed-point units of 2^-40, and the fp32 weight.
__device__ __forceinline__ long long rel_fix(float a, float ref, float* w_out) {
  const float w = exp2f(a - ref);
  *w_out = w;
  return __float2ll_rn(w * 1099511627776.0f);  // 2^40
}

// bias[c] = E[prev] . Wt[v0 + c] for the TW columns of one tile (erow holds
// the previous token's E row in fp32): warp w takes columns w*TW/8 .. +TW/8,
// lanes split the rank dimension with 16-byte loads of the Wt row (r a
// multiple of 8, r <= 256); all of a warp's row loads are issued before the
// reductions so their latencies overlap.
template <int TW, class S>
__device__ __forceinline__ void tile_bias_recompute(const BiasSrc& b, int V, int v0,
                                                    const float* erow, float* bias) {
  constexpr int CPW = TW / S::kWarps;
  const int warp = S::tid() >> 5, lane = S::tid() & 31;
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
    if (lane == 0) bias[warp * CPW + c] = acc;
  }
  S::sync();
}

// With a stage buffer: copy the drawn token's E row (s.tok, set by the
// drawing thread before the last sync) to stage[n], where the next position's
// A operand is loaded from by TMA; the proxy fence orders these generic
// stores before that async-proxy read (r a multiple of 8, rows 16-byte aligned).
template <class S>
__device__ __forceinline__ void stage_row(FinishScratch& s, __nv_bfloat16* stage,
                                          const BiasSrc& b, int n) {
  if (stage == nullptr) return;
  const int tok = s.tok;
  const int tid = S::tid();
  if (tid < b.r / 8) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tok >= 0) v = *reinterpret_cast<const uint4*>(b.E + (size_t)tok * b.r + tid * 8);
    *reinterpret_cast<uint4*>(stage + (size_t)n * b.r + tid * 8) = v;
  }
  sm100::fence_proxy_async_all();
  S::sync();
}

// The draw inside tile tsel from its 16-token group sums: the group (placed
// by the caller, or the last group with mass after a fallback) is recomputed
// exactly (warp w takes the group's tokens 2w and 2w + 1; lanes split the
// rank with 16-byte loads) together with those tokens' E rows, so the drawn
// token's row is staged from registers.  F, g: the fixed-point total of the
// request's partials (sum_v 2^a_v = F * 2^g).
template <typename T, class S, bool kDeferLog>
__device__ __forceinline__ void finish_group(FinishScratch& s, int n, int V, int tsel, bool fallback,
                                          size_t out, long long F, int g, const T* __restrict__ z,
                                          const BiasSrc& bsrc, ScalePair sc, const float* sub,
                                          int n_tiles, int32_t* tokens, double* q_lse,
                                          float* q_tok, __nv_bfloat16* stage);

// Where the draw falls inside a tile, from the tile's eight 16-token group
// sums gs (any common unit) and the fraction f in [0, 1) of the tile's mass
// below the draw: the first group whose running sum exceeds f * total, and
// the fraction of that group's mass below the draw (fp32 throughout: a
// group boundary moves by rounding only for draws within ~1e-7 of it).  No
// group crossed: the last group with mass and *f_in = 2 (its last token).
__device__ __forceinline__ int pick_group(const float (&gs)[8], float f, float* f_in) {
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += gs[i];
  const float tgt = f * tot;
  float cum = 0.f, before = 0.f, gsel = 1.f;
  int j = -1, lastg = -1;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float g = gs[i];
    if (g > 0.f) {
      if (j < 0 && cum + g > tgt) {
        j = i;
        before = cum;
        gsel = g;
      }
      lastg = i;
    }
    cum += g;
  }
  if (j < 0) {
    *f_in = 2.0f;
    return lastg;
  }
  *f_in = fminf(fmaxf((tgt - before) / gsel, 0.f), 1.f);
  return j;
}

// num / den for 0 <= num < den < 2^63, to fp32 precision, from the top 24
// bits of both (integer shifts: no 64-bit conversions).
__device__ __forceinline__ float ratio_ll(long long num, long long den) {
  const int sh = max(0, 40 - __clzll(den));  // den >> sh < 2^24
  return (float)(unsigned)(num >> sh) / (float)(unsigned)(den >> sh);
}

__device__ __forceinline__ void load_groups(const float* sub, float (&gs)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(sub));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(sub) + 1);
  gs[0] = a.x; gs[1] = a.y; gs[2] = a.z; gs[3] = a.w;
  gs[4] = b.x; gs[5] = b.y; gs[6] = b.z; gs[7] = b.w;
}

// The finish of request n at draft position k, by the S::kWarps warps of
// one finish group (S::tid() their thread index).  part: [R][n_tiles] tile partials (doubles; greedy:
// ArgMax pairs) of width TW.  Writes tokens / q_lse / q_tok [n][k].
// With sub ([R][n_tiles][8] group sums of 128-token partials) the draw is
// placed in a 16-token group first and only that group is recomputed;
// without, the whole tile is.  Partials and previous tokens may have been
// written by other blocks of the same kernel, so they are read past L1
// (ld.global.cg).
template <typename T, int TW, class S, bool kDeferLog>
__device__ void finish_request(FinishScratch& s, int n, int V, int gamma, int k, int n_tiles,
                               const T* __restrict__ z, const BiasSrc& bsrc, ScalePair sc,
                               int greedy, const double* part, const float* __restrict__ u,
                               int32_t* tokens, double* q_lse, float* q_tok, uint32_t* status,
                               __nv_bfloat16* stage = nullptr, const float* sub = nullptr) {
  constexpr int NT = S::kWarps * 32;
  const int tid = S::tid();
  const size_t out = (size_t)n * gamma + k;
  const float u_out = greedy ? 0.0f : u[out];  // issued early: needed after the scan
  if (greedy) {
    const ArgMax* P = reinterpret_cast<const ArgMax*>(part) + (size_t)n * n_tiles;
    ArgMax best{-INFINITY, 0x7fffffff};
    for (int t = tid; t < n_tiles; t += NT) {
      const long long raw = __ldcg(reinterpret_cast<const long long*>(P + t));
      ArgMax am;
      am.v = __int_as_float((int)(raw & 0xffffffffll));
      am.i = (int)(raw >> 32);
      best = better(best, am);
    }
    best = g_argmax<S>(best, s.sha);
    if (tid == 0) {
      int tok = best.i;
      if (tok < 0 || tok >= V) {
        set_flag(status, kFlagNonFinite);
        tok = 0;
      }
      tokens[out] = tok;
      q_lse[out] = (double)best.v;
      q_tok[out] = 1.0f;
      s.tok = tok;
    }
    S::sync();
    stage_row<S>(s, stage, bsrc, n);
    return;
  }
  if (bsrc.bias == nullptr) {
    // the previous token's E row, needed once the tile is chosen: load it now
    int tok = n * bsrc.prev_stride;  // no token list: row n * stride (the RNN states)
    if (bsrc.prev != nullptr) {
      tok = __ldcg(bsrc.prev + (size_t)n * bsrc.prev_stride);
      if (tok >= V || tok < -1) {
        if (tid == 0) set_flag(status, kFlagTokenRange);
        tok = -1;
      }
    }
    for (int i = tid; i < bsrc.r; i += NT)
      s.erow[i] = tok >= 0 ? __bfloat162float(bsrc.E[(size_t)tok * bsrc.r + i]) : 0.f;
  }
  // The partials are exact doubles; they are summed exactly as integers in
  // units of 2^g, g chosen from the largest partial's exponent so that the
  // sum of all n_tiles partials stays below 2^62.  Thread tid owns the
  // contiguous tiles [t0, t0 + seg); up to kMaxSeg of them (2048 tiles in
  // all: V <= 2^18 on the tensor-core path) are loaded once into registers,
  // longer segments are re-read from L2 in each pass.
  constexpr int kMaxSeg = 8;
  const double* S_ = part + (size_t)n * n_tiles;
  const int seg = (n_tiles + NT - 1) / NT;
  const bool fast = seg <= kMaxSeg;
  const int t0 = min(n_tiles, tid * seg), t1 = min(n_tiles, t0 + seg);
  double pv[kMaxSeg];
  int emax = INT_MIN;
  if (fast) {
#pragma unroll
    for (int i = 0; i < kMaxSeg; ++i) pv[i] = t0 + i < t1 ? __ldcg(S_ + t0 + i) : 0.0;
#pragma unroll
    for (int i = 0; i < kMaxSeg; ++i) emax = max(emax, double_exponent(pv[i]));
  } else {
    for (int t = t0; t < t1; ++t) emax = max(emax, double_exponent(__ldcg(S_ + t)));
  }
  emax = g_max_i<S>(emax, s.shi);
  if (emax == INT_MIN) {  // no token has mass
    if (tid == 0) {
      set_flag(status, kFlagNonFinite);
      tokens[out] = 0;
      q_lse[out] = kDeferLog ? 0.0 : -INFINITY;
      q_tok[out] = 0.0f;
    }
    S::sync();
    return;
  }
  const int g = emax + 2 + (32 - __clz(n_tiles)) - 62;
  long long fx[kMaxSeg], loc = 0;
  if (fast) {
#pragma unroll
    for (int i = 0; i < kMaxSeg; ++i) {
      fx[i] = double_to_fix(pv[i], g);
      loc += fx[i];
    }
  } else {
    for (int t = t0; t < t1; ++t) loc += double_to_fix(__ldcg(S_ + t), g);
  }
  long long F;
  const long long incl = g_scan_ll<S>(loc, s.shl, &F);
  // the draw is the first token whose running sum exceeds u*F; for integer
  // running sums that is "exceeds floor(u*F)"
  const long long thr = floor_mul(u_out, F);
  int cand = 0x7fffffff, last = -1;
  long long base = 0, ssel = 0;
  {
    long long run = incl - loc;
    if (fast) {
#pragma unroll
      for (int i = 0; i < kMaxSeg; ++i) {
        const long long nx = run + fx[i];
        if (cand == 0x7fffffff && t0 + i < t1 && nx > thr) {
          cand = t0 + i;
          base = run;
          ssel = fx[i];
        }
        if (fx[i] > 0) last = t0 + i;
        run = nx;
      }
    } else {
      for (int t = t0; t < t1; ++t) {
        const long long f = double_to_fix(__ldcg(S_ + t), g);
        const long long nx = run + f;
        if (cand == 0x7fffffff && nx > thr) {
          cand = t;
          base = run;
          ssel = f;
        }
        if (f > 0) last = t;
        run = nx;
      }
    }
  }
  // With group sums, the thread whose segment holds the crossing places it
  // in a group now, so that load overlaps the reduction that picks the tile.
  int grp = -1;
  float f2 = 2.0f;
  if (TW == 128 && sub != nullptr && cand != 0x7fffffff) {
    float gs[8];
    load_groups(sub + ((size_t)n * n_tiles + cand) * 8, gs);
    grp = pick_group(gs, ratio_ll(thr - base, ssel), &f2);
  }
  int tsel = g_min_i<S>(cand, s.shi);
  if (tsel == 0x7fffffff) {
    // u outside [0, 1): the last tile with mass
    tsel = g_max_i<S>(last, s.shi);
    if (tsel < 0) tsel = 0;
    if (tid == 0) {
      s.fallback = 1;
      s.grp = -1;
    }
  } else if (cand == tsel) {
    s.base = base;
    s.ssel = ssel;
    s.fallback = 0;
    s.grp = grp;
    s.f2 = f2;
  }
  S::sync();
  const bool fallback = s.fallback != 0;
  if (TW == 128 && sub != nullptr) {
    finish_group<T, S, kDeferLog>(s, n, V, tsel, fallback, out, F, g, z, bsrc, sc, sub, n_tiles,
                                  tokens, q_lse, q_tok, stage);
    return;
  }
  base = s.base;
  const long long S_sel = s.ssel;
  // Recompute the chosen tile.
  const int v = tsel * TW + tid;
  const bool ok = tid < TW && v < V;
  const float zv = ok ? ldf(z, out * V + v) : 0.f;  // issued before the bias loads
  float bv = 0.f;
  if (bsrc.bias != nullptr) {
    if (ok) bv = bsrc.bias[(size_t)n * V + v];
  } else {
    tile_bias_recompute<TW, S>(bsrc, V, tsel * TW, s.erow, s.bias);
    bv = tid < TW ? s.bias[tid] : 0.f;
  }
  float y = -INFINITY;
  if (ok) y = zv + bv;
  if (ok && (isnan(y) || y == INFINITY)) y = -INFINITY;
  const float a = scaled(y, sc);
  const float amax = g_max_f<S>(a, s.shf);
  const float ref = ceilf(amax);
  float w = 0.f;
  const long long f = (ok && a > -INFINITY && amax > -INFINITY) ? rel_fix(a, ref, &w) : 0ll;
  long long mass;
  const long long cum = g_scan_ll<S>(f, s.shl, &mass);
  // The recomputed tile can differ from its partial in the last bits, so the
  // crossing is placed at the same fraction of the recomputed tile:
  //   cum / mass > (thr - base) / S_sel  <=>  cum * S_sel > (thr - base) * mass
  // compared exactly in 128-bit products.
  const unsigned long long need = (unsigned long long)(thr - base);
  int pick = 0x7fffffff;
  if (!fallback && f > 0 &&
      mul_gt((unsigned long long)cum, (unsigned long long)S_sel, need, (unsigned long long)mass))
    pick = tid;
  int isel = g_min_i<S>(pick, s.shi);
  if (isel == 0x7fffffff) isel = g_max_i<S>(f > 0 ? tid : -1, s.shi);
  if (isel < 0) isel = 0;
  if (tid == isel) {
    tokens[out] = tsel * TW + isel;
    const double total = fix_to_double(F, g);  // sum_v 2^a_v
    q_lse[out] = kDeferLog ? total : (double)fix_log(F, g);
    // q(x) = 2^a / total = w * 2^ref / (F * 2^g)
    const int fm = 63 - __clzll(F);
    q_tok[out] = scale_pow2(w / fix_to_float(F, -fm), (int)ref - g - fm);
    s.tok = tsel * TW + isel;
  }
  S::sync();
  stage_row<S>(s, stage, bsrc, n);
}

template <typename T, class S, bool kDeferLog>
__device__ __forceinline__ void finish_group(FinishScratch& s, int n, int V, int tsel, bool fallback,
                                          size_t out, long long F, int g, const T* __restrict__ z,
                                          const BiasSrc& bsrc, ScalePair sc, const float* sub,
                                          int n_tiles, int32_t* tokens, double* q_lse,
                                          float* q_tok, __nv_bfloat16* stage) {
  constexpr int TPW = 16 / S::kWarps;  // the group's tokens per warp
  const int tid = S::tid(), lane = tid & 31, w = tid >> 5;
  const int grp0 = s.grp;
  if (fallback || grp0 < 0) {
    // the last group with mass, its last token with mass
    S::sync();  // every thread has read s.grp before it is rewritten
    if (tid == 0) {
      float gs[8];
      load_groups(sub + ((size_t)n * n_tiles + tsel) * 8, gs);
      int lastg = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (gs[i] > 0.f) lastg = i;
      s.grp = lastg;
      s.f2 = 2.0f;
    }
    S::sync();
  }
  const int gv0 = tsel * 128 + s.grp * 16;
  const float f2 = s.f2;
  // bias of tokens gv0 + TPW w + c; with up to two tokens a warp their E
  // rows ride along (the drawn token's is staged from registers), with more
  // the drawn token's row is read once it is known (fewer live registers)
  constexpr bool kRide = TPW <= 2;
  const int j = lane * 8;
  const bool lane_on = j < bsrc.r;
  uint4 wr[TPW], er[kRide ? TPW : 1];
#pragma unroll
  for (int c = 0; c < TPW; ++c) {
    const int v = gv0 + TPW * w + c;
    const bool ok = lane_on && v < V;
    wr[c] = ok ? *reinterpret_cast<const uint4*>(bsrc.Wt + (size_t)v * bsrc.r + j)
               : make_uint4(0, 0, 0, 0);
    if constexpr (kRide)
      er[c] = (ok && stage != nullptr)
                  ? *reinterpret_cast<const uint4*>(bsrc.E + (size_t)v * bsrc.r + j)
                  : make_uint4(0, 0, 0, 0);
  }
  const int vz = gv0 + lane;
  const float zv = (w == 0 && lane < 16 && vz < V) ? ldf(z, out * V + vz) : 0.f;
  float e8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e8[i] = lane_on ? s.erow[j + i] : 0.f;
#pragma unroll
  for (int c = 0; c < TPW; ++c) {
    const uint32_t w4[4] = {wr[c].x, wr[c].y, wr[c].z, wr[c].w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(w4[e] << 16), e8[2 * e], acc);
      acc = fmaf(__uint_as_float(w4[e] & 0xffff0000u), e8[2 * e + 1], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) s.bias[TPW * w + c] = acc;
  }
  S::sync();
  if (w == 0) {
    // lanes 0-15: the group's tokens.  Weights 2^(a - ref) <= 1 in 32-bit
    // fixed point (2^-27 units: 16 of them stay below 2^31) and their scan,
    // all in 32-bit integer arithmetic.
    const bool ok = lane < 16 && vz < V;
    float y = ok ? zv + s.bias[lane] : -INFINITY;
    if (ok && (isnan(y) || y == INFINITY)) y = -INFINITY;
    const float a = scaled(y, sc);
    const float amax = warp_max_nonan(a);  // y was cleaned: no NaN
    const float ref = ceilf(amax);
    const float wt = (ok && a > -INFINITY && amax > -INFINITY) ? exp2f(a - ref) : 0.f;
    const uint32_t f = __float2uint_rn(wt * 134217728.0f);  // 2^27
    uint32_t cum = f;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, cum, o);
      if (lane >= o) cum += x;
    }
    const uint32_t mass = __shfl_sync(0xffffffffu, cum, 15);
    // the draw is the first token whose running sum exceeds f2 * mass
    const uint32_t thr_g =
        f2 < 1.5f ? __umulhi(__float2uint_rz(f2 * 4294967040.0f), mass) : 0xffffffffu;
    const unsigned hit = __ballot_sync(0xffffffffu, lane < 16 && f > 0 && cum > thr_g);
    const unsigned has = __ballot_sync(0xffffffffu, lane < 16 && f > 0);
    const int isel = hit ? __ffs(hit) - 1 : (has ? 31 - __clz(has) : 0);
    if (lane == isel) {
      const int tok = gv0 + isel;
      tokens[out] = tok;
      const double total = fix_to_double(F, g);  // sum_v 2^a_v
      q_lse[out] = kDeferLog ? total : (double)fix_log(F, g);
      // q(x) = 2^a / total = wt * 2^ref / (F * 2^g)
      const int fm = 63 - __clzll(F);
      q_tok[out] = scale_pow2(wt / fix_to_float(F, -fm), (int)ref - g - fm);
      s.tok = isel;
    }
  }
  S::sync();
  if (stage != nullptr) {
    const int isel = s.tok;
    if constexpr (kRide) {
      if (w == isel / TPW && lane_on) {
        uint4 row = er[0];
#pragma unroll
        for (int c = 1; c < TPW; ++c)
          if (isel % TPW == c) row = er[c];
        *reinterpret_cast<uint4*>(stage + (size_t)n * bsrc.r + j) = row;
      }
    } else if (w == 0 && lane_on && gv0 + isel < V) {
      *reinterpret_cast<uint4*>(stage + (size_t)n * bsrc.r + j) =
          *reinterpret_cast<const uint4*>(bsrc.E + (size_t)(gv0 + isel) * bsrc.r + j);
    }
    sm100::fence_proxy_async_all();
    S::sync();
  }
}

}  // namespace dspark
