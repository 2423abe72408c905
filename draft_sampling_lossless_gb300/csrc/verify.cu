// Lossless rejection-sampling and greedy verification.
//
// Forum post "为什么DSpark 可以加速推理？以及DSpark会不会导致降智？", lossless
// proof: accept the drafted token with probability min(1, p/q); on rejection
// draw from max(0, p - q) normalised; the emitted marginal is p.  Explainer
// "DSpark.让每一轮计算，多走几步", lossless panel: if the whole block passes,
// one more (bonus) token comes from the next target distribution.  CSDN
// tutorial, section 五: the first rejection ends the block.
//
// Launches on the bf16 tensor-core path (the common case):
//   rows   -- verify_rows_tma_kernel: every verified target row streamed once
//             (4096-token items, 2 KiB bulk copies through a per-warp ring),
//             each item's exact fixed-point sum of 2^(t*log2e/T - ref) (greedy:
//             its argmax); the block that completes a request's last item then
//             runs that request's decide: row normalisers, p_lse, the accept
//             tests u < p(x)/q(x) in order, n_acc, the accepted tokens and the
//             final draw's state
//   final  -- final_tc_kernel (draft_tc.cu): the rejected position's bias on
//             the tensor cores and, per 128-token half tile, the exact sums of
//             p and of max(0, p - q), both normalised
//   pick   -- per request: inverse CDF over the half tiles, then inside the
//             chosen one by recomputing it with the same arithmetic, compared
//             with u*total in exact integer arithmetic
// Other shapes (fp32, R > 1024, unaligned rows) use plain-load rows, a
// separate decide kernel and the CUDA-core bias / final / pick kernels.
// Greedy verification needs only the rows and the decide.
#include "common.cuh"
#include "f32x2.cuh"
#include "finish.cuh"

namespace dspark {

namespace {

constexpr int kRowChunk = kChunkV;          // tokens per row-pass item
constexpr int kRowSub = 1024;               // tokens per sub-chunk (one bulk copy)
constexpr int kRowGroup = kRowChunk / kRowSub;  // sub-chunks per item
constexpr int kFinTile = 256;    // tokens per warp item of the final pass

// ---------------------------------------------------------------- rows

// load8 with an L2 evict-first cache policy: the row pass streams every
// verified target row once, and should not push the draft's W (kept with an
// evict-last policy for the final draw) out of L2.
template <typename T>
__device__ __forceinline__ void load8_stream(const T* p, int v0, int V, float (&o)[8], float fill,
                                             uint64_t pol);
template <>
__device__ __forceinline__ void load8_stream<__nv_bfloat16>(const __nv_bfloat16* p, int v0, int V,
                                                            float (&o)[8], float fill,
                                                            uint64_t pol) {
  if (v0 + 8 <= V) {
    uint32_t w[4];
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "l"(p + v0), "l"(pol));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    load8<__nv_bfloat16>(p, v0, V, o, fill);
  }
}
template <>
__device__ __forceinline__ void load8_stream<float>(const float* p, int v0, int V, float (&o)[8],
                                                    float fill, uint64_t pol) {
  if (v0 + 8 <= V) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                   : "=f"(o[4 * h]), "=f"(o[4 * h + 1]), "=f"(o[4 * h + 2]), "=f"(o[4 * h + 3])
                   : "l"(p + v0 + 4 * h), "l"(pol));
  } else {
    load8<float>(p, v0, V, o, fill);
  }
}

// 1024 tokens of one row as raw 16-byte vectors: lane l holds tokens
// i*256 + l*8 .. +7 of group i (bf16: one uint4 per group; fp32: two).
template <typename T>
struct RowRaw;
template <>
struct RowRaw<__nv_bfloat16> {
  uint4 q[4];
  __device__ __forceinline__ void load(const __nv_bfloat16* p, int lim, uint64_t pol) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v0 = i * 256 + lane * 8;
      if (v0 + 8 <= lim) {
        asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=r"(q[i].x), "=r"(q[i].y), "=r"(q[i].z), "=r"(q[i].w)
                     : "l"(p + v0), "l"(pol));
      } else {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t lo = v0 + 2 * k < lim ? (uint32_t)__bfloat16_as_ushort(p[v0 + 2 * k]) : 0xff80u;
          const uint32_t hi = v0 + 2 * k + 1 < lim ? (uint32_t)__bfloat16_as_ushort(p[v0 + 2 * k + 1]) : 0xff80u;
          w[k] = lo | (hi << 16);  // 0xff80 = -inf
        }
        q[i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  __device__ __forceinline__ void get(int i, float (&o)[8]) const {
    const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      o[2 * k] = __uint_as_float(w[k] << 16);
      o[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  // the largest of the 32 values (NaN ignored), on bf16 pairs
  __device__ __forceinline__ float max() const {
    __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162*>(&q[0].x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    }
    return fmaxf(__low2float(m), __high2float(m));
  }
};
template <>
struct RowRaw<float> {
  float x[4][8];
  __device__ __forceinline__ void load(const float* p, int lim, uint64_t pol) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) load8_stream<float>(p, i * 256 + lane * 8, lim, x[i], -INFINITY, pol);
  }
  __device__ __forceinline__ void get(int i, float (&o)[8]) const {
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = x[i][e];
  }
  __device__ __forceinline__ float max() const {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, x[i][e]);
    return m;
  }
};

// Running state of one warp item (kRowChunk tokens of a verified row, taken
// as kRowGroup sub-chunks of kRowSub tokens): per lane the fixed-point sum of
// 2^(a - ref) in 2^-40 units against the lane's own power-of-two reference
// that only grows (the sum is shifted down when it does), or the greedy
// argmax.  a = y * c with c = log2(e)/T rounded to fp32: the largest a is
// the scaled largest y (c > 0), each exponent argument is one FMA (-inf
// weighs 0).  Per sub-chunk a lane adds its 32 weights as an fp32 tree and
// converts the tree once; no warp-wide step until the item's partial, where
// the lanes' sums are brought to the largest reference (shifted down, so
// each lane loses less than one 2^-40 unit of it) and added exactly.  A NaN
// surfaces in a tree, +inf in a maximum: both flag the row non-finite and
// weigh 0.
struct RowState {
  long long acc = 0;
  int ref = INT_MIN;
  bool bad = false;
  ArgMax am{-INFINITY, 0x7fffffff};

  template <typename T>
  __device__ __forceinline__ void add(const RowRaw<T>& raw, int v0, int V, ScalePair sc,
                                      int greedy) {
    const int lane = threadIdx.x & 31;
    if (greedy) {
      // the 32 values' maximum (NaN ignored), its first index in token order,
      // then one comparison with the item's best.  Values past V were loaded
      // as -inf, so they never come before a token of the row.
      const float m = raw.max();
      int idx = 31;
#pragma unroll
      for (int i = 3; i >= 0; --i) {
        float x[8];
        raw.get(i, x);
#pragma unroll
        for (int e = 7; e >= 0; --e) idx = x[e] == m ? i * 8 + e : idx;
      }
      am = better(am, ArgMax{m, v0 + (idx >> 3) * 256 + lane * 8 + (idx & 7)});
      return;
    }
    const float m = raw.max() * sc.hi;
    if (!(m < 3.0e38f)) {  // +inf or NaN
      bad = true;
      return;
    }
    if (m <= -1.0e38f) return;  // no mass in this lane's values
    const int cref = (int)ceilf(m);
    if (ref == INT_MIN) {
      ref = cref;
    } else if (cref > ref) {
      const int d = cref - ref;
      acc = d >= 63 ? 0 : (acc >> d);
      ref = cref;
    }
    const float fref = (float)ref;
    // pairs of tokens through the packed fp32 FMA and adds: the same
    // roundings, in the same tree, as one token at a time
    const unsigned long long c2 = pack2(sc.hi, sc.hi), r2 = pack2(-fref, -fref);
    float t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x[8];
      raw.get(i, x);
      unsigned long long p2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a, b;
        unpack2(fma2(pack2(x[2 * e], x[2 * e + 1]), c2, r2), a, b);
        p2[e] = pack2(ex2_fast(a), ex2_fast(b));
      }
      p2[0] = add2(p2[0], p2[2]);  // tokens e and e + 4
      p2[1] = add2(p2[1], p2[3]);
      p2[0] = add2(p2[0], p2[1]);  // e and e + 2
      float a, b;
      unpack2(p2[0], a, b);
      t[i] = a + b;
    }
    const float sum = (t[0] + t[1]) + (t[2] + t[3]);
    if (sum != sum) bad = true;
    else acc += __float2ll_rn(sum * 1099511627776.0f);  // 2^40
  }

  // the item's partial (sampling: a double of the exact fixed-point total)
  __device__ __forceinline__ void store(int greedy, double* out, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    if (greedy) {
      const ArgMax r = warp_argmax(am);
      if (lane == 0) *reinterpret_cast<ArgMax*>(out) = r;
      return;
    }
    const int rmax = __reduce_max_sync(0xffffffffu, ref);
    const int d = ref == INT_MIN ? 64 : rmax - ref;
    const long long f = warp_sum_nonneg_ll(d >= 63 ? 0ll : (acc >> d));
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_flag(status, kFlagNonFinite);
    if (lane == 0) *out = (rmax == INT_MIN || f <= 0) ? 0.0 : fix_to_double(f, rmax - kFixRel);
  }
};

// The verified-row list of the row pass, built by every block in shared
// memory: s_r0 = row_off, s_pre = exclusive prefix of the rows per request
// (1 + ell[n], 0 for an invalid ell -- the decide kernel reports it).
__device__ __forceinline__ int build_row_list(int R, int gamma, const int32_t* __restrict__ ell,
                                              const int32_t* __restrict__ row_off, int* s_r0,
                                              int* s_pre, int* s_scan) {
  int cnt[4], loc = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int n = threadIdx.x * 4 + q;
    cnt[q] = 0;
    if (n < R) {
      const int L = ell[n];
      s_r0[n] = row_off[n];
      cnt[q] = (L >= 0 && L <= gamma) ? L + 1 : 0;
    }
    loc += cnt[q];
  }
  const int incl = block_inclusive_scan(loc, s_scan);
  int run = incl - loc;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int n = threadIdx.x * 4 + q;
    if (n < R) s_pre[n] = run;
    run += cnt[q];
  }
  if (threadIdx.x == blockDim.x - 1) s_pre[R] = incl;
  __syncthreads();
  return s_pre[R];
}

constexpr int kRowsSmem = 1024;  // requests whose row list fits shared memory

template <typename T>
__device__ __noinline__ void decide_request(
    int n, int gamma, int V, int n_chunks, long long n_rows, const T* __restrict__ target,
    ScalePair sc, int greedy, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const double* __restrict__ q_lse,
    const float* __restrict__ q_tok, const int32_t* __restrict__ ell,
    const int32_t* __restrict__ row_off, const float* __restrict__ u_acc,
    const double* __restrict__ row_part, double* __restrict__ p_lse,
    int32_t* __restrict__ n_acc_out, int32_t* __restrict__ out_tokens,
    VerifyState* __restrict__ vstate, int32_t* __restrict__ prev_out, uint32_t* status);

// What the row pass needs to run each request's decide itself: the block that
// completes a request's last item runs it (per-request item counters in the
// workspace, returned to zero by that block).
struct DecideOut {
  int on;
  const int32_t* anchor;
  const int32_t* tokens;
  const double* q_lse;
  const float* q_tok;
  const float* u_acc;
  double* p_lse;
  int32_t* n_acc;
  int32_t* out_tokens;
  VerifyState* vstate;
  int32_t* prev;
  int* cnt;  // [R] items counted so far, zero between calls
};

// The row pass for bf16 targets with V % 8 == 0 (16-byte aligned rows).
// Item = (verified row, chunk of kRowChunk tokens), strided over the grid's
// warps.  Each warp streams its items' sub-chunks (2 KiB each) in order
// through a ring of kRowStages shared-memory slots with bulk copies (L2
// evict-first): lane 0 keeps the copies kRowStages units ahead of the
// reduction, so every warp has its next item's data in flight while it
// reduces the current one, at few registers.  Three slots a warp and the
// request list sized by R (after the rings) let four blocks share an SM, so
// the grid's warps outnumber the items of a typical verify batch and each
// warp streams about one item.  Every wait is bounded; a timeout sets the
// timeout flag.
constexpr int kRowStages = 3;
constexpr uint32_t kRowSlot = kRowSub * 2;  // bytes of one bf16 sub-chunk
constexpr size_t kRowsTmaSmem = 8 * kRowStages * kRowSlot;  // the rings; the lists follow
__host__ __device__ constexpr size_t rows_tma_smem(int R) {
  return kRowsTmaSmem + (size_t)(4 * R + 1) * sizeof(int);  // rings; r0, pre, items, winners
}

//
// kGreedy (T = 0: arg-max items) is a template parameter, so that each
// instantiation's sub-chunk loop holds one kind of reduction.
template <bool kGreedy>
__global__ void __launch_bounds__(256, 4) verify_rows_tma_kernel(
    int R, int gamma, int V, int n_chunks, long long n_rows,
    const __nv_bfloat16* __restrict__ target, const int32_t* __restrict__ ell,
    const int32_t* __restrict__ row_off, ScalePair sc, double* __restrict__ row_part,
    uint32_t* status, const DecideOut dec) {
  constexpr int greedy = kGreedy ? 1 : 0;
  extern __shared__ __align__(16) uint8_t rows_ring[];
  int* s_r0 = reinterpret_cast<int*>(rows_ring + kRowsTmaSmem);  // [R]
  int* s_pre = s_r0 + R;                                          // [R + 1]
  int* s_cnt = s_pre + R + 1;                                     // [R] items done here
  int* s_win = s_cnt + R;                                         // [R] requests decided here
  __shared__ int s_req[8][kRowStages];
  __shared__ int s_nwin;
  __shared__ int s_scan[32];
  __shared__ uint64_t bars[8][kRowStages];
  __shared__ double* s_out[8][kRowStages];  // the unit's item output (null: row out of range)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t pol = sm100::policy_evict_first();
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8 * kRowStages; ++i) sm100::mbar_init(sm100::smem_u32(&bars[0][0] + i), 1);
    sm100::fence_mbar_init();
  }
  for (int i = threadIdx.x; i < R; i += blockDim.x) s_cnt[i] = 0;
  grid_dependency_wait();  // ell, row_off
  const int n_verified = build_row_list(R, gamma, ell, row_off, s_r0, s_pre, s_scan);
  const int n_subs = (V + kRowSub - 1) / kRowSub;
  const uint32_t total = (uint32_t)n_verified * (uint32_t)n_chunks;
  const uint32_t nwarps = gridDim.x * 8, w0 = blockIdx.x * 8 + warp;
  uint8_t* ring = rows_ring + (size_t)warp * kRowStages * kRowSlot;
  auto subs_of = [&](uint32_t item) -> int {
    const int c = (int)(item % (uint32_t)n_chunks);
    return min(kRowGroup, n_subs - c * kRowGroup);
  };
  // producer cursor (lane 0): the next unit to copy
  uint32_t p_item = w0;
  int p_sub = 0, p_nsub = 0;
  const __nv_bfloat16* p_src = nullptr;  // sub-chunk 0 of p_item's chunk, null: nothing to copy
  double* p_out = nullptr;
  int p_req = 0, p_c = 0;
  auto p_decode = [&]() {
    p_sub = 0;
    if (p_item >= total) return;
    const int k = (int)(p_item / (uint32_t)n_chunks);
    const int c = (int)(p_item - (uint32_t)k * (uint32_t)n_chunks);
    p_c = c;
    p_nsub = min(kRowGroup, n_subs - c * kRowGroup);
    int lo = 0, hi = R - 1;  // the request n with s_pre[n] <= k < s_pre[n + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= k) lo = mid;
      else hi = mid - 1;
    }
    const int n = lo, j = k - s_pre[n];
    p_req = n;
    const long long row = (long long)s_r0[n] + j;
    if (row < 0 || row >= n_rows) {  // reported by the decide kernel
      p_src = nullptr;
      p_out = nullptr;
    } else {
      p_src = target + (size_t)row * V + (size_t)c * kRowChunk;
      p_out = row_part + ((size_t)n * (gamma + 1) + j) * n_chunks + c;
    }
  };
  auto p_issue = [&](int slot) {  // copy the producer's unit into `slot`, advance
    if (p_item >= total) return;
    const uint32_t bar = sm100::smem_u32(&bars[warp][slot]);
    s_out[warp][slot] = p_out;
    s_req[warp][slot] = p_req;
    if (p_src == nullptr) {
      sm100::mbar_arrive(bar);
    } else {
      const int v0 = p_c * kRowChunk + p_sub * kRowSub;
      const uint32_t bytes = (uint32_t)min(kRowSub, V - v0) * 2u;
      sm100::mbar_arrive_expect_tx(bar, bytes);
      sm100::bulk_load_hint(sm100::smem_u32(ring + slot * kRowSlot), p_src + p_sub * kRowSub,
                            bytes, bar, pol);
    }
    if (++p_sub == p_nsub) {
      p_item += nwarps;
      p_decode();
    }
  };
  if (lane == 0) {
    p_decode();
    for (int sl = 0; sl < kRowStages; ++sl) p_issue(sl);
  }
  __syncwarp();
  uint32_t u = 0;  // units consumed by this warp
  for (uint32_t item = w0; item < total; item += nwarps) {
    const int c = (int)(item % (uint32_t)n_chunks), nsub = subs_of(item);
    RowState st;
    double* out = nullptr;
    int req = 0;
    bool failed = false;
    for (int sb = 0; sb < nsub; ++sb, ++u) {
      const int slot = (int)(u % kRowStages);
      const bool ok = sm100::mbar_wait(sm100::smem_u32(&bars[warp][slot]), (u / kRowStages) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
      out = s_out[warp][slot];
      req = s_req[warp][slot];
      if (out != nullptr) {
        const int v0 = c * kRowChunk + sb * kRowSub, lim = V - v0;
        RowRaw<__nv_bfloat16> x;
        const uint8_t* sl = ring + slot * kRowSlot;
        if (lim >= kRowSub) {  // every sub-chunk but the vocabulary's last
#pragma unroll
          for (int i = 0; i < 4; ++i)
            x.q[i] = *reinterpret_cast<const uint4*>(sl + (i * 256 + lane * 8) * 2);
        } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e0 = i * 256 + lane * 8;
          if (e0 + 8 <= lim) {
            x.q[i] = *reinterpret_cast<const uint4*>(sl + e0 * 2);
          } else {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint16_t* h = reinterpret_cast<const uint16_t*>(sl) + e0 + 2 * k;
              const uint32_t lo = e0 + 2 * k < lim ? h[0] : 0xff80u;  // -inf past V
              const uint32_t hi = e0 + 2 * k + 1 < lim ? h[1] : 0xff80u;
              w[k] = lo | (hi << 16);
            }
            x.q[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        }
        st.add(x, v0, V, sc, greedy);
      }
      __syncwarp();
      if (lane == 0) {
        sm100::fence_proxy_async_smem();  // this slot's generic reads before the refill
        p_issue(slot);
      }
      __syncwarp();
    }
    if (failed) {
      // give up: flag it, then wait (bounded) for this warp's copies in flight
      if (lane == 0) {
        set_flag(status, kFlagWaitTimeout);
        for (uint32_t r = u + 1; r < u + kRowStages; ++r)
          sm100::mbar_wait(sm100::smem_u32(&bars[warp][r % kRowStages]), (r / kRowStages) & 1);
      }
      break;
    }
    if (out != nullptr) st.store(greedy, out, status);
    if (dec.on && lane == 0) atomicAdd(s_cnt + req, 1);
  }
  if (!dec.on) return;
  // Each request's decide, by the block that completes its last item: the
  // block publishes its item counts (its partials ordered before them by the
  // block barrier and the fence); the one whose count completes a request
  // (1 + l rows of n_chunks items) runs the decide and zeroes the counter.
  // A request with no verified rows (an invalid l) is decided by block
  // n mod gridDim.x.
  __syncthreads();
  if (threadIdx.x == 0) s_nwin = 0;
  __syncthreads();
  for (int n = threadIdx.x; n < R; n += blockDim.x) {
    const int items = (s_pre[n + 1] - s_pre[n]) * n_chunks;
    const int c = s_cnt[n];
    bool win = false;
    if (items == 0) {
      win = n % (int)gridDim.x == (int)blockIdx.x;
    } else if (c > 0) {
      __threadfence();
      const int old = atomicAdd(dec.cnt + n, c);
      if (old + c == items) {
        win = true;
        dec.cnt[n] = 0;
      }
    }
    if (win) s_win[atomicAdd(&s_nwin, 1)] = n;
  }
  __syncthreads();
  const int nw = s_nwin;
  if (nw == 0) return;
  __threadfence();  // the other blocks' partials, published before their counts
  for (int i = 0; i < nw; ++i) {
    decide_request<__nv_bfloat16>(s_win[i], gamma, V, n_chunks, n_rows, target, sc, greedy,
                                  dec.anchor, dec.tokens, dec.q_lse, dec.q_tok, ell, row_off,
                                  dec.u_acc, row_part, dec.p_lse, dec.n_acc, dec.out_tokens,
                                  dec.vstate, dec.prev, status);
    __syncthreads();
  }
}

// The same pass for the other cases (R > kRowsSmem, fp32 targets, rows not
// 16-byte aligned): items (n, j, c) over every request and position, ell
// and row_off read from global memory, unverified j skipped, the sub-chunks
// loaded with plain vector loads.
template <typename T>
__global__ void __launch_bounds__(256) verify_rows_wide_kernel(
    int R, int gamma, int V, int n_chunks, long long n_rows, const T* __restrict__ target,
    const int32_t* __restrict__ ell, const int32_t* __restrict__ row_off, ScalePair sc,
    int greedy, double* __restrict__ row_part, uint32_t* status) {
  const uint64_t pol = sm100::policy_evict_first();
  grid_dependency_wait();  // ell, row_off
  const long long total = (long long)R * (gamma + 1) * n_chunks;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long item = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       item < total; item += nwarps) {
    const long long nj = item / n_chunks;
    const int c = (int)(item - nj * n_chunks);
    const int n = (int)(nj / (gamma + 1)), j = (int)(nj - (long long)n * (gamma + 1));
    const int L = ell[n];
    if (j > L || L > gamma) continue;
    const long long row = (long long)row_off[n] + j;
    if (row < 0 || row >= n_rows) continue;  // reported by the decide kernel
    RowState st;
    for (int sb = 0; sb < kRowGroup; ++sb) {
      const int v0 = c * kRowChunk + sb * kRowSub;
      if (v0 >= V) break;
      RowRaw<T> x;
      x.load(target + (size_t)row * V + v0, V - v0, pol);
      st.add(x, v0, V, sc, greedy);
    }
    st.store(greedy, row_part + ((size_t)n * (gamma + 1) + j) * n_chunks + c, status);
  }
}

// ---------------------------------------------------------------- decide

// u < p(x) / q(x) with p(x) = 2^a / Sp, a = t_x * log2(e) / T, in fp32
// (Sp = F * 2^g = m * 2^e with m = F's top 24 bits in [1, 2)): the result can
// differ from the exact comparison only when u lies within about 1e-6 of the
// ratio.
__device__ __forceinline__ bool accept_test(float tx, ScalePair sc, long long F, int g, float qx,
                                            float u) {
  if (F <= 0) return false;
  const int msb = 63 - __clzll(F);
  const uint32_t top =
      msb >= 23 ? (uint32_t)(F >> (msb - 23)) : (uint32_t)((unsigned long long)F << (23 - msb));
  const float ms = __uint_as_float(0x3f800000u | (top & 0x7fffffu));  // [1, 2)
  const float p = exp2f(scaled(tx, sc) - (float)(msb + g)) / ms;
  return u < p / qx;
}

// A row's chunk partials are exact doubles of fixed-point sums: their total
// F * 2^g is formed exactly as an integer sum in units of 2^g, g from the
// largest exponent so that n_chunks of them stay below 2^62 (one warp; every
// lane gets F and g).  No double instruction is used.  Non-finite partials
// are counted as 0 and reported in *bad.
__device__ __forceinline__ long long warp_fix_total(const double* __restrict__ pj, int n_chunks,
                                                    int* g_out, bool* bad) {
  const int lane = threadIdx.x & 31;
  constexpr int kReg = 8;  // chunks per lane kept in registers (n_chunks <= 256)
  const bool fast = n_chunks <= 32 * kReg;
  auto clean = [&](double x) -> double {
    if (((__double_as_longlong(x) >> 52) & 0x7ff) == 0x7ff) {
      *bad = true;
      return 0.0;
    }
    return x;
  };
  double pv[kReg];
  int emax = INT_MIN;
  if (fast) {
#pragma unroll
    for (int i = 0; i < kReg; ++i) {
      const int c = lane + 32 * i;
      pv[i] = c < n_chunks ? clean(__ldcg(pj + c)) : 0.0;
      emax = max(emax, double_exponent(pv[i]));
    }
  } else {
    for (int c = lane; c < n_chunks; c += 32)
      emax = max(emax, double_exponent(clean(__ldcg(pj + c))));
  }
  emax = __reduce_max_sync(0xffffffffu, emax);
  if (emax == INT_MIN) {
    *g_out = 0;
    return 0;
  }
  const int g = emax + 2 + (32 - __clz(n_chunks)) - 62;
  long long loc = 0;
  if (fast) {
#pragma unroll
    for (int i = 0; i < kReg; ++i) loc += double_to_fix(pv[i], g);
  } else {
    for (int c = lane; c < n_chunks; c += 32) loc += double_to_fix(clean(__ldcg(pj + c)), g);
  }
  *g_out = g;
  return warp_sum_nonneg_ll(loc);
}


// The accept tests and the final-draw state of request n, by one block of 256
// threads (every thread must call it; it returns with warps at different
// points, so a caller's next block barrier orders what follows).  Used by the
// decide kernel and by the row pass's block that completes request n's last
// item (row partials written by other blocks of that kernel: L2 loads).
template <typename T>
__device__ __noinline__ void decide_request(
    int n, int gamma, int V, int n_chunks, long long n_rows, const T* __restrict__ target,
    ScalePair sc, int greedy, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const double* __restrict__ q_lse,
    const float* __restrict__ q_tok, const int32_t* __restrict__ ell,
    const int32_t* __restrict__ row_off, const float* __restrict__ u_acc,
    const double* __restrict__ row_part, double* __restrict__ p_lse,
    int32_t* __restrict__ n_acc_out, int32_t* __restrict__ out_tokens,
    VerifyState* __restrict__ vstate, int32_t* __restrict__ prev_out, uint32_t* status) {
  __shared__ long long SpF[kMaxGamma + 1];  // target row totals F * 2^g
  __shared__ int Spg[kMaxGamma + 1];
  __shared__ ArgMax am_s[kMaxGamma + 1];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int L = ell[n];
  const long long r0 = row_off[n];
  // the same for every thread of the block
  const bool bad = L < 0 || L > gamma || r0 < 0 || r0 + L >= n_rows;
  int32_t* ot = out_tokens + (size_t)n * (gamma + 1);
  if (bad) {
    if (tid == 0) set_flag(status, kFlagRowRange);
    for (int j = tid; j <= gamma; j += blockDim.x) ot[j] = -1;
    if (tid == 0) {
      n_acc_out[n] = 0;
      VerifyState st{0, -1, 0, -1, {0.f, 0.f, 0}, {0.f, 0.f, 0}};
      vstate[n] = st;
      prev_out[n] = -1;
    }
    return;
  }
  // warp 0, lane j < L: drafted token j, its target logit, q, u and q_lse
  // (the q_lse and the previous token of the rejected position are taken
  // from these registers later); lane 0 also the anchor.  Issued before the
  // row totals' loads, which do not wait for them.
  int x_pre = -1, anc = -1;
  float tx_pre = 0.f, qx_pre = 1.f, u_pre = 1.f;
  double ql_pre = 0.0;
  if (wid == 0 && lane < L) {
    x_pre = tokens[(size_t)n * gamma + lane];
    if (!greedy) {
      qx_pre = q_tok[(size_t)n * gamma + lane];
      u_pre = u_acc[(size_t)n * gamma + lane];
      ql_pre = q_lse[(size_t)n * gamma + lane];
    }
    if (x_pre >= 0 && x_pre < V) tx_pre = to_f32<T>(target[(size_t)(r0 + lane) * V + x_pre]);
  }
  if (wid == 0 && lane == 0 && anchor != nullptr) anc = anchor[n];
  const double* part = row_part + (size_t)n * (gamma + 1) * n_chunks;
  for (int j = wid; j <= L; j += blockDim.x >> 5) {
    const double* pj = part + (size_t)j * n_chunks;
    if (greedy) {
      ArgMax am{-INFINITY, 0x7fffffff};
      for (int c = lane; c < n_chunks; c += 32) {
        const long long raw = __ldcg(reinterpret_cast<const long long*>(pj) + c);
        am = better(am, ArgMax{__int_as_float((int)(raw & 0xffffffffll)), (int)(raw >> 32)});
      }
      am = warp_argmax(am);
      if (lane == 0) {
        am_s[j] = am;
        if (p_lse) p_lse[r0 + j] = (double)am.v;
      }
    } else {
      int g;
      bool nonfinite = false;
      const long long F = warp_fix_total(pj, n_chunks, &g, &nonfinite);
      if (nonfinite) set_flag(status, kFlagNonFinite);
      if (lane == 0) {
        SpF[j] = F;
        Spg[j] = g;
        if (F <= 0) set_flag(status, kFlagNonFinite);
        if (p_lse) p_lse[r0 + j] = F > 0 ? (double)fix_log(F, g) : -INFINITY;
      }
    }
  }
  __syncthreads();
  if (wid != 0) return;
  // warp 0: the accept tests of the L drafted positions, one lane each, then
  // n_acc = the first rejection
  bool acc = true;
  if (lane < L) {
    const int x = x_pre;
    if (x < 0 || x >= V) {
      set_flag(status, kFlagTokenRange);
      acc = false;
    } else if (greedy) {
      acc = (x == am_s[lane].i);
    } else {
      acc = accept_test(tx_pre, sc, SpF[lane], Spg[lane], qx_pre, u_pre);
    }
  }
  const unsigned live = L >= 32 ? 0xffffffffu : ((1u << L) - 1u);
  const unsigned rej = __ballot_sync(0xffffffffu, !acc) & live;
  const int nacc = rej ? __ffs(rej) - 1 : L;
  for (int j = lane; j <= gamma; j += 32) {
    int v = -1;
    if (j < nacc) v = tokens[(size_t)n * gamma + j];
    else if (j == nacc && greedy) v = am_s[nacc].i;
    ot[j] = v;
  }
  // the rejected position's q_lse and the token before it (nacc < L when a
  // position is rejected, so both are in lanes below L)
  const double ql_rej = __shfl_sync(0xffffffffu, ql_pre, nacc & 31);
  const int x_before = __shfl_sync(0xffffffffu, x_pre, nacc > 0 ? (nacc - 1) & 31 : 0);
  if (lane != 0) return;
  n_acc_out[n] = nacc;
  VerifyState st;
  st.n_acc = nacc;
  st.mode = greedy ? -1 : (nacc == L ? 0 : 1);
  st.final_row = (int)(r0 + nacc);
  st.prev = -1;
  st.ip = greedy ? InvPair{0.f, 0.f, 0} : inv_fix(SpF[nacc], Spg[nacc]);
  st.iq = InvPair{0.f, 0.f, 0};
  if (st.mode == 1) {
    // the bias row of the rejected position: the Markov row of the token
    // before it, or (no anchors: the RNN head) the state S[n][nacc]
    st.prev = anchor == nullptr ? n * gamma + nacc : (nacc == 0 ? anc : x_before);
    st.iq = exp_neg_pair(ql_rej);
  }
  vstate[n] = st;
  prev_out[n] = st.prev;
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
  grid_dependency_wait();  // the row partials
  decide_request<T>(blockIdx.x, gamma, V, n_chunks, n_rows, target, sc, greedy, anchor, tokens,
                    q_lse, q_tok, ell, row_off, u_acc, row_part, p_lse, n_acc_out, out_tokens,
                    vstate, prev_out, status);
}

// ---------------------------------------------------------------- final draw

// (hi, lo) fp32 pair of 2^ref / S from the request's InvPair of 1/S.
__device__ __forceinline__ ScalePair norm_pair(int ref, InvPair ip) {
  return ScalePair{scale_pow2(ip.hi, ref + ip.e), scale_pow2(ip.lo, ref + ip.e)};
}

// One warp, one 256-token tile of request n's final draw: per lane the eight
// tokens t*256 + lane*8 .. +7.  fp / fr = the normalised target probability
// p and the residual max(0, p - q) (= p for a bonus draw) in units of 2^-60.
// The pick kernel calls this again for the chosen tile and gets identical
// values.
template <typename T>
__device__ __forceinline__ void final_warp_tile(int gamma, int V, int t,
                                                const T* __restrict__ z,
                                                const float* __restrict__ bias,
                                                const T* __restrict__ target, ScalePair sc,
                                                const VerifyState& st, int n, long long (&fr)[8],
                                                long long (&fp)[8]) {
  const int lane = threadIdx.x & 31;
  const int v0 = t * kFinTile + lane * 8;
  float ap[8], aq[8], bb[8];
  // all loads first (one memory round trip), then the arithmetic
  load8<T>(target + (size_t)st.final_row * V, v0, V, ap, -INFINITY);
  if (st.mode == 1) {
    load8<T>(z + ((size_t)n * gamma + st.n_acc) * V, v0, V, aq, -INFINITY);
    load8<float>(bias + (size_t)n * V, v0, V, bb, 0.f);
  }
  float mp = -3.0e38f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ap[e] = scaled_clamped(ap[e], sc);
    mp = fmaxf(mp, ap[e]);
  }
  mp = warp_max(mp);
  float mq = -3.0e38f;
  if (st.mode == 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      aq[e] = scaled_clamped(aq[e] + bb[e], sc);
      mq = fmaxf(mq, aq[e]);
    }
    mq = warp_max(mq);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) aq[e] = -3.0e38f;
  }
  const int refp = mp > -1.0e38f ? (int)ceilf(mp) : 0;
  const int refq = mq > -1.0e38f ? (int)ceilf(mq) : 0;
  const ScalePair kp = mp > -1.0e38f ? norm_pair(refp, st.ip) : ScalePair{0.f, 0.f};
  const ScalePair kq = mq > -1.0e38f ? norm_pair(refq, st.iq) : ScalePair{0.f, 0.f};
  constexpr float k2_60 = 1152921504606846976.0f;  // 2^60
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float wp = ex2_fast(ap[e] - (float)refp);
    const float p = fmaf(wp, kp.hi, wp * kp.lo);
    float rho = p;
    if (st.mode == 1) {
      const float wq = ex2_fast(aq[e] - (float)refq);
      rho = fmaxf(0.0f, p - fmaf(wq, kq.hi, wq * kq.lo));
    }
    fp[e] = __float2ll_rn(p * k2_60);
    fr[e] = __float2ll_rn(rho * k2_60);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) final_partial_kernel(
    int gamma, int V, int n_tiles, const T* __restrict__ z, const float* __restrict__ bias,
    const T* __restrict__ target, ScalePair sc, const VerifyState* __restrict__ vstate,
    long long* __restrict__ fin_part) {
  const int n = blockIdx.y;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= n_tiles) return;
  const VerifyState st = vstate[n];
  long long* out = fin_part + ((size_t)n * n_tiles + t) * 2;
  if (st.mode < 0) {
    if ((threadIdx.x & 31) == 0) out[0] = out[1] = 0;
    return;
  }
  long long fr[8], fp[8];
  final_warp_tile<T>(gamma, V, t, z, bias, target, sc, st, n, fr, fp);
  long long sr = 0, sp = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sr += fr[e];
    sp += fp[e];
  }
  sr = warp_sum(sr);
  sp = warp_sum(sp);
  if ((threadIdx.x & 31) == 0) {
    out[0] = sr;
    out[1] = sp;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) final_pick_kernel(
    int gamma, int V, int n_tiles, const T* __restrict__ z, const float* __restrict__ bias,
    const T* __restrict__ target, ScalePair sc, const VerifyState* __restrict__ vstate,
    const long long* __restrict__ fin_part, const float* __restrict__ u_fin,
    int32_t* __restrict__ out_tokens, uint32_t* status) {
  __shared__ long long shl[32];
  __shared__ int shi[32];
  __shared__ long long incl_s[256];
  __shared__ long long base_s;
  __shared__ int tsel_s;
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
  if (cand == tsel) {
    base_s = base;
    tsel_s = tsel;
  }
  __syncthreads();
  if (tid >= 32) return;
  // warp 0: the chosen tile again, then its inclusive prefix in token order
  long long fr[8], fp[8];
  final_warp_tile<T>(gamma, V, tsel_s, z, bias, target, sc, st, n, fr, fp);
  long long w[8], lsum = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w[e] = col == 0 ? fr[e] : fp[e];
    lsum += w[e];
  }
  long long lincl = lsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, lincl, o);
    if (tid >= o) lincl += y;
  }
  long long run = base_s + (lincl - lsum);
  int pick = 0x7fffffff, last = -1;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    run += w[e];
    if (w[e] > 0) last = tid * 8 + e;
    if (pick == 0x7fffffff && w[e] > 0 && run > thr) pick = tid * 8 + e;
  }
  pick = __reduce_min_sync(0xffffffffu, pick);
  last = __reduce_max_sync(0xffffffffu, last);
  if (tid == 0) {
    const int idx = pick != 0x7fffffff ? pick : (last >= 0 ? last : 0);
    out_tokens[(size_t)n * (gamma + 1) + st.n_acc] = tsel_s * kFinTile + idx;
  }
}

// Pick of the final draw on the tensor-core path.  The partials are per
// 128-token half tile and were formed with the tensor-core bias; the chosen
// half tile is recomputed here with the bias on CUDA cores, so its running
// sums can differ from its partial in the last bits.  The crossing is placed
// at the same fraction of the recomputed half tile (exact 128-bit
// cross-multiplication), as in the draft finish.
__global__ void __launch_bounds__(256) final_pick_tc_kernel(
    int gamma, int V, int r, int n_halves, const __nv_bfloat16* __restrict__ z,
    const __nv_bfloat16* __restrict__ target, const __nv_bfloat16* __restrict__ E,
    const __nv_bfloat16* __restrict__ Wt, ScalePair sc, const VerifyState* __restrict__ vstate,
    const long long* __restrict__ fin_part, const float* __restrict__ u_fin,
    int32_t* __restrict__ out_tokens, uint32_t* status) {
  __shared__ FinishScratch s;
  const int n = blockIdx.x, tid = threadIdx.x;
  // The verification state was complete before the final pass (the kernel
  // this one waits for) could finish: it, the uniform and the previous
  // token's E row are read before the wait; the partials after it.
  const VerifyState st = vstate[n];
  if (st.mode < 0) return;
  const bool resid = st.mode == 1;
  if (resid) {  // the previous token's E row, needed once the half tile is known
    for (int i = tid; i < r; i += 256)
      s.erow[i] = st.prev >= 0 ? __bfloat162float(E[(size_t)st.prev * r + i]) : 0.f;
  }
  const float u = u_fin[n];
  grid_dependency_wait();  // the final partials
  const long long* P = fin_part + (size_t)n * n_halves * 2;
  const int seg = (n_halves + 255) / 256;
  const int t0 = min(n_halves, tid * seg), t1 = min(n_halves, t0 + seg);
  long long lr = 0, lp = 0;
  for (int t = t0; t < t1; ++t) {
    lr += P[2 * t];
    lp += P[2 * t + 1];
  }
  // both columns' scans at once; the residual column unless p and q agree
  // everywhere (then p itself)
  long long ir = lr, ip = lp, Fr, Fp;
  g_scan_ll2<BlockSync>(ir, ip, s.shl, s.shl2, &Fr, &Fp);
  const int col = (resid && Fr > 0) ? 0 : 1;
  const long long loc = col == 0 ? lr : lp;
  const long long F = col == 0 ? Fr : Fp;
  const long long incl = col == 0 ? ir : ip;
  if (F <= 0) {
    if (tid == 0) {
      set_flag(status, kFlagNonFinite);
      out_tokens[(size_t)n * (gamma + 1) + st.n_acc] = 0;
    }
    return;
  }
  const long long thr = floor_mul(u, F);  // C > u*F  <=>  C > floor(u*F)
  int cand = 0x7fffffff;
  long long base = 0, ssel = 0;
  {
    long long run = incl - loc;
    for (int t = t0; t < t1; ++t) {
      const long long x = P[2 * t + col];
      const long long nx = run + x;
      if (cand == 0x7fffffff && nx > thr) {
        cand = t;
        base = run;
        ssel = x;
      }
      run = nx;
    }
  }
  const int hsel = g_min_i<BlockSync>(cand, s.shi);  // found: F > thr
  if (cand == hsel) {
    s.base = base;
    s.ssel = ssel;
  }
  __syncthreads();
  base = s.base;
  ssel = s.ssel;
  // recompute the chosen half tile: thread tid < 128 takes token hsel*128 + tid
  const int v = hsel * 128 + tid;
  const bool ok = tid < 128 && v < V;
  const float tv = ok ? __bfloat162float(target[(size_t)st.final_row * V + v]) : -INFINITY;
  float zv = 0.f;
  if (resid && ok) zv = __bfloat162float(z[((size_t)n * gamma + st.n_acc) * V + v]);
  float bv = 0.f;
  if (resid) {
    const BiasSrc b{nullptr, E, Wt, nullptr, 0, r};
    tile_bias_recompute<128, BlockSync>(b, V, hsel * 128, s.erow, s.bias);
    bv = tid < 128 ? s.bias[tid] : 0.f;
  }
  // the same arithmetic as the final pass's blocks: a = y * c (c rounded to
  // fp32), p = 2^(a + e) * (hi + lo) with 1/Sp = (hi + lo) * 2^e, q alike
  const float yp = ok ? tv : -INFINITY;
  const float yq = ok && resid ? zv + bv : -INFINITY;
  long long f = 0;
  if (ok && st.ip.hi != 0.f) {
    const float wp = ex2_fast(fmaf(yp, sc.hi, (float)st.ip.e));
    const float pv = fmaf(wp, st.ip.hi, wp * st.ip.lo);
    float rho = pv;
    if (resid && st.iq.hi != 0.f) {
      const float wq = ex2_fast(fmaf(yq, sc.hi, (float)st.iq.e));
      rho = fmaxf(0.0f, pv - fmaf(wq, st.iq.hi, wq * st.iq.lo));
    }
    const float val = col == 0 ? rho : pv;
    if (val == val) f = __float2ll_rn(val * 1152921504606846976.0f);  // 2^60
  }
  long long mass;
  const long long cum = g_scan_ll<BlockSync>(f, s.shl, &mass);
  //   cum / mass > (thr - base) / ssel  <=>  cum * ssel > (thr - base) * mass
  int pick = 0x7fffffff;
  if (f > 0 && mul_gt((unsigned long long)cum, (unsigned long long)ssel,
                      (unsigned long long)(thr - base), (unsigned long long)mass))
    pick = tid;
  int isel = g_min_i<BlockSync>(pick, s.shi);
  if (isel == 0x7fffffff) isel = g_max_i<BlockSync>(f > 0 ? tid : -1, s.shi);
  if (isel < 0) isel = 0;
  if (tid == 0) out_tokens[(size_t)n * (gamma + 1) + st.n_acc] = hsel * 128 + isel;
}

// The row pass's grid: as many blocks as fit on the GPU at once (every block
// strides over the items), at most one warp per item.
template <typename K>
int row_grid(K kernel, long long items, size_t dyn_smem) {
  int per_sm = blocks_per_sm((const void*)kernel, 256, dyn_smem);
  if (per_sm < 1) per_sm = 1;
  const long long resident = (long long)per_sm * sm_count();
  const long long blocks = (items + 7) / 8;
  return (int)(blocks < resident ? (blocks < 1 ? 1 : blocks) : resident);
}

template <typename T>
cudaError_t run_verify(const VerifyArgs& a, cudaStream_t st) {
  const bool greedy = a.T == 0.0f;
  const ScalePair sc = make_scale(greedy ? 1.0 : 1.4426950408889634 / (double)a.T);
  const int n_chunks = (a.V + kRowChunk - 1) / kRowChunk;
  const int n_tiles = (a.V + kFinTile - 1) / kFinTile;
  const T* z = (const T*)a.z;
  const T* tg = (const T*)a.target;
  const long long items = (long long)a.R * (a.gamma + 1) * n_chunks;
  // rows of E the final draw may read: tokens, or (RNN head) the states
  const int lim = a.anchor == nullptr ? a.R * a.gamma : a.V;
  const bool staged = sizeof(T) == 2 && a.R <= kRowsSmem && a.V % 8 == 0 &&
                      ((uintptr_t)a.target & 15) == 0;
  // the staged row pass runs every request's decide itself
  const DecideOut dec{staged && a.vcnt != nullptr ? 1 : 0, a.anchor, a.tokens, a.q_lse, a.q_tok,
                      a.u_acc, a.p_lse, a.n_acc, a.out_tokens, a.vstate, a.prev, a.vcnt};
  if (staged) {
    // the opt-in for the largest list, once per device; the resident grid
    // for this list size (cached per device and size)
    const size_t dyn = rows_tma_smem(a.R);
    auto kern = greedy ? verify_rows_tma_kernel<true> : verify_rows_tma_kernel<false>;
    cudaError_t ea = ensure_smem_attr((const void*)kern, (int)rows_tma_smem(kRowsSmem));
    if (ea != cudaSuccess) return ea;
    const int grid = row_grid(kern, 1ll << 40, dyn);
    const int g = (int)(grid < (items + 7) / 8 ? grid : (items + 7) / 8);
    DSPARK_LAUNCH(kKindVerifyRows, st,
                  launch_pdl(kern, dim3(g), dim3(256), dyn, st, a.R, a.gamma, a.V, n_chunks,
                             a.n_rows, reinterpret_cast<const __nv_bfloat16*>(tg), a.ell,
                             a.row_off, sc, a.row_part, a.status, dec));
  } else {
    DSPARK_LAUNCH(kKindVerifyRows, st,
                  launch_pdl(verify_rows_wide_kernel<T>,
                             dim3(row_grid(verify_rows_wide_kernel<T>, items, 0)), dim3(256), 0,
                             st, a.R, a.gamma, a.V, n_chunks, a.n_rows, tg, a.ell, a.row_off, sc,
                             (int)greedy, a.row_part, a.status));
  }
  if (!dec.on)
    DSPARK_LAUNCH(kKindVerifyDecide, st,
                  launch_pdl(verify_decide_kernel<T>, dim3(a.R), dim3(256), 0, st, a.gamma, a.V,
                             n_chunks, a.n_rows, tg, sc, (int)greedy, a.anchor, a.tokens,
                             a.q_lse, a.q_tok, a.ell, a.row_off, a.u_acc,
                             (const double*)a.row_part, a.p_lse, a.n_acc, a.out_tokens, a.vstate,
                             a.prev, a.status));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || greedy) return e;
  if (tc_shape_supported(a.dt, a.V, a.r, a.z, a.E, a.Wt) &&
      (((uintptr_t)a.target & 15) == 0)) {
    // bias, p and the residual in one tensor-core pass; the pick recomputes
    // its half tile
    e = launch_final_tc(a, a.vstate, a.fin_part, st);
    if (e != cudaSuccess) return e;
    const int n_halves = (a.V + 127) / 128;
    DSPARK_LAUNCH(kKindFinalPick, st,
                  launch_pdl(final_pick_tc_kernel, dim3(a.R), dim3(256), 0, st, a.gamma, a.V,
                             a.r, n_halves, (const __nv_bfloat16*)a.z,
                             (const __nv_bfloat16*)a.target, (const __nv_bfloat16*)a.E,
                             (const __nv_bfloat16*)a.Wt, sc, (const VerifyState*)a.vstate,
                             (const long long*)a.fin_part, a.u_fin, a.out_tokens, a.status));
    return cudaGetLastError();
  }
  e = tc_shape_supported(a.dt, a.V, a.r, a.z, a.E, a.Wt)
          ? launch_bias_tc(a.R, a.V, a.r, a.E, a.Wt, a.prev, 1, lim, a.bias, a.status, st)
          : launch_bias(a.R, a.V, a.r, a.dt, a.E, a.Wt, a.prev, 1, lim, a.bias, a.status, st);
  if (e != cudaSuccess) return e;
  DSPARK_LAUNCH(kKindFinalPartial, st,
                final_partial_kernel<T><<<dim3((n_tiles + 7) / 8, a.R), 256, 0, st>>>(
                    a.gamma, a.V, n_tiles, z, a.bias, tg, sc, a.vstate, a.fin_part));
  DSPARK_LAUNCH(kKindFinalPick, st,
                final_pick_kernel<T><<<a.R, 256, 0, st>>>(a.gamma, a.V, n_tiles, z, a.bias, tg,
                                                         sc, a.vstate, a.fin_part, a.u_fin,
                                                         a.out_tokens, a.status));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t st) {
  return a.dt == 0 ? run_verify<__nv_bfloat16>(a, st) : run_verify<float>(a, st);
}

}  // namespace dspark
