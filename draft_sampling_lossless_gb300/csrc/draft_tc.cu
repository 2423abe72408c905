// The tensor-core kernels of the draft and of the final draw (5th-generation
// tensor cores: tcgen05 MMA into TMEM accumulators, TMA operand loads).
//
// "DSpark.让每一轮计算，多走几步" (explainer), Markov head panel, and the news
// article "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", innovation 1, second stage: at draft
// position k every request's previous token selects a row of the low-rank
// table E, and bias = E[x_{k-1}] . W is added to the backbone logits before
// the draw.  The bias is never written to memory: per vocabulary tile the MMA
//     D[m][v] = sum_i E[x_{k-1}(m)][i] * Wt[v][i]          (M=128, N=256, K=r)
// lands in tensor memory, and the epilogue turns each thread's row of D plus
// the matching slice of z into y = z + bias, a = y * log2(e)/T and, per
// 128-token half tile, the exact fixed-point sum of 2^(a - ref) (greedy: the
// half tile's max and argmax) with its 16-token group sums.
//
// Kernels:
//   draft_persistent_kernel  every draft position in one cooperative launch
//       (the main path): partial pass, grid barrier, the per-request finish
//       (finish.cuh) that draws x_k and stages E[x_k] for the next A operand,
//       grid barrier; optionally also the confidence head and the scheduler
//       (dspark_draft_schedule).
//   draft_fused_tc_kernel    one draft position's partial pass (the fallback
//       when a cooperative launch is not possible; the finish is a separate
//       launch), or in bias-out mode the fp32 bias rows.
//   final_tc_kernel          the verification's final draw: the rejected
//       position's bias in TMEM and, per half tile, the fixed-point sums of
//       the target's p and of max(0, p - q).
//
// Warp roles (352 threads, one CTA an SM):
//   warps 0-7  epilogue: warp w reads TMEM lane quadrant w % 4 and token
//              half w / 4 of the accumulator; also the gathers and finishes
//   warp 8     TMA producer of Wt K-chunks [256 tokens x 64] (3-stage ring)
//   warp 9     TMEM allocation and the single MMA-issuing thread
//   warp 10    producer of z (TMA boxes) or of the final draw's rows
// A operands are in the 128-byte swizzled K-major layout; with R <= 64 the
// paired layout puts two vocabulary tiles in one accumulator.  Two 256-column
// accumulators alternate so the MMA of one unit overlaps the epilogue of the
// previous one.  Every wait is bounded (about one second on an mbarrier, two
// on a grid barrier); a timeout sets DSPARK_DEVFLAG_TIMEOUT, makes the other
// waits of the CTA give up at once, and the kernel runs to completion.
#include <climits>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "confidence.cuh"
#include "f32x2.cuh"
#include "finish.cuh"
#include "schedule.cuh"
#include "sm100.cuh"

namespace dspark {

namespace {

using namespace sm100;

constexpr int BM = 128;           // requests per tile (MMA M, TMEM lanes)
constexpr int BN = 256;           // tokens per tile (MMA N)
constexpr int BK = 64;            // K chunk = one 128-byte swizzle row of bf16
constexpr int kHalf = BN / 2;     // tokens per epilogue warp per tile = partial width
constexpr int kStagesB = 3;
constexpr int kZBoxes = 4;        // 64-token boxes of z per tile
constexpr int kEpiWarps = 8;
constexpr int kThreads = (kEpiWarps + 3) * 32;
constexpr int kWarpW = kEpiWarps, kWarpMma = kEpiWarps + 1, kWarpZ = kEpiWarps + 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kABytesPerChunk = BM * BK * 2;  // 16 KiB
constexpr uint32_t kBBytes = BN * BK * 2;          // 32 KiB
constexpr uint32_t kZBytes = BM * 64 * 2;          // 16 KiB
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);
constexpr uint32_t kFlagTimeout = 0x10u;
// mbarriers: fullB[3] @0, emptyB[3] @3, fullZ[2][4] @6, emptyZ[2][4] @14,
// accFull[2] @22, accEmpty[2] @24, drain @26, aFull @27 (persistent kernel:
// the staged A operand); the TMEM address word @28
constexpr int kBars = 29;

struct TcParams {
  int R, gamma, V, r, k, nK, n_vt, n_parts;
  int greedy;
  ScalePair sc;
  float c12, crest;  // log2(e)/T = c12 + crest, c12 with 12 significant bits
  const __nv_bfloat16* E;
  const int32_t* prev;  // null: row n * prev_stride of E (the RNN states)
  int prev_stride;
  int prev_limit;   // rows of E: larger previous-token entries are flagged
  double* part;     // [R][n_parts] partials (draft mode)
  float* sub;       // [R][n_parts][8] 16-token group sums of each partial (sampling)
  float* bias_out;  // [R][V] (bias-out mode)
  uint32_t* status;
};

size_t tc_smem_bytes(int nK) {
  return 1024 + (size_t)nK * kABytesPerChunk + kStagesB * kBBytes + kZBoxes * kZBytes +
         kBars * sizeof(uint64_t) + 16;
}

// Bounded wait that also gives up at once when another role of the CTA has
// already timed out, so a broken pipeline ends the kernel quickly.
// After the first tries the thread sleeps in the wait (woken by the phase
// completion), so waiting roles leave the issue slots to working warps.
// limit_ns: how long to wait before giving up (the kernels use about 1 s).
constexpr uint64_t kMbarLimitNs = 1000000000ull;
constexpr uint64_t kGridLimitNs = 2000000000ull;

__device__ __forceinline__ bool wait_abortable(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, uint32_t* status,
                                               uint64_t limit_ns = kMbarLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      set_flag(status, kFlagTimeout);
      return false;
    }
  }
}

// The z ring.  Slot s holding a box that token half h reads is guarded by
// the barrier pair (fullZ[h][s], emptyZ[h][s]).  With fewer slots than boxes
// per tile a slot is read alternately by both halves; one barrier pair per
// (half, slot) keeps each barrier's phases consecutive for its only reader,
// so a parity wait can never match an older phase.  The producer remembers
// which half read each slot last and waits for that half's release.
struct ZRing {
  uint32_t epar = 0;  // bit h*4+s: parity of the next release of (h, s) to wait for
  uint32_t last = 0;  // two bits per slot: 1 + the half that read it last, 0 = unused
  __device__ __forceinline__ void acquire(uint32_t b_emptyZ, int s, int h, volatile int* abort_flag,
                                          uint32_t* status) {
    const uint32_t lu = (last >> (2 * s)) & 3u;
    if (lu != 0) {
      const int bit = (int)(lu - 1) * 4 + s;
      wait_abortable(b_emptyZ + 8 * bit, (epar >> bit) & 1u, abort_flag, status);
      epar ^= 1u << bit;
    }
    last = (last & ~(3u << (2 * s))) | ((uint32_t)(h + 1) << (2 * s));
  }
};

// Slot and phase of a stage ring, advanced by increment and wrap so that
// the single MMA-issuing thread spends no cycles on divisions.
struct RingPos {
  uint32_t s = 0, ph = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// The four K=16 MMAs of one 64-wide K chunk.  Both descriptors start at
// their operand's chunk and advance 32 bytes (2 in the descriptor's 16-byte
// address units) per step inside the 128-byte swizzle row.
__device__ __forceinline__ void mma_chunk(uint32_t d_tmem, uint64_t da, uint64_t db,
                                          bool accumulate) {
  mma_bf16(d_tmem, da, db, kIdesc, accumulate ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < BK / 16; ++kk) mma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, kIdesc, 1u);
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Per-thread running state of one (request, half tile) partial.
struct Part {
  long long acc;  // sum of 2^(a - ref) in units of 2^-40
  int ref;        // power-of-two reference, INT_MIN = no mass yet
  int bad;        // a NaN or +inf input was seen
  ArgMax best;    // greedy
};


// TwoSum (Knuth): s = RN(a + b) and the exact error a + b - s, for any
// order of magnitudes; the packed form does two pairs at once.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err) {
  s = a + b;
  const float bb = s - a;
  err = (a - (s - bb)) + (b - bb);
}
__device__ __forceinline__ void two_sum2(unsigned long long a, unsigned long long b,
                                         unsigned long long& s, unsigned long long& err) {
  const unsigned long long t = add2(a, b);
  const unsigned long long bb = sub2(t, a);
  err = add2(sub2(a, sub2(t, bb)), sub2(b, bb));
  s = t;
}

// round(x * 2^40) for 0 <= x < 2^22, from the float's bits (no conversion
// instruction): exact once x * 2^40 >= 2^23, where the float holds an
// integer; below, the bits under 2^-40 are dropped (less than one unit).
__device__ __forceinline__ long long fix40(float x) {
  const uint32_t b = __float_as_uint(x);
  const int e = (int)(b >> 23);  // x >= 0: the biased exponent
  const unsigned long long m = (b & 0x7fffffu) | (e ? 0x800000u : 0u);
  const int sh = e - 110;  // x * 2^40 = m * 2^(e - 150 + 40)
  return (long long)(sh >= 0 ? m << sh : (sh > -24 ? m >> -sh : 0ull));
}

// Greedy: the arg-max of y = z + b over 32 consecutive tokens of one
// request row (one 32-column accumulator load b and the z words zq), half h
// (tokens v0 + 32h ..) of a 64-token block; `lim` = number of the block's
// tokens below V.  The half's maximum first (NaN-propagating, so a NaN shows
// in it; then the maximum of the other values is taken again), then its
// first index, then one comparison with the running best (lowest index on
// ties: the halves come in token order).  NaN and +inf set s.bad.
template <bool kRagged>
__device__ __forceinline__ void epi_half_greedy(const uint32_t (&b)[32], const uint4 (&zq)[4],
                                                int h, int v0, int lim, Part& s) {
  const int t0 = h * 32;
  float y[32];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t zw = (&zq[0].x)[k];
    unpack2(add2(pack2(bf_lo(zw), bf_hi(zw)),
                 pack2(__uint_as_float(b[2 * k]), __uint_as_float(b[2 * k + 1]))),
            y[2 * k], y[2 * k + 1]);
    if (kRagged) {
      if (t0 + 2 * k >= lim) y[2 * k] = -INFINITY;
      if (t0 + 2 * k + 1 >= lim) y[2 * k + 1] = -INFINITY;
    }
  }
  float mx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mx[e] = fmax_nan(fmax_nan(y[e], y[e + 8]), fmax_nan(y[e + 16], y[e + 24]));
#pragma unroll
  for (int w = 4; w > 0; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) mx[e] = fmax_nan(mx[e], mx[e + w]);
  float m = mx[0];
  if (!(m < INFINITY)) {  // NaN or +inf: flagged; the maximum of the non-NaN values
    s.bad = 1;
    if (m != m) {
      m = -INFINITY;
#pragma unroll
      for (int k = 0; k < 32; ++k) m = fmaxf(m, y[k]);
    }
  }
  int idx = 31;  // the first token holding the maximum (all NaN: the last, -inf weight)
#pragma unroll
  for (int k = 30; k >= 0; --k) idx = y[k] == m ? k : idx;
  s.best = better(s.best, ArgMax{m, v0 + t0 + idx});
}

// One weight 2^(x c + e) for two tokens at once, with the exponent split as
// in the draft epilogue: x c = P + x' (P = x_hi c12 exact for a bf16 x_hi;
// x' the rest), n = rint(P + bq c12 + e) clamped at -125, the fraction
// f = (P - rint(P + bq c12)) + bq c12 + (x_hi + bq) crest in [-1/2, 1/2]
// to ex2, 2^n from the magic number's bits.  xx: the bf16 values (z);
// bb: the Markov bias.
__device__ __forceinline__ unsigned long long pow2_split2(unsigned long long xx,
                                                          unsigned long long bb,
                                                          unsigned long long c12,
                                                          unsigned long long cr2,
                                                          unsigned long long k2, float klo) {
  const unsigned long long P = mul2(xx, c12);
  float qa, qb;
  unpack2(add2(fma2(bb, c12, P), k2), qa, qb);  // 1.5 * 2^23 + n
  qa = fmaxf(qa, klo);
  qb = fmaxf(qb, klo);
  const unsigned long long M = sub2(pack2(qa, qb), k2);
  unsigned long long F = fma2(bb, c12, sub2(P, M));
  F = fma2(xx, cr2, fma2(bb, cr2, F));
  float fa, fb;
  unpack2(F, fa, fb);
  const float sa = __uint_as_float(__float_as_uint(qa) * 8388608u + 0x3f800000u);  // 2^n
  const float sb = __uint_as_float(__float_as_uint(qb) * 8388608u + 0x3f800000u);
  return pack2(ex2_approx(fa) * sa, ex2_approx(fb) * sb);
}

// The same with the bias scaled by cf = c rounded to fp32 (one fused
// multiply-add fewer: bq c12 + bq crest becomes bq cf, whose rounding moves
// f by about 2^-24 |bq| c, far below ex2's own error).  The final draw's
// residual weights use it.
__device__ __forceinline__ unsigned long long pow2_split2_cf(unsigned long long xx,
                                                             unsigned long long bb,
                                                             unsigned long long c12,
                                                             unsigned long long cf2,
                                                             unsigned long long cr2,
                                                             unsigned long long k2, float klo) {
  const unsigned long long P = mul2(xx, c12);
  float qa, qb;
  unpack2(add2(fma2(bb, cf2, P), k2), qa, qb);  // 1.5 * 2^23 + n
  qa = fmaxf(qa, klo);
  qb = fmaxf(qb, klo);
  const unsigned long long M = sub2(pack2(qa, qb), k2);
  float fa, fb;
  unpack2(fma2(xx, cr2, fma2(bb, cf2, sub2(P, M))), fa, fb);
  const float sa = __uint_as_float(__float_as_uint(qa) * 8388608u + 0x3f800000u);  // 2^n
  const float sb = __uint_as_float(__float_as_uint(qb) * 8388608u + 0x3f800000u);
  return pack2(ex2_approx(fa) * sa, ex2_approx(fb) * sb);
}

// The same without a bias (the target logits): n = rint(P + e) clamped at
// -125, f = (P - rint(P)) + x_hi crest.
__device__ __forceinline__ unsigned long long pow2_split2_nb(unsigned long long xx,
                                                             unsigned long long c12,
                                                             unsigned long long cr2,
                                                             unsigned long long k2, float klo) {
  const unsigned long long P = mul2(xx, c12);
  float qa, qb;
  unpack2(add2(P, k2), qa, qb);  // 1.5 * 2^23 + n
  qa = fmaxf(qa, klo);
  qb = fmaxf(qb, klo);
  const unsigned long long M = sub2(pack2(qa, qb), k2);
  float fa, fb;
  unpack2(fma2(xx, cr2, sub2(P, M)), fa, fb);
  const float sa = __uint_as_float(__float_as_uint(qa) * 8388608u + 0x3f800000u);  // 2^n
  const float sb = __uint_as_float(__float_as_uint(qb) * 8388608u + 0x3f800000u);
  return pack2(ex2_approx(fa) * sa, ex2_approx(fb) * sb);
}

// (h, l) += (x, y) for double-float pairs: TwoSum of the high parts, the low
// parts added (their rounding is 2^-24 of a 2^-24 term).
__device__ __forceinline__ void add_pair(float& h, float& l, float x, float y) {
  float t, e;
  two_sum(h, x, t, e);
  h = t;
  l += e + y;
}

// TwoSum tree over 8 packed pairs (16 values): the sum as (hi, lo).
// Plain packed adds form the four-value partial sums (each a rounding near
// 2^-25 of a partial, about the size of one weight's own fp32 rounding);
// TwoSum the two levels above, so no rounding of a 16-token or larger sum
// reaches the fixed-point totals.
__device__ __forceinline__ void sum16(unsigned long long (&v)[8], float& hi, float& lo) {
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = add2(v[e], v[e + 4]);
#pragma unroll
  for (int e = 0; e < 2; ++e) v[e] = add2(v[e], v[e + 2]);
  unsigned long long s2, e2;
  two_sum2(v[0], v[1], s2, e2);
  float ha, hb, la, lb, er;
  unpack2(s2, ha, hb);
  unpack2(e2, la, lb);
  two_sum(ha, hb, hi, er);
  lo = er + (la + lb);
}

// Sampling: 32 consecutive tokens of one request row (one 32-column
// accumulator load b = the Markov bias, and the z words zq), half h (tokens
// 32h .. 32h + 31) of a 64-token block; `lim` = number of the block's tokens
// below V.  Adds the fixed-point sum of 2^t, t = (z + b) log2(e)/T - ref, to
// s.acc (units of 2^(s.ref - 40)), the sums of the half's two 16-token groups
// to gs[2h], gs[2h + 1] (units of 2^s.ref), and the low parts of their
// compensated sums to lo (converted once per block by the caller).  When the
// half raises the lane's reference, s.acc, lo and the groups already summed
// are rescaled exactly.
//
// The reference: ref = ceil(max y * c) from fp32 y = z + b (rounded
// monotone in y, c = log2(e)/T > 0); NaN and +inf surface in that maximum
// and drop the half (flagged); -inf (a masked token) weighs 0.
// Each weight is formed without rounding y or t at the magnitude of the
// logits (an fp32 y or t near 8 is off by up to 5e-7, which would shift
// every CDF boundary after it):
//   c = c12 + crest, c12 with 12 significant bits, so P = z c12 is exact
//   (z is bf16); Q = P + b c12 (rounded) only picks the integer M = rint(Q)
//   (a magic-number round) and n = M - ref (clamped at -125 so 2^n stays
//   normal); P - M is exact; the fraction f = (P - M) + b c12 + (z + b) crest
//   lies in [-1/2, 1/2] and is rounded twice at that magnitude (about 2e-8);
//   2^f comes from ex2 (5.5e-8 RMS relative error on [-1/2, 1/2], measured on
//   this GPU); 2^n scales it exactly, built from the magic number's bits.
// The sums are compensated: plain packed adds form four-token partials,
// TwoSum the levels above; a group's high part is converted to 2^-40 units
// exactly with integer operations.
// kRagged: the block holds the vocabulary's end (its last block only), so
// tokens at or past lim are masked; a template parameter, so that the
// unrolled pairs of the common case carry no branch.
template <bool kRagged>
__device__ __forceinline__ void epi_half(const uint32_t (&b)[32], const uint4 (&zq)[4], int h,
                                         int lim, const TcParams& p, Part& s, float (&gs)[4],
                                         float& lo) {
  const int t0 = h * 32;
  constexpr bool ragged = kRagged;
  float mx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t zw = (&zq[0].x)[k];
    float ya, yb;
    unpack2(add2(pack2(bf_lo(zw), bf_hi(zw)),
                 pack2(__uint_as_float(b[2 * k]), __uint_as_float(b[2 * k + 1]))),
            ya, yb);
    if (ragged) {
      if (t0 + 2 * k >= lim) ya = -INFINITY;
      if (t0 + 2 * k + 1 >= lim) yb = -INFINITY;
    }
    mx[k & 7] = fmax_nan(mx[k & 7], fmax_nan(ya, yb));
  }
#pragma unroll
  for (int w = 4; w > 0; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) mx[e] = fmax_nan(mx[e], mx[e + w]);
  const float cmax = mx[0] * p.sc.hi;
  if (!(cmax < 3.0e38f)) {  // NaN or +inf among the inputs
    s.bad = 1;
    return;
  }
  if (cmax <= -1.0e38f) return;  // no mass in these tokens
  const int cref = static_cast<int>(ceilf(fmaxf(cmax, -2.0e9f)));
  if (s.ref == INT_MIN) {
    s.ref = cref;
  } else if (cref > s.ref) {
    const int d = cref - s.ref;
    s.acc = d >= 63 ? 0 : (s.acc >> d);
    const float sc = __int_as_float((127 - min(d, 126)) << 23);  // 2^-d, exact
    lo *= sc;
#pragma unroll
    for (int g = 0; g < 4; ++g) gs[g] *= sc;
    s.ref = cref;
  }
  const float kmag = 12582912.0f - static_cast<float>(s.ref);  // 1.5 * 2^23 - ref, exact
  const float klo = 12582912.0f - 125.0f;
  const unsigned long long c12 = pack2(p.c12, p.c12), cr2 = pack2(p.crest, p.crest);
  const unsigned long long k2 = pack2(kmag, kmag);
#pragma unroll
  for (int gg = 0; gg < 2; ++gg) {
    unsigned long long w2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = gg * 8 + e;  // the token pair (t0 + 2k, t0 + 2k + 1)
      const uint32_t zw = (&zq[0].x)[k];
      w2[e] = pow2_split2(pack2(bf_lo(zw), bf_hi(zw)),
                          pack2(__uint_as_float(b[2 * k]), __uint_as_float(b[2 * k + 1])), c12,
                          cr2, k2, klo);
      if (ragged) {
        float wa, wb;
        unpack2(w2[e], wa, wb);
        w2[e] = pack2(t0 + 2 * k < lim ? wa : 0.f, t0 + 2 * k + 1 < lim ? wb : 0.f);
      }
    }
    float hi, glo;
    sum16(w2, hi, glo);
    gs[h * 2 + gg] = hi + glo;
    s.acc += fix40(hi);
    lo += glo;
  }
}

// One 64-token block of a request row: its two 32-column halves one after
// the other, the second loaded once the first is done (fewer live registers).
// b0 must hold the first half's load, already issued at column tcol.  Every
// lane of the warp calls this (the loads are warp-collective); `valid`
// lanes compute.
template <bool kGreedy>
__device__ __forceinline__ void epi_block(uint32_t (&b0)[32], uint32_t (&b1)[32], uint32_t tcol,
                                          const uint4 (&z0)[4], const uint4 (&z1)[4], int v0,
                                          int lim, bool valid, const TcParams& p, Part& s,
                                          float (&gs)[4]) {
  float lo = 0.f;
  tmem_wait_ld_regs(b0);
  if (valid) {
    if (kGreedy && lim < 64)
      epi_half_greedy<true>(b0, z0, 0, v0, lim, s);
    else if (kGreedy)
      epi_half_greedy<false>(b0, z0, 0, v0, lim, s);
    else if (lim < 64)
      epi_half<true>(b0, z0, 0, lim, p, s, gs, lo);
    else
      epi_half<false>(b0, z0, 0, lim, p, s, gs, lo);
  }
  __syncwarp();
  tmem_ld_32x32b_x32(tcol + 32, b1);
  tmem_wait_ld_regs(b1);
  if (valid) {
    if (kGreedy) {
      if (lim < 64)
        epi_half_greedy<true>(b1, z1, 1, v0, lim, s);
      else
        epi_half_greedy<false>(b1, z1, 1, v0, lim, s);
    } else {
      if (lim < 64)
        epi_half<true>(b1, z1, 1, lim, p, s, gs, lo);
      else
        epi_half<false>(b1, z1, 1, lim, p, s, gs, lo);
      s.acc += __float2ll_rn(lo * 1099511627776.0f);  // one 64-bit conversion a block
    }
  }
}

// Stores the four 16-token group sums gs of block jj (0, 1) of a 128-token
// partial, all eight in one unit: block 0's reference ref0 (the first block
// with mass).  Block 1's sums, in units of 2^ref, are scaled up by
// 2^(ref - ref0) (capped at 2^100: block 0 then weighs under 2^-100).
__device__ __forceinline__ void store_groups(float* dst, int jj, const float (&gs)[4], int ref,
                                             int& ref0) {
  float sc = 1.f;
  if (jj == 0) {
    ref0 = ref;
  } else if (ref0 != INT_MIN && ref > ref0) {
    sc = __int_as_float((127 + min(ref - ref0, 100)) << 23);
  }
  *reinterpret_cast<float4*>(dst + jj * 4) = make_float4(gs[0] * sc, gs[1] * sc, gs[2] * sc, gs[3] * sc);
}

// kGreedy: T = 0, its own instantiation (one kind of epilogue a kernel).
template <bool kBiasOut, bool kGreedy>
__global__ void __launch_bounds__(kThreads, 1)
    draft_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_w,
                          const __grid_constant__ CUtensorMap tm_z, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ int s_tok[BM];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + p.nK * kABytesPerChunk;
  uint8_t* sZ = sB + kStagesB * kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sZ + kZBoxes * kZBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars - 1);
  const uint32_t b_fullB = smem_u32(bars + 0);      // [3]
  const uint32_t b_emptyB = smem_u32(bars + 3);     // [3]
  const uint32_t b_fullZ = smem_u32(bars + 6);      // [2 halves][4 slots]
  const uint32_t b_emptyZ = smem_u32(bars + 14);    // [2 halves][4 slots]
  const uint32_t b_accFull = smem_u32(bars + 22);   // [2]
  const uint32_t b_accEmpty = smem_u32(bars + 24);  // [2]
  const uint32_t b_drain = smem_u32(bars + 26);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.y * BM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(b_fullB + 8 * i, 1);
      mbar_init(b_emptyB + 8 * i, 1);
    }
    for (int i = 0; i < 2 * kZBoxes; ++i) {
      mbar_init(b_fullZ + 8 * i, 1);
      mbar_init(b_emptyZ + 8 * i, 4);  // the four warps of one token half
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_accFull + 8 * i, 1);
      mbar_init(b_accEmpty + 8 * i, kEpiWarps);
    }
    mbar_init(b_drain, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpW && lane == 0) {
    tma_prefetch(&tm_w);
    if (!kBiasOut) tma_prefetch(&tm_z);
  }
  // A operand: the previous token's E row for each request of the tile, in
  // the 128-byte swizzled K-major layout (row m at m*128 bytes of its K
  // chunk, 16-byte granule g at position g ^ (m & 7)); rows past R are zero.
  // The tokens go to shared memory first, then every thread issues all of
  // its row loads before any store so the L2 latencies overlap.
  {
    if (threadIdx.x < BM) {
      const int n = r0 + threadIdx.x;
      int tok = -1;
      if (n < p.R && p.prev == nullptr) {
        tok = n * p.prev_stride;
      } else if (n < p.R) {
        tok = p.prev[(size_t)n * p.prev_stride];
        if (tok >= p.prev_limit || tok < -1) {
          set_flag(p.status, kFlagTokenRange);
          tok = -1;
        }
      }
      s_tok[threadIdx.x] = tok;
    }
    __syncthreads();
    const int per_row = p.nK * 8;
    constexpr int kPer = (BM * 32 + kThreads - 1) / kThreads;  // r <= 256: 32 granules a row
    uint4 val[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = threadIdx.x + i * kThreads;
      val[i] = make_uint4(0, 0, 0, 0);
      if (idx < BM * per_row) {
        const int m = idx / per_row, rem = idx - m * per_row;
        const int col = (rem >> 3) * BK + (rem & 7) * 8;
        const int tok = s_tok[m];
        if (tok >= 0 && col < p.r)
          val[i] = *reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.r + col);
      }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = threadIdx.x + i * kThreads;
      if (idx < BM * per_row) {
        const int m = idx / per_row, rem = idx - m * per_row;
        const int c = rem >> 3, g = rem & 7;
        *reinterpret_cast<uint4*>(sA + c * kABytesPerChunk + m * 128 + ((g ^ (m & 7)) << 4)) =
            val[i];
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpW) {
    // ---------------- Wt producer
    if (lane == 0) {
      // W is re-read at every draft position: keep it resident in L2
      const uint64_t pol = policy_evict_last();
      RingPos rb;
      for (int t = blockIdx.x; t < p.n_vt; t += gridDim.x) {
        for (int c = 0; c < p.nK; ++c, rb.next(kStagesB)) {
          wait_abortable(b_emptyB + 8 * rb.s, rb.ph ^ 1, &s_abort, p.status);
          mbar_arrive_expect_tx(b_fullB + 8 * rb.s, kBBytes);
          tma_load_2d_hint(smem_u32(sB + rb.s * kBBytes), &tm_w, b_fullB + 8 * rb.s, c * BK,
                           t * BN, pol);
        }
      }
    }
  } else if (warp == kWarpZ) {
    // ---------------- z producer
    if (!kBiasOut && lane == 0) {
      // each logit slice is read exactly once: do not let it displace W
      const uint64_t pol = policy_evict_first();
      uint32_t it = 0;
      ZRing zr;
      for (int t = blockIdx.x; t < p.n_vt; t += gridDim.x) {
        for (int j = 0; j < kZBoxes; ++j, ++it) {
          const int s = it % kZBoxes;
          zr.acquire(b_emptyZ, s, j >> 1, &s_abort, p.status);
          // the epilogue read this box through the generic proxy; order those
          // reads before the async-proxy (TMA) write that refills it
          fence_proxy_async_smem();
          const uint32_t fb = b_fullZ + 8 * ((j >> 1) * 4 + s);
          mbar_arrive_expect_tx(fb, kZBytes);
          tma_load_3d_hint(smem_u32(sZ + s * kZBytes), &tm_z, fb, t * BN + j * 64, p.k, r0, pol);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint64_t da0 = desc_kmajor_sw128(smem_u32(sA));
      const uint64_t db0 = desc_kmajor_sw128(smem_u32(sB));
      RingPos rb;
      uint32_t acc_it = 0;
      for (int t = blockIdx.x; t < p.n_vt; t += gridDim.x, ++acc_it) {
        const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
        wait_abortable(b_accEmpty + 8 * a, aph ^ 1, &s_abort, p.status);
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * BN;
        for (int c = 0; c < p.nK; ++c, rb.next(kStagesB)) {
          wait_abortable(b_fullB + 8 * rb.s, rb.ph, &s_abort, p.status);
          tc_fence_after();
          mma_chunk(d_tmem, da0 + ((uint32_t)c * (kABytesPerChunk >> 4)),
                    db0 + (rb.s * (kBBytes >> 4)), c != 0);
          mma_commit(b_emptyB + 8 * rb.s);
        }
        mma_commit(b_accFull + 8 * a);
      }
      // every MMA issued here completes before TMEM is released
      mma_commit(b_drain);
      if (!mbar_wait(b_drain, 0)) set_flag(p.status, kFlagTimeout);
    }
  } else {
    // ---------------- epilogue, warps 0-7
    const int quad = warp & 3, half = warp >> 2;
    const int m = quad * 32 + lane;  // request row of the tile = TMEM lane
    const int n = r0 + m;
    const bool valid = n < p.R;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t acc_it = 0, zit0 = 0, cpar = 0;
    for (int t = blockIdx.x; t < p.n_vt; t += gridDim.x, ++acc_it, zit0 += kZBoxes) {
      const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
      wait_abortable(b_accFull + 8 * a, aph, &s_abort, p.status);
      tc_fence_after();
      Part s{0, INT_MIN, 0, ArgMax{-INFINITY, 0x7fffffff}};
      int ref0 = INT_MIN;
      const size_t o = (size_t)n * p.n_parts + t * 2 + half;
      const bool own = !kBiasOut && valid && t * 2 + half < p.n_parts;
#pragma unroll 1
      for (int jj = 0; jj < 2; ++jj) {
        const int j = half * 2 + jj;  // z box (64 tokens) of this warp
        const int col = j * 64;
        const uint32_t tcol = tmem + lane_base + a * BN + col;
        const int v0 = t * BN + col;
        if (kBiasOut) {
          uint32_t b0[32], b1[32];
          __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
          tmem_ld_32x32b_x32(tcol, b0);
          tmem_ld_32x32b_x32(tcol + 32, b1);
          tmem_wait_ld_regs(b0, b1);
          if (valid) {
            float* dst = p.bias_out + (size_t)n * p.V;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              if (v0 + e + 4 <= p.V)
                *reinterpret_cast<uint4*>(dst + v0 + e) = make_uint4(b0[e], b0[e + 1], b0[e + 2], b0[e + 3]);
              if (v0 + 32 + e + 4 <= p.V)
                *reinterpret_cast<uint4*>(dst + v0 + 32 + e) =
                    make_uint4(b1[e], b1[e + 1], b1[e + 2], b1[e + 3]);
            }
          }
          continue;
        }
        uint32_t b0[32], b1[32];
        __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
        tmem_ld_32x32b_x32(tcol, b0);  // the first half, while the z box is awaited
        const uint32_t zs = (zit0 + j) % kZBoxes;
        wait_abortable(b_fullZ + 8 * (half * 4 + zs), (cpar >> zs) & 1u, &s_abort, p.status);
        cpar ^= 1u << zs;
        uint4 z0[4], z1[4];
        const uint8_t* zrow = sZ + zs * kZBytes + m * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          z0[q] = *reinterpret_cast<const uint4*>(zrow + ((q ^ (m & 7)) << 4));
          z1[q] = *reinterpret_cast<const uint4*>(zrow + (((q + 4) ^ (m & 7)) << 4));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(b_emptyZ + 8 * (half * 4 + zs));
        float gs[4] = {0.f, 0.f, 0.f, 0.f};
        epi_block<kGreedy>(b0, b1, tcol, z0, z1, v0, min(64, p.V - v0), valid, p, s, gs);
        if (own && !kGreedy) store_groups(p.sub + o * 8, jj, gs, s.ref, ref0);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_accEmpty + 8 * a);
      if (own) {
        if (s.bad) set_flag(p.status, kFlagNonFinite);
        if (kGreedy)
          reinterpret_cast<ArgMax*>(p.part)[o] = s.best;
        else
          p.part[o] = (s.ref == INT_MIN) ? 0.0 : fix_to_double(s.acc, s.ref - kFixRel);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- persistent

// All gamma draft positions in one cooperative launch.  Per position k:
//   epilogue warps gather A(k) (E rows of x_{k-1}), release the MMA warp,
//   run the partial pass over the CTA's tiles, grid barrier, run the finish
//   of the CTA's requests (scratch aliased on the A tile, idle by then), grid
//   barrier (none after the last position: nothing reads across CTAs after
//   it).  The Wt and z producers run ahead across positions through
//   their rings (neither operand depends on the drafted tokens), so their
//   loads overlap the finish and the barriers.  TMEM is allocated once.
// With `fuse` the launch also evaluates the confidence head and the
// scheduler, off the per-position path where it can: the hidden-state terms
// at position 0 while its first accumulator is computed, the head itself
// (c_k needs x_{k-1} only) at the last position while its first accumulator
// is computed, the candidates' ranks by the CTAs without a finish during the
// last finish, and the one-block cut by one CTA after the loop, once the
// ranking CTAs have signalled it (the other CTAs do not wait).
struct PersistParams {
  TcParams p;
  const __nv_bfloat16* z;
  const __nv_bfloat16* Wt;
  const int32_t* anchor;
  int32_t* tokens;
  double* q_lse;
  float* q_tok;
  const float* u;
  unsigned* grid_counter;  // [2], zeroed before the launch: grid barrier, ranking CTAs done
  int pair;                // R <= 64: two vocabulary tiles per accumulator
  __nv_bfloat16* stage;    // [R][r]: E rows of the tokens drawn at the last position
  int fuse;                // also the confidence head and the scheduler (f)
  DraftFuse f;
};

// Paired layout (R <= 64).  A 128-row accumulator holds two vocabulary tiles:
// rows 0-63 the requests against tile t1, rows 64-127 the same requests
// against tile t2.  The A operand lives in 8 KiB blocks of 64 swizzled rows,
// [0, E_0, 0, E_1, ..., E_{nK-1}, 0] (E_c = K-chunk c of the gathered E rows,
// 0 = zero rows): the descriptor starting at E_c reads [E_c; 0] and the one
// starting at the zero block before it reads [0; E_c], so one accumulator
// receives E W(t1) in its top half and E W(t2) in its bottom half from two
// K-passes, with no more MMA work than two unpaired tiles and every TMEM
// lane quadrant (hence every epilogue warp) holding live rows.
constexpr uint32_t kPairBlk = 64 * 128;  // 64 rows x 128 bytes
static_assert(sizeof(FinishScratch) <= kPairBlk, "finish scratch must fit one A block");
// two finish scratches (more requests than CTAs: unpaired layout) on A(0)
static_assert(2 * sizeof(FinishScratch) <= kABytesPerChunk, "two finish scratches must fit A(0)");
static_assert(sizeof(FinishScratch) % 16 == 0, "finish scratch alignment");

__host__ __device__ inline uint32_t persist_a_bytes(int nK, int pair) {
  return pair ? (uint32_t)(2 * nK + 1) * kPairBlk : (uint32_t)nK * kABytesPerChunk;
}
__host__ __device__ inline int persist_z_slots(int pair) { return pair ? 3 : kZBoxes; }

size_t persist_smem_bytes(int nK, int pair) {
  return 1024 + (size_t)persist_a_bytes(nK, pair) + kStagesB * kBBytes +
         (size_t)persist_z_slots(pair) * kZBytes + kBars * sizeof(uint64_t) + 16;
}

// Grid-wide barrier among the 256 epilogue threads of every CTA (bounded:
// gives up after about two seconds, setting the timeout flag).  The CTA
// barrier orders every thread's writes before thread 0's release-add, and
// thread 0's acquire-load of the full count orders the other CTAs' writes
// before everything after the second CTA barrier, so no full fence is needed.
__device__ __forceinline__ void grid_arrive_wait(unsigned* ctr, unsigned target,
                                                 volatile int* abort_flag, uint32_t* status,
                                                 uint64_t limit_ns = kGridLimitNs) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
  if (*abort_flag) return;
  const uint64_t t0 = globaltimer_ns();
  for (int spin = 1;; ++spin) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) break;
    if ((spin & 63) == 0 && globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      set_flag(status, kFlagTimeout);
      break;
    }
  }
}

__device__ __forceinline__ void grid_sync(unsigned* ctr, unsigned target, volatile int* abort_flag,
                                          uint32_t* status) {
  NamedSync<2, 256>::sync();
  if (threadIdx.x == 0) grid_arrive_wait(ctr, target, abort_flag, status);
  NamedSync<2, 256>::sync();
}

// Diagnostic of the bounded waits above: one CTA waits on an mbarrier that
// nothing arrives on, then on a grid-barrier target that only it counts
// towards, each with a short limit.  Both waits must give up, set the
// timeout bit and let the kernel return; the counter is put back to zero.
// out[0] = 1 if the mbarrier wait reported success (it must not),
// out[1] = the abort flag after the grid wait (it must be set).
__global__ void wait_check_kernel(uint64_t limit_ns, unsigned* ctr, uint32_t* status, int* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = wait_abortable(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    abort_flag = 0;
    grid_arrive_wait(ctr, 2u, &abort_flag, status, limit_ns);
    out[0] = ok ? 1 : 0;
    out[1] = abort_flag;
    atomicExch(ctr, 0u);
  }
}

// Confidence head at the last draft position (c_k needs x_{k-1} only, and
// every such token is drawn by then), for the CTA's own requests, by the
// epilogue warps while the position's first accumulator is computed; the
// lane partials of w_h . h were stored at position 0 by the same threads.
// Same per-warp arithmetic as the confidence kernel.
__device__ __noinline__ void fused_confidence(const PersistParams& pp, int cta, int n_ctas,
                                              float* s_conf) {
  const TcParams& p = pp.p;
  const DraftFuse& f = pp.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int nn = cta; nn < p.R; nn += n_ctas) {
    for (int kk = warp; kk < p.gamma; kk += 8) {
      const size_t idx = (size_t)nn * p.gamma + kk;
      float c;
      if (f.c_in != nullptr) {
        c = f.c_in[idx];
      } else {
        int prev = kk == 0 ? pp.anchor[nn] : pp.tokens[idx - 1];
        if (prev >= p.V || prev < -1) {
          if (lane == 0) set_flag(p.status, kFlagTokenRange);
          prev = -1;
        }
        const uint4 eq = conf::conf_load_e1(static_cast<const __nv_bfloat16*>(f.E1), prev, p.r);
        c = conf::conf_sigma(f.hpart[idx * 32 + lane], eq, prev, p.r, f.w + f.d, f.sts[kk]);
      }
      if (lane == 0) {
        if (!isfinite(c)) set_flag(p.status, kFlagNonFinite);
        s_conf[kk] = c;
        f.c_out[idx] = c;
      }
    }
    NamedSync<3, 256>::sync();
    if ((int)threadIdx.x < p.gamma) {
      // a_j = prod_{i <= j} c_i, each thread its own prefix
      float run = 1.0f;
      for (int j = 0; j <= (int)threadIdx.x; ++j) run = run * s_conf[j];
      f.a_out[(size_t)nn * p.gamma + threadIdx.x] = run;
    }
    NamedSync<3, 256>::sync();
  }
}

// Ranks of the scheduler's candidates, by the epilogue warps of the CTAs
// without a finish at the last draft position (every CTA when each has one),
// after that position's grid barrier (the survival values were written
// before it); the cut waits for their signal, nobody else does.  Each
// candidate's rank counts the i < e whose value is >= its own and the i > e
// whose value is above it (the cleaned values are >= +0, so their bits order
// like the values); a warp per candidate.  `ab` points into the Wt ring,
// idle after the last MMA: the values' bits, then their fixed-point images.
__device__ __noinline__ void fused_rank(const PersistParams& pp, int cta, int n_ctas,
                                        uint32_t* ab) {
  const TcParams& p = pp.p;
  const DraftFuse& f = pp.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.R * p.gamma;
  const int w0 = p.R < n_ctas ? p.R : 0, nwk = n_ctas - w0;  // worker CTAs
  if (cta < w0) return;
  long long* fx = reinterpret_cast<long long*>(ab + ((N + 1) & ~1));  // 8-byte aligned
  for (int e = threadIdx.x; e < N; e += 256) {
    const float v = sched::clean_a(__ldcg(f.a_out + e), p.status) + 0.0f;
    ab[e] = __float_as_uint(v);
    fx[e] = sched::to_fixed(v);
  }
  NamedSync<3, 256>::sync();
  // with its rank, each candidate's exact prefix S_rank (the sum of the
  // values ranked before it) and Theta_rank's key; the last-ranked one also
  // gives S_N and Theta_N
  for (int e = (cta - w0) + warp * nwk; e < N; e += 8 * nwk) {
    const uint32_t be = ab[e];
    int cnt = 0;
    long long sacc = 0;
    for (int i = lane; i < N; i += 32) {
      const uint32_t x = ab[i];
      const bool before = i < e ? (x >= be) : (i > e && x > be);
      cnt += before ? 1 : 0;
      sacc += before ? fx[i] : 0ll;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    const long long S = warp_sum_nonneg_ll(sacc);
    if (lane == 0) {
      f.rank[e] = cnt;
      f.spre[cnt] = S;
      if (cnt <= f.imax) f.tkey[cnt] = sched::theta_key_of(p.R, cnt, S, f.sps, p.status);
      if (cnt == N - 1) {
        f.spre[N] = S + fx[e];
        if (N <= f.imax) f.tkey[N] = sched::theta_key_of(p.R, N, S + fx[e], f.sps, p.status);
      }
    }
  }
}

// The scheduler's one-block cut, by one CTA after the last grid barrier
// (every rank written), every thread of the CTA; `buf` is the dynamic shared
// memory, idle by then.
__device__ __noinline__ void fused_cut(const PersistParams& pp, uint8_t* buf, int n_ctas,
                                       volatile int* s_abort) {
  const TcParams& p = pp.p;
  const DraftFuse& f = pp.f;
  const int N = p.R * p.gamma;
  // every ranking CTA has published its ranks (bounded wait, about 2 s)
  if (threadIdx.x == 0) {
    const unsigned want = (unsigned)(n_ctas - (p.R < n_ctas ? p.R : 0));
    const uint64_t t0 = globaltimer_ns();
    for (int spin = 1;; ++spin) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(pp.grid_counter + 1)
                   : "memory");
      if (v >= want) break;
      if ((spin & 63) == 0 && globaltimer_ns() - t0 > 2000000000ull) {
        *s_abort = 1;
        set_flag(p.status, kFlagTimeout);
        break;
      }
    }
  }
  __syncthreads();
  if (*s_abort) return;
  int32_t* rk = reinterpret_cast<int32_t*>(buf);
  for (int e = threadIdx.x; e < N; e += blockDim.x) rk[e] = __ldcg(f.rank + e);
  __syncthreads();
  sched::schedule_cut_keys(p.R, p.gamma, f.imax, f.early_stop, f.tkey, f.spre, rk, f.ell,
                           f.row_off, f.B_out, f.E_out);
}

// kGroups: finishes a CTA runs at once (8 / kGroups warps each) when it has
// many requests to finish; separate instantiations, so that the grouped
// finishes' registers do not weigh on the epilogue of every launch.
// kGreedy: T = 0 (argmax draws), its own instantiation for the same reason.
template <int kGroups, bool kGreedy>
__global__ void __launch_bounds__(kThreads, 1)
    draft_persistent_kernel(const __grid_constant__ CUtensorMap tm_w,
                            const __grid_constant__ CUtensorMap tm_z,
                            const __grid_constant__ CUtensorMap tm_a, const PersistParams pp) {
  const TcParams& p = pp.p;
  constexpr int greedy = kGreedy ? 1 : 0;  // p.greedy
  const bool pair = pp.pair != 0;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ int s_tok[BM];
  __shared__ float s_conf[kMaxGamma];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + persist_a_bytes(p.nK, pp.pair);
  uint8_t* sZ = sB + kStagesB * kBBytes;
  const int nzs = persist_z_slots(pp.pair);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sZ + nzs * kZBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars - 1);
  const uint32_t b_fullB = smem_u32(bars + 0);
  const uint32_t b_emptyB = smem_u32(bars + 3);
  const uint32_t b_fullZ = smem_u32(bars + 6);    // [2 halves][4 slots]
  const uint32_t b_emptyZ = smem_u32(bars + 14);  // [2 halves][4 slots]
  const uint32_t b_accFull = smem_u32(bars + 22);
  const uint32_t b_accEmpty = smem_u32(bars + 24);
  const uint32_t b_drain = smem_u32(bars + 26);
  const uint32_t b_aFull = smem_u32(bars + 27);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.y * BM;
  const unsigned n_ctas = gridDim.x * gridDim.y;
  const int cta = blockIdx.y * gridDim.x + blockIdx.x;
  // work units: one tile, or (paired) tiles 2u and 2u + 1
  const int n_units = pair ? (p.n_vt + 1) / 2 : p.n_vt;
  const int passes = pair ? 2 : 1;  // K passes per unit (one per tile)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(b_fullB + 8 * i, 1);
      mbar_init(b_emptyB + 8 * i, 1);
    }
    for (int i = 0; i < 2 * kZBoxes; ++i) {
      mbar_init(b_fullZ + 8 * i, 1);
      mbar_init(b_emptyZ + 8 * i, 4);  // the four warps of one token half
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_accFull + 8 * i, 1);
      mbar_init(b_accEmpty + 8 * i, kEpiWarps);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_aFull, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpW && lane == 0) {
    tma_prefetch(&tm_w);
    tma_prefetch(&tm_z);
    tma_prefetch(&tm_a);
  }
  if (pair && threadIdx.x < 256) {
    // the zero blocks of the paired A operand, written once
    for (int c = 0; c <= p.nK; ++c) {
      uint4* blk = reinterpret_cast<uint4*>(sA + (size_t)(2 * c) * kPairBlk);
      for (int i = threadIdx.x; i < (int)(kPairBlk / 16); i += 256) blk[i] = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpW) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      // W is not in L2 at the first position: ask for the tiles of this
      // CTA's later units now, so that they arrive while the first unit's
      // tiles stream through the ring (32 KiB prefetches of whole rows)
      for (int u = blockIdx.x + gridDim.x; u < n_units; u += gridDim.x)
        for (int pass = 0; pass < passes; ++pass) {
          const int t = pair ? 2 * u + pass : u;
          if (t >= p.n_vt) continue;
          const char* base = reinterpret_cast<const char*>(pp.Wt) + (size_t)t * BN * p.r * 2;
          const uint32_t bytes = (uint32_t)(min(BN, p.V - t * BN) * p.r * 2);
          for (uint32_t o = 0; o < bytes; o += 32768)
            prefetch_l2_bulk(base + o, min(32768u, bytes - o));
        }
      RingPos rb;
      for (int k = 0; k < p.gamma; ++k)
        for (int u = blockIdx.x; u < n_units; u += gridDim.x)
          for (int pass = 0; pass < passes; ++pass)
            for (int c = 0; c < p.nK; ++c, rb.next(kStagesB)) {
              const int t = pair ? 2 * u + pass : u;
              wait_abortable(b_emptyB + 8 * rb.s, rb.ph ^ 1, &s_abort, p.status);
              if (t < p.n_vt) {
                mbar_arrive_expect_tx(b_fullB + 8 * rb.s, kBBytes);
                tma_load_2d_hint(smem_u32(sB + rb.s * kBBytes), &tm_w, b_fullB + 8 * rb.s, c * BK,
                                 t * BN, pol);
              } else {
                // the odd last unit's second tile lies past V: no load, its
                // accumulator rows are never read
                mbar_arrive(b_fullB + 8 * rb.s);
              }
            }
    }
  } else if (warp == kWarpZ) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t it = 0;
      ZRing zr;
      for (int k = 0; k < p.gamma; ++k)
        for (int u = blockIdx.x; u < n_units; u += gridDim.x)
          for (int j = 0; j < kZBoxes; ++j, ++it) {
            const int s = it % nzs;
            zr.acquire(b_emptyZ, s, j >> 1, &s_abort, p.status);
            const uint32_t fb = b_fullZ + 8 * ((j >> 1) * 4 + s);
            fence_proxy_async_smem();  // generic reads of the slot before the TMA refill
            const uint32_t dst = smem_u32(sZ + s * kZBytes);
            if (pair) {
              // rows 0-63: the requests' logits of tile 2u; rows 64-127: of tile 2u + 1
              const bool second = 2 * u + 1 < p.n_vt;
              mbar_arrive_expect_tx(fb, second ? kZBytes : kZBytes / 2);
              tma_load_3d_hint(dst, &tm_z, fb, (2 * u) * BN + j * 64, k, 0, pol);
              if (second)
                tma_load_3d_hint(dst + kZBytes / 2, &tm_z, fb, (2 * u + 1) * BN + j * 64, k, 0,
                                 pol);
            } else {
              mbar_arrive_expect_tx(fb, kZBytes);
              tma_load_3d_hint(dst, &tm_z, fb, u * BN + j * 64, k, r0, pol);
            }
          }
    }
  } else if (warp == kWarpMma) {
    const uint64_t da0 = desc_kmajor_sw128(smem_u32(sA));
    const uint64_t db0 = desc_kmajor_sw128(smem_u32(sB));
    // A chunk c of pass 0 / pass 1, in 16-byte descriptor units: paired, the
    // first pass reads [E_c; 0] (block 2c + 1) against tile 2u and the
    // second [0; E_c] (block 2c) against tile 2u + 1
    const uint32_t a_step = (pair ? 2 * kPairBlk : kABytesPerChunk) >> 4;
    const uint32_t a_pass0 = pair ? kPairBlk >> 4 : 0;
    RingPos rb;
    uint32_t acc_it = 0;
    for (int k = 0; k < p.gamma; ++k) {
      NamedSync<1, 288>::sync();  // A(k) is in shared memory, or on its way by TMA
      if (lane == 0) {
        if (k > 0) wait_abortable(b_aFull, (k - 1) & 1, &s_abort, p.status);
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++acc_it) {
          const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
          wait_abortable(b_accEmpty + 8 * a, aph ^ 1, &s_abort, p.status);
          tc_fence_after();
          const uint32_t d_tmem = tmem + a * BN;
          for (int pass = 0; pass < passes; ++pass) {
            uint64_t da = da0 + (pass == 0 ? a_pass0 : 0);
            for (int c = 0; c < p.nK; ++c, da += a_step, rb.next(kStagesB)) {
              wait_abortable(b_fullB + 8 * rb.s, rb.ph, &s_abort, p.status);
              tc_fence_after();
              mma_chunk(d_tmem, da, db0 + rb.s * (kBBytes >> 4), (pass | c) != 0);
              mma_commit(b_emptyB + 8 * rb.s);
            }
          }
          mma_commit(b_accFull + 8 * a);
        }
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(b_drain);
      if (!mbar_wait(b_drain, 0)) set_flag(p.status, kFlagTimeout);
    }
  } else {
    // ---------------- epilogue warps 0-7 (also the gather and the finish)
    const int quad = warp & 3, half = warp >> 2;
    const int m = quad * 32 + lane;  // TMEM lane = row of the z slot
    // paired: lanes 0-63 are requests 0-63 on tile 2u, lanes 64-127 on 2u + 1
    const int n = pair ? (m & 63) : r0 + m;
    const int tsub = pair ? (m >> 6) : 0;
    const bool valid = n < p.R;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int rows = pair ? 64 : BM;  // gathered A rows
    uint32_t acc_it = 0, zit = 0, epoch = 0, cpar = 0;
    FinishScratch& fs = *reinterpret_cast<FinishScratch*>(pair ? sA + kPairBlk : sA);
    for (int k = 0; k < p.gamma; ++k) {
      const int32_t* prev = k == 0 ? pp.anchor : pp.tokens + (k - 1);
      const int stride = k == 0 ? 1 : p.gamma;
      if (k > 0) {
        // A(k) = the E rows the finishes staged at position k - 1: four TMA
        // boxes straight into the swizzled A blocks
        if (threadIdx.x == 0) {
          fence_proxy_async_all();
          const uint32_t box = pair ? kPairBlk : kABytesPerChunk;
          mbar_arrive_expect_tx(b_aFull, box * p.nK);
          for (int c = 0; c < p.nK; ++c)
            tma_load_2d(smem_u32(pair ? sA + (size_t)(2 * c + 1) * kPairBlk
                                      : sA + (size_t)c * kABytesPerChunk),
                        &tm_a, b_aFull, c * BK, pair ? 0 : r0);
        }
      } else {
      // gather A(0): the rows of E at the anchors
      if (threadIdx.x < rows) {
        const int nn = (pair ? 0 : r0) + threadIdx.x;
        int tok = -1;
        if (nn < p.R) {
          tok = __ldcg(prev + (size_t)nn * stride);
          if (tok >= p.V || tok < -1) {
            set_flag(p.status, kFlagTokenRange);
            tok = -1;
          }
        }
        s_tok[threadIdx.x] = tok;
      }
      NamedSync<3, 256>::sync();
      {
        const int per_row = p.nK * 8;
        constexpr int kPer = BM * 32 / 256;
        uint4 val[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = threadIdx.x + i * 256;
          val[i] = make_uint4(0, 0, 0, 0);
          if (idx < rows * per_row) {
            const int mm = idx / per_row, rem = idx - mm * per_row;
            const int col = (rem >> 3) * BK + (rem & 7) * 8;
            const int tok = s_tok[mm];
            if (tok >= 0 && col < p.r)
              val[i] = *reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.r + col);
          }
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = threadIdx.x + i * 256;
          if (idx < rows * per_row) {
            const int mm = idx / per_row, rem = idx - mm * per_row;
            const int c = rem >> 3, g = rem & 7;
            uint8_t* blk = pair ? sA + (size_t)(2 * c + 1) * kPairBlk : sA + c * kABytesPerChunk;
            *reinterpret_cast<uint4*>(blk + mm * 128 + ((g ^ (mm & 7)) << 4)) = val[i];
          }
        }
      }
      }
      fence_proxy_async_smem();
      NamedSync<1, 288>::sync();  // release the MMA warp
      if (k == 0 && pp.fuse && pp.f.c_in == nullptr) {
        // the confidence head's hidden-state term does not depend on the
        // draft: its lane partials while the first accumulator is computed
        for (int nn = cta; nn < p.R; nn += n_ctas)
          for (int kk = warp; kk < p.gamma; kk += 8) {
            const size_t idx = (size_t)nn * p.gamma + kk;
            uint4 hq[conf::kHLoads];
            conf::conf_load_h(static_cast<const __nv_bfloat16*>(pp.f.h) + idx * pp.f.d, pp.f.d,
                              hq);
            pp.f.hpart[idx * 32 + lane] = conf::conf_h_lane(hq, pp.f.w, pp.f.d);
          }
      }
      // c_k depends on x_{k-1} only: every confidence is known once the
      // last position's A is; evaluate the head while its first accumulator
      // is computed (written before this position's first grid barrier)
      if (k == p.gamma - 1 && pp.fuse) fused_confidence(pp, cta, (int)n_ctas, s_conf);
      // partial pass over this CTA's units
      for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++acc_it, zit += kZBoxes) {
        const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
        const int t = pair ? 2 * u + tsub : u;
        wait_abortable(b_accFull + 8 * a, aph, &s_abort, p.status);
        tc_fence_after();
        Part s{0, INT_MIN, 0, ArgMax{-INFINITY, 0x7fffffff}};
        int ref0 = INT_MIN;
        const size_t o = (size_t)n * p.n_parts + t * 2 + half;
        const bool own = valid && t * 2 + half < p.n_parts;
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
          const int j = half * 2 + jj;
          const int col = j * 64;
          const uint32_t tcol = tmem + lane_base + a * BN + col;
          uint32_t b0[32], b1[32];
          __syncwarp();
          tmem_ld_32x32b_x32(tcol, b0);  // the first half, while the z box is awaited
          const int v0 = t * BN + col;
          const uint32_t zs = (zit + j) % nzs;
          wait_abortable(b_fullZ + 8 * (half * 4 + zs), (cpar >> zs) & 1u, &s_abort, p.status);
          cpar ^= 1u << zs;
          uint4 z0[4], z1[4];
          const uint8_t* zrow = sZ + zs * kZBytes + m * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            z0[q] = *reinterpret_cast<const uint4*>(zrow + ((q ^ (m & 7)) << 4));
            z1[q] = *reinterpret_cast<const uint4*>(zrow + (((q + 4) ^ (m & 7)) << 4));
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(b_emptyZ + 8 * (half * 4 + zs));
          float gs[4] = {0.f, 0.f, 0.f, 0.f};
          epi_block<kGreedy>(b0, b1, tcol, z0, z1, v0, min(64, p.V - v0), valid, p, s, gs);
          if (own && !greedy) store_groups(p.sub + o * 8, jj, gs, s.ref, ref0);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_accEmpty + 8 * a);
        if (own) {
          if (s.bad) set_flag(p.status, kFlagNonFinite);
          if (greedy)
            reinterpret_cast<ArgMax*>(p.part)[o] = s.best;
          else
            p.part[o] = (s.ref == INT_MIN) ? 0.0 : fix_to_double(s.acc, s.ref - kFixRel);
        }
      }
      grid_sync(pp.grid_counter, (++epoch) * n_ctas, &s_abort, p.status);
      // finish of this CTA's requests; scratch on an A block (its MMAs are
      // done: order their async-proxy reads before these generic writes)
      fence_proxy_async_smem();
      const BiasSrc b{nullptr, p.E, pp.Wt, prev, stride, p.r};
      if constexpr (kGroups > 1) {
        // many requests a CTA: kGroups finishes at once (group g on warps
        // g * 8 / kGroups .., requests cta + g n_ctas, cta + (g + kGroups)
        // n_ctas, ...), each on its own scratch and named barrier
        constexpr int kNW = 8 / kGroups;
        const int grp = warp / kNW;
        FinishScratch& fg = (&fs)[grp];
        for (int nn = cta + grp * (int)n_ctas; nn < p.R; nn += kGroups * (int)n_ctas)
          finish_request<__nv_bfloat16, kHalf, GroupSync<4, kNW>, true>(
              fg, nn, p.V, p.gamma, k, p.n_parts, pp.z, b, p.sc, greedy, p.part, pp.u,
              pp.tokens, pp.q_lse, pp.q_tok, p.status, k + 1 < p.gamma ? pp.stage : nullptr,
              p.sub);
        NamedSync<3, 256>::sync();  // both groups done (the log pass reads their q_lse)
      } else {
        for (int nn = cta; nn < p.R; nn += n_ctas)
          finish_request<__nv_bfloat16, kHalf, NamedSync<3, 256>, true>(
              fs, nn, p.V, p.gamma, k, p.n_parts, pp.z, b, p.sc, greedy, p.part, pp.u,
              pp.tokens, pp.q_lse, pp.q_tok, p.status, k + 1 < p.gamma ? pp.stage : nullptr,
              p.sub);
      }
      if (k + 1 < p.gamma) {
        // the finish scratch (generic) is overwritten by the next A's TMA;
        // every CTA needs every staged row before it loads the next A
        fence_proxy_async_smem();
        grid_sync(pp.grid_counter, (++epoch) * n_ctas, &s_abort, p.status);
      } else if (pp.fuse && !s_abort) {
        // after the last position only the cut waits, for the ranks: the
        // ranking CTAs signal it (release) and nobody waits for the finishes
        fused_rank(pp, cta, (int)n_ctas, reinterpret_cast<uint32_t*>(sB));
        NamedSync<3, 256>::sync();
        if (threadIdx.x == 0 && cta >= (p.R < (int)n_ctas ? p.R : 0))
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(pp.grid_counter + 1)
                       : "memory");
      }
    }
    // The finishes left each q_lse entry holding its normaliser; take the
    // logarithms here, off the per-position path (same CTA, same requests).
    if (!greedy) {
      const int mine = p.R > cta ? (p.R - cta + (int)n_ctas - 1) / (int)n_ctas : 0;
      for (int i = threadIdx.x; i < mine * p.gamma; i += 256) {
        const size_t o = (size_t)(cta + (i / p.gamma) * (int)n_ctas) * p.gamma + i % p.gamma;
        const double tot = pp.q_lse[o];
        pp.q_lse[o] = (double)dbl_log(tot);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
  // the cut on a CTA without requests when there is one (no logarithm pass)
  if (pp.fuse && cta == (p.R < (int)n_ctas ? (int)n_ctas - 1 : 0) && !s_abort)
    fused_cut(pp, smem, (int)n_ctas, &s_abort);
}

// ---------------------------------------------------------------- final draw

// Final draw of the verification (the residual max(0, p - q) after a
// rejection, p itself for the bonus token): per (request, 128-token half
// tile) the exact fixed-point sums of both, in units of 2^-60 of the
// normalised probabilities.  The draft logits at the rejected position need
// the Markov bias of the token before it, which the tensor cores produce in
// TMEM as in the draft (with the paired accumulator layout when R <= 64).
// The z and target rows sit at request-dependent positions: the producer
// warp copies them 32 tokens (64 bytes) at a time with cp.async, four lanes
// per row so that every 16-byte copy of an instruction falls in one of eight
// row segments, into 64-byte slot rows whose 16-byte granules are permuted
// by row so that the epilogue's 16-byte reads across 32 rows hit distinct
// banks.
struct FinalParams {
  int R, V, r, nK, n_vt, n_halves, gamma, pair;
  int prev_limit;  // rows of E
  long long n_rows;
  ScalePair sc;
  float c12, crest;  // log2(e)/T = c12 + crest, c12 with 12 significant bits
  const __nv_bfloat16* E;       // Markov table, or the RNN states [R][gamma][r]
  const __nv_bfloat16* z;       // [R][gamma][V]
  const __nv_bfloat16* target;  // [n_rows][V]
  const int32_t* prev;          // [R] bias row of the rejected position (row of E), -1 none
  const VerifyState* vstate;    // [R]
  long long* fin_part;          // [R][n_halves][2]: residual, p
  uint32_t* status;
};

constexpr int kFinSteps = BN / 32;            // 32-token blocks per tile
constexpr uint32_t kRowPart = BM * 64;         // one tensor's 128 rows of 64 bytes
constexpr uint32_t kRowSlot = 2 * kRowPart;    // z rows + target rows of one block
constexpr int kFinSlots = 3;

size_t final_smem_bytes(int nK, int pair) {
  const size_t a = pair ? (size_t)(2 * nK + 1) * kPairBlk : (size_t)nK * kABytesPerChunk;
  return 1024 + a + (size_t)kStagesB * kBBytes + (size_t)kFinSlots * kRowSlot +
         kBars * sizeof(uint64_t) + 16;
}

// byte offset of 16-byte granule g (0..3) of slot row m
__device__ __forceinline__ uint32_t row_granule(int m, int g) {
  return (uint32_t)m * 64 + ((uint32_t)(g ^ ((m >> 1) & 3)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// The same, issued only when `on` is nonzero (a predicate inside the
// instruction, so that a run of them carries no branch).
__device__ __forceinline__ void cp_async16_if(uint32_t dst, const void* src, uint32_t on) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t"
      "@q cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(dst),
      "l"(src), "r"(on)
      : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (counts as one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// The final draw's weights for 32 tokens of one request row (accumulator
// load b = the Markov bias of the rejected position, z and target words):
// p = 2^(t c + ep) (hi + lo) with 1/Sp = (hi + lo) 2^ep (so p <= 2), and the
// residual max(0, p - q), q = 2^((z + b) c + eq) (iq.hi + iq.lo), or p itself
// for a bonus draw.  The exponents are split as in the draft epilogue (no
// fp32 rounding of t c or of z + b at the magnitude of the logits) and the
// 16-token sums are TwoSum trees; acc holds (residual hi, lo, p hi, lo).
// A NaN group is left out (the pick's recompute flags it).
// kRagged: the block holds the vocabulary's end (tokens at or past lim
// weigh 0); kQ: some lane of the warp draws from a residual (else no q is
// formed).  Template parameters, so that the unrolled pairs carry no branch.
template <bool kRagged, bool kQ>
__device__ __forceinline__ void fin_block(const uint32_t (&b)[32], const uint4 (&zq)[4],
                                          const uint4 (&tq)[4], int lim, bool resid, float c12,
                                          float cf, float crest, InvPair ip, InvPair iq,
                                          float (&acc)[4]) {
  if (ip.hi == 0.f) return;  // no target normaliser: no mass
  const bool qlive = resid && iq.hi != 0.f;
  const unsigned long long c2 = pack2(c12, c12), cr2 = pack2(crest, crest);
  const unsigned long long cf2 = pack2(cf, cf);
  const float kp = 12582912.0f + (float)ip.e, kq = 12582912.0f + (float)iq.e;
  const unsigned long long kp2 = pack2(kp, kp), kq2 = pack2(kq, kq);
  const float klo = 12582912.0f - 125.0f;
  const unsigned long long iph = pack2(ip.hi, ip.hi), ipl = pack2(ip.lo, ip.lo);
  const unsigned long long iqh = pack2(iq.hi, iq.hi), iql = pack2(iq.lo, iq.lo);
#pragma unroll
  for (int gg = 0; gg < 2; ++gg) {
    unsigned long long p2[8], r2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = gg * 8 + e;  // the token pair (2k, 2k + 1)
      const uint32_t tw = (&tq[0].x)[k];
      const unsigned long long wp =
          pow2_split2_nb(pack2(bf_lo(tw), bf_hi(tw)), c2, cr2, kp2, klo);
      p2[e] = fma2(wp, iph, mul2(wp, ipl));
      float pa, pb;
      unpack2(p2[e], pa, pb);
      if (kRagged) {
        pa = 2 * k < lim ? pa : 0.f;
        pb = 2 * k + 1 < lim ? pb : 0.f;
        p2[e] = pack2(pa, pb);
      }
      if (kQ) {
        // q for every lane of a warp with a residual (finite: a bonus lane's
        // z and bias are zero), the residual taken by select, so the
        // unrolled pairs have no branch
        const uint32_t zw = (&zq[0].x)[k];
        const unsigned long long wq =
            pow2_split2_cf(pack2(bf_lo(zw), bf_hi(zw)),
                           pack2(__uint_as_float(b[2 * k]), __uint_as_float(b[2 * k + 1])), c2,
                           cf2, cr2, kq2, klo);
        float da, db;  // p - q
        unpack2(sub2(p2[e], fma2(wq, iqh, mul2(wq, iql))), da, db);
        r2[e] = pack2(qlive ? fmaxf(0.0f, da) : pa, qlive ? fmaxf(0.0f, db) : pb);
      } else {
        r2[e] = p2[e];
      }
    }
    float ph, pl, rh, rl;
    sum16(p2, ph, pl);
    sum16(r2, rh, rl);
    // a NaN group is left out, by select (no branch between the groups)
    const bool okp = ph == ph, okr = rh == rh;
    add_pair(acc[2], acc[3], okp ? ph : 0.f, okp ? pl : 0.f);
    add_pair(acc[0], acc[1], okr ? rh : 0.f, okr ? rl : 0.f);
  }
}

// round(x * 2^60) for 0 <= x < 8, from the float's bits (exact once
// x * 2^60 >= 2^23; below, the bits under 2^-60 are dropped).
__device__ __forceinline__ long long fix60(float x) {
  const uint32_t b = __float_as_uint(x);
  const int e = (int)(b >> 23);
  const unsigned long long m = (b & 0x7fffffu) | (e ? 0x800000u : 0u);
  const int sh = e - 90;  // x * 2^60 = m * 2^(e - 150 + 60)
  return (long long)(sh >= 0 ? m << sh : (sh > -24 ? m >> -sh : 0ull));
}


__global__ void __launch_bounds__(kThreads, 1)
    final_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const FinalParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ int s_tok[BM];
  const bool pair = p.pair != 0;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + (pair ? (size_t)(2 * p.nK + 1) * kPairBlk : (size_t)p.nK * kABytesPerChunk);
  uint8_t* sZ = sB + kStagesB * kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sZ + kFinSlots * kRowSlot);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars - 1);
  const uint32_t b_fullB = smem_u32(bars + 0);
  const uint32_t b_emptyB = smem_u32(bars + 3);
  const uint32_t b_fullZ = smem_u32(bars + 6);    // [2 halves][4 slots]
  const uint32_t b_emptyZ = smem_u32(bars + 14);  // [2 halves][4 slots]
  const uint32_t b_accFull = smem_u32(bars + 22);
  const uint32_t b_accEmpty = smem_u32(bars + 24);
  const uint32_t b_drain = smem_u32(bars + 26);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.y * BM;
  // units: one tile, or (paired) tiles 2u and 2u + 1
  const int n_units = pair ? (p.n_vt + 1) / 2 : p.n_vt;
  const int passes = pair ? 2 : 1;  // K passes per unit (one per tile)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(b_fullB + 8 * i, 1);
      mbar_init(b_emptyB + 8 * i, 1);
    }
    for (int i = 0; i < 2 * kZBoxes; ++i) {
      mbar_init(b_fullZ + 8 * i, 32);  // every copier lane's arrival
      mbar_init(b_emptyZ + 8 * i, 4);  // the four warps of one token half
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_accFull + 8 * i, 1);
      mbar_init(b_accEmpty + 8 * i, kEpiWarps);
    }
    mbar_init(b_drain, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpW && lane == 0) tma_prefetch(&tm_w);
  if (pair && threadIdx.x < 256) {
    // the zero blocks of the paired A operand depend on nothing: before the wait
    for (int c = 0; c <= p.nK; ++c) {
      uint4* blk = reinterpret_cast<uint4*>(sA + (size_t)(2 * c) * kPairBlk);
      for (int i = threadIdx.x; i < (int)(kPairBlk / 16); i += 256) blk[i] = make_uint4(0, 0, 0, 0);
    }
  }
  grid_dependency_wait();  // the verification state and previous tokens
  // A operand: E rows of the token before each request's rejected position
  {
    const int rows = pair ? 64 : BM;
    if (threadIdx.x < rows) {
      const int n = r0 + threadIdx.x;
      int tok = -1;
      if (n < p.R) {
        tok = p.prev[n];
        if (tok >= p.prev_limit || tok < -1) {
          set_flag(p.status, kFlagTokenRange);
          tok = -1;
        }
      }
      s_tok[threadIdx.x] = tok;
    }
    __syncthreads();
    const int per_row = p.nK * 8;
    constexpr int kPer = (BM * 32 + kThreads - 1) / kThreads;
    uint4 val[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = threadIdx.x + i * kThreads;
      val[i] = make_uint4(0, 0, 0, 0);
      if (idx < rows * per_row) {
        const int m = idx / per_row, rem = idx - m * per_row;
        const int col = (rem >> 3) * BK + (rem & 7) * 8;
        const int tok = s_tok[m];
        if (tok >= 0 && col < p.r)
          val[i] = *reinterpret_cast<const uint4*>(p.E + (size_t)tok * p.r + col);
      }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = threadIdx.x + i * kThreads;
      if (idx < rows * per_row) {
        const int m = idx / per_row, rem = idx - m * per_row;
        const int c = rem >> 3, g = rem & 7;
        uint8_t* blk = pair ? sA + (size_t)(2 * c + 1) * kPairBlk : sA + c * kABytesPerChunk;
        *reinterpret_cast<uint4*>(blk + m * 128 + ((g ^ (m & 7)) << 4)) = val[i];
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpW) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      RingPos rb;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x)
        for (int pass = 0; pass < passes; ++pass)
          for (int c = 0; c < p.nK; ++c, rb.next(kStagesB)) {
            const int t = pair ? 2 * u + pass : u;
            wait_abortable(b_emptyB + 8 * rb.s, rb.ph ^ 1, &s_abort, p.status);
            if (t < p.n_vt) {
              mbar_arrive_expect_tx(b_fullB + 8 * rb.s, kBBytes);
              tma_load_2d_hint(smem_u32(sB + rb.s * kBBytes), &tm_w, b_fullB + 8 * rb.s, c * BK,
                               t * BN, pol);
            } else {
              mbar_arrive(b_fullB + 8 * rb.s);  // past V: nothing to load, rows never read
            }
          }
    }
  } else if (warp == kWarpZ) {
    // row copier: an instruction moves 8 slot rows, lanes 4i..4i+3 the four
    // 16-byte granules of row 8c + i
    const int sub = lane >> 2, g = lane & 3;
    const __nv_bfloat16* zr[16];
    const __nv_bfloat16* tr[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      zr[c] = nullptr;
      tr[c] = nullptr;
      const int m = 8 * c + sub;
      const int n = pair ? (m & 63) : r0 + m;
      if (n < p.R) {
        const VerifyState st = p.vstate[n];
        if (st.mode >= 0 && st.final_row >= 0 && st.final_row < p.n_rows)
          tr[c] = p.target + (size_t)st.final_row * p.V;
        if (st.mode == 1 && st.n_acc >= 0 && st.n_acc < p.gamma)
          zr[c] = p.z + ((size_t)n * p.gamma + st.n_acc) * p.V;
      }
    }
    // per lane, once: the slot offsets of its granules and which rows it
    // copies (a missing row: a valid dummy address, its copies not issued)
    uint32_t off[16], ton = 0, zon = 0;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      off[c] = row_granule(8 * c + sub, g);
      ton |= (tr[c] != nullptr ? 1u : 0u) << c;
      zon |= (zr[c] != nullptr ? 1u : 0u) << c;
      if (tr[c] == nullptr) tr[c] = p.target;
      if (zr[c] == nullptr) zr[c] = p.z;
    }
    uint32_t it = 0, s = 0;
    ZRing zring;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      // slot rows 0-63 read tile t0, rows 64-127 tile t1 (paired; else both t0)
      const int t0 = pair ? 2 * u : u, t1 = pair ? 2 * u + 1 : u;
      for (int j = 0; j < kFinSteps; ++j, ++it) {
        const int h = j / (kFinSteps / 2);
        zring.acquire(b_emptyZ, (int)s, h, &s_abort, p.status);
        fence_proxy_async_smem();
        const uint32_t zdst = smem_u32(sZ + s * kRowSlot), tdst = zdst + kRowPart;
        // V is a multiple of 8: a granule is all in or out
        const int v0 = t0 * BN + j * 32 + g * 8, v1 = t1 * BN + j * 32 + g * 8;
        const uint32_t in0 = v0 < p.V ? 0xffffu : 0u, in1 = v1 < p.V ? 0xffffu : 0u;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int v = c < 8 ? v0 : v1;
          const uint32_t in = c < 8 ? in0 : in1;
          cp_async16_if(tdst + off[c], tr[c] + v, (ton & in) & (1u << c));
          cp_async16_if(zdst + off[c], zr[c] + v, (zon & in) & (1u << c));
        }
        cp_async_arrive(b_fullZ + 8 * (h * 4 + s));
        if (++s == kFinSlots) s = 0;
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      const uint64_t da0 = desc_kmajor_sw128(smem_u32(sA));
      const uint64_t db0 = desc_kmajor_sw128(smem_u32(sB));
      // paired A chunks: pass 0 reads [E_c; 0] at block 2c + 1, pass 1 [0; E_c] at 2c
      const uint32_t a_step = (pair ? 2 * kPairBlk : kABytesPerChunk) >> 4;
      const uint32_t a_pass0 = pair ? kPairBlk >> 4 : 0;
      RingPos rb;
      uint32_t acc_it = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++acc_it) {
        const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
        wait_abortable(b_accEmpty + 8 * a, aph ^ 1, &s_abort, p.status);
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * BN;
        for (int pass = 0; pass < passes; ++pass) {
          uint64_t da = da0 + (pass == 0 ? a_pass0 : 0);
          for (int c = 0; c < p.nK; ++c, da += a_step, rb.next(kStagesB)) {
            wait_abortable(b_fullB + 8 * rb.s, rb.ph, &s_abort, p.status);
            tc_fence_after();
            mma_chunk(d_tmem, da, db0 + rb.s * (kBBytes >> 4), (pass | c) != 0);
            mma_commit(b_emptyB + 8 * rb.s);
          }
        }
        mma_commit(b_accFull + 8 * a);
      }
      mma_commit(b_drain);
      if (!mbar_wait(b_drain, 0)) set_flag(p.status, kFlagTimeout);
    }
  } else {
    // ---------------- epilogue, warps 0-7
    const int quad = warp & 3, half = warp >> 2;
    const int m = quad * 32 + lane;  // TMEM lane = slot row
    const int n = pair ? (m & 63) : r0 + m;
    const int tsub = pair ? (m >> 6) : 0;
    VerifyState st{0, -1, 0, -1, {0.f, 0.f, 0}, {0.f, 0.f, 0}};
    if (n < p.R) st = p.vstate[n];
    const bool live = n < p.R && st.mode >= 0;
    const bool resid = st.mode == 1;
    // a warp whose requests all draw a bonus token computes no q
    const bool warp_q = __any_sync(0xffffffffu, live && resid && st.iq.hi != 0.f);
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t acc_it = 0, zit = 0, cpar = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++acc_it, zit += kFinSteps) {
      const uint32_t a = acc_it & 1, aph = (acc_it >> 1) & 1;
      const int t = pair ? 2 * u + tsub : u;
      const bool valid = live && t < p.n_vt;
      wait_abortable(b_accFull + 8 * a, aph, &s_abort, p.status);
      tc_fence_after();
      float facc[4] = {0.f, 0.f, 0.f, 0.f};  // residual (hi, lo), p (hi, lo)
#pragma unroll 1
      for (int jj = 0; jj < kFinSteps / 2; ++jj) {
        const int j = half * (kFinSteps / 2) + jj;
        const int col = j * 32;
        uint32_t b[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tmem + lane_base + a * BN + col, b);
        const int v0 = t * BN + col;
        const uint32_t zs = (zit + j) % kFinSlots;
        wait_abortable(b_fullZ + 8 * (half * 4 + zs), (cpar >> zs) & 1u, &s_abort, p.status);
        cpar ^= 1u << zs;
        uint4 zq[4], tq[4];
        const uint8_t* zslot = sZ + zs * kRowSlot;
        const uint8_t* tslot = zslot + kRowPart;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          zq[q] = make_uint4(0, 0, 0, 0);
          tq[q] = make_uint4(0, 0, 0, 0);
          if (valid) {
            tq[q] = *reinterpret_cast<const uint4*>(tslot + row_granule(m, q));
            if (resid) zq[q] = *reinterpret_cast<const uint4*>(zslot + row_granule(m, q));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(b_emptyZ + 8 * (half * 4 + zs));
        tmem_wait_ld_regs(b);
        const int lim = min(32, p.V - v0);
        if (valid && lim < 32)  // only the vocabulary's last block
          fin_block<true, true>(b, zq, tq, lim, resid, p.c12, p.sc.hi, p.crest, st.ip, st.iq,
                                facc);
        else if (valid && warp_q)
          fin_block<false, true>(b, zq, tq, lim, resid, p.c12, p.sc.hi, p.crest, st.ip, st.iq,
                                 facc);
        else if (valid)
          fin_block<false, false>(b, zq, tq, lim, resid, p.c12, p.sc.hi, p.crest, st.ip, st.iq,
                                  facc);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_accEmpty + 8 * a);
      if (n < p.R && t < p.n_vt && t * 2 + half < p.n_halves) {
        long long* o = p.fin_part + ((size_t)n * p.n_halves + t * 2 + half) * 2;
        // 2^-60 units: the high parts from their bits, one conversion a low part
        o[0] = fix60(facc[0]) + __float2ll_rn(facc[1] * 1152921504606846976.0f);
        o[1] = fix60(facc[2]) + __float2ll_rn(facc[3] * 1152921504606846976.0f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// c = c12 + crest with c12 = c rounded to 12 significant bits (a bf16 times
// c12 is exact in fp32) and crest the fp32 rounding of the remainder.
void split12(double c, float* c12, float* crest) {
  int e = 0;
  const double m = frexp(c, &e);  // c = m 2^e, m in [1/2, 1)
  const double h = ldexp(nearbyint(ldexp(m, 12)), e - 12);
  *c12 = (float)h;
  *crest = (float)(c - h);
}

// The driver's tensor-map encoder (a process-wide entry point, the same for
// every device); resolved once, thread-safely, by the static's initialiser.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
  }();
  return fn;
}

cudaError_t encode_w(CUtensorMap* m, const void* Wt, int V, int r) {
  cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)V};
  cuuint64_t strides[1] = {(cuuint64_t)r * 2};
  cuuint32_t box[2] = {BK, BN};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(Wt), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

cudaError_t encode_z(CUtensorMap* m, const void* z, int R, int gamma, int V, int box_rows = BM) {
  cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)gamma, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)V * 2, (cuuint64_t)gamma * V * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(z), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

// The staged A rows, [R][r] bf16, as 64-element (128-byte) K chunks of
// box_rows rows, 128-byte swizzled like the A blocks they land in.
cudaError_t encode_stage(CUtensorMap* m, const void* stage, int R, int r, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)R};
  cuuint64_t strides[1] = {(cuuint64_t)r * 2};
  cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(stage), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

template <bool kBiasOut>
cudaError_t launch_tc(const CUtensorMap& tm_w, const CUtensorMap& tm_z, const TcParams& p,
                      cudaStream_t st) {
  // the bias-only pass has no epilogue draws: one instantiation
  auto kern = draft_fused_tc_kernel<kBiasOut, false>;
  if constexpr (!kBiasOut) {
    if (p.greedy) kern = draft_fused_tc_kernel<false, true>;
  }
  cudaError_t e = ensure_smem_attr((const void*)kern, (int)tc_smem_bytes(4));
  if (e != cudaSuccess) return e;
  const int n_rt = (p.R + BM - 1) / BM;
  int gx = sm_count() / n_rt;
  if (gx < 1) gx = 1;
  if (gx > p.n_vt) gx = p.n_vt;
  DSPARK_LAUNCH(kKindDraftFusedTc, st,
                kern<<<dim3(gx, n_rt), kThreads, tc_smem_bytes(p.nK), st>>>(tm_w, tm_z, p));
  return cudaGetLastError();
}

}  // namespace

bool tc_shape_supported(int dt, int V, int r, const void* a, const void* b, const void* c) {
  const uintptr_t mis = reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                        reinterpret_cast<uintptr_t>(c);
  return dt == 0 && r % 8 == 0 && r <= 256 && V % 8 == 0 && (mis & 15) == 0 &&
         encode_fn() != nullptr;
}

bool draft_tc_supported(const DraftArgs& a) {
  return tc_shape_supported(a.dt, a.V, a.r, a.z, a.E, a.Wt);
}

// Fused partial pass for draft position k (previous tokens at
// prev[n * prev_stride]): partials per (request, 128-token half tile) in
// a.part, ceil(V / 128) per request.
cudaError_t launch_draft_partial_tc(const DraftArgs& a, int k, const int32_t* prev,
                                    int prev_stride, cudaStream_t st) {
  CUtensorMap tm_w, tm_z;
  cudaError_t e = encode_w(&tm_w, a.Wt, a.V, a.r);
  if (e == cudaSuccess) e = encode_z(&tm_z, a.z, a.R, a.gamma, a.V);
  if (e != cudaSuccess) return e;
  TcParams p;
  p.R = a.R;
  p.gamma = a.gamma;
  p.V = a.V;
  p.r = a.r;
  p.k = k;
  p.nK = (a.r + BK - 1) / BK;
  p.n_vt = (a.V + BN - 1) / BN;
  p.n_parts = (a.V + kHalf - 1) / kHalf;
  p.greedy = a.T == 0.0f;
  p.sc = make_scale(p.greedy ? 1.0 : 1.4426950408889634 / (double)a.T);
  split12(p.greedy ? 1.0 : 1.4426950408889634 / (double)a.T, &p.c12, &p.crest);
  p.E = static_cast<const __nv_bfloat16*>(a.E);
  p.prev = prev;
  p.prev_stride = prev_stride;
  p.prev_limit = a.V;
  p.part = a.part;
  p.sub = a.sub;
  p.bias_out = nullptr;
  p.status = a.status;
  return launch_tc<false>(tm_w, tm_z, p, st);
}

// Every draft position in one cooperative launch (see draft_persistent_kernel).
// Returns cudaErrorNotSupported, launching nothing, when the GPU cannot hold
// one CTA per SM for the whole grid (the caller then launches per position).
cudaError_t launch_draft_persistent_tc(const DraftArgs& a, cudaStream_t st) {
  if (a.grid_counter == nullptr) return cudaErrorNotSupported;
  const int pair = a.R <= 64 ? 1 : 0;
  CUtensorMap tm_w, tm_z;
  cudaError_t e = encode_w(&tm_w, a.Wt, a.V, a.r);
  if (e == cudaSuccess) e = encode_z(&tm_z, a.z, a.R, a.gamma, a.V, pair ? 64 : BM);
  CUtensorMap tm_a;
  if (e == cudaSuccess) e = encode_stage(&tm_a, a.stage, a.R, a.r, pair ? 64 : BM);
  if (e != cudaSuccess) return e;
  PersistParams pp;
  TcParams& p = pp.p;
  p.R = a.R;
  p.gamma = a.gamma;
  p.V = a.V;
  p.r = a.r;
  p.k = 0;
  p.nK = (a.r + BK - 1) / BK;
  p.n_vt = (a.V + BN - 1) / BN;
  p.n_parts = (a.V + kHalf - 1) / kHalf;
  p.greedy = a.T == 0.0f;
  p.sc = make_scale(p.greedy ? 1.0 : 1.4426950408889634 / (double)a.T);
  split12(p.greedy ? 1.0 : 1.4426950408889634 / (double)a.T, &p.c12, &p.crest);
  p.E = static_cast<const __nv_bfloat16*>(a.E);
  p.prev = nullptr;
  p.prev_stride = 0;
  p.prev_limit = a.V;
  p.part = a.part;
  p.sub = a.sub;
  p.bias_out = nullptr;
  p.status = a.status;
  pp.z = static_cast<const __nv_bfloat16*>(a.z);
  pp.Wt = static_cast<const __nv_bfloat16*>(a.Wt);
  pp.anchor = a.anchor;
  pp.tokens = a.tokens;
  pp.q_lse = a.q_lse;
  pp.q_tok = a.q_tok;
  pp.u = a.u;
  pp.grid_counter = a.grid_counter;
  pp.pair = pair;
  pp.stage = static_cast<__nv_bfloat16*>(a.stage);
  pp.fuse = a.fuse != nullptr && draft_fuse_supported(a, *a.fuse) ? 1 : 0;
  // the scheduler's values, ranks and fixed-point sums (16 bytes a candidate)
  // go below the mbarriers in the dynamic shared memory
  if (16ull * a.R * a.gamma > persist_a_bytes(p.nK, pair) + (size_t)kStagesB * kBBytes +
                                  (size_t)persist_z_slots(pair) * kZBytes)
    pp.fuse = 0;
  if (pp.fuse) pp.f = *a.fuse;
  const int n_rt = (a.R + BM - 1) / BM;
  const int n_units = pair ? (p.n_vt + 1) / 2 : p.n_vt;
  int gx = sm_count() / n_rt;
  if (gx < 1) return cudaErrorNotSupported;
  if (gx > n_units) gx = n_units;
  // two concurrent finishes a CTA once a CTA has eight or more requests (at
  // four, the greedy workload, they measured slower)
  const int per_cta = (a.R + gx * n_rt - 1) / (gx * n_rt);
  // (greedy draws always finish one request at a time: the argmax finish is short)
  const int groups = per_cta >= 8 && !p.greedy ? 2 : 1;
  const void* kern = p.greedy      ? (const void*)draft_persistent_kernel<1, true>
                     : groups == 2 ? (const void*)draft_persistent_kernel<2, false>
                                   : (const void*)draft_persistent_kernel<1, false>;
  e = ensure_smem_attr(kern, (int)tc_smem_bytes(4));
  if (e != cudaSuccess) return e;
  const size_t smem = persist_smem_bytes(p.nK, pair);
  if (blocks_per_sm(kern, kThreads, smem) < 1) return cudaErrorNotSupported;
  e = cudaMemsetAsync(a.grid_counter, 0, 2 * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, n_rt);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.greedy)
    DSPARK_LAUNCH(kKindDraftPersistent, st,
                  e = cudaLaunchKernelEx(&cfg, draft_persistent_kernel<1, true>, tm_w, tm_z, tm_a,
                                         pp));
  else if (groups == 2)
    DSPARK_LAUNCH(kKindDraftPersistent, st,
                  e = cudaLaunchKernelEx(&cfg, draft_persistent_kernel<2, false>, tm_w, tm_z,
                                         tm_a, pp));
  else
    DSPARK_LAUNCH(kKindDraftPersistent, st,
                  e = cudaLaunchKernelEx(&cfg, draft_persistent_kernel<1, false>, tm_w, tm_z,
                                         tm_a, pp));
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e == cudaSuccess && a.fused != nullptr) *a.fused = pp.fuse;
  return e;
}

// The persistent draft can also run the confidence head and the scheduler
// when the head takes the confidence kernel's one-pass path (bf16 hidden
// states and embedding, d <= 4096 and a multiple of 8, 16-byte aligned rows
// and weights) or the confidences are given, and the candidates' values,
// ranks and fixed-point sums fit the kernel's shared memory.
bool draft_fuse_supported(const DraftArgs& a, const DraftFuse& f) {
  const long long N = (long long)a.R * a.gamma;
  if (N > kFuseMaxCandidates || a.dt != 0) return false;
  if (f.c_in != nullptr) return true;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(f.h) | reinterpret_cast<uintptr_t>(f.E1) |
                        reinterpret_cast<uintptr_t>(f.w);
  return f.h != nullptr && f.E1 != nullptr && (mis & 15) == 0 && f.d >= 1 &&
         f.d <= 32 * 8 * conf::kHLoads && f.d % 8 == 0 && a.r % 8 == 0 && a.r <= 256;
}

// bias[n][v] = E[prev[n * prev_stride]] . Wt[v] on the tensor cores (rows of
// requests with prev < 0 are zero).
cudaError_t launch_bias_tc(int R, int V, int r, const void* E, const void* Wt,
                           const int32_t* prev, int prev_stride, int prev_limit, float* bias,
                           uint32_t* status, cudaStream_t st) {
  CUtensorMap tm_w;
  cudaError_t e = encode_w(&tm_w, Wt, V, r);
  if (e != cudaSuccess) return e;
  TcParams p;
  p.R = R;
  p.gamma = 1;
  p.V = V;
  p.r = r;
  p.k = 0;
  p.nK = (r + BK - 1) / BK;
  p.n_vt = (V + BN - 1) / BN;
  p.n_parts = 0;
  p.greedy = 0;
  p.sc = ScalePair{1.f, 0.f};
  p.E = static_cast<const __nv_bfloat16*>(E);
  p.prev = prev;
  p.prev_stride = prev_stride;
  p.prev_limit = prev_limit;
  p.part = nullptr;
  p.sub = nullptr;
  p.bias_out = bias;
  p.status = status;
  return launch_tc<true>(tm_w, tm_w, p, st);
}

// Final-draw partial sums on the tensor cores (see final_tc_kernel):
// fin_part[R][ceil(V / 128)][2].
cudaError_t launch_final_tc(const VerifyArgs& a, const VerifyState* vstate, long long* fin_part,
                            cudaStream_t st) {
  CUtensorMap tm_w;
  cudaError_t e = encode_w(&tm_w, a.Wt, a.V, a.r);
  if (e != cudaSuccess) return e;
  FinalParams p;
  p.R = a.R;
  p.V = a.V;
  p.r = a.r;
  p.nK = (a.r + BK - 1) / BK;
  p.n_vt = (a.V + BN - 1) / BN;
  p.n_halves = (a.V + kHalf - 1) / kHalf;
  p.gamma = a.gamma;
  p.n_rows = a.n_rows;
  p.sc = make_scale(1.4426950408889634 / (double)a.T);
  split12(1.4426950408889634 / (double)a.T, &p.c12, &p.crest);
  p.E = static_cast<const __nv_bfloat16*>(a.E);
  p.z = static_cast<const __nv_bfloat16*>(a.z);
  p.target = static_cast<const __nv_bfloat16*>(a.target);
  p.prev = a.prev;
  p.prev_limit = a.anchor == nullptr ? a.R * a.gamma : a.V;
  p.vstate = vstate;
  p.fin_part = fin_part;
  p.status = a.status;
  p.pair = a.R <= 64 ? 1 : 0;
  e = ensure_smem_attr((const void*)final_tc_kernel, (int)final_smem_bytes(4, 1));
  if (e != cudaSuccess) return e;
  const int n_rt = (a.R + BM - 1) / BM;
  const int n_units = p.pair ? (p.n_vt + 1) / 2 : p.n_vt;
  int gx = sm_count() / n_rt;
  if (gx < 1) gx = 1;
  if (gx > n_units) gx = n_units;
  DSPARK_LAUNCH(kKindFinalTc, st,
                e = launch_pdl(final_tc_kernel, dim3(gx, n_rt), dim3(kThreads),
                               final_smem_bytes(p.nK, p.pair), st, tm_w, p));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_wait_check(uint64_t limit_ns, unsigned* ctr, uint32_t* status, int* out,
                              cudaStream_t st) {
  DSPARK_LAUNCH(kKindWaitCheck, st,
                wait_check_kernel<<<1, 32, 0, st>>>(limit_ns, ctr, status, out));
  return cudaGetLastError();
}

}  // namespace dspark
