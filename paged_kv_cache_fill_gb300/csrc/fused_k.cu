// Fused K path: RMSNorm -> RoPE -> paged write, one rounding.
// [kv_cache.rs] `fused_k_norm_rope_cache_write_bf16`: K stays above BF16
// precision through the norm and the rotation and is rounded once at the
// cache write. The same kernel serves the MRoPE variant
// (`fused_k_norm_rope_cache_write_bf16_mrope`: pair i turns by the position
// of stream i % 3) and the FP8-output variant
// (`fused_k_norm_rope_cache_write_fp8`: E4M3 of the result times inv_scale).
//
// Precision design. The rotation of a pair (y_i, y_j) can cancel, so an
// output element can be far smaller than its pair; to stay within 1 BF16 ulp
// of the exactly rounded result even then, the error must be small relative
// to the element, not to the pair. The kernel therefore
//   - keeps u = x * w exact (BF16 x BF16 fits a binary32 significand) and
//     applies the RMS factor r = 1/sqrt(mean(x^2) + eps) last, as a relative
//     error only: o = r * (u_i cos - u_j sin);
//   - reduces the angle pos * f_i modulo one turn exactly: the host passes,
//     per rotation pair, G_i = frac(f_i / (2 pi)) as a 96-bit fixed-point
//     fraction of a turn (f_i = theta^(-2i/R) in binary64, divided by 2 pi
//     through the 256-bit constant 2^256 / (2 pi)), and the kernel forms
//     pos * G_i mod 2^96 with integer multiplies, for any int32 position;
//   - takes sin/cos of the nearest multiple of 2 pi / 2048 from a table of
//     binary32 (hi, lo) pairs and finishes with the remainder r
//     (|r| <= pi / 2048, converted to radians as a binary32 pair): the
//     products with the table entries are formed exactly (FMA) and the
//     short series of sin r and cos r - 1 enter as small corrections,
//     largest last, for about 2^-43 absolute error;
//   - forms u_i cos - u_j sin inside one FMA against the rounded second
//     product, adding that product's exact error (FMA) afterwards, so the
//     cancellation is exact and the result is accurate to ~2^-23 of itself.
// Error-free transforms use __fmul_rn / __fadd_rn so that the compiler
// cannot fuse them into FMAs.
//
// Work split. A warp handles 256 / head_dim tokens at a time with
// head_dim / 8 lanes per token. Lane l of a token owns unit l of every head
// row of that token: when l < rotary_dim / 8 the rotation pairs 4l..4l+3
// (elements 4l..4l+3 and R/2+4l..R/2+4l+3), otherwise 8 pass-through
// elements (rotated by the identity, so that every lane runs the same code).
// A lane therefore needs sin/cos of its own four pairs only: it computes
// them once per token and uses them for every head, with no shared memory
// and no barriers. Each warp walks (token group, group of kHeadsPerStep
// heads) items and loads the next item's rows into registers before it
// computes the current one, so loads are always in flight.
#include <math.h>

#include "internal.h"
#include "rope_tables.h"

namespace pagedkv {

__device__ uint32_t g_fused_error;

namespace {

struct Dd {
  float hi, lo;
};

// |a| >= |b| (or a == 0)
__device__ __forceinline__ Dd fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// Per rotation pair i < rotary_dim / 2: frac(f_i / (2 pi)) * 2^96 as
// {bits 0..31, 32..63, 64..95, unused}. Computed on the host per call and
// passed by value.
struct TurnTable {
  uint4 g[128];
};

// sin and cos, as (hi, lo) pairs {sin_hi, sin_lo, cos_hi, cos_lo}, of the
// angle whose fraction of a turn is pos * G mod 1 (G in units of 2^-96 turn);
// `table` is the CTA's shared-memory copy of kSinCosTurn.
__device__ __forceinline__ float4 turn_sincos(int32_t pos, uint4 g, const float4* table) {
  // bits 32..95 of pos * G mod 2^96 (bits 0..31 are below the precision kept)
  const uint32_t pu = uint32_t(pos);
  const uint64_t mid = uint64_t(pu) * g.y + __umulhi(pu, g.x);
  uint64_t w = ((uint64_t(uint32_t(mid >> 32) + pu * g.z)) << 32) | uint32_t(mid);
  // a negative position was multiplied as pos + 2^32: take 2^32 * G back off
  const uint64_t neg = uint64_t(int64_t(pos >> 31));
  w -= ((uint64_t(g.y) << 32) | g.x) & neg;
  const uint32_t w2 = uint32_t(w >> 32), w1 = uint32_t(w);
  // nearest multiple m of 1/2048 turn, and the remainder
  // (u - 2^20 + w1 / 2^32) * 2^-32 turn with |u - 2^20| <= 2^20
  constexpr int kShift = 32 - kTurnTableBits;
  const uint32_t wr = w2 + (1u << (kShift - 1));
  const uint32_t m = wr >> kShift;
  const uint32_t u = wr & ((1u << kShift) - 1);
  // integers below 2^23 convert exactly through the 2^23 exponent pattern
  const float th = __fsub_rn(__uint_as_float(0x4B000000u | u), float(8388608 + (1 << (kShift - 1))));
  const float tl = __fmul_rn(__fsub_rn(__uint_as_float(0x4B000000u | (w1 >> 9)), 8388608.0f), 0x1p-23f);
  // r = (th + tl) * 2 pi / 2^32 as rh + rl
  const float rh = __fmul_rn(th, kTwoPiOver2p32Hi);
  const float rl = fmaf(th, kTwoPiOver2p32Lo, fmaf(tl, kTwoPiOver2p32Hi, fmaf(th, kTwoPiOver2p32Hi, -rh)));
  // {sin_hi, sin_lo, cos_hi, cos_lo} of 2 pi m / 2048
  const float4 T = table[m];
  // cos r = 1 + dh + dl (dh = -rh^2 / 2 exactly), sin r = rh + t
  const float r2 = __fmul_rn(rh, rh);
  const float r2e = fmaf(rh, rh, -r2);
  const float dh = __fmul_rn(-0.5f, r2);
  const float dl = fmaf(r2, __fmul_rn(r2, 1.0f / 24.0f), fmaf(-rh, rl, __fmul_rn(-0.5f, r2e)));
  const float t = fmaf(__fmul_rn(rh, r2), -1.0f / 6.0f, rl);
  // sin(A + r) = sin A (1 + d) + cos A (rh + t); |sin A| >= sin(2 pi / 2048)
  // or sin A == 0, and |cos A * rh| <= pi / 2048, so fast_two_sum applies
  const float p = __fmul_rn(T.z, rh);
  Dd s = fast_two_sum(T.x, p);
  float lo = fmaf(T.w, rh, fmaf(T.z, rh, -p));
  lo = fmaf(T.x, dl, lo);
  lo = __fadd_rn(__fadd_rn(lo, T.y), s.lo);
  lo = fmaf(T.z, t, lo);
  lo = fmaf(T.x, dh, lo);
  s = fast_two_sum(s.hi, lo);
  // cos(A + r) = cos A (1 + d) - sin A (rh + t)
  const float q = __fmul_rn(T.x, rh);
  Dd c = fast_two_sum(T.z, -q);
  lo = fmaf(-T.y, rh, -fmaf(T.x, rh, -q));
  lo = fmaf(T.z, dl, lo);
  lo = __fadd_rn(__fadd_rn(lo, T.w), c.lo);
  lo = fmaf(-T.x, t, lo);
  lo = fmaf(T.z, dh, lo);
  c = fast_two_sum(c.hi, lo);
  return make_float4(s.hi, s.lo, c.hi, c.lo);
}

// The low (kHi false) or high BF16 halves of a and b multiplied exactly and
// added to c with one rounding (mixed-precision FMA: no unpacking to binary32).
template <bool kHi>
__device__ __forceinline__ float fma_bf16(uint32_t a, uint32_t b, float c) {
  float d;
  if (kHi)
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
  else
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

// Sum of the squares of the 8 BF16 values in (a, b); each square is exact.
__device__ __forceinline__ float sum_sq8(uint2 a, uint2 b) {
  float s0 = fma_bf16<false>(a.x, a.x, 0.0f), s1 = fma_bf16<true>(a.x, a.x, 0.0f);
  s0 = fma_bf16<false>(a.y, a.y, s0);
  s1 = fma_bf16<true>(a.y, a.y, s1);
  s0 = fma_bf16<false>(b.x, b.x, s0);
  s1 = fma_bf16<true>(b.x, b.x, s1);
  s0 = fma_bf16<false>(b.y, b.y, s0);
  s1 = fma_bf16<true>(b.y, b.y, s1);
  return __fadd_rn(s0, s1);
}

// x * w for a pair of BF16 values (the word's halves): exact in binary32.
__device__ __forceinline__ F2 mul_bf16x2(uint32_t x, uint32_t w) {
  return f2_make(fma_bf16<false>(x, w, -0.0f), fma_bf16<true>(x, w, -0.0f));
}

// Sine and cosine of two rotation pairs, each as a (hi, lo) binary32 pair,
// packed pair by pair for the f32x2 rotation.
struct PairSinCos {
  F2 ch, cl, sh, nsh, sl;
};

// The rotation of two pairs at once: X holds their first elements, Y their
// partners (rotary_dim / 2 further on). out_x = X cos - Y sin and
// out_y = Y cos + X sin, each accurate to about 2^-23 of itself even when the
// two products cancel: the product that is subtracted is rounded once and its
// exact error (FMA against the negated sine) is added back with the low
// parts of sin and cos, after the main difference has been formed exactly
// inside one FMA and rounded once.
__device__ __forceinline__ void rotate2(F2 X, F2 Y, const PairSinCos& c, F2& out_x, F2& out_y) {
  const F2 nq = f2_mul(Y, c.nsh);             // -RN(Y sh)
  const F2 e = f2_fma(Y, c.sh, nq);           // Y sh - RN(Y sh), exact
  const F2 tx = f2_fma(X, c.ch, nq);          // X ch - RN(Y sh), one rounding
  const F2 sx = f2_sub(f2_mul(X, c.cl), f2_mul(Y, c.sl));
  out_x = f2_add(tx, f2_sub(sx, e));
  const F2 q = f2_mul(X, c.sh);               // RN(X sh)
  const F2 ne = f2_fma(X, c.nsh, q);          // RN(X sh) - X sh, exact
  const F2 ty = f2_fma(Y, c.ch, q);           // Y ch + RN(X sh), one rounding
  const F2 sy = f2_fma(Y, c.cl, f2_mul(X, c.sl));
  out_y = f2_add(ty, f2_sub(sy, ne));
}

// Launch shape: persistent, two 256-thread CTAs per SM, four head rows per
// lane per item (a sweep of threads, CTAs per SM and heads per item chose
// it; eight heads per item spilled or cut the occupancy).
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCtasPerSm = 2;
constexpr int kHeadsPerStep = 4;  // head rows a lane holds per item

// One item's inputs for this lane: its unit of kHeadsPerStep head rows of one
// token, the token's slot and (on the token's first item) its positions.
struct Item {
  uint2 xa[kHeadsPerStep], xb[kHeadsPerStep];
  int64_t slot;
  int32_t pos[3];
  uint32_t t, hg;
  bool valid;
};

// kFp8Out: store E4M3(o * inv_scale) (saturating, RNE) instead of BF16(o).
// kMrope: pair i takes its position from positions / pos_h / pos_w by i % 3.
template <int D, bool kFp8Out, bool kMrope>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) fused_k_norm_rope_kernel(
    const uint16_t* __restrict__ k_in, const uint16_t* __restrict__ k_norm_weight,
    const int32_t* __restrict__ positions, const int32_t* __restrict__ pos_h,
    const int32_t* __restrict__ pos_w, void* __restrict__ k_cache,
    const int64_t* __restrict__ slot_mapping, uint32_t num_tokens, uint32_t num_kv_heads,
    uint32_t rotary_dim, float rms_eps, const __grid_constant__ TurnTable tt, float inv_scale) {
  constexpr uint32_t kLanes = D / 8;        // lanes per token
  constexpr uint32_t kTokens = 32 / kLanes;  // tokens per warp step
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t sub = lane / kLanes;        // token of the step
  const uint32_t l = lane % kLanes;          // unit of the row
  const uint32_t half = rotary_dim / 2;
  const bool is_pair = l < rotary_dim / 8;
  // element offsets of this lane's two groups of four
  const uint32_t off_a = is_pair ? 4 * l : rotary_dim + 8 * (l - rotary_dim / 8);
  const uint32_t off_b = is_pair ? half + 4 * l : off_a + 4;
  const uint32_t head_groups = (num_kv_heads + kHeadsPerStep - 1) / kHeadsPerStep;

  // work of this warp: token steps gw, gw + W, ..., each in head_groups items
  const uint32_t warps_total = gridDim.x * kWarps;
  const uint32_t gw = blockIdx.x * kWarps + threadIdx.x / 32;
  const uint32_t steps_total = (num_tokens + kTokens - 1) / kTokens;
  const uint32_t my_steps = gw < steps_total ? (steps_total - gw + warps_total - 1) / warps_total : 0;
  const uint32_t n_items = my_steps * head_groups;

  auto load_item = [&](uint32_t k, Item& it) {
    const uint32_t step = gw + (k / head_groups) * warps_total;
    it.hg = k % head_groups;
    it.t = step * kTokens + sub;
    it.valid = it.t < num_tokens;
    it.slot = -1;
#pragma unroll
    for (int j = 0; j < kHeadsPerStep; ++j) it.xa[j] = it.xb[j] = make_uint2(0, 0);
    if (!it.valid) return;
    it.slot = __ldg(slot_mapping + it.t);
    if (it.hg == 0) {
      it.pos[0] = __ldg(positions + it.t);
      if (kMrope) {
        it.pos[1] = __ldg(pos_h + it.t);
        it.pos[2] = __ldg(pos_w + it.t);
      }
    }
    const uint16_t* src = k_in + (uint64_t(it.t) * num_kv_heads + it.hg * kHeadsPerStep) * D;
#pragma unroll
    for (int j = 0; j < kHeadsPerStep; ++j) {
      if (it.hg * kHeadsPerStep + j < num_kv_heads) {
        it.xa[j] = __ldcs(reinterpret_cast<const uint2*>(src + j * D + off_a));
        it.xb[j] = __ldcs(reinterpret_cast<const uint2*>(src + j * D + off_b));
      }
    }
  };

  Item A, B;
  if (n_items > 0) load_item(0, A);  // the first rows are on their way before the set-up below

  __shared__ uint4 s_turn[128];  // turn fractions of the rotation pairs
  // The sin/cos table in shared memory, one bulk copy per CTA issued now,
  // beside the first rows. A warp's 32 lookups at unrelated indices cost a
  // few shared-memory wavefronts here; read through L1 they touched ~32
  // distinct lines each, which at 4096 tokens was ~2 us of every warp's
  // first item.
  __shared__ __align__(128) float4 s_table[sizeof(kSinCosTurn) / sizeof(float4)];
  __shared__ uint64_t s_table_bar;
  if (threadIdx.x == 0) {
    mbar_init(&s_table_bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&s_table_bar, sizeof(kSinCosTurn));
    bulk_load(s_table, kSinCosTurn, sizeof(kSinCosTurn), &s_table_bar);
  }
  for (uint32_t i = threadIdx.x; i < half; i += kThreads) s_turn[i] = tt.g[i];
  // the norm weights of this lane's unit, as BF16 pairs
  const uint2 wa = *reinterpret_cast<const uint2*>(k_norm_weight + off_a);
  const uint2 wb = *reinterpret_cast<const uint2*>(k_norm_weight + off_b);
  // sin/cos of this lane's pairs (4l, 4l+1) and (4l+2, 4l+3) for the current
  // token; the identity for pass-through lanes
  PairSinCos sc[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    sc[k].ch = f2_make(1.0f, 1.0f);
    sc[k].cl = sc[k].sh = sc[k].nsh = sc[k].sl = f2_make(0.0f, 0.0f);
  }
  __syncthreads();  // s_turn written (and the table's barrier initialised); no barrier follows
  if (!mbar_wait(&s_table_bar, 0)) {
    // the copy did not land in time: flag it and let it land (bounded)
    // before the CTA can release its shared memory
    if ((threadIdx.x & 31) == 0) atomicOr(&g_fused_error, kErrWaitTimeout);
    mbar_wait(&s_table_bar, 0);
    return;
  }
  if (n_items == 0) return;

  auto process = [&](const Item& it) {
    if (it.hg == 0 && it.valid && is_pair) {
      float4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int32_t pos = it.pos[0];
        if (kMrope) {
          const uint32_t stream = (4 * l + q) % 3;
          pos = stream == 0 ? it.pos[0] : (stream == 1 ? it.pos[1] : it.pos[2]);
        }
        v[q] = turn_sincos(pos, s_turn[4 * l + q], s_table);  // {sin_hi, sin_lo, cos_hi, cos_lo}
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float4 a0 = v[2 * k], a1 = v[2 * k + 1];
        sc[k].ch = f2_make(a0.z, a1.z);
        sc[k].cl = f2_make(a0.w, a1.w);
        sc[k].sh = f2_make(a0.x, a1.x);
        sc[k].nsh = f2_make(-a0.x, -a1.x);
        sc[k].sl = f2_make(a0.y, a1.y);
      }
    }
    int64_t slot = it.slot;
#ifdef PAGEDKV_DEBUG_BOUNDS
    if (it.valid && slot >= 0 && !dbg_slot_ok(slot)) slot = -1;  // skipped like padding
#endif
    // sums of squares of every row first, then their reductions over the
    // token's lanes side by side, so that the shuffles do not wait on each
    // other (rows past the last head are zeros and are not stored)
    float ss[kHeadsPerStep];
#pragma unroll
    for (int j = 0; j < kHeadsPerStep; ++j) ss[j] = sum_sq8(it.xa[j], it.xb[j]);  // x^2 exact in binary32
#pragma unroll
    for (uint32_t o = kLanes / 2; o > 0; o >>= 1) {
#pragma unroll
      for (int j = 0; j < kHeadsPerStep; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], o);
    }
#pragma unroll
    for (int j = 0; j < kHeadsPerStep; ++j) {
      const uint32_t h = it.hg * kHeadsPerStep + j;
      if (!it.valid || slot < 0 || h >= num_kv_heads) continue;
      // 1/sqrt(mean + eps): a few-ulp binary32 factor, a relative error on the
      // whole row far below half a BF16 ulp
      const float r = rsqrtf(__fadd_rn(ss[j] * (1.0f / float(D)), rms_eps));
      // u = x * w (exact); X: elements 0..3 of the unit, Y: their partners 4..7
      const F2 x01 = mul_bf16x2(it.xa[j].x, wa.x), x23 = mul_bf16x2(it.xa[j].y, wa.y);
      const F2 y01 = mul_bf16x2(it.xb[j].x, wb.x), y23 = mul_bf16x2(it.xb[j].y, wb.y);
      F2 o[4];  // elements (0,1), (2,3), (4,5), (6,7)
      rotate2(x01, y01, sc[0], o[0], o[2]);
      rotate2(x23, y23, sc[1], o[1], o[3]);
      if constexpr (kFp8Out) {
        // no BF16 rounding: the binary32 result times r * inv_scale, cast once
        const float rs = __fmul_rn(r, inv_scale);
        const F2 rs2 = f2_make(rs, rs);
        uint32_t codes[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 a0 = f2_split(f2_mul(o[2 * e], rs2)), a1 = f2_split(f2_mul(o[2 * e + 1], rs2));
          codes[e] = uint32_t(f32x2_to_e4m3x2_satfinite(a0.x, a0.y)) |
                     (uint32_t(f32x2_to_e4m3x2_satfinite(a1.x, a1.y)) << 16);
        }
        uint8_t* dst = static_cast<uint8_t*>(k_cache) + (uint64_t(slot) * num_kv_heads + h) * D;
        *reinterpret_cast<uint32_t*>(dst + off_a) = codes[0];
        *reinterpret_cast<uint32_t*>(dst + off_b) = codes[1];
      } else {
        const F2 r2 = f2_make(r, r);
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a0 = f2_split(f2_mul(o[e], r2));
          packed[e] = f32x2_to_bf16x2(a0.x, a0.y);
        }
        uint16_t* dst = static_cast<uint16_t*>(k_cache) + (uint64_t(slot) * num_kv_heads + h) * D;
        *reinterpret_cast<uint2*>(dst + off_a) = make_uint2(packed[0], packed[1]);
        *reinterpret_cast<uint2*>(dst + off_b) = make_uint2(packed[2], packed[3]);
      }
    }
  };

  // two item buffers in turn: the next item's loads are issued before the
  // current item is computed
  for (uint32_t k = 0;;) {
    if (k + 1 < n_items) load_item(k + 1, B);
    process(A);
    if (++k >= n_items) break;
    if (k + 1 < n_items) load_item(k + 1, A);
    process(B);
    if (++k >= n_items) break;
  }
}

// frac(f / (2 pi)) * 2^96 for a binary64 f > 0, least significant word first.
// f = M * 2^(e - 53) with a 53-bit integer M, so f / (2 pi) * 2^96 =
// X * 2^(e - 213) with X = M * floor(2^256 / (2 pi)); its fraction's 96 bits
// are bits [213 - e, 309 - e) of X (the truncation of the constant moves them
// by less than 2^-200).
uint4 turn_fraction(double f) {
  int e = 0;
  const double fr = frexp(f, &e);
  const uint64_t M = uint64_t(ldexp(fr, 53));
  uint64_t X[5];
  unsigned __int128 carry = 0;
  for (int k = 0; k < 4; ++k) {
    const unsigned __int128 prod = (unsigned __int128)M * kInv2Pi256[3 - k] + carry;
    X[k] = uint64_t(prod);
    carry = prod >> 64;
  }
  X[4] = uint64_t(carry);
  auto word = [&](int bit) -> uint32_t {  // X's bits [bit, bit + 32); zero outside X
    uint32_t v = 0;
    for (int b = 0; b < 32; ++b) {
      const int at = bit + b;
      if (at >= 0 && at < 320 && ((X[at >> 6] >> (at & 63)) & 1u)) v |= 1u << b;
    }
    return v;
  };
  const int lo = 213 - e;
  return make_uint4(word(lo), word(lo + 32), word(lo + 64), 0u);
}

// The turn fractions of theta^(-2i/R), i < R/2, for the last (theta, R) this
// host thread launched with.
const TurnTable& turn_table(float theta, uint32_t rotary_dim) {
  thread_local TurnTable tt;
  thread_local float cached_theta = 0.0f;
  thread_local uint32_t cached_r = 0;
  if (cached_r != rotary_dim || cached_theta != theta) {
    const double c = -2.0 * log2(double(theta)) / double(rotary_dim);
    for (uint32_t i = 0; i < 128; ++i) tt.g[i] = i < rotary_dim / 2 ? turn_fraction(exp2(c * double(i))) : uint4{};
    cached_theta = theta;
    cached_r = rotary_dim;
  }
  return tt;
}

}  // namespace

template <int D>
static void launch_d(bool fp8_out, bool mrope, unsigned blocks, cudaStream_t stream, const uint16_t* k_in,
                     const uint16_t* w, const int32_t* pos, const int32_t* pos_h, const int32_t* pos_w, void* cache,
                     const int64_t* slots, uint32_t n, uint32_t H, uint32_t R, float eps, const TurnTable& tt,
                     float inv_scale) {
  if (fp8_out)
    fused_k_norm_rope_kernel<D, true, false><<<blocks, kThreads, 0, stream>>>(k_in, w, pos, pos_h, pos_w, cache,
                                                                              slots, n, H, R, eps, tt, inv_scale);
  else if (mrope)
    fused_k_norm_rope_kernel<D, false, true><<<blocks, kThreads, 0, stream>>>(k_in, w, pos, pos_h, pos_w, cache,
                                                                              slots, n, H, R, eps, tt, inv_scale);
  else
    fused_k_norm_rope_kernel<D, false, false><<<blocks, kThreads, 0, stream>>>(k_in, w, pos, pos_h, pos_w, cache,
                                                                               slots, n, H, R, eps, tt, inv_scale);
}

cudaError_t launch_fused_k_norm_rope(const uint16_t* k_in, const uint16_t* k_norm_weight,
                                     const int32_t* positions, const int32_t* pos_h, const int32_t* pos_w,
                                     void* k_cache, bool fp8_out, float inv_scale,
                                     const int64_t* slot_mapping, uint32_t num_tokens,
                                     uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                     float rms_eps, float theta, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  const uint32_t tokens_per_step = 256 / head_dim;
  const uint64_t steps = (uint64_t(num_tokens) + tokens_per_step - 1) / tokens_per_step;
  uint64_t blocks = uint64_t(dev.num_sms) * kCtasPerSm;  // persistent
  const uint64_t needed = (steps + kWarps - 1) / kWarps;   // one step per warp at least
  if (needed < blocks) blocks = needed;
  const bool mrope = pos_h != nullptr;
  const TurnTable& tt = turn_table(theta, rotary_dim);
  switch (head_dim) {
    case 64:
      launch_d<64>(fp8_out, mrope, unsigned(blocks), stream, k_in, k_norm_weight, positions, pos_h, pos_w, k_cache,
                   slot_mapping, num_tokens, num_kv_heads, rotary_dim, rms_eps, tt, inv_scale);
      break;
    case 128:
      launch_d<128>(fp8_out, mrope, unsigned(blocks), stream, k_in, k_norm_weight, positions, pos_h, pos_w, k_cache,
                    slot_mapping, num_tokens, num_kv_heads, rotary_dim, rms_eps, tt, inv_scale);
      break;
    case 256:
      launch_d<256>(fp8_out, mrope, unsigned(blocks), stream, k_in, k_norm_weight, positions, pos_h, pos_w, k_cache,
                    slot_mapping, num_tokens, num_kv_heads, rotary_dim, rms_eps, tt, inv_scale);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t read_and_clear_fused_error(uint32_t* bits) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_fused_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_fused_error, &zero, sizeof(uint32_t));
}

#ifdef PAGEDKV_DEBUG_BOUNDS
PAGEDKV_DEBUG_UNIT(fused_k)
#endif

}  // namespace pagedkv
