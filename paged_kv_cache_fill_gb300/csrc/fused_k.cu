// Fused K path: RMSNorm -> RoPE -> BF16 paged write, one rounding.
// [kv_cache.rs] `fused_k_norm_rope_cache_write_bf16`: K stays above BF16
// precision through the norm and the rotation and is rounded once at the
// cache write.
//
// Precision design. The rotation of a pair (y_i, y_j) can cancel, so an
// output element can be far smaller than its pair; to stay within 1 BF16 ulp
// of the exactly rounded result even then, the error must be small relative
// to the element, not to the pair. The kernel therefore
//   - keeps u = x * w exact (BF16 x BF16 fits a binary32 significand) and
//     applies the RMS factor r = 1/sqrt(mean(x^2) + eps) last, as a relative
//     error only: o = r * (u_i cos - u_j sin);
//   - carries the frequency theta^(-2i/R) as three binary32 parts (from a
//     binary64 exp2), forms pos * freq as a sum of exact products, reduces it
//     by pi/32 held in three parts, and evaluates sin and cos of the
//     remainder (|r| <= pi/64) by short Taylor series in double-binary32
//     arithmetic, combined with a table of sin/cos(m pi/32) held as (hi, lo)
//     pairs (rope_tables.h): about 2^-44 absolute error;
//   - forms u_i cos - u_j sin with exact product error terms (FMA), so the
//     cancellation is exact and the result is accurate to ~2^-23 of itself.
// The error-free transforms use __fmul_rn / __fadd_rn so that the compiler
// cannot fuse them into FMAs.
//
// Work split: a CTA handles 256 / (head_dim / 8) rows (token, head) per
// step, head_dim / 8 lanes per row and 8 elements per lane: lane l < R/8
// holds the rotation pairs (4l..4l+3, R/2+4l..R/2+4l+3), the other lanes 8
// pass-through elements. The sin/cos of a token are computed once per token
// into shared memory and shared by all its heads.
#include <math.h>

#include "internal.h"
#include "rope_tables.h"

namespace pagedkv {

namespace {

struct Dd {
  float hi, lo;
};

__device__ __forceinline__ Dd two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// |a| >= |b| (or a == 0)
__device__ __forceinline__ Dd fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ Dd two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, fmaf(a, b, -p)};
}

struct Freq {
  float h, m, l;  // h + m + l = the binary64 frequency
  float pad;
  double d;
};

// sin and cos of the remainder r = rh + rl (|r| <= ~pi/64), combined with
// the table entry m: returns (sin, cos) of m*pi/32 + r as (hi, lo) pairs.
__device__ __forceinline__ float4 sincos_from_remainder(float rh, float rl, int m) {
  // z = r^2
  const float zh = __fmul_rn(rh, rh);
  const float zl = fmaf(rh, rh, -zh) + 2.0f * rh * rl;
  // sin r = r + r^3 * (-1/6 + z/120 - z^2/5040)
  const float p = __fmul_rn(rh, zh);
  const float pe = fmaf(rh, zh, -p) + (rh * zl + rl * zh);
  const float c6h = -1.0f / 6.0f;
  const float c6l = float(-1.0 / 6.0 - double(-1.0f / 6.0f));  // folded at compile time
  const float poly = c6l + zh * (1.0f / 120.0f - zh * (1.0f / 5040.0f));
  const Dd m1 = two_prod(p, c6h);
  const float corr = m1.lo + (pe * c6h + p * poly);
  Dd sr = fast_two_sum(rh, m1.hi);
  sr.lo = sr.lo + (rl + corr);
  // cos r = 1 + d, d = -z/2 + z^2/24 - z^3/720
  const float dh = -0.5f * zh;
  const float dl = -0.5f * zl + (zh * zh) * (1.0f / 24.0f - zh * (1.0f / 720.0f));
  const float4 t = kSinCosPio32[m & 63];  // {sin_hi, sin_lo, cos_hi, cos_lo}
  // X + X*d + sign * Y*sin r
  auto combine = [&](float xh, float xl, float yh, float yl, float sign) -> Dd {
    const Dd t1 = two_prod(xh, dh);
    const float t1l = t1.lo + (xh * dl + xl * dh);
    const Dd t2 = two_prod(yh, sr.hi);
    const float t2h = sign * t2.hi;
    const float t2l = sign * (t2.lo + (yh * sr.lo + yl * sr.hi));
    Dd x = two_sum(xh, t2h);
    const Dd x2 = two_sum(x.hi, t1.hi);
    const float lo = ((xl + x.lo) + (x2.lo + t1l)) + t2l;
    return fast_two_sum(x2.hi, lo);
  };
  const Dd s = combine(t.x, t.y, t.z, t.w, 1.0f);
  const Dd c = combine(t.z, t.w, t.x, t.y, -1.0f);
  return make_float4(s.hi, s.lo, c.hi, c.lo);
}

// sin and cos of pos * freq as (hi, lo) pairs.
__device__ __forceinline__ float4 rope_sincos(int32_t pos, const Freq& f) {
  if (pos > -65536 && pos < 65536) {
    const float pf = float(pos);  // exact
    const Dd a1 = two_prod(pf, f.h);
    const Dd a2 = two_prod(pf, f.m);
    const float a3 = __fmul_rn(pf, f.l);
    const float k = rintf(__fmul_rn(a1.hi, k32OverPi));
    const Dd q1 = two_prod(k, kPio32P1);
    const Dd q2 = two_prod(k, kPio32P2);
    const float q3 = __fmul_rn(k, kPio32P3);
    float x = __fsub_rn(a1.hi, q1.hi);  // exact (Sterbenz)
    Dd s1 = two_sum(x, a1.lo);
    Dd s2 = two_sum(s1.hi, a2.hi);
    Dd s3 = two_sum(s2.hi, -q1.lo);
    Dd s4 = two_sum(s3.hi, -q2.hi);
    const float lo = ((s1.lo + s2.lo) + (s3.lo + s4.lo)) + ((a2.lo + a3) - (q2.lo + q3));
    const Dd r = fast_two_sum(s4.hi, lo);
    return sincos_from_remainder(r.hi, r.lo, int(k));
  }
  // Large positions: reduce in binary64.
  const double a = double(pos) * f.d;
  const double k = rint(a * (32.0 / 3.14159265358979323846));
  double r = fma(-k, kPio32D1, a);
  r = fma(-k, kPio32D2, r);
  const float rh = float(r);
  const float rl = float(r - double(rh));
  const long long km = (long long)k;
  return sincos_from_remainder(rh, rl, int(km & 63));
}

// Compensated u_a * c + sign * u_b * s with c = (ch, cl), s = (sh, sl).
__device__ __forceinline__ float rotate(float ua, float ub, float ch, float cl, float sh, float sl,
                                        float sign) {
  const Dd p1 = two_prod(ua, ch);
  const Dd p2 = two_prod(ub, sh);
  const Dd s = two_sum(p1.hi, sign * p2.hi);
  return s.hi + (s.lo + ((p1.lo + sign * p2.lo) + (ua * cl + sign * (ub * sl))));
}

__device__ __forceinline__ void unpack8(const uint32_t (&w)[4], float (&x)[8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = bf16_lo_to_f32(w[j]);
    x[2 * j + 1] = bf16_hi_to_f32(w[j]);
  }
}

constexpr int kThreads = 256;
constexpr int kMaxRows = 32;        // rows per step for head_dim 64
constexpr int kMaxTableEntries = 1024;  // tokens per step x rotary_dim/2

template <int D>
__global__ void __launch_bounds__(kThreads) fused_k_norm_rope_kernel(
    const uint16_t* __restrict__ k_in, const uint16_t* __restrict__ k_norm_weight,
    const int32_t* __restrict__ positions, uint16_t* __restrict__ k_cache,
    const int64_t* __restrict__ slot_mapping, uint32_t num_tokens, uint32_t num_kv_heads,
    uint32_t rotary_dim, float rms_eps, float theta) {
  constexpr int kLanes = D / 8;                 // lanes per row
  constexpr int kRows = kThreads / kLanes;      // rows per step
  static_assert(kRows <= kMaxRows, "rows per step");
  __shared__ Freq freq[128];
  __shared__ float4 table[2][kMaxTableEntries];

  const uint32_t half = rotary_dim / 2;
  // Frequencies theta^(-2i/R) in binary64, split into three binary32 parts.
  if (threadIdx.x < half) {
    const double c = -2.0 * log2(double(theta)) / double(rotary_dim);
    const double f = exp2(c * double(threadIdx.x));
    Freq e;
    e.h = float(f);
    e.m = float(f - double(e.h));
    e.l = float(f - double(e.h) - double(e.m));
    e.pad = 0.0f;
    e.d = f;
    freq[threadIdx.x] = e;
  }

  const uint32_t lane = threadIdx.x % kLanes;
  const uint32_t row_in_step = threadIdx.x / kLanes;
  const uint32_t pair_lanes = rotary_dim / 8;
  const bool is_pair = lane < pair_lanes;
  // element offsets of this lane's two groups of four (pair lanes) or one
  // group of eight (pass-through lanes)
  const uint32_t off_a = is_pair ? 4 * lane : rotary_dim + 8 * (lane - pair_lanes);
  const uint32_t off_b = is_pair ? half + 4 * lane : off_a + 4;

  float w[8];
  {
    const uint2 wa = *reinterpret_cast<const uint2*>(k_norm_weight + off_a);
    const uint2 wb = *reinterpret_cast<const uint2*>(k_norm_weight + off_b);
    const uint32_t ww[4] = {wa.x, wa.y, wb.x, wb.y};
    unpack8(ww, w);
  }
  __syncthreads();

  const uint64_t total_rows = uint64_t(num_tokens) * num_kv_heads;
  const uint64_t steps = (total_rows + kRows - 1) / kRows;
  uint32_t parity = 0;
  for (uint64_t step = blockIdx.x; step < steps; step += gridDim.x, parity ^= 1) {
    const uint64_t row0 = step * kRows;
    const uint64_t row = row0 + row_in_step;
    const bool active = row < total_rows;
    const uint32_t t_first = uint32_t(row0 / num_kv_heads);
    // rows past the end idle on the step's first token (in-bounds table reads)
    const uint32_t t = active ? uint32_t(row / num_kv_heads) : t_first;
    const uint32_t h = active ? uint32_t(row % num_kv_heads) : 0;
    uint64_t last_row = row0 + kRows - 1;
    if (last_row >= total_rows) last_row = total_rows - 1;
    const uint32_t ntok = uint32_t(last_row / num_kv_heads) - t_first + 1;

    // issue this row's loads first
    int64_t slot = -1;
    uint2 xa = make_uint2(0, 0), xb = make_uint2(0, 0);
    if (active) {
      slot = __ldg(slot_mapping + t);
      const uint16_t* src = k_in + (uint64_t(t) * num_kv_heads + h) * D;
      xa = __ldcs(reinterpret_cast<const uint2*>(src + off_a));
      xb = __ldcs(reinterpret_cast<const uint2*>(src + off_b));
    }
    // sin/cos of every (token of this step, frequency)
    for (uint32_t e = threadIdx.x; e < ntok * half; e += kThreads) {
      const uint32_t j = e / half, i = e % half;
      table[parity][j * half + i] = rope_sincos(__ldg(positions + t_first + j), freq[i]);
    }
    __syncthreads();

    float x[8];
    {
      const uint32_t xw[4] = {xa.x, xa.y, xb.x, xb.y};
      unpack8(xw, x);
    }
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);  // x^2 is exact in binary32
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(__fadd_rn(ss / float(D), rms_eps));

    float u[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) u[j] = __fmul_rn(x[j], w[j]);  // exact
    float out[8];
    if (is_pair && active) {
      const float4* tb = &table[parity][(t - t_first) * half + 4 * lane];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 sc = tb[q];  // {sin_hi, sin_lo, cos_hi, cos_lo}
        out[q] = rotate(u[q], u[4 + q], sc.z, sc.w, sc.x, sc.y, -1.0f);
        out[4 + q] = rotate(u[4 + q], u[q], sc.z, sc.w, sc.x, sc.y, 1.0f);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = u[j];
    }
    if (active && slot >= 0) {
      uint32_t packed[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        packed[j] = f32x2_to_bf16x2(__fmul_rn(out[2 * j], r), __fmul_rn(out[2 * j + 1], r));
      uint16_t* dst = k_cache + (uint64_t(slot) * num_kv_heads + h) * D;
      *reinterpret_cast<uint2*>(dst + off_a) = make_uint2(packed[0], packed[1]);
      *reinterpret_cast<uint2*>(dst + off_b) = make_uint2(packed[2], packed[3]);
    }
  }
}

}  // namespace

cudaError_t launch_fused_k_norm_rope(const uint16_t* k_in, const uint16_t* k_norm_weight,
                                     const int32_t* positions, uint16_t* k_cache,
                                     const int64_t* slot_mapping, uint32_t num_tokens,
                                     uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                     float rms_eps, float theta, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  const uint32_t rows_per_step = kThreads / (head_dim / 8);
  const uint64_t steps = (uint64_t(num_tokens) * num_kv_heads + rows_per_step - 1) / rows_per_step;
  uint64_t blocks = uint64_t(dev.num_sms) * 4;
  if (steps < blocks) blocks = steps;
  switch (head_dim) {
    case 64:
      fused_k_norm_rope_kernel<64><<<unsigned(blocks), kThreads, 0, stream>>>(
          k_in, k_norm_weight, positions, k_cache, slot_mapping, num_tokens, num_kv_heads,
          rotary_dim, rms_eps, theta);
      break;
    case 128:
      fused_k_norm_rope_kernel<128><<<unsigned(blocks), kThreads, 0, stream>>>(
          k_in, k_norm_weight, positions, k_cache, slot_mapping, num_tokens, num_kv_heads,
          rotary_dim, rms_eps, theta);
      break;
    case 256:
      fused_k_norm_rope_kernel<256><<<unsigned(blocks), kThreads, 0, stream>>>(
          k_in, k_norm_weight, positions, k_cache, slot_mapping, num_tokens, num_kv_heads,
          rotary_dim, rms_eps, theta);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pagedkv
