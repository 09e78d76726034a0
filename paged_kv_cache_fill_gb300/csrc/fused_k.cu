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
//   - forms u_i cos - u_j sin inside one FMA against the rounded second
//     product, adding that product's exact error (FMA) afterwards, so the
//     cancellation is exact and the result is accurate to ~2^-23 of itself.
// The error-free transforms use __fmul_rn / __fadd_rn so that the compiler
// cannot fuse them into FMAs.
//
// Work split: two 256-thread CTAs per SM (their phases interleave) take
// passes of up to tokens_per_pass() tokens (all their heads); the frequency
// ladder comes from the host with the launch. head_dim / 8 lanes per row and
// 8 elements per lane: lane l < R/8 holds the rotation pairs (4l..4l+3,
// R/2+4l..R/2+4l+3), the other lanes 8 pass-through elements; a thread keeps
// up to 4 rows. Each pass
// first issues every row load, then all threads build the pass's sin/cos
// table in shared memory (once per token, shared by its heads) while the
// loads are in flight, then normalises, rotates and stores every row.
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

// theta^(-2i/R) for every rotation pair i < R/2 (R <= 256), computed on the
// host per call (binary64 exp2/log2 are slow on this GPU) and passed by value.
struct FreqTable {
  Freq f[128];
};

// sin and cos of the remainder r = rh + rl (|r| <= ~pi/64), combined with
// the table entry m: returns (sin, cos) of m*pi/32 + r as (hi, lo) pairs.
__device__ __forceinline__ float4 sincos_from_remainder(float rh, float rl, int m, const float4* tab) {
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
  const float4 t = tab[m & 63];  // {sin_hi, sin_lo, cos_hi, cos_lo} of m*pi/32
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
__device__ __forceinline__ float4 rope_sincos(int32_t pos, const Freq& f, const float4* tab) {
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
    return sincos_from_remainder(r.hi, r.lo, int(k), tab);
  }
  // Large positions: reduce in binary64.
  const double a = double(pos) * f.d;
  const double k = rint(a * (32.0 / 3.14159265358979323846));
  double r = fma(-k, kPio32D1, a);
  r = fma(-k, kPio32D2, r);
  const float rh = float(r);
  const float rl = float(r - double(rh));
  const long long km = (long long)k;
  return sincos_from_remainder(rh, rl, int(km & 63), tab);
}

// u_a * c + sign * u_b * s with c = (ch, cl), s = (sh, sl), accurate to about
// 2^-23 of the result even when the two products cancel: p2 = RN(u_b * sh)
// with its exact error e2 (FMA); u_a * ch - p2 is formed exactly inside one
// FMA and rounded once; the small terms are added last.
__device__ __forceinline__ float rotate(float ua, float ub, float ch, float cl, float sh, float sl,
                                        float sign) {
  const float p2 = __fmul_rn(ub, sh);
  const float e2 = fmaf(ub, sh, -p2);
  const float t0 = fmaf(ua, ch, sign * p2);  // ua*ch + sign*p2, one rounding
  return t0 + (sign * e2 + (ua * cl + sign * (ub * sl)));
}

__device__ __forceinline__ void unpack8(const uint32_t (&w)[4], float (&x)[8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = bf16_lo_to_f32(w[j]);
    x[2 * j + 1] = bf16_hi_to_f32(w[j]);
  }
}

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 2;  // two CTAs per SM interleave their load / table / row phases
constexpr int kMaxRowsPerThread = 4;
constexpr int kTableEntries = 2048;  // sin/cos entries per pass: tokens x rotary_dim/2

// Tokens per pass for a head_dim/rotary/heads shape: bounded by the table and
// by 16 rows per thread.
__host__ __device__ inline uint32_t tokens_per_pass(uint32_t head_dim, uint32_t rotary_dim, uint32_t num_kv_heads) {
  const uint32_t rows_per_pass = (kThreads / (head_dim / 8)) * kMaxRowsPerThread;
  uint32_t t = kTableEntries / (rotary_dim / 2);
  const uint32_t by_rows = rows_per_pass / num_kv_heads;
  if (by_rows < t) t = by_rows;
  return t < 1 ? 1 : t;
}

// kFp8Out: store E4M3(o * inv_scale) (saturating, RNE) instead of BF16(o).
// kMrope: pair i takes its position from positions / pos_h / pos_w by i % 3.
template <int D, bool kFp8Out, bool kMrope>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) fused_k_norm_rope_kernel(
    const uint16_t* __restrict__ k_in, const uint16_t* __restrict__ k_norm_weight,
    const int32_t* __restrict__ positions, const int32_t* __restrict__ pos_h,
    const int32_t* __restrict__ pos_w, void* __restrict__ k_cache,
    const int64_t* __restrict__ slot_mapping, uint32_t num_tokens, uint32_t num_kv_heads,
    uint32_t rotary_dim, float rms_eps, const __grid_constant__ FreqTable ft, float inv_scale, uint32_t tok_pass) {
  constexpr int kLanes = D / 8;              // lanes per row
  constexpr int kRows = kThreads / kLanes;   // rows per sweep of the CTA
  __shared__ Freq freq[128];
  __shared__ float4 table[kTableEntries];
  __shared__ float4 sincos_pio32[64];  // lanes index it by position: shared, not constant, memory
  if (threadIdx.x < 64) sincos_pio32[threadIdx.x] = kSinCosPio32[threadIdx.x];

  const uint32_t half = rotary_dim / 2;
  if (threadIdx.x < half) freq[threadIdx.x] = ft.f[threadIdx.x];  // visible after the pass's first barrier

  const uint32_t lane = threadIdx.x % kLanes;
  const uint32_t row_in_sweep = threadIdx.x / kLanes;
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

  const uint32_t passes = (num_tokens + tok_pass - 1) / tok_pass;
  for (uint32_t pass = blockIdx.x; pass < passes; pass += gridDim.x) {
    const uint32_t t0 = pass * tok_pass;
    const uint32_t ntok = num_tokens - t0 < tok_pass ? num_tokens - t0 : tok_pass;
    const uint32_t nrows = ntok * num_kv_heads;

    // 1. every load of the pass first: this thread's rows and their slots
    uint2 xa[kMaxRowsPerThread], xb[kMaxRowsPerThread];
    int64_t slot[kMaxRowsPerThread];
    uint32_t tok_of[kMaxRowsPerThread], head_of[kMaxRowsPerThread];  // token in the pass, head
#pragma unroll
    for (int k = 0; k < kMaxRowsPerThread; ++k) {
      const uint32_t row = row_in_sweep + k * kRows;
      xa[k] = xb[k] = make_uint2(0, 0);
      slot[k] = -1;
      tok_of[k] = row / num_kv_heads;
      head_of[k] = row - tok_of[k] * num_kv_heads;
      if (row < nrows) {
        const uint32_t t = t0 + tok_of[k], h = head_of[k];
        const uint16_t* src = k_in + (uint64_t(t) * num_kv_heads + h) * D;
        xa[k] = __ldcs(reinterpret_cast<const uint2*>(src + off_a));
        xb[k] = __ldcs(reinterpret_cast<const uint2*>(src + off_b));
        slot[k] = __ldg(slot_mapping + t);
#ifdef PAGEDKV_DEBUG_BOUNDS
        if (slot[k] >= 0 && !dbg_slot_ok(slot[k])) slot[k] = -1;  // skipped like padding
#endif
      }
    }
    if (pass == blockIdx.x) __syncthreads();  // freq and sincos_pio32 written
    // 2. sin/cos of every (token of the pass, frequency), by all threads.
    // Pair i = 4 l + q (lane l, group q) sits at [token][q][l], so the 16
    // lanes of a row read 16 consecutive entries (no bank conflicts).
    const uint32_t quarter = half >> 2;  // rotary_dim is a multiple of 8
    for (uint32_t e = threadIdx.x; e < ntok * half; e += kThreads) {
      const uint32_t j = e / half, i = e % half;
      const int32_t* pos_src = positions;
      if (kMrope) pos_src = (i % 3 == 0) ? positions : (i % 3 == 1 ? pos_h : pos_w);
      table[j * half + (i & 3) * quarter + (i >> 2)] = rope_sincos(__ldg(pos_src + t0 + j), freq[i], sincos_pio32);
    }
    __syncthreads();

    // 3. normalise, rotate, round once and store every row
#pragma unroll
    for (int k = 0; k < kMaxRowsPerThread; ++k) {
      const uint32_t row = row_in_sweep + k * kRows;
      if (k * kRows >= nrows) break;  // uniform across the CTA
      const bool active = row < nrows;
      float x[8];
      {
        const uint32_t xw[4] = {xa[k].x, xa[k].y, xb[k].x, xb[k].y};
        unpack8(xw, x);
      }
      float ss = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);  // x^2 is exact in binary32
#pragma unroll
      for (int o = kLanes / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      // 1/sqrt(mean + eps): a few-ulp binary32 factor, a relative error on the
      // whole row far below half a BF16 ulp
      const float r = rsqrtf(__fadd_rn(ss * (1.0f / float(D)), rms_eps));
      float u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) u[j] = __fmul_rn(x[j], w[j]);  // exact
      float out[8];
      if (is_pair && active) {
        const float4* tb = &table[tok_of[k] * half + lane];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 sc = tb[q * quarter];  // pair 4 lane + q: {sin_hi, sin_lo, cos_hi, cos_lo}
          out[q] = rotate(u[q], u[4 + q], sc.z, sc.w, sc.x, sc.y, -1.0f);
          out[4 + q] = rotate(u[4 + q], u[q], sc.z, sc.w, sc.x, sc.y, 1.0f);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) out[j] = u[j];
      }
      if (active && slot[k] >= 0) {
        if constexpr (kFp8Out) {
          // no BF16 rounding: the binary32 result times inv_scale, cast once
          const float rs = __fmul_rn(r, inv_scale);
          uint32_t codes[2];
#pragma unroll
          for (int j = 0; j < 2; ++j)
            codes[j] = uint32_t(f32x2_to_e4m3x2_satfinite(__fmul_rn(out[4 * j], rs), __fmul_rn(out[4 * j + 1], rs))) |
                       (uint32_t(f32x2_to_e4m3x2_satfinite(__fmul_rn(out[4 * j + 2], rs),
                                                           __fmul_rn(out[4 * j + 3], rs))) << 16);
          uint8_t* dst = static_cast<uint8_t*>(k_cache) + (uint64_t(slot[k]) * num_kv_heads + head_of[k]) * D;
          *reinterpret_cast<uint32_t*>(dst + off_a) = codes[0];
          *reinterpret_cast<uint32_t*>(dst + off_b) = codes[1];
        } else {
          uint32_t packed[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            packed[j] = f32x2_to_bf16x2(__fmul_rn(out[2 * j], r), __fmul_rn(out[2 * j + 1], r));
          uint16_t* dst = static_cast<uint16_t*>(k_cache) + (uint64_t(slot[k]) * num_kv_heads + head_of[k]) * D;
          *reinterpret_cast<uint2*>(dst + off_a) = make_uint2(packed[0], packed[1]);
          *reinterpret_cast<uint2*>(dst + off_b) = make_uint2(packed[2], packed[3]);
        }
      }
    }
    __syncthreads();  // the next pass rewrites the table
  }
}

}  // namespace

template <int D>
static void launch_d(bool fp8_out, bool mrope, unsigned blocks, cudaStream_t stream, const uint16_t* k_in,
                     const uint16_t* w, const int32_t* pos, const int32_t* pos_h, const int32_t* pos_w, void* cache,
                     const int64_t* slots, uint32_t n, uint32_t H, uint32_t R, float eps, const FreqTable& ft,
                     float inv_scale, uint32_t tok_pass) {
  if (fp8_out)
    fused_k_norm_rope_kernel<D, true, false><<<blocks, kThreads, 0, stream>>>(
        k_in, w, pos, pos_h, pos_w, cache, slots, n, H, R, eps, ft, inv_scale, tok_pass);
  else if (mrope)
    fused_k_norm_rope_kernel<D, false, true><<<blocks, kThreads, 0, stream>>>(
        k_in, w, pos, pos_h, pos_w, cache, slots, n, H, R, eps, ft, inv_scale, tok_pass);
  else
    fused_k_norm_rope_kernel<D, false, false><<<blocks, kThreads, 0, stream>>>(
        k_in, w, pos, pos_h, pos_w, cache, slots, n, H, R, eps, ft, inv_scale, tok_pass);
}

cudaError_t launch_fused_k_norm_rope(const uint16_t* k_in, const uint16_t* k_norm_weight,
                                     const int32_t* positions, const int32_t* pos_h, const int32_t* pos_w,
                                     void* k_cache, bool fp8_out, float inv_scale,
                                     const int64_t* slot_mapping, uint32_t num_tokens,
                                     uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                     float rms_eps, float theta, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  const uint32_t tok_pass = tokens_per_pass(head_dim, rotary_dim, num_kv_heads);
  const uint64_t passes = (uint64_t(num_tokens) + tok_pass - 1) / tok_pass;
  uint64_t blocks = uint64_t(dev.num_sms) * kCtasPerSm;  // persistent
  if (passes < blocks) blocks = passes;
  const bool mrope = pos_h != nullptr;
  // theta^(-2i/R) in binary64, split into three binary32 parts
  FreqTable ft{};
  const double c = -2.0 * log2(double(theta)) / double(rotary_dim);
  for (uint32_t i = 0; i < rotary_dim / 2 && i < 128; ++i) {
    const double f = exp2(c * double(i));
    Freq& e = ft.f[i];
    e.h = float(f);
    e.m = float(f - double(e.h));
    e.l = float(f - double(e.h) - double(e.m));
    e.pad = 0.0f;
    e.d = f;
  }
  switch (head_dim) {
    case 64:
      launch_d<64>(fp8_out, mrope, unsigned(blocks), stream, k_in, k_norm_weight, positions, pos_h, pos_w, k_cache,
                   slot_mapping, num_tokens, num_kv_heads, rotary_dim, rms_eps, ft, inv_scale, tok_pass);
      break;
    case 128:
      launch_d<128>(fp8_out, mrope, unsigned(blocks), stream, k_in, k_norm_weight, positions, pos_h, pos_w, k_cache,
                    slot_mapping, num_tokens, num_kv_heads, rotary_dim, rms_eps, ft, inv_scale, tok_pass);
      break;
    case 256:
      launch_d<256>(fp8_out, mrope, unsigned(blocks), stream, k_in, k_norm_weight, positions, pos_h, pos_w, k_cache,
                    slot_mapping, num_tokens, num_kv_heads, rotary_dim, rms_eps, ft, inv_scale, tok_pass);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

#ifdef PAGEDKV_DEBUG_BOUNDS
PAGEDKV_DEBUG_UNIT(fused_k)
#endif

}  // namespace pagedkv
