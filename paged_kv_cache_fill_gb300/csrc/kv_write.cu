// Slot filling and the BF16 / V-only / FP8-K / FP8 K+V cache writes.
//
// [kv_cache.rs] `fill_slots_from_block_table`, `reshape_and_cache` (BF16),
// `reshape_and_cache_flash_v_only`, `reshape_and_cache_fp8` (K and V as
// k / k_scale and v / v_scale in E4M3); [kv_cache_fp8k.rs] module
// invariants (K stored as k / k_scale in E4M3).
//
// The writes are pure HBM streams: every token's row is read once and
// written once. A warp owns one token at a time and moves its K and V rows as
// 16-byte vectors, several per lane in flight before any store, with enough
// resident warps per SM to keep ~100+ KB of loads outstanding. The grid is a
// fixed multiple of the SM count and warps stride over tokens.
#include "internal.h"

namespace pagedkv {

// ------------------------------------------------------------ slot filling
__global__ void __launch_bounds__(256) fill_slots_kernel(int64_t* __restrict__ slots,
                                                         const int32_t* __restrict__ block_table,
                                                         uint32_t start_pos, uint32_t count,
                                                         uint32_t block_size) {
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += gridDim.x * blockDim.x) {
    const uint64_t p = uint64_t(start_pos) + i;
    const int64_t block = __ldg(block_table + p / block_size);
#ifdef PAGEDKV_DEBUG_BOUNDS
    if (block >= 0) dbg_block_ok(block);  // flagged here; the write skips the slot it gives
#endif
    slots[i] = block * int64_t(block_size) + int64_t(p % block_size);
  }
}

cudaError_t launch_fill_slots(int64_t* slots, const int32_t* block_table, uint32_t start_pos,
                              uint32_t count, uint32_t block_size, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  uint32_t blocks = (count + 255) / 256;
  blocks = blocks < uint32_t(dev.num_sms * 8) ? blocks : uint32_t(dev.num_sms * 8);
  fill_slots_kernel<<<blocks, 256, 0, stream>>>(slots, block_table, start_pos, count, block_size);
  return cudaGetLastError();
}

// ------------------------------------------------------------ row copies
// Copy token rows to their slots. `src1`/`dst1` null means V-only (one
// tensor). V is uint4 (16-byte vectors) when every row start and the row
// length are 16-byte aligned, else uint16_t (one BF16 element). Row lengths
// and strides are in units of V.
template <typename V, int kUnroll>
__global__ void __launch_bounds__(256) copy_rows_kernel(const V* __restrict__ src0,
                                                        const V* __restrict__ src1,
                                                        V* __restrict__ dst0, V* __restrict__ dst1,
                                                        const int64_t* __restrict__ slot_mapping,
                                                        uint32_t num_tokens, uint32_t row_vecs,
                                                        uint32_t stride0_vecs,
                                                        uint32_t stride1_vecs) {
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t num_warps = (gridDim.x * blockDim.x) >> 5;
  const bool two = src1 != nullptr;
  for (uint32_t t = warp; t < num_tokens; t += num_warps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
#ifdef PAGEDKV_DEBUG_BOUNDS
    if (!dbg_slot_ok(slot)) continue;
#endif
    const V* s0 = src0 + size_t(t) * stride0_vecs;
    const V* s1 = two ? src1 + size_t(t) * stride1_vecs : nullptr;
    V* d0 = dst0 + size_t(slot) * row_vecs;
    V* d1 = two ? dst1 + size_t(slot) * row_vecs : nullptr;
    for (uint32_t base = lane; base < row_vecs; base += 32u * kUnroll) {
      V a[kUnroll], b[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t c = base + 32u * u;
        if (c < row_vecs) {
          a[u] = __ldcs(s0 + c);
          if (two) b[u] = __ldcs(s1 + c);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t c = base + 32u * u;
        if (c < row_vecs) {
          d0[c] = a[u];
          if (two) d1[c] = b[u];
        }
      }
    }
  }
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static uint32_t copy_grid(const DeviceInfo& dev, uint32_t num_tokens) {
  // 8 warps per block; at most 8 blocks per SM resident, one token per warp.
  uint32_t blocks = (num_tokens + 7) / 8;
  const uint32_t cap = uint32_t(dev.num_sms) * 8;
  return blocks < cap ? blocks : cap;
}

cudaError_t launch_copy_rows(const uint16_t* src0, const uint16_t* src1, uint16_t* dst0,
                             uint16_t* dst1, const int64_t* slot_mapping, uint32_t num_tokens,
                             uint32_t row_elems, uint32_t stride0, uint32_t stride1,
                             cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  const uint32_t blocks = copy_grid(dev, num_tokens);
  const bool vec = (row_elems % 8 == 0) && (stride0 % 8 == 0) && (!src1 || stride1 % 8 == 0) &&
                   aligned16(src0) && aligned16(dst0) && (!src1 || (aligned16(src1) && aligned16(dst1)));
  if (vec) {
    copy_rows_kernel<uint4, 4><<<blocks, 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(src0), reinterpret_cast<const uint4*>(src1),
        reinterpret_cast<uint4*>(dst0), reinterpret_cast<uint4*>(dst1), slot_mapping, num_tokens,
        row_elems / 8, stride0 / 8, stride1 / 8);
  } else {
    copy_rows_kernel<uint16_t, 8><<<blocks, 256, 0, stream>>>(src0, src1, dst0, dst1, slot_mapping,
                                                             num_tokens, row_elems, stride0,
                                                             stride1);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ FP8 writes
// K (and V when it is FP8 too): 8 BF16 in (16 B) -> 8 E4M3 out (8 B) per
// vector; the quotient is the IEEE binary32 division (correctly rounded),
// then one saturating RNE conversion. A BF16 V is a 16-byte copy.
//
// The correctly rounded quotient comes from one of two routes. The exact
// division __fdiv_rn works for any scale. The division-free route is for
// scales s in [2^-60, 2^60]. It takes y = RN(1/s) once per thread
// (__frcp_rn), q0 = RN(x*y), and two residual corrections
// q' = RN(q + RN(x - s*q)*y); each residual is exact by FMA.
// The first correction leaves q1 within one ulp of x/s, since its error
// before rounding is |q0 - x/s| * |1 - s*y| <= 2^-24 |q0 - x/s|. From q1,
// Markstein's theorem gives RN(x/s) exactly, provided no intermediate
// underflows or overflows (P. Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990;
// J.-M. Muller et al., Handbook of Floating-Point Arithmetic, division with
// an FMA). That holds while |q0| lies in [2^-20, 2^20] and s in
// [2^-60, 2^60]. Outside that range of |q0| the quotient is below 2^-10 or
// above 448, so q0 gives the same E4M3 code (+-0, or +-448 when
// saturated), as do NaN and infinite inputs.
constexpr float kFastScaleMin = 0x1p-60f, kFastScaleMax = 0x1p60f;

__device__ __forceinline__ float quotient_rn(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, x), y, q0);
  const float q2 = __fmaf_rn(__fmaf_rn(-q1, s, x), y, q1);
  const float a = fabsf(q0);
  return (a >= 0x1p-20f && a <= 0x1p20f) ? q2 : q0;
}

template <bool kFast>
__device__ __forceinline__ float quotient(float x, float s, float y) {
  if constexpr (kFast)
    return quotient_rn(x, s, y);
  else
    return __fdiv_rn(x, s);
}

template <bool kFast>
__device__ __forceinline__ uint2 encode8(uint4 k, float scale, float recip) {
  const uint32_t w[4] = {k.x, k.y, k.z, k.w};
  uint32_t out[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float q0 = quotient<kFast>(bf16_lo_to_f32(w[2 * j]), scale, recip);
    const float q1 = quotient<kFast>(bf16_hi_to_f32(w[2 * j]), scale, recip);
    const float q2 = quotient<kFast>(bf16_lo_to_f32(w[2 * j + 1]), scale, recip);
    const float q3 = quotient<kFast>(bf16_hi_to_f32(w[2 * j + 1]), scale, recip);
    out[j] = uint32_t(f32x2_to_e4m3x2_satfinite(q0, q1)) |
             (uint32_t(f32x2_to_e4m3x2_satfinite(q2, q3)) << 16);
  }
  return make_uint2(out[0], out[1]);
}

__device__ __forceinline__ uint8_t encode1(uint16_t k, float k_scale) {
  const float q = __fdiv_rn(__uint_as_float(uint32_t(k) << 16), k_scale);
  return uint8_t(f32x2_to_e4m3x2_satfinite(q, 0.0f) & 0xFF);
}

// kFp8V: V is quantised like K (v / v_scale, 16 B in -> 8 B out) instead of
// copied. kFast: the division-free quotient (both scales in its range).
template <int kUnroll, bool kFp8V, bool kFast>
__global__ void __launch_bounds__(256) write_fp8_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value, uint2* __restrict__ k_cache,
    void* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, uint32_t num_tokens,
    uint32_t row_vecs, uint32_t kstride_vecs, uint32_t vstride_vecs, float k_scale, float v_scale) {
  const float k_recip = kFast ? __frcp_rn(k_scale) : 0.0f;
  const float v_recip = kFast ? __frcp_rn(v_scale) : 0.0f;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t num_warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t t = warp; t < num_tokens; t += num_warps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
#ifdef PAGEDKV_DEBUG_BOUNDS
    if (!dbg_slot_ok(slot)) continue;
#endif
    const uint4* ks = key + size_t(t) * kstride_vecs;
    const uint4* vs = value + size_t(t) * vstride_vecs;
    uint2* kd = k_cache + size_t(slot) * row_vecs;
    for (uint32_t base = lane; base < row_vecs; base += 32u * kUnroll) {
      uint4 a[kUnroll], b[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t c = base + 32u * u;
        if (c < row_vecs) {
          a[u] = __ldcs(ks + c);
          b[u] = __ldcs(vs + c);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t c = base + 32u * u;
        if (c < row_vecs) {
          kd[c] = encode8<kFast>(a[u], k_scale, k_recip);
          if constexpr (kFp8V)
            static_cast<uint2*>(v_cache)[size_t(slot) * row_vecs + c] = encode8<kFast>(b[u], v_scale, v_recip);
          else
            static_cast<uint4*>(v_cache)[size_t(slot) * row_vecs + c] = b[u];
        }
      }
    }
  }
}

// Unaligned fallback: one element per lane step.
template <bool kFp8V>
__global__ void __launch_bounds__(256) write_fp8_scalar_kernel(
    const uint16_t* __restrict__ key, const uint16_t* __restrict__ value,
    uint8_t* __restrict__ k_cache, void* __restrict__ v_cache,
    const int64_t* __restrict__ slot_mapping, uint32_t num_tokens, uint32_t row_elems,
    uint32_t key_stride, uint32_t value_stride, float k_scale, float v_scale) {
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t num_warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t t = warp; t < num_tokens; t += num_warps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
#ifdef PAGEDKV_DEBUG_BOUNDS
    if (!dbg_slot_ok(slot)) continue;
#endif
    for (uint32_t c = lane; c < row_elems; c += 32) {
      const size_t dst = size_t(slot) * row_elems + c;
      k_cache[dst] = encode1(key[size_t(t) * key_stride + c], k_scale);
      const uint16_t v = value[size_t(t) * value_stride + c];
      if constexpr (kFp8V)
        static_cast<uint8_t*>(v_cache)[dst] = encode1(v, v_scale);
      else
        static_cast<uint16_t*>(v_cache)[dst] = v;
    }
  }
}

template <bool kFp8V>
static void launch_write_fp8_t(bool vec, uint32_t blocks, cudaStream_t stream, const uint16_t* key,
                               const uint16_t* value, uint8_t* k_cache_fp8, void* v_cache,
                               const int64_t* slot_mapping, uint32_t num_tokens, uint32_t row_elems,
                               uint32_t key_stride, uint32_t value_stride, float k_scale, float v_scale) {
  auto in_fast_range = [](float sc) { return sc >= kFastScaleMin && sc <= kFastScaleMax; };
  const bool fast = in_fast_range(k_scale) && (!kFp8V || in_fast_range(v_scale));
  if (vec && fast)
    write_fp8_kernel<4, kFp8V, true><<<blocks, 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(key), reinterpret_cast<const uint4*>(value),
        reinterpret_cast<uint2*>(k_cache_fp8), v_cache, slot_mapping, num_tokens, row_elems / 8, key_stride / 8,
        value_stride / 8, k_scale, v_scale);
  else if (vec)
    write_fp8_kernel<4, kFp8V, false><<<blocks, 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(key), reinterpret_cast<const uint4*>(value),
        reinterpret_cast<uint2*>(k_cache_fp8), v_cache, slot_mapping, num_tokens, row_elems / 8, key_stride / 8,
        value_stride / 8, k_scale, v_scale);
  else
    write_fp8_scalar_kernel<kFp8V><<<blocks, 256, 0, stream>>>(key, value, k_cache_fp8, v_cache, slot_mapping,
                                                               num_tokens, row_elems, key_stride, value_stride,
                                                               k_scale, v_scale);
}

cudaError_t launch_write_fp8(const uint16_t* key, const uint16_t* value, uint8_t* k_cache_fp8, void* v_cache,
                             bool fp8_v, const int64_t* slot_mapping, uint32_t num_tokens, uint32_t row_elems,
                             uint32_t key_stride, uint32_t value_stride, float k_scale, float v_scale,
                             cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  const uint32_t blocks = copy_grid(dev, num_tokens);
  const uintptr_t v_align = fp8_v ? 7u : 15u;
  const bool vec = (row_elems % 8 == 0) && (key_stride % 8 == 0) && (value_stride % 8 == 0) &&
                   aligned16(key) && aligned16(value) && (reinterpret_cast<uintptr_t>(v_cache) & v_align) == 0 &&
                   (reinterpret_cast<uintptr_t>(k_cache_fp8) & 7u) == 0;
  if (fp8_v)
    launch_write_fp8_t<true>(vec, blocks, stream, key, value, k_cache_fp8, v_cache, slot_mapping, num_tokens,
                             row_elems, key_stride, value_stride, k_scale, v_scale);
  else
    launch_write_fp8_t<false>(vec, blocks, stream, key, value, k_cache_fp8, v_cache, slot_mapping, num_tokens,
                              row_elems, key_stride, value_stride, k_scale, v_scale);
  return cudaGetLastError();
}

#ifdef PAGEDKV_DEBUG_BOUNDS
PAGEDKV_DEBUG_UNIT(kv_write)
#endif

}  // namespace pagedkv
