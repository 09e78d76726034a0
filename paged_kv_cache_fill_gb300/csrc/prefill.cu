// Multi-token (chunked-prefill) paged attention over a BF16, an FP8-E4M3-K /
// BF16-V or an FP8-E4M3 K and V paged cache.
//
// [kv_cache.rs] "Batched prefill variants (N tokens)" (a heading only), read
// as: sequence s brings n_s = query_start_loc[s+1] - query_start_loc[s]
// query tokens, the last n_s of its seq_lens[s] cached positions; query j
// (row query_start_loc[s] + j, position P = seq_lens[s] - n_s + j) attends
// positions [start, P], start = max(0, P + 1 - sliding_window) when
// sliding_window > 0, else 0 -- what the paged decode ([kv_cache.rs]
// `paged_decode_attn_fp8`) attends for a sequence of length P + 1. GQA as in
// the decode: query head h reads KV head h / (num_q_heads / num_kv_heads).
//
// GB300 design (tcgen05 / TMEM). Rows are (query token, query head of the
// KV head's group) pairs, token-major, so a CTA's rows -- 128 per
// tcgen05.mma (its M) -- share every K/V tile it loads. One kernel,
// prefill_tc2_kernel, with two 128-row Q tiles per CTA (one tile's
// products cover the other's drain in the tensor pipe), runs every call.
// A CTA owns one (sequence, KV head, block of 256 rows) item; items run
// longest key range first across all sequences (by a length class of each
// sequence's key range), and the grid holds an upper bound of the item count
// (CTAs past the last item exit at once). The kernel's own comment gives
// its warp roles, TMEM map and barriers.
#include <math.h>

#include "../../include/pagedkv.h"
#include "internal.h"

namespace pagedkv {

__device__ uint32_t g_prefill_error;

namespace {

constexpr int kSub = 16;                // keys per TMA box
constexpr int kTcBM = 128, kTcBN = 128, kTcStages = 2;  // rows per Q tile, keys per K/V tile, ring stages
constexpr float kLog2e = 1.4426950408889634f;

struct PrefillParams {
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;  // query_start_loc
  float* output;
  uint32_t max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, group;
  uint32_t block_size, block_shift, q_stride, sliding_window;
  float score_scale;  // inv_sqrt_d * log2(e) (times k_scale for FP8)
  float out_scale;    // E4M3 V: v_scale (the V codes enter the PV product as they are)
};

// An E4M3 tile [chunk of 128 dims][128 keys][128 B] (head_dim 64: [128
// keys][64 B], 64-byte swizzled) -> the f16 tile [chunk of 64 dims][128
// keys][128 B], 128-byte swizzled; rows at or past `live`
// become zeros. Exact (every E4M3 value is an f16 value). Lane l takes keys
// l, l + 32 (first pass) and l + 64, l + 96 (second). Each pass loads its
// two rows (16 x 16 B) before any store: the stores could alias the loads as
// far as the compiler knows, so interleaving them would serialise every
// load behind the previous unit's stores. A dead row's codes are replaced by
// zeros as loaded (E4M3 0 is f16 0), which costs far fewer instructions than
// selecting every converted word. Not inlined and the passes not unrolled,
// so that the converting warp runs one short body (inlined, unrolled
// converter copies in several warps have stalled a kernel's warps on
// instruction fetch).
template <int D>
__device__ __noinline__ void e4m3_tile_to_f16(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                              int32_t live, uint32_t lane) {
  constexpr uint32_t kUnits = D < 128 ? D / 16 : 8;  // 16-byte units of a source row per chunk
  constexpr uint32_t kSrcChunks = (D + 127) / 128;
  // unit u of key r in source chunk c8
  auto src_unit = [&](uint32_t c8, uint32_t r, uint32_t u) -> const uint4* {
    if constexpr (D == 64) return reinterpret_cast<const uint4*>(src + r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
    else return reinterpret_cast<const uint4*>(src + c8 * (128 * 128) + r * 128 + ((u ^ (r & 7)) << 4));
  };
#pragma unroll 1
  for (uint32_t r0 = 0; r0 < 128u; r0 += 64) {
#pragma unroll
    for (uint32_t c8 = 0; c8 < kSrcChunks; ++c8) {
      uint4 w[2][kUnits];
#pragma unroll
      for (uint32_t k = 0; k < 2; ++k) {
        const uint32_t r = r0 + 32 * k + lane;
        const bool keep = int32_t(r) < live;
#pragma unroll
        for (uint32_t u = 0; u < kUnits; ++u) {
          w[k][u] = *src_unit(c8, r, u);
          if (!keep) w[k][u] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (uint32_t k = 0; k < 2; ++k) {
        const uint32_t r = r0 + 32 * k + lane;
#pragma unroll
        for (uint32_t u = 0; u < kUnits; ++u) {  // 16 dims per 16-byte unit
          const uint32_t ws[4] = {w[k][u].x, w[k][u].y, w[k][u].z, w[k][u].w};
          uint32_t h[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            h[2 * j] = e4m3x2_to_f16x2(uint16_t(ws[j]));
            h[2 * j + 1] = e4m3x2_to_f16x2(uint16_t(ws[j] >> 16));
          }
          // dims 128 c8 + 16 u .. + 15: f16 chunk 2 c8 + u / 4, units 2 (u % 4) and + 1
          const uint32_t c = 2 * c8 + (u >> 2), u0 = 2 * (u & 3);
          uint8_t* drow = dst + c * (128 * 128) + r * 128;
          *reinterpret_cast<uint4*>(drow + ((u0 ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(drow + (((u0 + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
    }
  }
}

struct Item {
  int32_t seq, kv_head, row0, rows;  // rows [row0, row0 + rows) of the sequence's n * group
  int32_t n, qstart, len;            // query tokens, their first row in q, cached positions
};

template <int BM>
__device__ __forceinline__ uint32_t row_blocks(int64_t n, uint32_t group) {
  return uint32_t((n * group + BM - 1) / BM);
}

// Items run longest key range first across all sequences (a CTA launched
// late then runs a short item, so the last wave ends evenly): the order is
// by length class of the sequence's key range, descending, then by
// sequence, then by row block (the last block, with the most keys, first).
// Classes are log-linear in 128-key tiles, eight per octave, so items of one
// class differ in length by at most 1/8.
constexpr uint32_t kLenClasses = 128;

__device__ __forceinline__ uint32_t len_class(uint64_t tiles) {
  if (tiles == 0) return 0;
  const uint32_t msb = 63 - __clzll(tiles);
  const uint32_t frac = uint32_t(msb >= 3 ? tiles >> (msb - 3) : tiles << (3 - msb)) & 7u;
  const uint32_t c = msb * 8 + frac;
  return c < kLenClasses ? c : kLenClasses - 1;
}

// Sequence s's share of the item list: its query tokens n, its items (row
// blocks x KV heads) and the length class of its queries' key range.
// A bad query layout counts as no queries (flagged once, by the caller's
// first pass).
template <int BM>
__device__ __forceinline__ uint32_t seq_items(const PrefillParams& p, uint32_t s, bool flag, int64_t& n,
                                              uint32_t& cls) {
  n = 0;
  cls = 0;
  if (s >= p.num_seqs) return 0;
  const int32_t a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
  n = int64_t(b) - a;
  if (a < 0 || n < 0 || uint32_t(b) > p.num_q_tokens) {
    if (flag) atomicOr(&g_prefill_error, kErrQueryLayout);
    n = 0;
  }
  int64_t L = __ldg(p.seq_lens + s);
  const int64_t cap = int64_t(p.max_blocks_per_seq) << p.block_shift;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  int64_t k_lo = 0;
  if (p.sliding_window > 0 && L - n + 1 - int64_t(p.sliding_window) > 0) k_lo = L - n + 1 - p.sliding_window;
  const int64_t tiles = (L + kTcBN - 1) / kTcBN - k_lo / kTcBN;
  cls = len_class(tiles > 0 ? uint64_t(tiles) : 0);
  return row_blocks<BM>(n, p.group) * p.num_kv_heads;
}

// The item of CTA `target` (seq < 0: none), items of BM rows. Run by one
// warp; `hist` is kLenClasses words of scratch shared memory.
template <int BM>
__device__ Item locate(uint32_t target, const PrefillParams& p, uint32_t lane, uint32_t* hist) {
  Item it{};
  it.seq = -1;
  for (uint32_t c = lane; c < kLenClasses; c += 32) hist[c] = 0;
  __syncwarp();
  // items per length class
  for (uint32_t s = lane; s < p.num_seqs; s += 32) {
    int64_t n;
    uint32_t cls;
    const uint32_t items = seq_items<BM>(p, s, true, n, cls);
    if (items) atomicAdd(&hist[cls], items);
  }
  __syncwarp();
  // the class that holds item `target`, longest class first (lane l of a
  // round takes class c0 + 31 - l)
  uint64_t before = 0;
  int32_t cls_t = -1;
  for (int32_t c0 = int32_t(kLenClasses) - 32; c0 >= 0 && cls_t < 0; c0 -= 32) {
    const uint32_t cnt = hist[uint32_t(c0) + 31 - lane];
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= uint32_t(o)) incl += v;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    if (uint64_t(target) < before + total) {
      const uint32_t rel = uint32_t(target - before);
      const uint32_t sl = __ffs(__ballot_sync(0xffffffffu, incl > rel)) - 1;
      cls_t = c0 + 31 - int32_t(sl);
      before += __shfl_sync(0xffffffffu, incl, sl) - __shfl_sync(0xffffffffu, cnt, sl);
    } else {
      before += total;
    }
  }
  if (cls_t < 0) return it;
  // the sequence of that class, in sequence order, that holds it
  uint64_t rel = uint64_t(target) - before;
  for (uint32_t s0 = 0; s0 < p.num_seqs; s0 += 32) {
    const uint32_t s = s0 + lane;
    int64_t n;
    uint32_t cls;
    uint32_t items = seq_items<BM>(p, s, false, n, cls);
    if (int32_t(cls) != cls_t) items = 0;
    uint32_t incl = items;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= uint32_t(o)) incl += v;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    if (rel < total) {
      const uint32_t sl = __ffs(__ballot_sync(0xffffffffu, incl > uint32_t(rel))) - 1;
      const uint32_t local =
          uint32_t(rel) - (__shfl_sync(0xffffffffu, incl, sl) - __shfl_sync(0xffffffffu, items, sl));
      const int64_t ns = __shfl_sync(0xffffffffu, n, sl);
      const uint32_t nblk = row_blocks<BM>(ns, p.group);
      const uint32_t blk = nblk - 1 - local / p.num_kv_heads;  // longest key range first
      it.seq = int32_t(s0 + sl);
      it.kv_head = int32_t(local % p.num_kv_heads);
      it.row0 = int32_t(blk * BM);
      const int64_t rows_total = ns * p.group;
      it.rows = int32_t(rows_total - it.row0 < BM ? rows_total - it.row0 : BM);
      it.n = int32_t(ns);
      it.qstart = __ldg(p.qsl + it.seq);
      int32_t L = __ldg(p.seq_lens + it.seq);
      if (L < 0) L = 0;
      const int64_t cap = int64_t(p.max_blocks_per_seq) << p.block_shift;
      if (L > cap) {
        L = int32_t(cap);
        if (lane == 0 && it.kv_head == 0) atomicOr(&g_prefill_error, kErrSeqLenClamped);
      }
      it.len = L;
      return it;
    }
    rel -= total;
  }
  return it;
}

constexpr float kRescaleLog2 = 8.0f;  // reference-max slack of the online softmax (base 2)

// ------------------------------------------------- the two-tile kernel
// BF16, E4M3-K / BF16-V (kFp8) or E4M3 K and V (kFp8V) caches. One CTA
// per (sequence, KV head, block of 256 rows): two 128-row Q tiles, A (rows
// 0..127) and B (rows 128..255), share every K/V tile the CTA loads. Each Q tile has its own S/P and O in tensor memory
// (S_A [0, 128), O_A [128, 128 + D), S_B [256, 384), O_B [384, 384 + D)); Q
// lives in shared memory (the S product's A operand). A tile's S product
// writes the columns its P occupied, so it must wait until the tile's PV
// product before it has finished (one thread's tcgen05.mma operations are
// ordered only for the same accumulator); with one Q tile the tensor pipe
// idled through that hand-off and the softmax that follows. Here per K/V
// tile j the MMA thread issues PV_A(j), S_A(j + 1) as soon as PV_A(j) is
// done, then PV_B(j), and S_B(j + 1) as soon as PV_B(j) is done: while one
// tile's softmax runs, the other tile's products keep the pipe busy, and a
// tile's S product never waits behind the other tile's PV product (that
// order measured slower).
// The PV product is one f16 x f16 product: the weights as one f16 rounding
// of 2^7 P (relative error <= 2^-11), every V tile converted to f16 in
// shared memory before it (E4M3 codes exactly; BF16 values times 2^-8,
// exact for 2^-6 <= |v| < 2^24, which the output scale undoes). 384
// threads, three warpgroups:
//   warpgroup 0 (registers cut to tc2_regs_low() with setmaxnreg):
//     warp 0      TMA producer of 128-key K tiles, warp 2 of V tiles, each a
//                 2-stage ring whose stage is free once the MMA thread's
//                 commit after its last reader has arrived on its empty
//                 barrier; with an E4M3 V cache warp 2 converts each V
//                 tile into its f16 stage before it loads the next: at
//                 head_dim 128 in place, the tile loaded into the upper
//                 half of its f16 stage (E4M3 row r lies where the f16
//                 tile's second chunk puts row r, and a lane reads the
//                 whole row before it writes), at head_dim 64 from a ring
//                 of its own;
//     warp 1      owns TMEM (all 512 columns) and issues every tcgen05.mma;
//     warp 3      with an E4M3 K cache: turns each E4M3 K tile, loaded by
//                 warp 0 into a ring of its own, into the f16 K stage the
//                 S product reads (exact); with a BF16 K cache: converts
//                 the second half of each BF16 V tile (below);
//   warpgroups 1, 2 (registers raised to tc2_regs_high()): the softmax of tile
//     A and of tile B, one thread per row (TMEM lane) over all 128 keys of a
//     tile, so no row is shared between threads; they also write the Q rows
//     (with an E4M3 K cache: as f16, the row scaled by a power of two that
//     the row's score scale undoes) and, with a
//     BF16 V cache, convert V tile j + 1 in place right after publishing
//     their P of tile j, off the path of that tile's PV product (each
//     warpgroup half of it with an E4M3 K cache; with a BF16 K cache a
//     quarter each, warp 3 the other half: one warp converting a whole
//     tile per cycle became the serial path). At the end each thread stages its O / l row in the
//     then free Q tiles and K/V stages and stores it with one bulk copy
//     (direct stores of a row per thread wrote 16 bytes per 32-byte sector
//     and took ~3 us per CTA).
constexpr int kTc2Rows = 256;
// registers per thread of warpgroup 0 and of the softmax warpgroups after
// setmaxnreg (per variant, the split that ptxas fits without spills or the
// faster one measured): 128 x low + 256 x high <= 384 x 168 at launch
template <bool kFp8V>
__host__ __device__ constexpr uint32_t tc2_regs_low() { return kFp8V ? 72u : 96u; }
template <bool kFp8V>
__host__ __device__ constexpr uint32_t tc2_regs_high() { return kFp8V ? 208u : 192u; }
static_assert(128 * tc2_regs_low<false>() + 256 * tc2_regs_high<false>() <= 384 * 168, "register split");
static_assert(128 * tc2_regs_low<true>() + 256 * tc2_regs_high<true>() <= 384 * 168, "register split");

template <int D, bool kFp8, bool kFp8V>
struct Tc2Layout {  // byte offsets from the 1024-aligned shared base
  static constexpr uint32_t kChunks = D / 64;
  static constexpr uint32_t kQBytes = kChunks * kTcBM * 128;  // one Q tile [chunk][128 rows][128 B]
  static constexpr uint32_t kQ0 = 0;
  static constexpr uint32_t kKBytes = kChunks * kTcBN * 128;  // [chunk][128 keys][128 B]
  static constexpr uint32_t kStage0 = 2 * kQBytes;
  static constexpr uint32_t kStageBytes = 2 * kKBytes;        // K (f16 when converted), then V
  // E4M3 K as loaded, one ring of stages: [chunk of 128 dims][128 keys][128
  // B], or for head_dim 64 [128 keys][64 B] (kE4Row bytes of a key's row)
  static constexpr uint32_t kE4Row = D < 128 ? D : 128;
  static constexpr uint32_t kK8Chunks = (D + 127) / 128;
  static constexpr uint32_t kK8Bytes = kFp8 ? kK8Chunks * kTcBN * kE4Row : 0;
  static constexpr uint32_t kK80 = kStage0 + kTcStages * kStageBytes;
  // E4M3 V as loaded: at head_dim 128 a V tile lands inside its f16 V stage
  // (converted in place, no ring of its own: the shared memory is full);
  // at head_dim 64 in a ring of its own, [128 keys][64 B]
  static constexpr bool kV8Ring = kFp8V && D == 64;
  static constexpr uint32_t kV8Bytes = kV8Ring ? kTcBN * kE4Row : 0;
  static constexpr uint32_t kV80 = kK80 + kTcStages * kK8Bytes;
  static constexpr uint32_t kBytes = kV80 + kTcStages * kV8Bytes;
  static constexpr uint32_t kTmemCols = 512;
  // tile t's S/P columns and O columns
  static __device__ __forceinline__ constexpr uint32_t s_col(uint32_t t) { return t << 8; }
  static __device__ __forceinline__ constexpr uint32_t o_col(uint32_t t) { return 128u + (t << 8); }
};

template <int D, bool kFp8, bool kFp8V>
__global__ void __launch_bounds__(32 * 12, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const PrefillParams p) {
  static_assert(kFp8 || !kFp8V, "an E4M3 V cache comes with an E4M3 K cache");
  using Lay = Tc2Layout<D, kFp8, kFp8V>;
  constexpr uint32_t kChunks = Lay::kChunks;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  __shared__ uint64_t k_full[kTcStages], v_full[kTcStages], k_empty[kTcStages], v_empty[kTcStages];
  __shared__ uint64_t k8_full[kTcStages], k8_empty[kTcStages];  // E4M3 K: loaded, read by the converter
  __shared__ uint64_t v8_full[kTcStages];                        // E4M3 V: loaded
  __shared__ uint64_t s_full[2], p_full[2], o_full[2];  // per Q tile
  __shared__ uint64_t q_full, mma_done;
  __shared__ uint32_t tmem_base_s;
  __shared__ Item s_item;

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&k_full[s], kFp8 ? 32 : 1);  // E4M3 K: the converter warp's arrivals
      // once the tile is f16: E4M3 V, warp 2's lanes; BF16 V, the eight
      // softmax warps (and warp 3 with a BF16 K cache)
      mbar_init(&v_full[s], kFp8V ? 32 : (kFp8 ? 8 : 9));
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&k8_full[s], 1);
      mbar_init(&k8_empty[s], 32);
      mbar_init(&v8_full[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], kTcBM);
      mbar_init(&o_full[t], 1);
    }
    mbar_init(&q_full, 2 * kTcBM);
    mbar_init(&mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    const Item it = locate<kTc2Rows>(blockIdx.x, p, lane, reinterpret_cast<uint32_t*>(smem));  // (free until the Q rows)
    if (lane == 0) s_item = it;
  }
  __syncthreads();
  const Item it = s_item;
  if (it.seq < 0) return;
  if (warp == 1) tmem_alloc(&tmem_base_s, Lay::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  const int32_t g = int32_t(p.group);
  const bool two = it.rows > kTcBM;  // tile B holds rows
  const int32_t pos_first = it.len - it.n + it.row0 / g;
  const int32_t pos_last = it.len - it.n + (it.row0 + it.rows - 1) / g;
  const int32_t k_hi = pos_last + 1;  // keys [k_lo, k_hi)
  const int32_t W = int32_t(p.sliding_window);
  int32_t k_lo = 0;
  if (W > 0 && pos_first + 1 - W > 0) k_lo = pos_first + 1 - W;
  const int32_t t_begin = k_lo / kTcBN;
  const int32_t t_end = k_hi > 0 ? (k_hi + kTcBN - 1) / kTcBN : t_begin;
  const int32_t T = t_end - t_begin;

  if (warp < 4) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(tc2_regs_low<kFp8V>()));
   if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == 0;
    const bool e4m3 = is_k ? kFp8 : kFp8V;  // this tensor's cache holds E4M3 codes
    const bool self_converts = kFp8V && !is_k;
    const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
    uint64_t* full = is_k ? (kFp8 ? k8_full : k_full) : v8_full;  // V: converted before v_full
    uint64_t* empty = is_k ? (kFp8 ? k8_empty : k_empty) : v_empty;
    const uint32_t chunks = e4m3 ? Lay::kK8Chunks : kChunks;
    const uint32_t row_bytes = e4m3 ? Lay::kE4Row : 128u;  // of a key's row per box
    // E4M3 V tile j -> its f16 stage (in place at head_dim 128, from its own
    // ring at head_dim 64); rows at or past the item's last key (not
    // loaded, or positions past every query) become zeros
    auto convert_v = [&](int32_t j) -> bool {
      const uint32_t sj = uint32_t(j) % kTcStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&v8_full[sj], uint32_t(j / kTcStages) & 1))) return false;
      uint8_t* vt = smem + Lay::kStage0 + sj * Lay::kStageBytes + Lay::kKBytes;  // [chunk][128 keys][128 B]
      const int32_t live = k_hi - (t_begin + j) * kTcBN;
      if constexpr (Lay::kV8Ring) {
        e4m3_tile_to_f16<D>(smem + Lay::kV80 + sj * Lay::kV8Bytes, vt, live, lane);
      } else {
#pragma unroll 1
        for (uint32_t r = lane; r < uint32_t(kTcBN); r += 32) {
          uint8_t* row1 = vt + kTcBN * 128 + r * 128;  // the E4M3 row, and the f16 tile's chunk 1 row r
          uint4 w[8];
#pragma unroll
          for (uint32_t u = 0; u < 8; ++u) w[u] = *reinterpret_cast<const uint4*>(row1 + ((u ^ (r & 7)) << 4));
          if (int32_t(r) >= live) {
#pragma unroll
            for (uint32_t u = 0; u < 8; ++u) w[u] = make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (uint32_t u = 0; u < 8; ++u) {  // dims 16 u ..: f16 chunk u / 4, units 2 (u % 4) and + 1
            const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              h[2 * q] = e4m3x2_to_f16x2(uint16_t(ws[q]));
              h[2 * q + 1] = e4m3x2_to_f16x2(uint16_t(ws[q] >> 16));
            }
            const uint32_t u0 = 2 * (u & 3);
            uint8_t* drow = vt + (u >> 2) * (kTcBN * 128) + r * 128;
            *reinterpret_cast<uint4*>(drow + ((u0 ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(drow + (((u0 + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        }
      }
      fence_async_smem();
      mbar_arrive(&v_full[sj]);
      return true;
    };
    tma_prefetch_desc(map);
    const int32_t* table = p.block_tables + uint64_t(it.seq) * p.max_blocks_per_seq;
    bool ok = true;
    int32_t issued = 0;
    for (int32_t i = 0; i < T && ok; ++i) {
      // E4M3 V: the tile before this one is converted as soon as it has
      // landed, before this tile's stage is waited for (PV two tiles back)
      if (self_converts && i >= 1 && !(ok = convert_v(i - 1))) break;
      const uint32_t st = uint32_t(i) % kTcStages;
      const int32_t key0 = (t_begin + i) * kTcBN + int32_t(lane) * kSub;
      const bool mine = lane < uint32_t(kTcBN / kSub) && key0 < k_hi;
      const int32_t block_id = mine ? __ldg(table + (key0 >> p.block_shift)) : 0;
      // stage st was last filled for tile i - 2: free once its last reader is done
      if (lane == 0 && i >= kTcStages && !mbar_wait(&empty[st], uint32_t((i - kTcStages) / kTcStages) & 1))
        ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t loaded = __popc(__ballot_sync(0xffffffffu, mine));
      if (lane == 0) mbar_arrive_expect_tx(&full[st], loaded * chunks * (kSub * row_bytes));
      __syncwarp();
      if (mine) {
#ifdef PAGEDKV_DEBUG_BOUNDS
        const int32_t slot0 =
            ((dbg_block_ok(block_id) ? block_id : 0) << p.block_shift) + (key0 & int32_t(p.block_size - 1));
#else
        const int32_t slot0 = (block_id << p.block_shift) + (key0 & int32_t(p.block_size - 1));
#endif
        // E4M3 K: its own ring; E4M3 V: the upper half of its f16 stage
        // (head_dim 128) or its own ring (head_dim 64)
        uint8_t* dst =
            smem +
            (is_k ? (e4m3 ? Lay::kK80 + st * Lay::kK8Bytes : Lay::kStage0 + st * Lay::kStageBytes)
                  : (Lay::kV8Ring ? Lay::kV80 + st * Lay::kV8Bytes
                                  : Lay::kStage0 + st * Lay::kStageBytes + Lay::kKBytes + (e4m3 ? kTcBN * 128u : 0u))) +
            lane * (kSub * row_bytes);
        for (uint32_t c = 0; c < chunks; ++c)
          tma_load_3d(dst + c * (kTcBN * row_bytes), map, 0, slot0, it.kv_head * chunks + c, &full[st]);
      }
      issued = i + 1;
    }
    if (self_converts && ok && T > 0) ok = convert_v(T - 1);
    if (!ok) {
      // a wait gave up: let this warp's loads still in flight land (bounded)
      if (lane == 0) atomicOr(&g_prefill_error, kErrWaitTimeout);
      for (int32_t j = issued > kTcStages ? issued - kTcStages : 0; j < issued; ++j)
        mbar_wait(&full[uint32_t(j) % kTcStages], uint32_t(j / kTcStages) & 1);
    }
   } else if (!kFp8 && warp == 3) {
    // ------------------------------------------------------------ BF16 V
    // With a BF16 K cache this warp is free: it turns the second half of
    // each BF16 V tile into f16 (the same rounding as the softmax warps'
    // quarters, below), leaving the softmax warps a quarter each.
    bool ok = true;
    const F2 down = f2_make(0.00390625f, 0.00390625f);
    constexpr uint32_t kHalf = uint32_t(kTcBN) * kChunks * 4;
    for (int32_t j = 0; j < T && ok; ++j) {
      const uint32_t sj = uint32_t(j) % kTcStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&v8_full[sj], uint32_t(j / kTcStages) & 1));
      if (!ok) break;
      uint4* units = reinterpret_cast<uint4*>(smem + Lay::kStage0 + sj * Lay::kStageBytes + Lay::kKBytes);
      const int32_t live = k_hi - (t_begin + j) * kTcBN;
#pragma unroll 1
      for (uint32_t e0 = kHalf; e0 < 2 * kHalf; e0 += 8 * 32) {
        uint4 w[8];
#pragma unroll
        for (uint32_t u = 0; u < 8; ++u) w[u] = units[e0 + 32 * u + lane];
#pragma unroll
        for (uint32_t u = 0; u < 8; ++u) {
          uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = f2_split(
                f2_mul(f2_make(__uint_as_float(ws[q] << 16), __uint_as_float(ws[q] & 0xffff0000u)), down));
            ws[q] = f32x2_to_f16x2(f.x, f.y);
          }
          w[u] = make_uint4(ws[0], ws[1], ws[2], ws[3]);
        }
        if (live < kTcBN) {
#pragma unroll
          for (uint32_t u = 0; u < 8; ++u)
            if (int32_t(((e0 + 32 * u + lane) >> 3) % uint32_t(kTcBN)) >= live) w[u] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (uint32_t u = 0; u < 8; ++u) units[e0 + 32 * u + lane] = w[u];
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&v_full[sj]);
    }
    if (!ok && lane == 0) atomicOr(&g_prefill_error, kErrWaitTimeout);
   } else if (kFp8 && warp == 3) {
    // ------------------------------------------------------------ E4M3 -> f16
    // Each loaded E4M3 K tile into the f16 K stage the S products read
    // (exact: every E4M3 value is an f16 value). The f16 stage is free once
    // both S products of the tile two back are done (k_empty), the E4M3
    // stage once this warp has read it (k8_empty). Inline and one key row at
    // a time: this warpgroup runs on tc2_regs_low() registers.
    bool ok = true;
    for (int32_t j = 0; j < T && ok; ++j) {
      const uint32_t st = uint32_t(j) % kTcStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&k8_full[st], uint32_t(j / kTcStages) & 1));
      if (ok && j >= kTcStages)
        ok = __all_sync(0xffffffffu, mbar_wait(&k_empty[st], uint32_t((j - kTcStages) / kTcStages) & 1));
      if (!ok) break;
      const uint8_t* __restrict__ src = smem + Lay::kK80 + st * Lay::kK8Bytes;
      uint8_t* __restrict__ dst = smem + Lay::kStage0 + st * Lay::kStageBytes;
      constexpr uint32_t kUnits = Lay::kE4Row / 16;  // 16-byte units of a source row per chunk
#pragma unroll 1
      for (uint32_t r = lane; r < uint32_t(kTcBN); r += 32) {
#pragma unroll
        for (uint32_t c8 = 0; c8 < Lay::kK8Chunks; ++c8) {
          uint4 w[kUnits];
#pragma unroll
          for (uint32_t u = 0; u < kUnits; ++u) {
            const uint32_t off = D == 64 ? r * 64 + ((u ^ ((r >> 1) & 3)) << 4)
                                         : c8 * (kTcBN * 128) + r * 128 + ((u ^ (r & 7)) << 4);
            w[u] = *reinterpret_cast<const uint4*>(src + off);
          }
#pragma unroll
          for (uint32_t u = 0; u < kUnits; ++u) {  // 16 dims: f16 chunk 2 c8 + u / 4, units 2 (u % 4), + 1
            const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              h[2 * q] = e4m3x2_to_f16x2(uint16_t(ws[q]));
              h[2 * q + 1] = e4m3x2_to_f16x2(uint16_t(ws[q] >> 16));
            }
            const uint32_t cf = 2 * c8 + (u >> 2), u0 = 2 * (u & 3);
            uint8_t* drow = dst + cf * (kTcBN * 128) + r * 128;
            *reinterpret_cast<uint4*>(drow + ((u0 ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(drow + (((u0 + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        }
      }
      fence_async_smem();
      mbar_arrive(&k8_empty[st]);
      mbar_arrive(&k_full[st]);
    }
    if (!ok && lane == 0) atomicOr(&g_prefill_error, kErrWaitTimeout);
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      // S: BF16 Q and K, or f16 Q rows scaled by powers of two against K converted to f16
      constexpr uint32_t idesc_s =
          kFp8 ? umma_idesc_f16(kTcBM, kTcBN, false) : umma_idesc_bf16(kTcBM, kTcBN, false);
      // PV: f16 P x V converted to f16
      constexpr uint32_t idesc_o = umma_idesc_f16(kTcBM, D, true);
      const uint64_t k_desc0 = umma_desc_sw128(sbase + Lay::kStage0, 16, 1024);
      const uint64_t v_desc0 = umma_desc_sw128(sbase + Lay::kStage0 + Lay::kKBytes, kTcBN * 128, 1024);
      const uint64_t q_desc0 = umma_desc_sw128(sbase + Lay::kQ0, 16, 1024);
      constexpr uint64_t kStageStep = Lay::kStageBytes >> 4;
      constexpr uint64_t kQStep = Lay::kQBytes >> 4;
      const uint32_t ntiles = two ? 2u : 1u;
      bool ok = mbar_wait(&q_full, 0);
      tc_fence_after();
      // S_t(j) = Q_t K(j)^T into tile t's S columns
      auto issue_s = [&](int32_t j, uint32_t t) {
        const uint64_t kd = k_desc0 + uint64_t(uint32_t(j) % kTcStages) * kStageStep;
        const uint64_t qd = q_desc0 + t * kQStep;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // chunk kk / 4 is 128 rows of 128 B further; 16 dims are 32 B
          const uint64_t off = uint64_t((kk >> 2) * (kTcBN * 128) + (kk & 3) * 32) >> 4;
          umma_f16kind_ss(tmem + Lay::s_col(t), qd + off, kd + off, idesc_s, kk > 0);
        }
        umma_commit(&s_full[t]);
      };
      if (ok && T > 0) {
        ok = mbar_wait(&k_full[0], 0);
        tc_fence_after();
        if (ok) {
          for (uint32_t t = 0; t < ntiles; ++t) issue_s(0, t);
          umma_commit(&k_empty[0]);
        }
      }
      // Per K/V tile j: PV_A(j); S_A(j + 1) as soon as PV_A(j) is done; then
      // PV_B(j) and S_B(j + 1) the same way. Each S product follows its own
      // tile's PV directly, so a tile's loop (softmax, PV, S) is not held up
      // by the other tile's PV product in the in-order pipe.
      for (int32_t j = 0; j < T && ok; ++j) {
        const uint32_t st = uint32_t(j) % kTcStages;
        const bool more = j + 1 < T;
        const uint32_t sn = uint32_t(j + 1) % kTcStages;
        if (!mbar_wait(&v_full[st], uint32_t(j / kTcStages) & 1)) {
          ok = false;
          break;
        }
        const uint64_t vd = v_desc0 + st * kStageStep;
        for (uint32_t t = 0; t < ntiles && ok; ++t) {
          if (!mbar_wait(&p_full[t], uint32_t(j) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t pt = tmem + Lay::s_col(t);  // P of tile t: keys 2m, 2m + 1 in column m
#pragma unroll
          for (int kk = 0; kk < kTcBN / 16; ++kk) {
            const uint64_t v_k = vd + uint64_t(kk * (16 * 128) >> 4);
            umma_f16kind_tmem_a(tmem + Lay::o_col(t), pt + 8 * kk, v_k, idesc_o, j > 0 || kk > 0);
          }
          umma_commit(&o_full[t]);
          if (t + 1 == ntiles) umma_commit(&v_empty[st]);
          if (more) {
            // tile t's S columns hold P_t(j) until PV_t(j) is done
            if (t == 0 && !mbar_wait(&k_full[sn], uint32_t((j + 1) / kTcStages) & 1)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&o_full[t], uint32_t(j) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(j + 1, t);
            if (t + 1 == ntiles) umma_commit(&k_empty[sn]);
          }
        }
      }
      if (!ok) atomicOr(&g_prefill_error, kErrWaitTimeout);
      // every issued MMA has finished before TMEM is released
      umma_commit(&mma_done);
      mbar_wait(&mma_done, 0);
    }
    __syncwarp();
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(tc2_regs_high<kFp8V>()));
    // ------------------------------------------------------------ softmax
    const uint32_t t = (warp - 4) >> 2;         // the Q tile
    const uint32_t row = (warp & 3) * 32 + lane;  // the row within the tile = TMEM lane
    const uint32_t lane_addr = ((warp & 3) * 32u) << 16;
    const int32_t r = int32_t(t * kTcBM + row);  // the item's row
    const bool valid = r < it.rows;
    const int32_t grow = it.row0 + r;
    const int32_t tok = grow / g, hh = grow % g;
    const int32_t pos = valid ? it.len - it.n + tok : -1;  // -1: attends nothing
    const int32_t lo = W > 0 ? pos + 1 - W : INT32_MIN;
    // the Q row into the tile's shared-memory tile ([chunk][row][128 B],
    // 128-byte swizzled), zeros past the item. E4M3 K cache: the row as f16,
    // times 2^e with e chosen so that its largest magnitude lies in
    // [2^14, 2^15) (exact for BF16 values in range), and the row's score
    // scale rs undoes 2^e.
    float rs = p.score_scale;
    {
      const uint16_t* qr = valid ? p.q + uint64_t(it.qstart + tok) * p.q_stride + uint64_t(it.kv_head * g + hh) * D
                                 : nullptr;
      uint8_t* qt = smem + Lay::kQ0 + t * Lay::kQBytes;
      uint4 qv[D / 8];
#pragma unroll
      for (uint32_t u = 0; u < D / 8; ++u)
        qv[u] = qr ? *reinterpret_cast<const uint4*>(qr + 8 * u) : make_uint4(0, 0, 0, 0);
      if constexpr (kFp8) {
        float amax = 0.0f;
#pragma unroll
        for (uint32_t u = 0; u < D / 8; ++u) {
          const uint32_t w4[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo_to_f32(w4[q])), fabsf(bf16_hi_to_f32(w4[q]))));
        }
        int e = 0;
        if (amax > 0.0f && amax < INFINITY) {
          int ex;
          frexpf(amax, &ex);
          e = 15 - ex;
        }
        const float sc = ldexpf(1.0f, e);
        rs = p.score_scale * ldexpf(1.0f, -e);
#pragma unroll
        for (uint32_t u = 0; u < D / 8; ++u) {
          uint32_t w4[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) w4[q] = f32x2_to_f16x2(bf16_lo_to_f32(w4[q]) * sc, bf16_hi_to_f32(w4[q]) * sc);
          qv[u] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
#pragma unroll
      for (uint32_t u = 0; u < D / 8; ++u)  // 16-byte unit u: chunk u / 8, unit u % 8 of its 128-byte row
        *reinterpret_cast<uint4*>(qt + (u >> 3) * (kTcBM * 128) + row * 128 + (((u & 7) ^ (row & 7)) << 4)) = qv[u];
    }
    fence_async_smem();
    mbar_arrive(&q_full);
    if (t == 1 && !two) {
      // no rows in tile B: nothing more to do
    } else {
      const uint32_t scol = tmem + lane_addr + Lay::s_col(t);
      const uint32_t ocol = tmem + lane_addr + Lay::o_col(t);
      // BF16 V tile j -> f16 in place, part h of it: each warpgroup one part
      // (tile A's both when tile B holds no rows), a half of the tile with an
      // E4M3 K cache, a quarter with a BF16 K cache, where warp 3 takes the
      // second half: each value times
      // 2^-8, rounded to f16 (exact for 2^-6 <= |v| < 2^24, within 2^-17
      // absolute below; the output scale undoes 2^-8). Rows at or past the
      // item's last key (not loaded, or positions past every query) become
      // zeros. Elementwise, so the swizzle does not matter: 16-byte unit e of
      // the tile ([chunk][128 keys][128 B]) holds key row (e / 8) % 128, and
      // a warp's access covers 32 consecutive units.
      auto convert_v_half = [&](int32_t j, uint32_t h) -> bool {
        constexpr uint32_t kHalf = uint32_t(kTcBN) * kChunks * (kFp8 ? 4 : 2);  // units per part
        constexpr uint32_t kPer = kHalf / kTcBM;                                 // per thread
        const uint32_t sj = uint32_t(j) % kTcStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&v8_full[sj], uint32_t(j / kTcStages) & 1))) return false;
        uint4* units = reinterpret_cast<uint4*>(smem + Lay::kStage0 + sj * Lay::kStageBytes + Lay::kKBytes);
        const int32_t live = k_hi - (t_begin + j) * kTcBN;
        const F2 down = f2_make(0.00390625f, 0.00390625f);
        constexpr uint32_t kPass = kPer < 4 ? kPer : 4;  // units per pass
#pragma unroll 1
        for (uint32_t u0 = 0; u0 < kPer; u0 += kPass) {
          uint4 w[kPass];
#pragma unroll
          for (uint32_t u = 0; u < kPass; ++u) w[u] = units[h * kHalf + (u0 + u) * kTcBM + row];
#pragma unroll
          for (uint32_t u = 0; u < kPass; ++u) {
            uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = f2_split(
                  f2_mul(f2_make(__uint_as_float(ws[q] << 16), __uint_as_float(ws[q] & 0xffff0000u)), down));
              ws[q] = f32x2_to_f16x2(f.x, f.y);
            }
            w[u] = make_uint4(ws[0], ws[1], ws[2], ws[3]);
          }
          if (live < kTcBN) {  // the item's last tile
#pragma unroll
            for (uint32_t u = 0; u < kPass; ++u)
              if (int32_t(((h * kHalf + (u0 + u) * kTcBM + row) >> 3) % uint32_t(kTcBN)) >= live)
                w[u] = make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (uint32_t u = 0; u < kPass; ++u) units[h * kHalf + (u0 + u) * kTcBM + row] = w[u];
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&v_full[sj]);
        return true;
      };
      auto convert_v = [&](int32_t j) -> bool {
        if constexpr (kFp8V) return true;  // E4M3 V: converted by the V producer warp
        const uint32_t h1 = two ? t + 1 : 2u;
#pragma unroll 1
        for (uint32_t h = two ? t : 0u; h < h1; ++h)
          if (!convert_v_half(j, h)) return false;
        return true;
      };
      float m_run = -INFINITY, l_run = 0.0f;
      bool ok = T == 0 || convert_v(0);
      for (int32_t j = 0; j < T && ok; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], uint32_t(j) & 1));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[kTcBN];
#pragma unroll
        for (int c = 0; c < kTcBN / 32; ++c)
          tmem_ld32(scol + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
        tmem_wait_ld();
        float x[kTcBN];
#pragma unroll
        for (int k = 0; k < kTcBN; ++k) x[k] = __uint_as_float(sv[k]);
        const int32_t key_base = (t_begin + j) * kTcBN;
        if (key_base + kTcBN - 1 > pos || key_base < lo) {
#pragma unroll
          for (int k = 0; k < kTcBN; ++k)
            if (key_base + k > pos || key_base + k < lo) x[k] = -INFINITY;
        }
        // the tile max: eight partial maxima, two scores into each per
        // three-input max
        float xm8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) xm8[q] = x[q];
#pragma unroll
        for (int k = 8; k + 8 < kTcBN; k += 16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) xm8[q] = fmax3(xm8[q], x[k + q], x[k + 8 + q]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) xm8[q] = fmaxf(xm8[q], x[kTcBN - 8 + q]);
        const float xm = fmax3(fmax3(xm8[0], xm8[1], xm8[2]), fmax3(xm8[3], xm8[4], xm8[5]), fmaxf(xm8[6], xm8[7]));
        // the row's reference max moves only when the tile max exceeds it
        // by more than kRescaleLog2 (or on its first finite score)
        const float tile_max = xm * rs;
        const float mx = (m_run == -INFINITY || tile_max > m_run + kRescaleLog2) ? fmaxf(m_run, tile_max) : m_run;
        const float mb = mx == -INFINITY ? 0.0f : mx;
        // the weights are formed as 2^7 P (<= 2^15), so that they stay above
        // f16's subnormal range down to P = 2^-21; the sum l takes the same
        // factor
        const float mbp = mb - 7.0f;
        // x * score_scale - mbp and the row sum two keys per packed operation;
        // each pair of weights goes to f16 as soon as it is formed (|P - P16|
        // <= 2^-11 P above 2^-21 P, the weights being 2^7 P), so that few
        // packed words stay live
        const F2 sc2 = f2_make(rs, rs), nmb2 = f2_make(-mbp, -mbp);
        F2 sum2[4] = {0ull, 0ull, 0ull, 0ull};
        // P over the S columns, keys 2m, 2m + 1 in column m, 32 keys at a
        // time (the V rows of keys at or past k_hi were zeroed as the tile
        // was converted)
#pragma unroll
        for (int c = 0; c < kTcBN / 32; ++c) {
          uint32_t pw[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int k = 16 * c + q;
            const float2 a = f2_split(f2_fma(f2_make(x[2 * k], x[2 * k + 1]), sc2, nmb2));
            const float e0 = fast_exp2(a.x), e1 = fast_exp2(a.y);
            sum2[q & 3] = f2_add(sum2[q & 3], f2_make(e0, e1));
            pw[q] = f32x2_to_f16x2(e0, e1);
          }
          tmem_st16(scol + 16 * c, pw);
        }
        const float2 s01 = f2_split(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])));
        const float sum = s01.x + s01.y;
        const float al = fast_exp2(m_run - mb);
        const bool rescale = j > 0 && __any_sync(0xffffffffu, mx != m_run);
        if (rescale) {
          // O changes only once PV_t(j - 1) is done
          ok = __all_sync(0xffffffffu, mbar_wait(&o_full[t], uint32_t(j - 1) & 1));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (uint32_t c0 = 0; c0 < uint32_t(D); c0 += 32) {
            uint32_t ov[32];
            tmem_ld32(ocol + c0, ov);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * al);
            tmem_st32(ocol + c0, ov);
          }
        }
        l_run = l_run * al + sum;
        m_run = mx;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        // the next V tile, off the path of this tile's PV product
        if (j + 1 < T) ok = convert_v(j + 1);
      }
      if (!ok && lane == 0) atomicOr(&g_prefill_error, kErrWaitTimeout);
      // ---- O / l to the output row
      // the PV product summed E4M3 codes (v_scale dequantises them) or BF16
      // values times 2^-8
      const float inv = l_run > 0.0f ? (kFp8V ? p.out_scale : 256.0f) / l_run : 0.0f;
      float* o = valid ? p.output + (uint64_t(it.qstart + tok) * p.num_q_heads + uint64_t(it.kv_head * g + hh)) * D
                       : nullptr;
      bool done = __all_sync(0xffffffffu, ok);
      if (T == 0) {  // no key for any query of the item: zeros
        if (o && done)
          for (uint32_t c = 0; c < uint32_t(D); c += 4) *reinterpret_cast<float4*>(o + c) = make_float4(0, 0, 0, 0);
      } else if (done) {
        // once every product is done, the Q tiles and the K/V stages are free:
        // the row is staged there (rows D * 4 + 16 bytes apart, so that the
        // warp's 16-byte stores fall in distinct banks) and goes out as one
        // bulk copy
        done = __all_sync(0xffffffffu, mbar_wait(&mma_done, 0));
        tc_fence_after();
        constexpr uint32_t kRowStride = D * 4 + 16;
        static_assert(2 * kTcBM * kRowStride <= Lay::kStage0 + kTcStages * Lay::kStageBytes,
                      "the staged O rows fit in the Q tiles and the K/V stages");
        float* stage = reinterpret_cast<float*>(smem + (t * kTcBM + row) * kRowStride);
#pragma unroll 1
        for (uint32_t c0 = 0; c0 < uint32_t(D) && done; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(ocol + c0, ov);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(stage + c0 + k) =
                make_float4(__uint_as_float(ov[k]) * inv, __uint_as_float(ov[k + 1]) * inv,
                            __uint_as_float(ov[k + 2]) * inv, __uint_as_float(ov[k + 3]) * inv);
        }
        if (o && done) {
          fence_async_smem();
          bulk_store(o, stage, D * 4);
          bulk_store_wait_read();
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <int D, bool kFp8, bool kFp8V>
int launch_prefill_tc2(const PrefillArgs& a, cudaStream_t stream, PrefillParams& p) {
  CUtensorMap mk, mv;
  if (!encode_pool_map(&mk, a.k_cache, kFp8, a.num_kv_heads, D, 1, 1) ||
      !encode_pool_map(&mv, a.v_cache, kFp8V, a.num_kv_heads, D, 1, 1))
    return KV_ERR_CUDA;
  // grid: an upper bound of the item count, sum over sequences of
  // ceil(n_s * group / 256) <= num_q_tokens * group / 256 + num_seqs
  const uint64_t grid =
      uint64_t(a.num_kv_heads) * ((uint64_t(a.num_q_tokens) * p.group + kTc2Rows - 1) / kTc2Rows + a.num_seqs);
  if (grid == 0) return KV_OK;
  if (grid > 0x7fffffffull) return KV_ERR_UNSUPPORTED;
  // all 512 TMEM columns: no second CTA may be resident on an SM
  constexpr int kNeed = int(1024 + Tc2Layout<D, kFp8, kFp8V>::kBytes);
  const int smem = kNeed > 120 * 1024 ? kNeed : 120 * 1024;
  auto kern = prefill_tc2_kernel<D, kFp8, kFp8V>;
  static int set_bytes[64] = {0};
  const int dev_id = device_info().device;
  if (dev_id < 0 || dev_id >= 64) return KV_ERR_CUDA;
  if (set_bytes[dev_id] < smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return KV_ERR_CUDA;
    set_bytes[dev_id] = smem;
  }
  kern<<<unsigned(grid), 32 * 12, smem, stream>>>(mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

}  // namespace

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  PrefillParams p{};
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  p.output = a.output;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_tokens = a.num_q_tokens;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.block_shift = uint32_t(__builtin_ctz(a.block_size));
  p.q_stride = a.q_stride;
  p.sliding_window = a.sliding_window;
  p.score_scale = a.inv_sqrt_d * kLog2e * (a.fp8 ? a.k_scale : 1.0f);
  p.out_scale = a.fp8_v ? a.v_scale : 1.0f;
  const int key = (a.fp8_v ? 200 : a.fp8 ? 100 : 0) + int(a.head_dim);
  switch (key) {
    case 64: return launch_prefill_tc2<64, false, false>(a, stream, p);  // tcgen05 / TMEM, two Q tiles per CTA
    case 128: return launch_prefill_tc2<128, false, false>(a, stream, p);
    case 164: return launch_prefill_tc2<64, true, false>(a, stream, p);
    case 228: return launch_prefill_tc2<128, true, false>(a, stream, p);
    case 264: return launch_prefill_tc2<64, true, true>(a, stream, p);
    case 328: return launch_prefill_tc2<128, true, true>(a, stream, p);
    default: return KV_ERR_UNSUPPORTED;
  }
}

cudaError_t read_and_clear_prefill_error(uint32_t* bits) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_prefill_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(uint32_t));
}

#ifdef PAGEDKV_DEBUG_BOUNDS
PAGEDKV_DEBUG_UNIT(prefill)
#endif

}  // namespace pagedkv
