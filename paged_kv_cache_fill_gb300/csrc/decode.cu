// Paged decode attention over a BF16, FP8-E4M3-K / BF16-V or FP8 K+V paged
// cache.
//
// [kv_cache.rs] `paged_decode_attn_fp8` doc (one query per (query head,
// sequence), block_tables i32[num_seqs * max_blocks_per_seq], seq_lens
// i32[num_seqs]; K and V scaled by k_scale and v_scale);
// `paged_decode_attn_bf16k_turbo3v` argument list (q_stride,
// sliding_window); [kv_cache_fp8k.rs] module invariants (FP8 K is multiplied
// by k_scale).
//
// GB300 design (the pages launch one 256-thread block per (query head,
// sequence); that re-reads each KV head's bytes once per query head of its
// group, so it is not followed):
//   * The unit of work is a 16-token tile of one (sequence, group of HG KV
//     heads). One persistent CTA per SM (two for the FP8 K+V variant where
//     they fit). With a workspace (split-KV), the tiles of all (sequence,
//     head group) pairs form one stream, in sequence order, which is cut
//     into equal chunks, about one per CTA (stream-K):
//     every CTA gets the same number of tiles whatever the length mix, and a
//     sequence is split only where a chunk boundary falls inside it. Without
//     one, a CTA takes whole (sequence, head group) items b, b+G, ...
//     Every KV byte is read exactly once per call.
//   * Warp 0 is the producer: it walks its chunk's pieces (the part of one
//     (sequence, head group) inside the chunk) and the block table, and
//     issues TMA tiled loads of each 16-token tile of K and V for the HG
//     heads (one 16-row x 128-byte box per head and 128-byte chunk, swizzled
//     so that ldmatrix over 8 token rows is bank-conflict free) plus, on a
//     piece's first tile, a bulk copy of its query rows, into a ring of
//     stages guarded by full/empty mbarriers.
//   * Warps 1..HG*NT are consumers, one per (KV head, 8-query-head tile). Per
//     tile: S^T = K Q^T with mma.sync m16n8k16 (16 tokens x 8 query heads),
//     base-2 online softmax in fp32 with warp-shuffle max, then O^T += V^T P^T
//     with P split into BF16 hi + lo parts (two MMAs) so the weights keep
//     ~16 significant bits. FP8 K converts exactly to f16 in registers
//     (cvt e4m3x2 -> f16x2) against f16 queries scaled by a power of two.
//     FP8 V converts exactly to f16 too, after a transposing ldmatrix that
//     gives each lane two tokens of two adjacent dims; P then enters as f16
//     hi + lo parts scaled by 2^8 (keeping small weights out of the f16
//     subnormal range), and v_scale / 2^8 is applied at the end.
//   * Split-KV (flash-decoding): the pieces of a sequence cut by chunk
//     boundaries write unnormalised partial outputs with their running max
//     and sum to a caller-provided workspace; a combine kernel merges them in
//     piece order, so the result is deterministic. A piece that holds a whole
//     sequence is written directly.
#include <cudaTypedefs.h>
#include <math.h>

#include "internal.h"
#include "../../include/pagedkv.h"

namespace pagedkv {

namespace {

__device__ uint32_t g_decode_error;

constexpr int kTile = 16;            // tokens per stage
constexpr int kHeaderBytes = 256;    // workspace header (work and done counters)
constexpr int kChunksPerCta = 1;     // chunks of the tile stream per CTA
constexpr int kMinChunkTiles = 4;    // smallest chunk: 64 positions
constexpr int kSplitUnitTiles = 16;  // the workspace-size formula's split unit: 256 positions
constexpr float kLog2e = 1.4426950408889634f;

enum : int32_t {
  kFirst = 1,    // first tile of an item
  kLast = 2,     // last tile of an item
  kEmpty = 4,    // the item has no positions: write zeros
  kSingle = 8,   // the sequence is one item per head group: write the output directly
  kSentinel = 16 // no more work
};

struct StageMeta {
  int32_t seq, hg, split, tile, start, len, flags, pad;
};

struct DecodeParams {
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  float* output;
  float* ws_o;          // [num_seqs, max_splits, Hq, D] partial outputs (unnormalised)
  float* ws_ml;         // [num_seqs, max_splits, Hq, 2] running max (log2 units) and sum
  uint32_t* ws_count;   // [num_seqs, num_head_groups] pieces of each (sequence, head group)
  uint32_t* ws_header;  // [1] work counter, [2] done counter
  uint32_t max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, block_size, block_shift;
  uint32_t group;       // query heads per KV head
  uint32_t heads_per_item;  // HG
  uint32_t num_head_groups;
  uint32_t q_stride, sliding_window;
  uint32_t max_splits;  // 0: no workspace, one item per (sequence, head group)
  uint32_t min_chunk_tiles;  // chunks at least this long keep every sequence within max_splits pieces
  float score_scale;    // inv_sqrt_d * log2(e)   (times k_scale for FP8)
  float out_scale;      // FP8 V: v_scale / 2^8 (P enters the MMA scaled by 2^8)
  uint32_t stages, stage_bytes, k_bytes, v_bytes;  // shared-memory ring geometry
};

// -------------------------------------------------------------- item walk
struct SeqSpan {
  int32_t len, start, t0, ntiles;
};

__device__ __forceinline__ SeqSpan seq_span(int32_t raw_len, const DecodeParams& p) {
  SeqSpan s;
  int32_t L = raw_len < 0 ? 0 : raw_len;
  const int64_t cap = int64_t(p.max_blocks_per_seq) << p.block_shift;
  if (L > cap) {
    L = int32_t(cap);
    atomicOr(&g_decode_error, kErrSeqLenClamped);
  }
  s.len = L;
  s.start = (p.sliding_window > 0 && int64_t(L) > int64_t(p.sliding_window))
                ? int32_t(int64_t(L) - int64_t(p.sliding_window))
                : 0;
  s.t0 = s.start / kTile;
  s.ntiles = L > 0 ? (L + kTile - 1) / kTile - s.t0 : 0;
  return s;
}

// The producer walks the tile stream 32 sequences at a time: each lane
// holds one sequence's tile count (times the head groups) and the warp keeps
// an inclusive prefix of the chunk.
struct Walker {
  uint32_t chunk_seq;    // first sequence of the cached chunk
  uint64_t chunk_base;   // stream tiles before the chunk
  uint64_t incl;         // inclusive prefix of stream tiles within the chunk (this lane)
  uint64_t chunk_total;  // stream tiles of the chunk
  int32_t raw_len;       // seq_lens of sequence chunk_seq + lane

  __device__ void load(uint32_t first_seq, const DecodeParams& p, uint32_t lane) {
    chunk_seq = first_seq;
    const uint32_t s = first_seq + lane;
    raw_len = s < p.num_seqs ? __ldg(p.seq_lens + s) : 0;
    incl = s < p.num_seqs ? uint64_t(seq_span(raw_len, p).ntiles) * p.num_head_groups : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= uint32_t(o)) incl += v;
    }
    chunk_total = __shfl_sync(0xffffffffu, incl, 31);
  }
};

// -------------------------------------------------------------- tile layout
// Shared-memory address of 16-byte unit u of row `row` (a slot) in one head's
// tile of a stage, whose head rows are RB bytes:
//   RB a multiple of 128: [128-byte chunk][16 slots][128 B], 128-byte
//     swizzle (unit u % 8 of chunk u / 8 sits at (u % 8) ^ (row % 8));
//   RB = 64 (E4M3 rows of head_dim 64): [16 slots][64 B], 64-byte swizzle
//     (unit u at u ^ ((row / 2) % 4)).
// Both are what the TMA box of the matching tensor map writes (encode_pool_map)
// into a 1024-byte-aligned tile, and both keep ldmatrix over 8 rows free of
// bank conflicts.
template <int RB>
__device__ __forceinline__ uint32_t tile_addr(uint32_t head_base, uint32_t row, uint32_t u) {
  if constexpr (RB == 64) {
    return head_base + row * 64 + ((u ^ ((row >> 1) & 3)) << 4);
  } else {
    static_assert(RB % 128 == 0, "head rows of 64 bytes or whole 128-byte chunks");
    return head_base + (u >> 3) * (kTile * 128) + row * 128 + (((u & 7) ^ (row & 7)) << 4);
  }
}

// -------------------------------------------------------------- O^T += V^T P^T
// One 16-token tile of the PV product for one warp: acc[i] holds the 16-dim
// block i of O^T (8 query-head columns). B fragments (bh*, bl*) are the hi and
// lo parts of P^T; kMask zeroes the V values of masked positions (their rows
// may hold NaN), with vmask01 / vmask89 covering this lane's tokens 2c4, 2c4+1
// and 2c4+8, 2c4+9.
//   BF16 V: per 16-dim block one transposing ldmatrix (rows: 16 tokens).
//   FP8 V: one transposing ldmatrix covers 32 dims x 16 tokens: matrix m holds
//     tokens 8(m&1).. of 16-byte unit 2(jj&3)+(m>>1) and gives this lane the
//     byte pairs (dims 2g8, 2g8+1) of tokens 2c4 and 2c4+1; one byte
//     permutation regroups them by dim and each pair converts exactly to f16.
//     A-row g8 is dim 2g8 and A-row g8+8 dim 2g8+1 of the 16-dim block, so
//     the accumulator rows come out in that order too.
template <bool kFp8V, int D, bool kMask>
__device__ __forceinline__ void pv_tile(float (&acc)[D / 16][4], uint32_t vbase, uint32_t row, uint32_t unit_lo,
                                        uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1, uint32_t vmask01,
                                        uint32_t vmask89) {
  constexpr int kVRow = D * (kFp8V ? 1 : 2);  // bytes of one head's V row
  if constexpr (!kFp8V) {
    uint32_t a[D / 16][4];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      ldmatrix_x4_trans(a[i], tile_addr<kVRow>(vbase, row, 2 * i + unit_lo));
      if constexpr (kMask) {
        a[i][0] &= vmask01;
        a[i][1] &= vmask01;
        a[i][2] &= vmask89;
        a[i][3] &= vmask89;
      }
      mma_bf16(acc[i], a[i], bh0, bh1);
    }
    // the lo parts after every hi part: no MMA waits on the one before
#pragma unroll
    for (int i = 0; i < D / 16; ++i) mma_bf16(acc[i], a[i], bl0, bl1);
  } else {
#pragma unroll
    for (int jj = 0; jj < D / 32; ++jj) {
      uint32_t r[4];
      ldmatrix_x4_trans(r, tile_addr<kVRow>(vbase, row, 2 * jj + unit_lo));
      uint32_t a[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // bytes [t0 d0, t0 d1, t1 d0, t1 d1] -> [t0 d0, t1 d0, t0 d1, t1 d1]
        const uint32_t w0 = __byte_perm(r[2 * h], 0u, 0x3120u);
        const uint32_t w1 = __byte_perm(r[2 * h + 1], 0u, 0x3120u);
        a[h][0] = e4m3x2_to_f16x2(uint16_t(w0));
        a[h][1] = e4m3x2_to_f16x2(uint16_t(w0 >> 16));
        a[h][2] = e4m3x2_to_f16x2(uint16_t(w1));
        a[h][3] = e4m3x2_to_f16x2(uint16_t(w1 >> 16));
        if constexpr (kMask) {
          a[h][0] &= vmask01;
          a[h][1] &= vmask01;
          a[h][2] &= vmask89;
          a[h][3] &= vmask89;
        }
      }
      // hi, hi, lo, lo: no MMA waits on the accumulator of the one before
      mma_f16(acc[2 * jj], a[0], bh0, bh1);
      mma_f16(acc[2 * jj + 1], a[1], bh0, bh1);
      mma_f16(acc[2 * jj], a[0], bl0, bl1);
      mma_f16(acc[2 * jj + 1], a[1], bl0, bl1);
    }
  }
}

// -------------------------------------------------------------- the kernel
// The FP8 K+V variant does 1.5x the per-byte work of the others and is
// bound by dependent-instruction latency: for head_dim up to 128 and one
// 8-head tile per KV head it is built to run two CTAs per SM (registers for
// two, a ring in half the shared memory) where the ring fits
// (launch_decode); with head_dim 256 or two tiles the accumulators do not
// fit two CTAs' registers.
template <bool kFp8V, int D, int NT>
constexpr bool two_ctas_per_sm() { return kFp8V && D <= 128 && NT == 1; }

template <bool kFp8, bool kFp8V, int D, int NT>
__global__ void __launch_bounds__(32 * 9, two_ctas_per_sm<kFp8V, D, NT>() ? 2 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeParams p) {
  constexpr int kKRow = D * (kFp8 ? 1 : 2), kVRow = D * (kFp8V ? 1 : 2);  // bytes of one head's row
  // the tensor maps' third coordinate per head: 128-byte chunks, or one
  // 64-byte row (encode_pool_map)
  constexpr int kKCoord = kKRow >= 128 ? kKRow / 128 : 1;
  constexpr int kVCoord = kVRow >= 128 ? kVRow / 128 : 1;
  static_assert(kFp8 || !kFp8V, "an FP8 V cache comes with an FP8 K cache");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes);
  uint64_t* empty = full + p.stages;
  StageMeta* meta = reinterpret_cast<StageMeta*>(empty + p.stages);
  __shared__ uint64_t s_chunk, s_total;

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t num_consumers = p.heads_per_item * NT;
  const uint64_t wait_ns = pipeline_wait_limit();  // fixed in the product build

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], num_consumers);
    }
    fence_mbar_init();
    s_total = 0;
  }
  __syncthreads();

  // Chunk size: the stream's tiles over kChunksPerCta chunks per CTA, never
  // below the minimum chunk (or the larger one a small workspace imposes).
  if (p.max_splits > 0) {
    uint64_t local = 0;
    for (uint32_t s = threadIdx.x; s < p.num_seqs; s += blockDim.x)
      local += uint64_t(seq_span(__ldg(p.seq_lens + s), p).ntiles);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if (lane == 0 && local) atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), local);
    __syncthreads();
    if (threadIdx.x == 0) {
      s_total *= p.num_head_groups;
      const uint64_t parts = uint64_t(gridDim.x) * kChunksPerCta;
      const uint64_t want = (s_total + parts - 1) / parts;
      s_chunk = want > p.min_chunk_tiles ? want : p.min_chunk_tiles;
    }
    __syncthreads();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    // Stages whose last fill was issued with TMA (bit s) and the parity the
    // consumers wait on for that fill: drained before the CTA exits.
    uint32_t issued = 0, issued_parity = 0;

    // One piece: tiles [tile_begin, tile_end) of sequence s for head group
    // hg, the split'th piece of that pair (no tiles: one meta-only stage
    // tells the consumers to write zeros).
    auto emit = [&](uint32_t s, uint32_t hg, uint32_t split, const SeqSpan& span, int32_t tile_begin,
                    int32_t tile_end, int32_t base_flags) {
      const uint32_t heads_here = (hg + 1) * p.heads_per_item <= p.num_kv_heads
                                      ? p.heads_per_item
                                      : p.num_kv_heads - hg * p.heads_per_item;
      const uint32_t q_bytes = heads_here * p.group * D * 2;
      const uint16_t* q_src = p.q + uint64_t(s) * p.q_stride + uint64_t(hg) * p.heads_per_item * p.group * D;
      if (tile_begin >= tile_end) {
        if (lane == 0) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wait_ns)) ok = false;
          if (ok) {
            issued &= ~(1u << stage);  // the stage's previous fill was taken, so it landed
            meta[stage] = StageMeta{int32_t(s), int32_t(hg), int32_t(split), 0, 0, 0,
                                    kFirst | kLast | kEmpty | base_flags, 0};
            mbar_arrive(&full[stage]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (++stage == p.stages) { stage = 0; phase ^= 1; }
        return;
      }
      const int32_t* table = p.block_tables + uint64_t(s) * p.max_blocks_per_seq;
      const int32_t tiles_per_block_shift = int32_t(p.block_shift) - 4;  // block_size >= 16
      int32_t cached_first_block = -1;  // first logical block held by the lanes
      int32_t cached_block_id = 0;
      for (int32_t tile = tile_begin; tile < tile_end && ok; ++tile) {
        const int32_t lblock = tile >> tiles_per_block_shift;
        if (cached_first_block < 0 || lblock >= cached_first_block + 32) {
          cached_first_block = lblock;
          const int32_t want = lblock + int32_t(lane);
          cached_block_id = want < int32_t(p.max_blocks_per_seq) ? __ldg(table + want) : 0;
        }
        const int32_t block_id = __shfl_sync(0xffffffffu, cached_block_id, lblock - cached_first_block);
        if (lane == 0) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wait_ns)) ok = false;
          if (ok) {
            issued &= ~(1u << stage);
            int32_t flags = base_flags;
            if (tile == tile_begin) flags |= kFirst;
            if (tile == tile_end - 1) flags |= kLast;
            meta[stage] = StageMeta{int32_t(s), int32_t(hg), int32_t(split), tile, span.start,
                                    span.len, flags, 0};
            // one box per tensor covers all heads of the piece (chunks past
            // the last head are zero-filled and still counted in the box bytes)
            const uint32_t bytes = p.k_bytes + p.v_bytes + ((flags & kFirst) ? q_bytes : 0u);
            mbar_arrive_expect_tx(&full[stage], bytes);
            uint8_t* st = smem + stage * p.stage_bytes;
#ifdef PAGEDKV_DEBUG_BOUNDS
            // a block id outside the pool is flagged and block 0 read instead
            const int32_t slot0 =
                ((dbg_block_ok(block_id) ? block_id : 0) << p.block_shift) + ((tile << 4) & int32_t(p.block_size - 1));
#else
            const int32_t slot0 = (block_id << p.block_shift) + ((tile << 4) & int32_t(p.block_size - 1));
#endif
            const int32_t head0 = int32_t(hg * p.heads_per_item);
            tma_load_3d(st, &tmap_k, 0, slot0, head0 * kKCoord, &full[stage]);
            tma_load_3d(st + p.k_bytes, &tmap_v, 0, slot0, head0 * kVCoord, &full[stage]);
            if (flags & kFirst) bulk_load(st + p.k_bytes + p.v_bytes, q_src, q_bytes, &full[stage]);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (++stage == p.stages) { stage = 0; phase ^= 1; }
      }
    };

    if (p.max_splits > 0) {
      // Stream-K: chunk k holds stream tiles [k C, (k + 1) C). CTA b takes
      // chunk b; chunks past the grid (more than one per CTA) come from an
      // atomic counter in the workspace header, in increasing order, so the
      // walker only moves forward. The piece of (sequence, head group) range
      // [a, b) that lies in chunk k is its piece k - floor(a / C).
      const uint64_t C = s_chunk, total = s_total;
      const uint64_t nchunks = (total + C - 1) / C;
      uint32_t* const work = p.ws_header + 1;
      Walker wk;
      wk.chunk_base = 0;
      wk.load(0, p, lane);
      uint64_t k = blockIdx.x;
      while (ok && k < nchunks) {
        uint64_t g = k * C;
        const uint64_t g1 = g + C < total ? g + C : total;
        while (ok && g < g1) {
          while (wk.chunk_seq < p.num_seqs && g >= wk.chunk_base + wk.chunk_total) {
            wk.chunk_base += wk.chunk_total;
            wk.load(wk.chunk_seq + 32, p, lane);
          }
          if (wk.chunk_seq >= p.num_seqs) break;  // not reached: g < total
          const uint64_t rel = g - wk.chunk_base;
          const uint32_t sl = __ffs(__ballot_sync(0xffffffffu, wk.incl > rel)) - 1;
          const uint32_t s = wk.chunk_seq + sl;
          const SeqSpan span = seq_span(__shfl_sync(0xffffffffu, wk.raw_len, sl), p);
          const uint64_t nt = uint64_t(span.ntiles);  // > 0: the ballot skips empty sequences
          const uint64_t seq_base = wk.chunk_base + __shfl_sync(0xffffffffu, wk.incl, sl) - nt * p.num_head_groups;
          const uint32_t hg = uint32_t((g - seq_base) / nt);
          const uint64_t a = seq_base + uint64_t(hg) * nt, b = a + nt;
          const uint64_t e = b < g1 ? b : g1;
          const uint32_t split = uint32_t(k - a / C);
          // the piece that ends the pair records how many pieces it has
          if (e == b && lane == 0) p.ws_count[uint64_t(s) * p.num_head_groups + hg] = split + 1;
          emit(s, hg, split, span, span.t0 + int32_t(g - a), span.t0 + int32_t(e - a),
               (g == a && e == b) ? kSingle : 0);
          g = e;
        }
        if (nchunks <= gridDim.x) break;
        k = gridDim.x + __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(work, 1u) : 0u, 0);
      }
    } else {
      // no workspace: whole (sequence, head group) items, statically strided
      const uint64_t items = uint64_t(p.num_seqs) * p.num_head_groups;
      for (uint64_t it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const uint32_t s = uint32_t(it / p.num_head_groups), hg = uint32_t(it % p.num_head_groups);
        const SeqSpan span = seq_span(__ldg(p.seq_lens + s), p);
        emit(s, hg, 0, span, span.t0, span.t0 + span.ntiles, kSingle);
      }
    }
    // sentinel: no more work
    if (ok && lane == 0) {
      if (mbar_wait(&empty[stage], phase ^ 1, wait_ns)) {
        issued &= ~(1u << stage);
        meta[stage].flags = kSentinel;
        mbar_arrive(&full[stage]);
      } else {
        ok = false;
      }
    }
    if (!__all_sync(0xffffffffu, ok) && lane == 0) atomicOr(&g_decode_error, kErrWaitTimeout);
    // No copy may land in shared memory after the CTA exits: wait (bounded,
    // with the fixed limit even where the pipeline's is shorter) until every
    // TMA fill not yet known to have landed has completed. A bit is cleared
    // when the producer next waits the stage's empty barrier out (the
    // consumers took that fill). After a normal run the fills still marked
    // are ones the consumers wait on too, so they have landed or are about
    // to; the drain matters when a wait above, or a consumer's, gave up.
    if (lane == 0) {
      for (uint32_t st = 0; st < p.stages; ++st)
        if ((issued >> st) & 1u)
          if (!mbar_wait(&full[st], (issued_parity >> st) & 1u)) atomicOr(&g_decode_error, kErrWaitTimeout);
    }
    // The last CTA to finish resets the counters for the next launch.
    if (p.max_splits > 0 && lane == 0) {
      __threadfence();
      if (atomicAdd(p.ws_header + 2, 1u) == gridDim.x - 1) {
        atomicExch(p.ws_header + 1, 0u);
        atomicExch(p.ws_header + 2, 0u);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const uint32_t task = warp - 1;
  if (task >= num_consumers) return;
  const uint32_t hl = task / NT;   // KV head within the item
  const uint32_t qt = task % NT;   // 8-query-head tile within the group
  const uint32_t g8 = lane >> 2;   // fragment row group
  const uint32_t c4 = lane & 3;    // fragment column pair
  // ldmatrix row/unit of this lane: K (non-transposed A) and V (transposed A)
  const uint32_t k_row = (lane & 7) + ((lane >> 3) & 1) * 8, k_unit = lane >> 4;
  const uint32_t v_row = (lane & 7) + (lane >> 4) * 8, v_unit = (lane >> 3) & 1;

  float acc[D / 16][4];
  float m_run[2], l_run[2];
  uint32_t qf[D / 16][2];
  float head_scale[2];

  uint32_t stage = 0, phase = 0;
  while (true) {
    if (!mbar_wait(&full[stage], phase, wait_ns)) {
      // the producer drains the copies it issued before the CTA exits
      if (lane == 0) atomicOr(&g_decode_error, kErrWaitTimeout);
      return;
    }
    const StageMeta mt = meta[stage];
    if (mt.flags & kSentinel) break;
    const uint8_t* st = smem + stage * p.stage_bytes;
    const uint32_t kv_head = mt.hg * p.heads_per_item + hl;
    const bool head_ok = kv_head < p.num_kv_heads;
    // query heads of this warp's tile: qt*8 + n for n < 8, valid if < group
    const uint32_t q_in_group_row = qt * 8 + g8;  // the head this lane loads for B fragments

    if (head_ok && (mt.flags & kFirst)) {
#pragma unroll
      for (int i = 0; i < D / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.0f;
      if (!(mt.flags & kEmpty)) {
        const uint16_t* qs = reinterpret_cast<const uint16_t*>(st + p.k_bytes + p.v_bytes) +
                             (hl * p.group + q_in_group_row) * D;
        const bool row_ok = q_in_group_row < p.group;
        if constexpr (!kFp8) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][0] = row_ok ? *reinterpret_cast<const uint32_t*>(qs + kk * 16 + 2 * c4) : 0u;
            qf[kk][1] = row_ok ? *reinterpret_cast<const uint32_t*>(qs + kk * 16 + 2 * c4 + 8) : 0u;
          }
          head_scale[0] = head_scale[1] = p.score_scale;
        } else {
          // permuted k order: slot pair (2c, 2c+1) <-> d = 16kk + 4c + {0,1},
          // (2c+8, 2c+9) <-> d = 16kk + 4c + {2,3}
          float qv[D / 16][4];
          float amax = 0.0f;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint2 w = row_ok ? *reinterpret_cast<const uint2*>(qs + kk * 16 + 4 * c4) : make_uint2(0, 0);
            qv[kk][0] = bf16_lo_to_f32(w.x);
            qv[kk][1] = bf16_hi_to_f32(w.x);
            qv[kk][2] = bf16_lo_to_f32(w.y);
            qv[kk][3] = bf16_hi_to_f32(w.y);
#pragma unroll
            for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qv[kk][e]));
          }
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          // scale the row by 2^e so its largest magnitude lies in [2^14, 2^15)
          int e = 0;
          if (amax > 0.0f && amax < INFINITY) {
            int ex;
            frexpf(amax, &ex);
            e = 15 - ex;
          }
          const float sc = ldexpf(1.0f, e);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][0] = f32x2_to_f16x2(qv[kk][0] * sc, qv[kk][1] * sc);
            qf[kk][1] = f32x2_to_f16x2(qv[kk][2] * sc, qv[kk][3] * sc);
          }
          const float unscale = p.score_scale * ldexpf(1.0f, -e);
          head_scale[0] = __shfl_sync(0xffffffffu, unscale, (2 * c4) * 4);
          head_scale[1] = __shfl_sync(0xffffffffu, unscale, (2 * c4 + 1) * 4);
        }
      }
    }

    if (head_ok && !(mt.flags & kEmpty)) {
      const uint32_t kbase = smem_u32(st) + hl * (kTile * kKRow);
      const uint32_t vbase = smem_u32(st + p.k_bytes) + hl * (kTile * kVRow);
      // ---- S^T = K Q^T (16 tokens x 8 query heads), even and odd k-steps in
      // two accumulators so that consecutive MMAs do not wait on each other
      float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (!kFp8) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a[4];
          ldmatrix_x4(a, tile_addr<kKRow>(kbase, k_row, 2 * kk + k_unit));
          if (kk & 1) mma_bf16(s2, a, qf[kk][0], qf[kk][1]);
          else mma_bf16(s, a, qf[kk][0], qf[kk][1]);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < D / 32; ++jj) {
          uint32_t r[4];
          ldmatrix_x4(r, tile_addr<kKRow>(kbase, k_row, 2 * jj + k_unit));
          uint32_t a0[4], a1[4];
          a0[0] = e4m3x2_to_f16x2(uint16_t(r[0]));
          a0[1] = e4m3x2_to_f16x2(uint16_t(r[1]));
          a0[2] = e4m3x2_to_f16x2(uint16_t(r[0] >> 16));
          a0[3] = e4m3x2_to_f16x2(uint16_t(r[1] >> 16));
          a1[0] = e4m3x2_to_f16x2(uint16_t(r[2]));
          a1[1] = e4m3x2_to_f16x2(uint16_t(r[3]));
          a1[2] = e4m3x2_to_f16x2(uint16_t(r[2] >> 16));
          a1[3] = e4m3x2_to_f16x2(uint16_t(r[3] >> 16));
          mma_f16(s, a0, qf[2 * jj][0], qf[2 * jj][1]);
          mma_f16(s2, a1, qf[2 * jj + 1][0], qf[2 * jj + 1][1]);
        }
      }
      s[0] += s2[0];
      s[1] += s2[1];
      s[2] += s2[2];
      s[3] += s2[3];
      s[0] *= head_scale[0];
      s[1] *= head_scale[1];
      s[2] *= head_scale[0];
      s[3] *= head_scale[1];
      // ---- mask positions outside [start, len)
      const int32_t p0 = mt.tile * kTile;
      const bool boundary = p0 < mt.start || p0 + kTile > mt.len;
      if (boundary) {
        const int32_t pa = p0 + int32_t(g8), pb = pa + 8;
        if (pa < mt.start || pa >= mt.len) s[0] = s[1] = -INFINITY;
        if (pb < mt.start || pb >= mt.len) s[2] = s[3] = -INFINITY;
      }
      // ---- online softmax (base 2), per query head column
      float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
      // Rescale only when some column's running max moved (rare after the
      // first tiles); with the max unchanged the factor would be exactly 1.
      if (__any_sync(0xffffffffu, mn0 != m_run[0] || mn1 != m_run[1])) {
        const float al0 = fast_exp2(m_run[0] - mn0), al1 = fast_exp2(m_run[1] - mn1);
        l_run[0] *= al0;
        l_run[1] *= al1;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          acc[i][0] *= al0;
          acc[i][1] *= al1;
          acc[i][2] *= al0;
          acc[i][3] *= al1;
        }
      }
      m_run[0] = mn0;
      m_run[1] = mn1;
      const float e0 = fast_exp2(s[0] - mn0), e1 = fast_exp2(s[1] - mn1);
      const float e2 = fast_exp2(s[2] - mn0), e3 = fast_exp2(s[3] - mn1);
      l_run[0] += e0 + e2;
      l_run[1] += e1 + e3;
      // V rows of masked positions may hold anything (NaN): zero them
      uint32_t vmask01 = 0xffffffffu, vmask89 = 0xffffffffu;
      if (boundary) {
        const int32_t q0 = p0 + 2 * int32_t(c4);
        auto ok = [&](int32_t pos) { return pos >= mt.start && pos < mt.len; };
        vmask01 = (ok(q0) ? 0x0000ffffu : 0u) | (ok(q0 + 1) ? 0xffff0000u : 0u);
        vmask89 = (ok(q0 + 8) ? 0x0000ffffu : 0u) | (ok(q0 + 9) ? 0xffff0000u : 0u);
      }
      uint32_t bh0, bh1, bl0, bl1;
      if constexpr (!kFp8V) {
        // ---- P^T as B fragments: hi and lo BF16 parts, transposed by movmatrix
        const uint32_t hi01 = f32x2_to_bf16x2(e0, e1), hi23 = f32x2_to_bf16x2(e2, e3);
        const uint32_t lo01 = f32x2_to_bf16x2(e0 - bf16_lo_to_f32(hi01), e1 - bf16_hi_to_f32(hi01));
        const uint32_t lo23 = f32x2_to_bf16x2(e2 - bf16_lo_to_f32(hi23), e3 - bf16_hi_to_f32(hi23));
        bh0 = movmatrix_trans(hi01), bh1 = movmatrix_trans(hi23);
        bl0 = movmatrix_trans(lo01), bl1 = movmatrix_trans(lo23);
      } else {
        // ---- P^T as f16 hi + lo parts of 2^8 * P
        const float f0 = e0 * 256.0f, f1 = e1 * 256.0f, f2 = e2 * 256.0f, f3 = e3 * 256.0f;
        const uint32_t hi01 = f32x2_to_f16x2(f0, f1), hi23 = f32x2_to_f16x2(f2, f3);
        const uint32_t lo01 = f32x2_to_f16x2(f0 - f16_lo_to_f32(hi01), f1 - f16_hi_to_f32(hi01));
        const uint32_t lo23 = f32x2_to_f16x2(f2 - f16_lo_to_f32(hi23), f3 - f16_hi_to_f32(hi23));
        bh0 = movmatrix_trans(hi01), bh1 = movmatrix_trans(hi23);
        bl0 = movmatrix_trans(lo01), bl1 = movmatrix_trans(lo23);
      }
      // ---- O^T += V^T P^T; only a tile with masked positions pays for the masks
      const uint32_t vrow = kFp8V ? k_row : v_row, vunit = kFp8V ? k_unit : v_unit;
      if (boundary)
        pv_tile<kFp8V, D, true>(acc, vbase, vrow, vunit, bh0, bh1, bl0, bl1, vmask01, vmask89);
      else
        pv_tile<kFp8V, D, false>(acc, vbase, vrow, vunit, bh0, bh1, bl0, bl1, 0u, 0u);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);

    if (head_ok && (mt.flags & kLast)) {
      // ---- finish the item
      float l0 = l_run[0], l1 = l_run[1];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
      }
      const uint32_t col0 = qt * 8 + 2 * c4;  // query head within the group of column 0
      const uint32_t hq0 = kv_head * p.group + col0;
      const bool ok0 = col0 < p.group, ok1 = col0 + 1 < p.group;
      if (mt.flags & kSingle) {
        const float sc = kFp8V ? p.out_scale : 1.0f;
        const float inv0 = (mt.flags & kEmpty) ? 0.0f : sc / l0;
        const float inv1 = (mt.flags & kEmpty) ? 0.0f : sc / l1;
        float* o0 = p.output + (uint64_t(mt.seq) * p.num_q_heads + hq0) * D;
        float* o1 = o0 + D;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          if constexpr (kFp8V) {
            // accumulator rows g8 / g8+8 are dims 2g8 / 2g8+1
            const uint32_t d = i * 16 + 2 * g8;
            if (ok0) *reinterpret_cast<float2*>(o0 + d) = make_float2(acc[i][0] * inv0, acc[i][2] * inv0);
            if (ok1) *reinterpret_cast<float2*>(o1 + d) = make_float2(acc[i][1] * inv1, acc[i][3] * inv1);
          } else {
            const uint32_t d = i * 16 + g8;
            if (ok0) {
              o0[d] = (mt.flags & kEmpty) ? 0.0f : acc[i][0] * inv0;
              o0[d + 8] = (mt.flags & kEmpty) ? 0.0f : acc[i][2] * inv0;
            }
            if (ok1) {
              o1[d] = (mt.flags & kEmpty) ? 0.0f : acc[i][1] * inv1;
              o1[d + 8] = (mt.flags & kEmpty) ? 0.0f : acc[i][3] * inv1;
            }
          }
        }
      } else {
        const uint64_t row = (uint64_t(mt.seq) * p.max_splits + mt.split) * p.num_q_heads + hq0;
        float* o0 = p.ws_o + row * D;
        float* o1 = o0 + D;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          if constexpr (kFp8V) {
            const uint32_t d = i * 16 + 2 * g8;
            const float sc = p.out_scale;
            if (ok0) *reinterpret_cast<float2*>(o0 + d) = make_float2(acc[i][0] * sc, acc[i][2] * sc);
            if (ok1) *reinterpret_cast<float2*>(o1 + d) = make_float2(acc[i][1] * sc, acc[i][3] * sc);
          } else {
            const uint32_t d = i * 16 + g8;
            if (ok0) {
              o0[d] = acc[i][0];
              o0[d + 8] = acc[i][2];
            }
            if (ok1) {
              o1[d] = acc[i][1];
              o1[d + 8] = acc[i][3];
            }
          }
        }
        if (g8 == 0) {
          if (ok0) *reinterpret_cast<float2*>(p.ws_ml + row * 2) = make_float2(m_run[0], l0);
          if (ok1) *reinterpret_cast<float2*>(p.ws_ml + (row + 1) * 2) = make_float2(m_run[1], l1);
        }
      }
    }
    if (++stage == p.stages) { stage = 0; phase ^= 1; }
  }
}

// Merge the partials of every (sequence, query head) whose sequence was cut
// into more than one piece: o = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i,
// in piece order, in one pass: M is the running max of the pieces' maxima,
// and the sums so far are scaled by 2^(M_old - M_new) when it moves. One
// warp per (sequence, query head), lane k holding dims k, k + 32, ...: the
// piece count, then each piece's (m, l) and the lane's dims of its partial
// output, whose loads do not depend on one another. A sequence with no
// positions has no piece in the tile stream: its output row is written as
// zeros here.
constexpr uint32_t kCombineWarps = 8;  // per CTA

template <int D>
__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(const DecodeParams p) {
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t item = uint64_t(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);  // s * Hq + h
  if (item >= uint64_t(p.num_seqs) * p.num_q_heads) return;
  const uint32_t s = uint32_t(item / p.num_q_heads), h = uint32_t(item % p.num_q_heads);
  float* out = p.output + item * D;
  const SeqSpan span = seq_span(__ldg(p.seq_lens + s), p);
  if (span.ntiles == 0) {
#pragma unroll
    for (uint32_t k = 0; k < D / 32; ++k) out[lane + 32 * k] = 0.0f;
    return;
  }
  const uint32_t hg = h / p.group / p.heads_per_item;
  const int32_t nsplit = int32_t(__ldg(p.ws_count + uint64_t(s) * p.num_head_groups + hg));
  if (nsplit <= 1) return;
  const uint64_t row0 = uint64_t(s) * p.max_splits * p.num_q_heads + h;  // piece i at row0 + i * Hq
  float M = -INFINITY, den = 0.0f, acc[D / 32];
#pragma unroll
  for (uint32_t k = 0; k < D / 32; ++k) acc[k] = 0.0f;
#pragma unroll 4
  for (int32_t i = 0; i < nsplit; ++i) {
    const uint64_t row = row0 + uint64_t(i) * p.num_q_heads;
    const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + row * 2);
    float v[D / 32];
#pragma unroll
    for (uint32_t k = 0; k < D / 32; ++k) v[k] = p.ws_o[row * D + lane + 32 * k];
    const float Mn = fmaxf(M, ml.x);
    const float a = M == -INFINITY ? 0.0f : fast_exp2(M - Mn);
    const float w = ml.x == -INFINITY ? 0.0f : fast_exp2(ml.x - Mn);
    den = den * a + w * ml.y;
#pragma unroll
    for (uint32_t k = 0; k < D / 32; ++k) acc[k] = acc[k] * a + w * v[k];
    M = Mn;
  }
#pragma unroll
  for (uint32_t k = 0; k < D / 32; ++k) out[lane + 32 * k] = acc[k] / den;
}

// ---------------------------------------------------------------- host side
}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Tensor map over a cache pool for one TMA box per 16-position tile and
// item: dim 0 the elements of a 128-byte chunk, dim 1 the slot (stride
// heads * head_dim * elem bytes), dim 2 the 128-byte chunk of a slot's row
// (stride 128 bytes; a head owns head_dim * elem / 128 consecutive chunks).
// Box: one chunk x 16 slots x (heads per item * chunks per head), so the
// shared-memory tile is [chunk][slot][128 bytes], 128-byte swizzled by slot
// row. (Dim 1's stride exceeds dim 2's; the encoder accepts any order.)
bool encode_pool_map(CUtensorMap* map, const void* base, bool fp8, uint32_t num_kv_heads,
                     uint32_t head_dim, uint32_t heads_per_item, uint32_t box_chunks) {
  auto encode = get_encode();
  if (!encode) return false;
  const uint32_t elem = fp8 ? 1 : 2;
  if (head_dim * elem == 64) {
    // E4M3 rows of head_dim 64: dim 0 a head's 64-byte row, dim 1 the slot,
    // dim 2 the head (stride 64 bytes); box: one row x 16 slots x the item's
    // heads, 64-byte swizzled ([head][slot][64 B] in shared memory)
    cuuint64_t dims[3] = {64, cuuint64_t(1) << 31, num_kv_heads};
    cuuint64_t strides[2] = {cuuint64_t(num_kv_heads) * 64, 64};
    cuuint32_t box[3] = {64, kTile, box_chunks ? box_chunks : heads_per_item};
    cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const uint32_t chunk_elems = 128 / elem;
  const uint32_t chunks_per_head = head_dim * elem / 128;
  cuuint64_t dims[3] = {chunk_elems, cuuint64_t(1) << 31, cuuint64_t(num_kv_heads) * chunks_per_head};
  cuuint64_t strides[2] = {cuuint64_t(num_kv_heads) * head_dim * elem, 128};
  cuuint32_t box[3] = {chunk_elems, kTile, box_chunks ? box_chunks : heads_per_item * chunks_per_head};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

struct Geometry {
  uint32_t heads_per_item, nt, stages, stage_bytes, k_bytes, v_bytes, smem_bytes;
  uint32_t ctas_per_sm;  // set by launch_decode
};

Geometry geometry(bool fp8, bool fp8_v, uint32_t head_dim, uint32_t num_kv_heads, uint32_t group, int smem_max) {
  Geometry g{};
  g.nt = (group + 7) / 8;
  uint32_t hg = 8 / g.nt;
  if (hg > num_kv_heads) hg = num_kv_heads;
  const uint32_t krow = head_dim * (fp8 ? 1 : 2), vrow = head_dim * (fp8_v ? 1 : 2);  // bytes per head row
  for (;; hg = (hg + 1) / 2) {
    g.heads_per_item = hg;
    g.k_bytes = hg * kTile * krow;
    g.v_bytes = hg * kTile * vrow;
    const uint32_t q_bytes = (hg * group * head_dim * 2 + 1023) / 1024 * 1024;
    g.stage_bytes = g.k_bytes + g.v_bytes + q_bytes;
    const uint32_t extra = 1024 + 64 * (2 * 8 + 32);  // alignment slack, barriers, meta
    uint32_t stages = (uint32_t(smem_max) - extra) / g.stage_bytes;
    if (stages > 4) stages = 4;
    g.stages = stages;
    g.smem_bytes = stages * g.stage_bytes + extra;
    // Keep all heads of a group in one item (8 consumer warps per CTA) even
    // at 3 stages: 4 heads per item with a 6-stage ring measured slower (the
    // per-tile MMA/softmax work of 4 warps becomes the limit).
    if (stages >= 2 || hg == 1) break;
  }
  return g;
}

template <bool kFp8, bool kFp8V, int D, int NT>
int launch_decode_t(const DecodeArgs& a, cudaStream_t stream, const Geometry& geo, DecodeParams& p) {
  CUtensorMap mk, mv;
  if (!encode_pool_map(&mk, a.k_cache, kFp8, a.num_kv_heads, D, geo.heads_per_item) ||
      !encode_pool_map(&mv, a.v_cache, kFp8V, a.num_kv_heads, D, geo.heads_per_item))
    return KV_ERR_CUDA;
  auto kern = decode_kernel<kFp8, kFp8V, D, NT>;
  // The dynamic shared-memory opt-in is set once per device and size (so
  // that calls made while a stream is being captured into a CUDA graph after
  // a first eager call issue no attribute change).
  static int set_bytes[64] = {0};
  const int dev_id = device_info().device;
  if (dev_id < 0 || dev_id >= 64) return KV_ERR_CUDA;
  if (set_bytes[dev_id] < int(geo.smem_bytes)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(geo.smem_bytes)) !=
        cudaSuccess)
      return KV_ERR_CUDA;
    set_bytes[dev_id] = int(geo.smem_bytes);
  }
  const DeviceInfo& dev = device_info();
  const uint32_t threads = 32 * (1 + geo.heads_per_item * geo.nt);
  if (geo.ctas_per_sm > 1 && !two_ctas_per_sm<kFp8V, D, NT>()) return KV_ERR_CUDA;  // not reached
  kern<<<dev.num_sms * geo.ctas_per_sm, threads, geo.smem_bytes, stream>>>(mk, mv, p);
  if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
  if (p.max_splits > 0) {
    const uint64_t items = uint64_t(p.num_seqs) * p.num_q_heads;
    combine_kernel<D><<<unsigned((items + kCombineWarps - 1) / kCombineWarps), 32 * kCombineWarps, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
  }
  return KV_OK;
}

}  // namespace

namespace {

// Pieces a sequence of up to max_tiles tiles can be cut into by chunks of
// c tiles: a range [a, a + n) meets floor((a + n - 1) / c) - floor(a / c) + 1
// chunks, at most ceil((n - 1) / c) + 1.
uint64_t max_pieces(uint64_t max_tiles, uint64_t c) {
  return max_tiles <= 1 ? max_tiles : (max_tiles - 2) / c + 2;
}

// The per-(sequence, head group) piece counts, ahead of the partials.
uint64_t count_bytes(uint32_t num_seqs, uint32_t num_kv_heads) {
  return (uint64_t(num_seqs) * num_kv_heads * 4 + kHeaderBytes - 1) / kHeaderBytes * kHeaderBytes;
}

}  // namespace

size_t decode_workspace_bytes(uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                              uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size) {
  const uint64_t max_tiles = (uint64_t(max_blocks_per_seq) * block_size + kTile - 1) / kTile;
  const uint64_t max_splits = max_pieces(max_tiles, kSplitUnitTiles);
  return kHeaderBytes + count_bytes(num_seqs, num_kv_heads) +
         uint64_t(num_seqs) * max_splits * num_q_heads * (uint64_t(head_dim) + 2) * 4;
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  const uint32_t group = a.num_q_heads / a.num_kv_heads;
  const bool fp8_v = a.fp8 && a.fp8_v;
  Geometry geo = geometry(a.fp8, fp8_v, a.head_dim, a.num_kv_heads, group, dev.max_smem_optin);
  if (geo.stages < 2) return KV_ERR_UNSUPPORTED;
  geo.ctas_per_sm = 1;
  if (fp8_v && a.head_dim <= 128 && geo.nt == 1) {  // two_ctas_per_sm()
    // two CTAs per SM when a ring of two or more stages with the same heads
    // per item fits in half of the SM's shared memory (1 KB of it is
    // reserved per CTA): 0.957 -> 0.883 ms on the mixed-length FP8 K+V
    // decode, 1.344 -> 1.248 ms on 128 sequences of 32,768 positions; the
    // other variants were 1-3% slower so
    const Geometry half = geometry(a.fp8, fp8_v, a.head_dim, a.num_kv_heads, group,
                                   dev.max_smem_sm / 2 - 1024 - 256);  // 256: the kernel's static shared memory
    if (half.stages >= 2 && half.heads_per_item == geo.heads_per_item) {
      geo = half;
      geo.ctas_per_sm = 2;
    }
  }

  DecodeParams p{};
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.output = a.output;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.block_shift = uint32_t(__builtin_ctz(a.block_size));
  p.group = group;
  p.heads_per_item = geo.heads_per_item;
  p.num_head_groups = (a.num_kv_heads + geo.heads_per_item - 1) / geo.heads_per_item;
  p.q_stride = a.q_stride;
  p.sliding_window = a.sliding_window;
  p.score_scale = a.inv_sqrt_d * kLog2e * (a.fp8 ? a.k_scale : 1.0f);
  p.out_scale = fp8_v ? a.v_scale * (1.0f / 256.0f) : 1.0f;
  p.stages = geo.stages;
  p.stage_bytes = geo.stage_bytes;
  p.k_bytes = geo.k_bytes;
  p.v_bytes = geo.v_bytes;

  // Split-KV (stream-K chunks) when a workspace is registered and holds the
  // header, the piece counts and partials for the most pieces a sequence can
  // be cut into: chunks are at least kMinChunkTiles long, longer if the
  // workspace holds fewer pieces per sequence than that needs.
  const uint64_t max_tiles = (uint64_t(a.max_blocks_per_seq) * a.block_size + kTile - 1) / kTile;
  const uint64_t fixed = kHeaderBytes + count_bytes(a.num_seqs, a.num_kv_heads);
  p.max_splits = 0;
  p.min_chunk_tiles = 0;
  if (a.workspace && a.workspace_bytes > fixed && max_tiles > 1) {
    const uint64_t per_split = uint64_t(a.num_seqs) * a.num_q_heads * (a.head_dim + 2) * 4;
    const uint64_t fit = (a.workspace_bytes - fixed) / per_split;
    uint64_t c = 0;
    if (fit >= max_pieces(max_tiles, kMinChunkTiles))
      c = kMinChunkTiles;
    else if (fit >= 2)
      c = (max_tiles - 2) / (fit - 1) + 1;  // the least c with max_pieces(max_tiles, c) <= fit
    if (c) {
      if (a.workspace_fresh &&
          cudaMemsetAsync(a.workspace, 0, kHeaderBytes, stream) != cudaSuccess)
        return KV_ERR_CUDA;
      p.min_chunk_tiles = uint32_t(c);
      p.max_splits = uint32_t(max_pieces(max_tiles, c));
      uint8_t* ws = static_cast<uint8_t*>(a.workspace);
      p.ws_header = reinterpret_cast<uint32_t*>(ws);
      p.ws_count = reinterpret_cast<uint32_t*>(ws + kHeaderBytes);
      p.ws_o = reinterpret_cast<float*>(ws + fixed);
      p.ws_ml = p.ws_o + uint64_t(a.num_seqs) * p.max_splits * a.num_q_heads * a.head_dim;
    }
  }

  const int key = (fp8_v ? 200 : a.fp8 ? 100 : 0) + int(a.head_dim / 64) * 10 + int(geo.nt);
  switch (key) {
    case 11: return launch_decode_t<false, false, 64, 1>(a, stream, geo, p);
    case 12: return launch_decode_t<false, false, 64, 2>(a, stream, geo, p);
    case 21: return launch_decode_t<false, false, 128, 1>(a, stream, geo, p);
    case 22: return launch_decode_t<false, false, 128, 2>(a, stream, geo, p);
    case 41: return launch_decode_t<false, false, 256, 1>(a, stream, geo, p);
    case 42: return launch_decode_t<false, false, 256, 2>(a, stream, geo, p);
    case 111: return launch_decode_t<true, false, 64, 1>(a, stream, geo, p);
    case 112: return launch_decode_t<true, false, 64, 2>(a, stream, geo, p);
    case 121: return launch_decode_t<true, false, 128, 1>(a, stream, geo, p);
    case 122: return launch_decode_t<true, false, 128, 2>(a, stream, geo, p);
    case 141: return launch_decode_t<true, false, 256, 1>(a, stream, geo, p);
    case 142: return launch_decode_t<true, false, 256, 2>(a, stream, geo, p);
    case 211: return launch_decode_t<true, true, 64, 1>(a, stream, geo, p);
    case 212: return launch_decode_t<true, true, 64, 2>(a, stream, geo, p);
    case 221: return launch_decode_t<true, true, 128, 1>(a, stream, geo, p);
    case 222: return launch_decode_t<true, true, 128, 2>(a, stream, geo, p);
    case 241: return launch_decode_t<true, true, 256, 1>(a, stream, geo, p);
    case 242: return launch_decode_t<true, true, 256, 2>(a, stream, geo, p);
    default: return KV_ERR_UNSUPPORTED;
  }
}

cudaError_t read_and_clear_decode_error(uint32_t* bits) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_decode_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(uint32_t));
}

#ifdef PAGEDKV_DEBUG_BOUNDS
PAGEDKV_DEBUG_UNIT(decode)
#endif

}  // namespace pagedkv
