/*
 * pagedkv.h — C ABI of the GB300 (sm_103a) paged KV-cache library.
 *
 * The paged KV-cache hot path of an LLM decode server: slot filling, cache
 * writes (BF16, FP8-E4M3 K with BF16 V, fused RMSNorm/RoPE K, V only) and
 * paged decode attention (BF16 and FP8 K). The calls and their argument
 * order follow the Rust launchers on the pages
 *   "spark_model/layers/ops/kv_cache.rs"              (written [kv_cache.rs]) and
 *   "metrale_model_layers/layers/ops/kv_cache_fp8k.rs" (written [kv_cache_fp8k.rs]),
 * with the launcher's GPU/kernel handles dropped and the stream last.
 *
 * Conventions for every call
 *   - Pointers marked "device" are CUDA device (or managed) memory owned by
 *     the caller; the library never allocates, frees or keeps them, and never
 *     synchronises. Every call is asynchronous on `stream` and returns once
 *     the work is queued. The stream is a cudaStream_t passed as void* (NULL
 *     means the legacy default stream), so that this header and its callers
 *     (C code, ctypes) need no CUDA header; the scope table's listing writes
 *     it as cudaStream_t.
 *   - BF16 data are passed as their 16-bit patterns (kv_bf16_t), FP8 data as
 *     E4M3 ("FN": no infinities, max 448, NaN 0x7F/0xFF) codes (kv_e4m3_t).
 *   - Cache pools are [num_blocks, block_size, num_kv_heads, head_dim], row
 *     major ("NHD" within a block). A flat slot s is row s % block_size of
 *     block s / block_size, so its num_kv_heads * head_dim elements start at
 *     element s * num_kv_heads * head_dim of the pool base pointer.
 *   - A negative slot in slot_mapping marks a padding token: nothing is
 *     written for it.
 *   - Return value: KV_OK, or an error code below. Argument errors are found
 *     on the host before anything is queued. Errors in device-resident data
 *     (a slot or block id outside the pool, a table shorter than a sequence)
 *     cannot be seen on the host; keeping them in range is the caller's
 *     contract, as with the pages' kernels. Calls with no work
 *     (count == 0, num_tokens == 0, num_seqs == 0) return KV_OK and launch
 *     nothing, as [kv_cache.rs] `fill_slots_from_block_table` does for
 *     count == 0.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PAGEDKV_API __attribute__((visibility("default")))
#else
#define PAGEDKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kv_bf16_t; /* BF16 bit pattern */
typedef uint8_t kv_e4m3_t;  /* FP8 E4M3 code */

enum kv_status {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,  /* null pointer with work to do, bad shape or stride */
    KV_ERR_UNSUPPORTED = 2,  /* legal but outside what the kernels implement */
    KV_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed */
    KV_ERR_DEVICE = 4        /* kv_get_device_error only: a kernel reported a fault in device
                                data or a wait timeout since the last read */
};

/* Human-readable text of a status code (static storage). */
PAGEDKV_API const char *kv_status_string(int status);

/* ------------------------------------------------------------------------
 * Slot filling.  [kv_cache.rs] `fill_slots_from_block_table`.
 *
 * slots[i] = block_table[p / block_size] * block_size + p % block_size for
 * p = start_pos + i, i < count.
 *   slots        device int64[count], written.
 *   block_table  device int32[ceil((start_pos + count) / block_size)], the
 *                sequence's physical block ids in logical order. A negative
 *                id gives a negative (skipped) slot.
 *   block_size   > 0.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_fill_slots(int64_t *slots, const int32_t *block_table, uint32_t start_pos, uint32_t count,
                  uint32_t block_size, void *stream);

/* ------------------------------------------------------------------------
 * BF16 cache write.  [kv_cache.rs] `reshape_and_cache` ("BF16 reshape and
 * cache — no quantization, direct BF16 copy"; its kernel-name line is a
 * garbled FP8 name and is not followed).
 *
 * For token t < num_tokens with slot = slot_mapping[t] >= 0 and head h:
 *   k_cache[slot][h][:] = key[t * key_stride + h * head_dim + :]
 *   v_cache[slot][h][:] = value[t * value_stride + h * head_dim + :]
 * bit for bit.
 *   key, value        device bf16, row t at element t * key_stride (resp.
 *                     value_stride); strides >= num_kv_heads * head_dim.
 *   k_cache, v_cache  device bf16 pools.
 *   slot_mapping      device int64[num_tokens].
 * Distinct tokens must not share a slot (their order is then unspecified).
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_write_bf16(const kv_bf16_t *key, const kv_bf16_t *value, kv_bf16_t *k_cache,
                  kv_bf16_t *v_cache, const int64_t *slot_mapping, uint32_t num_tokens,
                  uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                  uint32_t key_stride, uint32_t value_stride, void *stream);

/* ------------------------------------------------------------------------
 * FP8-K / BF16-V cache write.  [kv_cache_fp8k.rs] module invariants: K is
 * stored as k / k_scale in E4M3 in the NHD layout; argument order of
 * `reshape_and_cache_fp8k_turbo3v` without its TurboQuant-V arguments. V is a
 * BF16 copy as in kv_write_bf16.
 *
 * code = E4M3(round-to-nearest-even, saturating to +-448)(fp32(k) / k_scale),
 * where the quotient is the IEEE binary32 division rounded to nearest; NaN
 * inputs give 0x7F. Bit-exact.
 *   k_cache_fp8  device uint8 pool; v_cache device bf16 pool.
 *   k_scale      per-tensor scale, finite and > 0.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_write_fp8k(const kv_bf16_t *key, const kv_bf16_t *value, kv_e4m3_t *k_cache_fp8,
                  kv_bf16_t *v_cache, const int64_t *slot_mapping, uint32_t num_tokens,
                  uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                  uint32_t key_stride, uint32_t value_stride, float k_scale, void *stream);

/* ------------------------------------------------------------------------
 * FP8 K and V cache write.  [kv_cache.rs] `reshape_and_cache_fp8`: K stored
 * as k / k_scale and V as v / v_scale, both E4M3 with the rule of
 * kv_write_fp8k, into two uint8 pools of the NHD layout. Argument order of
 * that launcher (scales before strides); its cache_stride is implied by the
 * layout and dropped. Bit-exact.
 *   k_scale, v_scale  per-tensor scales, finite and > 0.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_write_fp8(const kv_bf16_t *key, const kv_bf16_t *value, kv_e4m3_t *k_cache_fp8,
                             kv_e4m3_t *v_cache_fp8, const int64_t *slot_mapping, uint32_t num_tokens,
                             uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size, float k_scale,
                             float v_scale, uint32_t key_stride, uint32_t value_stride, void *stream);

/* ------------------------------------------------------------------------
 * Fused K path.  [kv_cache.rs] `fused_k_norm_rope_cache_write_bf16`: RMSNorm,
 * then RoPE, then the BF16 paged write in one kernel, K kept above BF16
 * precision throughout and rounded once at the write.
 *
 * For token t with slot >= 0 and head h, x = k_in[t][h][:] (contiguous
 * [num_tokens, num_kv_heads, head_dim], no stride argument on the page):
 *   y_d = x_d / sqrt(mean(x^2) + rms_eps) * k_norm_weight[d]
 *   for i < rotary_dim/2, angle = positions[t] * theta^(-2i/rotary_dim):
 *     o_i = y_i cos - y_{i+R/2} sin,  o_{i+R/2} = y_{i+R/2} cos + y_i sin
 *   o_d = y_d for d >= rotary_dim
 *   k_cache[slot][h][d] = BF16_RNE(o_d)
 * The result is within 1 BF16 ulp of the exactly rounded value.
 *   k_norm_weight  device bf16[head_dim], shared by all heads.
 *   positions      device int32[num_tokens], >= 0.
 *   rotary_dim     even, 8 <= rotary_dim <= head_dim, multiple of 8.
 * The V half goes through kv_write_v_only.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_write_fused_k_norm_rope_bf16(const kv_bf16_t *k_in, const kv_bf16_t *k_norm_weight,
                                    const int32_t *positions, kv_bf16_t *k_cache,
                                    const int64_t *slot_mapping, uint32_t num_tokens,
                                    uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                    uint32_t block_size, float rms_eps, float theta, void *stream);

/* ------------------------------------------------------------------------
 * MRoPE-interleaved fused K path. [kv_cache.rs]
 * `fused_k_norm_rope_cache_write_bf16_mrope`: as
 * kv_write_fused_k_norm_rope_bf16, but rotation pair i of token t turns by
 * pos * theta^(-2i/rotary_dim) with pos = (pos_t, pos_h, pos_w)[i % 3][t].
 * With pos_t == pos_h == pos_w the result is bit-identical to
 * kv_write_fused_k_norm_rope_bf16.
 *   pos_t, pos_h, pos_w  device int32[num_tokens] each.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_write_fused_k_norm_rope_bf16_mrope(
    const kv_bf16_t *k_in, const kv_bf16_t *k_norm_weight, const int32_t *pos_t, const int32_t *pos_h,
    const int32_t *pos_w, kv_bf16_t *k_cache, const int64_t *slot_mapping, uint32_t num_tokens,
    uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim, uint32_t block_size, float rms_eps,
    float theta, void *stream);

/* ------------------------------------------------------------------------
 * FP8-output fused K path. [kv_cache.rs] `fused_k_norm_rope_cache_write_fp8`:
 * the same RMSNorm and RoPE with no BF16 rounding; the result times
 * inv_scale (finite, > 0; inv_scale = 1 / k_scale of the FP8-K decode) is
 * cast once to E4M3, round to nearest even, saturating to +-448. The code
 * equals the correctly rounded one except where the exact scaled value lies
 * within ~2^-19 (relative) of the midpoint between two codes; there either
 * neighbour may be stored.
 *   k_cache_fp8  device uint8 pool [num_blocks, block_size, num_kv_heads, head_dim].
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_write_fused_k_norm_rope_fp8(const kv_bf16_t *k_in, const kv_bf16_t *k_norm_weight,
                                               const int32_t *positions, kv_e4m3_t *k_cache_fp8,
                                               const int64_t *slot_mapping, uint32_t num_tokens,
                                               uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                               uint32_t block_size, float rms_eps, float theta, float inv_scale,
                                               void *stream);

/* ------------------------------------------------------------------------
 * V-only write.  [kv_cache.rs] `reshape_and_cache_flash_v_only`: the V half
 * of kv_write_bf16, so that the fused K kernel stays the only writer of K.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_write_v_only(const kv_bf16_t *value, kv_bf16_t *v_cache, const int64_t *slot_mapping,
                    uint32_t num_tokens, uint32_t num_kv_heads, uint32_t head_dim,
                    uint32_t block_size, uint32_t value_stride, void *stream);

/* ------------------------------------------------------------------------
 * Paged decode attention.  [kv_cache.rs] `paged_decode_attn_fp8` doc (one
 * query per (query head, sequence); block_tables int32[num_seqs *
 * max_blocks_per_seq]; seq_lens int32[num_seqs]) and the argument list of
 * `paged_decode_attn_bf16k_turbo3v` without its TurboQuant-V arguments
 * (q_stride, sliding_window). [kv_cache_fp8k.rs]: the FP8 variant multiplies
 * the stored K by k_scale, which follows inv_sqrt_d in the argument list.
 *
 * For sequence s and query head h, with g = num_q_heads / num_kv_heads and
 * KV head h / g, L = seq_lens[s] (cached tokens, the current token included)
 * and start = (sliding_window > 0 ? max(0, L - sliding_window) : 0):
 *   position p in [start, L) lives at row p % block_size of block
 *   block_tables[s * max_blocks_per_seq + p / block_size];
 *   score_p = inv_sqrt_d * (q[s * q_stride + h * head_dim + :] . k_p)
 *   output[s][h][:] = sum_p softmax(score)_p * v_p     (zeros if L == 0)
 *   q       device bf16; q_stride (elements between sequences) >= num_q_heads * head_dim.
 *   output  device float32[num_seqs, num_q_heads, head_dim], written.
 *   seq_lens[s] <= max_blocks_per_seq * block_size.
 * Supported: head_dim in {64, 128, 256}; block_size a power
 * of two in [16, 256]; g <= 16; q, caches and q_stride 16-byte aligned;
 * output 8-byte aligned. Anything else returns KV_ERR_UNSUPPORTED.
 * With a workspace registered by kv_set_decode_workspace, the positions of
 * all sequences are shared out equally among the CTAs and a sequence split
 * between CTAs is merged afterwards (flash-decoding); without one every
 * (sequence, KV head group) runs in one CTA (same result, less parallelism).
 * ---------------------------------------------------------------------- */
PAGEDKV_API int paged_decode_attn_bf16(const kv_bf16_t *q, const kv_bf16_t *k_cache, const kv_bf16_t *v_cache,
                           float *output, const int32_t *block_tables, const int32_t *seq_lens,
                           uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                           uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                           float inv_sqrt_d, uint32_t q_stride, uint32_t sliding_window,
                           void *stream);

PAGEDKV_API int paged_decode_attn_fp8k(const kv_bf16_t *q, const kv_e4m3_t *k_cache_fp8,
                           const kv_bf16_t *v_cache, float *output, const int32_t *block_tables,
                           const int32_t *seq_lens, uint32_t max_blocks_per_seq,
                           uint32_t num_seqs, uint32_t num_q_heads, uint32_t num_kv_heads,
                           uint32_t head_dim, uint32_t block_size, float inv_sqrt_d,
                           float k_scale, uint32_t q_stride, uint32_t sliding_window,
                           void *stream);

/* ------------------------------------------------------------------------
 * FP8 K and V paged decode.  [kv_cache.rs] `paged_decode_attn_fp8` (its
 * argument order, with num_seqs, q_stride and sliding_window as in the
 * calls above and cache_stride dropped): as paged_decode_attn_fp8k, with
 * v_p = E4M3 code * v_scale (v_scale finite and > 0) read from a uint8 V
 * pool. Supported head_dim: {128, 256}.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int paged_decode_attn_fp8(const kv_bf16_t *q, const kv_e4m3_t *k_cache_fp8,
                                      const kv_e4m3_t *v_cache_fp8, float *output, const int32_t *block_tables,
                                      const int32_t *seq_lens, uint32_t max_blocks_per_seq, uint32_t num_seqs,
                                      uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                      uint32_t block_size, float inv_sqrt_d, float k_scale, float v_scale,
                                      uint32_t q_stride, uint32_t sliding_window, void *stream);

/* ------------------------------------------------------------------------
 * Multi-token (chunked-prefill) paged attention.  [kv_cache.rs] "Batched
 * prefill variants (N tokens)" gives only the heading; the reading here:
 * sequence s brings n_s = query_start_loc[s+1] - query_start_loc[s] query
 * tokens, the last n_s of its seq_lens[s] cached positions (their K/V
 * already written). Query j of s (row query_start_loc[s] + j of q, at
 * position P = seq_lens[s] - n_s + j) attends causally, over positions
 * [start, P] with start = (sliding_window > 0 ? max(0, P + 1 -
 * sliding_window) : 0): exactly what the paged decode attends for that
 * sequence cut to length P + 1. A query with P < 0 gives zeros. GQA,
 * inv_sqrt_d, the block tables and (FP8) k_scale are as in the decode calls.
 *   q                bf16 rows [num_q_tokens], row stride q_stride elements,
 *                    head h at +h * head_dim.
 *   query_start_loc  device int32[num_seqs + 1], non-decreasing, from 0 to
 *                    num_q_tokens (a violation sets bit 2 of the device
 *                    fault word and that sequence's rows are skipped).
 *   output           device float32[num_q_tokens, num_q_heads, head_dim].
 * Precision: scores and sums in fp32; the PV product takes the softmax
 * weights as f16 (one rounding, relative error at most 2^-11) against V as
 * f16: E4M3 codes exactly, BF16 values as v * 2^-8 rounded to f16, exact for
 * 2^-6 <= |v| < 2^24 and within 2^-17 below. BF16 V values of magnitude
 * 2^24 or more are outside the supported range: the outputs of every query
 * whose keys share a 128-key tile with one are not finite.
 * Supported: head_dim 64 or 128; block_size a power of two in
 * [16, 256]; q, caches, q_stride and output 16-byte aligned. No workspace
 * is used.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int paged_prefill_attn_bf16(const kv_bf16_t *q, const kv_bf16_t *k_cache, const kv_bf16_t *v_cache,
                                        float *output, const int32_t *block_tables, const int32_t *seq_lens,
                                        const int32_t *query_start_loc, uint32_t max_blocks_per_seq,
                                        uint32_t num_seqs, uint32_t num_q_tokens, uint32_t num_q_heads,
                                        uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                                        float inv_sqrt_d, uint32_t q_stride, uint32_t sliding_window,
                                        void *stream);

PAGEDKV_API int paged_prefill_attn_fp8k(const kv_bf16_t *q, const kv_e4m3_t *k_cache_fp8,
                                        const kv_bf16_t *v_cache, float *output, const int32_t *block_tables,
                                        const int32_t *seq_lens, const int32_t *query_start_loc,
                                        uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_tokens,
                                        uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                        uint32_t block_size, float inv_sqrt_d, float k_scale, uint32_t q_stride,
                                        uint32_t sliding_window, void *stream);

/* Multi-token paged attention over an FP8 K and V cache (the cache that
 * kv_write_fp8 fills and paged_decode_attn_fp8 reads): as
 * paged_prefill_attn_fp8k, with v_p = E4M3 code * v_scale (v_scale finite and
 * > 0) read from a uint8 V pool. head_dim 64 or 128. */
PAGEDKV_API int paged_prefill_attn_fp8(const kv_bf16_t *q, const kv_e4m3_t *k_cache_fp8,
                                       const kv_e4m3_t *v_cache_fp8, float *output, const int32_t *block_tables,
                                       const int32_t *seq_lens, const int32_t *query_start_loc,
                                       uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_tokens,
                                       uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                       uint32_t block_size, float inv_sqrt_d, float k_scale, float v_scale,
                                       uint32_t q_stride, uint32_t sliding_window, void *stream);

/* ------------------------------------------------------------------------
 * FP8-K paged decode without any caller-provided memory. The source pages
 * have no counterpart of this call; it exists for callers that cannot give
 * the library a device allocation: applications whose device memory belongs
 * to another allocator (a framework memory pool, a serving engine that
 * reserves all of HBM for its KV cache) cannot set a raw buffer aside for a
 * library, and a cudaMalloc of their own would fail or break that
 * allocator's accounting. Like every call here it uses the CUDA API, so it
 * must not be made from a host function enqueued with cudaLaunchHostFunc.
 *
 * Same arguments, results and limits as paged_decode_attn_fp8k; the
 * split-KV scratch comes from a fixed 64 MiB array in the library's own
 * device memory, which every GPU that loads the library keeps until the
 * process exits. The call allocates and frees nothing. It returns
 * KV_ERR_UNSUPPORTED when the shape's worst-case scratch
 * (kv_decode_workspace_bytes of the same arguments) exceeds 64 MiB.
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and caches it: make that
 * first call before any stream capture, and do not call it on a device
 * after a cudaDeviceReset in the same process (the cached address belonged
 * to the reset context). All calls share the one array, which keeps the
 * previous call's contents; each call clears the counters that must start
 * at zero on its own stream first. Calls whose work may overlap on the GPU
 * (different streams, other devices' calls aside) race on the array: order
 * them.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int paged_decode_attn_fp8k_static_scratch(
    const kv_bf16_t *q, const kv_e4m3_t *k_cache_fp8, const kv_bf16_t *v_cache, float *output,
    const int32_t *block_tables, const int32_t *seq_lens, uint32_t max_blocks_per_seq, uint32_t num_seqs,
    uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size, float inv_sqrt_d,
    float k_scale, uint32_t q_stride, uint32_t sliding_window, void *stream);

/* ------------------------------------------------------------------------
 * Split-KV workspace (not on the pages: flash-decoding partials and the
 * combine step need scratch). The caller allocates device memory of at
 * least kv_decode_workspace_bytes(...) for the largest decode it will run
 * and registers it for the current device; NULL (or 0 bytes) unregisters.
 *
 * kv_decode_workspace_bytes takes the decode's table geometry
 * (max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim,
 * block_size: the same values the decode call gets) rather than a split
 * count: the kernel cuts the tiles of all sequences (16 positions each),
 * taken in sequence order, into equal chunks, about one per SM, sized on
 * the device from the actual sequence lengths, and a sequence is split
 * where a chunk boundary falls inside it; a caller cannot know those splits
 * in advance. The size covers the worst case, a sequence as long as its
 * table allows (T = ceil(max_blocks_per_seq * block_size / 16) tiles) cut
 * by chunks of 16 tiles into P = (T <= 1 ? T : (T - 2) / 16 + 2) pieces
 * (integer division): 256 bytes of header, then num_seqs * num_kv_heads
 * 4-byte piece counts rounded up to a multiple of 256 bytes, then
 * num_seqs * P * num_q_heads * (head_dim + 2) * 4 bytes of partials. A
 * smaller registered workspace is still used, with longer chunks (or none
 * where it holds fewer than two pieces per sequence), and gives the same
 * results.
 * Decode calls on that device use it in stream order, so decode calls that
 * may run concurrently on different streams need separate devices or must be
 * ordered by the caller. The library never frees it.
 * ---------------------------------------------------------------------- */
PAGEDKV_API size_t kv_decode_workspace_bytes(uint32_t max_blocks_per_seq, uint32_t num_seqs,
                                 uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                                 uint32_t block_size);
PAGEDKV_API int kv_set_decode_workspace(void *device_ptr, size_t bytes);

/* ------------------------------------------------------------------------
 * Device-side fault word. Kernels that meet bad device data (a slot mapping
 * or table value they refuse to use, a pipeline wait that ran out of time)
 * skip the work, set a bit here and return instead of faulting or hanging.
 * kv_get_device_error synchronises the current device, returns the bits seen
 * since the last clear (0 = none) in *bits and clears them. Its status is
 * KV_ERR_DEVICE when any bit was set, KV_OK when none was, KV_ERR_CUDA when
 * the synchronisation or a read failed (*bits then unspecified) and
 * KV_ERR_INVALID_ARG for a null bits pointer. The other calls never
 * synchronise, so they cannot see these faults and never return
 * KV_ERR_DEVICE.
 *   bit 0: a decode pipeline wait timed out
 *   bit 1: seq_lens[s] exceeded max_blocks_per_seq * block_size (clamped)
 *   bit 2: a prefill query_start_loc was decreasing, negative or past
 *          num_q_tokens (that sequence skipped)
 *   bit 3: (bounds-checking build only) a slot or block id outside the pool
 *          set by kv_debug_set_pool
 *   (bit 0 also covers the prefill pipeline and the fused K write's wait
 *   for its shared-memory copy of the sin/cos table)
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_get_device_error(uint32_t *bits);

/* ------------------------------------------------------------------------
 * Bounds checking (a separate build of this library, compiled with
 * PAGEDKV_DEBUG_BOUNDS: libpagedkv_debug.so). Device data that index the
 * pools (slot mappings, block tables) are the caller's contract and go
 * unchecked in the product build. In the bounds-checking build every kernel
 * checks each slot against num_blocks * block_size and each block id
 * against num_blocks, as set here for the current device (num_blocks 0:
 * unchecked, the initial state). A write skips a row whose slot is out of
 * the pool; an attention call reads block 0 in place of a block id out of
 * the pool; either sets bit 3 of the fault word. Nothing traps. The call
 * synchronises. The product build returns KV_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------- */
PAGEDKV_API int kv_debug_set_pool(uint32_t num_blocks, uint32_t block_size);

/* Bounds-checking build only: how long each pipeline wait of the paged
 * decode kernels (a consumer waiting for a loaded tile, the loader waiting
 * for a free stage) may take on the current device before the kernel gives
 * up, sets bit 0 of the fault word and returns; 0 restores the default of
 * 2 s, which the product build always uses. Whatever the limit, a decode CTA
 * that gave up first waits (with the 2 s limit) until every copy it issued
 * into its shared memory has landed, so that nothing is left in flight.
 * The call synchronises. The product build returns KV_ERR_UNSUPPORTED. */
PAGEDKV_API int kv_debug_set_wait_limit(uint64_t nanoseconds);

/* Number of decode CTAs per SM and SM count the library launches with on the
 * current device, for benchmarks (optional outputs may be NULL). */
PAGEDKV_API int kv_device_info(int *num_sms, int *decode_ctas);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
