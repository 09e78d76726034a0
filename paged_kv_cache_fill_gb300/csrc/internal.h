// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace pagedkv {

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int max_smem_optin = 0;  // bytes of shared memory a block may opt into
  int max_smem_sm = 0;     // bytes of shared memory per SM (each resident block also reserves 1 KB)
  int cc_major = 0, cc_minor = 0;
};

// Cached properties of the current device (queried once per device).
const DeviceInfo& device_info();

// Launchers (asynchronous on `stream`; return the launch's cudaError_t).
cudaError_t launch_fill_slots(int64_t* slots, const int32_t* block_table, uint32_t start_pos,
                              uint32_t count, uint32_t block_size, cudaStream_t stream);

cudaError_t launch_copy_rows(const uint16_t* src0, const uint16_t* src1, uint16_t* dst0,
                             uint16_t* dst1, const int64_t* slot_mapping, uint32_t num_tokens,
                             uint32_t row_elems, uint32_t stride0, uint32_t stride1,
                             cudaStream_t stream);

// FP8 K write; V is copied as BF16 (fp8_v false) or quantised by v_scale.
cudaError_t launch_write_fp8(const uint16_t* key, const uint16_t* value, uint8_t* k_cache_fp8, void* v_cache,
                             bool fp8_v, const int64_t* slot_mapping, uint32_t num_tokens, uint32_t row_elems,
                             uint32_t key_stride, uint32_t value_stride, float k_scale, float v_scale,
                             cudaStream_t stream);

// Fused RMSNorm/RoPE K write. pos_h/pos_w non-null selects the MRoPE
// variant (position of pair i from positions/pos_h/pos_w by i % 3); fp8_out
// stores E4M3(o * inv_scale) into a uint8 pool instead of BF16(o).
cudaError_t launch_fused_k_norm_rope(const uint16_t* k_in, const uint16_t* k_norm_weight,
                                     const int32_t* positions, const int32_t* pos_h, const int32_t* pos_w,
                                     void* k_cache, bool fp8_out, float inv_scale,
                                     const int64_t* slot_mapping, uint32_t num_tokens,
                                     uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                     float rms_eps, float theta, cudaStream_t stream);

// Tensor map over a cache pool [num_blocks, block_size, num_kv_heads,
// head_dim] (bf16, or e4m3 when fp8) whose box is one 128-byte chunk x 16
// slots x (heads_per_item x chunks per head, or box_chunks when nonzero):
// the shared-memory tile is [chunk][slot][128 B], 128-byte swizzled by slot
// row.
bool encode_pool_map(CUtensorMap* map, const void* base, bool fp8, uint32_t num_kv_heads, uint32_t head_dim,
                     uint32_t heads_per_item, uint32_t box_chunks = 0);

// Multi-token (chunked-prefill) paged attention; returns a KV_* status.
struct PrefillArgs {
  const uint16_t* q;
  const void* k_cache;  // bf16 or e4m3 pool
  const void* v_cache;  // bf16 or (fp8_v) e4m3 pool
  float* output;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  uint32_t max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, block_size;
  float inv_sqrt_d, k_scale, v_scale;
  uint32_t q_stride, sliding_window;
  bool fp8, fp8_v;  // fp8_v implies fp8
};
int launch_prefill(const PrefillArgs& a, cudaStream_t stream);
cudaError_t read_and_clear_prefill_error(uint32_t* bits);

// Paged decode. `workspace` may be null (then no split-KV).
struct DecodeArgs {
  const uint16_t* q;
  const void* k_cache;  // bf16 or e4m3 pool
  const void* v_cache;  // bf16 pool, or e4m3 when fp8_v
  float* output;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  uint32_t max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  float inv_sqrt_d, k_scale;
  uint32_t q_stride, sliding_window;
  bool fp8;
  bool fp8_v;     // V is E4M3 too (requires fp8), dequantised by v_scale
  float v_scale;
  void* workspace;
  size_t workspace_bytes;
  bool workspace_fresh;  // registered since the last decode: its counters must be zeroed first
};

size_t decode_workspace_bytes(uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                              uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size);

// Returns KV_* status (host-side checks) and launches on `stream`.
int launch_decode(const DecodeArgs& a, cudaStream_t stream);

// The decode kernels' device fault word (read and clear).
cudaError_t read_and_clear_decode_error(uint32_t* bits);

// The fused K write's device fault word (read and clear).
cudaError_t read_and_clear_fused_error(uint32_t* bits);

#ifdef PAGEDKV_DEBUG_BOUNDS
// The bounds-checking build's per-unit pool size and fault word (common.cuh).
cudaError_t debug_set_pool_kv_write(uint32_t num_blocks, uint32_t block_size);
cudaError_t debug_set_pool_fused_k(uint32_t num_blocks, uint32_t block_size);
cudaError_t debug_set_pool_decode(uint32_t num_blocks, uint32_t block_size);
cudaError_t debug_set_pool_prefill(uint32_t num_blocks, uint32_t block_size);
cudaError_t debug_read_and_clear_kv_write(uint32_t* bits);
cudaError_t debug_read_and_clear_fused_k(uint32_t* bits);
cudaError_t debug_read_and_clear_decode(uint32_t* bits);
cudaError_t debug_read_and_clear_prefill(uint32_t* bits);
cudaError_t debug_set_wait_limit_decode(uint64_t ns);
#endif

}  // namespace pagedkv
