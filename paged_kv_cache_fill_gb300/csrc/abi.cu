// C ABI of the paged KV-cache library: argument checks, dispatch to the
// kernels, the per-device split-KV workspace registry and device queries.
// Every entry point validates on the host, queues its kernels on the
// caller's stream and returns; nothing here allocates or synchronises except
// kv_get_device_error (documented).
#include <math.h>

#include <mutex>

#include "../../include/pagedkv.h"
#include "internal.h"

namespace pagedkv {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
void* g_ws_ptr[kMaxDevices];
size_t g_ws_bytes[kMaxDevices];
bool g_ws_fresh[kMaxDevices];

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}
}  // namespace

const DeviceInfo& device_info() {
  static DeviceInfo invalid;
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return invalid;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& info = g_devices[d];
  if (info.device != d) {
    cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, d);
    cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    cudaDeviceGetAttribute(&info.max_smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
    cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, d);
    info.device = d;
  }
  return info;
}

}  // namespace pagedkv

using namespace pagedkv;

namespace {

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? KV_OK : KV_ERR_CUDA; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool is_pow2(uint32_t x) { return x && !(x & (x - 1)); }

// Shared checks of the row-copy style writes.
int check_rows(uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size) {
  if (num_kv_heads == 0 || head_dim == 0 || block_size == 0) return KV_ERR_INVALID_ARG;
  if (uint64_t(num_kv_heads) * head_dim > (1u << 20)) return KV_ERR_UNSUPPORTED;
  return KV_OK;
}

}  // namespace

extern "C" {

const char* kv_status_string(int status) {
  switch (status) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_UNSUPPORTED: return "unsupported shape, alignment or device";
    case KV_ERR_CUDA: return "CUDA error";
    case KV_ERR_DEVICE: return "a kernel reported a fault in device data or a wait timeout";
    default: return "unknown status";
  }
}

int kv_fill_slots(int64_t* slots, const int32_t* block_table, uint32_t start_pos, uint32_t count,
                  uint32_t block_size, void* stream) {
  if (count == 0) return KV_OK;
  if (!slots || !block_table || block_size == 0) return KV_ERR_INVALID_ARG;
  return from_cuda(launch_fill_slots(slots, block_table, start_pos, count, block_size, as_stream(stream)));
}

int kv_write_bf16(const kv_bf16_t* key, const kv_bf16_t* value, kv_bf16_t* k_cache, kv_bf16_t* v_cache,
                  const int64_t* slot_mapping, uint32_t num_tokens, uint32_t num_kv_heads,
                  uint32_t head_dim, uint32_t block_size, uint32_t key_stride, uint32_t value_stride,
                  void* stream) {
  if (num_tokens == 0) return KV_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return KV_ERR_INVALID_ARG;
  if (int r = check_rows(num_kv_heads, head_dim, block_size)) return r;
  const uint32_t row = num_kv_heads * head_dim;
  if (key_stride < row || value_stride < row) return KV_ERR_INVALID_ARG;
  return from_cuda(launch_copy_rows(key, value, k_cache, v_cache, slot_mapping, num_tokens, row, key_stride,
                                    value_stride, as_stream(stream)));
}

int kv_write_v_only(const kv_bf16_t* value, kv_bf16_t* v_cache, const int64_t* slot_mapping,
                    uint32_t num_tokens, uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                    uint32_t value_stride, void* stream) {
  if (num_tokens == 0) return KV_OK;
  if (!value || !v_cache || !slot_mapping) return KV_ERR_INVALID_ARG;
  if (int r = check_rows(num_kv_heads, head_dim, block_size)) return r;
  const uint32_t row = num_kv_heads * head_dim;
  if (value_stride < row) return KV_ERR_INVALID_ARG;
  return from_cuda(launch_copy_rows(value, nullptr, v_cache, nullptr, slot_mapping, num_tokens, row,
                                    value_stride, 0, as_stream(stream)));
}

int kv_write_fp8k(const kv_bf16_t* key, const kv_bf16_t* value, kv_e4m3_t* k_cache_fp8,
                  kv_bf16_t* v_cache, const int64_t* slot_mapping, uint32_t num_tokens,
                  uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size, uint32_t key_stride,
                  uint32_t value_stride, float k_scale, void* stream) {
  if (num_tokens == 0) return KV_OK;
  if (!key || !value || !k_cache_fp8 || !v_cache || !slot_mapping) return KV_ERR_INVALID_ARG;
  if (int r = check_rows(num_kv_heads, head_dim, block_size)) return r;
  const uint32_t row = num_kv_heads * head_dim;
  if (key_stride < row || value_stride < row) return KV_ERR_INVALID_ARG;
  if (!(k_scale > 0.0f) || !isfinite(k_scale)) return KV_ERR_INVALID_ARG;
  return from_cuda(launch_write_fp8(key, value, k_cache_fp8, v_cache, false, slot_mapping, num_tokens, row,
                                    key_stride, value_stride, k_scale, 1.0f, as_stream(stream)));
}

int kv_write_fp8(const kv_bf16_t* key, const kv_bf16_t* value, kv_e4m3_t* k_cache_fp8, kv_e4m3_t* v_cache_fp8,
                 const int64_t* slot_mapping, uint32_t num_tokens, uint32_t num_kv_heads, uint32_t head_dim,
                 uint32_t block_size, float k_scale, float v_scale, uint32_t key_stride, uint32_t value_stride,
                 void* stream) {
  if (num_tokens == 0) return KV_OK;
  if (!key || !value || !k_cache_fp8 || !v_cache_fp8 || !slot_mapping) return KV_ERR_INVALID_ARG;
  if (int r = check_rows(num_kv_heads, head_dim, block_size)) return r;
  const uint32_t row = num_kv_heads * head_dim;
  if (key_stride < row || value_stride < row) return KV_ERR_INVALID_ARG;
  if (!(k_scale > 0.0f) || !isfinite(k_scale) || !(v_scale > 0.0f) || !isfinite(v_scale))
    return KV_ERR_INVALID_ARG;
  return from_cuda(launch_write_fp8(key, value, k_cache_fp8, v_cache_fp8, true, slot_mapping, num_tokens, row,
                                    key_stride, value_stride, k_scale, v_scale, as_stream(stream)));
}

static int fused_common(const kv_bf16_t* k_in, const kv_bf16_t* k_norm_weight, const int32_t* positions,
                        const int32_t* pos_h, const int32_t* pos_w, bool mrope, void* k_cache, bool fp8_out,
                        float inv_scale, const int64_t* slot_mapping, uint32_t num_tokens, uint32_t num_kv_heads,
                        uint32_t head_dim, uint32_t rotary_dim, uint32_t block_size, float rms_eps, float theta,
                        void* stream) {
  if (num_tokens == 0) return KV_OK;
  if (!k_in || !k_norm_weight || !positions || !k_cache || !slot_mapping) return KV_ERR_INVALID_ARG;
  if (mrope && (!pos_h || !pos_w)) return KV_ERR_INVALID_ARG;
  if (num_kv_heads == 0 || head_dim == 0 || block_size == 0) return KV_ERR_INVALID_ARG;
  if (rotary_dim == 0 || rotary_dim % 2 || rotary_dim > head_dim) return KV_ERR_INVALID_ARG;
  if (!(rms_eps >= 0.0f) || !isfinite(rms_eps) || !(theta > 0.0f) || !isfinite(theta))
    return KV_ERR_INVALID_ARG;
  if (fp8_out && (!(inv_scale > 0.0f) || !isfinite(inv_scale))) return KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KV_ERR_UNSUPPORTED;
  if (rotary_dim % 8) return KV_ERR_UNSUPPORTED;
  if (!aligned(k_in, 16) || !aligned(k_norm_weight, 16) || !aligned(k_cache, 16)) return KV_ERR_UNSUPPORTED;
  return from_cuda(launch_fused_k_norm_rope(k_in, k_norm_weight, positions, mrope ? pos_h : nullptr,
                                            mrope ? pos_w : nullptr, k_cache, fp8_out, inv_scale, slot_mapping,
                                            num_tokens, num_kv_heads, head_dim, rotary_dim, rms_eps, theta,
                                            as_stream(stream)));
}

int kv_write_fused_k_norm_rope_bf16(const kv_bf16_t* k_in, const kv_bf16_t* k_norm_weight,
                                    const int32_t* positions, kv_bf16_t* k_cache,
                                    const int64_t* slot_mapping, uint32_t num_tokens,
                                    uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                    uint32_t block_size, float rms_eps, float theta, void* stream) {
  return fused_common(k_in, k_norm_weight, positions, nullptr, nullptr, false, k_cache, false, 1.0f, slot_mapping,
                      num_tokens, num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta, stream);
}

int kv_write_fused_k_norm_rope_bf16_mrope(const kv_bf16_t* k_in, const kv_bf16_t* k_norm_weight,
                                          const int32_t* pos_t, const int32_t* pos_h, const int32_t* pos_w,
                                          kv_bf16_t* k_cache, const int64_t* slot_mapping, uint32_t num_tokens,
                                          uint32_t num_kv_heads, uint32_t head_dim, uint32_t rotary_dim,
                                          uint32_t block_size, float rms_eps, float theta, void* stream) {
  return fused_common(k_in, k_norm_weight, pos_t, pos_h, pos_w, true, k_cache, false, 1.0f, slot_mapping,
                      num_tokens, num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta, stream);
}

int kv_write_fused_k_norm_rope_fp8(const kv_bf16_t* k_in, const kv_bf16_t* k_norm_weight,
                                   const int32_t* positions, kv_e4m3_t* k_cache_fp8,
                                   const int64_t* slot_mapping, uint32_t num_tokens, uint32_t num_kv_heads,
                                   uint32_t head_dim, uint32_t rotary_dim, uint32_t block_size, float rms_eps,
                                   float theta, float inv_scale, void* stream) {
  return fused_common(k_in, k_norm_weight, positions, nullptr, nullptr, false, k_cache_fp8, true, inv_scale,
                      slot_mapping, num_tokens, num_kv_heads, head_dim, rotary_dim, block_size, rms_eps, theta,
                      stream);
}

static int decode_common(const kv_bf16_t* q, const void* k_cache, const void* v_cache, float* output,
                         const int32_t* block_tables, const int32_t* seq_lens, uint32_t max_blocks_per_seq,
                         uint32_t num_seqs, uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                         uint32_t block_size, float inv_sqrt_d, float k_scale, uint32_t q_stride,
                         uint32_t sliding_window, bool fp8, bool fp8_v, float v_scale, void* stream) {
  if (num_seqs == 0) return KV_OK;
  if (!q || !k_cache || !v_cache || !output || !block_tables || !seq_lens) return KV_ERR_INVALID_ARG;
  if (num_kv_heads == 0 || num_q_heads == 0 || num_q_heads % num_kv_heads) return KV_ERR_INVALID_ARG;
  if (head_dim == 0 || block_size == 0) return KV_ERR_INVALID_ARG;
  if (uint64_t(q_stride) < uint64_t(num_q_heads) * head_dim) return KV_ERR_INVALID_ARG;
  if (!isfinite(inv_sqrt_d)) return KV_ERR_INVALID_ARG;
  if (fp8 && (!(k_scale > 0.0f) || !isfinite(k_scale))) return KV_ERR_INVALID_ARG;
  if (fp8_v && (!(v_scale > 0.0f) || !isfinite(v_scale))) return KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KV_ERR_UNSUPPORTED;
  if (!is_pow2(block_size) || block_size < 16 || block_size > 256) return KV_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > 16) return KV_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || (q_stride * 2u) % 16)
    return KV_ERR_UNSUPPORTED;
  if (!aligned(output, 8)) return KV_ERR_UNSUPPORTED;
  if (uint64_t(max_blocks_per_seq) * block_size >= (1ull << 31)) return KV_ERR_UNSUPPORTED;
  const DeviceInfo& dev = device_info();
  if (dev.device < 0) return KV_ERR_CUDA;
  if (dev.cc_major < 10) return KV_ERR_UNSUPPORTED;

  DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.output = output;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.inv_sqrt_d = inv_sqrt_d;
  a.k_scale = k_scale;
  a.q_stride = q_stride;
  a.sliding_window = sliding_window;
  a.fp8 = fp8;
  a.fp8_v = fp8_v;
  a.v_scale = v_scale;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    a.workspace = g_ws_ptr[dev.device];
    a.workspace_bytes = g_ws_bytes[dev.device];
    a.workspace_fresh = g_ws_fresh[dev.device];
  }
  const int status = launch_decode(a, as_stream(stream));
  if (status == KV_OK && a.workspace_fresh) {
    // the work counters were zeroed on this call's stream; the kernels keep
    // them at zero from here on
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_ws_ptr[dev.device] == a.workspace) g_ws_fresh[dev.device] = false;
  }
  return status;
}

int paged_decode_attn_bf16(const kv_bf16_t* q, const kv_bf16_t* k_cache, const kv_bf16_t* v_cache,
                           float* output, const int32_t* block_tables, const int32_t* seq_lens,
                           uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                           uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size, float inv_sqrt_d,
                           uint32_t q_stride, uint32_t sliding_window, void* stream) {
  return decode_common(q, k_cache, v_cache, output, block_tables, seq_lens, max_blocks_per_seq, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, 1.0f, q_stride,
                       sliding_window, false, false, 1.0f, stream);
}

int paged_decode_attn_fp8k(const kv_bf16_t* q, const kv_e4m3_t* k_cache_fp8, const kv_bf16_t* v_cache,
                           float* output, const int32_t* block_tables, const int32_t* seq_lens,
                           uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                           uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size, float inv_sqrt_d,
                           float k_scale, uint32_t q_stride, uint32_t sliding_window, void* stream) {
  return decode_common(q, k_cache_fp8, v_cache, output, block_tables, seq_lens, max_blocks_per_seq, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, k_scale, q_stride,
                       sliding_window, true, false, 1.0f, stream);
}

int paged_decode_attn_fp8(const kv_bf16_t* q, const kv_e4m3_t* k_cache_fp8, const kv_e4m3_t* v_cache_fp8,
                          float* output, const int32_t* block_tables, const int32_t* seq_lens,
                          uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                          uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size, float inv_sqrt_d,
                          float k_scale, float v_scale, uint32_t q_stride, uint32_t sliding_window,
                          void* stream) {
  return decode_common(q, k_cache_fp8, v_cache_fp8, output, block_tables, seq_lens, max_blocks_per_seq,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, k_scale, q_stride,
                       sliding_window, true, true, v_scale, stream);
}

static int prefill_common(const kv_bf16_t* q, const void* k_cache, const void* v_cache, float* output,
                          const int32_t* block_tables, const int32_t* seq_lens, const int32_t* query_start_loc,
                          uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_tokens,
                          uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                          float inv_sqrt_d, float k_scale, float v_scale, uint32_t q_stride,
                          uint32_t sliding_window, bool fp8, bool fp8_v, void* stream) {
  if (num_seqs == 0 || num_q_tokens == 0) return KV_OK;
  if (!q || !k_cache || !v_cache || !output || !block_tables || !seq_lens || !query_start_loc)
    return KV_ERR_INVALID_ARG;
  if (num_kv_heads == 0 || num_q_heads == 0 || num_q_heads % num_kv_heads) return KV_ERR_INVALID_ARG;
  if (head_dim == 0 || block_size == 0) return KV_ERR_INVALID_ARG;
  if (uint64_t(q_stride) < uint64_t(num_q_heads) * head_dim) return KV_ERR_INVALID_ARG;
  if (!isfinite(inv_sqrt_d)) return KV_ERR_INVALID_ARG;
  if (fp8 && (!(k_scale > 0.0f) || !isfinite(k_scale))) return KV_ERR_INVALID_ARG;
  if (fp8_v && (!(v_scale > 0.0f) || !isfinite(v_scale))) return KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return KV_ERR_UNSUPPORTED;
  if (!is_pow2(block_size) || block_size < 16 || block_size > 256) return KV_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || (q_stride * 2u) % 16)
    return KV_ERR_UNSUPPORTED;
  if (!aligned(output, 16)) return KV_ERR_UNSUPPORTED;
  if (uint64_t(max_blocks_per_seq) * block_size >= (1ull << 31)) return KV_ERR_UNSUPPORTED;
  if (uint64_t(num_q_tokens) * num_q_heads >= (1ull << 31)) return KV_ERR_UNSUPPORTED;
  const DeviceInfo& dev = device_info();
  if (dev.device < 0) return KV_ERR_CUDA;
  if (dev.cc_major < 10) return KV_ERR_UNSUPPORTED;
  PrefillArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.output = output;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.query_start_loc = query_start_loc;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_q_tokens = num_q_tokens;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.inv_sqrt_d = inv_sqrt_d;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.q_stride = q_stride;
  a.sliding_window = sliding_window;
  a.fp8 = fp8;
  a.fp8_v = fp8_v;
  return launch_prefill(a, as_stream(stream));
}

int paged_prefill_attn_bf16(const kv_bf16_t* q, const kv_bf16_t* k_cache, const kv_bf16_t* v_cache, float* output,
                            const int32_t* block_tables, const int32_t* seq_lens, const int32_t* query_start_loc,
                            uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_tokens,
                            uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size,
                            float inv_sqrt_d, uint32_t q_stride, uint32_t sliding_window, void* stream) {
  return prefill_common(q, k_cache, v_cache, output, block_tables, seq_lens, query_start_loc, max_blocks_per_seq,
                        num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, block_size, inv_sqrt_d, 1.0f,
                        1.0f, q_stride, sliding_window, false, false, stream);
}

int paged_prefill_attn_fp8k(const kv_bf16_t* q, const kv_e4m3_t* k_cache_fp8, const kv_bf16_t* v_cache,
                            float* output, const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* query_start_loc, uint32_t max_blocks_per_seq, uint32_t num_seqs,
                            uint32_t num_q_tokens, uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                            uint32_t block_size, float inv_sqrt_d, float k_scale, uint32_t q_stride,
                            uint32_t sliding_window, void* stream) {
  return prefill_common(q, k_cache_fp8, v_cache, output, block_tables, seq_lens, query_start_loc,
                        max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                        inv_sqrt_d, k_scale, 1.0f, q_stride, sliding_window, true, false, stream);
}

int paged_prefill_attn_fp8(const kv_bf16_t* q, const kv_e4m3_t* k_cache_fp8, const kv_e4m3_t* v_cache_fp8,
                           float* output, const int32_t* block_tables, const int32_t* seq_lens,
                           const int32_t* query_start_loc, uint32_t max_blocks_per_seq, uint32_t num_seqs,
                           uint32_t num_q_tokens, uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim,
                           uint32_t block_size, float inv_sqrt_d, float k_scale, float v_scale, uint32_t q_stride,
                           uint32_t sliding_window, void* stream) {
  return prefill_common(q, k_cache_fp8, v_cache_fp8, output, block_tables, seq_lens, query_start_loc,
                        max_blocks_per_seq, num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                        inv_sqrt_d, k_scale, v_scale, q_stride, sliding_window, true, true, stream);
}

size_t kv_decode_workspace_bytes(uint32_t max_blocks_per_seq, uint32_t num_seqs, uint32_t num_q_heads,
                                 uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size) {
  return decode_workspace_bytes(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size);
}

int kv_set_decode_workspace(void* device_ptr, size_t bytes) {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return KV_ERR_CUDA;
  if (device_ptr && !aligned(device_ptr, 256)) return KV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  g_ws_ptr[d] = bytes ? device_ptr : nullptr;
  g_ws_bytes[d] = device_ptr ? bytes : 0;
  g_ws_fresh[d] = g_ws_ptr[d] != nullptr;
  return KV_OK;
}

int kv_get_device_error(uint32_t* bits) {
  if (!bits) return KV_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return KV_ERR_CUDA;
  uint32_t decode_bits = 0, prefill_bits = 0, fused_bits = 0;
  if (read_and_clear_decode_error(&decode_bits) != cudaSuccess ||
      read_and_clear_prefill_error(&prefill_bits) != cudaSuccess ||
      read_and_clear_fused_error(&fused_bits) != cudaSuccess)
    return KV_ERR_CUDA;
  *bits = decode_bits | prefill_bits | fused_bits;
#ifdef PAGEDKV_DEBUG_BOUNDS
  uint32_t d[4] = {0, 0, 0, 0};
  if (debug_read_and_clear_kv_write(&d[0]) != cudaSuccess || debug_read_and_clear_fused_k(&d[1]) != cudaSuccess ||
      debug_read_and_clear_decode(&d[2]) != cudaSuccess || debug_read_and_clear_prefill(&d[3]) != cudaSuccess)
    return KV_ERR_CUDA;
  *bits |= d[0] | d[1] | d[2] | d[3];
#endif
  return *bits ? KV_ERR_DEVICE : KV_OK;
}

int kv_debug_set_pool(uint32_t num_blocks, uint32_t block_size) {
#ifdef PAGEDKV_DEBUG_BOUNDS
  if (num_blocks && !block_size) return KV_ERR_INVALID_ARG;
  if (device_info().device < 0) return KV_ERR_CUDA;
  if (debug_set_pool_kv_write(num_blocks, block_size) != cudaSuccess ||
      debug_set_pool_fused_k(num_blocks, block_size) != cudaSuccess ||
      debug_set_pool_decode(num_blocks, block_size) != cudaSuccess ||
      debug_set_pool_prefill(num_blocks, block_size) != cudaSuccess)
    return KV_ERR_CUDA;
  return KV_OK;
#else
  (void)num_blocks;
  (void)block_size;
  return KV_ERR_UNSUPPORTED;  // only the bounds-checking build checks indices
#endif
}

int kv_debug_set_wait_limit(uint64_t nanoseconds) {
#ifdef PAGEDKV_DEBUG_BOUNDS
  if (device_info().device < 0) return KV_ERR_CUDA;
  const uint64_t ns = nanoseconds ? nanoseconds : kWaitLimitNs;
  return from_cuda(debug_set_wait_limit_decode(ns));
#else
  (void)nanoseconds;
  return KV_ERR_UNSUPPORTED;  // the product build's limit is fixed
#endif
}

int kv_device_info(int* num_sms, int* decode_ctas) {
  const DeviceInfo& dev = device_info();
  if (dev.device < 0) return KV_ERR_CUDA;
  if (num_sms) *num_sms = dev.num_sms;
  if (decode_ctas) *decode_ctas = dev.num_sms;
  return KV_OK;
}

}  // extern "C"
