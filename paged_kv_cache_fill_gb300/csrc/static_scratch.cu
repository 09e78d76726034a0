// paged_decode_attn_fp8k_static_scratch: the FP8-K paged decode for callers
// that cannot hand the library a device allocation.
//
// The regular decode takes its split-KV scratch from a buffer the caller
// allocates and registers. Some callers cannot do that: an application whose
// device memory is owned end to end by another allocator (a framework's
// memory pool, a serving engine that reserves all of HBM for its KV cache up
// front) has no way to set a raw buffer aside for a third-party library, and
// a cudaMalloc of its own would fail or break that allocator's accounting.
// This entry point needs no allocation from anyone: its scratch is a
// fixed-size array in the library's own device memory. (It is an ordinary
// CUDA call like every other one here: it must not be made from a host
// function enqueued with cudaLaunchHostFunc, where the CUDA API may not be
// called.)
//
// The array is g_static_scratch below (kStaticScratchBytes = 64 MiB). Every
// GPU that loads the library reserves it until the process exits. Host code
// must not use the array's name as a device address, so the first call on
// each device (with that device current) looks up the array's device address
// with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture. A device reset (cudaDeviceReset) ends the context that
// address belongs to: do not call this entry point on a device after
// resetting it in the same process.
#include <math.h>

#include <mutex>

#include "../../include/pagedkv.h"
#include "internal.h"

namespace pagedkv {
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr int kMaxStaticDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mutex;
void* g_static_ptr[kMaxStaticDevices];  // device address of g_static_scratch, per device

// Device address of the static scratch array on the current device, looked
// up once per device; nullptr on failure.
void* static_scratch_address(int device) {
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_ptr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
    g_static_ptr[device] = p;
  }
  return g_static_ptr[device];
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" int paged_decode_attn_fp8k_static_scratch(
    const kv_bf16_t* q, const kv_e4m3_t* k_cache_fp8, const kv_bf16_t* v_cache, float* output,
    const int32_t* block_tables, const int32_t* seq_lens, uint32_t max_blocks_per_seq, uint32_t num_seqs,
    uint32_t num_q_heads, uint32_t num_kv_heads, uint32_t head_dim, uint32_t block_size, float inv_sqrt_d,
    float k_scale, uint32_t q_stride, uint32_t sliding_window, void* stream) {
  // the same argument rules as paged_decode_attn_fp8k
  if (num_seqs == 0) return KV_OK;
  if (!q || !k_cache_fp8 || !v_cache || !output || !block_tables || !seq_lens) return KV_ERR_INVALID_ARG;
  if (num_kv_heads == 0 || num_q_heads == 0 || num_q_heads % num_kv_heads) return KV_ERR_INVALID_ARG;
  if (head_dim == 0 || block_size == 0) return KV_ERR_INVALID_ARG;
  if (uint64_t(q_stride) < uint64_t(num_q_heads) * head_dim) return KV_ERR_INVALID_ARG;
  if (!isfinite(inv_sqrt_d) || !(k_scale > 0.0f) || !isfinite(k_scale)) return KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KV_ERR_UNSUPPORTED;
  if (block_size < 16 || block_size > 256 || (block_size & (block_size - 1))) return KV_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > 16) return KV_ERR_UNSUPPORTED;
  const auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (misaligned(q, 16) || misaligned(k_cache_fp8, 16) || misaligned(v_cache, 16) || (q_stride * 2u) % 16 ||
      misaligned(output, 8))
    return KV_ERR_UNSUPPORTED;
  if (uint64_t(max_blocks_per_seq) * block_size >= (1ull << 31)) return KV_ERR_UNSUPPORTED;
  // The whole split-KV scratch this shape can need must fit the fixed array.
  if (decode_workspace_bytes(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size) >
      kStaticScratchBytes)
    return KV_ERR_UNSUPPORTED;

  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxStaticDevices) return KV_ERR_CUDA;
  const DeviceInfo& dev = device_info();
  if (dev.device < 0) return KV_ERR_CUDA;
  if (dev.cc_major < 10) return KV_ERR_UNSUPPORTED;
  void* scratch = static_scratch_address(device);
  if (!scratch) return KV_ERR_CUDA;

  DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache_fp8;
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
  a.fp8 = true;
  a.workspace = scratch;
  a.workspace_bytes = kStaticScratchBytes;
  // The array keeps whatever the previous call left in it: have the decode
  // clear its work counters on this call's stream before it starts.
  a.workspace_fresh = true;
  return launch_decode(a, static_cast<cudaStream_t>(stream));
}
