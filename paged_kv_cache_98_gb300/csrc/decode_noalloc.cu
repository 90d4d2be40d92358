// Decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc, or hand this library a workspace: a
// host framework that owns every byte of device memory through its own pool
// and forbids plugins from allocating, or a latency-critical serving loop that
// must not pay the implicit device synchronisation of cudaMalloc/cudaFree.
// For them pkv_paged_attention_decode_noalloc keeps the split-K scratch (the
// per-partition partial outputs and log-sum-exp values) in a fixed
// file-scope device array instead of a caller workspace.
//
// The array lives in this translation unit's own module, so only processes
// that use this entry point load it; every GPU that does holds it until the
// process exits.  Its address is looked up once per device, with that device
// current, on the first call made on that device.

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = PKV_DECODE_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// Split-K scratch shared by every call on a device.  Host code sees only a
// stand-in for this name; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_decode_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // do not leave the lookup failure pending for later calls
      return PKV_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_heads,
    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
    int max_context_len, float scale, pkv_dtype q_dtype, pkv_dtype kv_dtype, float k_scale,
    float v_scale, int partition_size, uint32_t* device_errors, void* stream) {
  if (partition_size != 0 &&
      (partition_size % 16 != 0 || partition_size < 16 || partition_size > 512))
    return PKV_ERR_INVALID_ARG;
  const size_t need = pkv_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len,
                                                partition_size);
  if (need > kScratchBytes) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&scratch);
    if (rc != PKV_OK) return rc;
  }
  return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                                    num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                    max_blocks_per_seq, num_blocks, max_context_len, scale,
                                    q_dtype, kv_dtype, k_scale, v_scale, partition_size, scratch,
                                    need > 0 ? kScratchBytes : 0, device_errors, stream);
}
