// Whole-block copies, the device half of copy-on-write (openeuler.csdn.net
// PagedAttention notes, "机制 2：写时复制": before a request writes into a
// block it shares, it gets a private copy of that block).  With the cache
// layout [num_blocks][num_kv_heads][block_size][head_dim] a block of one cache
// is one contiguous run of num_kv_heads * block_size * head_dim elements, so
// each (pair, cache) copy is a straight 16-byte-vector memcpy.
//
// Grid: x = pairs (grid-stride), y = 2 (K cache, V cache); each CTA copies one
// block of one cache with 256 threads, loads and stores fully coalesced.

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int32_t* __restrict__ pairs, int num_pairs, int num_blocks,
                   int64_t block_vecs, uint32_t* errors) {
  uint4* cache = blockIdx.y ? v_cache : k_cache;
  for (int i = blockIdx.x; i < num_pairs; i += gridDim.x) {
    const int src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(errors, PKV_DEVERR_BLOCK_ID);
      continue;
    }
    const uint4* s = cache + (int64_t)src * block_vecs;
    uint4* d = cache + (int64_t)dst * block_vecs;
    for (int64_t j = threadIdx.x; j < block_vecs; j += blockDim.x) d[j] = s[j];
  }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs,
                               int num_pairs, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, pkv_dtype cache_dtype, uint32_t* device_errors,
                               void* stream) {
  if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) & 15u) || (reinterpret_cast<uintptr_t>(v_cache) & 15u))
    return PKV_ERR_INVALID_ARG;
  if (block_size != pkv::kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (cache_dtype != PKV_F16 && cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3)
    return PKV_ERR_UNSUPPORTED;
  const int64_t elem = cache_dtype == PKV_FP8_E4M3 ? 1 : 2;
  const int64_t block_bytes = (int64_t)num_kv_heads * block_size * head_dim * elem;
  if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  const int grid = num_pairs < 4096 ? num_pairs : 4096;
  pkv::copy_blocks_kernel<<<dim3(grid, 2), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_pairs, num_pairs,
      num_blocks, block_bytes / 16, device_errors);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
