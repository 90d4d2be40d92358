// Cache write: scatter new K/V rows into the paged block pool through a slot
// mapping (devpress.csdn.net vLLM overview, "8、推理流程": K and V of the layer
// are stored into the paged cache; openeuler.csdn.net PagedAttention notes,
// "Block Table 数据结构": slot = physical_block * block_size + offset).
//
// One thread moves one 16-byte chunk of one source row; consecutive threads
// take consecutive chunks of a row, so both the loads from k/v and the stores
// into the (block, head) tile are 128-bit and coalesced.  The FP8 variant
// divides by the per-tensor scale (IEEE division) and rounds to E4M3 with
// saturation, eight elements per thread.

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

template <typename SRC>
__device__ __forceinline__ uint2 quantize8(const uint4& w, float scale) {
  float f[8];
  to_float(w, f, SRC());
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    __nv_fp8_storage_t b = __nv_cvt_float_to_fp8(__fdiv_rn(f[i], scale), __NV_SATFINITE, __NV_E4M3);
    out[i / 4] |= static_cast<uint32_t>(b) << (8 * (i % 4));
  }
  return make_uint2(out[0], out[1]);
}

template <typename SRC, bool FP8>
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                         uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                         const int64_t* __restrict__ slots, int num_tokens, int num_kv_heads,
                         int head_dim, int64_t num_slots, float k_scale, float v_scale,
                         uint32_t* errors) {
  const int chunks = head_dim / 8;  // 16-byte chunks per source row
  const int64_t per_token = 2LL * num_kv_heads * chunks;
  const int64_t total = per_token * num_tokens;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / per_token);
    int rem = (int)(i - (int64_t)t * per_token);
    const int kv = rem / (num_kv_heads * chunks);
    rem -= kv * num_kv_heads * chunks;
    const int h = rem / chunks;
    const int c = rem - h * chunks;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (kv == 0 && h == 0 && c == 0) flag_error(errors, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / kBlockSize;
    const int off = (int)(slot - blk * kBlockSize);
    const int64_t src_idx = ((int64_t)t * num_kv_heads + h) * chunks + c;
    const uint4 w = kv ? __ldg(v + src_idx) : __ldg(k + src_idx);
    const int64_t row = (blk * num_kv_heads + h) * kBlockSize + off;
    uint8_t* cache = kv ? v_cache : k_cache;
    if constexpr (FP8) {
      const uint2 q = quantize8<SRC>(w, kv ? v_scale : k_scale);
      reinterpret_cast<uint2*>(cache + row * head_dim)[c] = q;
    } else {
      reinterpret_cast<uint4*>(cache + row * head_dim * 2)[c] = w;
    }
  }
}

}  // namespace

int launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int num_blocks, int src_dtype, int cache_dtype,
                             float k_scale, float v_scale, uint32_t* errors,
                             cudaStream_t stream) {
  const int64_t total = 2LL * num_tokens * num_kv_heads * (head_dim / 8);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152LL * 64) blocks = 152LL * 64;
  const int64_t num_slots = (int64_t)num_blocks * kBlockSize;
  auto kk = static_cast<const uint4*>(k);
  auto vv = static_cast<const uint4*>(v);
  auto kc = static_cast<uint8_t*>(k_cache);
  auto vc = static_cast<uint8_t*>(v_cache);
  const bool fp8 = cache_dtype == PKV_FP8_E4M3;
  if (src_dtype == PKV_BF16) {
    if (fp8)
      reshape_and_cache_kernel<BF16, true><<<(unsigned)blocks, threads, 0, stream>>>(
          kk, vv, kc, vc, slot_mapping, num_tokens, num_kv_heads, head_dim, num_slots, k_scale,
          v_scale, errors);
    else
      reshape_and_cache_kernel<BF16, false><<<(unsigned)blocks, threads, 0, stream>>>(
          kk, vv, kc, vc, slot_mapping, num_tokens, num_kv_heads, head_dim, num_slots, k_scale,
          v_scale, errors);
  } else {
    if (fp8)
      reshape_and_cache_kernel<F16, true><<<(unsigned)blocks, threads, 0, stream>>>(
          kk, vv, kc, vc, slot_mapping, num_tokens, num_kv_heads, head_dim, num_slots, k_scale,
          v_scale, errors);
    else
      reshape_and_cache_kernel<F16, false><<<(unsigned)blocks, threads, 0, stream>>>(
          kk, vv, kc, vc, slot_mapping, num_tokens, num_kv_heads, head_dim, num_slots, k_scale,
          v_scale, errors);
  }
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
