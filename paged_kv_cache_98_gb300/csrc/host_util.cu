// Host helpers shared by the tensor-core kernels: TMA tensor-map encoding
// (through the driver entry point, so nothing links against libcuda) and the
// SM count.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

bool tmap_available() { return encode_fn() != nullptr; }

// Rows of 128 16-bit elements; boxes of 64 columns x box_rows rows; 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, bool bf16, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128 * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of 128 one-byte E4M3 values; boxes of 128 columns x box_rows rows; 128-byte swizzle.
bool make_map_e4m3(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 q viewed as [tokens][heads][128 B]: boxes of 128 columns x box_heads
// heads x box_tokens tokens (token-major rows of 128 bytes), 128-byte swizzle.
bool make_map_q3d_e4m3(CUtensorMap* m, const void* base, uint64_t tokens, uint32_t heads,
                       uint32_t box_heads, uint32_t box_tokens) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {128, (cuuint64_t)heads * 128};
  cuuint32_t box[3] = {128, box_heads, box_tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q viewed as [tokens][heads][128]: boxes of 64 columns x box_heads heads x
// box_tokens tokens, 128-byte swizzle (the box lands as box_heads*box_tokens
// rows of 128 bytes, token-major).
bool make_map_q3d(CUtensorMap* m, const void* base, uint64_t tokens, uint32_t heads, bool bf16,
                  uint32_t box_heads, uint32_t box_tokens) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  cuuint32_t box[3] = {64, box_heads, box_tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace pkv
