// Combination of the partitions of one row: with lse_p the base-2
// log-sum-exp of partition p and o_p its normalised partial output,
//   L = log2(sum_p 2^lse_p),  out = sum_p 2^(lse_p - L) o_p.
// This is the renormalised form of the per-block combination sketched in
// devpress.csdn.net vLLM overview, "3、PagedAttention (3)", using the running
// max / sum of exponentials of "9、FlashAttention (4)".
//
// One CTA per (row, head), one thread per output element; the weights of all
// partitions are computed once into shared memory.  In cascade decode the
// partitions of a row are the chunks of its group's shared prefix followed by
// those of its own keys.

#include "common.cuh"
#include "launch.h"
#include "rows.cuh"

namespace pkv {
namespace {

template <class QT, int D>
__global__ void __launch_bounds__(D) lse_merge_kernel(const AttnParams p) {
  using OutT = typename QT::T;
  extern __shared__ float s_w[];  // [max_parts]
  __shared__ float s_red[D / 32];
  const int row = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int seq;
  const int keys = row_keys(p, row, &seq);
  // cascade decode: the shared prefix's partials, then the sequence's own
  const int pre = cascade_prefix(p, seq, keys, false);
  int np = cascade_slots(p, pre) + (keys - pre + p.partition - 1) / p.partition;
  if (np > p.max_parts) {  // a prefix longer than the launch was sized for
    if (tid == 0) flag_error(p.errors, PKV_DEVERR_CONTEXT);
    np = p.max_parts;
  }
  const size_t head = (size_t)row * p.num_heads + h;
  OutT* out = static_cast<OutT*>(p.out) + head * D;
  if (np == 0) {
    store_out(out + tid, 0.0f);
    return;
  }
  // a single partition was written to out directly, except in cascade decode
  if (np == 1 && p.prefix_lens == nullptr) return;
  const float* lse = p.lse + head * p.max_parts;

  float m = -INFINITY;
  for (int i = tid; i < np; i += D) m = fmaxf(m, lse[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  m = s_red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) m = fmaxf(m, s_red[w]);
  __syncthreads();

  float sum = 0.0f;
  for (int i = tid; i < np; i += D) {
    const float e = exp2f(lse[i] - m);
    s_w[i] = e;
    sum += e;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  if (lane == 0) s_red[warp] = sum;
  __syncthreads();
  sum = 0.0f;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) sum += s_red[w];

  const float* op = p.o_part + head * p.max_parts * D + tid;
  float acc0 = 0.0f, acc1 = 0.0f, acc2 = 0.0f, acc3 = 0.0f;
  int i = 0;
  for (; i + 4 <= np; i += 4) {
    acc0 = fmaf(s_w[i], op[(size_t)i * D], acc0);
    acc1 = fmaf(s_w[i + 1], op[(size_t)(i + 1) * D], acc1);
    acc2 = fmaf(s_w[i + 2], op[(size_t)(i + 2) * D], acc2);
    acc3 = fmaf(s_w[i + 3], op[(size_t)(i + 3) * D], acc3);
  }
  for (; i < np; ++i) acc0 = fmaf(s_w[i], op[(size_t)i * D], acc0);
  store_out(out + tid, ((acc0 + acc1) + (acc2 + acc3)) / sum);
}

template <class QT>
int launch_merge_typed(const AttnParams& p, int head_dim, cudaStream_t stream) {
  dim3 grid(p.num_rows, p.num_heads);
  const size_t smem = (size_t)p.max_parts * sizeof(float);
  if (head_dim == 64) {
    auto k = lse_merge_kernel<QT, 64>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return PKV_ERR_CUDA;
    k<<<grid, 64, smem, stream>>>(p);
  } else {
    auto k = lse_merge_kernel<QT, 128>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return PKV_ERR_CUDA;
    k<<<grid, 128, smem, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int launch_lse_merge(const AttnParams& p, int q_dtype, int head_dim, cudaStream_t stream) {
  return q_dtype == PKV_BF16 ? launch_merge_typed<BF16>(p, head_dim, stream)
                             : launch_merge_typed<F16>(p, head_dim, stream);
}

}  // namespace pkv
