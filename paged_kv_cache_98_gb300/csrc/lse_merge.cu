// Combination of the partitions of one row: with lse_p the base-2
// log-sum-exp of partition p and o_p its normalised partial output,
//   L = log2(sum_p 2^lse_p),  out = sum_p 2^(lse_p - L) o_p.
// This is the renormalised form of the per-block combination sketched in
// devpress.csdn.net vLLM overview, "3、PagedAttention (3)", using the running
// max / sum of exponentials of "9、FlashAttention (4)".  In cascade decode the
// partitions of a row are the chunks of its group's shared prefix followed by
// those of its own keys.
//
// Two shapes of the same computation, chosen by the launch's partition count:
// - few partitions (up to kWarpParts = 64): one warp per (row, head), eight
//   per CTA.  Lane j computes the weights of partitions j and j + 32 once
//   (shuffle reductions for the max and the sum); each lane owns four output
//   dimensions (one float4 of each partial) and walks the partitions with
//   four loads in flight, taking each weight from its lane by shuffle;
// - many partitions: one CTA of eight warps per (row, head).  The weights go
//   to shared memory once; warp w takes partitions w, w + 8, ... for all
//   dimensions (float4 per lane) and the eight partial sums meet in shared
//   memory.
// Either way every partial is read once, with 16-byte loads.

#include "common.cuh"
#include "launch.h"
#include "rows.cuh"

namespace pkv {
namespace {

constexpr int kWarpParts = 64;  // at most this many partitions: a warp per (row, head)
constexpr int kMergeWarps = 8;

// Partitions holding this (row, head)'s partials; 0 for an empty context.
// Returns -1 when the partition was written to out directly (no merge).
__device__ __forceinline__ int row_parts(const AttnParams& p, int row) {
  int seq;
  const int keys = row_keys(p, row, &seq);
  const int pre = cascade_prefix(p, seq, keys, false);
  int np = cascade_slots(p, pre) + (keys - pre + p.partition - 1) / p.partition;
  if (np > p.max_parts) {  // a prefix longer than the launch was sized for
    if ((threadIdx.x & 31) == 0) flag_error(p.errors, PKV_DEVERR_CONTEXT);
    np = p.max_parts;
  }
  // a single partition was written to out directly, except in cascade decode
  if (np == 1 && p.prefix_lens == nullptr) return -1;
  return np;
}

template <class OutT>
__device__ __forceinline__ void store4(OutT* dst, float4 v) {
  store_out(dst + 0, v.x);
  store_out(dst + 1, v.y);
  store_out(dst + 2, v.z);
  store_out(dst + 3, v.w);
}

__device__ __forceinline__ float4 fma4(float w, const float4& a, float4 c) {
  c.x = fmaf(w, a.x, c.x);
  c.y = fmaf(w, a.y, c.y);
  c.z = fmaf(w, a.z, c.z);
  c.w = fmaf(w, a.w, c.w);
  return c;
}

// One warp per (row, head); D / 4 lanes own four dimensions each.
template <class QT, int D>
__global__ void __launch_bounds__(32 * kMergeWarps) lse_merge_warp_kernel(const AttnParams p) {
  using OutT = typename QT::T;
  const int lane = threadIdx.x & 31;
  const long long pair = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (pair >= (long long)p.num_rows * p.num_heads) return;
  const int row = (int)(pair / p.num_heads), h = (int)(pair % p.num_heads);
  const int np = row_parts(p, row);
  if (np < 0) return;
  const size_t head = (size_t)row * p.num_heads + h;
  OutT* out = static_cast<OutT*>(p.out) + head * D;
  constexpr int kLanes = D / 4;  // lanes holding dimensions
  if (np == 0) {
    if (lane < kLanes) store4(out + 4 * lane, make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const float4* op = reinterpret_cast<const float4*>(p.o_part + head * p.max_parts * D) +
                     (lane < kLanes ? lane : 0);
  constexpr int kStride = D / 4;  // float4s per partial
  // the first partials are requested before the weights are known
  constexpr int kPre = 8;
  float4 pf[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j)
    pf[j] = j < np ? __ldg(op + (size_t)j * kStride) : make_float4(0.f, 0.f, 0.f, 0.f);
  // lane j holds the weights of partitions j and j + 32 (np <= kWarpParts = 64)
  const float* lse = p.lse + head * p.max_parts;
  const float l0 = lane < np ? __ldg(lse + lane) : -INFINITY;
  const float l1 = lane + 32 < np ? __ldg(lse + lane + 32) : -INFINITY;
  float m = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  const float e0 = exp2f(l0 - m), e1 = exp2f(l1 - m);
  float sum = e0 + e1;
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
  // the whole warp walks the partitions (the weights come by shuffle)
  auto wt = [&](int i) { return __shfl_sync(kFull, i < 32 ? e0 : e1, i & 31); };
#pragma unroll
  for (int j = 0; j < kPre; j += 2) {  // weights past np are 0 (their lse is -inf)
    a0 = fma4(wt(j), pf[j], a0);
    a1 = fma4(wt(j + 1), pf[j + 1], a1);
  }
  int i = kPre;
  for (; i + 4 <= np; i += 4) {
    const float4 v0 = __ldg(op + (size_t)i * kStride), v1 = __ldg(op + (size_t)(i + 1) * kStride);
    const float4 v2 = __ldg(op + (size_t)(i + 2) * kStride), v3 = __ldg(op + (size_t)(i + 3) * kStride);
    a0 = fma4(wt(i), v0, a0);
    a1 = fma4(wt(i + 1), v1, a1);
    a2 = fma4(wt(i + 2), v2, a2);
    a3 = fma4(wt(i + 3), v3, a3);
  }
  for (; i < np; ++i) a0 = fma4(wt(i), __ldg(op + (size_t)i * kStride), a0);
  if (lane >= kLanes) return;
  const float inv = 1.0f / sum;
  store4(out + 4 * lane, make_float4(((a0.x + a1.x) + (a2.x + a3.x)) * inv,
                                     ((a0.y + a1.y) + (a2.y + a3.y)) * inv,
                                     ((a0.z + a1.z) + (a2.z + a3.z)) * inv,
                                     ((a0.w + a1.w) + (a2.w + a3.w)) * inv));
}

// One CTA of eight warps per (row, head), for many partitions.
template <class QT, int D>
__global__ void __launch_bounds__(32 * kMergeWarps) lse_merge_cta_kernel(const AttnParams p) {
  using OutT = typename QT::T;
  extern __shared__ float s_w[];  // [max_parts] weights, then [kMergeWarps][D] partial sums
  __shared__ float s_red[kMergeWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x, h = blockIdx.y;
  const int np = row_parts(p, row);
  if (np < 0) return;
  const size_t head = (size_t)row * p.num_heads + h;
  OutT* out = static_cast<OutT*>(p.out) + head * D;
  constexpr int kLanes = D / 4;
  if (np == 0) {
    if (tid < kLanes) store4(out + 4 * tid, make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const float* lse = p.lse + head * p.max_parts;
  float m = -INFINITY;
  for (int i = tid; i < np; i += 32 * kMergeWarps) m = fmaxf(m, __ldg(lse + i));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  m = s_red[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) m = fmaxf(m, s_red[w]);
  __syncthreads();
  float sum = 0.0f;
  for (int i = tid; i < np; i += 32 * kMergeWarps) {
    const float e = exp2f(__ldg(lse + i) - m);
    s_w[i] = e;
    sum += e;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  if (lane == 0) s_red[warp] = sum;
  __syncthreads();
  sum = 0.0f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) sum += s_red[w];
  float* s_acc = s_w + ((p.max_parts + 3) & ~3);
  if (lane < kLanes) {
    const float4* op =
        reinterpret_cast<const float4*>(p.o_part + head * p.max_parts * D) + lane;
    constexpr int kStride = D / 4;
    constexpr int W = kMergeWarps;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
    int i = warp;
    for (; i + 3 * W < np; i += 4 * W) {  // four loads in flight
      const float4 v0 = __ldg(op + (size_t)i * kStride);
      const float4 v1 = __ldg(op + (size_t)(i + W) * kStride);
      const float4 v2 = __ldg(op + (size_t)(i + 2 * W) * kStride);
      const float4 v3 = __ldg(op + (size_t)(i + 3 * W) * kStride);
      a0 = fma4(s_w[i], v0, a0);
      a1 = fma4(s_w[i + W], v1, a1);
      a2 = fma4(s_w[i + 2 * W], v2, a2);
      a3 = fma4(s_w[i + 3 * W], v3, a3);
    }
    for (; i < np; i += W) a0 = fma4(s_w[i], __ldg(op + (size_t)i * kStride), a0);
    reinterpret_cast<float4*>(s_acc + warp * D)[lane] =
        make_float4((a0.x + a1.x) + (a2.x + a3.x), (a0.y + a1.y) + (a2.y + a3.y),
                    (a0.z + a1.z) + (a2.z + a3.z), (a0.w + a1.w) + (a2.w + a3.w));
  }
  __syncthreads();
  if (tid < D) {
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) acc += s_acc[w * D + tid];
    store_out(out + tid, acc / sum);
  }
}

template <class QT, int D>
int launch_merge_shape(const AttnParams& p, cudaStream_t stream) {
  if (p.max_parts <= kWarpParts) {
    const long long pairs = (long long)p.num_rows * p.num_heads;
    const long long ctas = (pairs + kMergeWarps - 1) / kMergeWarps;
    if (ctas > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    lse_merge_warp_kernel<QT, D><<<(unsigned)ctas, 32 * kMergeWarps, 0, stream>>>(p);
  } else {
    auto k = lse_merge_cta_kernel<QT, D>;
    const size_t smem = ((size_t)(p.max_parts + 3) / 4 * 4 + kMergeWarps * D) * sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
      return PKV_ERR_CUDA;
    k<<<dim3(p.num_rows, p.num_heads), 32 * kMergeWarps, smem, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <class QT>
int launch_merge_typed(const AttnParams& p, int head_dim, cudaStream_t stream) {
  return head_dim == 64 ? launch_merge_shape<QT, 64>(p, stream)
                        : launch_merge_shape<QT, 128>(p, stream);
}

}  // namespace

int launch_lse_merge(const AttnParams& p, int q_dtype, int head_dim, cudaStream_t stream) {
  return q_dtype == PKV_BF16 ? launch_merge_typed<BF16>(p, head_dim, stream)
                             : launch_merge_typed<F16>(p, head_dim, stream);
}

}  // namespace pkv
