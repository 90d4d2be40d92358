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
// - many partitions: one CTA of sixteen warps per (row, head).  The weights
//   go to shared memory once; warp w takes partitions w, w + 16, ... for all
//   dimensions (float4 per lane), its first eight partials requested before
//   the weights and eight in flight after, and the sixteen partial sums meet
//   in shared memory.
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

// The merge is launched as a programmatic dependent of the attention launch
// before it (its launch overlaps that grid's end); it reads the partials only
// once that grid has completed and its writes are visible.  Without the
// launch attribute this returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  grid_dependency_wait();
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

// One CTA of sixteen warps per (row, head), for many partitions.
constexpr int kCtaWarps = 16;

template <class QT, int D>
__global__ void __launch_bounds__(32 * kCtaWarps) lse_merge_cta_kernel(const AttnParams p) {
  using OutT = typename QT::T;
  extern __shared__ float s_w[];  // [max_parts] weights, then [kCtaWarps][D] partial sums
  __shared__ float s_red[kCtaWarps];
  grid_dependency_wait();
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
  // warp w's partitions are w, w + W, ...: its first kIn partials are
  // requested before the weights are known (their latency overlaps the
  // log-sum-exp pass), then kIn stay in flight
  constexpr int W = kCtaWarps;
  constexpr int kIn = 8;
  constexpr int kStride = D / 4;
  const float4* op = reinterpret_cast<const float4*>(p.o_part + head * p.max_parts * D) + lane;
  const bool dims = lane < kLanes;
  float4 pf[kIn];
#pragma unroll
  for (int j = 0; j < kIn; ++j) {
    const int i = warp + j * W;
    pf[j] = dims && i < np ? __ldg(op + (size_t)i * kStride) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float* lse = p.lse + head * p.max_parts;
  float m = -INFINITY;
  for (int i = tid; i < np; i += 32 * W) m = fmaxf(m, __ldg(lse + i));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  m = s_red[0];
#pragma unroll
  for (int w = 1; w < W; ++w) m = fmaxf(m, s_red[w]);
  __syncthreads();
  float sum = 0.0f;
  for (int i = tid; i < np; i += 32 * W) {
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
  for (int w = 0; w < W; ++w) sum += s_red[w];
  float* s_acc = s_w + ((p.max_parts + 3) & ~3);
  float4 a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0;; base += kIn) {
    // partials base .. base + kIn - 1 of this warp are in pf
#pragma unroll
    for (int j = 0; j < kIn; ++j) {
      const int i = warp + (base + j) * W;
      if (i < np) a[j & 3] = fma4(s_w[i], pf[j], a[j & 3]);
    }
    if (warp + (base + kIn) * W >= np) break;
#pragma unroll
    for (int j = 0; j < kIn; ++j) {
      const int i = warp + (base + kIn + j) * W;
      pf[j] = dims && i < np ? __ldg(op + (size_t)i * kStride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (dims)
    reinterpret_cast<float4*>(s_acc + warp * D)[lane] =
        make_float4((a[0].x + a[1].x) + (a[2].x + a[3].x), (a[0].y + a[1].y) + (a[2].y + a[3].y),
                    (a[0].z + a[1].z) + (a[2].z + a[3].z), (a[0].w + a[1].w) + (a[2].w + a[3].w));
  __syncthreads();
  if (tid < D) {
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < W; ++w) acc += s_acc[w * D + tid];
    store_out(out + tid, acc / sum);
  }
}

// Launches kernel k on `stream` as a programmatic dependent of the launch
// before it (the kernels wait for it with grid_dependency_wait).
template <class K>
int launch_dependent(K k, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     const AttnParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <class QT, int D>
int launch_merge_shape(const AttnParams& p, cudaStream_t stream) {
  int rc;
  if (p.max_parts <= kWarpParts) {
    const long long pairs = (long long)p.num_rows * p.num_heads;
    const long long ctas = (pairs + kMergeWarps - 1) / kMergeWarps;
    if (ctas > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    rc = launch_dependent(lse_merge_warp_kernel<QT, D>, dim3((unsigned)ctas),
                          dim3(32 * kMergeWarps), 0, stream, p);
  } else {
    auto k = lse_merge_cta_kernel<QT, D>;
    const size_t smem = ((size_t)(p.max_parts + 3) / 4 * 4 + kCtaWarps * D) * sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
      return PKV_ERR_CUDA;
    rc = launch_dependent(k, dim3(p.num_rows, p.num_heads), dim3(32 * kCtaWarps), smem, stream, p);
  }
  return rc == PKV_OK && cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
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
