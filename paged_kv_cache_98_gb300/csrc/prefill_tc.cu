// Chunked-prefill attention on tcgen05: the kernel and its launcher.  The
// device code (design notes, roles, modes) is in prefill_tc.cuh, shared with
// the fused mixed-batch kernel.

#include <atomic>

#include "prefill_pair.cuh"

namespace pkv {

// Kernel for causal and draft-tree chunks (pkv_debug_prefill_pairs): 1 CTA
// pairs, 0 one CTA per tile, 2 (the default) pairs for draft trees only.
// Measured on one GB300: draft trees 0.867 -> 0.831 ms on pairs (a tree's rows
// per KV head become one item, so its context is read once), causal chunks of
// the mixed batch 0.0822 ms either way.
std::atomic<int> g_prefill_pairs{2};

namespace {
using namespace pre_tc;

// kTree: draft-tree mode (per-row ancestor masks over the chunk's keys);
// kAlt: shared-prefix mode (non-causal, key chunks, partial outputs)
// kFP8: E4M3 caches (causal or draft-tree chunks)
template <class QT, bool kTree, bool kAlt, bool kFP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, int kv_rows) {
  extern __shared__ uint8_t smem_raw[];
  // shared-prefix pass: the cascade's own-keys decode, launched after it as a
  // dependent, may start on the SMs this grid's last wave leaves free
  if constexpr (kAlt) tc::launch_dependents();
  prefill_body<QT, kTree, kAlt, kFP8>(p, tm_k, tm_v, tm_q, kv_rows, blockIdx.x, gridDim.x,
                                      smem_raw);
}

// The query of an E4M3-cache prefill, split per (row, head) for 8-bit MMAs:
// q / s = hi + lo with hi = E4M3(q / s), lo = E4M3(q / s - hi) and
// s = max|q| / 448 (1 for a zero row); together about 8 significant bits.
// Sixteen lanes per (row, head), eight elements (one 16-byte load) per lane;
// each half-warp splits kPerHalf consecutive (row, head)s, their loads issued
// first.  hi rows [rows][heads][128 B], then the lo rows, then s [rows][heads].
constexpr int kPerHalf = 2;

template <class QT>
__global__ void __launch_bounds__(256) split_query_kernel(const typename QT::T* __restrict__ q,
                                                          uint8_t* __restrict__ hi,
                                                          uint8_t* __restrict__ lo,
                                                          float* __restrict__ scale,
                                                          long long row_heads) {
  const long long half = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
  const int lane = threadIdx.x & 15;
  uint4 raw[kPerHalf];
#pragma unroll
  for (int j = 0; j < kPerHalf; ++j) {
    const long long w = half * kPerHalf + j;
    raw[j] = w < row_heads ? __ldg(reinterpret_cast<const uint4*>(q + w * kD) + lane)
                           : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < kPerHalf; ++j) {
    const long long w = half * kPerHalf + j;
    float f[8];
    to_float(raw[j], f, QT());
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o, 16));
    const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;
    uint32_t h4[2] = {0, 0}, l4[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float x0 = f[i] * inv, x1 = f[i + 1] * inv;
      const __nv_fp8x2_storage_t h2 =
          __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
      __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3);
      const float2 hv = __half22float2(*reinterpret_cast<__half2*>(&hr));
      const __nv_fp8x2_storage_t l2 =
          __nv_cvt_float2_to_fp8x2(make_float2(x0 - hv.x, x1 - hv.y), __NV_SATFINITE, __NV_E4M3);
      h4[i >> 2] |= (uint32_t)h2 << (8 * (i & 3));
      l4[i >> 2] |= (uint32_t)l2 << (8 * (i & 3));
    }
    if (w < row_heads) {
      reinterpret_cast<uint2*>(hi + w * kD)[lane] = make_uint2(h4[0], h4[1]);
      reinterpret_cast<uint2*>(lo + w * kD)[lane] = make_uint2(l4[0], l4[1]);
      if (lane == 0) scale[w] = amax > 0.0f ? amax / 448.0f : 1.0f;
    }
  }
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Causal and draft-tree chunks on CTA pairs (prefill_pair.cuh).
template <class QT, bool kTree>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, int kv_rows) {
  extern __shared__ uint8_t smem_raw[];
  prefill_pair_body<QT, kTree>(p, tm_k, tm_v, tm_q, kv_rows, blockIdx.x >> 1, gridDim.x >> 1,
                               smem_raw);
}

template <class QT>
int launch_pairs(const AttnParams& p, int total_q, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tq, int kv_rows, cudaStream_t stream) {
  const size_t smem = sizeof(PairSmem) + 1024;
  static_assert(sizeof(PairSmem) + 1024 <= 232448, "shared memory budget of one CTA");
  static_assert(offsetof(PairSmem, ring) % 1024 == 0 && offsetof(PairSmem, q) % 1024 == 0 &&
                    offsetof(PairSmem, tail) % 1024 == 0,
                "swizzled buffers must start on 1024-byte boundaries");
  const bool tree = p.tree_mask != nullptr;
  auto kern = tree ? prefill_pair_kernel<QT, true> : prefill_pair_kernel<QT, false>;
  static int max_pairs[2] = {0, 0};  // clusters of two that fit on the GPU at once
  int& mp = max_pairs[tree ? 1 : 0];
  if (mp == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sm_count());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return PKV_ERR_CUDA;
    if (n < 1) return PKV_ERR_UNSUPPORTED;
    mp = n;
  }
  // an upper bound of the items: every sequence's 256-row tile pairs, times the KV heads
  const long long tiles =
      ((long long)total_q * p.group + (long long)p.num_seqs * (kRowsPair - 1)) / kRowsPair;
  const long long items = (tiles + p.num_seqs) / 2 * p.num_kv_heads;
  const int pairs = (int)(items < mp ? (items > 0 ? items : 1) : mp);
  kern<<<2 * pairs, kThreads, smem, stream>>>(p, tk, tv, tq, kv_rows);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// q8: E4M3 caches, the split query (hi rows then lo rows) or null.
template <class QT>
int launch_typed(const AttnParams& p, int total_q, cudaStream_t stream, const uint8_t* q8 = nullptr) {
  const bool bf16 = std::is_same<QT, BF16>::value;
  const bool fp8 = q8 != nullptr;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv, tq;
  const bool maps =
      fp8 ? make_map_e4m3(&tk, p.k_cache, kv_rows, 16) && make_map_e4m3(&tv, p.v_cache, kv_rows, 16) &&
                make_map_q3d_e4m3(&tq, q8, 2 * (uint64_t)total_q, (uint32_t)p.num_heads,
                                  (uint32_t)p.group, (uint32_t)(kRowsM / p.group))
          : make_map_2d(&tk, p.k_cache, kv_rows, bf16, 16) &&
                make_map_2d(&tv, p.v_cache, kv_rows, bf16, 16) &&
                make_map_q3d(&tq, p.q, (uint64_t)total_q, (uint32_t)p.num_heads, bf16,
                             (uint32_t)p.group, (uint32_t)(kRowsM / p.group));
  if (!maps) return PKV_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget of one CTA");
  static_assert(offsetof(Smem, ring) % 1024 == 0 && offsetof(Smem, q) % 1024 == 0 &&
                    offsetof(Smem, tail) % 1024 == 0,
                "swizzled buffers must start on 1024-byte boundaries");
  static_assert(offsetof(Smem, q) == offsetof(Smem, ring) + kStages * kTileBytes,
                "q[0] is the ring's fifth stage in shared-prefix mode");
  const int mode = p.tree_mask != nullptr ? 1 : (p.partial_out ? 2 : 0);
  const int pairs = g_prefill_pairs.load(std::memory_order_relaxed);
  if (!fp8 && mode != 2 && p.seq_rows == nullptr && (pairs == 1 || (pairs == 2 && mode == 1))) {
    const int rc = launch_pairs<QT>(p, total_q, tk, tv, tq, (int)kv_rows, stream);
    if (rc != PKV_ERR_UNSUPPORTED) return rc;  // (no pair fits: the single-CTA kernel)
  }
  if (fp8 && mode == 2) return PKV_ERR_UNSUPPORTED;
  auto kern = fp8 ? (mode == 1 ? prefill_tc_kernel<QT, true, false, true>
                               : prefill_tc_kernel<QT, false, false, true>)
              : mode == 1 ? prefill_tc_kernel<QT, true, false>
              : mode == 2 ? prefill_tc_kernel<QT, false, true>
                          : prefill_tc_kernel<QT, false, false>;
  const int slot = mode + (fp8 ? 3 : 0);
  static bool configured[6] = {false, false, false, false, false, false};
  if (!configured[slot]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    configured[slot] = true;
  }
  // an upper bound of the items: every sequence's tile pairs, times the KV heads
  const long long tiles = ((long long)total_q * p.group + (long long)p.num_seqs * (kRowsM - 1)) /
                          kRowsM;
  const long long items = (tiles + p.num_seqs) / 2 * p.num_kv_heads;
  int grid = sm_count();
  // (key chunks multiply the items of the shared-prefix pass)
  if (!p.partial_out && items < grid) grid = (int)(items > 0 ? items : 1);
  kern<<<grid, kThreads, smem, stream>>>(p, tk, tv, tq, (int)kv_rows);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

bool tc_prefill_supported(const AttnParams& p, int q_dtype, int kv_dtype, int head_dim) {
  if (head_dim != kD || p.query_start_loc == nullptr) return false;
  // E4M3 caches: causal and draft-tree chunks (the shared-prefix pass is 16-bit)
  if (kv_dtype != q_dtype && !(kv_dtype == PKV_FP8_E4M3 && !p.partial_out)) return false;
  if (p.group < 1 || p.group > kRowsM || kRowsM % p.group != 0) return false;
  if (p.num_seqs > kMaxSeqs) return false;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  if (kv_rows + 16 >= (1ull << 31)) return false;
  if ((uint64_t)p.num_rows * p.num_heads >= (1ull << 31)) return false;
  return tmap_available();
}

int launch_prefill_tc(const AttnParams& p, int q_dtype, int total_q, cudaStream_t stream) {
  return q_dtype == PKV_BF16 ? launch_typed<BF16>(p, total_q, stream)
                             : launch_typed<F16>(p, total_q, stream);
}

// hi rows, the lo rows right after them (one tensor map spans both), then s
size_t prefill_q8_bytes(int total_q, int num_heads) {
  const size_t rh = (size_t)total_q * num_heads;
  return round256(2 * rh * kD) + round256(rh * sizeof(float));
}

int launch_prefill_tc_fp8(const AttnParams& p, int q_dtype, int total_q, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  const size_t need = prefill_q8_bytes(total_q, p.num_heads);
  if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKV_ERR_INVALID_ARG;
  const size_t rh = (size_t)total_q * p.num_heads;
  uint8_t* hi = static_cast<uint8_t*>(workspace);
  uint8_t* lo = hi + rh * kD;
  float* scale = reinterpret_cast<float*>(hi + round256(2 * rh * kD));
  // sixteen threads per kPerHalf (row, head)s
  const long long blocks = (((long long)rh + kPerHalf - 1) / kPerHalf * 16 + 255) / 256;
  if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  AttnParams c = p;
  c.q8_scale = scale;
  if (q_dtype == PKV_BF16) {
    split_query_kernel<BF16><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(p.q), hi, lo, scale, (long long)rh);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    return launch_typed<BF16>(c, total_q, stream, hi);
  }
  split_query_kernel<F16><<<(unsigned)blocks, 256, 0, stream>>>(
      static_cast<const __half*>(p.q), hi, lo, scale, (long long)rh);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return launch_typed<F16>(c, total_q, stream, hi);
}

}  // namespace pkv
