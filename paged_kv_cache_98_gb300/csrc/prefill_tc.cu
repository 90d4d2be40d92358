// Chunked-prefill attention on tcgen05: the kernel and its launcher.  The
// device code (design notes, roles, modes) is in prefill_tc.cuh, shared with
// the fused mixed-batch kernel.

#include <atomic>

#include "prefill_pair.cuh"

namespace pkv {

// Causal and draft-tree chunks on CTA pairs (1) or on the single-CTA kernel
// (0, the default); see pkv_debug_prefill_pairs.
std::atomic<int> g_prefill_pairs{0};

namespace {
using namespace pre_tc;

// kTree: draft-tree mode (per-row ancestor masks over the chunk's keys);
// kAlt: shared-prefix mode (non-causal, key chunks, partial outputs)
template <class QT, bool kTree, bool kAlt>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, int kv_rows) {
  extern __shared__ uint8_t smem_raw[];
  prefill_body<QT, kTree, kAlt>(p, tm_k, tm_v, tm_q, kv_rows, blockIdx.x, gridDim.x, smem_raw);
}

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

template <class QT>
int launch_typed(const AttnParams& p, int total_q, cudaStream_t stream) {
  const bool bf16 = std::is_same<QT, BF16>::value;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv, tq;
  if (!make_map_2d(&tk, p.k_cache, kv_rows, bf16, 16) ||
      !make_map_2d(&tv, p.v_cache, kv_rows, bf16, 16) ||
      !make_map_q3d(&tq, p.q, (uint64_t)total_q, (uint32_t)p.num_heads, bf16, (uint32_t)p.group,
                    (uint32_t)(kRowsM / p.group)))
    return PKV_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget of one CTA");
  static_assert(offsetof(Smem, ring) % 1024 == 0 && offsetof(Smem, q) % 1024 == 0 &&
                    offsetof(Smem, tail) % 1024 == 0,
                "swizzled buffers must start on 1024-byte boundaries");
  static_assert(offsetof(Smem, q) == offsetof(Smem, ring) + kStages * kTileBytes,
                "q[0] is the ring's fifth stage in shared-prefix mode");
  const int mode = p.tree_mask != nullptr ? 1 : (p.partial_out ? 2 : 0);
  if (mode != 2 && p.seq_rows == nullptr && g_prefill_pairs.load(std::memory_order_relaxed)) {
    const int rc = launch_pairs<QT>(p, total_q, tk, tv, tq, (int)kv_rows, stream);
    if (rc != PKV_ERR_UNSUPPORTED) return rc;  // (no pair fits: the single-CTA kernel)
  }
  auto kern = mode == 1   ? prefill_tc_kernel<QT, true, false>
              : mode == 2 ? prefill_tc_kernel<QT, false, true>
                          : prefill_tc_kernel<QT, false, false>;
  static bool configured[3] = {false, false, false};
  if (!configured[mode]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    configured[mode] = true;
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
  if (head_dim != kD || kv_dtype != q_dtype || p.query_start_loc == nullptr) return false;
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

}  // namespace pkv
