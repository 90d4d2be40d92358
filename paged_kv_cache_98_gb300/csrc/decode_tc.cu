// Grouped-query paged decode on tcgen05: the kernel and its launcher.  The
// device code (design notes, layouts, roles) is in decode_tc.cuh, shared with
// the fused mixed-batch kernel.

#include "decode_tc.cuh"

namespace pkv {
namespace {
using namespace dec_tc;

// kH: heads the softmax computes (4 for groups of at most 4, else all rows)
template <class QT, bool G16, bool FP8, int kH>
__global__ void __launch_bounds__(tc_threads(G16, FP8), 1)
    paged_decode_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_q, int kv_rows) {
  extern __shared__ uint8_t smem_raw[];
  // launched as a dependent (cascade decode), this grid does not read its
  // predecessor but ends only after it.  (Letting the merge start early here
  // was measured slower: its resident CTAs slowed the decode.)
  decode_body<QT, G16, FP8, tc_threads(G16, FP8), kH>(p, tm_k, tm_v, tm_q, kv_rows, blockIdx.x,
                                                     gridDim.x, smem_raw);
  tc::grid_dependency_wait();
}

// ---- host side ---------------------------------------------------------------------------
template <class QT, bool G16, bool FP8, int kH = (G16 ? 16 : 8)>
int launch_tc_typed(const AttnParams& p, cudaStream_t stream, bool dependent) {
  const bool bf16 = std::is_same<QT, BF16>::value;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv;
  const bool maps = FP8 ? make_map_e4m3(&tk, p.k_cache, kv_rows, 16) &&
                              make_map_e4m3(&tv, p.v_cache, kv_rows, 16)
                        : make_map_2d(&tk, p.k_cache, kv_rows, bf16, 16) &&
                              make_map_2d(&tv, p.v_cache, kv_rows, bf16, 16);
  if (!maps) return PKV_ERR_CUDA;
  using SM = Smem<G16, FP8>;
  using L = Layout<G16, FP8>;
  const size_t smem = sizeof(SM) + 1024;
  static_assert(sizeof(SM) + 1024 <= 232448, "shared memory budget of one CTA");
  static_assert(offsetof(SM, kring) % 1024 == 0 && offsetof(SM, vring) % 1024 == 0 &&
                    offsetof(SM, q) % 1024 == 0 && offsetof(SM, pmat) % 1024 == 0 &&
                    offsetof(SM, tail) % 1024 == 0 && L::kTileBytes % 1024 == 0 &&
                    L::kQHalf % 1024 == 0 && L::kQBytes % 1024 == 0,
                "swizzled buffers must start on 1024-byte boundaries");
  static_assert(L::kStepKeys * L::kRowBytes == kTailBytes, "tail buffer = one MMA step of V");
  auto kern = paged_decode_tc_kernel<QT, G16, FP8, kH>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    configured = true;
  }
  using OutT = typename QT::T;
  // launches of at most kMaxSeqs sequences each (their rows are independent)
  for (int r0 = 0; r0 < p.num_rows; r0 += kMaxSeqs) {
    AttnParams c = p;
    c.num_rows = p.num_rows - r0 < kMaxSeqs ? p.num_rows - r0 : kMaxSeqs;
    c.num_seqs = c.num_rows;
    const size_t head0 = (size_t)r0 * p.num_heads;
    c.out = static_cast<OutT*>(p.out) + head0 * kD;
    c.q = static_cast<const OutT*>(p.q) + head0 * kD;
    c.block_tables = p.block_tables + (size_t)r0 * p.max_blocks_per_seq;
    c.context_lens = p.context_lens + r0;
    if (p.prefix_lens) c.prefix_lens = p.prefix_lens + r0;
    if (p.lse) {
      c.lse = p.lse + head0 * p.max_parts;
      c.o_part = p.o_part + head0 * p.max_parts * kD;
    }
    CUtensorMap tq;  // read by TMA on 16-bit caches, unused on E4M3 (split query)
    if (!make_map_2d(&tq, c.q, (uint64_t)c.num_rows * p.num_heads, bf16, L::kRows))
      return PKV_ERR_CUDA;
    const long long items = (long long)c.num_rows * p.num_kv_heads * p.max_parts;
    int grid = sm_count();
    if (items < grid) grid = (int)items;
    if (grid < 1) grid = 1;
    if (dependent && r0 == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(tc_threads(G16, FP8));
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr.val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, kern, c, tk, tv, tq, (int)kv_rows) != cudaSuccess)
        return PKV_ERR_CUDA;
    } else {
      kern<<<grid, tc_threads(G16, FP8), smem, stream>>>(c, tk, tv, tq, (int)kv_rows);
    }
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace

bool tc_decode_supported(const AttnParams& p, int q_dtype, int kv_dtype, int head_dim) {
  if (head_dim != kD || (kv_dtype != q_dtype && kv_dtype != PKV_FP8_E4M3)) return false;
  if (p.query_start_loc != nullptr || p.partition != kPart) return false;
  if (p.group < 2 || p.group > 16) return false;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  if (kv_rows + 16 >= (1ull << 31)) return false;
  if ((uint64_t)p.num_rows * p.num_heads + 16 >= (1ull << 31)) return false;
  if ((long long)p.num_rows * p.num_kv_heads * p.max_parts >= (1ll << 31)) return false;
  // the packed per-sequence table holds up to 2^22 (sequence, partition) pairs
  if ((long long)kMaxSeqs * p.max_parts >= (1ll << (31 - kLenBits))) return false;
  return tmap_available();
}

int launch_paged_decode_tc(const AttnParams& p, int q_dtype, int kv_dtype, cudaStream_t stream,
                           bool dependent) {
  const bool g16 = p.group > 8, g4 = p.group <= 4;
  if (kv_dtype == PKV_FP8_E4M3) {
    if (q_dtype == PKV_BF16)
      return g16  ? launch_tc_typed<BF16, true, true>(p, stream, dependent)
             : g4 ? launch_tc_typed<BF16, false, true, 4>(p, stream, dependent)
                  : launch_tc_typed<BF16, false, true>(p, stream, dependent);
    return g16  ? launch_tc_typed<F16, true, true>(p, stream, dependent)
           : g4 ? launch_tc_typed<F16, false, true, 4>(p, stream, dependent)
                : launch_tc_typed<F16, false, true>(p, stream, dependent);
  }
  if (q_dtype == PKV_BF16)
    return g16  ? launch_tc_typed<BF16, true, false>(p, stream, dependent)
           : g4 ? launch_tc_typed<BF16, false, false, 4>(p, stream, dependent)
                : launch_tc_typed<BF16, false, false>(p, stream, dependent);
  return g16  ? launch_tc_typed<F16, true, false>(p, stream, dependent)
         : g4 ? launch_tc_typed<F16, false, false, 4>(p, stream, dependent)
              : launch_tc_typed<F16, false, false>(p, stream, dependent);
}

}  // namespace pkv
