// A mixed batch in one launch: single-token decode rows and prefill chunks
// ("第32讲 … Prefill vs Decode …" §5.4, chunked prefill: a step's batch holds
// both the running decodes and slices of new prompts; devpress.csdn.net vLLM
// overview, "8、推理流程").
//
// The two kinds of work want different things from an SM: decode streams K/V
// at whatever rate the SM's copy engine sustains (HBM-bound in aggregate),
// the chunks keep the tensor pipe and the softmax warps busy on K/V tiles
// that mostly come from L2.  Run back to back, each launch spreads over every
// SM and the step pays both tails; here the CTAs are split between the two:
// CTAs [0, n_pre) run the prefill kernel body over the chunks, the others the
// decode kernel body over the decode rows, each body sharing its items among
// its own CTAs.  Every CTA computes the same split at start from the batch
// (decode keys and prefill key tiles, weighed by their per-SM costs), so no
// host-side view of the lengths is needed.
//
// The decode rows use the decode body's split-K partitions; their partials
// are merged by the usual log-sum-exp merge launch afterwards.

#include "decode_tc.cuh"
#include "prefill_tc.cuh"

namespace pkv {
namespace {

constexpr int kMixThreads = 384;  // the prefill body's CTA; decode uses 320 of them
// Per-SM cost model of the split (SM nanoseconds), from the two kernels' own
// rates on one GB300: a 128-key tile of a prefill item (two 128-row query
// tiles) takes about 2.6 us; a decode SM streams about 40 GB/s of K/V, i.e.
// 12.8 ns per key and KV head at head_dim 128 in 16 bits (K and V rows).
constexpr double kPreNsPerTile = 2600.0;
constexpr double kDecNsPerKey = 12.8;

// CTAs for the chunks (the rest decode), the same in every CTA.  scratch holds
// 2 x (threads / 32) int64 values.
__device__ int split_ctas(const AttnParams& pd, const AttnParams& pp, int forced,
                          long long* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long wd = 0, wp = 0, items = 0;
  const int cap = pd.max_blocks_per_seq * kBlockSize;
  for (int s = tid; s < pd.num_rows; s += kMixThreads) {
    const int k = __ldg(pd.context_lens + s);
    wd += k < 0 ? 0 : (k > cap ? cap : k);
  }
  const int rpt = 128 / pp.group;  // query tokens per 128-row tile
  for (int s = tid; s < pp.num_seqs; s += kMixThreads) {
    const int q0 = __ldg(pp.query_start_loc + s);
    int qlen = __ldg(pp.query_start_loc + s + 1) - q0;
    int ctx = __ldg(pp.context_lens + s);
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    qlen = qlen < 0 ? 0 : (qlen > ctx ? ctx : qlen);
    const int tiles = (qlen + rpt - 1) / rpt;
    const int pairs = (tiles + 1) / 2;
    const int kt = (ctx - qlen / 2 + 127) / 128;
    wp += (long long)pairs * (kt > 0 ? kt : 1);
    items += pairs;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    wd += __shfl_xor_sync(kFull, wd, o);
    wp += __shfl_xor_sync(kFull, wp, o);
    items += __shfl_xor_sync(kFull, items, o);
  }
  if (lane == 0) {
    scratch[warp] = wd;
    scratch[kMixThreads / 32 + warp] = wp;
    scratch[2 * (kMixThreads / 32) + warp] = items;
  }
  __syncthreads();
  wd = wp = items = 0;
  for (int w = 0; w < kMixThreads / 32; ++w) {
    wd += scratch[w];
    wp += scratch[kMixThreads / 32 + w];
    items += scratch[2 * (kMixThreads / 32) + w];
  }
  __syncthreads();  // the scratch is the bodies' shared memory
  const int grid = gridDim.x;
  items *= pp.num_kv_heads;  // prefill work items
  int n;
  if (forced > 0) {
    n = forced;
  } else {
    const double cp = (double)wp * pp.num_kv_heads * kPreNsPerTile;
    const double cd = (double)wd * pd.num_kv_heads * kDecNsPerKey;
    n = (int)(grid * cp / (cp + cd) + 0.5);
  }
  if (n > items) n = (int)items;
  if (n > grid - 1) n = grid - 1;
  return n < 1 ? 1 : n;
}

// kH: heads the decode softmax computes (4 for groups of at most 4, else 8)
template <class QT, int kH>
__global__ void __launch_bounds__(kMixThreads, 1)
    mixed_tc_kernel(const AttnParams pd, const AttnParams pp,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_qd,
                    const __grid_constant__ CUtensorMap tm_qp, int kv_rows, int forced) {
  extern __shared__ uint8_t smem_raw[];
  long long* scratch = reinterpret_cast<long long*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int n_pre = split_ctas(pd, pp, forced, scratch);
  if ((int)blockIdx.x < n_pre)
    pre_tc::prefill_body<QT, false, false>(pp, tm_k, tm_v, tm_qp, kv_rows, blockIdx.x, n_pre,
                                           smem_raw);
  else
    dec_tc::decode_body<QT, false, false, kMixThreads, kH>(pd, tm_k, tm_v, tm_qd, kv_rows,
                                                       blockIdx.x - n_pre, gridDim.x - n_pre,
                                                       smem_raw);
}

template <class QT>
int launch_mixed_typed(const AttnParams& pd, const AttnParams& pp, int total_q, int forced,
                       cudaStream_t stream) {
  const bool bf16 = std::is_same<QT, BF16>::value;
  const uint64_t kv_rows = (uint64_t)pd.num_blocks * pd.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv, tqd, tqp;
  using DL = dec_tc::Layout<false, false>;
  if (!make_map_2d(&tk, pd.k_cache, kv_rows, bf16, 16) ||
      !make_map_2d(&tv, pd.v_cache, kv_rows, bf16, 16) ||
      !make_map_2d(&tqd, pd.q, (uint64_t)pd.num_rows * pd.num_heads, bf16, DL::kRows) ||
      !make_map_q3d(&tqp, pp.q, (uint64_t)total_q, (uint32_t)pp.num_heads, bf16,
                    (uint32_t)pp.group, (uint32_t)(pre_tc::kRowsM / pp.group)))
    return PKV_ERR_CUDA;
  constexpr size_t kDecSmem = sizeof(dec_tc::Smem<false, false>);
  constexpr size_t kPreSmem = sizeof(pre_tc::Smem);
  constexpr size_t smem = (kDecSmem > kPreSmem ? kDecSmem : kPreSmem) + 1024;
  static_assert(smem <= 232448, "shared memory budget of one CTA");
  static_assert(3 * (kMixThreads / 32) * sizeof(long long) <= kPreSmem, "split scratch");
  const bool g4 = pd.group <= 4;
  auto kern = g4 ? mixed_tc_kernel<QT, 4> : mixed_tc_kernel<QT, 8>;
  static bool configured[2] = {false, false};
  if (!configured[g4]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    configured[g4] = true;
  }
  const int grid = sm_count();
  if (grid < 2) return PKV_ERR_UNSUPPORTED;
  kern<<<grid, kMixThreads, smem, stream>>>(pd, pp, tk, tv, tqd, tqp, (int)kv_rows, forced);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

bool tc_mixed_supported(const AttnParams& pd, const AttnParams& pp, int q_dtype, int kv_dtype,
                        int head_dim) {
  if (kv_dtype != q_dtype || pd.group > 8) return false;
  if (pd.num_rows > dec_tc::kMaxSeqs || pp.num_seqs > pre_tc::kMaxSeqs) return false;
  return tc_decode_supported(pd, q_dtype, kv_dtype, head_dim) &&
         tc_prefill_supported(pp, q_dtype, kv_dtype, head_dim);
}

int launch_mixed_tc(const AttnParams& pd, const AttnParams& pp, int q_dtype, int total_q,
                    int prefill_ctas, cudaStream_t stream) {
  return q_dtype == PKV_BF16 ? launch_mixed_typed<BF16>(pd, pp, total_q, prefill_ctas, stream)
                             : launch_mixed_typed<F16>(pd, pp, total_q, prefill_ctas, stream);
}

}  // namespace pkv
