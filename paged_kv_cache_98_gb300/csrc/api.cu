// C ABI of libpagedkv.so: argument validation and kernel dispatch.  The
// declarations, data model and error conventions are in include/pagedkv.h.

#include <atomic>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "launch.h"

namespace {

constexpr int kDefaultPartition = 512;
constexpr int kCascadeChunk = 2048;  // keys per partial of the shared-prefix pass

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is16bit(int dt) { return dt == PKV_F16 || dt == PKV_BF16; }

int effective_partition(int partition_size, int max_context_len) {
  int ps = partition_size == 0 ? kDefaultPartition : partition_size;
  (void)max_context_len;
  return ps;
}

int parts_for(int max_context_len, int partition) {
  int n = (max_context_len + partition - 1) / partition;
  return n < 1 ? 1 : n;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t split_workspace(size_t rows, int num_heads, int head_dim, int max_parts) {
  if (max_parts <= 1) return 0;
  const size_t heads = rows * (size_t)num_heads * (size_t)max_parts;
  return round_up(heads * sizeof(float), 256) + round_up(heads * head_dim * sizeof(float), 256);
}

int pow2_at_least(int g) {
  int p = 1;
  while (p < g) p <<= 1;
  return p;
}

// Checks shared by decode and prefill.
int check_attention_args(const void* out, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                         int num_blocks, int max_context_len, float scale, int q_dtype,
                         int kv_dtype, float k_scale, float v_scale) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0 || max_context_len < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (block_size != pkv::kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_heads / num_kv_heads > 16) return PKV_ERR_UNSUPPORTED;
  if (!is16bit(q_dtype)) return PKV_ERR_UNSUPPORTED;
  if (kv_dtype != q_dtype && kv_dtype != PKV_FP8_E4M3) return PKV_ERR_UNSUPPORTED;
  if (kv_dtype == PKV_FP8_E4M3) {
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || !std::isfinite(k_scale) ||
        !std::isfinite(v_scale))
      return PKV_ERR_INVALID_ARG;
  }
  if ((long long)max_blocks_per_seq * pkv::kBlockSize > (1LL << 30)) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

int run_attention(pkv::AttnParams& p, int q_dtype, int kv_dtype, int head_dim, float scale,
                  float k_scale, float v_scale, void* workspace, size_t ws_need,
                  size_t workspace_bytes, cudaStream_t stream) {
  if (ws_need > 0) {
    if (!workspace || workspace_bytes < ws_need) return PKV_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKV_ERR_INVALID_ARG;
    const size_t heads = (size_t)p.num_rows * p.num_heads * p.max_parts;
    p.lse = static_cast<float*>(workspace);
    p.o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        round_up(heads * sizeof(float), 256));
  } else {
    p.lse = nullptr;
    p.o_part = nullptr;
  }
  const bool fp8 = kv_dtype == PKV_FP8_E4M3;
  p.q_scale = scale * pkv::kLog2e * (fp8 ? k_scale : 1.0f);
  p.v_scale = fp8 ? v_scale : 1.0f;
  const int g_pad = pow2_at_least(p.group);
  pkv::take_debug_hook(p);
  int rc;
  if (pkv::tc_decode_supported(p, q_dtype, kv_dtype, head_dim))
    rc = pkv::launch_paged_decode_tc(p, q_dtype, kv_dtype, stream);
  else
    rc = pkv::launch_paged_attention_simt(p, q_dtype, kv_dtype, head_dim, g_pad, stream);
  if (rc != PKV_OK) return rc;
  if (p.max_parts > 1) rc = pkv::launch_lse_merge(p, q_dtype, head_dim, stream);
  return rc;
}

}  // namespace

namespace pkv {

// The failure-detection test hook armed by pkv_debug_arm_wait_timeout: taken
// (and cleared) by the next attention call.
extern std::atomic<int> g_prefill_pairs;  // prefill_tc.cu
std::atomic<int> g_hook_skip{0};
std::atomic<unsigned long long> g_hook_limit_ns{0};

void take_debug_hook(AttnParams& p) {
  if (g_hook_skip.load(std::memory_order_relaxed) == 0) return;
  p.skip_copy = g_hook_skip.exchange(0);
  p.wait_limit_ns = g_hook_limit_ns.exchange(0);
}

int launch_paged_attention_simt(const AttnParams& p, int q_dtype, int kv_dtype, int head_dim,
                                int g_pad, cudaStream_t stream) {
  if (q_dtype == PKV_F16)
    return kv_dtype == PKV_FP8_E4M3 ? launch_simt_f16_e4m3(p, head_dim, g_pad, stream)
                                    : launch_simt_f16_f16(p, head_dim, g_pad, stream);
  return kv_dtype == PKV_FP8_E4M3 ? launch_simt_bf16_e4m3(p, head_dim, g_pad, stream)
                                  : launch_simt_bf16_bf16(p, head_dim, g_pad, stream);
}
}  // namespace pkv

extern "C" {

int pkv_version(void) { return 100; }

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE: return "device-side check failed";
    case PKV_ERR_TIMEOUT: return "device-side wait timed out";
    case PKV_ERR_NO_BLOCKS: return "block pool exhausted";
    default: return "unknown status";
  }
}

int pkv_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, pkv_dtype src_dtype,
                          pkv_dtype cache_dtype, float k_scale, float v_scale,
                          uint32_t* device_errors, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (block_size != pkv::kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (!is16bit(src_dtype)) return PKV_ERR_UNSUPPORTED;
  if (cache_dtype != src_dtype && cache_dtype != PKV_FP8_E4M3) return PKV_ERR_UNSUPPORTED;
  if (cache_dtype == PKV_FP8_E4M3 &&
      (!(k_scale > 0.0f) || !(v_scale > 0.0f) || !std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return PKV_ERR_INVALID_ARG;
  return pkv::launch_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                       num_kv_heads, head_dim, num_blocks, src_dtype,
                                       cache_dtype, k_scale, v_scale, device_errors,
                                       static_cast<cudaStream_t>(stream));
}

size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                 int partition_size) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
  const int ps = effective_partition(partition_size, max_context_len);
  if (ps <= 0) return 0;
  return split_workspace((size_t)num_seqs, num_heads, head_dim, parts_for(max_context_len, ps));
}

int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int max_blocks_per_seq, int num_blocks,
                               int max_context_len, float scale, pkv_dtype q_dtype,
                               pkv_dtype kv_dtype, float k_scale, float v_scale,
                               int partition_size, void* workspace, size_t workspace_bytes,
                               uint32_t* device_errors, void* stream) {
  int rc = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                num_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, num_blocks, max_context_len, scale, q_dtype,
                                kv_dtype, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (partition_size != 0 &&
      (partition_size % pkv::kBlockSize != 0 || partition_size < pkv::kBlockSize ||
       partition_size > 512))
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  const int ps = effective_partition(partition_size, max_context_len);
  pkv::AttnParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start_loc = nullptr;
  p.num_seqs = num_seqs;
  p.num_rows = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.partition = ps;
  p.max_parts = parts_for(max_context_len, ps);
  if (p.max_parts > 16384) return PKV_ERR_UNSUPPORTED;
  p.errors = device_errors;
  const size_t need = split_workspace((size_t)num_seqs, num_heads, head_dim, p.max_parts);
  return run_attention(p, q_dtype, kv_dtype, head_dim, scale, k_scale, v_scale, workspace, need,
                       workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t pkv_prefill_workspace_size(int total_q, int num_heads, int head_dim, int max_context_len,
                                  int max_q_len) {
  (void)max_q_len;
  if (total_q <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
  // CUDA-core path: split-K partials; E4M3 caches on tensor cores: the split query
  const size_t simt = split_workspace((size_t)total_q, num_heads, head_dim,
                                      parts_for(max_context_len, kDefaultPartition));
  const size_t q8 = head_dim == 128 ? pkv::prefill_q8_bytes(total_q, num_heads) : 0;
  return simt > q8 ? simt : q8;
}

int pkv_paged_attention_prefill_chunk(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens,
                                      const int32_t* query_start_loc, int num_seqs, int total_q,
                                      int max_q_len, int num_heads, int num_kv_heads,
                                      int head_dim, int block_size, int max_blocks_per_seq,
                                      int num_blocks, int max_context_len, float scale,
                                      pkv_dtype q_dtype, pkv_dtype kv_dtype, float k_scale,
                                      float v_scale, void* workspace, size_t workspace_bytes,
                                      uint32_t* device_errors, void* stream) {
  int rc = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                num_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, num_blocks, max_context_len, scale, q_dtype,
                                kv_dtype, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (!query_start_loc || total_q < 0 || max_q_len < 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  pkv::AttnParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start_loc = query_start_loc;
  p.num_seqs = num_seqs;
  p.num_rows = total_q;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.partition = kDefaultPartition;
  p.max_parts = parts_for(max_context_len, kDefaultPartition);
  if (p.max_parts > 16384) return PKV_ERR_UNSUPPORTED;
  p.errors = device_errors;
  if (pkv::tc_prefill_supported(p, q_dtype, kv_dtype, head_dim)) {
    // tensor-core path: one pass over the keys per tile, no workspace
    const bool fp8 = kv_dtype == PKV_FP8_E4M3;
    p.q_scale = scale * pkv::kLog2e * (fp8 ? k_scale : 1.0f);
    p.v_scale = fp8 ? v_scale : 1.0f;
    pkv::take_debug_hook(p);
    if (fp8)
      return pkv::launch_prefill_tc_fp8(p, q_dtype, total_q, workspace, workspace_bytes,
                                        static_cast<cudaStream_t>(stream));
    return pkv::launch_prefill_tc(p, q_dtype, total_q, static_cast<cudaStream_t>(stream));
  }
  const size_t need = split_workspace((size_t)total_q, num_heads, head_dim, p.max_parts);
  return run_attention(p, q_dtype, kv_dtype, head_dim, scale, k_scale, v_scale, workspace, need,
                       workspace_bytes, static_cast<cudaStream_t>(stream));
}

int pkv_paged_attention_prefill_tree(void* out, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables,
                                     const int32_t* context_lens, const int32_t* query_start_loc,
                                     const uint64_t* tree_mask, int num_seqs, int total_q,
                                     int max_q_len, int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_blocks_per_seq, int num_blocks,
                                     int max_context_len, float scale, pkv_dtype q_dtype,
                                     pkv_dtype kv_dtype, float k_scale, float v_scale,
                                     uint32_t* device_errors, void* stream) {
  int rc = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                num_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, num_blocks, max_context_len, scale, q_dtype,
                                kv_dtype, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (!query_start_loc || !tree_mask || total_q < 0 || max_q_len < 0 || max_q_len > 64)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  pkv::AttnParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start_loc = query_start_loc;
  p.tree_mask = tree_mask;
  p.num_seqs = num_seqs;
  p.num_rows = total_q;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.partition = kDefaultPartition;
  p.max_parts = parts_for(max_context_len, kDefaultPartition);
  if (p.max_parts > 16384) return PKV_ERR_UNSUPPORTED;
  p.errors = device_errors;
  // the tensor-core prefill kernel carries the mask; other shapes (and E4M3
  // caches, whose query split needs a workspace this call does not take) are
  // unsupported
  if (kv_dtype != q_dtype || !pkv::tc_prefill_supported(p, q_dtype, kv_dtype, head_dim))
    return PKV_ERR_UNSUPPORTED;
  p.q_scale = scale * pkv::kLog2e;
  p.v_scale = 1.0f;
  pkv::take_debug_hook(p);
  return pkv::launch_prefill_tc(p, q_dtype, total_q, static_cast<cudaStream_t>(stream));
}

size_t pkv_mixed_workspace_size(int num_decode, int total_q, int num_heads, int head_dim,
                                int max_context_len) {
  const size_t d = pkv_decode_workspace_size(num_decode, num_heads, head_dim, max_context_len, 0);
  const size_t p =
      pkv_prefill_workspace_size(total_q - num_decode, num_heads, head_dim, max_context_len, 0);
  return d > p ? d : p;
}

int pkv_paged_attention_mixed(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* context_lens,
                              const int32_t* query_start_loc, int num_decode, int num_seqs,
                              int total_q, int max_q_len, int num_heads, int num_kv_heads,
                              int head_dim, int block_size, int max_blocks_per_seq,
                              int num_blocks, int max_context_len, float scale,
                              pkv_dtype q_dtype, pkv_dtype kv_dtype, float k_scale,
                              float v_scale, int prefill_ctas, void* workspace,
                              size_t workspace_bytes, uint32_t* device_errors, void* stream) {
  int rc = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                num_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, num_blocks, max_context_len, scale, q_dtype,
                                kv_dtype, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (!query_start_loc || num_decode < 0 || num_decode > num_seqs || total_q < num_decode ||
      max_q_len < 0 || prefill_ctas < 0)
    return PKV_ERR_INVALID_ARG;
  const int num_chunks = num_seqs - num_decode;
  // the chunks' block-table rows, lengths and offsets follow the decode rows'
  const int32_t* bt_pre = block_tables + (size_t)num_decode * max_blocks_per_seq;
  if (num_chunks == 0 || total_q == num_decode)
    return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                                      num_decode, num_heads, num_kv_heads, head_dim, block_size,
                                      max_blocks_per_seq, num_blocks, max_context_len, scale,
                                      q_dtype, kv_dtype, k_scale, v_scale, 0, workspace,
                                      workspace_bytes, device_errors, stream);
  if (num_decode == 0)
    return pkv_paged_attention_prefill_chunk(
        out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_seqs, total_q,
        max_q_len, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
        max_context_len, scale, q_dtype, kv_dtype, k_scale, v_scale, workspace, workspace_bytes,
        device_errors, stream);
  pkv::AttnParams pd{};
  pd.out = out;
  pd.q = q;
  pd.k_cache = static_cast<const uint8_t*>(k_cache);
  pd.v_cache = static_cast<const uint8_t*>(v_cache);
  pd.block_tables = block_tables;
  pd.context_lens = context_lens;
  pd.num_seqs = pd.num_rows = num_decode;
  pd.num_heads = num_heads;
  pd.num_kv_heads = num_kv_heads;
  pd.group = num_heads / num_kv_heads;
  pd.max_blocks_per_seq = max_blocks_per_seq;
  pd.num_blocks = num_blocks;
  pd.partition = kDefaultPartition;
  pd.max_parts = parts_for(max_context_len, kDefaultPartition);
  if (pd.max_parts > 16384) return PKV_ERR_UNSUPPORTED;
  pd.errors = device_errors;
  pkv::AttnParams pp = pd;
  pp.block_tables = bt_pre;
  pp.context_lens = context_lens + num_decode;
  pp.query_start_loc = query_start_loc + num_decode;
  pp.num_seqs = num_chunks;
  pp.num_rows = total_q;
  const bool fused = pkv::tc_mixed_supported(pd, pp, q_dtype, kv_dtype, head_dim);
  if (!fused) {
    // the two launches the fused kernel replaces, sharing the workspace in stream order
    rc = pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                                    num_decode, num_heads, num_kv_heads, head_dim, block_size,
                                    max_blocks_per_seq, num_blocks, max_context_len, scale,
                                    q_dtype, kv_dtype, k_scale, v_scale, 0, workspace,
                                    workspace_bytes, device_errors, stream);
    if (rc != PKV_OK) return rc;
    return pkv_paged_attention_prefill_chunk(
        out, q, k_cache, v_cache, bt_pre, context_lens + num_decode, query_start_loc + num_decode,
        num_chunks, total_q, max_q_len, num_heads, num_kv_heads, head_dim, block_size,
        max_blocks_per_seq, num_blocks, max_context_len, scale, q_dtype, kv_dtype, k_scale,
        v_scale, workspace, workspace_bytes, device_errors, stream);
  }
  const size_t need = split_workspace((size_t)num_decode, num_heads, head_dim, pd.max_parts);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKV_ERR_INVALID_ARG;
    const size_t heads = (size_t)num_decode * num_heads * pd.max_parts;
    pd.lse = static_cast<float*>(workspace);
    pd.o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         round_up(heads * sizeof(float), 256));
  }
  pd.q_scale = pp.q_scale = scale * pkv::kLog2e;
  pd.v_scale = pp.v_scale = 1.0f;
  pkv::take_debug_hook(pd);
  pp.skip_copy = pd.skip_copy;
  pp.wait_limit_ns = pd.wait_limit_ns;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = pkv::launch_mixed_tc(pd, pp, q_dtype, total_q, prefill_ctas, st);
  if (rc != PKV_OK) return rc;
  if (pd.max_parts > 1) rc = pkv::launch_lse_merge(pd, q_dtype, head_dim, st);
  return rc;
}

size_t pkv_cascade_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                  int max_prefix_len) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
      max_prefix_len < 0)
    return 0;
  // the shared prefix's chunks, then the sequence's own partitions; the
  // partials always go through the workspace
  const int slots = 2 * ((max_prefix_len + kCascadeChunk - 1) / kCascadeChunk) +
                    parts_for(max_context_len, kDefaultPartition);
  const size_t heads = (size_t)num_seqs * num_heads * slots;
  return round_up(heads * sizeof(float), 256) + round_up(heads * head_dim * sizeof(float), 256);
}

int pkv_paged_attention_decode_cascade(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* group_start,
                                       const int32_t* prefix_lens, int num_seqs, int num_groups,
                                       int num_heads, int num_kv_heads, int head_dim,
                                       int block_size, int max_blocks_per_seq, int num_blocks,
                                       int max_context_len, int max_prefix_len, float scale,
                                       pkv_dtype q_dtype, pkv_dtype kv_dtype, float k_scale,
                                       float v_scale, void* workspace, size_t workspace_bytes,
                                       uint32_t* device_errors, void* stream) {
  int rc = check_attention_args(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                num_heads, num_kv_heads, head_dim, block_size,
                                max_blocks_per_seq, num_blocks, max_context_len, scale, q_dtype,
                                kv_dtype, k_scale, v_scale);
  if (rc != PKV_OK) return rc;
  if (!group_start || !prefix_lens || num_groups < 0 || max_prefix_len < 0 ||
      max_prefix_len > max_context_len)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (kv_dtype != q_dtype || head_dim != 128) return PKV_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  pkv::AttnParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.num_seqs = num_seqs;
  p.num_rows = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.partition = kDefaultPartition;
  p.max_parts = 2 * ((max_prefix_len + kCascadeChunk - 1) / kCascadeChunk) +
                parts_for(max_context_len, kDefaultPartition);
  if (p.max_parts > 16384) return PKV_ERR_UNSUPPORTED;
  p.errors = device_errors;
  p.q_scale = scale * pkv::kLog2e;
  p.v_scale = 1.0f;
  p.prefix_chunk = kCascadeChunk;
  pkv::take_debug_hook(p);
  // pass 1: every member's query over its group's shared prefix (the prefill
  // kernel, no causal mask, one partial per chunk of the prefix)
  pkv::AttnParams pp = p;
  pp.query_start_loc = group_start;
  pp.num_seqs = num_groups;
  pp.context_lens = prefix_lens;
  pp.seq_rows = group_start;
  pp.non_causal = 1;
  pp.partial_out = 1;
  // pass 2: each sequence over its own keys (the decode kernel), then the merge
  pkv::AttnParams ps = p;
  ps.prefix_lens = prefix_lens;
  if (!pkv::tc_decode_supported(ps, q_dtype, kv_dtype, head_dim) ||
      (num_groups > 0 && !pkv::tc_prefill_supported(pp, q_dtype, kv_dtype, head_dim)))
    return PKV_ERR_UNSUPPORTED;
  const size_t need =
      pkv_cascade_workspace_size(num_seqs, num_heads, head_dim, max_context_len, max_prefix_len);
  if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PKV_ERR_INVALID_ARG;
  const size_t heads = (size_t)num_seqs * num_heads * p.max_parts;
  float* lse = static_cast<float*>(workspace);
  float* o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                           round_up(heads * sizeof(float), 256));
  pp.lse = ps.lse = lse;
  pp.o_part = ps.o_part = o_part;
  if (num_groups > 0 && max_prefix_len > 0) {
    rc = pkv::launch_prefill_tc(pp, q_dtype, num_seqs, st);
    if (rc != PKV_OK) return rc;
  }
  // the own-keys pass reads nothing the prefix pass writes: it may fill the
  // prefix pass's last wave (programmatic dependent launch)
  rc = pkv::launch_paged_decode_tc(ps, q_dtype, kv_dtype, st, num_groups > 0 && max_prefix_len > 0);
  if (rc != PKV_OK) return rc;
  return pkv::launch_lse_merge(ps, q_dtype, head_dim, st);
}

int pkv_debug_prefill_pairs(int mode) {
  if (mode < 0 || mode > 2) return PKV_ERR_INVALID_ARG;
  return pkv::g_prefill_pairs.exchange(mode);
}

int pkv_debug_arm_wait_timeout(int skip_copy, unsigned wait_limit_us) {
  if (skip_copy <= 0) return PKV_ERR_INVALID_ARG;
  pkv::g_hook_limit_ns.store((unsigned long long)wait_limit_us * 1000ull);
  pkv::g_hook_skip.store(skip_copy);
  return PKV_OK;
}

int pkv_check_errors(uint32_t* device_errors, uint32_t* bits_out, void* stream) {
  if (!device_errors) return PKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, device_errors, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaMemset(device_errors, 0, sizeof(uint32_t)) != cudaSuccess) return PKV_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  if (bits & PKV_DEVERR_TIMEOUT) return PKV_ERR_TIMEOUT;
  return bits ? PKV_ERR_DEVICE : PKV_OK;
}

}  // extern "C"
