// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Longest a device-side wait may take before the kernel gives up, flags
// PKV_DEVERR_TIMEOUT and returns (about 2 s).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// One launch of the paged attention kernels.  A "row" is one query token:
// a decode sequence (query_start_loc == nullptr, row = sequence) or one query
// of a prefill chunk (row = index into q, its sequence found through
// query_start_loc).
struct AttnParams {
  void* out;                      // [rows][num_heads][head_dim], q dtype
  const void* q;                  // [rows][num_heads][head_dim], q dtype
  const uint8_t* k_cache;         // [num_blocks][num_kv_heads][16][head_dim]
  const uint8_t* v_cache;
  const int32_t* block_tables;    // [num_seqs][max_blocks_per_seq]
  const int32_t* context_lens;    // [num_seqs]
  const int32_t* query_start_loc; // [num_seqs + 1] or nullptr (decode)
  int num_seqs;
  int num_rows;
  int num_heads;
  int num_kv_heads;
  int group;                      // num_heads / num_kv_heads
  int max_blocks_per_seq;
  int num_blocks;
  int partition;                  // tokens per partition (multiple of 16)
  int max_parts;                  // partitions launched per row
  float q_scale;                  // softmax scale * log2(e) (* k_scale for E4M3)
  float v_scale;                  // 1, or v_scale for E4M3
  float* o_part;                  // [rows][num_heads][max_parts][head_dim] (split only)
  float* lse;                     // [rows][num_heads][max_parts], base-2 units (split only)
  uint32_t* errors;               // device error word or nullptr
  // Cascade decode (a prompt shared by a group of sequences is read once per
  // group) and the prefill kernel's options for its shared-prefix pass.
  // Zero / null for plain decode and prefill.
  const int32_t* prefix_lens;     // decode, merge: [num_seqs] shared prefix tokens of each
                                  // sequence (whole blocks); its partials come first
  const int32_t* seq_rows;        // prefill: block-table and context_lens row of each
                                  // sequence (null: the sequence itself)
  int prefix_chunk;               // keys per partial of the shared-prefix pass (multiple of 512)
  int non_causal;                 // prefill: every query sees all keys of its context
  int partial_out;                // prefill: write (o, lse) partials, one slot per key chunk
  // Draft-tree verification (prefill): per query row, bit j = the chunk's key
  // j is visible (its ancestors and itself); null = causal.
  const uint64_t* tree_mask;
  // Failure-detection test hook (zero in normal calls): the longest any
  // device-side wait of the launch may take (0: kWaitLimitNs), and a copy
  // the first producer of CTA 0 never issues (n > 0: its n-th tile copy,
  // counted from 1), so that the waits for that tile run out.
  unsigned long long wait_limit_ns;
  int skip_copy;
  // Prefill on E4M3 caches: per (query row, head) scale s of the split query
  // (q / s = hi + lo, both E4M3), [rows][num_heads]; null otherwise.
  const float* q8_scale;
};

// Limit of the launch's device-side waits.
__host__ __device__ inline unsigned long long wait_limit(const AttnParams& p) {
  return p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs;
}

// Applies and clears the armed test hook (pkv_debug_arm_wait_timeout), if any.
void take_debug_hook(AttnParams& p);

int launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int num_blocks, int src_dtype, int cache_dtype,
                             float k_scale, float v_scale, uint32_t* errors,
                             cudaStream_t stream);

// CUDA-core paged attention (any group size up to 16) plus the merge of
// partitions when p.max_parts > 1.  g_pad is the group size rounded up to a
// power of two.
int launch_paged_attention_simt(const AttnParams& p, int q_dtype, int kv_dtype, int head_dim,
                                int g_pad, cudaStream_t stream);

// Per-(q dtype, kv dtype) launchers, one translation unit each.
int launch_simt_f16_f16(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s);
int launch_simt_f16_e4m3(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s);
int launch_simt_bf16_bf16(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s);
int launch_simt_bf16_e4m3(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s);

// tcgen05 grouped-query decode (head_dim 128, 16-bit or E4M3 caches, 2..16
// heads per KV head, 512-token partitions, decode rows only).
bool tc_decode_supported(const AttnParams& p, int q_dtype, int kv_dtype, int head_dim);
// dependent: launched as a programmatic dependent of the launch before it on
// the stream, which it does not read; its CTAs may start while that grid ends
// and wait for it before they exit (so whatever waits for this grid also
// sees that one's writes).
int launch_paged_decode_tc(const AttnParams& p, int q_dtype, int kv_dtype, cudaStream_t stream,
                           bool dependent = false);

// tcgen05 chunked-prefill attention (head_dim 128, 16-bit caches, 128 % g == 0).
bool tc_prefill_supported(const AttnParams& p, int q_dtype, int kv_dtype, int head_dim);
int launch_prefill_tc(const AttnParams& p, int q_dtype, int total_q, cudaStream_t stream);
// Device bytes the E4M3-cache prefill needs for its split query (0 otherwise).
size_t prefill_q8_bytes(int total_q, int num_heads);
// The E4M3-cache prefill: splits q into the workspace, then launches the kernel.
int launch_prefill_tc_fp8(const AttnParams& p, int q_dtype, int total_q, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

// One launch for a mixed batch: pd describes the decode rows (as for
// launch_paged_decode_tc), pp the prefill chunks (as for launch_prefill_tc);
// the CTAs are split between the two (prefill_ctas > 0 fixes the chunks'
// share, 0 lets the kernel weigh the batch).  16-bit caches, group <= 8.
bool tc_mixed_supported(const AttnParams& pd, const AttnParams& pp, int q_dtype, int kv_dtype,
                        int head_dim);
int launch_mixed_tc(const AttnParams& pd, const AttnParams& pp, int q_dtype, int total_q,
                    int prefill_ctas, cudaStream_t stream);

// Host helpers (host_util.cu).
bool tmap_available();
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, bool bf16, uint32_t box_rows);
bool make_map_q3d(CUtensorMap* m, const void* base, uint64_t tokens, uint32_t heads, bool bf16,
                  uint32_t box_heads, uint32_t box_tokens);
bool make_map_e4m3(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows);
bool make_map_q3d_e4m3(CUtensorMap* m, const void* base, uint64_t tokens, uint32_t heads,
                       uint32_t box_heads, uint32_t box_tokens);
int sm_count();

int launch_lse_merge(const AttnParams& p, int q_dtype, int head_dim, cudaStream_t stream);

}  // namespace pkv
