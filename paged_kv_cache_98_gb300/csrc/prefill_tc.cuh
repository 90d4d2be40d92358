// Chunked-prefill paged attention on the tcgen05 tensor cores (head_dim 128,
// fp16/bf16 caches, group sizes dividing 128).
//
// Sources: "第32讲 … Prefill vs Decode …", §5.4 (a prompt is processed in
// chunks; each chunk's queries attend the paged prior context and, causally,
// the chunk itself) and §3.4 (query heads grouped on a KV head);
// devpress.csdn.net vLLM overview, "9、FlashAttention (3)/(4)" (query blocks
// against streamed key/value blocks, running max and sum of exponentials).
//
// A query tile is 128 rows, a row being a (query token, head of the group)
// pair, token-major, so that the g heads of a KV head share every K/V tile.
// Work item = (sequence, KV head, two consecutive query tiles a and b): each
// K/V tile brought into shared memory feeds both.  Per 128-key tile j:
//   S_x = Q_x K_j^T     tcgen05, M = 128 rows, N = 128 keys, fp32 in TMEM
//   softmax of tile x   warpgroup x (thread = row = TMEM lane): scores -> P,
//                       written back over S_x in TMEM as packed 16-bit pairs
//   O_x += P_x V_j      tcgen05 with A = P_x read from TMEM, B = V_j
// for x = a, b.  The two softmax warpgroups alternate with the MMAs: while
// warpgroup a turns S_a into P_a, the tensor pipe computes S_b, and the other
// way round.  The running max only moves (and O is rescaled in TMEM) when a
// row's tile max exceeds it by more than 8 in base-2 units; the final
// division by the row sum is exact.
//
// Shared-prefix mode (cascade decode): the "sequences" are groups of decode
// sequences sharing a prompt, their query rows are the members' single
// tokens, every query sees every key of the prompt (no causal mask), the
// prompt's block-table and length row is the group's first member, items are
// further split into 2048-key chunks, and each chunk writes normalised partial
// outputs and their log-sum-exps (merged later with the members' own keys).
// A group's members rarely fill more than one query tile, so in this mode both
// warpgroups take the same query tile and alternate key tiles (even / odd),
// each writing its own partial: the two softmaxes then overlap as they do for
// two query tiles.  The second query buffer is then not needed: the query
// tile sits in q[1] and q[0], right after the ring, becomes a fifth ring
// stage; and V tiles trail K tiles by one (K0, K1, V0, K2, V1, ...), the order
// the alternating MMAs take them in, so a V tile waiting for its softmax does
// not hold back the next score tile's K.
//
// Draft-tree mode (speculative verification): a chunk of at most 64 draft
// tokens whose queries each see the prior context and, of the chunk's own
// keys, only those in their row of a 64-bit ancestor mask.  When the prior
// context is shorter than kFewKeys a draft token may see only a handful of
// keys, where rounding its softmax weights to 16 bits does not average out:
// the rows of such chunks are recomputed in fp32 after the main loop, as the
// causal rows at the start of a prompt are.
//
// Warps: 0-3 softmax + epilogue of tile a, 4-7 of tile b, 8 TMEM owner + MMA
// issuer, 9-11 TMA producers.  A K/V tile is 16 boxes of 16 rows x 128 B (one
// per block and half); the boxes of each tile are spread over the three
// producer warps, since one warp issuing boxes of this size moves about 31
// GB/s per SM and three about 40.  Producer 0 also loads Q (one 3-D box per
// half) and the partial last block of V.

#ifndef PKV_PREFILL_TC_CUH
#define PKV_PREFILL_TC_CUH

#include <cuda.h>

#include <climits>
#include <cstddef>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace pkv {
namespace pre_tc {
namespace {

constexpr int kThreads = 384;
constexpr int kProducers = 3;  // warps 9..11
constexpr int kD = 128;
constexpr int kTileKeys = 128;
constexpr int kRowsM = 128;
constexpr int kStages = 4;     // ring stages (5 in shared-prefix mode: q[0] joins the ring)
constexpr int kMaxStages = 5;
constexpr int kStages8 = 8;    // E4M3 caches: tiles of 16 KB, eight in the same ring
constexpr int kRingBars = 8;   // barriers for the deepest ring
constexpr int kTileBytes = 128 * kD * 2;  // 32 KB: [2 halves][128 rows][128 B]
constexpr int kHalf = kTileBytes / 2;
constexpr int kTailBytes = kBlockSize * kD * 2;  // one block of V: [2 halves][16 rows][128 B]
constexpr int kMaxSeqs = 1024;
constexpr int kTmemCols = 512;  // S/P a, S/P b, O a, O b
constexpr uint32_t kColO = 256;
constexpr float kRescaleAt = 8.0f;
// E4M3 weights: P holds 16 w with w <= 2^4 (the running max moves once a tile
// exceeds it by 4), so P stays below E4M3's largest value (448) while weights
// down to 2^-13 keep a code.
constexpr float kRescaleAt8 = 4.0f;
constexpr float kPScale8 = 16.0f;
// Causal rows that see at most this many keys are recomputed in fp32 on the
// CUDA cores after the main loop: with so few keys the 16-bit rounding of the
// softmax weights (relative 2^-9 each) does not average out.
constexpr int kFewKeys = 32;
constexpr int kBeyond = INT_MIN;  // block past the context (the box reads zeros)

struct Smem {
  alignas(1024) uint8_t ring[kStages][kTileBytes];
  alignas(1024) uint8_t q[2][kTileBytes];  // must follow the ring (fifth stage)
  alignas(1024) uint8_t tail[kTailBytes];
  int seq_start[kMaxSeqs + 1];  // prefix of tile pairs per sequence
  int seq_qlen[kMaxSeqs];
  int seq_ctx[kMaxSeqs];
  int seq_q0[kMaxSeqs];
  int few_start[kMaxSeqs + 1];  // prefix of rows seeing at most kFewKeys keys
  int scan[kThreads / 32];
  int scan2[kThreads / 32];
  uint64_t full[kRingBars];
  uint64_t empty[kRingBars];
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t s_ready[2];  // per query tile
  uint64_t p_ready[2];
  uint64_t o_done[2];
  uint64_t o_free[2];
  uint64_t tail_full;
  uint64_t tail_free;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int seq, kvh, ctx, q0;
  int trow;          // block-table row of the sequence
  int t0[2], nt[2];  // first token (within the chunk) and tokens of tiles a, b (nt[1] = 0: none)
  int pos0[2];       // absolute position of each tile's first token (last key without mask)
  int kt0;           // first key tile of the item (key chunks in shared-prefix mode)
  int nkt[2];        // end (exclusive) of the key tiles each query tile attends in the item
  int nk;            // end of the item's key tiles (max of the two)
  int chunk;         // key chunk of the item (its partial slots)
  int first[2];      // first key tile of each warpgroup in the item
  int last[2];       // last key tile of each warpgroup (-1: none)
  int step;          // key tiles between a warpgroup's tiles: 1, or 2 (shared-prefix mode)
  int tail_step;     // 16-key MMA step of the last key tile holding a partial block, else -1
};

// Key chunks of a sequence: all its key tiles in one item, or (shared-prefix
// mode) prefix_chunk keys per item.
template <bool kAlt>
__device__ __forceinline__ int key_chunks(const AttnParams& p, int ctx) {
  if (!kAlt || p.prefix_chunk <= 0) return 1;
  const int tiles = (ctx + kTileKeys - 1) / kTileKeys, per = p.prefix_chunk / kTileKeys;
  return (tiles + per - 1) / per;
}

// kFP8: E4M3 caches, whose P.V MMAs take 32 keys per step (16 for 16-bit).
template <bool kAlt, bool kFP8 = false>
__device__ __forceinline__ bool next_item(const AttnParams& p, const Smem& sm, int& idx,
                                          int total, Item& it, int stride) {
  if (idx >= total) return false;
  const int k = idx;
  idx += stride;
  const int kvh = k % p.num_kv_heads;
  const int pair = k / p.num_kv_heads;
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.seq_start[mid] <= pair) lo = mid; else hi = mid - 1;
  }
  const int rpt = kRowsM / p.group;  // tokens per tile
  const int qlen = sm.seq_qlen[lo];
  it.seq = lo;
  it.kvh = kvh;
  it.ctx = sm.seq_ctx[lo];
  it.q0 = sm.seq_q0[lo];
  it.trow = p.seq_rows ? __ldg(p.seq_rows + lo) : lo;
  const int nch = key_chunks<kAlt>(p, it.ctx);
  const int npairs = (sm.seq_start[lo + 1] - sm.seq_start[lo]) / nch;
  const int in_seq = pair - sm.seq_start[lo];
  const int mp = npairs - 1 - in_seq / nch;  // longest pairs first
  constexpr bool alt = kAlt;  // one query tile, alternating key tiles
  it.chunk = in_seq % nch;
  it.kt0 = kAlt && p.prefix_chunk > 0 ? it.chunk * (p.prefix_chunk / kTileKeys) : 0;
  const int kt1 = kAlt && p.prefix_chunk > 0 ? it.kt0 + p.prefix_chunk / kTileKeys : INT_MAX;
  it.nk = 0;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    it.t0[x] = (alt ? mp : 2 * mp + x) * rpt;
    it.nt[x] = max(0, min(rpt, qlen - it.t0[x]));
    it.pos0[x] = kAlt ? it.ctx - 1 : it.ctx - qlen + it.t0[x];
    const int last = kAlt ? it.pos0[x] : it.pos0[x] + it.nt[x] - 1;
    it.nkt[x] = it.nt[x] > 0 ? min(kt1, last / kTileKeys + 1) : 0;
    it.nk = max(it.nk, it.nkt[x]);
  }
  const bool partial = (it.ctx & (kBlockSize - 1)) != 0;
  it.tail_step = partial && (it.ctx - 1) / kTileKeys == it.nk - 1
                     ? ((it.ctx - 1) % kTileKeys) / (kFP8 ? 2 * kBlockSize : kBlockSize)
                     : -1;
  it.step = alt ? 2 : 1;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    it.first[x] = it.kt0 + (alt ? x : 0);
    const int end = alt ? it.nk : it.nkt[x];
    it.last[x] = it.nt[x] > 0 && end > it.first[x]
                     ? it.first[x] + (end - 1 - it.first[x]) / it.step * it.step
                     : -1;
  }
  return true;
}

// Rows of a chunk (qlen queries after ctx - qlen prior tokens) recomputed in
// fp32: causal rows that see at most kFewKeys keys (positions below
// kFewKeys); in draft-tree mode every row of a chunk whose prior context is
// shorter than kFewKeys (a row then sees its prior and its ancestors only);
// none in shared-prefix mode.
template <bool kTree, bool kAlt>
__device__ __forceinline__ int few_rows(int qlen, int ctx) {
  if (kAlt) return 0;
  if (kTree) return ctx - qlen < kFewKeys ? qlen : 0;
  const int n = kFewKeys - (ctx - qlen);
  return n <= 0 ? 0 : (n < qlen ? n : qlen);
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         unsigned long long limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// All 128 threads of softmax warpgroup x agree on `ok` (named barrier 1 + x).
__device__ __forceinline__ bool all_group(bool ok, int x) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(1 + x)
      : "memory");
  return r != 0;
}

template <class QT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (std::is_same<QT, BF16>::value) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Softmax weights of 32 keys of a row (sv[0..31]) as 16 packed 16-bit pairs,
// with their sums added to the row's partial sums: x = s * qa - m on packed
// fp32 pairs (one rounding, as fmaf), 2^x on the MUFU.  Each pair's weights go
// to sums l2[c % 4], the same chains as unpacked code would use.
template <class QT>
__device__ __forceinline__ void exp_pairs(const float* sv, float qa, float m, float2* l2,
                                          float* pk) {
  const float2 qa2 = make_float2(qa, qa), nm2 = make_float2(-m, -m);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const float e0 = fast_exp2(fmaf(sv[2 * c], qa, -m)), e1 = fast_exp2(fmaf(sv[2 * c + 1], qa, -m));
    l2[c & 3] = __fadd2_rn(l2[c & 3], make_float2(e0, e1));
    pk[c] = __uint_as_float(pack2<QT>(e0, e1));
  }
}

// The same for E4M3 weights: 32 keys (sv[0..31]) as 8 columns of four E4M3
// codes of kPScale8 * 2^x, sums of the unrounded weights.
__device__ __forceinline__ void exp_quads8(const float* sv, float qa, float m, float2* l2,
                                           float* pk) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = fast_exp2(fmaf(sv[4 * c + i], qa, -m));
    l2[(2 * c) & 3] = __fadd2_rn(l2[(2 * c) & 3], make_float2(e[0], e[1]));
    l2[(2 * c + 1) & 3] = __fadd2_rn(l2[(2 * c + 1) & 3], make_float2(e[2], e[3]));
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(e[0] * kPScale8, e[1] * kPScale8), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(e[2] * kPScale8, e[3] * kPScale8), __NV_SATFINITE, __NV_E4M3);
    pk[c] = __uint_as_float(lo | (hi << 16));
  }
}

// D[tmem] (+)= A[tmem] * B[smem]^T, 16-bit operands: A is M lanes x K
// elements, two elements per 32-bit column (the lower half holds the even one).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The MMAs of one tile, from values passed in registers (nothing in the
// issue loop is read from memory, so consecutive MMAs issue back to back).
// Scores: S (128 rows x 128 keys, fp32 in TMEM at d) = Q K^T over head_dim
// 128, in K-steps of 16 elements within the two 64-element swizzle halves.
__device__ __forceinline__ void issue_scores(uint32_t d, uint64_t dq, uint64_t dk, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
    tc::mma_f16(d, dq + off, dk + off, idesc, kk > 0);
  }
}

// Output: O (at d) (+)= P (TMEM at a, 16 keys per 8 columns) V, 16 keys per
// step; step ts (if >= 0) takes its V rows from the tail buffer.
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t a, uint64_t dv, uint64_t dtail, int ts,
                                         uint32_t acc0, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kTileKeys / 16; ++kk) {
    const uint64_t b = kk == ts ? dtail : dv + (uint64_t)((kk * (kBlockSize * 128)) >> 4);
    mma_f16_tmem_a(d, a + kk * 8, b, idesc, acc0 | (kk != 0 ? 1u : 0u));
  }
}

// D[tmem] (+)= A[tmem] * B[smem]^T, 8-bit operands (kind::f8f6f4): A is M
// lanes x K elements, four elements per 32-bit column.
__device__ __forceinline__ void mma_f8_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// E4M3 caches.  Scores: S = Q_hi K^T + Q_lo K^T, with the query split per row
// as q / s = hi + lo (E4M3 each, [128 rows][128 B] apiece, lo 16 KB after hi)
// and K [128 keys][128 B]; K-steps of 32 dims.
__device__ __forceinline__ void issue_scores8(uint32_t d, uint64_t dq, uint64_t dk, uint32_t idesc) {
#pragma unroll
  for (int part = 0; part < 2; ++part) {
#pragma unroll
    for (int kk = 0; kk < kD / 32; ++kk)
      tc::mma_f8(d, dq + (uint64_t)((part * (kTileBytes / 2) + kk * 32) >> 4),
                 dk + (uint64_t)((kk * 32) >> 4), idesc, (part | kk) != 0);
  }
}

// O (+)= P V with P as E4M3 in TMEM (32 keys per 8 columns) and V [128 keys][128
// B] (MN-major, one swizzle atom wide), 32 keys per step; step ts (if >= 0)
// takes its V rows from the tail buffer.
__device__ __forceinline__ void issue_pv8(uint32_t d, uint32_t a, uint64_t dv, uint64_t dtail,
                                          int ts, uint32_t acc0, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kTileKeys / 32; ++kk) {
    const uint64_t b = kk == ts ? dtail : dv + (uint64_t)((kk * (32 * 128)) >> 4);
    mma_f8_tmem_a(d, a + kk * 8, b, idesc, acc0 | (kk != 0 ? 1u : 0u));
  }
}

// kTree: draft-tree mode (per-row ancestor masks over the chunk's keys);
// kAlt: shared-prefix mode (non-causal, key chunks, partial outputs)
// The rows that see few keys (few_rows), recomputed in fp32 from the caches
// (the plain online softmax over the keys in order, exp2f).  Four
// lanes share a row, 32 dimensions each: partial dot products summed across
// the four, then each lane's share of the output.  Unit u of F x H x 4 (F
// such rows): lane quarter u % 4, head (u / 4) % H, row (u / 4) / H.  Keys in
// a block outside the pool count as zero vectors (the main pass flags them).
// kFP8: E4M3 caches (codes decoded; k_scale is in q_scale, v_scale applied).
template <class QT, bool kTree, class SM, bool kFP8 = false>
__device__ __noinline__ void few_key_rows(const AttnParams& p, const SM& sm, int first,
                                          int stride) {
  constexpr int kElem = kFP8 ? 1 : 2;
  using T = typename QT::T;
  const int H = p.num_heads, S = p.num_seqs;
  const int lane = threadIdx.x & 31;
  const unsigned gmask = 0xFu << (lane & 28);
  const long long units = (long long)sm.few_start[S] * H * 4;
  for (long long u = first; u < units; u += stride) {
    const int quarter = (int)(u & 3);
    const long long ru = u >> 2;
    const int h = (int)(ru % H);
    const int f = (int)(ru / H);
    int lo = 0, hi = S - 1;  // largest s with few_start[s] <= f
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sm.few_start[mid] <= f) lo = mid; else hi = mid - 1;
    }
    const int i = f - sm.few_start[lo];
    const int prior = sm.seq_ctx[lo] - sm.seq_qlen[lo];
    const int pos = prior + i;  // causal: keys 0 .. pos
    // draft-tree mode: the prior keys, then the chunk keys in the row's mask
    const uint64_t tmask = kTree ? __ldg(p.tree_mask + sm.seq_q0[lo] + i) : 0ull;
    const int kend = kTree ? sm.seq_ctx[lo] : pos + 1;
    const int row = sm.seq_q0[lo] + i;
    const int kvh = h / p.group;
    const int trow = p.seq_rows ? __ldg(p.seq_rows + lo) : lo;
    float qf[32];
    const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                     ((size_t)row * H + h) * kD + quarter * 32);
#pragma unroll
    for (int c = 0; c < 4; ++c) to_float(__ldg(qp + c), qf + 8 * c, QT());
    float m = -INFINITY, l = 0.0f, acc[32];
#pragma unroll
    for (int d = 0; d < 32; ++d) acc[d] = 0.0f;
    for (int j = 0; j < kend; ++j) {
      if (kTree && j >= prior && !((tmask >> (j - prior)) & 1ull)) continue;
      const int blk = __ldg(p.block_tables + (size_t)trow * p.max_blocks_per_seq + j / kBlockSize);
      const bool bok = blk >= 0 && blk < p.num_blocks;
      const size_t off = ((((size_t)(bok ? blk : 0) * p.num_kv_heads + kvh) * kBlockSize +
                           j % kBlockSize) * kD + quarter * 32) * kElem;
      float kv[32];
      float dot = 0.0f;
      if (bok) {
        const uint4* kp = reinterpret_cast<const uint4*>(p.k_cache + off);
#pragma unroll
        for (int c = 0; c < 32 * kElem / 16; ++c) {
          if constexpr (kFP8) to_float(__ldg(kp + c), kv + 16 * c, E4M3());
          else to_float(__ldg(kp + c), kv + 8 * c, QT());
        }
#pragma unroll
        for (int d = 0; d < 32; ++d) dot = fmaf(qf[d], kv[d], dot);
      }
      dot += __shfl_xor_sync(gmask, dot, 1);
      dot += __shfl_xor_sync(gmask, dot, 2);
      const float sc = dot * p.q_scale;  // base-2 units
      if (sc > m) {
        const float a = exp2f(m - sc);
        l *= a;
#pragma unroll
        for (int d = 0; d < 32; ++d) acc[d] *= a;
        m = sc;
      }
      const float w = exp2f(sc - m);
      l += w;
      if (bok) {
        const uint4* vp = reinterpret_cast<const uint4*>(p.v_cache + off);
#pragma unroll
        for (int c = 0; c < 32 * kElem / 16; ++c) {
          if constexpr (kFP8) to_float(__ldg(vp + c), kv + 16 * c, E4M3());
          else to_float(__ldg(vp + c), kv + 8 * c, QT());
        }
#pragma unroll
        for (int d = 0; d < 32; ++d) acc[d] = fmaf(w, kv[d], acc[d]);
      }
    }
    const float inv = p.v_scale / l;
    uint4* op = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)row * H + h) * kD +
                                         quarter * 32);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 w;
      w.x = pack2<QT>(acc[8 * c + 0] * inv, acc[8 * c + 1] * inv);
      w.y = pack2<QT>(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv);
      w.z = pack2<QT>(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv);
      w.w = pack2<QT>(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv);
      op[c] = w;
    }
  }
}

// The kernel body, run as CTA `cta` of `ncta` that share the items.
// Barriers, tensor memory, and the per-sequence tables (query length,
// context, first query row, the prefix of work units, the prefix of rows
// recomputed in fp32) of a prefill launch; ends with the CTA synchronised.
template <bool kTree, bool kAlt>
__device__ __forceinline__ void prefill_setup(const AttnParams& p, Smem& sm,
                                              const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                              const CUtensorMap& tm_q) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group;
  // ---- set-up ---------------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingBars; ++s) {
      mbar_init(&sm.full[s], kProducers);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.s_ready[x], 1);
      mbar_init(&sm.p_ready[x], 1);
      mbar_init(&sm.o_done[x], 1);
      mbar_init(&sm.o_free[x], 1);
    }
    mbar_init(&sm.tail_full, 1);
    mbar_init(&sm.tail_free, 1);
    mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp >= 9 && lane == 0) {
    tc::prefetch_tmap(&tm_k);
    tc::prefetch_tmap(&tm_v);
    tc::prefetch_tmap(&tm_q);
  }
  if (warp == 8) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  {
    // per-sequence query length, context, first query row, and the prefix
    // of tile pairs
    const int S = p.num_seqs, tid = threadIdx.x;
    const int chunk = (S + kThreads - 1) / kThreads;
    const int cap = p.max_blocks_per_seq * kBlockSize;
    int local = 0, local2 = 0;
    for (int i = 0; i < chunk; ++i) {
      const int sq = tid * chunk + i;
      if (sq < S) {
        const int q0 = __ldg(p.query_start_loc + sq);
        int qlen = __ldg(p.query_start_loc + sq + 1) - q0;
        int ctx = __ldg(p.context_lens + (p.seq_rows ? __ldg(p.seq_rows + sq) : sq));
        if (ctx < 0 || ctx > cap || qlen < 0 || (!kAlt && qlen > ctx) || q0 < 0 ||
            q0 + qlen > p.num_rows || (kTree && qlen > 64)) {
          flag_error(p.errors, PKV_DEVERR_CONTEXT);
          ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
          qlen = qlen < 0 ? 0 : (!kAlt && qlen > ctx ? ctx : qlen);
          if (kTree && qlen > 64) qlen = 64;  // the mask covers 64 chunk keys
          if (q0 < 0 || q0 + qlen > p.num_rows) qlen = 0;
        }
        sm.seq_qlen[sq] = qlen;
        sm.seq_ctx[sq] = ctx;
        sm.seq_q0[sq] = q0;
        const int tiles = (qlen * g + kRowsM - 1) / kRowsM;
        const int units = kAlt ? tiles : (tiles + 1) / 2;
        local += ctx > 0 ? units * key_chunks<kAlt>(p, ctx) : 0;
        local2 += few_rows<kTree, kAlt>(qlen, ctx);
      }
    }
    int incl = local, incl2 = local2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      const int y2 = __shfl_up_sync(kFull, incl2, o);
      if (lane >= o) {
        incl += y;
        incl2 += y2;
      }
    }
    if (lane == 31) {
      sm.scan[warp] = incl;
      sm.scan2[warp] = incl2;
    }
    __syncthreads();
    int base = 0, base2 = 0;
    for (int w = 0; w < warp; ++w) {
      base += sm.scan[w];
      base2 += sm.scan2[w];
    }
    int run = base + incl - local, run2 = base2 + incl2 - local2;
    for (int i = 0; i < chunk; ++i) {
      const int sq = tid * chunk + i;
      if (sq < S) {
        sm.few_start[sq] = run2;
        run2 += few_rows<kTree, kAlt>(sm.seq_qlen[sq], sm.seq_ctx[sq]);
        sm.seq_start[sq] = run;
        const int c = sm.seq_ctx[sq];
        const int tiles = (sm.seq_qlen[sq] * g + kRowsM - 1) / kRowsM;
        run += c > 0 ? (kAlt ? tiles : (tiles + 1) / 2) * key_chunks<kAlt>(p, c) : 0;
      }
    }
    if (tid == kThreads - 1) {
      sm.seq_start[S] = base + incl;
      sm.few_start[S] = base2 + incl2;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

// The TMA producer warps (9..11) of a prefill launch: per work item the query
// tile(s), then per key tile its K boxes, the tail rows of V where the tile
// holds the context's partial last block, and its V boxes, into the ring.
template <bool kAlt, bool kFP8>
__device__ __forceinline__ void prefill_producers(const AttnParams& p, Smem& sm,
                                                  const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                                  const CUtensorMap& tm_q, int kv_rows, int cta,
                                                  int ncta, int total, volatile int* abort,
                                                  unsigned long long lim) {
  constexpr int kStageBytes = kFP8 ? kTileBytes / 2 : kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group;
  {
    // ---- TMA producers (ring order K0, V0, K1, V1, ...) -----------------------------------
    // Producer pw issues the boxes of blocks j with j % 3 == pw of every tile.
    const int pw = warp - 9;
    const int mine = (8 - pw + kProducers - 1) / kProducers;  // blocks per tile: 3, 3, 2
    const bool my_lane = (lane & 7) % kProducers == pw;
    constexpr bool alt = kAlt;  // shared-prefix mode
    constexpr int nst = kFP8 ? kStages8 : (alt ? kMaxStages : kStages);
    uint8_t* const ring = &sm.ring[0][0];  // stage 4 (shared-prefix mode) is q[0]
    int idx = cta;
    uint32_t pos = 0;
    int nitem = 0, ntail = 0;
    bool ok = true;
    Item x;
    // block id of block 32c + lane of the item's context (kBeyond past it);
    // read ahead of its use, checked when used
    auto fetch = [&](int c) -> int {
      const int b = 32 * c + lane;
      return b < (x.ctx + kBlockSize - 1) / kBlockSize
                 ? __ldg(p.block_tables + (size_t)x.trow * p.max_blocks_per_seq + b)
                 : kBeyond;
    };
    auto to_row = [&](int blk) -> int {
      if (blk == kBeyond) return kv_rows;
      if (blk >= 0 && blk < p.num_blocks) return (blk * p.num_kv_heads + x.kvh) * kBlockSize;
      flag_error(p.errors, PKV_DEVERR_BLOCK_ID);
      return kv_rows;
    };
    auto issue = [&](int t, int row, bool is_v) -> bool {
      const int st = pos % nst;
      // test hook: these boxes are never issued, so every wait for the tile runs out
      const bool skip = pw == 0 && cta == 0 && p.skip_copy > 0 && pos + 1 == (uint32_t)p.skip_copy;
      bool good = true;
      if (lane == 0) {
        if (pos >= (uint32_t)nst) good = wait_bar(&sm.empty[st], ((pos / nst) - 1) & 1, abort, lim);
        if (good && !skip) mbar_arrive_expect_tx(&sm.full[st], mine * (kStageBytes / 8));
      }
      if (!__shfl_sync(kFull, (int)good, 0)) return false;
      if (!skip && (lane >> 3) == (t & 3) && my_lane) {
        uint8_t* dst = ring + (size_t)st * kStageBytes + (lane & 7) * (kBlockSize * 128);
        const CUtensorMap* map = is_v ? &tm_v : &tm_k;
        tc::tma_load_2d(dst, map, 0, row, &sm.full[st]);
        if (!kFP8) tc::tma_load_2d(dst + kHalf, map, 64, row, &sm.full[st]);
      }
      __syncwarp();
      ++pos;
      return true;
    };
    // V rows of the partial last block, rows past the context as zeros, into
    // the tail buffer with the ring's swizzle (0 * NaN would poison the MMA)
    auto load_tail = [&]() -> bool {
      bool good = true;
      if (lane == 0 && ntail >= 1) good = wait_bar(&sm.tail_free, (ntail - 1) & 1, abort, lim);
      if (!__shfl_sync(kFull, (int)good, 0)) return false;
      if constexpr (kFP8) {
        // the 32 rows of the MMA step that holds the partial block, [32][128 B]
        const int key0 = (x.nk - 1) * kTileKeys + x.tail_step * 2 * kBlockSize;
#pragma unroll
        for (int i = 0; i < kTailBytes / 16 / 32; ++i) {
          const int c = lane + 32 * i;
          const int r = c >> 3, ch = c & 7;
          const int key = key0 + r;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (key < x.ctx) {
            const int blk =
                __ldg(p.block_tables + (size_t)x.trow * p.max_blocks_per_seq + key / kBlockSize);
            if (blk >= 0 && blk < p.num_blocks)
              v = __ldg(reinterpret_cast<const uint4*>(
                            p.v_cache + (((size_t)blk * p.num_kv_heads + x.kvh) * kBlockSize +
                                         (key & (kBlockSize - 1))) * kD) + ch);
          }
          *reinterpret_cast<uint4*>(&sm.tail[0] + r * 128 + ((ch ^ (r & 7)) << 4)) = v;
        }
      } else {
        const int bi = (x.ctx - 1) / kBlockSize;
        const int blk = __ldg(p.block_tables + (size_t)x.trow * p.max_blocks_per_seq + bi);
        const bool bok = blk >= 0 && blk < p.num_blocks;
        const uint8_t* src =
            p.v_cache + ((size_t)(bok ? blk : 0) * p.num_kv_heads + x.kvh) * kBlockSize * (kD * 2);
        const int rows = x.ctx - bi * kBlockSize;
#pragma unroll
        for (int i = 0; i < kTailBytes / 16 / 32; ++i) {
          const int c = lane + 32 * i;
          const int r = c >> 4, ch = c & 15;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (bok && r < rows) v = __ldg(reinterpret_cast<const uint4*>(src + r * (kD * 2)) + ch);
          *reinterpret_cast<uint4*>(&sm.tail[0] + (ch >> 3) * (kTailBytes / 2) + r * 128 +
                                    (((ch & 7) ^ (r & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tail_full);
      ++ntail;
      return true;
    };
    while (ok && next_item<kAlt, kFP8>(p, sm, idx, total, x, ncta)) {
      bool good = true;
      if (pw == 0 && lane == 0) {
        if (nitem >= 1) good = wait_bar(&sm.q_empty, (nitem - 1) & 1, abort, lim);
        if (good) {
          // shared-prefix mode: one query tile, in q[1]
          const int nq = alt ? 1 : (x.nt[1] > 0 ? 2 : 1);
          mbar_arrive_expect_tx(&sm.q_full, nq * kTileBytes);
          for (int qt = 0; qt < nq; ++qt) {
            uint8_t* dq = &sm.q[alt ? 1 : qt][0];
            const int tok = x.q0 + x.t0[qt];
            if constexpr (kFP8) {
              // E4M3 hi rows, then the lo rows (num_rows tokens further on)
              tc::tma_load_3d(dq, &tm_q, 0, x.kvh * g, tok, &sm.q_full);
              tc::tma_load_3d(dq + kHalf, &tm_q, 0, x.kvh * g, p.num_rows + tok, &sm.q_full);
            } else {
              tc::tma_load_3d(dq, &tm_q, 0, x.kvh * g, tok, &sm.q_full);
              tc::tma_load_3d(dq + kHalf, &tm_q, 64, x.kvh * g, tok, &sm.q_full);
            }
          }
        }
      }
      ok = __shfl_sync(kFull, (int)good, 0) != 0;
      // Block rows of the 32-block table chunks (4 key tiles each) the tiles
      // being issued fall in: two chunks cached (K runs a tile ahead of V in
      // shared-prefix mode), the next one read ahead.
      // (two named slots rather than an array: a runtime index would put them
      // in local memory)
      int rc_c0 = -1, rc_c1 = -1, rc_row0 = kv_rows, rc_row1 = kv_rows;
      int pre_c = x.kt0 >> 2, pre_raw = fetch(pre_c);
      auto row_for = [&](int t) -> int {
        const int c = t >> 2;
        if (rc_c0 == c) return rc_row0;
        if (rc_c1 == c) return rc_row1;
        const int r = to_row(pre_c == c ? pre_raw : fetch(c));
        if (rc_c0 < rc_c1) {  // replace the older chunk
          rc_c0 = c;
          rc_row0 = r;
        } else {
          rc_c1 = c;
          rc_row1 = r;
        }
        pre_c = c + 1;
        pre_raw = 4 * pre_c < x.nk ? fetch(pre_c) : kBeyond;
        return r;
      };
      if (!alt) {
        for (int t = x.kt0; ok && t < x.nk; ++t) {
          ok = issue(t, row_for(t), false);
          if (ok && pw == 0 && t == x.nk - 1 && x.tail_step >= 0) ok = load_tail();
          if (ok) ok = issue(t, row_for(t), true);
        }
      } else {
        // K0, K1, V0, K2, V1, ...
        ok = issue(x.kt0, row_for(x.kt0), false);
        for (int t = x.kt0; ok && t < x.nk; ++t) {
          if (t + 1 < x.nk) ok = issue(t + 1, row_for(t + 1), false);
          if (ok && pw == 0 && t == x.nk - 1 && x.tail_step >= 0) ok = load_tail();
          if (ok) ok = issue(t, row_for(t), true);
        }
      }
      ++nitem;
    }
    if (!ok && lane == 0) {
      flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      for (uint32_t y = pos > (uint32_t)nst ? pos - nst : 0; y < pos; ++y)
        mbar_wait(&sm.full[y % nst], (y / nst) & 1, 10000000ull);
    }
  }
}

// kFP8: E4M3 caches (not with kAlt).  K and V tiles are [128 keys][128 B] (16
// KB, one box per block), eight to the ring; the query comes split per row as
// q / s = hi + lo in E4M3 (rows of hi, then the same rows of lo, at token
// offset num_rows in tm_q; s in p.q8_scale); scores are S = (Q_hi + Q_lo) K^T
// on 8-bit MMAs, scaled by s and k_scale in the softmax; P is E4M3 of
// kPScale8 w in TMEM, O = P V on 8-bit MMAs, divided by kPScale8 l and
// multiplied by v_scale.
template <class QT, bool kTree, bool kAlt, bool kFP8 = false>
__device__ __forceinline__ void prefill_body(const AttnParams& p, const CUtensorMap& tm_k,
                                             const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                                             int kv_rows, int cta, int ncta, uint8_t* smem_raw) {
  static_assert(!(kFP8 && kAlt), "E4M3 caches have no shared-prefix mode");
  constexpr int kStageBytes = kFP8 ? kTileBytes / 2 : kTileBytes;
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t kAB = std::is_same<QT, BF16>::value ? 1u : 0u;
  // kind::f16 (0 f16, 1 bf16) or, on E4M3 caches, kind::f8f6f4 (0 = E4M3)
  constexpr uint32_t kIdescS = tc::idesc_f16(kFP8 ? 0u : kAB, 0, 0, 128, 128);
  constexpr uint32_t kIdescO = tc::idesc_f16(kFP8 ? 0u : kAB, 0, 1, 128, 128);
  const int g = p.group;

  prefill_setup<kTree, kAlt>(p, sm, tm_k, tm_v, tm_q);
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const unsigned long long lim = wait_limit(p);
  const int total = sm.seq_start[p.num_seqs] * p.num_kv_heads;

  if (warp >= 9) {
    prefill_producers<kAlt, kFP8>(p, sm, tm_k, tm_v, tm_q, kv_rows, cta, ncta, total, abort, lim);
  } else if (warp == 8) {
    // ---- MMA issuer --------------------------------------------------------------------
    // Order per item: S_a(0), S_b(0), then for each key tile t:
    //   P_a(t) V_t, S_a(t+1), P_b(t) V_t, S_b(t+1)
    // so each softmax warpgroup works while the tensor pipe serves the other.
    // Shared-prefix mode (warpgroup a even tiles, b odd): S_a(0), S_b(1), then
    //   P_a(t) V_t, S_a(t+2), P_b(t+1) V_t+1, S_b(t+3)   for t = 0, 2, ...
    // The whole warp runs the loop (waits, counters and descriptors stay warp-
    // uniform); one elected lane issues the MMAs and commits.
    {
      const bool leader = tc::elect_one();
      auto commit = [&](uint64_t* bar) {
        if (leader) tc::mma_commit(bar);
      };
      // every lane takes the same result
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __shfl_sync(kFull, (int)wait_bar(bar, parity, abort, lim), 0) != 0;
      };
      int idx = cta;
      uint32_t pos = 0;
      uint32_t np[2] = {0, 0};   // P tiles consumed per query tile
      uint32_t nit[2] = {0, 0};  // items per query tile
      int nitem = 0, ntail = 0;
      bool ok = true;
      Item x;
      const uint32_t qaddr[2] = {smem_u32(&sm.q[0][0]), smem_u32(&sm.q[1][0])};
      const uint32_t taddr = smem_u32(&sm.tail[0]);
      constexpr bool alt = kAlt;  // shared-prefix mode
      constexpr int nst = kFP8 ? kStages8 : (alt ? kMaxStages : kStages);
      auto acquire = [&](int& st) -> bool {
        st = pos % nst;
        const bool r = wait(&sm.full[st], (pos / nst) & 1);
        ++pos;
        if (r) tc::fence_after_sync();
        return r;
      };
      // Operand descriptors are built once; a step moves the start address
      // field (bytes / 16 in the low bits, no carry below 256 KB).
      // (shared-prefix mode: both warpgroups' scores from the query tile in q[1])
      const uint64_t dq[2] = {tc::smem_desc(qaddr[alt ? 1 : 0], 16, 1024, tc::kLayoutSw128),
                              tc::smem_desc(qaddr[1], 16, 1024, tc::kLayoutSw128)};
      const uint64_t dk0 = tc::smem_desc(smem_u32(&sm.ring[0][0]), 16, 1024, tc::kLayoutSw128);
      // V: 16-bit [2 halves][128 keys][128 B] (MN-major, the halves kHalf apart);
      // E4M3 [128 keys][128 B], one swizzle atom wide
      const uint64_t dv0 = tc::smem_desc(smem_u32(&sm.ring[0][0]), kFP8 ? 16 : kHalf, 1024,
                                         tc::kLayoutSw128);
      const uint64_t dtail =
          tc::smem_desc(taddr, kFP8 ? 16 : kTailBytes / 2, 1024, tc::kLayoutSw128);
      auto mma_s = [&](int qt, int st) {
        if (leader) {
          const uint64_t dk = dk0 + (uint64_t)(st * (kStageBytes >> 4));
          if constexpr (kFP8) issue_scores8(tmem + qt * 128, qt ? dq[1] : dq[0], dk, kIdescS);
          else issue_scores(tmem + qt * 128, qt ? dq[1] : dq[0], dk, kIdescS);
        }
        commit(&sm.s_ready[qt]);
      };
      auto mma_pv = [&](int qt, int st, int t) -> bool {
        if (!wait(&sm.p_ready[qt], np[qt] & 1)) return false;
        ++np[qt];
        if (t == x.first[qt] && nit[qt] >= 1 &&
            !wait(&sm.o_free[qt], (nit[qt] - 1) & 1))
          return false;  // the previous item's O has been read out
        tc::fence_after_sync();
        if (leader) {
          const uint64_t dv = dv0 + (uint64_t)(st * (kStageBytes >> 4));
          const int ts = t == x.nk - 1 ? x.tail_step : -1;
          if constexpr (kFP8)
            issue_pv8(tmem + kColO + qt * 128, tmem + qt * 128, dv, dtail, ts, t != x.first[qt],
                      kIdescO);
          else
            issue_pv(tmem + kColO + qt * 128, tmem + qt * 128, dv, dtail, ts, t != x.first[qt],
                     kIdescO);
        }
        if (t == x.last[qt]) commit(&sm.o_done[qt]);
        return true;
      };
      // K(t) into S of warpgroup qt, its stage released, and Q released after
      // the item's last S
      auto s_tile = [&](int qt, int t) -> bool {
        int st = 0;
        if (!acquire(st)) return false;
        mma_s(qt, st);
        commit(&sm.empty[st]);
        if (t == x.nk - 1) commit(&sm.q_empty);
        return true;
      };
      auto tail_wait = [&](int t) -> bool {
        if (t != x.nk - 1 || x.tail_step < 0) return true;
        const bool r = wait(&sm.tail_full, ntail & 1);
        if (r) tc::fence_after_sync();
        return r;
      };
      // shared-prefix mode: the two warpgroups on alternate key tiles; the
      // ring holds K0, K1, V0, K2, V1, K3, ... in the order taken here
      auto alternate = [&]() -> bool {
        int va = 0, vb = 0;
        const bool hb = x.last[1] >= 0;
        if (!s_tile(0, x.kt0)) return false;
        if (hb && !s_tile(1, x.kt0 + 1)) return false;
        for (int t = x.kt0; t < x.nk; t += 2) {
          if (!(acquire(va) && tail_wait(t) && mma_pv(0, va, t))) return false;
          commit(&sm.empty[va]);
          if (t + 2 < x.nk && !s_tile(0, t + 2)) return false;
          if (t + 1 < x.nk) {
            if (!(acquire(vb) && tail_wait(t + 1) && mma_pv(1, vb, t + 1))) return false;
            commit(&sm.empty[vb]);
            if (t + 3 < x.nk && !s_tile(1, t + 3)) return false;
          }
        }
        return true;
      };
      while (ok && next_item<kAlt, kFP8>(p, sm, idx, total, x, ncta)) {
        const bool ha = x.last[0] >= 0;
        const bool hb = x.last[1] >= 0;
        int kst = 0, vst = 0;
        ok = wait(&sm.q_full, nitem & 1);
        if (ok) tc::fence_after_sync();
        if (ok && x.step == 2) {
          ok = alternate();
        } else if (ok) {
          ok = acquire(kst);
          if (ok) {
            if (ha) mma_s(0, kst);
            if (hb) mma_s(1, kst);
            commit(&sm.empty[kst]);
            if (x.nk - x.kt0 == 1) commit(&sm.q_empty);
          }
          for (int t = x.kt0; ok && t < x.nk; ++t) {
            const bool more = t + 1 < x.nk;
            ok = acquire(vst);
            if (ok) ok = tail_wait(t);
            if (ok && t <= x.last[0]) ok = mma_pv(0, vst, t);
            if (ok && more) {
              ok = acquire(kst);
              if (ok && t + 1 <= x.last[0]) mma_s(0, kst);
            }
            if (ok && hb) ok = mma_pv(1, vst, t);
            if (!ok) break;
            commit(&sm.empty[vst]);
            if (more) {
              if (hb) mma_s(1, kst);
              commit(&sm.empty[kst]);
              if (t + 1 == x.nk - 1) commit(&sm.q_empty);
            }
          }
        }
        if (ok && x.tail_step >= 0) {
          commit(&sm.tail_free);
          ++ntail;
        }
        if (ha) ++nit[0];
        if (hb) ++nit[1];
        ++nitem;
      }
      if (!ok && leader) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, 100000000ull);
    }
  } else {
    // ---- softmax + epilogue: warpgroup qt = 0 (tile a) or 1 (tile b) --------------------
    const int qt = warp >> 2;
    const int tid = threadIdx.x & 127;  // row = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_off + qt * 128;
    const uint32_t o_col = tmem + lane_off + kColO + qt * 128;
    const float qs = p.q_scale;
    using OutT = typename QT::T;
    // Scores are scaled inside the exponent: exp2(s * |q_scale| - m) with m the
    // scaled running max.  A negative scale is folded in by negating the
    // scores; a zero scale is taken as 1e-30 (exp2 of s * 1e-30 rounds to 1).
    const bool neg = qs < 0.0f;
    const float qa = fmaxf(fabsf(qs), 1e-30f);
    int idx = cta;
    uint32_t ns = 0, nit = 0;  // S tiles and items of this query tile
    bool ok = true;
    Item x;
    while (ok && next_item<kAlt, kFP8>(p, sm, idx, total, x, ncta)) {
      // this warpgroup's fields of the item, in registers
      const int nt = qt ? x.nt[1] : x.nt[0];
      const int t0 = qt ? x.t0[1] : x.t0[0];
      const int pos0 = qt ? x.pos0[1] : x.pos0[0];
      const int first = qt ? x.first[1] : x.first[0];
      const int last = qt ? x.last[1] : x.last[0];
      const int step = x.step;
      const int tok = tid / g;  // token within the tile
      // rows past the tile's tokens compute on whatever Q holds there; their
      // output is never stored
      const bool valid = tid < nt * g;
      // shared-prefix mode: the warpgroup's partial slot of this key chunk
      const size_t head = (size_t)(x.q0 + t0 + tok) * p.num_heads + (size_t)x.kvh * g + tid % g;
      const int slot = 2 * x.chunk + qt;
      if (last < 0) {
        // no key tile for this warpgroup here (no tile b, or a one-tile chunk in
        // shared-prefix mode, whose empty partial then weighs nothing)
        if (kAlt && valid && nt > 0 && slot < p.max_parts) {
          p.lse[head * p.max_parts + slot] = -INFINITY;
          float4* z = reinterpret_cast<float4*>(p.o_part + (head * p.max_parts + slot) * kD);
#pragma unroll 4
          for (int i = 0; i < kD / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
      const int qpos = pos0 + (kAlt ? 0 : tok);
      // E4M3 caches: the row's query scale s (q / s = hi + lo) joins the score scale
      const float qa_r = kFP8 ? qa * (valid ? __ldg(p.q8_scale + head) : 1.0f) : qa;
      // draft-tree mode: the row's visible chunk keys, from the chunk's first position
      const int cbase = pos0 - t0;
      const uint64_t tmask = kTree && valid ? __ldg(p.tree_mask + x.q0 + t0 + tok) : 0ull;
      float m_run = -INFINITY;
      float2 l2[4];  // partial row sums (independent chains, packed pairs)
#pragma unroll
      for (int i = 0; i < 4; ++i) l2[i] = make_float2(0.0f, 0.0f);
      for (int t = first; t <= last; t += step, ++ns) {
        ok = all_group(wait_bar(&sm.s_ready[qt], ns & 1, abort, lim), qt);
        if (!ok) break;
        tc::fence_after_sync();
        float sv[kTileKeys];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_col + 32 * c, sv + 32 * c);
        tc::tmem_wait_ld();
        const int kbase = t * kTileKeys;
        if (neg) {
#pragma unroll
          for (int c = 0; c < kTileKeys; ++c) sv[c] = -sv[c];
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
        if (kTree && kbase + kTileKeys - 1 >= cbase) {
          // Chunk keys in this tile are visible when the row's mask has their
          // bit; keys before the chunk always are.  Visibility of the tile's
          // 128 keys as four 32-bit words: key 32 w + i is bit i of vw[w].
          const int nrel = x.ctx - cbase;  // keys in the chunk (<= 64)
          uint32_t vw[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int r0 = kbase + 32 * w - cbase;  // chunk index of the word's first key
            const uint64_t bits = r0 >= 0 ? (r0 < 64 ? tmask >> r0 : 0ull)
                                          : (-r0 < 64 ? tmask << -r0 : 0ull);
            const int lim = nrel - r0;  // keys i < lim are before the chunk's end
            const uint32_t keep = lim <= 0 ? 0u : (lim >= 32 ? ~0u : (1u << lim) - 1u);
            const uint32_t prior = r0 >= 0 ? 0u : (-r0 >= 32 ? ~0u : (1u << -r0) - 1u);
            vw[w] = prior | ((uint32_t)bits & keep);
          }
#pragma unroll
          for (int c = 0; c < kTileKeys; ++c) {
            sv[c] = (vw[c >> 5] >> (c & 31)) & 1u ? sv[c] : -INFINITY;
            mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
          }
        } else if (kbase + kTileKeys - 1 > pos0) {
          // the causal boundary crosses this tile: hidden keys become -inf
#pragma unroll
          for (int c = 0; c < kTileKeys; ++c) {
            sv[c] = kbase + c <= qpos ? sv[c] : -INFINITY;
            mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kTileKeys; c += 2)
            mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], sv[c], sv[c + 1]);
        }
        const float mt =
            fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * qa_r;
        // move the running max (and rescale O) only on a large increase; O is
        // complete up to tile t-1 (S of tile t was issued after its product)
        const bool need = mt > m_run + (kFP8 ? kRescaleAt8 : kRescaleAt);
        float alpha = 1.0f;
        if (need) {
          alpha = (t == first) ? 0.0f : fast_exp2(m_run - mt);
          m_run = mt;
#pragma unroll
          for (int i = 0; i < 4; ++i) l2[i] = __fmul2_rn(l2[i], make_float2(alpha, alpha));
        }
        if constexpr (kFP8) {
          // P over the first 32 columns of S: keys 4c .. 4c + 3 in column c
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float pk[16];
            exp_quads8(sv + h * 64, qa_r, m_run, l2, pk);
            exp_quads8(sv + h * 64 + 32, qa_r, m_run, l2, pk + 8);
            tc::tmem_st16(s_col + 16 * h, pk);
          }
        } else {
          // P over the first 64 columns of S: keys 2c and 2c+1 in column c
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float pk[16];
            exp_pairs<QT>(sv + h * 32, qa_r, m_run, l2, pk);
            tc::tmem_st16(s_col + 16 * h, pk);
          }
        }
        // the product of tile t adds onto O: rescale it first when a row's max moved
        if (t > first && __any_sync(kFull, need)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float ov[32];
            tc::tmem_ld32(o_col + 32 * c, ov);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] *= alpha;
            tc::tmem_st32(o_col + 32 * c, ov);
          }
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::named_sync(1 + qt, 128);
        if (tid == 0) mbar_arrive(&sm.p_ready[qt]);
      }
      if (!ok) break;
      // ---- epilogue: O / l --------------------------------------------------------------
      ok = all_group(wait_bar(&sm.o_done[qt], nit & 1, abort, lim), qt);
      if (!ok) break;
      tc::fence_after_sync();
      const float l = ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y)) +
                      ((l2[2].x + l2[2].y) + (l2[3].x + l2[3].y));
      // (E4M3: P held kPScale8 w, and V its codes: v_scale / (kPScale8 l))
      const float inv = valid ? (kFP8 ? p.v_scale / (kPScale8 * l) : 1.0f / l) : 0.0f;
      OutT* orow = static_cast<OutT*>(p.out) + head * kD;
      // shared-prefix mode: the normalised partial and its log-sum-exp (base 2,
      // scaled units), in the warpgroup's slot of the chunk
      const bool part = kAlt && slot < p.max_parts;
      float* prow = part ? p.o_part + (head * p.max_parts + slot) * kD : nullptr;
      if (part && valid) p.lse[head * p.max_parts + slot] = m_run + log2f(l);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float ov[32];
        tc::tmem_ld32(o_col + 32 * c, ov);
        tc::tmem_wait_ld();
        if (part) {
          if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              reinterpret_cast<float4*>(prow + 32 * c)[q4] =
                  make_float4(ov[q4 * 4] * inv, ov[q4 * 4 + 1] * inv, ov[q4 * 4 + 2] * inv,
                              ov[q4 * 4 + 3] * inv);
          }
        } else if (valid && !(!kAlt && (kTree ? cbase < kFewKeys : qpos < kFewKeys))) {
          // (rows of few keys are written by few_key_rows after the loop)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack2<QT>(ov[q4 * 8 + 0] * inv, ov[q4 * 8 + 1] * inv);
            w.y = pack2<QT>(ov[q4 * 8 + 2] * inv, ov[q4 * 8 + 3] * inv);
            w.z = pack2<QT>(ov[q4 * 8 + 4] * inv, ov[q4 * 8 + 5] * inv);
            w.w = pack2<QT>(ov[q4 * 8 + 6] * inv, ov[q4 * 8 + 7] * inv);
            reinterpret_cast<uint4*>(orow + 32 * c)[q4] = w;
          }
        }
      }
      tc::fence_before_sync();
      tc::named_sync(1 + qt, 128);
      if (tid == 0) mbar_arrive(&sm.o_free[qt]);
      ++nit;
    }
    if (!ok && tid == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
    if constexpr (!kAlt) {
      if (ok) few_key_rows<QT, kTree, Smem, kFP8>(p, sm, cta * 256 + qt * 128 + tid, ncta * 256);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace pre_tc
}  // namespace pkv

#endif  // PKV_PREFILL_TC_CUH
