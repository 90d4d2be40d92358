// Grouped-query paged decode attention on the tcgen05 tensor cores (head_dim
// 128, fp16/bf16 or E4M3 caches, 2..16 query heads per KV head).
//
// Sources: "第32讲 … Prefill vs Decode …", §3.4 (a KV head serves a group of
// query heads, so one K/V read feeds g query heads: a dense contraction of
// width g); openeuler.csdn.net PagedAttention notes, "Attention 计算时的 Block
// 映射（CUDA Kernel 伪代码）" (gather through the block table); devpress.csdn.net
// vLLM overview, "3、PagedAttention (3)" and "9、FlashAttention (4)" (per-block
// partials combined through max / sum of exponentials); "第34讲 …", §4.4 (E4M3
// KV cache).
//
// Work item = (sequence, KV head, 512-token partition); a persistent CTA per SM
// walks the items.  Per item, with the 512 keys cut into 128-key tiles:
//   S^T[128 keys x N] = K_tile[128 x 128] * Q^T        (tcgen05, M = 128)
//   softmax over the partition's keys per query head   (CUDA cores, from TMEM)
//   O^T[128 dims x 16] += V_tile^T[128 x 128] * P^T    (tcgen05, M = 128)
// The group's query heads are the N side of the MMAs ("swap-AB": the keys, not
// the few query heads, fill the M = 128 rows).
//
// Warp roles: 0-3 softmax + epilogue (thread = TMEM lane); 4 K producer (and
// the query on 16-bit caches); 5 TMEM owner + issuer of the score MMAs; 6 V
// producer; then on 16-bit caches 7 the tail loader (and 8-9 second K and V
// producers with at most 8 heads per group), on E4M3 caches 7-10 the query
// converters and tail loader.  On 16-bit caches one more warp (the last)
// issues the P.V MMAs: with the two products issued by separate warps, the K
// stream (scores of the next items) never waits behind a P.V product that
// waits for its softmax, and the V stream never waits behind K tiles still in
// flight (70B-GQA decode 0.209 -> 0.174 ms).  E4M3 caches keep one issuer,
// running S(i+1) then P.V(i): their softmax warps, not the streams, set the
// pace, and the extra warp's registers cost more than it returns.  One warp issuing 16-row boxes moves about 31 GB/s per SM, two
// per ring more, so the 16-bit rings' boxes are spread over two warps where
// registers allow (the E4M3 kernel is bound by its softmax warps, and second
// producers bought it nothing).  K and V tiles stream through separate
// shared-memory rings, so K tiles of later items keep arriving (and their
// scores keep being computed) while V tiles of the current item wait for its
// softmax.  TMEM holds two items.
//
// 16-bit tiles are [2 halves][128 rows][64 dims] with the 128-byte swizzle,
// filled by two 16-row TMA boxes per block; the same layout serves K as a
// K-major and V as an MN-major operand.  E4M3 tiles are [128 rows][128 dims]
// (one swizzle atom wide) and feed 8-bit MMAs (kind::f8f6f4, fp32
// accumulation) directly.  E4M3 scores: each query row is split as
// q / s = hi + lo with hi, lo in E4M3 and s = max|q| / 448 (together about 8
// significant bits, like bf16); hi rows and lo rows are the N columns of one
// MMA (fewer, wider MMAs issue faster) and the softmax adds them.  E4M3
// output: P is rounded to E4M3 after a 2^8 scale.  Shared-memory traffic stays at two bytes per byte read from HBM.
//
// The last block of a context is usually partial: rows past the last key hold
// whatever the pool had there.  Their weights are zero, but 0 * NaN is NaN
// inside the MMA, so the V rows of the MMA step holding that block are not
// taken from the ring: the tail loader copies them (rows past the context as
// zeros) into a small buffer of their own, which that one step reads instead.

#ifndef PKV_DECODE_TC_CUH
#define PKV_DECODE_TC_CUH

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "rows.cuh"
#include "tc.cuh"

namespace pkv {
namespace dec_tc {
namespace {

// producer warps per ring, and threads: the 16-bit, 16-head variant needs
// more registers than 320 threads leave
constexpr int tc_prod(bool g16, bool fp8) { return (fp8 || g16) ? 1 : 2; }
// (16-bit caches: one more warp issues the P.V MMAs, see decode_body)
constexpr bool tc_split_mma(bool fp8) { return !fp8; }
constexpr int tc_threads(bool g16, bool fp8) { return fp8 ? 352 : (g16 ? 288 : 352); }
constexpr int kTileKeys = 128;
constexpr int kPart = 512;
constexpr int kTilesPerPart = kPart / kTileKeys;
constexpr int kD = 128;
constexpr int kHalfBytes = kTileKeys * 128;       // 16 KB: 128 rows x 128 B
constexpr int kPGroupStride = (kPart / 8) * 128;  // 8 KB between 8-head groups of 16-bit P
constexpr int kMaxSeqs = 1024;                    // sequences per launch (host chunks more)
constexpr int kLenBits = 9;                       // seq_pack: start << 9 | (last length - 1)
constexpr int kTailBytes = 4096;                  // one MMA K step of V rows

// With at most 8 heads (G16 false) the 16-bit Q and P keep 8 rows and the
// descriptors' 8-row group stride is 0 (rows 8-15 alias rows 0-7; their
// products are never read); the E4M3 Q holds the hi rows, then the lo rows.
template <bool G16, bool FP8>
struct Layout {
  static constexpr int kTileBytes = FP8 ? kTileKeys * kD : kTileKeys * kD * 2;
  // 16-bit, at most 8 heads: three K and three V stages of 32 KB.  A clock64
  // trace of the 70B-GQA decode with two K and four V stages had the score
  // MMAs waiting ~1,100 SM cycles for every K tile (two stages cover one load
  // latency per two tiles) while the V stream kept up; 3 + 3 took the call
  // from 0.1715 to 0.1563 ms, 4 + 2 to 0.162 ms.
  static constexpr int kKStages = FP8 ? 4 : (G16 ? 2 : 3);
  static constexpr int kVStages = FP8 ? (G16 ? 7 : 8) : 3;
  static constexpr int kRows = G16 ? 16 : 8;               // query heads held (Q / P rows)
  static constexpr int kQRows = FP8 ? 2 * kRows : kRows;   // E4M3: hi rows, then lo rows
  static constexpr int kQHalf = kRows * 128;               // one 64-dim half of 16-bit Q
  static constexpr int kQBytes = FP8 ? kQRows * 128 : 2 * kQHalf;
  static constexpr int kQSbo = (FP8 || G16) ? 1024 : 0;
  static constexpr int kSCols = FP8 ? kQRows : 16;         // score columns per key tile
  static constexpr int kOCol = kTilesPerPart * kSCols;     // first O^T column of an item
  static constexpr int kBufCols = kOCol + 16 <= 128 ? 128 : 256;
  static constexpr int kTmemCols = 2 * kBufCols;           // two items in flight
  static constexpr int kPElem = FP8 ? 1 : 2;               // P bytes per element
  static constexpr int kPBytes = kRows * kPart * kPElem;
  static constexpr int kPSbo = G16 ? (kPart / (16 / kPElem)) * 128 : 0;
  // keys of one PV MMA step (16 for 16-bit, 32 for 8-bit operands)
  static constexpr int kStepKeys = FP8 ? 32 : 16;
  static constexpr int kRowBytes = FP8 ? kD : 2 * kD;      // one cache row
};

template <bool G16, bool FP8>
struct Smem {
  using L = Layout<G16, FP8>;
  // every TMA destination / MMA operand sits on a 1024-byte boundary (the
  // 128-byte swizzle repeats every 8 rows of 128 bytes)
  alignas(1024) uint8_t kring[L::kKStages][L::kTileBytes];
  alignas(1024) uint8_t vring[L::kVStages][L::kTileBytes];
  alignas(1024) uint8_t q[2][L::kQBytes];
  alignas(1024) uint8_t pmat[2][L::kPBytes];
  alignas(1024) uint8_t tail[2][kTailBytes];  // V rows of a partial block, alternating
  float stat_inv[2][16];  // v_scale / l per head
  float stat_lse[2][16];  // m + log2(l) per head
  float red_max[4][16];
  float red_sum[4][16];
  float qscale[4][16];    // E4M3: per-row scale s of the split query, by item % 4
  uint64_t kfull[L::kKStages];
  uint64_t kempty[L::kKStages];
  uint64_t vfull[L::kVStages];
  uint64_t vempty[L::kVStages];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_ready[2];
  uint64_t p_ready[2];
  uint64_t o_ready[2];
  uint64_t v_fixed[4];   // by (items with a partial block so far) % 4
  uint64_t tail_free[2];  // tail[i] read by the products: by that count % 2
  uint64_t qs_ready[4];  // by item % 4
  uint64_t s_free[2];    // the softmax has read S of buffer b (item % 2)
  uint64_t mma_done;
  uint64_t pv_done;
  // per sequence: first (sequence, partition) pair << 9 | (keys of its last
  // partition - 1); entry [S] holds the total << 9
  int seq_pack[kMaxSeqs + 1];
  int scan[12];  // per-warp partial sums
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int seq, kvh, part, nparts, n, ntiles;
  int kstart;  // first key of the sequence's own part (cascade decode: after its shared prefix)
  int slot;    // partial slot of this partition
};

// Context of sequence s, clamped to the block table and the launched partitions.
__device__ __forceinline__ int clamped_keys(const AttnParams& p, int s, bool report) {
  const int cap_t = p.max_blocks_per_seq * kBlockSize, cap_l = p.max_parts * kPart;
  const int cap = cap_t < cap_l ? cap_t : cap_l;
  int keys = __ldg(p.context_lens + s);
  if (keys < 0 || keys > cap) {
    if (report) flag_error(p.errors, PKV_DEVERR_CONTEXT);
    keys = keys < 0 ? 0 : cap;
  }
  return keys;
}

// Items are the non-empty (sequence, partition) pairs in sequence order, each
// split over the KV heads (KV head fastest): item k has KV head k % Hkv and
// pair k / Hkv.  Consecutive items read neighbouring (block, head) tiles.
//
// A CTA visits items first, first + stride, ...  Its cursor carries the next
// item's KV head and pair (advanced by adds, not divisions) and the sequence
// of the last one: pairs only grow, so the next sequence is found by stepping
// forward from there (a binary search for the first item, or when more than
// a few sequences lie in between).  A trace of the 70B-GQA decode had the
// divisions and the full binary search take ~1,250 SM cycles per item in
// every warp role.
struct Cursor {
  int k, kvh, pair, seq;  // next item, its KV head and pair; sequence of the last (-1: none)
  int dq, dr;             // stride = dq pairs + dr KV heads
};

__device__ __forceinline__ Cursor first_cursor(const AttnParams& p, int first, int stride) {
  Cursor c;
  c.k = first;
  c.kvh = first % p.num_kv_heads;
  c.pair = first / p.num_kv_heads;
  c.seq = -1;
  c.dq = stride / p.num_kv_heads;
  c.dr = stride % p.num_kv_heads;
  return c;
}

template <class SM>
__device__ __forceinline__ bool next_item(const AttnParams& p, const SM& sm, Cursor& c,
                                          int total, Item& it, int stride) {
  if (c.k >= total) return false;
  const int pair = c.pair;
  const int S = p.num_rows;
  // largest s with start(s) <= pair
  int lo = c.seq < 0 ? 0 : c.seq, hi = S - 1;
  int steps = c.seq < 0 ? 4 : 0;
  while (steps < 4 && lo < hi && (sm.seq_pack[lo + 1] >> kLenBits) <= pair) {
    ++lo;
    ++steps;
  }
  if (steps == 4) {
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((sm.seq_pack[mid] >> kLenBits) <= pair) lo = mid; else hi = mid - 1;
    }
  }
  c.seq = lo;
  const int pk = sm.seq_pack[lo];
  const int start = pk >> kLenBits;
  it.seq = lo;
  it.kvh = c.kvh;
  it.part = pair - start;
  it.nparts = (sm.seq_pack[lo + 1] >> kLenBits) - start;
  it.n = it.part == it.nparts - 1 ? (pk & ((1 << kLenBits) - 1)) + 1 : kPart;
  it.ntiles = (it.n + kTileKeys - 1) / kTileKeys;
  it.kstart = 0;
  it.slot = it.part;
  if (p.prefix_lens != nullptr) {  // cascade decode: the keys after the shared prefix
    it.kstart = cascade_prefix(p, lo, clamped_keys(p, lo, false), false);
    it.slot += cascade_slots(p, it.kstart);
  }
  c.k += stride;
  c.pair += c.dq;
  c.kvh += c.dr;
  if (c.kvh >= p.num_kv_heads) {
    c.kvh -= p.num_kv_heads;
    ++c.pair;
  }
  return true;
}

// Rows that see at most this many keys are recomputed in fp32 on the CUDA
// cores after the main loop: with so few keys the rounding of the softmax
// weights to the MMA's 16-bit (or E4M3) input does not average out.
constexpr int kFewKeys = 32;

// Decode rows with at most kFewKeys keys (one partition, no shared prefix):
// the plain online softmax over the keys in order, in fp32 with exp2f, from
// the caches (E4M3 codes decoded and scaled).  Four lanes share a (sequence,
// query head) row, 32 dimensions each; unit u of rows x heads x 4: lane
// quarter u % 4, head (u / 4) % H, sequence (u / 4) / H.  Keys in a block
// outside the pool count as zero vectors (the main pass flags them).
template <class QT, bool FP8, class SM>
__device__ __noinline__ void few_key_rows(const AttnParams& p, const SM& sm, int first,
                                          int stride) {
  using T = typename QT::T;
  const int H = p.num_heads;
  const int lane = threadIdx.x & 31;
  const unsigned gmask = 0xFu << (lane & 28);
  const long long units = (long long)p.num_rows * H * 4;
  for (long long u = first; u < units; u += stride) {
    const int quarter = (int)(u & 3);
    const long long ru = u >> 2;
    const int h = (int)(ru % H);
    const int s = (int)(ru / H);
    const int pk = sm.seq_pack[s];
    if ((sm.seq_pack[s + 1] >> kLenBits) - (pk >> kLenBits) != 1) continue;
    const int keys = (pk & ((1 << kLenBits) - 1)) + 1;
    if (keys > kFewKeys) continue;
    const int kvh = h / p.group;
    float qf[32];
    const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                     ((size_t)s * H + h) * kD + quarter * 32);
#pragma unroll
    for (int c = 0; c < 4; ++c) to_float(__ldg(qp + c), qf + 8 * c, QT());
    float m = -INFINITY, l = 0.0f, acc[32];
#pragma unroll
    for (int d = 0; d < 32; ++d) acc[d] = 0.0f;
    constexpr int kElem = FP8 ? 1 : 2;
    for (int j = 0; j < keys; ++j) {
      const int blk = __ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + j / kBlockSize);
      const bool bok = blk >= 0 && blk < p.num_blocks;
      const size_t off = ((((size_t)(bok ? blk : 0) * p.num_kv_heads + kvh) * kBlockSize +
                           j % kBlockSize) * kD + quarter * 32) * kElem;
      float kv[32];
      float dot = 0.0f;
      if (bok) {
        const uint4* kp = reinterpret_cast<const uint4*>(p.k_cache + off);
#pragma unroll
        for (int c = 0; c < 32 * kElem / 16; ++c) {
          if constexpr (FP8) to_float(__ldg(kp + c), kv + 16 * c, E4M3());
          else to_float(__ldg(kp + c), kv + 8 * c, QT());
        }
#pragma unroll
        for (int d = 0; d < 32; ++d) dot = fmaf(qf[d], kv[d], dot);
      }
      dot += __shfl_xor_sync(gmask, dot, 1);
      dot += __shfl_xor_sync(gmask, dot, 2);
      const float sc = dot * p.q_scale;  // base 2 (with k_scale for E4M3)
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
          if constexpr (FP8) to_float(__ldg(vp + c), kv + 16 * c, E4M3());
          else to_float(__ldg(vp + c), kv + 8 * c, QT());
        }
#pragma unroll
        for (int d = 0; d < 32; ++d) acc[d] = fmaf(w, kv[d], acc[d]);
      }
    }
    const float inv = p.v_scale / l;
    T* op = static_cast<T*>(p.out) + ((size_t)s * H + h) * kD + quarter * 32;
#pragma unroll
    for (int d = 0; d < 32; ++d) store_out(op + d, acc[d] * inv);
  }
}

// Wait bounded by limit_ns that also gives up when another role has aborted.
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

// All 128 threads of a group agree on `ok` (named barrier `id`).
template <int id>
__device__ __forceinline__ bool all_of_group(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(id)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool all_softmax(bool ok) { return all_of_group<1>(ok); }

// The kernel body, for kCta threads (at least tc_threads(G16, FP8); warps
// beyond the roles below only take part in the CTA-wide barriers), running
// as CTA `cta` of `ncta` that share the items.  The softmax computes kH heads
// (at least the group size): 4 for groups of at most 4 query heads, which
// halves its exponentials, shuffles and P stores against the 8 rows Q and P
// hold; the rows past kH keep the zeros P starts with.
template <class QT, bool G16, bool FP8, int kCta, int kH = (G16 ? 16 : 8)>
__device__ __forceinline__ void decode_body(const AttnParams& p, const CUtensorMap& tm_k,
                                            const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                                            int kv_rows, int cta, int ncta, uint8_t* smem_raw) {
  static_assert(kCta >= tc_threads(G16, FP8) && kCta <= 384 && kCta % 32 == 0, "CTA size");
  using L = Layout<G16, FP8>;
  static_assert(kH % 2 == 0 && kH <= L::kRows, "heads of the softmax");
  constexpr int KS = L::kKStages, VS = L::kVStages;
  constexpr int kThreads = kCta;
  constexpr int kProd = tc_prod(G16, FP8);
  // second producers of the K and V rings, and the P.V issuer (the last warp)
  constexpr int kWarpK1 = kProd == 2 ? 8 : -1;
  constexpr int kWarpV1 = kProd == 2 ? 9 : -1;
  constexpr int kWarpPV = tc_split_mma(FP8) ? tc_threads(G16, FP8) / 32 - 1 : -1;
  Smem<G16, FP8>& sm = *reinterpret_cast<Smem<G16, FP8>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // partials and a merge: several partitions, or cascade decode (prefix partials)
  const bool split = p.max_parts > 1 || p.prefix_lens != nullptr;
  // kind::f16 (16-bit operands: 0 f16, 1 bf16) or kind::f8f6f4 (0 = E4M3)
  constexpr uint32_t kAB = (!FP8 && std::is_same<QT, BF16>::value) ? 1u : 0u;
  constexpr uint32_t kIdescS = tc::idesc_f16(kAB, 0, 0, 128, L::kSCols);
  constexpr uint32_t kIdescO = tc::idesc_f16(kAB, 1, 0, 128, 16);

  // ---- set-up -------------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(&sm.kfull[s], kProd);
      mbar_init(&sm.kempty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&sm.vfull[s], kProd);
      mbar_init(&sm.vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_empty[b], 1);
      mbar_init(&sm.s_ready[b], 1);
      mbar_init(&sm.p_ready[b], 1);
      mbar_init(&sm.o_ready[b], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&sm.v_fixed[i], 1);
      mbar_init(&sm.qs_ready[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tail_free[i], 1);
      mbar_init(&sm.s_free[i], 1);
    }
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.pv_done, 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tc::prefetch_tmap(&tm_k);
    tc::prefetch_tmap(&tm_q);
  }
  if (warp == 6 && lane == 0) tc::prefetch_tmap(&tm_v);
  if (warp == 5) {
    tc::tmem_alloc(&sm.tmem_base, L::kTmemCols);
    tc::tmem_relinquish();
  }
  // per-sequence partition counts, their prefix, and the last partition's length
  {
    const int S = p.num_rows, tid = threadIdx.x;
    const int chunk = (S + kThreads - 1) / kThreads;
    // keys of the sequence's own part (cascade decode: those after its shared prefix)
    auto keys_of = [&](int sq, bool report) {
      const int keys = clamped_keys(p, sq, report);
      return keys - cascade_prefix(p, sq, keys, report);
    };
    int local = 0;
    for (int i = 0; i < chunk; ++i) {
      const int sq = tid * chunk + i;
      if (sq < S) local += (keys_of(sq, true) + kPart - 1) / kPart;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sm.scan[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += sm.scan[w];
    int run = base + incl - local;
    for (int i = 0; i < chunk; ++i) {
      const int sq = tid * chunk + i;
      if (sq < S) {
        const int keys = keys_of(sq, false);
        const int np = (keys + kPart - 1) / kPart;
        const int last = keys - (np > 0 ? np - 1 : 0) * kPart;  // 1..512 when np > 0
        sm.seq_pack[sq] = (run << kLenBits) | (np > 0 ? last - 1 : 0);
        run += np;
      }
    }
    if (tid == kThreads - 1) sm.seq_pack[S] = (base + incl) << kLenBits;
  }
  // P starts as zeros (every row a tile multiplies is rewritten per item)
  for (int i = threadIdx.x; i < 2 * L::kPBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(&sm.pmat[0][0])[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const unsigned long long lim = wait_limit(p);
  const int total = (sm.seq_pack[p.num_rows] >> kLenBits) * p.num_kv_heads;

  if (warp == 4 || warp == 6 || warp == kWarpK1 || warp == kWarpV1) {
    // ---- TMA producers: K (warp 4, and the 16-bit query) and V (warp 6) --------------------
    // Lane j reads the table entry of block j of an item's 32-block partition;
    // producer pi of a ring issues the boxes of blocks j with j % kProd == pi.
    const bool is_v = warp == 6 || warp == kWarpV1;
    const int pi = (warp == 4 || warp == 6) ? 0 : 1;
    const bool my_block = (lane & 7) % kProd == pi;
    const CUtensorMap* map = is_v ? &tm_v : &tm_k;
    uint64_t* full = is_v ? sm.vfull : sm.kfull;
    uint64_t* empty = is_v ? sm.vempty : sm.kempty;
    const uint32_t nst = is_v ? VS : KS;
    uint8_t* ring = is_v ? &sm.vring[0][0] : &sm.kring[0][0];
    Cursor idx = first_cursor(p, cta, ncta);
    uint32_t pos = 0;
    int it = 0;
    bool ok = true;
    // cache row of block `lane` of an item's partition in the [block][kv head][16]
    // row space (past the end, where the box reads zeros, when not part of it)
    auto block_row = [&](const Item& x) -> int {
      const int nblk = (x.n + kBlockSize - 1) / kBlockSize;
      int row = kv_rows;
      if (lane < nblk) {
        const int blk = __ldg(p.block_tables + (size_t)x.seq * p.max_blocks_per_seq +
                              x.kstart / kBlockSize + x.part * (kPart / kBlockSize) + lane);
        if (blk >= 0 && blk < p.num_blocks)
          row = (blk * p.num_kv_heads + x.kvh) * kBlockSize;
        else if (!is_v && pi == 0)
          flag_error(p.errors, PKV_DEVERR_BLOCK_ID);
      }
      return row;
    };
    auto load_q = [&](const Item& x, int k) -> bool {
      if constexpr (FP8) return true;  // the converter warps build the split query
      const int b = k & 1;
      bool good = true;
      if (lane == 0) {
        if (k >= 2) good = wait_bar(&sm.q_empty[b], ((k - 2) >> 1) & 1, abort, lim);
        if (good) {
          mbar_arrive_expect_tx(&sm.q_full[b], L::kQBytes);
          const int row = x.seq * p.num_heads + x.kvh * p.group;
          tc::tma_load_2d(&sm.q[b][0], &tm_q, 0, row, &sm.q_full[b]);
          tc::tma_load_2d(&sm.q[b][L::kQHalf], &tm_q, 64, row, &sm.q_full[b]);
        }
      }
      return __shfl_sync(kFull, (int)good, 0) != 0;
    };
    auto load_tiles = [&](const Item& x, int row) -> bool {
      for (int t = 0; t < x.ntiles; ++t, ++pos) {
        const uint32_t st = pos % nst;
        // test hook: this copy is never issued, so every wait for the tile runs out
        const bool skip = !is_v && pi == 0 && cta == 0 && p.skip_copy > 0 &&
                          pos + 1 == (uint32_t)p.skip_copy;
        bool good = true;
        if (lane == 0) {
          if (pos >= nst) good = wait_bar(&empty[st], ((pos / nst) - 1) & 1, abort, lim);
          if (good && !skip) mbar_arrive_expect_tx(&full[st], L::kTileBytes / kProd);
        }
        if (!__shfl_sync(kFull, (int)good, 0)) return false;
        if (!skip && (lane >> 3) == t && my_block) {
          uint8_t* dst = ring + (size_t)st * L::kTileBytes + (lane & 7) * (kBlockSize * 128);
          tc::tma_load_2d(dst, map, 0, row, &full[st]);
          if (!FP8) tc::tma_load_2d(dst + kHalfBytes, map, 64, row, &full[st]);
        }
        __syncwarp();
      }
      return true;
    };
    Item cur, nxt;
    bool has = next_item(p, sm, idx, total, cur, ncta);
    int row_cur = has ? block_row(cur) : kv_rows;
    while (has && ok) {
      // block rows are read one item ahead of their first use
      const bool has_n = next_item(p, sm, idx, total, nxt, ncta);
      const int row_nxt = has_n ? block_row(nxt) : kv_rows;
      if (!is_v && pi == 0) ok = load_q(cur, it);
      if (ok) ok = load_tiles(cur, row_cur);
      cur = nxt;
      row_cur = row_nxt;
      has = has_n;
      ++it;
    }
    if (!ok && lane == 0) {
      flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      // let copies already issued land before the CTA goes away
      for (uint32_t x = pos > nst ? pos - nst : 0; x < pos; ++x)
        mbar_wait(&full[x % nst], (x / nst) & 1, 10000000ull);
    }
  } else if (warp == 5 || warp == kWarpPV) {
    // ---- MMA issuers: scores (warp 5) and P.V products (the last warp) -------------------
    // Each warp runs its loop whole (waits, counters and descriptors stay warp-
    // uniform); one elected lane issues the MMAs and commits (a commit tracks
    // the MMAs of the thread that issued them).
    {
      const bool leader = tc::elect_one();
      auto commit = [&](uint64_t* bar) {
        if (leader) tc::mma_commit(bar);
      };
      // every lane takes the same result
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __shfl_sync(kFull, (int)wait_bar(bar, parity, abort, lim), 0) != 0;
      };
      Cursor idx = first_cursor(p, cta, ncta);
      uint32_t kpos = 0, vpos = 0;
      int ntail = 0;  // items with a partial last block so far
      Item cur;
      int it = 0;
      bool ok = true;
      auto mma_s = [&](const Item& x, int k) -> bool {
        const int b = k & 1;
        if (!wait(&sm.q_full[b], (k >> 1) & 1)) return false;
        const uint32_t qa = smem_u32(&sm.q[b][0]);
        for (int t = 0; t < x.ntiles; ++t, ++kpos) {
          const int st = kpos % KS;
          if (!wait(&sm.kfull[st], (kpos / KS) & 1)) return false;
          tc::fence_after_sync();
          const uint32_t ka = smem_u32(&sm.kring[st][0]);
          const uint32_t d = tmem + b * L::kBufCols + t * L::kSCols;
          if constexpr (FP8) {
            // S^T = K (E4M3, K-major) x [hi; lo]^T, 32 dims per instruction
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < kD / 32; ++kk)
                tc::mma_f8(d, tc::smem_desc(ka + kk * 32, 16, 1024, tc::kLayoutSw128),
                           tc::smem_desc(qa + kk * 32, 16, L::kQSbo, tc::kLayoutSw128), kIdescS,
                           kk > 0);
            }
          } else if (leader) {
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32u;
              tc::mma_f16(d,
                          tc::smem_desc(ka + (kk >> 2) * kHalfBytes + off, 16, 1024,
                                        tc::kLayoutSw128),
                          tc::smem_desc(qa + (kk >> 2) * L::kQHalf + off, 16, L::kQSbo,
                                        tc::kLayoutSw128),
                          kIdescS, kk > 0);
            }
          }
          commit(&sm.kempty[st]);
        }
        commit(&sm.s_ready[b]);
        commit(&sm.q_empty[b]);
        return true;
      };
      auto mma_pv = [&](const Item& x, int k) -> bool {
        const int b = k & 1;
        if (!wait(&sm.p_ready[b], (k >> 1) & 1)) return false;
        // the MMA step that holds the partial block reads the tail buffer
        const bool has_tail = (x.n & (kBlockSize - 1)) != 0;
        const int tail_step = has_tail ? ((x.n - 1) % kTileKeys) / L::kStepKeys : -1;
        const int slot = ntail & 1;
        if (has_tail) {
          if (!wait(&sm.v_fixed[ntail & 3], (ntail >> 2) & 1)) return false;
          ++ntail;
        }
        tc::fence_after_sync();
        const uint32_t pa = smem_u32(&sm.pmat[b][0]);
        const uint32_t ta = smem_u32(&sm.tail[slot][0]);
        const uint32_t d = tmem + b * L::kBufCols + L::kOCol;
        for (int t = 0; t < x.ntiles; ++t, ++vpos) {
          const int st = vpos % VS;
          if (!wait(&sm.vfull[st], (vpos / VS) & 1)) return false;
          tc::fence_after_sync();
          const uint32_t va = smem_u32(&sm.vring[st][0]);
          const int ts = t == x.ntiles - 1 ? tail_step : -1;
          if constexpr (FP8) {
            // V^T (E4M3, MN-major: 128 dims = one swizzle atom wide) x
            // P^T (E4M3, K-major), 32 keys per instruction
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < kTileKeys / 32; ++kk) {
                const uint32_t a = kk == ts ? ta : va + kk * (32 * 128);
                tc::mma_f8(d, tc::smem_desc(a, 16, 1024, tc::kLayoutSw128),
                           tc::smem_desc(pa + (t * (kTileKeys / 16) + kk * 2) * 128, 128,
                                         L::kPSbo, tc::kLayoutNone),
                           kIdescO, (t | kk) != 0);
              }
            }
          } else if (leader) {
            // V^T (MN-major: two 64-dim atoms) x P^T (K-major), 16 keys per instruction
#pragma unroll
            for (int kk = 0; kk < kTileKeys / 16; ++kk) {
              const bool tk = kk == ts;
              tc::mma_f16(d,
                          tc::smem_desc(tk ? ta : va + kk * (16 * 128),
                                        tk ? kTailBytes / 2 : kHalfBytes, 1024,
                                        tc::kLayoutSw128),
                          tc::smem_desc(pa + (t * (kTileKeys / 8) + kk * 2) * 128, 128, L::kPSbo,
                                        tc::kLayoutNone),
                          kIdescO, (t | kk) != 0);
            }
          }
          commit(&sm.vempty[st]);
        }
        if (has_tail) commit(&sm.tail_free[slot]);
        commit(&sm.o_ready[b]);
        return true;
      };
      if (!tc_split_mma(FP8)) {
        // one issuer: S(0), then per item i: S(i+1), P.V(i)
        Item nxt;
        bool has = next_item(p, sm, idx, total, cur, ncta);
        if (has) ok = mma_s(cur, 0);
        while (has && ok) {
          const bool has_n = next_item(p, sm, idx, total, nxt, ncta);
          if (has_n) ok = mma_s(nxt, it + 1);
          if (ok) ok = mma_pv(cur, it);
          cur = nxt;
          has = has_n;
          ++it;
        }
      } else if (warp == 5) {
        // S of item k goes to TMEM buffer k % 2 once the softmax has read item k - 2's
        while (ok && next_item(p, sm, idx, total, cur, ncta)) {
          const int b = it & 1;
          if (it >= 2) {
            ok = wait(&sm.s_free[b], ((it - 2) >> 1) & 1);
            if (ok) tc::fence_after_sync();
          }
          if (ok) ok = mma_s(cur, it);
          ++it;
        }
      } else {
        while (ok && next_item(p, sm, idx, total, cur, ncta)) ok = mma_pv(cur, it++);
      }
      if (!ok && leader) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      // no MMA of ours may still be running when TMEM is released
      uint64_t* done = warp == 5 ? &sm.mma_done : &sm.pv_done;
      commit(done);
      mbar_wait(done, 0, 100000000ull);
    }
  } else if (warp == 7 || (FP8 && warp >= 8 && warp <= 10)) {
    // ---- tail loader (16-bit: warp 7) / query converters + tail loader (E4M3: 7-10) -----
    constexpr int kGroup = FP8 ? 128 : 32;
    const int gtid = threadIdx.x - 224;
    Cursor idx = first_cursor(p, cta, ncta);
    int it = 0, ntail = 0;
    bool ok = true;
    auto group_all = [&](bool v) -> bool {
      if constexpr (FP8) return all_of_group<2>(v);
      return __all_sync(kFull, v) != 0;
    };
    auto group_sync = [&]() {
      if constexpr (FP8) tc::named_sync(2, 128);
      else __syncwarp();
    };
    // V rows of the MMA step that holds an item's partial last block, rows past
    // the context as zeros, into tail[m % 2] (m counts such items) with the
    // ring's swizzle.  The slot was last read by the products of item m - 2,
    // whose completion tail_free reports (item m's cannot complete before its
    // v_fixed, so the parity is unambiguous).
    auto load_tail = [&](const Item& x) -> bool {
      if ((x.n & (kBlockSize - 1)) == 0) return true;
      constexpr int kChunksPerRow = L::kRowBytes / 16;
      constexpr int kPer = L::kStepKeys * kChunksPerRow / kGroup;  // 16-B chunks per thread
      const int key0 = ((x.n - 1) / L::kStepKeys) * L::kStepKeys;  // first key of the step
      const uint8_t* cache = static_cast<const uint8_t*>(p.v_cache);
      uint4 v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int c = gtid + i * kGroup;
        const int key = key0 + c / kChunksPerRow;
        v[i] = make_uint4(0, 0, 0, 0);
        if (key < x.n) {
          const int blk = __ldg(p.block_tables + (size_t)x.seq * p.max_blocks_per_seq +
                                x.kstart / kBlockSize + x.part * (kPart / kBlockSize) +
                                key / kBlockSize);
          if (blk >= 0 && blk < p.num_blocks) {
            const size_t row =
                ((size_t)blk * p.num_kv_heads + x.kvh) * kBlockSize + (key & (kBlockSize - 1));
            v[i] = __ldg(reinterpret_cast<const uint4*>(cache + row * L::kRowBytes) +
                         c % kChunksPerRow);
          }
        }
      }
      const int m = ntail;
      bool good = true;
      if (m >= 2) good = wait_bar(&sm.tail_free[m & 1], ((m - 2) >> 1) & 1, abort, lim);
      if (!group_all(good)) return false;
      uint8_t* slot = &sm.tail[m & 1][0];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int c = gtid + i * kGroup;
        const int r = c / kChunksPerRow, ch = c % kChunksPerRow;
        // 16-bit: [2 halves][16 rows][128 B]; E4M3: [32 rows][128 B]
        const int half = ch >> 3, c8 = ch & 7;
        *reinterpret_cast<uint4*>(slot + half * (kTailBytes / 2) + r * 128 +
                                  ((c8 ^ (r & 7)) << 4)) = v[i];
      }
      fence_proxy_async_smem();
      group_sync();
      if (gtid == 0) mbar_arrive(&sm.v_fixed[m & 3]);
      ++ntail;
      return true;
    };
    if constexpr (FP8) {
      // Query rows split as q / s = hi + lo (E4M3 each, s = max|q| / 448), hi
      // rows 0..kRows-1 and lo rows kRows.., 128-byte swizzled (K-major).  The
      // rows of the next item are fetched into registers one item ahead.
      using QElem = typename QT::T;
      constexpr int TPR = 128 / L::kRows;  // threads per query row
      constexpr int EPT = kD / TPR;        // elements per thread: 8 or 16
      const int qr = gtid / TPR, qj = gtid % TPR;
      auto q_fetch = [&](const Item& x, uint4* buf) {
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) buf[i] = make_uint4(0, 0, 0, 0);
        if (qr < p.group) {
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const QElem*>(p.q) +
              ((size_t)x.seq * p.num_heads + (size_t)x.kvh * p.group + qr) * kD + qj * EPT);
#pragma unroll
          for (int i = 0; i < EPT / 8; ++i) buf[i] = __ldg(src + i);
        }
      };
      auto conv_q = [&](const uint4* buf, int k) -> bool {
        const int b = k & 1;
        bool good = true;
        if (k >= 2) good = wait_bar(&sm.q_empty[b], ((k - 2) >> 1) & 1, abort, lim);
        if (!all_of_group<2>(good)) return false;
        float f[EPT];
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) to_float(buf[i], f + 8 * i, QT());
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
        for (int o = TPR / 2; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;
        uint8_t hi[EPT], lo[EPT];
#pragma unroll
        for (int e = 0; e < EPT; e += 2) {
          const float x0 = f[e] * inv, x1 = f[e + 1] * inv;
          const __nv_fp8x2_storage_t h2 =
              __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
          __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3);
          const float2 hv = __half22float2(*reinterpret_cast<__half2*>(&hr));
          const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(
              make_float2(x0 - hv.x, x1 - hv.y), __NV_SATFINITE, __NV_E4M3);
          hi[e] = (uint8_t)(h2 & 0xff);
          hi[e + 1] = (uint8_t)(h2 >> 8);
          lo[e] = (uint8_t)(l2 & 0xff);
          lo[e + 1] = (uint8_t)(l2 >> 8);
        }
        const int d0 = qj * EPT;  // first dim of this thread
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int row = qr + part * L::kRows;
          const uint8_t* v = part ? lo : hi;
          uint8_t* dst = &sm.q[b][0] + row * 128 + (((d0 >> 4) ^ (row & 7)) * 16) + (d0 & 15);
          if constexpr (EPT == 16) {
            uint4 w;
            memcpy(&w, v, 16);
            *reinterpret_cast<uint4*>(dst) = w;
          } else {
            uint2 w;
            memcpy(&w, v, 8);
            *reinterpret_cast<uint2*>(dst) = w;
          }
        }
        if (qj == 0) sm.qscale[k & 3][qr] = sc;
        fence_proxy_async_smem();
        tc::named_sync(2, 128);
        if (gtid == 0) {
          mbar_arrive(&sm.q_full[b]);
          mbar_arrive(&sm.qs_ready[k & 3]);
        }
        return true;
      };
      uint4 qbuf[EPT / 8];
      Item cur, nxt, nxt2;
      bool has = next_item(p, sm, idx, total, cur, ncta);
      if (has) {
        q_fetch(cur, qbuf);
        ok = conv_q(qbuf, 0);
      }
      bool has_n = has && next_item(p, sm, idx, total, nxt, ncta);
      if (has_n) q_fetch(nxt, qbuf);
      while (has && ok) {
        const bool has_n2 = has_n && next_item(p, sm, idx, total, nxt2, ncta);
        if (has_n) {
          ok = conv_q(qbuf, it + 1);
          if (has_n2) q_fetch(nxt2, qbuf);
        }
        if (ok) ok = load_tail(cur);
        cur = nxt;
        nxt = nxt2;
        has = has_n;
        has_n = has_n2;
        ++it;
      }
    } else {
      Item cur;
      while (ok && next_item(p, sm, idx, total, cur, ncta)) ok = load_tail(cur);
    }
    if (!ok && gtid == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
  } else if (warp >= tc_threads(G16, FP8) / 32) {
    // not a role of this kernel: only the CTA-wide barriers below
  } else {
    // ---- softmax + epilogue (warps 0-3, thread = TMEM lane) ---------------------------
    const int tid = threadIdx.x;  // 0..127
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    using OutT = typename QT::T;
    const float qs = p.q_scale;
    // rows of sequences without context get zeros when no merge follows
    if (!split) {
      for (int s = cta; s < p.num_rows; s += ncta) {
        if ((sm.seq_pack[s + 1] >> kLenBits) == (sm.seq_pack[s] >> kLenBits)) {
          OutT* o = static_cast<OutT*>(p.out) + (size_t)s * p.num_heads * kD;
          for (int i = tid; i < p.num_heads * kD; i += 128) store_out(o + i, 0.0f);
        }
      }
    }
    Cursor idx = first_cursor(p, cta, ncta);
    Item cur, nxt, prev;
    int it = 0;
    bool has = next_item(p, sm, idx, total, cur, ncta);

    auto epilogue = [&](const Item& x, int k) -> bool {
      const int b = k & 1;
      const bool ok = all_softmax(wait_bar(&sm.o_ready[b], (k >> 1) & 1, abort, lim));
      if (!ok) return false;
      tc::fence_after_sync();
      float o[16];
      tc::tmem_ld16(tmem + lane_off + b * L::kBufCols + L::kOCol, o);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      const int d = tid;
      // one partition and no shared prefix: straight to out
      const bool direct = !split || (x.nparts == 1 && p.prefix_lens == nullptr);
      const size_t head0 = (size_t)x.seq * p.num_heads + (size_t)x.kvh * p.group;
      // rows with few keys (always direct) are recomputed after the loop
      const bool few = x.nparts == 1 && p.prefix_lens == nullptr && x.n <= kFewKeys;
      if (direct) {
        if (few) return true;
        OutT* dst = static_cast<OutT*>(p.out) + head0 * kD + d;
#pragma unroll
        for (int h = 0; h < kH; ++h)
          if (h < p.group) store_out(dst + h * kD, o[h] * sm.stat_inv[b][h]);
      } else if (x.slot < p.max_parts) {
        float* dst = p.o_part + (head0 * p.max_parts + x.slot) * kD + d;
        const size_t stride = (size_t)p.max_parts * kD;
#pragma unroll
        for (int h = 0; h < kH; ++h)
          if (h < p.group) dst[h * stride] = o[h] * sm.stat_inv[b][h];
        if (d < p.group) p.lse[(head0 + d) * p.max_parts + x.slot] = sm.stat_lse[b][d];
      }
      return true;
    };

    bool have_prev = false;
    bool ok = true;
    while (has) {
      const bool has_n = next_item(p, sm, idx, total, nxt, ncta);
      const int b = it & 1;
      ok = all_softmax(wait_bar(&sm.s_ready[b], (it >> 1) & 1, abort, lim));
      if (!ok) break;
      tc::fence_after_sync();
      float qsh[16];  // scale of each head's scores (base 2)
      if constexpr (FP8) {
        // per-row scales of the split query: published by the converters
        ok = all_softmax(wait_bar(&sm.qs_ready[it & 3], (it >> 2) & 1, abort, lim));
        if (!ok) break;
#pragma unroll
        for (int h = 0; h < kH; ++h) qsh[h] = qs * sm.qscale[it & 3][h];
      }
      float s[kTilesPerPart][16];
      if constexpr (FP8 && G16) {
        // 32 columns (16 hi, 16 lo) per tile: one tile at a time
#pragma unroll
        for (int t = 0; t < kTilesPerPart; ++t) {
          if (t < cur.ntiles) {
            float hl[32];
            tc::tmem_ld16(tmem + lane_off + b * L::kBufCols + t * L::kSCols, hl);
            tc::tmem_ld16(tmem + lane_off + b * L::kBufCols + t * L::kSCols + 16, hl + 16);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 16; ++h) s[t][h] = hl[h] + hl[h + 16];
          }
        }
      } else {
#pragma unroll
        for (int t = 0; t < kTilesPerPart; ++t)
          if (t < cur.ntiles)
            tc::tmem_ld16(tmem + lane_off + b * L::kBufCols + t * L::kSCols, s[t]);
        tc::tmem_wait_ld();
        if constexpr (FP8) {
          // columns 0-7 hi, 8-15 lo
#pragma unroll
          for (int t = 0; t < kTilesPerPart; ++t)
#pragma unroll
            for (int h = 0; h < kH; ++h) s[t][h] += s[t][h + 8];
        }
      }
      // Running max per head over this thread's keys, then over the CTA.  All
      // kRows heads are reduced and written to P: heads past the group hold
      // finite scores (the next group's queries, or zeros past the tensor) and
      // are never stored, and loops without per-head branches let the
      // independent shuffle chains of the heads interleave.
      float mx[16];
#pragma unroll
      for (int h = 0; h < kH; ++h) mx[h] = -INFINITY;
#pragma unroll
      for (int t = 0; t < kTilesPerPart; ++t) {
        const bool valid = t < cur.ntiles && t * kTileKeys + tid < cur.n;
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          s[t][h] = valid ? s[t][h] * (FP8 ? qsh[h] : qs) : -INFINITY;
          mx[h] = fmaxf(mx[h], s[t][h]);
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int h = 0; h < kH; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], o));
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kH; ++h) sm.red_max[warp][h] = mx[h];
      }
      tc::fence_before_sync();
      tc::named_sync(1, 128);
      if (tc_split_mma(FP8) && tid == 0) mbar_arrive(&sm.s_free[b]);  // S is in registers
      float sum[16];
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        sum[h] = 0.0f;
        mx[h] = fmaxf(fmaxf(sm.red_max[0][h], sm.red_max[1][h]),
                      fmaxf(sm.red_max[2][h], sm.red_max[3][h]));
      }
      // P[h][key] in the K-major core-matrix layout (8 keys per 16-byte row of a
      // 16-bit core matrix, 16 keys for E4M3), and its row sums
      uint8_t* pm = &sm.pmat[b][0];
#pragma unroll
      for (int t = 0; t < kTilesPerPart; ++t) {
        if (t < cur.ntiles) {
          const int key = t * kTileKeys + tid;
#pragma unroll
          for (int h = 0; h < kH; h += 2) {
            const float e0 = fast_exp2(s[t][h] - mx[h]);
            const float e1 = fast_exp2(s[t][h + 1] - mx[h + 1]);
            sum[h] += e0;
            sum[h + 1] += e1;
            if constexpr (FP8) {
              // E4M3 with a 2^8 scale (weights are <= 1)
              const __nv_fp8x2_storage_t q2 = __nv_cvt_float2_to_fp8x2(
                  make_float2(e0 * 256.0f, e1 * 256.0f), __NV_SATFINITE, __NV_E4M3);
              uint8_t* c8 = pm + (key >> 4) * 128 + (h >> 3) * L::kPSbo + (h & 7) * 16 + (key & 15);
              c8[0] = (uint8_t)(q2 & 0xffu);
              c8[16] = (uint8_t)(q2 >> 8);
            } else {
              uint32_t pr;
              if constexpr (std::is_same<QT, BF16>::value) {
                __nv_bfloat162 v2 = __floats2bfloat162_rn(e0, e1);
                pr = *reinterpret_cast<uint32_t*>(&v2);
              } else {
                __half2 v2 = __floats2half2_rn(e0, e1);
                pr = *reinterpret_cast<uint32_t*>(&v2);
              }
              uint8_t* c0 = pm + (key >> 3) * 128 + (key & 7) * 2 + (h >> 3) * kPGroupStride +
                            (h & 7) * 16;
              *reinterpret_cast<uint16_t*>(c0) = (uint16_t)(pr & 0xffffu);
              *reinterpret_cast<uint16_t*>(c0 + 16) = (uint16_t)(pr >> 16);
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int h = 0; h < kH; ++h) sum[h] += __shfl_xor_sync(kFull, sum[h], o);
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kH; ++h) sm.red_sum[warp][h] = sum[h];
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::named_sync(1, 128);  // P complete; every warp's partial sums written
      if (tid == 0) mbar_arrive(&sm.p_ready[b]);
      // read by this item's epilogue, after the next item's barriers
      if (tid < 16 && tid < p.group) {
        const float m = fmaxf(fmaxf(sm.red_max[0][tid], sm.red_max[1][tid]),
                              fmaxf(sm.red_max[2][tid], sm.red_max[3][tid]));
        const float l =
            (sm.red_sum[0][tid] + sm.red_sum[1][tid]) + (sm.red_sum[2][tid] + sm.red_sum[3][tid]);
        sm.stat_inv[b][tid] = p.v_scale / (FP8 ? l * 256.0f : l);
        sm.stat_lse[b][tid] = m + log2f(l);
      }

      if (have_prev) {
        ok = epilogue(prev, it - 1);
        if (!ok) break;
      }
      prev = cur;
      have_prev = true;
      cur = nxt;
      has = has_n;
      ++it;
    }
    if (ok && have_prev) ok = epilogue(prev, it - 1);
    if (!ok && tid == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
    if (ok && p.prefix_lens == nullptr) few_key_rows<QT, FP8>(p, sm, cta * 128 + tid, ncta * 128);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace
}  // namespace dec_tc
}  // namespace pkv

#endif  // PKV_DECODE_TC_CUH
