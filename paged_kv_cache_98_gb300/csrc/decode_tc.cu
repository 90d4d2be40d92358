// Grouped-query paged decode attention on the tcgen05 tensor cores (head_dim
// 128, fp16/bf16 caches, 2..16 query heads per KV head).
//
// Sources: "第32讲 … Prefill vs Decode …", §3.4 (a KV head serves a group of
// query heads, so one K/V read feeds g query heads: a dense contraction of
// width g); openeuler.csdn.net PagedAttention notes, "Attention 计算时的 Block
// 映射（CUDA Kernel 伪代码）" (gather through the block table); devpress.csdn.net
// vLLM overview, "3、PagedAttention (3)" and "9、FlashAttention (4)" (per-block
// partials combined through max / sum of exponentials).
//
// Work item = (sequence, KV head, 512-token partition); a persistent CTA per SM
// walks the items.  Per item, with the 512 keys cut into 128-key tiles:
//   S^T[128 keys x 16] = K_tile[128 x 128] * Q^T      (tcgen05, M=128, N=16)
//   softmax over the partition's keys per query head   (CUDA cores, from TMEM)
//   O^T[128 dims x 16] += V_tile^T[128 x 128] * P^T    (tcgen05, M=128, N=16)
// with the group's g query heads padded to N = 16 ("swap-AB": the keys, not
// the few query heads, fill the M = 128 rows of the MMA).
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue (one TMEM lane each),
// warp 4 TMA producer, warp 5 TMEM owner and MMA issuer.  The producer runs
// one item ahead (K tiles of item i+1 before V tiles of item i) so HBM keeps
// streaming while the softmax of item i runs; TMEM holds two items.
//
// Shared memory: a ring of 32 KB tile stages.  A tile is [2 halves][128 rows]
// [64 dims] with the 128-byte swizzle, filled by 16 two-dimensional TMA boxes
// of 16 rows (one per block and half); the same layout serves K as a K-major
// and V as an MN-major operand.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace pkv {
namespace {

// warps 0-3 softmax/epilogue, 4 producer, 5 MMA, then 6 the V-tail fixer
// (16-bit caches) or 6-9 the E4M3 -> fp16 converters (E4M3 caches)
constexpr int tc_threads(bool fp8) { return fp8 ? 320 : 224; }
constexpr int kTileKeys = 128;
constexpr int kPart = 512;
constexpr int kTilesPerPart = kPart / kTileKeys;
constexpr int kD = 128;
constexpr int kStageBytes = kTileKeys * kD * 2;  // 32 KB
constexpr int kHalfBytes = kStageBytes / 2;      // 16 KB: 128 rows x 128 B
constexpr int kPGroupStride = (kPart / 8) * 128;  // 8 KB between 8-head groups of P
constexpr int kTmemCols = 256;                    // two items x (64 S + 16 O, padded)
constexpr int kMaxSeqs = 1024;                    // sequences per launch (host chunks more)

// Layout for groups of up to 8 (G16 false) or up to 16 (G16 true) query heads.
// The MMA always has N = 16; with at most 8 heads, Q and P keep 8 rows and the
// descriptors' 8-row group stride is 0, so rows 8-15 alias rows 0-7 (their
// products are never read).  The shared memory saved buys a sixth ring stage.
// E4M3 caches: TMA brings raw 16 KB tiles into a deep ring.  K tiles are
// turned into fp16 by converter warps (E4M3 -> fp16 is exact) for the score
// MMA; V tiles feed the P V product directly as 8-bit operands
// (kind::f8f6f4), with P rounded to E4M3 after scaling by 2^8.  That keeps the
// shared-memory traffic near four bytes per byte read from HBM.
template <bool G16, bool FP8>
struct Layout {
  static constexpr int kStages = FP8 ? 2 : (G16 ? 5 : 6);        // 16-bit tiles (E4M3: K only)
  static constexpr int kRawStages = FP8 ? 8 : 1;                 // E4M3 tiles (K and V)
  static constexpr int kRawBytes = FP8 ? kTileKeys * kD : 16;
  static constexpr int kRows = G16 ? 16 : 8;               // Q / P rows held
  static constexpr int kQHalf = kRows * 128;               // one 64-dim half of Q
  static constexpr int kQBytes = 2 * kQHalf;
  static constexpr int kQSbo = G16 ? 1024 : 0;
  // P: 16-bit, or E4M3 (1 byte) on E4M3 caches; 8-head groups in the N direction
  static constexpr int kPElem = FP8 ? 1 : 2;
  static constexpr int kPBytes = kRows * kPart * kPElem;
  static constexpr int kPSbo = G16 ? (kPart / (16 / kPElem)) * 128 : 0;
};

template <bool G16, bool FP8>
struct Smem {
  using L = Layout<G16, FP8>;
  static constexpr int kStages = L::kStages;
  // every TMA destination / MMA operand sits on a 1024-byte boundary (the
  // 128-byte swizzle repeats every 8 rows of 128 bytes)
  alignas(1024) uint8_t ring[kStages][kStageBytes];
  alignas(1024) uint8_t raw[L::kRawStages][L::kRawBytes];
  alignas(1024) uint8_t q[2][L::kQBytes];
  alignas(1024) uint8_t pmat[2][L::kPBytes];
  float stat_inv[2][16];  // v_scale / l per head
  float stat_lse[2][16];  // m + log2(l) per head
  float red_max[4][16];
  float red_sum[4][16];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t raw_full[L::kRawStages];
  uint64_t raw_empty[L::kRawStages];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_ready[2];
  uint64_t p_ready[2];
  uint64_t o_ready[2];
  uint64_t v_fixed[2];
  uint64_t mma_done;
  int seq_keys[kMaxSeqs];       // clamped context length of each sequence
  int seq_start[kMaxSeqs + 1];  // prefix sum of partitions per sequence
  int scan[10];  // per-warp partial sums (up to 10 warps)
  uint32_t tmem_base;
  int abort;
  uint32_t issued;  // ring positions the producer has issued so far
};

struct Item {
  int seq, kvh, part, n, ntiles, keys;
};

// Items are the non-empty (sequence, partition) pairs in sequence order, each
// split over the KV heads (KV head fastest): item k has KV head k % Hkv and
// pair k / Hkv.  Consecutive items read neighbouring (block, head) tiles.
template <class SM>
__device__ __forceinline__ bool next_item(const AttnParams& p, const SM& sm, int& idx,
                                          int total, Item& it) {
  if (idx >= total) return false;
  const int k = idx;
  idx += gridDim.x;
  const int kvh = k % p.num_kv_heads;
  const int pair = k / p.num_kv_heads;
  int lo = 0, hi = p.num_rows - 1;  // largest s with seq_start[s] <= pair
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.seq_start[mid] <= pair) lo = mid; else hi = mid - 1;
  }
  const int keys = sm.seq_keys[lo];
  const int part = pair - sm.seq_start[lo];
  it.seq = lo;
  it.kvh = kvh;
  it.part = part;
  it.keys = keys;
  it.n = min(kPart, keys - part * kPart);
  it.ntiles = (it.n + kTileKeys - 1) / kTileKeys;
  return true;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > 2000000000ull) {
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

// 16 E4M3 values -> 16 fp16 values equal to value * 2^-8, exactly, as two
// 16-byte words.  Placing an E4M3 code's exponent and mantissa bits (e, m) at
// fp16 bits 10..13 and 7..9 gives 2^(e-15)(1 + m/8) for e > 0 and
// 2^-14 (m/8) for e = 0, i.e. the E4M3 value 2^(e-7)(1 + m/8) or 2^-6 (m/8)
// times 2^-8; the sign bit moves from bit 7 to bit 15.  (The NaN codes
// 0x7f / 0xff read as +-480 here; the cache write never produces them from
// finite inputs.)  The 2^8 is folded into the softmax and output scales.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t w) {
  return (w & 0x80008000u) | ((w >> 1) & 0x3F803F80u);
}
__device__ __forceinline__ void e4m3x16_to_f16(const uint4& v, uint4& lo, uint4& hi) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = e4m3x2_to_f16x2_scaled(__byte_perm(u[i], 0u, 0x1404));      // bytes 0, 1
    o[2 * i + 1] = e4m3x2_to_f16x2_scaled(__byte_perm(u[i], 0u, 0x3424));  // bytes 2, 3
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <class QT, bool G16, bool FP8>
__global__ void __launch_bounds__(tc_threads(FP8), 1)
    paged_decode_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_q, int kv_rows) {
  extern __shared__ uint8_t smem_raw[];
  using L = Layout<G16, FP8>;
  constexpr int kStages = L::kStages;
  constexpr int kRaw = L::kRawStages;
  constexpr int kQBytes = L::kQBytes;
  constexpr int kPBytes = L::kPBytes;
  constexpr int kTcThreads = tc_threads(FP8);
  // operands of the MMAs: fp16 when the cache is E4M3 (converted), else q's type
  using PT = typename std::conditional<FP8, F16, QT>::type;
  Smem<G16, FP8>& sm = *reinterpret_cast<Smem<G16, FP8>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool split = p.max_parts > 1;
  constexpr uint32_t kAB = std::is_same<PT, BF16>::value ? 1u : 0u;
  constexpr uint32_t kIdescS = tc::idesc_f16(kAB, 0, 0, 128, 16);
  constexpr uint32_t kIdescO = tc::idesc_f16(kAB, 1, 0, 128, 16);

  // ---- set-up -------------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kRaw; ++s) {
      mbar_init(&sm.raw_full[s], 1);
      mbar_init(&sm.raw_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_empty[b], 1);
      mbar_init(&sm.s_ready[b], 1);
      mbar_init(&sm.p_ready[b], 1);
      mbar_init(&sm.o_ready[b], 1);
      mbar_init(&sm.v_fixed[b], 1);
    }
    mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    sm.issued = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tc::prefetch_tmap(&tm_k);
    tc::prefetch_tmap(&tm_v);
    tc::prefetch_tmap(&tm_q);
  }
  if (warp == 5) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  // per-sequence key counts and the prefix of their partition counts
  {
    const int S = p.num_rows, tid = threadIdx.x;
    const int chunk = (S + kTcThreads - 1) / kTcThreads;
    const int cap_t = p.max_blocks_per_seq * kBlockSize, cap_l = p.max_parts * kPart;
    const int cap = cap_t < cap_l ? cap_t : cap_l;
    int local = 0;
    for (int i = 0; i < chunk; ++i) {
      const int sq = tid * chunk + i;
      if (sq < S) {
        int keys = __ldg(p.context_lens + sq);
        if (keys < 0 || keys > cap) {
          flag_error(p.errors, PKV_DEVERR_CONTEXT);
          keys = keys < 0 ? 0 : cap;
        }
        sm.seq_keys[sq] = keys;
        local += (keys + kPart - 1) / kPart;
      }
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
        sm.seq_start[sq] = run;
        run += (sm.seq_keys[sq] + kPart - 1) / kPart;
      }
    }
    if (tid == kTcThreads - 1) sm.seq_start[S] = base + incl;
  }
  // padded rows of P stay zero for the whole kernel
  for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(&sm.pmat[0][0])[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const int total = sm.seq_start[p.num_rows] * p.num_kv_heads;

  if (warp == 4) {
    // ---- TMA producer (whole warp: lane j owns block j of the partition) ----------------
    int idx = blockIdx.x;
    uint32_t pos = 0;
    Item cur, nxt;
    int it = 0;
    bool ok = true;
    auto load_q = [&](const Item& x, int k) -> bool {
      if constexpr (FP8) return true;  // the converter warps build fp16 Q
      const int b = k & 1;
      bool good = true;
      if (lane == 0) {
        if (k >= 2) good = wait_bar(&sm.q_empty[b], ((k - 2) >> 1) & 1, abort);
        if (good) {
          mbar_arrive_expect_tx(&sm.q_full[b], kQBytes);
          const int row = x.seq * p.num_heads + x.kvh * p.group;
          tc::tma_load_2d(&sm.q[b][0], &tm_q, 0, row, &sm.q_full[b]);
          tc::tma_load_2d(&sm.q[b][L::kQHalf], &tm_q, 64, row, &sm.q_full[b]);
        }
      }
      return __shfl_sync(kFull, (int)good, 0) != 0;
    };
    // Row of block `lane` of an item's partition in the [block][kv head][16]
    // row space of the caches (past the end when the block is not part of it).
    auto block_row = [&](const Item& x) -> int {
      const int nblk = (x.n + kBlockSize - 1) / kBlockSize;
      int row = kv_rows;
      if (lane < nblk) {
        const int blk = __ldg(p.block_tables + (size_t)x.seq * p.max_blocks_per_seq +
                              x.part * (kPart / kBlockSize) + lane);
        if (blk >= 0 && blk < p.num_blocks)
          row = (blk * p.num_kv_heads + x.kvh) * kBlockSize;
        else
          flag_error(p.errors, PKV_DEVERR_BLOCK_ID);
      }
      return row;
    };
    auto load_tiles = [&](const Item& x, int row, const CUtensorMap* map) -> bool {
      if constexpr (FP8) {
        // raw E4M3 tiles: one 16-row box of 128 bytes per block
        for (int t = 0; t < x.ntiles; ++t, ++pos) {
          const int st = pos % kRaw;
          bool good = true;
          if (lane == 0) {
            if (pos >= kRaw) good = wait_bar(&sm.raw_empty[st], ((pos / kRaw) - 1) & 1, abort);
            if (good) mbar_arrive_expect_tx(&sm.raw_full[st], kTileKeys * kD);
          }
          if (!__shfl_sync(kFull, (int)good, 0)) return false;
          if ((lane >> 3) == t)
            tc::tma_load_2d(&sm.raw[st][0] + (lane & 7) * (kBlockSize * 128), map, 0, row,
                            &sm.raw_full[st]);
          __syncwarp();
          if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&sm.issued) = pos + 1;
        }
        return true;
      }
      for (int t = 0; t < x.ntiles; ++t, ++pos) {
        const int st = pos % kStages;
        bool good = true;
        if (lane == 0) {
          if (pos >= kStages) good = wait_bar(&sm.empty[st], ((pos / kStages) - 1) & 1, abort);
          if (good) mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
        }
        if (!__shfl_sync(kFull, (int)good, 0)) return false;
        if ((lane >> 3) == t) {
          uint8_t* dst = &sm.ring[st][0] + (lane & 7) * (kBlockSize * 128);
          tc::tma_load_2d(dst, map, 0, row, &sm.full[st]);
          tc::tma_load_2d(dst + kHalfBytes, map, 64, row, &sm.full[st]);
        }
        __syncwarp();
        if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&sm.issued) = pos + 1;
      }
      return true;
    };
    Item nxt2;
    bool has = next_item(p, sm, idx, total, cur);
    int row_cur = has ? block_row(cur) : kv_rows;
    if (has) ok = load_q(cur, 0) && load_tiles(cur, row_cur, &tm_k);
    bool has_n = has && next_item(p, sm, idx, total, nxt);
    int row_nxt = has_n ? block_row(nxt) : kv_rows;
    while (has && ok) {
      // block rows are read one item ahead of their first use
      const bool has_n2 = has_n && next_item(p, sm, idx, total, nxt2);
      const int row_nxt2 = has_n2 ? block_row(nxt2) : kv_rows;
      if (has_n) ok = load_q(nxt, it + 1) && load_tiles(nxt, row_nxt, &tm_k);
      if (ok) ok = load_tiles(cur, row_cur, &tm_v);
      cur = nxt;
      row_cur = row_nxt;
      has = has_n;
      nxt = nxt2;
      row_nxt = row_nxt2;
      has_n = has_n2;
      ++it;
    }
    if (!ok && lane == 0) {
      flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      // let copies already issued land before the CTA goes away
      if constexpr (FP8) {
        for (uint32_t x = pos > kRaw ? pos - kRaw : 0; x < pos; ++x)
          mbar_wait(&sm.raw_full[x % kRaw], (x / kRaw) & 1, 10000000ull);
      } else {
        for (uint32_t x = pos > kStages ? pos - kStages : 0; x < pos; ++x)
          mbar_wait(&sm.full[x % kStages], (x / kStages) & 1, 10000000ull);
      }
    }
  } else if (warp == 5) {
    // ---- MMA issuer ---------------------------------------------------------------------
    if (lane == 0) {
      int idx = blockIdx.x;
      uint32_t pos = 0;   // position in the producer's ring
      uint32_t kpos = 0;  // E4M3: position in the converted-K ring
      Item cur, nxt;
      int it = 0;
      bool ok = true;
      auto mma_s = [&](const Item& x, int k) -> bool {
        const int b = k & 1;
        if (!wait_bar(&sm.q_full[b], (k >> 1) & 1, abort)) return false;
        const uint32_t qa = smem_u32(&sm.q[b][0]);
        for (int t = 0; t < x.ntiles; ++t, ++pos) {
          const uint32_t rp = FP8 ? kpos++ : pos;
          const int st = rp % kStages;
          if (!wait_bar(&sm.full[st], (rp / kStages) & 1, abort)) return false;
          tc::fence_after_sync();
          const uint32_t ka = smem_u32(&sm.ring[st][0]);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32u;
            const uint64_t a = tc::smem_desc(ka + (kk >> 2) * kHalfBytes + off, 16, 1024,
                                             tc::kLayoutSw128);
            const uint64_t bq = tc::smem_desc(qa + (kk >> 2) * L::kQHalf + off, 16, L::kQSbo,
                                              tc::kLayoutSw128);
            tc::mma_f16(tmem + b * 128 + t * 16, a, bq, kIdescS, kk > 0);
          }
          tc::mma_commit(&sm.empty[st]);
        }
        tc::mma_commit(&sm.s_ready[b]);
        tc::mma_commit(&sm.q_empty[b]);
        return true;
      };
      auto mma_pv = [&](const Item& x, int k) -> bool {
        const int b = k & 1;
        if (!wait_bar(&sm.p_ready[b], (k >> 1) & 1, abort)) return false;
        if (!wait_bar(&sm.v_fixed[b], (k >> 1) & 1, abort)) return false;
        tc::fence_after_sync();
        const uint32_t pa = smem_u32(&sm.pmat[b][0]);
        if constexpr (FP8) {
          // V^T (raw E4M3, MN-major: 128 dims = one swizzle atom wide) times
          // P^T (E4M3, K-major), 32 keys per instruction
          for (int t = 0; t < x.ntiles; ++t, ++pos) {
            const int st = pos % kRaw;
            if (!wait_bar(&sm.raw_full[st], (pos / kRaw) & 1, abort)) return false;
            tc::fence_after_sync();
            const uint32_t va = smem_u32(&sm.raw[st][0]);
#pragma unroll
            for (int kk = 0; kk < kTileKeys / 32; ++kk) {
              const uint64_t a = tc::smem_desc(va + kk * (32 * 128), 16, 1024, tc::kLayoutSw128);
              const uint64_t bp = tc::smem_desc(pa + (t * (kTileKeys / 16) + kk * 2) * 128, 128,
                                                L::kPSbo, tc::kLayoutNone);
              tc::mma_f8(tmem + b * 128 + 64, a, bp, kIdescO, (t | kk) != 0);
            }
            tc::mma_commit(&sm.raw_empty[st]);
          }
          tc::mma_commit(&sm.o_ready[b]);
          return true;
        }
        for (int t = 0; t < x.ntiles; ++t, ++pos) {
          const int st = pos % kStages;
          if (!wait_bar(&sm.full[st], (pos / kStages) & 1, abort)) return false;
          tc::fence_after_sync();
          const uint32_t va = smem_u32(&sm.ring[st][0]);
#pragma unroll
          for (int kk = 0; kk < kTileKeys / 16; ++kk) {
            const uint64_t a = tc::smem_desc(va + kk * (16 * 128), kHalfBytes, 1024,
                                             tc::kLayoutSw128);
            const uint64_t bp = tc::smem_desc(pa + (t * (kTileKeys / 8) + kk * 2) * 128, 128,
                                              L::kPSbo, tc::kLayoutNone);
            tc::mma_f16(tmem + b * 128 + 64, a, bp, kIdescO, (t | kk) != 0);
          }
          tc::mma_commit(&sm.empty[st]);
        }
        tc::mma_commit(&sm.o_ready[b]);
        return true;
      };
      bool has = next_item(p, sm, idx, total, cur);
      if (has) ok = mma_s(cur, 0);
      while (has && ok) {
        const bool has_n = next_item(p, sm, idx, total, nxt);
        if (has_n) ok = mma_s(nxt, it + 1);
        if (ok) ok = mma_pv(cur, it);
        cur = nxt;
        has = has_n;
        ++it;
      }
      if (!ok) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      // no MMA of ours may still be running when TMEM is released
      tc::mma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, 100000000ull);
    }
  } else if (FP8 && warp >= 6) {
    // ---- E4M3 -> fp16 converters (warps 6-9) ---------------------------------------------
    // Same item order as the producer: Q and K tiles of the next item, then V
    // tiles of the current one.  Thread = tile row (key).  V rows at or past
    // the partition's last key become zeros (0 * NaN would poison the MMA).
    const int ctid = threadIdx.x - 192;
    int idx = blockIdx.x;
    uint32_t pos = 0;
    Item cur, nxt;
    int it = 0;
    bool ok = true;
    using QElem = typename QT::T;
    auto conv_q = [&](const Item& x, int k) -> bool {
      const int b = k & 1;
      bool good = true;
      if (k >= 2) good = wait_bar(&sm.q_empty[b], ((k - 2) >> 1) & 1, abort);
      if (!all_of_group<2>(good)) return false;
      for (int i = ctid; i < L::kRows * 16; i += 128) {
        const int r = i >> 4, c = i & 15;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (r < p.group) {
          const QElem* src = static_cast<const QElem*>(p.q) +
                             ((size_t)x.seq * p.num_heads + (size_t)x.kvh * p.group + r) * kD;
          float f[8];
          to_float(__ldg(reinterpret_cast<const uint4*>(src) + c), f, QT());
          w = pack8(f, F16());
        }
        *reinterpret_cast<uint4*>(&sm.q[b][0] + (c >> 3) * L::kQHalf + r * 128 +
                                  (((c & 7) ^ (r & 7)) * 16)) = w;
      }
      fence_proxy_async_smem();
      tc::named_sync(2, 128);
      if (ctid == 0) mbar_arrive(&sm.q_full[b]);
      return true;
    };
    uint32_t kpos = 0;  // position in the converted-K ring
    // Waits until the producer has issued ring position x: every earlier use
    // of that stage is then complete, so a parity wait names this use.
    auto wait_issued = [&](uint32_t x) -> bool {
      const uint64_t t0 = globaltimer_ns();
      while (*reinterpret_cast<volatile uint32_t*>(&sm.issued) <= x) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > 2000000000ull) {
          *abort = 1;
          return false;
        }
      }
      return true;
    };
    auto conv_k = [&](const Item& x) -> bool {
      for (int t = 0; t < x.ntiles; ++t, ++pos, ++kpos) {
        const int rs = pos % kRaw, cs = kpos % kStages;
        bool good = wait_issued(pos) && wait_bar(&sm.raw_full[rs], (pos / kRaw) & 1, abort);
        if (good && kpos >= kStages)
          good = wait_bar(&sm.empty[cs], ((kpos / kStages) - 1) & 1, abort);
        if (!all_of_group<2>(good)) return false;
        const int r = ctid;
        const int sw = r & 7;
        const uint8_t* src = &sm.raw[rs][0] + r * 128;
        uint8_t* dst = &sm.ring[cs][0] + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16 E4M3 values = dims 16c .. 16c+15
          uint4 lo, hi;
          e4m3x16_to_f16(*reinterpret_cast<const uint4*>(src + ((c ^ sw) * 16)), lo, hi);
          uint8_t* h = dst + (c >> 2) * kHalfBytes;
          *reinterpret_cast<uint4*>(h + ((((2 * c) & 7) ^ sw) * 16)) = lo;
          *reinterpret_cast<uint4*>(h + ((((2 * c + 1) & 7) ^ sw) * 16)) = hi;
        }
        fence_proxy_async_smem();
        tc::named_sync(2, 128);
        if (ctid == 0) {
          mbar_arrive(&sm.full[cs]);
          mbar_arrive(&sm.raw_empty[rs]);
        }
      }
      return true;
    };
    // V tiles go to the MMA raw; rows at or past the partition's last key in a
    // partial last block hold whatever the pool had there and become zeros
    // (0 * NaN would poison the MMA).  At most one item ahead of the MMA.
    auto fix_v = [&](const Item& x, int k) -> bool {
      const int b = k & 1;
      const uint32_t last = pos + x.ntiles - 1;
      pos += x.ntiles;
      bool good = true;
      if (k >= 2) good = wait_bar(&sm.o_ready[b], ((k - 2) >> 1) & 1, abort);
      const int tail = x.n & (kBlockSize - 1);
      if (good && tail) good = wait_issued(last) && wait_bar(&sm.raw_full[last % kRaw], (last / kRaw) & 1, abort);
      if (!all_of_group<2>(good)) return false;
      if (tail) {
        const int jb = ((x.n - 1) % kTileKeys) / kBlockSize;
        const int rows = kBlockSize - tail;
        uint8_t* base = &sm.raw[last % kRaw][0] + (jb * kBlockSize + tail) * 128;
        for (int i = ctid; i < rows * 8; i += 128)
          reinterpret_cast<uint4*>(base + (i >> 3) * 128)[i & 7] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      tc::named_sync(2, 128);
      if (ctid == 0) mbar_arrive(&sm.v_fixed[b]);
      return true;
    };
    bool has = next_item(p, sm, idx, total, cur);
    if (has) ok = conv_q(cur, 0) && conv_k(cur);
    while (has && ok) {
      const bool has_n = next_item(p, sm, idx, total, nxt);
      if (has_n) ok = conv_q(nxt, it + 1) && conv_k(nxt);
      if (ok) ok = fix_v(cur, it);
      cur = nxt;
      has = has_n;
      ++it;
    }
    if (!ok && ctid == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
  } else if (!FP8 && warp == 6) {
    // ---- V tail fixer -------------------------------------------------------------------
    // V rows past the context in a partial last block hold whatever the pool
    // had there; their P is zero, but 0 * NaN is NaN inside the MMA, so they
    // are zeroed in shared memory once the tile has landed.  The MMA issuer
    // waits for this warp's signal before the item's V products.
    int idx = blockIdx.x;
    uint32_t pos = 0;
    Item cur, nxt;
    int it = 0;
    bool ok = true;
    bool has = next_item(p, sm, idx, total, cur);
    if (has) pos = cur.ntiles;
    while (has && ok) {
      const bool has_n = next_item(p, sm, idx, total, nxt);
      const int b = it & 1;
      // ring position of this item's last V tile (the producer's order: K of
      // the next item, then V of this one)
      if (has_n) pos += nxt.ntiles;
      const uint32_t v_last = pos + cur.ntiles - 1;
      pos += cur.ntiles;
      bool good = true;
      if (lane == 0) {
        // at most one item ahead of the MMA issuer: item it-2 has been multiplied
        if (it >= 2) good = wait_bar(&sm.o_ready[b], ((it - 2) >> 1) & 1, abort);
      }
      const int tail = cur.n & (kBlockSize - 1);
      if (good && tail && lane == 0) {
        // Once the producer has issued position v_last, every earlier use of
        // that stage has completed, so the parity below names this use.
        const uint64_t t0 = globaltimer_ns();
        while (*reinterpret_cast<volatile uint32_t*>(&sm.issued) <= v_last) {
          if (*abort || globaltimer_ns() - t0 > 2000000000ull) {
            *abort = 1;
            good = false;
            break;
          }
        }
        if (good) good = wait_bar(&sm.full[v_last % kStages], (v_last / kStages) & 1, abort);
      }
      ok = __shfl_sync(kFull, (int)good, 0) != 0;
      if (!ok) break;
      if (tail) {
        const int jb = ((cur.n - 1) % kTileKeys) / kBlockSize;  // block within the tile
        const int rows = kBlockSize - tail;
        uint8_t* base = &sm.ring[v_last % kStages][0] + (jb * kBlockSize + tail) * 128;
        for (int i = lane; i < rows * 2 * 8; i += 32) {
          const int half = i / (rows * 8), r = (i / 8) % rows, c = i % 8;
          reinterpret_cast<uint4*>(base + half * kHalfBytes + r * 128)[c] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.v_fixed[b]);
      cur = nxt;
      has = has_n;
      ++it;
    }
    if (!ok && lane == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
  } else {
    // ---- softmax + epilogue (warps 0-3, thread = TMEM lane) ---------------------------
    const int tid = threadIdx.x;  // 0..127
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    using OutT = typename QT::T;
    const float qs = p.q_scale;
    // rows of sequences without context get zeros when no merge follows
    if (!split) {
      for (int s = blockIdx.x; s < p.num_rows; s += gridDim.x) {
        if (sm.seq_keys[s] == 0) {
          OutT* o = static_cast<OutT*>(p.out) + (size_t)s * p.num_heads * kD;
          for (int i = tid; i < p.num_heads * kD; i += 128) store_out(o + i, 0.0f);
        }
      }
    }
    int idx = blockIdx.x;
    Item cur, nxt, prev;
    int it = 0;
    bool has = next_item(p, sm, idx, total, cur);

    auto epilogue = [&](const Item& x, int k) -> bool {
      const int b = k & 1;
      const bool ok = all_softmax(wait_bar(&sm.o_ready[b], (k >> 1) & 1, abort));
      if (!ok) return false;
      tc::fence_after_sync();
      float o[16];
      tc::tmem_ld16(tmem + lane_off + b * 128 + 64, o);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      const int d = tid;
      const int nparts = (x.keys + kPart - 1) / kPart;
      const bool direct = !split || nparts == 1;
      const size_t head0 = (size_t)x.seq * p.num_heads + (size_t)x.kvh * p.group;
      if (direct) {
        OutT* dst = static_cast<OutT*>(p.out) + head0 * kD + d;
#pragma unroll
        for (int h = 0; h < L::kRows; ++h)
          if (h < p.group) store_out(dst + h * kD, o[h] * sm.stat_inv[b][h]);
      } else {
        float* dst = p.o_part + (head0 * p.max_parts + x.part) * kD + d;
        const size_t stride = (size_t)p.max_parts * kD;
#pragma unroll
        for (int h = 0; h < L::kRows; ++h)
          if (h < p.group) dst[h * stride] = o[h] * sm.stat_inv[b][h];
        if (d < p.group) p.lse[(head0 + d) * p.max_parts + x.part] = sm.stat_lse[b][d];
      }
      return true;
    };

    bool have_prev = false;
    bool ok = true;
    while (has) {
      const bool has_n = next_item(p, sm, idx, total, nxt);
      const int b = it & 1;
      ok = all_softmax(wait_bar(&sm.s_ready[b], (it >> 1) & 1, abort));
      if (!ok) break;
      tc::fence_after_sync();
      float s[kTilesPerPart][16];
#pragma unroll
      for (int t = 0; t < kTilesPerPart; ++t)
        if (t < cur.ntiles) tc::tmem_ld16(tmem + lane_off + b * 128 + t * 16, s[t]);
      tc::tmem_wait_ld();
      // running max per head over this thread's keys, then over the CTA
      float mx[16];
#pragma unroll
      for (int h = 0; h < L::kRows; ++h) mx[h] = -INFINITY;
#pragma unroll
      for (int t = 0; t < kTilesPerPart; ++t) {
        const bool valid = t < cur.ntiles && t * kTileKeys + tid < cur.n;
#pragma unroll
        for (int h = 0; h < L::kRows; ++h) {
          s[t][h] = valid ? s[t][h] * qs : -INFINITY;
          mx[h] = fmaxf(mx[h], s[t][h]);
        }
      }
#pragma unroll
      for (int h = 0; h < L::kRows; ++h) {
        if (h < p.group) {
#pragma unroll
          for (int o = 16; o; o >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], o));
          if (lane == 0) sm.red_max[warp][h] = mx[h];
        }
      }
      tc::named_sync(1, 128);
      float sum[16];
#pragma unroll
      for (int h = 0; h < L::kRows; ++h) {
        sum[h] = 0.0f;
        if (h < p.group)
          mx[h] = fmaxf(fmaxf(sm.red_max[0][h], sm.red_max[1][h]),
                        fmaxf(sm.red_max[2][h], sm.red_max[3][h]));
      }
      // P[h][key] in the K-major core-matrix layout, and its row sums
      uint8_t* pm = &sm.pmat[b][0];
#pragma unroll
      for (int t = 0; t < kTilesPerPart; ++t) {
        if (t < cur.ntiles) {
          const int key = t * kTileKeys + tid;
          uint8_t* col = pm + (key >> 3) * 128 + (key & 7) * 2;
#pragma unroll
          for (int h = 0; h < L::kRows; h += 2) {
            if (h < p.group) {
              const float e0 = fast_exp2(s[t][h] - mx[h]);
              const float e1 = h + 1 < p.group ? fast_exp2(s[t][h + 1] - mx[h + 1]) : 0.0f;
              sum[h] += e0;
              sum[h + 1] += e1;
              if constexpr (FP8) {
                // E4M3 with a 2^8 scale (weights are <= 1), core matrices of 16 keys
                const __nv_fp8x2_storage_t q2 =
                    __nv_cvt_float2_to_fp8x2(make_float2(e0 * 256.0f, e1 * 256.0f),
                                             __NV_SATFINITE, __NV_E4M3);
                uint8_t* c8 = pm + (key >> 4) * 128 + (h >> 3) * L::kPSbo + (h & 7) * 16 + (key & 15);
                c8[0] = (uint8_t)(q2 & 0xffu);
                if (h + 1 < p.group) c8[16] = (uint8_t)(q2 >> 8);
                continue;
              }
              uint32_t pr;
              if constexpr (std::is_same<PT, BF16>::value) {
                __nv_bfloat162 v2 = __floats2bfloat162_rn(e0, e1);
                pr = *reinterpret_cast<uint32_t*>(&v2);
              } else {
                __half2 v2 = __floats2half2_rn(e0, e1);
                pr = *reinterpret_cast<uint32_t*>(&v2);
              }
              uint8_t* c0 = col + (h >> 3) * kPGroupStride + (h & 7) * 16;
              *reinterpret_cast<uint16_t*>(c0) = (uint16_t)(pr & 0xffffu);
              if (h + 1 < p.group) *reinterpret_cast<uint16_t*>(c0 + 16) = (uint16_t)(pr >> 16);
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < L::kRows; ++h) {
        if (h < p.group) {
#pragma unroll
          for (int o = 16; o; o >>= 1) sum[h] += __shfl_xor_sync(kFull, sum[h], o);
          if (lane == 0) sm.red_sum[warp][h] = sum[h];
        }
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
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host side ---------------------------------------------------------------------------
template <class QT, bool G16, bool FP8>
int launch_tc_typed(const AttnParams& p, cudaStream_t stream) {
  const bool bf16 = std::is_same<QT, BF16>::value;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv;
  const bool maps = FP8 ? make_map_e4m3(&tk, p.k_cache, kv_rows, 16) &&
                              make_map_e4m3(&tv, p.v_cache, kv_rows, 16)
                        : make_map_2d(&tk, p.k_cache, kv_rows, bf16, 16) &&
                              make_map_2d(&tv, p.v_cache, kv_rows, bf16, 16);
  if (!maps) return PKV_ERR_CUDA;
  using SM = Smem<G16, FP8>;
  const size_t smem = sizeof(SM) + 1024;
  static_assert(sizeof(SM) + 1024 <= 232448, "shared memory budget of one CTA");
  static_assert(offsetof(SM, ring) % 1024 == 0 && offsetof(SM, raw) % 1024 == 0 &&
                    offsetof(SM, q) % 1024 == 0 && offsetof(SM, pmat) % 1024 == 0 &&
                    kStageBytes % 1024 == 0 && Layout<G16, FP8>::kQHalf % 1024 == 0,
                "swizzled buffers must start on 1024-byte boundaries");
  auto kern = paged_decode_tc_kernel<QT, G16, FP8>;
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
    if (FP8) c.q_scale *= 256.0f;  // the converted K tiles hold value * 2^-8
    c.num_rows = p.num_rows - r0 < kMaxSeqs ? p.num_rows - r0 : kMaxSeqs;
    c.num_seqs = c.num_rows;
    const size_t head0 = (size_t)r0 * p.num_heads;
    c.out = static_cast<OutT*>(p.out) + head0 * kD;
    c.q = static_cast<const OutT*>(p.q) + head0 * kD;
    c.block_tables = p.block_tables + (size_t)r0 * p.max_blocks_per_seq;
    c.context_lens = p.context_lens + r0;
    if (p.lse) {
      c.lse = p.lse + head0 * p.max_parts;
      c.o_part = p.o_part + head0 * p.max_parts * kD;
    }
    CUtensorMap tq;  // read by TMA on 16-bit caches, unused (converted Q) on E4M3
    if (!make_map_2d(&tq, c.q, (uint64_t)c.num_rows * p.num_heads, bf16,
                     Layout<G16, FP8>::kRows))
      return PKV_ERR_CUDA;
    const long long items = (long long)c.num_rows * p.num_kv_heads * p.max_parts;
    int grid = sm_count();
    if (items < grid) grid = (int)items;
    if (grid < 1) grid = 1;
    kern<<<grid, tc_threads(FP8), smem, stream>>>(c, tk, tv, tq, (int)kv_rows);
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
  return tmap_available();
}

int launch_paged_decode_tc(const AttnParams& p, int q_dtype, int kv_dtype, cudaStream_t stream) {
  const bool g16 = p.group > 8;
  if (kv_dtype == PKV_FP8_E4M3) {
    if (q_dtype == PKV_BF16)
      return g16 ? launch_tc_typed<BF16, true, true>(p, stream)
                 : launch_tc_typed<BF16, false, true>(p, stream);
    return g16 ? launch_tc_typed<F16, true, true>(p, stream)
               : launch_tc_typed<F16, false, true>(p, stream);
  }
  if (q_dtype == PKV_BF16)
    return g16 ? launch_tc_typed<BF16, true, false>(p, stream)
               : launch_tc_typed<BF16, false, false>(p, stream);
  return g16 ? launch_tc_typed<F16, true, false>(p, stream)
             : launch_tc_typed<F16, false, false>(p, stream);
}

}  // namespace pkv
