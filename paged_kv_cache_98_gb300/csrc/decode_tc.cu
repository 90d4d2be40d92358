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

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace pkv {
namespace {

constexpr int kTcThreads = 224;
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
template <bool G16>
struct Layout {
  static constexpr int kStages = G16 ? 5 : 6;
  static constexpr int kRows = G16 ? 16 : 8;               // Q / P rows held
  static constexpr int kQHalf = kRows * 128;               // one 64-dim half of Q
  static constexpr int kQBytes = 2 * kQHalf;
  static constexpr int kQSbo = G16 ? 1024 : 0;
  static constexpr int kPBytes = kRows * kPart * 2;
  static constexpr int kPSbo = G16 ? kPGroupStride : 0;
};

template <bool G16>
struct Smem {
  static constexpr int kStages = Layout<G16>::kStages;
  uint8_t ring[kStages][kStageBytes];
  uint8_t q[2][Layout<G16>::kQBytes];
  uint8_t pmat[2][Layout<G16>::kPBytes];
  float stat_m[2][16];
  float stat_l[2][16];
  float red_max[4][16];
  float red_sum[4][16];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_ready[2];
  uint64_t p_ready[2];
  uint64_t o_ready[2];
  uint64_t v_fixed[2];
  uint64_t mma_done;
  int seq_keys[kMaxSeqs];       // clamped context length of each sequence
  int seq_start[kMaxSeqs + 1];  // prefix sum of partitions per sequence
  int scan[kTcThreads / 32];
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

// All 128 softmax threads agree on `ok` (named barrier 1).
__device__ __forceinline__ bool all_softmax(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

template <class QT, bool G16>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_q, int kv_rows) {
  extern __shared__ uint8_t smem_raw[];
  using L = Layout<G16>;
  constexpr int kStages = L::kStages;
  constexpr int kQBytes = L::kQBytes;
  constexpr int kPBytes = L::kPBytes;
  Smem<G16>& sm = *reinterpret_cast<Smem<G16>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool split = p.max_parts > 1;
  constexpr uint32_t kAB = std::is_same<QT, BF16>::value ? 1u : 0u;
  constexpr uint32_t kIdescS = tc::idesc_f16(kAB, 0, 0, 128, 16);
  constexpr uint32_t kIdescO = tc::idesc_f16(kAB, 1, 0, 128, 16);

  // ---- set-up -------------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
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
      for (uint32_t x = pos > kStages ? pos - kStages : 0; x < pos; ++x)
        mbar_wait(&sm.full[x % kStages], (x / kStages) & 1, 10000000ull);
    }
  } else if (warp == 5) {
    // ---- MMA issuer ---------------------------------------------------------------------
    if (lane == 0) {
      int idx = blockIdx.x;
      uint32_t pos = 0;
      Item cur, nxt;
      int it = 0;
      bool ok = true;
      auto mma_s = [&](const Item& x, int k) -> bool {
        const int b = k & 1;
        if (!wait_bar(&sm.q_full[b], (k >> 1) & 1, abort)) return false;
        const uint32_t qa = smem_u32(&sm.q[b][0]);
        for (int t = 0; t < x.ntiles; ++t, ++pos) {
          const int st = pos % kStages;
          if (!wait_bar(&sm.full[st], (pos / kStages) & 1, abort)) return false;
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
  } else if (warp == 6) {
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
#pragma unroll
      for (int h = 0; h < L::kRows; ++h) {
        if (h < p.group) {
          const float val = o[h] * (p.v_scale / sm.stat_l[b][h]);
          const size_t head = (size_t)x.seq * p.num_heads + (size_t)x.kvh * p.group + h;
          if (direct) {
            store_out(static_cast<OutT*>(p.out) + head * kD + d, val);
          } else {
            p.o_part[(head * p.max_parts + x.part) * kD + d] = val;
            if (d == 0) p.lse[head * p.max_parts + x.part] = sm.stat_m[b][h] + log2f(sm.stat_l[b][h]);
          }
        }
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
          for (int h = 0; h < L::kRows; ++h) {
            if (h < p.group) {
              const float e = fast_exp2(s[t][h] - mx[h]);
              sum[h] += e;
              OutT pv;
              store_out(&pv, e);
              *reinterpret_cast<OutT*>(col + (h >> 3) * kPGroupStride + (h & 7) * 16) = pv;
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
        sm.stat_m[b][tid] = fmaxf(fmaxf(sm.red_max[0][tid], sm.red_max[1][tid]),
                                  fmaxf(sm.red_max[2][tid], sm.red_max[3][tid]));
        sm.stat_l[b][tid] =
            (sm.red_sum[0][tid] + sm.red_sum[1][tid]) + (sm.red_sum[2][tid] + sm.red_sum[3][tid]);
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
template <class QT, bool G16>
int launch_tc_typed(const AttnParams& p, cudaStream_t stream) {
  const bool bf16 = std::is_same<QT, BF16>::value;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  CUtensorMap tk, tv;
  if (!make_map_2d(&tk, p.k_cache, kv_rows, bf16, 16) || !make_map_2d(&tv, p.v_cache, kv_rows, bf16, 16))
    return PKV_ERR_CUDA;
  const size_t smem = sizeof(Smem<G16>) + 1024;
  static_assert(sizeof(Smem<G16>) + 1024 <= 232448, "shared memory budget of one CTA");
  auto kern = paged_decode_tc_kernel<QT, G16>;
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
    if (p.lse) {
      c.lse = p.lse + head0 * p.max_parts;
      c.o_part = p.o_part + head0 * p.max_parts * kD;
    }
    CUtensorMap tq;
    if (!make_map_2d(&tq, c.q, (uint64_t)c.num_rows * p.num_heads, bf16, Layout<G16>::kRows))
      return PKV_ERR_CUDA;
    const long long items = (long long)c.num_rows * p.num_kv_heads * p.max_parts;
    int grid = sm_count();
    if (items < grid) grid = (int)items;
    if (grid < 1) grid = 1;
    kern<<<grid, kTcThreads, smem, stream>>>(c, tk, tv, tq, (int)kv_rows);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace

bool tc_decode_supported(const AttnParams& p, int q_dtype, int kv_dtype, int head_dim) {
  if (head_dim != kD || kv_dtype != q_dtype) return false;
  if (p.query_start_loc != nullptr || p.partition != kPart) return false;
  if (p.group < 2 || p.group > 16) return false;
  const uint64_t kv_rows = (uint64_t)p.num_blocks * p.num_kv_heads * kBlockSize;
  if (kv_rows + 16 >= (1ull << 31)) return false;
  if ((uint64_t)p.num_rows * p.num_heads + 16 >= (1ull << 31)) return false;
  if ((long long)p.num_rows * p.num_kv_heads * p.max_parts >= (1ll << 31)) return false;
  return tmap_available();
}

int launch_paged_decode_tc(const AttnParams& p, int q_dtype, cudaStream_t stream) {
  const bool g16 = p.group > 8;
  if (q_dtype == PKV_BF16)
    return g16 ? launch_tc_typed<BF16, true>(p, stream) : launch_tc_typed<BF16, false>(p, stream);
  return g16 ? launch_tc_typed<F16, true>(p, stream) : launch_tc_typed<F16, false>(p, stream);
}

}  // namespace pkv
