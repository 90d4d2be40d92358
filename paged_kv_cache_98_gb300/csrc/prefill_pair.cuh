// Chunked-prefill and draft-tree attention on CTA pairs: two CTAs of a
// cluster share every 256-row query tile through tcgen05.mma.cta_group::2.
//
// Sources: as prefill_tc.cuh ("第32讲 … Prefill vs Decode …", §5.4 chunked
// prefill; devpress.csdn.net vLLM overview, "9、FlashAttention (3)/(4)";
// openeuler.csdn.net notes, "MEDUSA推理框架" Tree Attention).
//
// The single-CTA kernel (prefill_tc.cuh) brings a whole 32 KB K tile and a
// whole 32 KB V tile into each SM for every 256 query rows it holds, as 32
// TMA boxes of one block half each (the paged layout allows no larger box),
// and a few warps issuing such boxes move only about 40 GB/s per SM.  Here a
// pair of CTAs computes one 256-row tile per MMA:
//   S = Q K^T     M = 256 rows (128 per CTA, from its own shared memory),
//                 N = 128 keys: CTA r holds keys 64 r .. 64 r + 63 of the tile
//                 (its 4 blocks, both 64-dim halves: 8 boxes, 16 KB)
//   O += P V      A = P from each CTA's own TMEM (its 128 rows), N = 128
//                 dims: CTA r holds dims 64 r .. 64 r + 63 of all 128 keys
//                 (one half of all 8 blocks: 8 boxes, 16 KB)
// so each SM loads half of every K and V tile for the same tensor work.  Each
// CTA's TMEM receives its own 128 rows of S and O, so the softmax, the lazy
// rescale, the masks and the epilogue run per CTA exactly as in the single
// kernel.  Nothing is broadcast: every load lands in the issuing CTA's own
// shared memory and counts its bytes on the even CTA's barrier (the MMAs
// read both CTAs' halves at the same offsets).
//
// Work item = (sequence, KV head, two 256-row query tiles a and b), longest
// first; a draft tree of 64 tokens at 8 heads per KV head is one item, so its
// context is streamed once.
//
// Barriers.  The even CTA's warp 8 issues every MMA and waits on its own
// CTA's barriers: full[stage] (3 producers x 2 CTAs arrive, both CTAs' bytes),
// q_full, tail_full, p_ready and o_free (one arrival per softmax warp of each
// CTA).  Each MMA
// commit that releases a resource (empty, q_empty, tail_free) or publishes a
// result (s_ready, o_done) arrives on that barrier in both CTAs.  The odd
// CTA's warp 8 only allocates and frees its TMEM with the pair.

#ifndef PKV_PREFILL_PAIR_CUH
#define PKV_PREFILL_PAIR_CUH

#include "prefill_tc.cuh"

namespace pkv {
namespace pre_tc {
namespace {

constexpr int kRowsPair = 256;               // rows of a pair tile (128 per CTA)
constexpr int kPairStages = 8;               // ring stages: K and V halves alternate
constexpr int kHalfTile = kTileBytes / 2;    // 16 KB: this CTA's half of a K or V tile
constexpr int kPairTail = kBlockSize * 128;  // 2 KB: this CTA's 64 dims of one V block

struct PairSmem {
  alignas(1024) uint8_t ring[kPairStages][kHalfTile];
  alignas(1024) uint8_t q[2][kTileBytes];  // this CTA's 128 rows of tiles a and b
  alignas(1024) uint8_t tail[kPairTail];
  int seq_start[kMaxSeqs + 1];  // prefix of items per sequence
  int seq_qlen[kMaxSeqs];
  int seq_ctx[kMaxSeqs];
  int seq_q0[kMaxSeqs];
  int few_start[kMaxSeqs + 1];  // prefix of rows seeing at most kFewKeys keys
  int scan[kThreads / 32];
  int scan2[kThreads / 32];
  uint64_t full[kPairStages];
  uint64_t empty[kPairStages];
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t s_ready[2];
  uint64_t p_ready[2];
  uint64_t o_done[2];
  uint64_t o_free[2];
  uint64_t tail_full;
  uint64_t tail_free;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// Items of a pair: (sequence, KV head, tiles 2m and 2m + 1 of 256 rows).
__device__ __forceinline__ bool next_pair_item(const AttnParams& p, const PairSmem& sm, int& idx,
                                               int total, Item& it, int stride) {
  if (idx >= total) return false;
  const int k = idx;
  idx += stride;
  const int kvh = k % p.num_kv_heads;
  const int unit = k / p.num_kv_heads;
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.seq_start[mid] <= unit) lo = mid; else hi = mid - 1;
  }
  const int rpt = kRowsPair / p.group;  // tokens per pair tile
  const int qlen = sm.seq_qlen[lo];
  it.seq = lo;
  it.kvh = kvh;
  it.ctx = sm.seq_ctx[lo];
  it.q0 = sm.seq_q0[lo];
  it.trow = lo;
  const int mp = sm.seq_start[lo + 1] - 1 - unit;  // longest tiles first
  it.chunk = 0;
  it.kt0 = 0;
  it.nk = 0;
  it.step = 1;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    it.t0[x] = (2 * mp + x) * rpt;
    it.nt[x] = max(0, min(rpt, qlen - it.t0[x]));
    it.pos0[x] = it.ctx - qlen + it.t0[x];
    it.nkt[x] = it.nt[x] > 0 ? (it.pos0[x] + it.nt[x] - 1) / kTileKeys + 1 : 0;
    it.nk = max(it.nk, it.nkt[x]);
    it.first[x] = 0;
    it.last[x] = it.nkt[x] > 0 ? it.nkt[x] - 1 : -1;
  }
  const bool partial = (it.ctx & (kBlockSize - 1)) != 0;
  it.tail_step = partial && (it.ctx - 1) / kTileKeys == it.nk - 1
                     ? ((it.ctx - 1) % kTileKeys) / kBlockSize
                     : -1;
  return true;
}

// Bounded wait, acquiring at cluster scope, for the barrier the other CTA's
// thread-written tail rows are published on.
__device__ __forceinline__ bool wait_bar_c(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           unsigned long long limit_ns) {
  if (tc::mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (tc::mbar_test_cluster(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Spins for about `ns` nanoseconds (used only after a wait gave up, so that
// copies this CTA issued have landed before the pair leaves).
__device__ __forceinline__ void settle(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) {
  }
}

// Scores of one key tile for the pair: Q (this CTA's [2 halves][128 rows][128
// B]) times this CTA's K half ([2 halves][64 keys][128 B]), K-steps of 16 dims.
__device__ __forceinline__ void issue_scores_pair(uint32_t d, uint64_t dq, uint64_t dk,
                                                  uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t oq = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
    const uint32_t ok = ((kk >> 2) * (kHalfTile / 2) + (kk & 3) * 32) >> 4;
    tc::mma_pair_f16(d, dq + oq, dk + ok, idesc, kk > 0);
  }
}

// O (+)= P V over one key tile, 16 keys per step; V is this CTA's 64 dims of
// the 128 keys ([128 keys][128 B], MN-major); step ts reads the tail buffer.
__device__ __forceinline__ void issue_pv_pair(uint32_t d, uint32_t a, uint64_t dv, uint64_t dtail,
                                              int ts, uint32_t acc0, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kTileKeys / 16; ++kk) {
    const uint64_t b = kk == ts ? dtail : dv + (uint64_t)((kk * (kBlockSize * 128)) >> 4);
    tc::mma_pair_f16_tmem_a(d, a + kk * 8, b, idesc, acc0 | (kk != 0 ? 1u : 0u));
  }
}

// The kernel body, run by both CTAs of pair `pair` of `npairs` that share the
// items.  kTree: draft-tree mode (per-row ancestor masks over the chunk's keys).
template <class QT, bool kTree>
__device__ __forceinline__ void prefill_pair_body(const AttnParams& p, const CUtensorMap& tm_k,
                                                  const CUtensorMap& tm_v,
                                                  const CUtensorMap& tm_q, int kv_rows, int pair,
                                                  int npairs, uint8_t* smem_raw) {
  PairSmem& sm = *reinterpret_cast<PairSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  constexpr uint32_t kAB = std::is_same<QT, BF16>::value ? 1u : 0u;
  constexpr uint32_t kIdescS = tc::idesc_f16(kAB, 0, 0, kRowsPair, 128);
  constexpr uint32_t kIdescO = tc::idesc_f16(kAB, 0, 1, kRowsPair, 128);
  const int g = p.group;

  // ---- set-up ---------------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&sm.full[s], 2 * kProducers);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.q_full, 2);
    mbar_init(&sm.q_empty, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.s_ready[x], 1);
      mbar_init(&sm.p_ready[x], 8);  // one arrival per softmax warp of each CTA
      mbar_init(&sm.o_done[x], 1);
      mbar_init(&sm.o_free[x], 8);
    }
    mbar_init(&sm.tail_full, 2);
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
    tc::tmem_alloc_pair(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish_pair();
  }
  {
    // per-sequence query length, context, first query row, and the prefix of items
    const int S = p.num_seqs, tid = threadIdx.x;
    const int chunk = (S + kThreads - 1) / kThreads;
    const int cap = p.max_blocks_per_seq * kBlockSize;
    int local = 0, local2 = 0;
    for (int i = 0; i < chunk; ++i) {
      const int sq = tid * chunk + i;
      if (sq < S) {
        const int q0 = __ldg(p.query_start_loc + sq);
        int qlen = __ldg(p.query_start_loc + sq + 1) - q0;
        int ctx = __ldg(p.context_lens + sq);
        if (ctx < 0 || ctx > cap || qlen < 0 || qlen > ctx || q0 < 0 || q0 + qlen > p.num_rows ||
            (kTree && qlen > 64)) {
          flag_error(p.errors, PKV_DEVERR_CONTEXT);
          ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
          qlen = qlen < 0 ? 0 : (qlen > ctx ? ctx : qlen);
          if (kTree && qlen > 64) qlen = 64;  // the mask covers 64 chunk keys
          if (q0 < 0 || q0 + qlen > p.num_rows) qlen = 0;
        }
        sm.seq_qlen[sq] = qlen;
        sm.seq_ctx[sq] = ctx;
        sm.seq_q0[sq] = q0;
        const int tiles = (qlen * g + kRowsPair - 1) / kRowsPair;
        local += ctx > 0 ? (tiles + 1) / 2 : 0;
        local2 += few_rows<kTree, false>(qlen, ctx);
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
        run2 += few_rows<kTree, false>(sm.seq_qlen[sq], sm.seq_ctx[sq]);
        sm.seq_start[sq] = run;
        const int tiles = (sm.seq_qlen[sq] * g + kRowsPair - 1) / kRowsPair;
        run += sm.seq_ctx[sq] > 0 ? (tiles + 1) / 2 : 0;
      }
    }
    if (tid == kThreads - 1) {
      sm.seq_start[S] = base + incl;
      sm.few_start[S] = base2 + incl2;
    }
  }
  // both CTAs' barriers are initialised before either CTA arrives on the other's
  tc::fence_before_sync();
  tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const unsigned long long lim = wait_limit(p);
  const int total = sm.seq_start[p.num_seqs] * p.num_kv_heads;
  // a barrier's address in the even CTA (rank 0) and in the odd one (rank 1)
  auto at0 = [&](const void* b) { return tc::map_rank(smem_u32(b), 0); };
  auto at1 = [&](const void* b) { return tc::map_rank(smem_u32(b), 1); };
  const int tok_off = (int)rank * (kRowsM / g);  // this CTA's first token of a pair tile
  bool ok = true;

  if (warp >= 9) {
    // ---- TMA producers (ring order K0, V0, K1, V1, ...) ------------------------------------
    // Lane 8 (t % 4) + j holds block j of key tile t.  K: this CTA's blocks
    // (j / 4 == rank), both dim halves, block j % 4 issued by producer
    // (j % 4) % 3.  V: all 8 blocks, this CTA's dim half, block j issued by
    // producer (j + 1) % 3.
    const int pw = warp - 9;
    const int jt = lane & 7;
    const bool k_mine = (jt >> 2) == (int)rank && (jt & 3) % kProducers == pw;
    const bool v_mine = (jt + 1) % kProducers == pw;
    uint32_t kbytes = 0, vbytes = 0;  // this producer's bytes per K / V stage
#pragma unroll
    for (int j = 0; j < 4; ++j) kbytes += j % kProducers == pw ? 2 * (kBlockSize * 128) : 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) vbytes += (j + 1) % kProducers == pw ? kBlockSize * 128 : 0;
    int idx = pair;
    uint32_t pos = 0;
    int nitem = 0, ntail = 0;
    Item x;
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
      const int st = pos % kPairStages;
      // test hook: these boxes are never issued, so every wait for the tile runs out
      const bool skip = pw == 0 && pair == 0 && rank == 0 && p.skip_copy > 0 &&
                        pos + 1 == (uint32_t)p.skip_copy;
      const uint32_t bar = at0(&sm.full[st]);
      bool good = true;
      if (lane == 0) {
        if (pos >= (uint32_t)kPairStages)
          good = wait_bar(&sm.empty[st], ((pos / kPairStages) - 1) & 1, abort, lim);
        if (good && !skip) tc::mbar_arrive_expect_tx_cluster(bar, is_v ? vbytes : kbytes);
      }
      if (!__shfl_sync(kFull, (int)good, 0)) return false;
      if (!skip && (lane >> 3) == (t & 3) && (is_v ? v_mine : k_mine)) {
        uint8_t* dst = &sm.ring[st][0];
        if (is_v) {
          tc::tma_load_2d_pair(dst + jt * (kBlockSize * 128), &tm_v, 64 * (int)rank, row, bar);
        } else {
          uint8_t* d0 = dst + (jt & 3) * (kBlockSize * 128);
          tc::tma_load_2d_pair(d0, &tm_k, 0, row, bar);
          tc::tma_load_2d_pair(d0 + kHalfTile / 2, &tm_k, 64, row, bar);
        }
      }
      __syncwarp();
      ++pos;
      return true;
    };
    // this CTA's 64 dims of the V rows of the partial last block, rows past the
    // context as zeros, swizzled like the ring (0 * NaN would poison the MMA)
    auto load_tail = [&]() -> bool {
      bool good = true;
      if (lane == 0 && ntail >= 1) good = wait_bar(&sm.tail_free, (ntail - 1) & 1, abort, lim);
      if (!__shfl_sync(kFull, (int)good, 0)) return false;
      const int bi = (x.ctx - 1) / kBlockSize;
      const int blk = __ldg(p.block_tables + (size_t)x.trow * p.max_blocks_per_seq + bi);
      const bool bok = blk >= 0 && blk < p.num_blocks;
      const uint8_t* src = p.v_cache +
                           ((size_t)(bok ? blk : 0) * p.num_kv_heads + x.kvh) * kBlockSize * (kD * 2) +
                           rank * 128;
      const int rows = x.ctx - bi * kBlockSize;
#pragma unroll
      for (int i = 0; i < kPairTail / 16 / 32; ++i) {
        const int c = lane + 32 * i;
        const int r = c >> 3, ch = c & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (bok && r < rows) v = __ldg(reinterpret_cast<const uint4*>(src + r * (kD * 2)) + ch);
        *reinterpret_cast<uint4*>(&sm.tail[0] + r * 128 + ((ch ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster_release(at0(&sm.tail_full));
      ++ntail;
      return true;
    };
    while (ok && next_pair_item(p, sm, idx, total, x, npairs)) {
      bool good = true;
      if (pw == 0 && lane == 0) {
        if (nitem >= 1) good = wait_bar(&sm.q_empty, (nitem - 1) & 1, abort, lim);
        if (good) {
          const int nq = x.nt[1] > 0 ? 2 : 1;
          const uint32_t bar = at0(&sm.q_full);
          tc::mbar_arrive_expect_tx_cluster(bar, nq * kTileBytes);
          for (int qt = 0; qt < nq; ++qt) {
            uint8_t* dq = &sm.q[qt][0];
            const int tok = x.q0 + x.t0[qt] + tok_off;
            tc::tma_load_3d_pair(dq, &tm_q, 0, x.kvh * g, tok, bar);
            tc::tma_load_3d_pair(dq + kHalf, &tm_q, 64, x.kvh * g, tok, bar);
          }
        }
      }
      ok = __shfl_sync(kFull, (int)good, 0) != 0;
      // block rows of the 32-block table chunk (4 key tiles) being issued, the
      // next chunk read ahead
      int rc_c = -1, rc_row = kv_rows;
      int pre_c = 0, pre_raw = fetch(0);
      auto row_for = [&](int t) -> int {
        const int c = t >> 2;
        if (rc_c != c) {
          rc_row = to_row(pre_c == c ? pre_raw : fetch(c));
          rc_c = c;
          pre_c = c + 1;
          pre_raw = 4 * pre_c < x.nk ? fetch(pre_c) : kBeyond;
        }
        return rc_row;
      };
      for (int t = 0; ok && t < x.nk; ++t) {
        const int row = row_for(t);
        ok = issue(t, row, false);
        if (ok && pw == 0 && t == x.nk - 1 && x.tail_step >= 0) ok = load_tail();
        if (ok) ok = issue(t, row, true);
      }
      ++nitem;
    }
    if (!ok) {
      if (lane == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      // the copies issued so far count on the even CTA's barriers: let them land
      settle(5000000ull);
    }
  } else if (warp == 8) {
    // ---- MMA issuer (even CTA) ---------------------------------------------------------
    // Order per item: S_a(0), S_b(0), then for each key tile t:
    //   P_a(t) V_t, S_a(t+1), P_b(t) V_t, S_b(t+1)
    // as in the single-CTA kernel.  The whole warp runs the loop; one elected
    // lane issues the MMAs and commits.
    if (rank == 0) {
      const bool leader = tc::elect_one();
      // releases and results go to the barrier in both CTAs
      auto commit2 = [&](uint64_t* bar) {
        if (leader) {
          tc::mma_pair_commit(smem_u32(bar));
          tc::mma_pair_commit(at1(bar));
        }
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __shfl_sync(kFull, (int)wait_bar(bar, parity, abort, lim), 0) != 0;
      };
      int idx = pair;
      uint32_t pos = 0;
      uint32_t np[2] = {0, 0};
      uint32_t nit[2] = {0, 0};
      int nitem = 0, ntail = 0;
      Item x;
      const uint64_t dq[2] = {tc::smem_desc(smem_u32(&sm.q[0][0]), 16, 1024, tc::kLayoutSw128),
                              tc::smem_desc(smem_u32(&sm.q[1][0]), 16, 1024, tc::kLayoutSw128)};
      const uint64_t dk0 = tc::smem_desc(smem_u32(&sm.ring[0][0]), 16, 1024, tc::kLayoutSw128);
      // V halves are one 64-dim swizzle atom wide (the leading offset is not used)
      const uint64_t dv0 =
          tc::smem_desc(smem_u32(&sm.ring[0][0]), kHalfTile, 1024, tc::kLayoutSw128);
      const uint64_t dtail =
          tc::smem_desc(smem_u32(&sm.tail[0]), kPairTail, 1024, tc::kLayoutSw128);
      auto acquire = [&](int& st) -> bool {
        st = pos % kPairStages;
        const bool r = wait(&sm.full[st], (pos / kPairStages) & 1);
        ++pos;
        if (r) tc::fence_after_sync();
        return r;
      };
      // has the next ring stage landed? (a test, no wait)
      auto landed = [&]() -> bool {
        return __shfl_sync(kFull, (int)mbar_peek(&sm.full[pos % kPairStages],
                                                  (pos / kPairStages) & 1), 0) != 0;
      };
      auto mma_s = [&](int qt, int st) {
        if (leader)
          issue_scores_pair(tmem + qt * 128, dq[qt], dk0 + (uint64_t)(st * (kHalfTile >> 4)),
                            kIdescS);
        commit2(&sm.s_ready[qt]);
      };
      auto mma_pv = [&](int qt, int st, int t) -> bool {
        if (!wait(&sm.p_ready[qt], np[qt] & 1)) return false;
        ++np[qt];
        if (t == 0 && nit[qt] >= 1 && !wait(&sm.o_free[qt], (nit[qt] - 1) & 1))
          return false;  // both CTAs have read out the previous item's O
        tc::fence_after_sync();
        if (leader)
          issue_pv_pair(tmem + kColO + qt * 128, tmem + qt * 128,
                        dv0 + (uint64_t)(st * (kHalfTile >> 4)), dtail,
                        t == x.nk - 1 ? x.tail_step : -1, t != 0, kIdescO);
        if (t == x.last[qt]) commit2(&sm.o_done[qt]);
        return true;
      };
      auto tail_wait = [&](int t) -> bool {
        if (t != x.nk - 1 || x.tail_step < 0) return true;
        const bool r =
            __shfl_sync(kFull, (int)wait_bar_c(&sm.tail_full, ntail & 1, abort, lim), 0) != 0;
        if (r) tc::fence_after_sync();
        return r;
      };
      while (ok && next_pair_item(p, sm, idx, total, x, npairs)) {
        const bool ha = x.last[0] >= 0;
        const bool hb = x.last[1] >= 0;
        int kst = 0, vst = 0;
        ok = wait(&sm.q_full, nitem & 1);
        if (ok) tc::fence_after_sync();
        if (ok) ok = acquire(kst);
        if (ok) {
          if (ha) mma_s(0, kst);
          if (hb) mma_s(1, kst);
          commit2(&sm.empty[kst]);
          if (x.nk == 1) commit2(&sm.q_empty);
        }
        for (int t = 0; ok && t < x.nk; ++t) {
          const bool more = t + 1 < x.nk;
          ok = acquire(vst);
          if (ok) ok = tail_wait(t);
          // K(t + 1) is taken before P_a(t) is awaited when it has landed
          bool k_taken = false;
          if (ok && more && landed()) {
            ok = acquire(kst);
            k_taken = true;
          }
          if (ok && t <= x.last[0]) ok = mma_pv(0, vst, t);
          if (ok && more && !k_taken) ok = acquire(kst);
          if (ok && more && t + 1 <= x.last[0]) mma_s(0, kst);
          if (ok && hb) ok = mma_pv(1, vst, t);
          if (!ok) break;
          commit2(&sm.empty[vst]);
          if (more) {
            if (hb) mma_s(1, kst);
            commit2(&sm.empty[kst]);
            if (t + 1 == x.nk - 1) commit2(&sm.q_empty);
          }
        }
        if (ok && x.tail_step >= 0) {
          commit2(&sm.tail_free);
          ++ntail;
        }
        if (ha) ++nit[0];
        if (hb) ++nit[1];
        ++nitem;
      }
      if (!ok && leader) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      // no MMA of the pair may still run when either CTA releases its TMEM
      if (leader) tc::mma_pair_commit(smem_u32(&sm.mma_done));
      mbar_wait(&sm.mma_done, 0, 100000000ull);
    }
  } else {
    // ---- softmax + epilogue: warpgroup qt = 0 (tile a) or 1 (tile b) --------------------
    // As in the single-CTA kernel, for this CTA's 128 rows of each pair tile.
    const int qt = warp >> 2;
    const int tid = threadIdx.x & 127;  // row = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_off + qt * 128;
    const uint32_t o_col = tmem + lane_off + kColO + qt * 128;
    const float qs = p.q_scale;
    using OutT = typename QT::T;
    const bool neg = qs < 0.0f;
    const float qa = fmaxf(fabsf(qs), 1e-30f);
    const uint32_t p_ready0 = at0(&sm.p_ready[qt]);
    const uint32_t o_free0 = at0(&sm.o_free[qt]);
    int idx = pair;
    uint32_t ns = 0, nit = 0;
    Item x;
    while (ok && next_pair_item(p, sm, idx, total, x, npairs)) {
      // this warpgroup's fields of the item, in registers
      const int nt = qt ? x.nt[1] : x.nt[0];
      const int t0 = qt ? x.t0[1] : x.t0[0];
      const int pos0 = qt ? x.pos0[1] : x.pos0[0];
      const int last = qt ? x.last[1] : x.last[0];
      if (last < 0) continue;  // no tile b in this item
      const int tok = tok_off + tid / g;  // token within the pair tile
      // rows past the tile's tokens compute on whatever Q holds there; their
      // output is never stored
      const bool valid = tok < nt;
      const size_t head = (size_t)(x.q0 + t0 + tok) * p.num_heads + (size_t)x.kvh * g + tid % g;
      const int qpos = pos0 + tok;
      const int cbase = pos0 - t0;  // the chunk's first position
      const uint64_t tmask = kTree && valid ? __ldg(p.tree_mask + x.q0 + t0 + tok) : 0ull;
      const int first_pos = pos0 + tok_off;  // this CTA's first row's position
      float m_run = -INFINITY;
      float2 l2[4];  // partial row sums (independent chains, packed pairs)
#pragma unroll
      for (int i = 0; i < 4; ++i) l2[i] = make_float2(0.0f, 0.0f);
      // each warp waits and signals on its own: no barrier across the warpgroup
      for (int t = 0; t <= last; ++t, ++ns) {
        ok = __all_sync(kFull, wait_bar(&sm.s_ready[qt], ns & 1, abort, lim));
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
          // chunk keys are visible when the row's mask has their bit; keys
          // before the chunk always are (key 32 w + i of the tile: bit i of vw[w])
          const int nrel = x.ctx - cbase;
          uint32_t vw[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int r0 = kbase + 32 * w - cbase;
            const uint64_t bits = r0 >= 0 ? (r0 < 64 ? tmask >> r0 : 0ull)
                                          : (-r0 < 64 ? tmask << -r0 : 0ull);
            const int lim2 = nrel - r0;
            const uint32_t keep = lim2 <= 0 ? 0u : (lim2 >= 32 ? ~0u : (1u << lim2) - 1u);
            const uint32_t prior = r0 >= 0 ? 0u : (-r0 >= 32 ? ~0u : (1u << -r0) - 1u);
            vw[w] = prior | ((uint32_t)bits & keep);
          }
#pragma unroll
          for (int c = 0; c < kTileKeys; ++c) {
            sv[c] = (vw[c >> 5] >> (c & 31)) & 1u ? sv[c] : -INFINITY;
            mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
          }
        } else if (!kTree && kbase + kTileKeys - 1 > first_pos) {
          // the causal boundary of some row of this CTA crosses this tile
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
                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * qa;
        // move the running max (and rescale O) only on a large increase
        const bool need = mt > m_run + kRescaleAt;
        float alpha = 1.0f;
        if (need) {
          alpha = t == 0 ? 0.0f : fast_exp2(m_run - mt);
          m_run = mt;
#pragma unroll
          for (int i = 0; i < 4; ++i) l2[i] = __fmul2_rn(l2[i], make_float2(alpha, alpha));
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float pk[16];
          exp_pairs<QT>(sv + h * 32, qa, m_run, l2, pk);
          tc::tmem_st16(s_col + 16 * h, pk);
        }
        if (t > 0 && __any_sync(kFull, need)) {
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
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(p_ready0);
      }
      if (!ok) break;
      // ---- epilogue: O / l --------------------------------------------------------------
      ok = __all_sync(kFull, wait_bar(&sm.o_done[qt], nit & 1, abort, lim));
      if (!ok) break;
      tc::fence_after_sync();
      const float l = ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y)) +
                      ((l2[2].x + l2[2].y) + (l2[3].x + l2[3].y));
      const float inv = valid ? 1.0f / l : 0.0f;
      OutT* orow = static_cast<OutT*>(p.out) + head * kD;
      const bool store = valid && !(kTree ? cbase < kFewKeys : qpos < kFewKeys);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float ov[32];
        tc::tmem_ld32(o_col + 32 * c, ov);
        tc::tmem_wait_ld();
        if (store) {
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
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(o_free0);
      ++nit;
    }
    if (!ok && lane == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
    if (ok) few_key_rows<QT, kTree>(p, sm, blockIdx.x * 256 + qt * 128 + tid, gridDim.x * 256);
  }

  if (!ok) settle(5000000ull);  // the other CTA may still be giving up
  tc::fence_before_sync();
  tc::cluster_sync();
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace pre_tc
}  // namespace pkv

#endif  // PKV_PREFILL_PAIR_CUH
