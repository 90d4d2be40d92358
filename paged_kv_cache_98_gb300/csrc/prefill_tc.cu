// Chunked-prefill paged attention on the tcgen05 tensor cores (head_dim 128,
// fp16/bf16 caches, group sizes dividing 128).
//
// Sources: "第32讲 … Prefill vs Decode …", §5.4 (a prompt is processed in
// chunks; each chunk's queries attend the paged prior context and, causally,
// the chunk itself) and §3.4 (query heads grouped on a KV head);
// devpress.csdn.net vLLM overview, "9、FlashAttention (3)/(4)" (query blocks
// against streamed key/value blocks, running max and sum of exponentials).
//
// Work item = (sequence, KV head, tile of 128 query rows), a row being a
// (query token, head of the group) pair, token-major, so that the g heads of a
// KV head share every K/V tile.  Per 128-key tile j of the visible context:
//   S_j = Q K_j^T              tcgen05, M = 128 rows, N = 128 keys, fp32 in TMEM
//   online softmax per row     four warps, thread = row = TMEM lane; causal mask
//   O  += P_j V_j              tcgen05, A = P (bf16/fp16 in shared memory), B = V
// The running max is only moved (and O rescaled in TMEM) when a row's tile max
// exceeds it by more than 8 in base-2 units, so exponentials stay <= 2^8 and
// most tiles need no rescale; the final division by the row sum is exact.
// The MMA issuer runs S one tile ahead of the P V product (S double-buffered
// in TMEM), so the softmax of tile j overlaps the MMAs of tile j+1.
//
// Warps: 0-3 softmax + epilogue, 4 TMA producer (Q with one 3-D box per half,
// K/V with one 16-row box per block and half), 5 TMEM owner + MMA issuer.

#include <cuda.h>

#include <cstddef>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 192;
constexpr int kD = 128;
constexpr int kTileKeys = 128;
constexpr int kRowsM = 128;
constexpr int kStages = 3;
constexpr int kTileBytes = 128 * kD * 2;  // 32 KB: [2 halves][128 rows][128 B]
constexpr int kHalf = kTileBytes / 2;
constexpr int kMaxSeqs = 1024;
constexpr int kTmemCols = 512;  // S (2 x 128) + O (128), rounded up
constexpr float kRescaleAt = 8.0f;

struct Smem {
  alignas(1024) uint8_t ring[kStages][kTileBytes];
  alignas(1024) uint8_t q[kTileBytes];
  alignas(1024) uint8_t pmat[2][kTileBytes];
  int seq_start[kMaxSeqs + 1];  // prefix of query-row tiles per sequence
  int seq_qlen[kMaxSeqs];
  int seq_ctx[kMaxSeqs];
  int seq_q0[kMaxSeqs];
  int scan[kThreads / 32];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t s_ready[2];
  uint64_t p_ready[2];
  uint64_t o_done[2];
  uint64_t o_free;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  uint32_t issued;
};

struct Item {
  int seq, kvh, t0, nt, qlen, ctx, q0, pos0, nkt;
};

__device__ __forceinline__ bool next_item(const AttnParams& p, const Smem& sm, int& idx,
                                          int total, Item& it) {
  if (idx >= total) return false;
  const int k = idx;
  idx += gridDim.x;
  const int kvh = k % p.num_kv_heads;
  const int pair = k / p.num_kv_heads;
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.seq_start[mid] <= pair) lo = mid; else hi = mid - 1;
  }
  const int ntile = sm.seq_start[lo + 1] - sm.seq_start[lo];
  const int mt = ntile - 1 - (pair - sm.seq_start[lo]);  // longest tiles first
  const int rpt = kRowsM / p.group;                      // tokens per tile
  it.seq = lo;
  it.kvh = kvh;
  it.qlen = sm.seq_qlen[lo];
  it.ctx = sm.seq_ctx[lo];
  it.q0 = sm.seq_q0[lo];
  it.t0 = mt * rpt;
  it.nt = min(rpt, it.qlen - it.t0);
  it.pos0 = it.ctx - it.qlen + it.t0;
  it.nkt = (it.pos0 + it.nt - 1) / kTileKeys + 1;
  return true;
}

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

template <class QT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, int kv_rows) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t kAB = std::is_same<QT, BF16>::value ? 1u : 0u;
  constexpr uint32_t kIdescS = tc::idesc_f16(kAB, 0, 0, 128, 128);
  constexpr uint32_t kIdescO = tc::idesc_f16(kAB, 0, 1, 128, 128);
  const int g = p.group;

  // ---- set-up ---------------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_ready[b], 1);
      mbar_init(&sm.p_ready[b], 1);
      mbar_init(&sm.o_done[b], 1);
    }
    mbar_init(&sm.o_free, 1);
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
  {
    // per-sequence query length, context, first query row, and the prefix
    // of 128-row tiles
    const int S = p.num_seqs, tid = threadIdx.x;
    const int chunk = (S + kThreads - 1) / kThreads;
    const int cap = p.max_blocks_per_seq * kBlockSize;
    int local = 0;
    for (int i = 0; i < chunk; ++i) {
      const int sq = tid * chunk + i;
      if (sq < S) {
        const int q0 = __ldg(p.query_start_loc + sq);
        int qlen = __ldg(p.query_start_loc + sq + 1) - q0;
        int ctx = __ldg(p.context_lens + sq);
        if (ctx < 0 || ctx > cap || qlen < 0 || qlen > ctx || q0 < 0 || q0 + qlen > p.num_rows) {
          flag_error(p.errors, PKV_DEVERR_CONTEXT);
          ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
          qlen = qlen < 0 ? 0 : (qlen > ctx ? ctx : qlen);
          if (q0 < 0 || q0 + qlen > p.num_rows) qlen = 0;
        }
        sm.seq_qlen[sq] = qlen;
        sm.seq_ctx[sq] = ctx;
        sm.seq_q0[sq] = q0;
        local += (qlen * g + kRowsM - 1) / kRowsM;
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
        run += (sm.seq_qlen[sq] * g + kRowsM - 1) / kRowsM;
      }
    }
    if (tid == kThreads - 1) sm.seq_start[S] = base + incl;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  const int total = sm.seq_start[p.num_seqs] * p.num_kv_heads;

  if (warp == 4) {
    // ---- TMA producer ---------------------------------------------------------------------
    int idx = blockIdx.x;
    uint32_t pos = 0;
    int nitem = 0;
    bool ok = true;
    Item x;
    // lane j: cache row of block 32*c + j of the item's key range
    auto rows_for = [&](int c) -> int {
      const int b = 32 * c + lane;
      const int nblk = (x.ctx + kBlockSize - 1) / kBlockSize;
      int row = kv_rows;
      if (b < nblk) {
        const int blk = __ldg(p.block_tables + (size_t)x.seq * p.max_blocks_per_seq + b);
        if (blk >= 0 && blk < p.num_blocks)
          row = (blk * p.num_kv_heads + x.kvh) * kBlockSize;
        else
          flag_error(p.errors, PKV_DEVERR_BLOCK_ID);
      }
      return row;
    };
    // Block rows of K chunk ck (current), ck-1 (still needed by the V tiles,
    // which lag one tile) and ck+1 (loaded one chunk ahead so its latency hides).
    int ck = 0, r_prev = kv_rows, r_cur = kv_rows, r_next = kv_rows;
    auto issue = [&](int t, bool is_v) -> bool {
      const int c = t >> 2;
      if (!is_v && c != ck) {  // K moves to the next chunk
        r_prev = r_cur;
        r_cur = r_next;
        r_next = rows_for(c + 1);
        ck = c;
      }
      const int row = (is_v && c != ck) ? r_prev : r_cur;
      const int st = pos % kStages;
      bool good = true;
      if (lane == 0) {
        if (pos >= kStages) good = wait_bar(&sm.empty[st], ((pos / kStages) - 1) & 1, abort);
        if (good) mbar_arrive_expect_tx(&sm.full[st], kTileBytes);
      }
      if (!__shfl_sync(kFull, (int)good, 0)) return false;
      if ((lane >> 3) == (t & 3)) {
        uint8_t* dst = &sm.ring[st][0] + (lane & 7) * (kBlockSize * 128);
        const CUtensorMap* map = is_v ? &tm_v : &tm_k;
        tc::tma_load_2d(dst, map, 0, row, &sm.full[st]);
        tc::tma_load_2d(dst + kHalf, map, 64, row, &sm.full[st]);
      }
      __syncwarp();
      if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&sm.issued) = pos + 1;
      ++pos;
      return true;
    };
    while (ok && next_item(p, sm, idx, total, x)) {
      ck = 0;
      r_prev = kv_rows;
      r_cur = rows_for(0);
      r_next = rows_for(1);
      bool good = true;
      if (lane == 0) {
        if (nitem >= 1) good = wait_bar(&sm.q_empty, (nitem - 1) & 1, abort);
        if (good) {
          mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
          const int tok = x.q0 + x.t0;
          tc::tma_load_3d(&sm.q[0], &tm_q, 0, x.kvh * g, tok, &sm.q_full);
          tc::tma_load_3d(&sm.q[kHalf], &tm_q, 64, x.kvh * g, tok, &sm.q_full);
        }
      }
      ok = __shfl_sync(kFull, (int)good, 0) != 0;
      // ring order = MMA order: K0, then (K_t, V_{t-1}) ..., then V_last
      if (ok) ok = issue(0, false);
      for (int t = 1; ok && t < x.nkt; ++t) {
        ok = issue(t, false);
        if (ok) ok = issue(t - 1, true);
      }
      if (ok) ok = issue(x.nkt - 1, true);
      ++nitem;
    }
    if (!ok && lane == 0) {
      flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      for (uint32_t y = pos > kStages ? pos - kStages : 0; y < pos; ++y)
        mbar_wait(&sm.full[y % kStages], (y / kStages) & 1, 10000000ull);
    }
  } else if (warp == 5) {
    // ---- MMA issuer --------------------------------------------------------------------
    if (lane == 0) {
      int idx = blockIdx.x;
      uint32_t pos = 0, J = 0;  // ring position, global S-tile counter
      int nitem = 0;
      bool ok = true;
      Item x;
      const uint32_t qa = smem_u32(&sm.q[0]);
      auto mma_s = [&](uint32_t j) -> bool {
        const int st = pos % kStages;
        if (!wait_bar(&sm.full[st], (pos / kStages) & 1, abort)) return false;
        tc::fence_after_sync();
        const uint32_t ka = smem_u32(&sm.ring[st][0]);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_f16(tmem + (j & 1) * 128, tc::smem_desc(qa + off, 16, 1024, tc::kLayoutSw128),
                      tc::smem_desc(ka + off, 16, 1024, tc::kLayoutSw128), kIdescS, kk > 0);
        }
        tc::mma_commit(&sm.empty[st]);
        tc::mma_commit(&sm.s_ready[j & 1]);
        ++pos;
        return true;
      };
      auto mma_pv = [&](uint32_t j, bool first) -> bool {
        if (!wait_bar(&sm.p_ready[j & 1], (j >> 1) & 1, abort)) return false;
        const int st = pos % kStages;
        if (!wait_bar(&sm.full[st], (pos / kStages) & 1, abort)) return false;
        tc::fence_after_sync();
        const uint32_t pa = smem_u32(&sm.pmat[j & 1][0]);
        const uint32_t va = smem_u32(&sm.ring[st][0]);
#pragma unroll
        for (int kk = 0; kk < kTileKeys / 16; ++kk) {
          const uint64_t a = tc::smem_desc(pa + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024,
                                           tc::kLayoutSw128);
          const uint64_t b = tc::smem_desc(va + kk * (kBlockSize * 128), kHalf, 1024,
                                           tc::kLayoutSw128);
          tc::mma_f16(tmem + 256, a, b, kIdescO, (!first || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm.empty[st]);
        tc::mma_commit(&sm.o_done[j & 1]);
        ++pos;
        return true;
      };
      while (ok && next_item(p, sm, idx, total, x)) {
        if (!wait_bar(&sm.q_full, nitem & 1, abort)) { ok = false; break; }
        const uint32_t j0 = J;
        ok = mma_s(J++);
        for (int t = 1; ok && t < x.nkt; ++t) {
          ok = mma_s(J++);
          if (t == x.nkt - 1 && ok) tc::mma_commit(&sm.q_empty);
          if (ok && t == 1 && nitem >= 1)
            ok = wait_bar(&sm.o_free, (nitem - 1) & 1, abort);  // previous O read out
          if (ok) ok = mma_pv(j0 + t - 1, t == 1);
        }
        if (ok && x.nkt == 1) {
          tc::mma_commit(&sm.q_empty);
          if (nitem >= 1) ok = wait_bar(&sm.o_free, (nitem - 1) & 1, abort);
        }
        if (ok) ok = mma_pv(j0 + x.nkt - 1, x.nkt == 1);
        ++nitem;
      }
      if (!ok) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
      tc::mma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, 100000000ull);
    }
  } else {
    // ---- softmax + epilogue (warps 0-3, thread = row = TMEM lane) ----------------------------
    const int tid = threadIdx.x;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float qs = p.q_scale;
    using OutT = typename QT::T;
    int idx = blockIdx.x;
    uint32_t J = 0, pos = 0;
    bool ok = true;
    Item x;
    while (ok && next_item(p, sm, idx, total, x)) {
      const int tok = tid / g;  // token within the tile
      const bool valid = tid < x.nt * g;
      const int qpos = x.pos0 + tok;
      float m_run = -INFINITY, l = 0.0f;
      const uint32_t item_pos = pos;  // ring position of this item's K0
      pos += 2 * x.nkt;
      for (int t = 0; t < x.nkt; ++t, ++J) {
        ok = all_softmax(wait_bar(&sm.s_ready[J & 1], (J >> 1) & 1, abort));
        if (!ok) break;
        tc::fence_after_sync();
        float sv[kTileKeys];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32(tmem + lane_off + (J & 1) * 128 + 32 * c, sv + 32 * c);
        tc::tmem_wait_ld();
        const int kbase = t * kTileKeys;
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTileKeys; ++c) {
          const bool vis = valid && kbase + c <= qpos;
          sv[c] = vis ? sv[c] * qs : -INFINITY;
          mt = fmaxf(mt, sv[c]);
        }
        // move the running max (and rescale O) only on a large increase
        const bool need = valid && (mt > m_run + kRescaleAt);
        float alpha = 1.0f;
        if (need) {
          alpha = (t == 0) ? 0.0f : fast_exp2(m_run - mt);
          m_run = mt;
          l *= alpha;
        }
        if (t > 0 && __any_sync(kFull, need)) {
          // O must be complete up to tile t-1 before it is rescaled in place
          bool w = wait_bar(&sm.o_done[(J - 1) & 1], ((J - 1) >> 1) & 1, abort);
          if (!__all_sync(kFull, w)) { ok = false; }
          if (ok) {
            tc::fence_after_sync();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float ov[32];
              tc::tmem_ld32(tmem + lane_off + 256 + 32 * c, ov);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] *= alpha;
              tc::tmem_st32(tmem + lane_off + 256 + 32 * c, ov);
            }
            tc::tmem_wait_st();
          }
        }
        ok = all_softmax(ok);
        if (!ok) break;
        // P buffer J&1 was last read by the product of tile J-2
        if (J >= 2) {
          ok = all_softmax(wait_bar(&sm.o_done[J & 1], ((J - 2) >> 1) & 1, abort));
          if (!ok) break;
        }
        uint8_t* prow = &sm.pmat[J & 1][0] + tid * 128;
        const int sw = tid & 7;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {  // 16-byte chunks of 8 keys
          float e[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float v = sv[ch * 8 + i];
            e[i] = valid ? fast_exp2(v - m_run) : 0.0f;
            l += e[i];
          }
          uint4 w;
          w.x = pack2<QT>(e[0], e[1]);
          w.y = pack2<QT>(e[2], e[3]);
          w.z = pack2<QT>(e[4], e[5]);
          w.w = pack2<QT>(e[6], e[7]);
          const int half = ch >> 3, c16 = (ch & 7) ^ sw;
          *reinterpret_cast<uint4*>(prow + half * kHalf + c16 * 16) = w;
        }
        // V rows past the context in the last block are garbage (0 * NaN = NaN
        // inside the MMA): zero them once that tile has landed
        const int last = x.ctx - 1;
        const int tail = x.ctx & (kBlockSize - 1);
        if (t == x.nkt - 1 && tail && last >= kbase && last < kbase + kTileKeys) {
          const uint32_t vpos = item_pos + 2 * x.nkt - 1;
          bool w = true;
          const uint64_t t0 = globaltimer_ns();
          while (*reinterpret_cast<volatile uint32_t*>(&sm.issued) <= vpos) {
            if (*abort || globaltimer_ns() - t0 > 2000000000ull) {
              *abort = 1;
              w = false;
              break;
            }
          }
          if (w) w = wait_bar(&sm.full[vpos % kStages], (vpos / kStages) & 1, abort);
          ok = all_softmax(w);
          if (!ok) break;
          const int jb = (last - kbase) / kBlockSize;
          const int rows = kBlockSize - tail;
          uint8_t* vb = &sm.ring[vpos % kStages][0] + (jb * kBlockSize + tail) * 128;
          for (int i = tid; i < rows * 2 * 8; i += 128) {
            const int half = i / (rows * 8), r = (i / 8) % rows, c = i % 8;
            reinterpret_cast<uint4*>(vb + half * kHalf + r * 128)[c] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        tc::named_sync(1, 128);
        if (tid == 0) mbar_arrive(&sm.p_ready[J & 1]);
      }
      if (!ok) break;
      // ---- epilogue: O / l --------------------------------------------------------------
      const uint32_t jl = J - 1;
      ok = all_softmax(wait_bar(&sm.o_done[jl & 1], (jl >> 1) & 1, abort));
      if (!ok) break;
      tc::fence_after_sync();
      const float inv = valid ? 1.0f / l : 0.0f;
      OutT* orow = static_cast<OutT*>(p.out) +
                   ((size_t)(x.q0 + x.t0 + tok) * p.num_heads + (size_t)x.kvh * g + tid % g) * kD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float ov[32];
        tc::tmem_ld32(tmem + lane_off + 256 + 32 * c, ov);
        tc::tmem_wait_ld();
        if (valid) {
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
      tc::named_sync(1, 128);
      if (tid == 0) mbar_arrive(&sm.o_free);
    }
    if (!ok && tid == 0) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
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
                    offsetof(Smem, pmat) % 1024 == 0,
                "swizzled buffers must start on 1024-byte boundaries");
  auto kern = prefill_tc_kernel<QT>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    configured = true;
  }
  // an upper bound of the items: every sequence's tiles, times the KV heads
  const long long rows = (long long)total_q * p.group + (long long)p.num_seqs * (kRowsM - 1);
  const long long items = rows / kRowsM * p.num_kv_heads;
  int grid = sm_count();
  if (items < grid) grid = (int)(items > 0 ? items : 1);
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
