// Paged attention on CUDA cores, for any group size up to 16: one CTA per
// (row, KV head, partition of the row's context).
//
// Sources: openeuler.csdn.net PagedAttention notes, "Attention 计算时的 Block
// 映射（CUDA Kernel 伪代码）" (the per-token gather through the block table);
// devpress.csdn.net vLLM overview, "3、PagedAttention (3)" (per-block partial
// results that are then combined) and "9、FlashAttention (4)" (max and sum of
// exponentials, rescaled); "第32讲 … Prefill vs Decode …", §3.4 (each K/V head
// serves a group of query heads).
//
// Design (GB300):
//  * Each (block, KV head) K or V tile is one contiguous 16 x head_dim run
//    (cache layout [block][kv_head][16][head_dim]), so it arrives in shared
//    memory through a single 1-D bulk async copy (cp.async.bulk, mbarrier
//    completion).  Every warp owns a ring of stages and streams its own tiles
//    (blocks w, w+4, ... of the partition: first all K tiles, then all V
//    tiles), so no cross-warp handshake sits on the copy path and the V tiles
//    are already in flight while the last K tiles are scored.
//  * All query heads of the KV head's group are handled together, so each K/V
//    tile is read from HBM once per KV head.
//  * Scores: a lane owns a 16-byte column chunk of a tile and a subset of its
//    rows; partial dot products are summed over the lanes of a row with a
//    shuffle reduce-scatter (each step halves the vector a lane carries).
//  * Softmax is exact per partition (max, then exp2, then sum) in shared
//    memory; partitions of one row are combined by the log-sum-exp merge.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "rows.cuh"

namespace pkv {

constexpr int kSimtWarps = 4;
constexpr int kSimtThreads = kSimtWarps * 32;
constexpr int kMaxPartition = 512;

template <class KVT, int D, int G>
struct SimtGeom {
  static constexpr int kRow = D * KVT::kBytes;   // bytes of one token row
  static constexpr int kTile = 16 * kRow;        // bytes of one (block, head) tile
  static constexpr int kLpr = kRow / 16;         // lanes per row (16-byte chunks)
  static constexpr int kEpl = 16 / KVT::kBytes;  // elements per lane chunk
  static constexpr int kRpi = 32 / kLpr;         // rows per warp-wide access
  static constexpr int kTpl = 16 / kRpi;         // rows per lane per tile
  // Groups of at most 2 (matrix-vector work, bound by the bytes in flight):
  // four CTAs per SM with about 12 KB of tiles in flight per warp; a CTA's
  // ring fills at its start and drains at its end, and four CTAs in different
  // phases keep more of the SM's 192 KB in flight than two with 24 KB per warp
  // (LLaMA-2-7B decode 0.6385 -> 0.5989 ms).  Larger groups need the
  // registers of two CTAs per SM (four would spill) and keep 24 KB per warp.
  static constexpr int kCtasPerSm = G <= 2 ? 4 : 2;
  static constexpr int kStagesRaw = (G <= 2 ? 12288 : 24576) / kTile;
  static constexpr int kStages = kStagesRaw > 16 ? 16 : (kStagesRaw < 2 ? 2 : kStagesRaw);
  static constexpr int kRingBytes = kSimtWarps * kStages * kTile;
  static constexpr int kBarBytes = kSimtWarps * kStages * 8;
};

template <class KVT, int D, int G>
size_t simt_smem_bytes(int partition) {
  using Geo = SimtGeom<KVT, D, G>;
  size_t ring = Geo::kRingBytes;
  size_t red = (size_t)kSimtWarps * G * D * sizeof(float);  // reuses the ring at the end
  if (red > ring) ring = red;
  return ring + Geo::kBarBytes + 2 * G * sizeof(float) + (size_t)G * partition * sizeof(float);
}

// Sum each entry of v over the kLanes lanes that differ in the low bits of the
// lane id (xor masks kLanes/2 .. 1), halving the carried vector at every step
// while it has more than one entry.  Returns the index of the first original
// entry the lane now holds; the lane holds max(1, V / kLanes) entries.
template <int kLanes, int V>
__device__ __forceinline__ int reduce_scatter(float (&v)[V], int lane) {
  int base = 0;
#pragma unroll
  for (int step = 0; (kLanes >> (step + 1)) >= 1; ++step) {
    const int m = kLanes >> (step + 1);
    const int len = V >> step;
    if (len > 1) {
      const int half = len / 2;
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int j = 0; j < half; ++j) {
        const float send = upper ? v[j] : v[j + half];
        const float keep = upper ? v[j + half] : v[j];
        v[j] = keep + __shfl_xor_sync(kFull, send, m);
      }
      if (upper) base += half;
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], m);
    }
  }
  return base;
}

template <class QT, int N>
__device__ __forceinline__ void load_q(const typename QT::T* src, float* f, float scale) {
  static_assert(N % 8 == 0, "q chunks are 8 elements");
#pragma unroll
  for (int i = 0; i < N / 8; ++i) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + i);
    to_float(w, f + 8 * i, QT());
  }
#pragma unroll
  for (int e = 0; e < N; ++e) f[e] *= scale;
}

template <class QT, class KVT, int D, int G>
__global__ void __launch_bounds__(kSimtThreads, (SimtGeom<KVT, D, G>::kCtasPerSm))
    paged_attention_simt_kernel(const AttnParams p) {
  using Geo = SimtGeom<KVT, D, G>;
  constexpr int LPR = Geo::kLpr, EPL = Geo::kEpl, RPI = Geo::kRpi, TPL = Geo::kTpl;
  constexpr int STAGES = Geo::kStages, TILE = Geo::kTile, ROW = Geo::kRow;
  constexpr int V0 = TPL * G;
  constexpr int KLEN = V0 >= LPR ? V0 / LPR : 1;

  extern __shared__ __align__(1024) uint8_t smem[];
  size_t ring_bytes = Geo::kRingBytes;
  if ((size_t)kSimtWarps * G * D * sizeof(float) > ring_bytes)
    ring_bytes = (size_t)kSimtWarps * G * D * sizeof(float);
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes);
  float* s_m = reinterpret_cast<float*>(smem + ring_bytes + Geo::kBarBytes);
  float* s_l = s_m + G;
  float* logits = s_l + G;  // [G][partition]
  __shared__ int s_abort;

  const int row = blockIdx.x, kvh = blockIdx.y, part = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.partition;
  int seq;
  const int keys = row_keys(p, row, &seq);
  const int start = part * P;
  const bool split = p.max_parts > 1;
  const int nparts = (keys + P - 1) / P;
  using OutT = typename QT::T;

  if (start >= keys) {
    // Nothing to attend in this partition.  A row with no keys at all gets
    // zeros here when no merge follows (the merge writes them otherwise).
    if (!split && part == 0) {
      OutT* o = static_cast<OutT*>(p.out) + ((size_t)row * p.num_heads + kvh * p.group) * D;
      for (int i = threadIdx.x; i < p.group * D; i += kSimtThreads) store_out(o + i, 0.0f);
    }
    return;
  }
  const int n = min(P, keys - start);  // tokens of this partition
  const int nblk = (n + kBlockSize - 1) / kBlockSize;
  const int32_t* table = p.block_tables + (size_t)seq * p.max_blocks_per_seq + start / kBlockSize;

  if (threadIdx.x == 0) s_abort = 0;
  uint64_t* my_bars = bars + warp * STAGES;
  uint8_t* my_ring = ring + (size_t)warp * STAGES * TILE;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(&my_bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // This warp's tiles: blocks warp, warp+4, ...; K tiles first, then V tiles.
  const int nw = nblk > warp ? (nblk - warp + kSimtWarps - 1) / kSimtWarps : 0;
  const int ntiles = 2 * nw;
  auto issue = [&](int u) {
    const int st = u % STAGES;
    const bool is_v = u >= nw;
    const int j = warp + kSimtWarps * (is_v ? u - nw : u);
    int blk = __ldg(table + j);
    if (blk < 0 || blk >= p.num_blocks) {
      flag_error(p.errors, PKV_DEVERR_BLOCK_ID);
      blk = 0;
    }
    const uint8_t* src = (is_v ? p.v_cache : p.k_cache) + ((size_t)blk * p.num_kv_heads + kvh) * TILE;
    mbar_arrive_expect_tx(&my_bars[st], TILE);
    bulk_g2s(my_ring + (size_t)st * TILE, src, TILE, &my_bars[st]);
  };
  int issued = 0;
  if (lane == 0) {
    for (; issued < STAGES && issued < ntiles; ++issued) issue(issued);
  }

  const int c = lane % LPR, r = lane / LPR;
  // Query chunk of every head of the group, pre-scaled into base-2 units.
  float qr[G][EPL];
  {
    const typename QT::T* qbase = static_cast<const typename QT::T*>(p.q) +
                                  ((size_t)row * p.num_heads + (size_t)kvh * p.group) * D + c * EPL;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (h < p.group) {
        load_q<QT, EPL>(qbase + (size_t)h * D, qr[h], p.q_scale);
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) qr[h][e] = 0.0f;
      }
    }
  }
  __syncthreads();  // s_abort initialised

  // ---- scores: K tiles ----------------------------------------------------
  bool ok = true;
  int u = 0;
  for (; u < nw; ++u) {
    const int st = u % STAGES;
    if (!mbar_wait(&my_bars[st], (u / STAGES) & 1)) {
      ok = false;
      break;
    }
    const uint8_t* tile = my_ring + (size_t)st * TILE;
    float acc[V0];
#pragma unroll
    for (int i = 0; i < V0; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int i = 0; i < TPL; ++i) {
      const int t = r + RPI * i;
      const uint4 w = *reinterpret_cast<const uint4*>(tile + t * ROW + c * 16);
      float kf[EPL];
      to_float(w, kf, KVT());
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) a = fmaf(qr[h][e], kf[e], a);
        acc[i * G + h] = a;
      }
    }
    const int base = reduce_scatter<LPR, V0>(acc, lane);
    const int tok0 = (warp + kSimtWarps * u) * kBlockSize;
#pragma unroll
    for (int j = 0; j < KLEN; ++j) {
      const int idx = base + j;
      const int i = idx / G, h = idx % G;
      const int tok = tok0 + r + RPI * i;
      logits[h * P + tok] = tok < n ? acc[j] : -INFINITY;
    }
    __syncwarp();
    if (lane == 0 && issued < ntiles) {
      fence_proxy_async_smem();
      issue(issued++);
    }
  }
  if (!ok) {
    flag_error(p.errors, PKV_DEVERR_TIMEOUT);
    s_abort = 1;
  }
  __syncthreads();

  // ---- softmax over the partition: one warp per head -----------------------
  if (!s_abort) {
    for (int h = warp; h < p.group; h += kSimtWarps) {
      float* lh = logits + h * P;
      float m = -INFINITY;
      for (int t = lane; t < n; t += 32) m = fmaxf(m, lh[t]);
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      float sum = 0.0f;
      for (int t = lane; t < nblk * kBlockSize; t += 32) {
        const float e = t < n ? fast_exp2(lh[t] - m) : 0.0f;
        lh[t] = e;
        sum += e;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
      if (lane == 0) {
        s_m[h] = m;
        s_l[h] = sum;
      }
    }
  }
  __syncthreads();

  // ---- weighted sum of V tiles ----------------------------------------------
  float o[G][EPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[h][e] = 0.0f;
  const bool run = ok && !s_abort;
  if (run) {
    for (; u < ntiles; ++u) {
      const int st = u % STAGES;
      if (!mbar_wait(&my_bars[st], (u / STAGES) & 1)) {
        ok = false;
        break;
      }
      const uint8_t* tile = my_ring + (size_t)st * TILE;
      const int tok0 = (warp + kSimtWarps * (u - nw)) * kBlockSize;
#pragma unroll
      for (int i = 0; i < TPL; ++i) {
        const int t = r + RPI * i;
        const int tok = tok0 + t;
        if (tok < n) {
          const uint4 w = *reinterpret_cast<const uint4*>(tile + t * ROW + c * 16);
          float vf[EPL];
          to_float(w, vf, KVT());
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float pw = logits[h * P + tok];
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(pw, vf[e], o[h][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && issued < ntiles) {
        fence_proxy_async_smem();
        issue(issued++);
      }
    }
  }
  if (!ok || !run) {
    // Leave no copy of ours in flight: wait briefly for what was issued.
    if (!ok) flag_error(p.errors, PKV_DEVERR_TIMEOUT);
    for (int x = u; x < issued; ++x) mbar_wait(&my_bars[x % STAGES], (x / STAGES) & 1, 10000000ull);
  }

  // Sum over the lanes of a column chunk (they covered different rows).
#pragma unroll
  for (int m = LPR; m < 32; m <<= 1)
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[h][e] += __shfl_xor_sync(kFull, o[h][e], m);
  __syncthreads();  // every warp is done with the ring; reuse it for the reduction
  float* red = reinterpret_cast<float*>(ring);  // [warps][G][D]
  if (r == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < EPL; ++e) red[(warp * G + h) * D + c * EPL + e] = o[h][e];
  }
  __syncthreads();
  if (s_abort || !ok) return;

  const bool direct = !split || nparts == 1;
  for (int idx = threadIdx.x; idx < p.group * D; idx += kSimtThreads) {
    const int h = idx / D, d = idx - h * D;
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) acc += red[(w * G + h) * D + d];
    const float val = acc * (p.v_scale / s_l[h]);
    const size_t head = (size_t)row * p.num_heads + (size_t)kvh * p.group + h;
    if (direct) {
      store_out(static_cast<OutT*>(p.out) + head * D + d, val);
    } else {
      p.o_part[(head * p.max_parts + part) * D + d] = val;
      if (d == 0) p.lse[head * p.max_parts + part] = s_m[h] + log2f(s_l[h]);
    }
  }
}

template <class QT, class KVT, int D, int G>
int launch_simt_one(const AttnParams& p, cudaStream_t stream) {
  const size_t smem = simt_smem_bytes<KVT, D, G>(p.partition);
  auto kern = paged_attention_simt_kernel<QT, KVT, D, G>;
  static bool configured = false;  // per instantiation
  if (!configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)simt_smem_bytes<KVT, D, G>(kMaxPartition)) != cudaSuccess)
      return PKV_ERR_CUDA;
    configured = true;
  }
  dim3 grid(p.num_rows, p.num_kv_heads, p.max_parts);
  kern<<<grid, kSimtThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <class QT, class KVT>
int launch_simt_typed(const AttnParams& p, int head_dim, int g_pad, cudaStream_t s) {
#define PKV_G_CASES(DIM)                                      \
  switch (g_pad) {                                            \
    case 1: return launch_simt_one<QT, KVT, DIM, 1>(p, s);    \
    case 2: return launch_simt_one<QT, KVT, DIM, 2>(p, s);    \
    case 4: return launch_simt_one<QT, KVT, DIM, 4>(p, s);    \
    case 8: return launch_simt_one<QT, KVT, DIM, 8>(p, s);    \
    case 16: return launch_simt_one<QT, KVT, DIM, 16>(p, s);  \
    default: return PKV_ERR_UNSUPPORTED;                      \
  }
  if (head_dim == 64) {
    PKV_G_CASES(64)
  } else if (head_dim == 128) {
    PKV_G_CASES(128)
  }
#undef PKV_G_CASES
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
