// CPU oracle for paged KV-cache attention.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
// statement of what the paged attention path computes.  Only the test suite,
// the package smoke check and the CPU-baseline leg of the benchmark load it.
// It shares no code, header, table or constant generator with the CUDA
// library; the two meet only at the seeded inputs.
//
// Arithmetic is IEEE double for attention (the plain definition), IEEE float
// only where the method fixes it: the FP8 cache write divides a float by a
// float scale before rounding to E4M3.
//
// Sources (page title, section):
//  [P2]  openeuler.csdn.net, PagedAttention notes: "显存占用计算",
//        "机制1：按需分配", "机制 2：写时复制", "Block Table 数据结构",
//        "Attention 计算时的 Block 映射（CUDA Kernel 伪代码）".
//  [P1]  "第34讲 … vLLM 生产级系统架构全景剖析与四重加速引擎", §1.2
//        (KVCacheManager.allocate_slots / free in reverse order, BlockPool,
//        ref_cnt, FreeKVCacheBlockQueue), §2.2 (longest-prefix match, ref_cnt),
//        §2.3 (cached-free blocks, LRU eviction), §4.4 (FP8 E4M3 KV cache).
//  [P3]  "第32讲 … Prefill vs Decode …", §3.1 (softmax(QK^T/sqrt(d_k))V and
//        the decode step), §3.2 (per-token KV bytes), §3.4 (GQA grouping),
//        §5.4 (chunked prefill).
//  [P5]  devpress.csdn.net vLLM overview, "3、PagedAttention (3)" (block pool
//        with a free list), "8、推理流程" (K/V written into the cache, then
//        attention), "9、FlashAttention (4)" (online softmax: max, sum_exp,
//        rescale).
//
// Readings where the pages are silent (each also listed in the design notes):
//  * cache layout [num_blocks][num_kv_heads][block_size][head_dim];
//  * query head h reads KV head h / (H / H_kv) (consecutive groups, [P3] §3.4);
//  * context_lens include the token(s) being attended from, whose K/V the
//    cache write has already stored;
//  * a prefill-chunk query at absolute position pos sees keys 0..pos;
//  * a sequence with no context yields a zero output row;
//  * negative slots are padding and are skipped;
//  * FP8 uses one fp32 scale per tensor: stored = E4M3_RNE_SAT(x / scale),
//    read back as decode(stored) * scale.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <vector>

namespace {

// Element formats (these numbers are part of the data interface).
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

int elem_bytes(int dtype) { return dtype == ORC_E4M3 ? 1 : 2; }

// IEEE 754 binary16: 1 sign, 5 exponent bits (bias 15), 10 fraction bits.
double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = std::ldexp((double)f, -24);  // subnormal: f * 2^-14 * 2^-10
  } else if (e == 31) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = std::ldexp(1.0 + f / 1024.0, e - 15);
  }
  return sign ? -mag : mag;
}

// bfloat16: 1 sign, 8 exponent bits (bias 127), 7 fraction bits.
double decode_bf16(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int f = b & 0x7f;
  double mag;
  if (e == 0) {
    mag = std::ldexp((double)f, -133);  // f * 2^-126 * 2^-7
  } else if (e == 255) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = std::ldexp(1.0 + f / 128.0, e - 127);
  }
  return sign ? -mag : mag;
}

// OCP 8-bit floating point, E4M3 ("FN"): 1 sign, 4 exponent bits (bias 7),
// 3 fraction bits; exponent 0 is subnormal; S.1111.111 is NaN; no infinity.
// Largest finite magnitude 1.75 * 2^8 = 448.
double decode_e4m3(uint8_t x) {
  int sign = (x >> 7) & 1;
  int e = (x >> 3) & 0xf;
  int f = x & 0x7;
  double mag;
  if (e == 15 && f == 7) {
    mag = NAN;
  } else if (e == 0) {
    mag = std::ldexp((double)f, -9);  // f/8 * 2^(1-7)
  } else {
    mag = std::ldexp(1.0 + f / 8.0, e - 7);
  }
  return sign ? -mag : mag;
}

// Round a float to the nearest E4M3 value, ties to even, saturating finite
// values (and infinities) to +-448.  NaN maps to the NaN code.
uint8_t encode_e4m3(float xf) {
  double x = (double)xf;
  uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  if (std::isnan(x)) return (uint8_t)(sign | 0x7f);
  double a = std::fabs(x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  if (a == 0.0) return sign;
  // Spacing of representable values around a: 2^(e-3) for normal binade
  // [2^e, 2^(e+1)), e >= -6; subnormals share the spacing 2^-9.
  int e = (int)std::floor(std::log2(a));
  // log2 can be off by one at exact powers of two; correct it.
  if (std::ldexp(1.0, e) > a) e -= 1;
  if (std::ldexp(1.0, e + 1) <= a) e += 1;
  if (e < -6) e = -6;
  double quantum = std::ldexp(1.0, e - 3);
  double n = a / quantum;  // exact: a has <= 24 significant bits
  double fl = std::floor(n);
  double rem = n - fl;
  double k;
  if (rem > 0.5) {
    k = fl + 1.0;
  } else if (rem < 0.5) {
    k = fl;
  } else {
    k = (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  }
  double r = k * quantum;  // the rounded magnitude
  if (r > 448.0) r = 448.0;  // cannot happen below 448, kept for clarity
  if (r == 0.0) return sign;
  // Encode r exactly.
  int re = (int)std::floor(std::log2(r));
  if (std::ldexp(1.0, re) > r) re -= 1;
  if (std::ldexp(1.0, re + 1) <= r) re += 1;
  uint8_t code;
  if (re < -6) {
    // subnormal: r = f * 2^-9
    int f = (int)(r / std::ldexp(1.0, -9));
    code = (uint8_t)f;
  } else {
    int f = (int)((r / std::ldexp(1.0, re) - 1.0) * 8.0);
    code = (uint8_t)(((re + 7) << 3) | f);
  }
  return (uint8_t)(sign | code);
}

double decode_elem(const uint8_t* base, size_t idx, int dtype) {
  if (dtype == ORC_E4M3) return decode_e4m3(base[idx]);
  uint16_t bits;
  std::memcpy(&bits, base + 2 * idx, 2);
  return dtype == ORC_F16 ? decode_f16(bits) : decode_bf16(bits);
}

// ---------------------------------------------------------------------------
// Block pool and per-sequence block tables ([P5] "3、PagedAttention (3)";
// [P1] §1.2; [P2] "Block Table 数据结构", "机制 2：写时复制").
struct Pool {
  int num_blocks;
  std::vector<int> free_list;  // popped from the back
  std::vector<int> ref_cnt;
};

struct Seq {
  Pool* pool;
  int block_size;
  int num_tokens;
  std::vector<int> table;  // logical block j -> physical block id
};

int pool_alloc(Pool* p) {
  if (p->free_list.empty()) return -1;
  int id = p->free_list.back();
  p->free_list.pop_back();
  p->ref_cnt[id] = 1;
  return id;
}

int pool_decref(Pool* p, int id) {
  if (id < 0 || id >= p->num_blocks || p->ref_cnt[id] <= 0) return -1;
  if (--p->ref_cnt[id] == 0) p->free_list.push_back(id);
  return 0;
}

struct CacheView {
  uint8_t* k;
  uint8_t* v;
  size_t block_bytes;  // bytes of one physical block in one cache
};

// One attention of a single query row over keys 0..n_keys-1 of a sequence,
// gathered through its block table ([P2] CUDA-kernel pseudocode:
// block_idx = i // block_size, offset = i % block_size,
// physical_block = block_table[block_idx]).  The result is the plain
// definition softmax(scale * q K^T) V ([P3] §3.1), evaluated in double with
// the two-pass form: m = max z, w = exp(z - m), o = sum(w v) / sum(w).
// Returns 0, or -1 when a table entry names a block outside the pool.
int attend_row(double* out, const double* q, const int32_t* table, int n_keys,
               const uint8_t* k_cache, const uint8_t* v_cache, int kv_head,
               int num_kv_heads, int head_dim, int block_size, int num_blocks,
               double scale, int kv_dtype, double k_scale, double v_scale,
               double* lse_out) {
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (n_keys <= 0) {
    if (lse_out) *lse_out = -INFINITY;
    return 0;
  }
  const bool fp8 = kv_dtype == ORC_E4M3;
  std::vector<double> z(n_keys);
  for (int t = 0; t < n_keys; ++t) {
    int blk = table[t / block_size];
    if (blk < 0 || blk >= num_blocks) return -1;
    size_t row = ((size_t)blk * num_kv_heads + kv_head) * block_size + t % block_size;
    double acc = 0.0;
    for (int d = 0; d < head_dim; ++d) {
      double kd = decode_elem(k_cache, row * head_dim + d, kv_dtype);
      if (fp8) kd *= k_scale;
      acc += q[d] * kd;
    }
    z[t] = scale * acc;
  }
  double m = z[0];
  for (int t = 1; t < n_keys; ++t) m = z[t] > m ? z[t] : m;
  double l = 0.0;
  for (int t = 0; t < n_keys; ++t) {
    double w = std::exp(z[t] - m);
    l += w;
    int blk = table[t / block_size];
    size_t row = ((size_t)blk * num_kv_heads + kv_head) * block_size + t % block_size;
    for (int d = 0; d < head_dim; ++d) {
      double vd = decode_elem(v_cache, row * head_dim + d, kv_dtype);
      if (fp8) vd *= v_scale;
      out[d] += w * vd;
    }
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= l;
  if (lse_out) *lse_out = m + std::log(l);
  return 0;
}

// The same definition over an explicit set of key positions of the sequence
// (ascending): used for tree-masked chunks, where a query sees the prior
// context and only some of the chunk's own keys.
int attend_keys(double* out, const double* q, const int32_t* table, const std::vector<int>& keys,
                const uint8_t* k_cache, const uint8_t* v_cache, int kv_head, int num_kv_heads,
                int head_dim, int block_size, int num_blocks, double scale, int kv_dtype,
                double k_scale, double v_scale) {
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  const int n = (int)keys.size();
  if (n == 0) return 0;
  const bool fp8 = kv_dtype == ORC_E4M3;
  std::vector<double> z(n);
  for (int i = 0; i < n; ++i) {
    const int t = keys[i];
    int blk = table[t / block_size];
    if (blk < 0 || blk >= num_blocks) return -1;
    size_t row = ((size_t)blk * num_kv_heads + kv_head) * block_size + t % block_size;
    double acc = 0.0;
    for (int d = 0; d < head_dim; ++d) {
      double kd = decode_elem(k_cache, row * head_dim + d, kv_dtype);
      if (fp8) kd *= k_scale;
      acc += q[d] * kd;
    }
    z[i] = scale * acc;
  }
  double m = z[0];
  for (int i = 1; i < n; ++i) m = z[i] > m ? z[i] : m;
  double l = 0.0;
  for (int i = 0; i < n; ++i) {
    const int t = keys[i];
    double w = std::exp(z[i] - m);
    l += w;
    int blk = table[t / block_size];
    size_t row = ((size_t)blk * num_kv_heads + kv_head) * block_size + t % block_size;
    for (int d = 0; d < head_dim; ++d) {
      double vd = decode_elem(v_cache, row * head_dim + d, kv_dtype);
      if (fp8) vd *= v_scale;
      out[d] += w * vd;
    }
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= l;
  return 0;
}

bool dtype_ok(int dt) { return dt == ORC_F16 || dt == ORC_BF16 || dt == ORC_E4M3; }

}  // namespace

extern "C" {

// ---- codecs ---------------------------------------------------------------
double orc_decode_f16(uint16_t h) { return decode_f16(h); }
double orc_decode_bf16(uint16_t b) { return decode_bf16(b); }
double orc_decode_e4m3(uint8_t x) { return decode_e4m3(x); }
uint8_t orc_encode_e4m3(float x) { return encode_e4m3(x); }

void orc_decode_array(double* out, const void* src, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) out[i] = decode_elem((const uint8_t*)src, (size_t)i, dtype);
}

void orc_encode_e4m3_array(uint8_t* out, const float* src, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = encode_e4m3(src[i]);
}

// ---- byte model ([P3] §3.2; [P2] "显存占用计算") ---------------------------
// K and V, for every layer, every KV head, every head dimension.
uint64_t orc_kv_bytes_per_token(int layers, int kv_heads, int head_dim, int bytes_per_elem) {
  return 2ull * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim *
         (uint64_t)bytes_per_elem;
}

// Blocks a sequence of n tokens occupies: one block per started group of
// block_size tokens ([P2] "机制1：按需分配": ceil(100/16) = 7).
int64_t orc_blocks_for_tokens(int64_t n, int block_size) {
  int64_t blocks = 0;
  for (int64_t t = 0; t < n; ++t)
    if (t % block_size == 0) ++blocks;
  return blocks;
}

// ---- pool -----------------------------------------------------------------
// free_order (may be NULL) lists the block ids in the order they will be
// handed out; NULL hands out 0, 1, 2, ...
void* orc_pool_create(int num_blocks, const int32_t* free_order) {
  if (num_blocks < 0) return nullptr;
  Pool* p = new Pool;
  p->num_blocks = num_blocks;
  p->ref_cnt.assign(num_blocks, 0);
  p->free_list.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) {
    int id = free_order ? free_order[i] : i;
    p->free_list[num_blocks - 1 - i] = id;  // back of the vector = next out
  }
  return p;
}

void orc_pool_destroy(void* pool) { delete (Pool*)pool; }
int orc_pool_alloc(void* pool) { return pool_alloc((Pool*)pool); }
int orc_pool_decref(void* pool, int id) { return pool_decref((Pool*)pool, id); }
int orc_pool_incref(void* pool, int id) {
  Pool* p = (Pool*)pool;
  if (id < 0 || id >= p->num_blocks || p->ref_cnt[id] <= 0) return -1;
  ++p->ref_cnt[id];
  return 0;
}
int orc_pool_ref_cnt(void* pool, int id) {
  Pool* p = (Pool*)pool;
  if (id < 0 || id >= p->num_blocks) return -1;
  return p->ref_cnt[id];
}
int orc_pool_num_free(void* pool) { return (int)((Pool*)pool)->free_list.size(); }

// ---- sequences --------------------------------------------------------------
void* orc_seq_create(void* pool, int block_size) {
  if (!pool || block_size <= 0) return nullptr;
  Seq* s = new Seq;
  s->pool = (Pool*)pool;
  s->block_size = block_size;
  s->num_tokens = 0;
  return s;
}

// Releases the sequence's blocks tail first, so that prefix blocks are the
// last to go back ([P1] §1.2, KVCacheManager.free), then deletes it.
void orc_seq_destroy(void* seq) {
  Seq* s = (Seq*)seq;
  if (!s) return;
  for (int j = (int)s->table.size() - 1; j >= 0; --j) pool_decref(s->pool, s->table[j]);
  delete s;
}

// A new sequence sharing every block of seq by reference (ref_cnt + 1 each),
// as parallel samples share their prompt ([P2] "机制 2：写时复制").
void* orc_seq_fork(void* seq) {
  Seq* s = (Seq*)seq;
  Seq* c = new Seq(*s);
  for (int id : c->table) ++c->pool->ref_cnt[id];
  return c;
}

// Appends n tokens ([P2] BlockTable.append_token: a new block whenever the
// token count is a multiple of block_size; [P1] §1.2 allocate_slots: fill the
// last block first).  Before a token is written into a block that other
// sequences still reference, that block is copied on write: a fresh block
// receives the bytes of every head of the K and V caches (when the caches
// are given), the shared block loses one reference, and the table points at
// the copy.  slots_out (may be NULL) receives the slot of each new token,
// physical_block * block_size + offset ([P2] get_physical_indices).
// cache_block_bytes is the size of one physical block of one cache.
// Returns 0, or -1 if the pool ran out (tokens appended before that stay).
int orc_seq_append(void* seq, int n, uint8_t* k_cache, uint8_t* v_cache,
                   int64_t cache_block_bytes, int64_t* slots_out) {
  Seq* s = (Seq*)seq;
  for (int i = 0; i < n; ++i) {
    int pos = s->num_tokens;
    int j = pos / s->block_size;
    if (pos % s->block_size == 0) {
      int id = pool_alloc(s->pool);
      if (id < 0) return -1;
      s->table.push_back(id);
    } else if (s->pool->ref_cnt[s->table[j]] > 1) {
      int old = s->table[j];
      int id = pool_alloc(s->pool);
      if (id < 0) return -1;
      if (k_cache && cache_block_bytes > 0) {
        std::memcpy(k_cache + (size_t)id * cache_block_bytes,
                    k_cache + (size_t)old * cache_block_bytes, (size_t)cache_block_bytes);
      }
      if (v_cache && cache_block_bytes > 0) {
        std::memcpy(v_cache + (size_t)id * cache_block_bytes,
                    v_cache + (size_t)old * cache_block_bytes, (size_t)cache_block_bytes);
      }
      pool_decref(s->pool, old);
      s->table[j] = id;
    }
    if (slots_out) slots_out[i] = (int64_t)s->table[j] * s->block_size + pos % s->block_size;
    s->num_tokens = pos + 1;
  }
  return 0;
}

int orc_seq_num_tokens(void* seq) { return ((Seq*)seq)->num_tokens; }
int orc_seq_num_blocks(void* seq) { return (int)((Seq*)seq)->table.size(); }

// Copies up to max entries of the block table; returns the number of blocks.
int orc_seq_table(void* seq, int32_t* out, int max) {
  Seq* s = (Seq*)seq;
  int n = (int)s->table.size();
  for (int j = 0; j < n && j < max; ++j) out[j] = s->table[j];
  return n;
}

// Slot of logical position pos, or -1 if pos is not a token of the sequence.
int64_t orc_seq_slot(void* seq, int pos) {
  Seq* s = (Seq*)seq;
  if (pos < 0 || pos >= s->num_tokens) return -1;
  return (int64_t)s->table[pos / s->block_size] * s->block_size + pos % s->block_size;
}

// ---- cache write ([P5] "8、推理流程": the layer's K and V are stored into the
// paged cache; [P2] slot = physical_block * block_size + offset) -------------
// k, v: [num_tokens][num_kv_heads][head_dim] in src_dtype (f16 or bf16).
// Caches: [num_blocks][num_kv_heads][block_size][head_dim] in cache_dtype.
// Same dtype: the element bits are copied.  E4M3: E4M3_RNE_SAT(float(x) / s)
// with an IEEE float division.
// Returns 0; -1 bad argument; -2 a slot outside the pool; -3 duplicate slot.
int orc_reshape_and_cache(const void* k, const void* v, uint8_t* k_cache, uint8_t* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, int src_dtype,
                          int cache_dtype, float k_scale, float v_scale) {
  if (src_dtype != ORC_F16 && src_dtype != ORC_BF16) return -1;
  if (cache_dtype != src_dtype && cache_dtype != ORC_E4M3) return -1;
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  std::vector<char> seen((size_t)num_slots, 0);
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) return -2;
    if (seen[(size_t)slot]) return -3;
    seen[(size_t)slot] = 1;
  }
  const int cb = elem_bytes(cache_dtype);
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      size_t src_row = ((size_t)t * num_kv_heads + h) * head_dim;
      size_t dst_row = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
      for (int half = 0; half < 2; ++half) {
        const uint8_t* src = (const uint8_t*)(half ? v : k);
        uint8_t* dst = half ? v_cache : k_cache;
        float sc = half ? v_scale : k_scale;
        for (int d = 0; d < head_dim; ++d) {
          if (cache_dtype == src_dtype) {
            std::memcpy(dst + (dst_row + d) * cb, src + (src_row + d) * 2, 2);
          } else {
            float x = (float)decode_elem(src, src_row + d, src_dtype);
            dst[dst_row + d] = encode_e4m3(x / sc);
          }
        }
      }
    }
  }
  return 0;
}

// ---- decode attention -------------------------------------------------------
// out: [num_seqs][num_heads][head_dim] double.  q: [num_seqs][num_heads][head_dim]
// in q_dtype.  Query head h reads KV head h / (num_heads / num_kv_heads).
// Every query attends the first context_lens[s] tokens of its sequence.
// Returns 0; -1 bad argument; -2 a block id outside the pool.
int orc_paged_attention_decode(double* out, const void* q, const uint8_t* k_cache,
                               const uint8_t* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, int num_seqs, int num_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               int max_blocks_per_seq, int num_blocks, double scale,
                               int q_dtype, int kv_dtype, double k_scale, double v_scale) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
  if (!dtype_ok(q_dtype) || q_dtype == ORC_E4M3 || !dtype_ok(kv_dtype)) return -1;
  const int group = num_heads / num_kv_heads;
  std::vector<double> qrow(head_dim);
  for (int s = 0; s < num_seqs; ++s) {
    int ctx = context_lens[s];
    if (ctx < 0 || ctx > max_blocks_per_seq * block_size) return -1;
    const int32_t* table = block_tables + (size_t)s * max_blocks_per_seq;
    for (int h = 0; h < num_heads; ++h) {
      size_t row = (size_t)s * num_heads + h;
      for (int d = 0; d < head_dim; ++d)
        qrow[d] = decode_elem((const uint8_t*)q, row * head_dim + d, q_dtype);
      if (attend_row(out + row * head_dim, qrow.data(), table, ctx, k_cache, v_cache,
                     h / group, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     kv_dtype, k_scale, v_scale, nullptr))
        return -2;
    }
  }
  return 0;
}

// The same attention evaluated the partitioned way: the context is cut into
// pieces of partition_size tokens, each piece gives a normalised partial
// output o_p and its log-sum-exp lse_p, and the pieces are combined with
// weights exp(lse_p - L), L = log(sum_p exp(lse_p)).  This is the exact
// reformulation of the per-block combination that [P5] "3、PagedAttention (3)"
// sketches, with the renormalisation of [P5] "9、FlashAttention (4)".
int orc_paged_attention_decode_partitioned(double* out, const void* q, const uint8_t* k_cache,
                                           const uint8_t* v_cache, const int32_t* block_tables,
                                           const int32_t* context_lens, int num_seqs,
                                           int num_heads, int num_kv_heads, int head_dim,
                                           int block_size, int max_blocks_per_seq,
                                           int num_blocks, double scale, int q_dtype,
                                           int kv_dtype, double k_scale, double v_scale,
                                           int partition_size) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
  if (partition_size <= 0 || partition_size % block_size != 0) return -1;
  if (!dtype_ok(q_dtype) || q_dtype == ORC_E4M3 || !dtype_ok(kv_dtype)) return -1;
  const int group = num_heads / num_kv_heads;
  const int pb = partition_size / block_size;
  std::vector<double> qrow(head_dim), part(head_dim);
  for (int s = 0; s < num_seqs; ++s) {
    int ctx = context_lens[s];
    if (ctx < 0 || ctx > max_blocks_per_seq * block_size) return -1;
    const int32_t* table = block_tables + (size_t)s * max_blocks_per_seq;
    int np = (ctx + partition_size - 1) / partition_size;
    for (int h = 0; h < num_heads; ++h) {
      size_t row = (size_t)s * num_heads + h;
      double* o = out + row * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        qrow[d] = decode_elem((const uint8_t*)q, row * head_dim + d, q_dtype);
        o[d] = 0.0;
      }
      std::vector<double> lse(np);
      std::vector<double> parts((size_t)np * head_dim);
      for (int p = 0; p < np; ++p) {
        int n = ctx - p * partition_size;
        if (n > partition_size) n = partition_size;
        if (attend_row(parts.data() + (size_t)p * head_dim, qrow.data(), table + p * pb, n,
                       k_cache, v_cache, h / group, num_kv_heads, head_dim, block_size,
                       num_blocks, scale, kv_dtype, k_scale, v_scale, &lse[p]))
          return -2;
      }
      if (np == 0) continue;
      double mx = lse[0];
      for (int p = 1; p < np; ++p) mx = lse[p] > mx ? lse[p] : mx;
      double sum = 0.0;
      for (int p = 0; p < np; ++p) sum += std::exp(lse[p] - mx);
      double L = mx + std::log(sum);
      for (int p = 0; p < np; ++p) {
        double w = std::exp(lse[p] - L);
        for (int d = 0; d < head_dim; ++d) o[d] += w * parts[(size_t)p * head_dim + d];
      }
    }
  }
  return 0;
}

// ---- chunked-prefill attention ([P3] §5.4) ---------------------------------
// q, out: [total_q][num_heads][head_dim]; sequence s owns query rows
// query_start_loc[s] .. query_start_loc[s+1]-1, which are its last
// q_len = query_start_loc[s+1] - query_start_loc[s] tokens, so query i sits
// at absolute position pos = context_lens[s] - q_len + i and attends keys
// 0..pos (causal).  Returns 0; -1 bad argument; -2 a block id outside the pool.
int orc_paged_attention_prefill(double* out, const void* q, const uint8_t* k_cache,
                                const uint8_t* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, const int32_t* query_start_loc,
                                int num_seqs, int total_q, int num_heads, int num_kv_heads,
                                int head_dim, int block_size, int max_blocks_per_seq,
                                int num_blocks, double scale, int q_dtype, int kv_dtype,
                                double k_scale, double v_scale) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
  if (!dtype_ok(q_dtype) || q_dtype == ORC_E4M3 || !dtype_ok(kv_dtype)) return -1;
  if (query_start_loc[0] != 0 || query_start_loc[num_seqs] != total_q) return -1;
  const int group = num_heads / num_kv_heads;
  std::vector<double> qrow(head_dim);
  for (int s = 0; s < num_seqs; ++s) {
    int q0 = query_start_loc[s], q_len = query_start_loc[s + 1] - q0;
    int ctx = context_lens[s];
    if (q_len < 0 || q_len > ctx || ctx > max_blocks_per_seq * block_size) return -1;
    const int32_t* table = block_tables + (size_t)s * max_blocks_per_seq;
    for (int i = 0; i < q_len; ++i) {
      int pos = ctx - q_len + i;
      for (int h = 0; h < num_heads; ++h) {
        size_t row = (size_t)(q0 + i) * num_heads + h;
        for (int d = 0; d < head_dim; ++d)
          qrow[d] = decode_elem((const uint8_t*)q, row * head_dim + d, q_dtype);
        if (attend_row(out + row * head_dim, qrow.data(), table, pos + 1, k_cache, v_cache,
                       h / group, num_kv_heads, head_dim, block_size, num_blocks, scale,
                       kv_dtype, k_scale, v_scale, nullptr))
          return -2;
      }
    }
  }
  return 0;
}

// Tree-masked chunk attention, for verifying a tree of draft tokens
// ([P2] "MEDUSA推理框架", "Tree Attention": candidate tokens of several heads
// form a tree verified in one pass under an attention mask; "EAGLE2推理",
// "重排阶段": the mask is adjusted so that each token sees only its
// ancestors).  Sequence s's chunk holds q_len <= 64 draft tokens at positions
// base = ctx - q_len .. ctx - 1; query i sees every key before base, and the
// chunk key base + j when bit j of tree_mask[q0 + i] is set (its ancestors
// and itself).  A mask with bits 0..i for every i is ordinary causal prefill.
int orc_paged_attention_prefill_tree(double* out, const void* q, const uint8_t* k_cache,
                                     const uint8_t* v_cache, const int32_t* block_tables,
                                     const int32_t* context_lens, const int32_t* query_start_loc,
                                     const uint64_t* tree_mask, int num_seqs, int total_q,
                                     int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_blocks_per_seq, int num_blocks,
                                     double scale, int q_dtype, int kv_dtype, double k_scale,
                                     double v_scale) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
  if (!dtype_ok(q_dtype) || q_dtype == ORC_E4M3 || !dtype_ok(kv_dtype)) return -1;
  if (query_start_loc[0] != 0 || query_start_loc[num_seqs] != total_q) return -1;
  const int group = num_heads / num_kv_heads;
  std::vector<double> qrow(head_dim);
  std::vector<int> keys;
  for (int s = 0; s < num_seqs; ++s) {
    int q0 = query_start_loc[s], q_len = query_start_loc[s + 1] - q0;
    int ctx = context_lens[s];
    if (q_len < 0 || q_len > 64 || q_len > ctx || ctx > max_blocks_per_seq * block_size)
      return -1;
    const int32_t* table = block_tables + (size_t)s * max_blocks_per_seq;
    const int base = ctx - q_len;
    for (int i = 0; i < q_len; ++i) {
      keys.clear();
      for (int t = 0; t < base; ++t) keys.push_back(t);
      for (int j = 0; j < q_len; ++j)
        if ((tree_mask[q0 + i] >> j) & 1u) keys.push_back(base + j);
      for (int h = 0; h < num_heads; ++h) {
        size_t row = (size_t)(q0 + i) * num_heads + h;
        for (int d = 0; d < head_dim; ++d)
          qrow[d] = decode_elem((const uint8_t*)q, row * head_dim + d, q_dtype);
        if (attend_keys(out + row * head_dim, qrow.data(), table, keys, k_cache, v_cache,
                        h / group, num_kv_heads, head_dim, block_size, num_blocks, scale,
                        kv_dtype, k_scale, v_scale))
          return -2;
      }
    }
  }
  return 0;
}

}  // extern "C"

// ===========================================================================
// Prefix-caching block pool ([P1] §1.2 BlockPool, FreeKVCacheBlockQueue,
// KVCacheManager.allocate_slots / free; §2.2 longest-prefix match with ref_cnt;
// §2.3 cached-free blocks and LRU eviction).
//
// Written for plainness, not speed: the free queue is a vector searched
// linearly, and a cached block is keyed by its whole token prefix (every token
// from the sequence's start through the block's last), so equal keys mean
// equal contents by definition.
//
// Readings where the pages are silent:
//  * only full blocks are cached; a block is registered when its last slot is
//    filled;
//  * when a prefix is already registered to another block, the new block
//    stays unregistered (the first copy keeps serving hits);
//  * a match stops before the block holding the prompt's last token, so at
//    least one token is always left to compute;
//  * every block whose count drops to 0 goes to the queue's tail, registered
//    or not; allocation takes the head and drops the head's registration
//    (eviction).  A fresh pool's queue holds blocks 0, 1, 2, ... in order.
namespace {

struct CachePool {
  int num_blocks = 0, block_size = 0;
  std::vector<int> queue;                    // free blocks; front = next out
  std::vector<int> ref_cnt;
  std::vector<std::vector<int32_t>> key;     // registered prefix (empty: none)
  std::map<std::vector<int32_t>, int> cached;  // prefix -> block
};

struct CacheReq {
  CachePool* pool = nullptr;
  std::vector<int32_t> tokens;  // the request's tokens so far
  std::vector<int> table;       // logical block -> physical block
};

// A block leaves the free queue (wherever it is) and gains a reference.
void cp_take(CachePool* p, int id) {
  if (p->ref_cnt[id] == 0) {
    for (size_t i = 0; i < p->queue.size(); ++i) {
      if (p->queue[i] == id) {
        p->queue.erase(p->queue.begin() + i);
        break;
      }
    }
  }
  ++p->ref_cnt[id];
}

// The head of the queue, its registration dropped; -1 when the queue is empty.
int cp_alloc(CachePool* p) {
  if (p->queue.empty()) return -1;
  int id = p->queue.front();
  p->queue.erase(p->queue.begin());
  if (!p->key[id].empty()) {
    p->cached.erase(p->key[id]);
    p->key[id].clear();
  }
  p->ref_cnt[id] = 1;
  return id;
}

void cp_release(CachePool* p, int id) {
  if (--p->ref_cnt[id] == 0) p->queue.push_back(id);
}

}  // namespace

extern "C" {

void* orc_cpool_create(int num_blocks, int block_size) {
  if (num_blocks < 0 || block_size <= 0) return nullptr;
  CachePool* p = new CachePool;
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->ref_cnt.assign(num_blocks, 0);
  p->key.assign(num_blocks, {});
  for (int i = 0; i < num_blocks; ++i) p->queue.push_back(i);
  return p;
}

void orc_cpool_destroy(void* pool) { delete (CachePool*)pool; }
int orc_cpool_num_free(void* pool) { return (int)((CachePool*)pool)->queue.size(); }
int orc_cpool_num_cached(void* pool) { return (int)((CachePool*)pool)->cached.size(); }

int orc_cpool_ref_cnt(void* pool, int id) {
  CachePool* p = (CachePool*)pool;
  return id < 0 || id >= p->num_blocks ? -1 : p->ref_cnt[id];
}

// 1 when the block holds a registered prefix, 0 when not, -1 for a bad id.
int orc_cpool_is_cached(void* pool, int id) {
  CachePool* p = (CachePool*)pool;
  return id < 0 || id >= p->num_blocks ? -1 : (p->key[id].empty() ? 0 : 1);
}

// Copies up to max entries of the free queue, head first; returns its length.
int orc_cpool_queue(void* pool, int32_t* out, int max) {
  CachePool* p = (CachePool*)pool;
  int n = (int)p->queue.size();
  for (int i = 0; i < n && i < max; ++i) out[i] = p->queue[i];
  return n;
}

void* orc_creq_create(void* pool) {
  if (!pool) return nullptr;
  CacheReq* r = new CacheReq;
  r->pool = (CachePool*)pool;
  return r;
}

// Longest cached prefix of tokens[0..n) in whole blocks, for a request that
// holds no tokens yet: each hit block gains a reference (leaving the free
// queue if it was there) and joins the table.  Returns the number of tokens
// matched (a multiple of block_size, at most n - 1), or -1 if the request is
// not empty.
int orc_creq_match(void* req, const int32_t* tokens, int n) {
  CacheReq* r = (CacheReq*)req;
  CachePool* p = r->pool;
  if (!r->tokens.empty() || !r->table.empty()) return -1;
  int matched = 0;
  for (int end = p->block_size; end <= n - 1; end += p->block_size) {
    std::vector<int32_t> prefix(tokens, tokens + end);
    auto it = p->cached.find(prefix);
    if (it == p->cached.end()) break;
    cp_take(p, it->second);
    r->table.push_back(it->second);
    matched = end;
  }
  r->tokens.assign(tokens, tokens + matched);
  return matched;
}

// Appends n tokens with the given ids ([P1] §1.2 allocate_slots): the last
// block is filled first, then new blocks are taken from the queue's head.  If
// the last block is partial and shared with a forked request, it is copied
// on write first: cow_out (may be NULL) receives {source, copy}, or {-1, -1}
// when no copy was needed.  slots_out (may be NULL) receives each token's
// slot.  Blocks that become full are registered under their prefix.
// All or nothing: returns -1, changing nothing, when the queue holds fewer
// blocks than the append needs; 0 otherwise.
int orc_creq_append(void* req, const int32_t* ids, int n, int64_t* slots_out, int32_t* cow_out) {
  CacheReq* r = (CacheReq*)req;
  CachePool* p = r->pool;
  const int bs = p->block_size;
  const int t0 = (int)r->tokens.size();
  if (cow_out) cow_out[0] = cow_out[1] = -1;
  if (n <= 0) return n == 0 ? 0 : -1;
  const bool cow = t0 % bs != 0 && p->ref_cnt[r->table.back()] > 1;
  int need = cow ? 1 : 0;
  for (int pos = t0; pos < t0 + n; ++pos) need += pos % bs == 0 ? 1 : 0;
  if (need > (int)p->queue.size()) return -1;
  if (cow) {
    const int old = r->table.back();
    const int id = cp_alloc(p);
    cp_release(p, old);
    r->table.back() = id;
    if (cow_out) {
      cow_out[0] = old;
      cow_out[1] = id;
    }
  }
  for (int i = 0; i < n; ++i) {
    const int pos = t0 + i;
    if (pos % bs == 0) r->table.push_back(cp_alloc(p));
    const int id = r->table[pos / bs];
    if (slots_out) slots_out[i] = (int64_t)id * bs + pos % bs;
    r->tokens.push_back(ids[i]);
    if (pos % bs == bs - 1 && p->cached.find(r->tokens) == p->cached.end()) {
      p->cached[r->tokens] = id;
      p->key[id] = r->tokens;
    }
  }
  return 0;
}

// The copy half of copy-on-write ([P2] "机制 2：写时复制": the writer gets a
// private copy of the shared block before it writes): for each pair
// (source, destination) in order, the destination block's bytes in each cache
// become the source block's.  block_bytes is one block of one cache.
// Returns 0, or -1 (nothing copied) when an id is outside the pool.
int orc_copy_blocks(uint8_t* k_cache, uint8_t* v_cache, const int32_t* pairs, int num_pairs,
                    int num_blocks, int64_t block_bytes) {
  for (int i = 0; i < 2 * num_pairs; ++i)
    if (pairs[i] < 0 || pairs[i] >= num_blocks) return -1;
  for (int i = 0; i < num_pairs; ++i) {
    const size_t src = (size_t)pairs[2 * i] * block_bytes, dst = (size_t)pairs[2 * i + 1] * block_bytes;
    std::memmove(k_cache + dst, k_cache + src, (size_t)block_bytes);
    std::memmove(v_cache + dst, v_cache + src, (size_t)block_bytes);
  }
  return 0;
}

// A request sharing every block of req by reference ([P2] "机制 2：写时复制").
void* orc_creq_fork(void* req) {
  CacheReq* r = (CacheReq*)req;
  CacheReq* c = new CacheReq(*r);
  for (int id : c->table) ++c->pool->ref_cnt[id];
  return c;
}

// Releases the request's blocks tail first ([P1] §1.2 free) and deletes it.
void orc_creq_free(void* req) {
  CacheReq* r = (CacheReq*)req;
  if (!r) return;
  for (int j = (int)r->table.size() - 1; j >= 0; --j) cp_release(r->pool, r->table[j]);
  delete r;
}

int orc_creq_num_tokens(void* req) { return (int)((CacheReq*)req)->tokens.size(); }

int orc_creq_table(void* req, int32_t* out, int max) {
  CacheReq* r = (CacheReq*)req;
  int n = (int)r->table.size();
  for (int j = 0; j < n && j < max; ++j) out[j] = r->table[j];
  return n;
}

}  // extern "C"
