"""Seeded synthetic inputs for the paged KV-cache attention path.

This module is shared by the CUDA path's callers (tests, benchmark) and by the
CPU oracle's tests.  It only draws random numbers and lays out input indices:
which physical block each logical block of a sequence lives in, which source
token row each cache slot receives, context and query lengths.  It holds none
of the attention arithmetic.

Input recipe (one attention layer per workload):
  * numpy PCG64 with the given seed for every structural choice;
  * the pool's free list is a seeded random permutation, so block tables are
    scattered over the pool;
  * K/V/Q values are N(0,1) drawn in fp32 and rounded (round-to-nearest-even)
    to fp16/bf16; on CPU from numpy PCG64, on a GPU from torch's seeded
    device generator (Philox);
  * pools hold 1.25x the blocks the sequences need unless a size is given.

Slots follow the cache layout [num_blocks][num_kv_heads][block_size][head_dim]:
slot = physical_block * block_size + offset.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F16, BF16, E4M3 = 0, 1, 2
BLOCK_SIZE = 16


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


@dataclass
class Workload:
    """One batch of sequences over one paged K/V cache.

    Sequence s has context_lens[s] tokens, the last q_lens[s] of which are
    queries (1 for a decode sequence, a chunk for a prefill sequence).  Token
    position t of sequence s holds source row seq_rows[s][t] of the K/V source
    tensors; the cache is filled by writing source row fill_rows[i] to slot
    fill_slots[i] (set-up), and the step's own new tokens are new_rows[i] to
    new_slots[i] (timed).
    """

    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    q_dtype: int
    kv_dtype: int
    num_blocks: int
    context_lens: np.ndarray  # [S] int32
    q_lens: np.ndarray  # [S] int32
    block_tables: np.ndarray  # [S, MB] int32, padded with valid but unused ids
    seq_rows: list  # per sequence: int64 [ctx] source row of each position
    num_src_rows: int
    fill_rows: np.ndarray  # int64
    fill_slots: np.ndarray  # int64
    new_rows: np.ndarray  # int64
    new_slots: np.ndarray  # int64
    scale: float
    partition_size: int = 512
    block_size: int = BLOCK_SIZE
    src_dtype: int = BF16
    seed: int = 0
    shared_groups: list = field(default_factory=list)  # lists of sequence ids sharing a prompt

    @property
    def num_seqs(self) -> int:
        return len(self.context_lens)

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == E4M3 else 2

    def decode_ids(self) -> np.ndarray:
        return np.nonzero(self.q_lens == 1)[0]

    def prefill_ids(self) -> np.ndarray:
        return np.nonzero(self.q_lens > 1)[0]

    def cascade_groups(self):
        """Cascade-decode grouping of the decode sequences (in decode_ids
        order): (group_start [G + 1] int32, prefix_lens [S] int32).  Consecutive
        members of one sharing group form a group whose prefix is their common
        leading blocks (whole blocks within every member's context); runs of
        other sequences form groups with no shared prefix."""
        ids = [int(s) for s in self.decode_ids()]
        group_of = {s: gi for gi, g in enumerate(self.shared_groups) for s in g}
        starts, prefix = [0], np.zeros(len(ids), np.int32)
        i = 0
        while i < len(ids):
            gi = group_of.get(ids[i])
            j = i + 1
            if gi is not None:
                while j < len(ids) and group_of.get(ids[j]) == gi:
                    j += 1
            k = 0
            if j - i > 1:
                tabs = [self.block_tables[s] for s in ids[i:j]]
                n = min(int(self.context_lens[s]) for s in ids[i:j]) // BLOCK_SIZE
                while k < n and all(t[k] == tabs[0][k] for t in tabs):
                    k += 1
            if k == 0:  # nothing shared: extend the run of unshared sequences
                while j < len(ids) and (group_of.get(ids[j]) is None or
                                        len(self.shared_groups[group_of[ids[j]]]) < 2):
                    j += 1
            prefix[i:j] = k * BLOCK_SIZE
            starts.append(j)
            i = j
        return np.asarray(starts, np.int32), prefix

    def kv_read_bytes(self, ids=None) -> int:
        """Bytes of K and V one decode pass reads: every context token, once per KV head."""
        ids = self.decode_ids() if ids is None else ids
        toks = int(self.context_lens[ids].astype(np.int64).sum())
        return toks * 2 * self.num_kv_heads * self.head_dim * self.kv_elem_bytes


class _Allocator:
    """Hands out block ids in the order of a seeded permutation."""

    def __init__(self, order: np.ndarray):
        self.order = order
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        if self.next + n > len(self.order):
            raise ValueError("synthetic pool too small")
        out = self.order[self.next:self.next + n]
        self.next += n
        return out


def _slots(table: np.ndarray, positions: np.ndarray) -> np.ndarray:
    positions = np.asarray(positions, dtype=np.int64)
    return table[positions // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + positions % BLOCK_SIZE


def _assemble(name, r, ctx, q_lens, tables, seq_rows, num_src, fill_rows, fill_slots,
              num_blocks, H, Hkv, D, q_dtype, kv_dtype, src_dtype, seed, groups=(),
              partition_size=512):
    S = len(ctx)
    mb = max(1, max(len(t) for t in tables))
    bt = r.integers(0, num_blocks, size=(S, mb), dtype=np.int64).astype(np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    new_rows, new_slots = [], []
    for s in range(S):
        pos = np.arange(max(0, ctx[s] - q_lens[s]), ctx[s], dtype=np.int64)
        new_rows.append(seq_rows[s][pos])
        new_slots.append(_slots(np.asarray(tables[s]), pos))
    return Workload(
        name=name, num_heads=H, num_kv_heads=Hkv, head_dim=D, q_dtype=q_dtype,
        kv_dtype=kv_dtype, num_blocks=num_blocks,
        context_lens=np.asarray(ctx, dtype=np.int32), q_lens=np.asarray(q_lens, dtype=np.int32),
        block_tables=bt, seq_rows=seq_rows, num_src_rows=num_src,
        fill_rows=np.concatenate(fill_rows).astype(np.int64) if fill_rows else np.zeros(0, np.int64),
        fill_slots=np.concatenate(fill_slots).astype(np.int64) if fill_slots else np.zeros(0, np.int64),
        new_rows=np.concatenate(new_rows).astype(np.int64),
        new_slots=np.concatenate(new_slots).astype(np.int64),
        scale=1.0 / math.sqrt(D), partition_size=partition_size, src_dtype=src_dtype, seed=seed,
        shared_groups=[list(g) for g in groups])


def independent(name: str, seed: int, context_lens, H: int, Hkv: int, D: int, q_dtype: int,
                kv_dtype: int, q_lens=None, num_blocks: int | None = None,
                pool_factor: float = 1.25, partition_size: int = 512) -> Workload:
    """Sequences with private blocks only, scattered by a seeded permutation."""
    r = rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    q_lens = np.ones(len(ctx), np.int64) if q_lens is None else np.asarray(q_lens, np.int64)
    need = [-(-int(c) // BLOCK_SIZE) for c in ctx]
    demand = sum(need)
    nb = num_blocks if num_blocks is not None else max(1, int(math.ceil(pool_factor * demand)))
    alloc = _Allocator(r.permutation(nb).astype(np.int32))
    tables, seq_rows, fill_rows, fill_slots = [], [], [], []
    base = 0
    for s, c in enumerate(ctx):
        t = alloc.take(need[s])
        tables.append(t)
        rows = np.arange(base, base + c, dtype=np.int64)
        seq_rows.append(rows)
        prior = max(0, c - q_lens[s])
        fill_rows.append(rows[:prior])
        fill_slots.append(_slots(t, np.arange(prior)))
        base += c
    src = kv_dtype if kv_dtype != E4M3 else q_dtype
    return _assemble(name, r, ctx, q_lens, tables, seq_rows, base, fill_rows, fill_slots, nb,
                     H, Hkv, D, q_dtype, kv_dtype, src, seed, partition_size=partition_size)


def shared_prefix(name: str, seed: int, prompt_lens, tail_lens, H: int, Hkv: int, D: int,
                  q_dtype: int, kv_dtype: int, num_blocks: int | None = None,
                  pool_factor: float = 1.25) -> Workload:
    """Groups of parallel samples of one prompt.

    The prompt's full blocks are stored once and referenced by every sample of
    the group; a partial last prompt block is copied into each sample's first
    private block (copy on write), which then continues with the sample's own
    tail tokens.  prompt_lens[g] is the prompt of group g; tail_lens[g] lists
    the private tail length of each of its samples (>= 1 each).
    """
    r = rng(seed)
    groups, tables, seq_rows, ctx = [], [], [], []
    plan = []
    demand = 0
    for P, tails in zip(prompt_lens, tail_lens):
        full = P // BLOCK_SIZE
        demand += full
        for tl in tails:
            demand += -(-(P + tl - full * BLOCK_SIZE) // BLOCK_SIZE)
        plan.append((P, tails, full))
    nb = num_blocks if num_blocks is not None else max(1, int(math.ceil(pool_factor * demand)))
    alloc = _Allocator(r.permutation(nb).astype(np.int32))
    fill_rows, fill_slots = [], []
    base = 0
    for P, tails, full in plan:
        shared = alloc.take(full)
        prompt_rows = np.arange(base, base + P, dtype=np.int64)
        base += P
        nshared = full * BLOCK_SIZE
        fill_rows.append(prompt_rows[:nshared])
        fill_slots.append(_slots(shared, np.arange(nshared)))
        g = []
        for tl in tails:
            c = P + tl
            priv = alloc.take(-(-(c - nshared) // BLOCK_SIZE))
            table = np.concatenate([shared, priv]).astype(np.int32)
            rows = np.concatenate([prompt_rows, np.arange(base, base + tl, dtype=np.int64)])
            base += tl
            # the sample's private blocks: the rest of the prompt, then its tail
            # (all but the newest token, which the timed step writes)
            pos = np.arange(nshared, c - 1, dtype=np.int64)
            fill_rows.append(rows[pos])
            fill_slots.append(_slots(table, pos))
            g.append(len(tables))
            tables.append(table)
            seq_rows.append(rows)
            ctx.append(c)
        groups.append(g)
    q_lens = np.ones(len(ctx), np.int64)
    return _assemble(name, r, np.asarray(ctx, np.int64), q_lens, tables, seq_rows, base,
                     fill_rows, fill_slots, nb, H, Hkv, D, q_dtype, kv_dtype,
                     kv_dtype if kv_dtype != E4M3 else q_dtype, seed, groups=groups)


# ---- draft trees (speculative verification) ------------------------------------
def random_tree(r, n: int) -> np.ndarray:
    """Parents of an n-node draft tree in topological order: node 0 is the
    root (parent -1), every other node's parent has a smaller index."""
    parents = np.full(n, -1, np.int64)
    for i in range(1, n):
        parents[i] = r.integers(0, i)
    return parents


def tree_mask(parents) -> np.ndarray:
    """Per node, a 64-bit mask of the chunk keys it may see: itself and its
    ancestors (bit j = node j).  A chain (parent i - 1) gives bits 0..i."""
    n = len(parents)
    assert n <= 64
    m = np.zeros(n, np.uint64)
    for i in range(n):
        m[i] = np.uint64(1) << np.uint64(i)
        if parents[i] >= 0:
            m[i] |= m[parents[i]]
    return m


# ---- the named workloads ------------------------------------------------------
def tiny(seed: int = 0) -> Workload:
    """4 sequences, 4 q heads = 4 kv heads, head_dim 64, fp16, 64-block pool,
    context lengths uniform on [1, 100], scale 1/8."""
    r = rng(seed)
    ctx = r.integers(1, 101, size=4)
    return independent("tiny", seed, ctx, 4, 4, 64, F16, F16, num_blocks=64)


def llama2_7b(seed: int = 1, num_seqs: int = 64, context: int = 4096) -> Workload:
    """LLaMA-2-7B-shaped decode: 64 x 4096 tokens, 32 q = 32 kv heads, head_dim 128, bf16."""
    return independent("llama2-7b decode", seed, [context] * num_seqs, 32, 32, 128, BF16, BF16)


def gqa70b_shared(seed: int = 2, num_seqs: int = 128, group: int = 3) -> Workload:
    """70B-GQA-shaped decode with prefix sharing: 128 sequences, 64 q / 8 kv heads,
    head_dim 128, bf16.  Samples come in groups of 3 (the remainder forms a
    smaller group).  Prompt lengths are lognormal with median 2000 (sigma 1),
    clipped so that prompt + tail stays within [16, 32768]; each sample adds a
    private tail of U[1, 128] tokens."""
    r = rng(seed)
    sizes = [group] * (num_seqs // group) + ([num_seqs % group] if num_seqs % group else [])
    prompts, tails = [], []
    for gsz in sizes:
        P = int(round(float(np.exp(r.normal(math.log(2000.0), 1.0)))))
        P = min(max(P, 16), 32768 - 128)
        prompts.append(P)
        tails.append([int(x) for x in r.integers(1, 129, size=gsz)])
    return shared_prefix("70b-gqa decode shared-prefix", seed, prompts, tails, 64, 8, 128,
                         BF16, BF16)


def mixed(seed: int = 3, num_decode: int = 32, num_prefill: int = 4, chunk: int = 512,
          prior: int = 2048, kv_dtype: int = BF16) -> Workload:
    """Mixed chunked-prefill batch: 32 decode sequences (context U[1024, 8192]) and
    4 prefill chunks of 512 queries over 2048 prior tokens; 32 q / 8 kv heads,
    head_dim 128, bf16 (the cache in kv_dtype).  The decode sequences come first."""
    r = rng(seed)
    dctx = r.integers(1024, 8193, size=num_decode)
    ctx = np.concatenate([dctx, np.full(num_prefill, prior + chunk)])
    q_lens = np.concatenate([np.ones(num_decode, np.int64), np.full(num_prefill, chunk)])
    name = "mixed chunked-prefill" + (", e4m3 cache" if kv_dtype == E4M3 else "")
    return independent(name, seed, ctx, 32, 8, 128, BF16, kv_dtype, q_lens=q_lens)


def mixed_fp8(seed: int = 3) -> Workload:
    """The mixed chunked-prefill batch over an E4M3 cache (per-tensor scales)."""
    return mixed(seed, kv_dtype=E4M3)


def long_fp8(seed: int = 4, num_seqs: int = 8, context: int = 131072) -> Workload:
    """Long-context split-K decode: 8 x 131072 tokens, 32 q / 8 kv heads, head_dim 128,
    bf16 queries, E4M3 K/V cache with per-tensor fp32 scales, 512-token partitions."""
    return independent("long-context fp8 split-k decode", seed, [context] * num_seqs, 32, 8, 128,
                       BF16, E4M3, partition_size=512)


def llama2_7b_x16(seed: int = 1) -> Workload:
    """The LLaMA-2-7B decode shape with 16 sequences (1.07 GB of K/V): a smaller
    case of the same kernel for detailed profiling."""
    return llama2_7b(seed, num_seqs=16)


def long_fp8_x2(seed: int = 4) -> Workload:
    """The long-context FP8 shape with 2 sequences (0.54 GB of K/V): a smaller
    case of the same kernel for detailed profiling."""
    return long_fp8(seed, num_seqs=2)


NAMED = {
    "tiny": tiny,
    "llama2_7b": llama2_7b,
    "llama2_7b_x16": llama2_7b_x16,
    "gqa70b_shared": gqa70b_shared,
    "mixed": mixed,
    "mixed_fp8": mixed_fp8,
    "long_fp8": long_fp8,
    "long_fp8_x2": long_fp8_x2,
}


# ---- values --------------------------------------------------------------------
def _round_bits(x32: np.ndarray, dtype: int) -> np.ndarray:
    """fp32 -> fp16/bf16 round-to-nearest-even, returned as uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    t = t.to(torch.float16 if dtype == F16 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def normal_bits(seed: int, shape, dtype: int) -> np.ndarray:
    """N(0,1) in fp32 from PCG64(seed), rounded to fp16/bf16 bits (CPU)."""
    x = rng(seed).standard_normal(size=shape, dtype=np.float32)
    return _round_bits(x, dtype)


def values_cpu(w: Workload):
    """(k_src, v_src, q) as uint16 bit arrays: [rows, Hkv, D], [rows, Hkv, D], [TQ, H, D]."""
    shp = (w.num_src_rows, w.num_kv_heads, w.head_dim)
    k = normal_bits(w.seed * 1000 + 11, shp, w.src_dtype)
    v = normal_bits(w.seed * 1000 + 12, shp, w.src_dtype)
    q = normal_bits(w.seed * 1000 + 13, (int(w.q_lens.sum()), w.num_heads, w.head_dim), w.q_dtype)
    return k, v, q


def values_device(w: Workload, device):
    """(k_src, v_src, q) as torch fp16/bf16 tensors drawn on `device` with a seeded
    torch generator (used where the CPU draw would be slow)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1000 + 17)
    sd = torch.float16 if w.src_dtype == F16 else torch.bfloat16
    qd = torch.float16 if w.q_dtype == F16 else torch.bfloat16
    shp = (w.num_src_rows, w.num_kv_heads, w.head_dim)
    k = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(sd)
    v = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(sd)
    q = torch.randn((int(w.q_lens.sum()), w.num_heads, w.head_dim), generator=g, device=device,
                    dtype=torch.float32).to(qd)
    return k, v, q


def token_kv(seed: int, tokens, positions, Hkv: int, D: int, dtype: int, vocab: int = 1024,
             max_pos: int = 8192):
    """(k, v) bits [n, Hkv, D] for tokens at positions: per-token and
    per-position N(0,1) embeddings (fp32, from PCG64(seed)) summed and rounded,
    so equal (token, position) pairs always give equal K/V, as a cached prefix
    block must."""
    r = rng(seed)
    et = r.standard_normal(size=(2, vocab, Hkv, D), dtype=np.float32)
    ep = r.standard_normal(size=(2, max_pos, Hkv, D), dtype=np.float32)
    t = np.asarray(tokens, np.int64) % vocab
    p = np.asarray(positions, np.int64)
    return (_round_bits(et[0, t] + ep[0, p], dtype), _round_bits(et[1, t] + ep[1, p], dtype))


def query_start_loc(q_lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(q_lens, np.int64))]).astype(np.int32)
