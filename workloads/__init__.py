"""Seeded synthetic inputs for paged-attention decode.

This module only *generates* inputs: sequence lengths, block tables drawn from a
shuffled free list, and fp16 N(0, 1) query / key / value values.  It holds none
of the attention arithmetic, so both the CPU oracle and the CUDA path can take
their inputs from it without sharing any of the method's code.

Recipes follow the pages on vLLM:

* KV blocks hold 16 tokens each and a sequence's blocks need not be contiguous;
  a per-sequence block table maps logical block -> physical block
  ("vLLM 2026 推理引擎全解", §2.1; mjmagnets.cn vLLM tutorial, §2.1-§2.2).
* Blocks are taken one by one from a free list, ceil(tokens / block_size) per
  request, and exhausting the list is an out-of-memory error (doramagic.ai vLLM
  manual, "KVCacheManager 缓存管理").  Shuffling the list first gives the
  scattered placement the workloads ask for.
* Requests sharing a system prompt point their first table entries at the same
  physical blocks ("vLLM 2026 推理引擎全解", §2.3).
* The cache layout is [num_blocks, num_heads, block_size, head_dim]
  ("vLLM 2026 推理引擎全解", §2.2, the kernel sketch's k_cache comment).

Slots that no context covers (the tail of a sequence's last block and every
spare block of the pool) are filled with fp16 NaN, so that any read of them
shows up in the output.
"""
from __future__ import annotations

import math
import os
from collections import deque
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

BLOCK_SIZE = 16
# Normals are drawn in independently seeded chunks so that generation can run
# on all host cores while the values stay independent of the thread count.
_CHUNK = 1 << 22
F16_NAN = np.float16(np.nan)
BF16_NAN_BITS = np.uint16(0x7FC0)  # a quiet NaN in bfloat16
# Storage dtype per element type: fp16 arrays are numpy float16; bf16 arrays
# are uint16 arrays holding the bfloat16 bit patterns (numpy has no bfloat16).
STORAGE = {"f16": np.float16, "bf16": np.uint16}


class OutOfBlocks(RuntimeError):
    """The free list ran dry while building block tables."""


@dataclass
class DecodeCase:
    """One batch of decode inputs, all host numpy arrays.

    Shapes: q [S, H, D] fp16; k_cache / v_cache [N, H, B, D] fp16;
    block_tables [S, MB] int32 (entries past a sequence's last block are -1);
    context_lens [S] int32.  The optional new-token fields feed
    reshape_and_cache: k_new / v_new [T, H, D] fp16, slot_mapping [T] int32
    with slot = physical_block * B + offset.
    """

    name: str
    seed: int
    num_heads: int
    head_dim: int
    block_size: int
    scale: float
    context_lens: np.ndarray
    block_tables: np.ndarray
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    k_new: Optional[np.ndarray] = None
    v_new: Optional[np.ndarray] = None
    slot_mapping: Optional[np.ndarray] = None
    shared_prefix_blocks: int = 0
    meta: dict = field(default_factory=dict)
    dtype: str = "f16"
    # prefill cases: q holds total_q rows; sequence s owns rows
    # query_start[s] .. query_start[s + 1] - 1, its last tokens
    query_start: Optional[np.ndarray] = None

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_new_tokens(self) -> int:
        return 0 if self.slot_mapping is None else int(self.slot_mapping.shape[0])

    def blocks_used(self) -> np.ndarray:
        """Logical blocks each sequence covers: ceil(ctx / B)."""
        return (self.context_lens.astype(np.int64) + self.block_size - 1) // self.block_size


# ----------------------------------------------------------------------------
# random values
# ----------------------------------------------------------------------------

def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns of finite float32 values, rounded to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def fill_normal(out: np.ndarray, seed: int, stream: int) -> None:
    """Fill a contiguous fp16 array (or a uint16 array of bf16 bits) with
    seeded N(0, 1) draws rounded to the element type.

    Chunk i of stream `stream` uses Philox seeded by SeedSequence(seed,
    spawn_key=(stream,)).spawn(...)[i], so the values do not depend on how many
    threads run the chunks.
    """
    flat = out.reshape(-1)
    n = flat.size
    if n == 0:
        return
    nchunks = (n + _CHUNK - 1) // _CHUNK
    children = np.random.SeedSequence(seed, spawn_key=(stream,)).spawn(nchunks)

    def work(i: int) -> None:
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.Generator(np.random.Philox(children[i]))
        draws = g.standard_normal(hi - lo, dtype=np.float32)
        if flat.dtype == np.uint16:
            flat[lo:hi] = f32_to_bf16_bits(draws)
        else:
            flat[lo:hi] = draws

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))


fill_normal_f16 = fill_normal  # the name used before bf16 support


# ----------------------------------------------------------------------------
# block tables
# ----------------------------------------------------------------------------

def blocks_needed(num_tokens: int, block_size: int = BLOCK_SIZE) -> int:
    """ceil(tokens / block_size), the allocation rule of the KV cache manager."""
    return (int(num_tokens) + block_size - 1) // block_size


def allocate_tables(context_lens: np.ndarray, block_size: int, num_blocks: int,
                    max_blocks_per_seq: int, rng: np.random.Generator,
                    shared_prefix_blocks: int = 0) -> np.ndarray:
    """Block tables taken in sequence order from a shuffled free list.

    With shared_prefix_blocks = P > 0, the first P blocks popped form a common
    prefix that every sequence's table starts with; each sequence then pops its
    private blocks.  Unused table entries are -1.
    """
    S = int(context_lens.shape[0])
    free = deque(int(b) for b in rng.permutation(num_blocks))
    tables = np.full((S, max_blocks_per_seq), -1, dtype=np.int32)

    def pop() -> int:
        if not free:
            raise OutOfBlocks("KV cache exhausted")
        return free.popleft()

    prefix = [pop() for _ in range(shared_prefix_blocks)]
    for s in range(S):
        nb = blocks_needed(context_lens[s], block_size)
        if nb > max_blocks_per_seq:
            raise ValueError(f"sequence {s} needs {nb} blocks > max_blocks_per_seq")
        row = prefix[:min(nb, shared_prefix_blocks)]
        row += [pop() for _ in range(nb - len(row))]
        tables[s, :nb] = row
    return tables


def poison_unused(case: DecodeCase) -> None:
    """Write NaN into every cache slot that no sequence's context covers."""
    B = case.block_size
    covered = np.zeros((case.num_blocks, B), dtype=bool)
    for s in range(case.num_seqs):
        ctx = int(case.context_lens[s])
        nb = blocks_needed(ctx, B)
        for b in range(nb):
            phys = int(case.block_tables[s, b])
            n = min(B, ctx - b * B)
            covered[phys, :n] = True
    blk, off = np.nonzero(~covered)
    nan = BF16_NAN_BITS if case.dtype == "bf16" else F16_NAN
    for cache in (case.k_cache, case.v_cache):
        cache[blk, :, off, :] = nan


# ----------------------------------------------------------------------------
# cases
# ----------------------------------------------------------------------------

def build_case(name: str, context_lens, *, num_heads: int, head_dim: int,
               seed: int, block_size: int = BLOCK_SIZE,
               num_blocks: Optional[int] = None, spare_frac: float = 0.10,
               max_blocks_per_seq: Optional[int] = None,
               shared_prefix_blocks: int = 0, new_tokens: bool = False,
               poison: bool = True, values: bool = True, dtype: str = "f16",
               tables: Optional[np.ndarray] = None) -> DecodeCase:
    """Generic builder; the named workloads below are thin wrappers.

    The pool holds exactly the blocks the tables use plus `spare_frac` spare
    blocks (left NaN), unless num_blocks is given.  values=False skips drawing
    q/K/V (the arrays are allocated but left unfilled) for callers that only
    need lengths and tables.  `tables` (with num_blocks and
    max_blocks_per_seq) supplies ready-made block tables instead.
    """
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    S = int(ctx.shape[0])
    nb = [blocks_needed(c, block_size) for c in ctx]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, max(nb) if nb else 1)
    if shared_prefix_blocks:
        needed = shared_prefix_blocks + sum(max(0, n - shared_prefix_blocks) for n in nb)
    else:
        needed = sum(nb)
    if tables is not None:
        if num_blocks is None or tables.shape != (S, max_blocks_per_seq):
            raise ValueError("ready-made tables need num_blocks and a matching max_blocks_per_seq")
        tables = np.ascontiguousarray(tables, dtype=np.int32)
    else:
        if num_blocks is None:
            num_blocks = max(1, needed + int(math.ceil(spare_frac * needed)))
        tables = allocate_tables(ctx, block_size, num_blocks, max_blocks_per_seq, rng,
                                 shared_prefix_blocks)
    H, D = num_heads, head_dim
    st = STORAGE[dtype]
    q = np.empty((S, H, D), dtype=st)
    k_cache = np.empty((num_blocks, H, block_size, D), dtype=st)
    v_cache = np.empty_like(k_cache)
    if values:
        fill_normal_f16(q, seed, 1)
        fill_normal_f16(k_cache, seed, 2)
        fill_normal_f16(v_cache, seed, 3)
    case = DecodeCase(name=name, seed=seed, num_heads=H, head_dim=D,
                      block_size=block_size,
                      scale=float(np.float32(1.0 / math.sqrt(D))),
                      context_lens=ctx, block_tables=tables, q=q,
                      k_cache=k_cache, v_cache=v_cache,
                      shared_prefix_blocks=shared_prefix_blocks, dtype=dtype)
    if poison and values:
        poison_unused(case)
    if new_tokens:
        add_new_tokens(case)
    return case


def build_grouped_case(name: str, layout, *, num_heads: int, head_dim: int, seed: int,
                       block_size: int = BLOCK_SIZE, spare_frac: float = 0.10,
                       max_blocks_per_seq: Optional[int] = None, dtype: str = "f16",
                       new_tokens: bool = False):
    """A decode batch in groups that share a prompt prefix.

    layout = [(P, [ctx, ...]), ...] lists consecutive groups of sequences.  In
    a group with P > 0 the first P blocks are popped once from the shuffled
    free list and start every member's table (a shared system prompt, or
    samples forked from one prompt: "vLLM 2026 推理引擎全解", §2.3); each
    member then pops its private blocks.  Sequences of a P = 0 entry share
    nothing.  Unused slots are NaN-poisoned.  Returns (case, group_start
    [G + 1] int32, group_prefix_blocks [G] int32), one group per entry.
    """
    rng = np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(1,)))
    lens = [int(c) for _, members in layout for c in members]
    nb = [blocks_needed(c, block_size) for c in lens]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, max(nb) if nb else 1)
    needed = 0
    i = 0
    for P, members in layout:
        if P:
            needed += P
        for _ in members:
            needed += max(0, nb[i] - P)
            i += 1
    num_blocks = max(1, needed + int(math.ceil(spare_frac * needed)))
    free = deque(int(b) for b in rng.permutation(num_blocks))
    tables = np.full((len(lens), max_blocks_per_seq), -1, dtype=np.int32)
    group_start, group_prefix = [0], []
    s = 0
    for P, members in layout:
        prefix = [free.popleft() for _ in range(P)]
        for _ in members:
            if nb[s] > max_blocks_per_seq:
                raise ValueError(f"sequence {s} needs {nb[s]} blocks > max_blocks_per_seq")
            row = prefix[:min(nb[s], P)]
            row += [free.popleft() for _ in range(nb[s] - len(row))]
            tables[s, :nb[s]] = row
            s += 1
        group_start.append(s)
        group_prefix.append(P)
    case = build_case(name, lens, num_heads=num_heads, head_dim=head_dim, seed=seed,
                      block_size=block_size, num_blocks=num_blocks,
                      max_blocks_per_seq=max_blocks_per_seq, dtype=dtype, tables=tables,
                      new_tokens=new_tokens)
    return (case, np.asarray(group_start, dtype=np.int32),
            np.asarray(group_prefix, dtype=np.int32))


def build_prefill_case(name: str, context_lens, query_lens, *, num_heads: int, head_dim: int,
                       seed: int, **kw) -> DecodeCase:
    """A prefill batch: sequence s has context_lens[s] tokens in the cache, of
    which the last query_lens[s] are the queries (a chunk of its prompt, or
    all of it).  q is [sum(query_lens), H, D]."""
    ql = np.asarray(query_lens, dtype=np.int32)
    case = build_case(name, context_lens, num_heads=num_heads, head_dim=head_dim, seed=seed, **kw)
    if (ql > case.context_lens).any() or (ql < 0).any():
        raise ValueError("query_lens must lie in [0, context_lens]")
    qs = np.zeros(len(ql) + 1, dtype=np.int32)
    qs[1:] = np.cumsum(ql)
    q = np.empty((int(qs[-1]), num_heads, head_dim), dtype=case.q.dtype)
    fill_normal(q, seed, 6)
    case.q = q
    case.query_start = qs
    return case


PREFILL_WORKLOADS = ("prefill_llama7b", "prefill_chunked")


def make_prefill_workload(kind: str, seed: Optional[int] = None, **kw) -> DecodeCase:
    """prefill_llama7b  16 prompts of 1024 tokens each, prefilled whole, on a
                        LLaMA-7B layer (32 heads x 128).
    prefill_chunked     32 sequences with contexts U[512, 4096] whose last
                        256 tokens are a prompt chunk being prefilled."""
    seeds = {"prefill_llama7b": 21, "prefill_chunked": 22}
    if kind not in seeds:
        raise KeyError(kind)
    seed = seeds[kind] if seed is None else seed
    rng = np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(0,)))
    if kind == "prefill_llama7b":
        ctx = np.full(16, 1024)
        return build_prefill_case(kind, ctx, ctx, num_heads=32, head_dim=128, seed=seed,
                                  max_blocks_per_seq=64, **kw)
    ctx = rng.integers(512, 4096, size=32, endpoint=True)
    return build_prefill_case(kind, ctx, np.full(32, 256), num_heads=32, head_dim=128, seed=seed,
                              max_blocks_per_seq=256, **kw)


def prefill_algorithmic_flops(case: DecodeCase) -> int:
    """2 * D flops per (query, key) for q.k and again for p.V, over the
    causal pairs: query at position p sees p + 1 keys."""
    total = 0
    for s in range(case.num_seqs):
        ctx = int(case.context_lens[s])
        q_len = int(case.query_start[s + 1] - case.query_start[s])
        first = ctx - q_len
        keys = q_len * (first + 1) + q_len * (q_len - 1) // 2
        total += keys
    return 4 * case.head_dim * case.num_heads * total


def add_new_tokens(case: DecodeCase) -> None:
    """One new token per sequence with ctx > 0, written at position ctx - 1.

    The decode step that follows attends to it, so the newest token sees
    itself, as o_t = Attention(q_t, K_{1:t}, V_{1:t}) requires
    ("vLLM 2026 推理引擎全解", §1.1).
    """
    B = case.block_size
    slots = []
    for s in range(case.num_seqs):
        ctx = int(case.context_lens[s])
        if ctx <= 0:
            continue
        pos = ctx - 1
        slots.append(int(case.block_tables[s, pos // B]) * B + pos % B)
    T = len(slots)
    case.slot_mapping = np.asarray(slots, dtype=np.int32)
    case.k_new = np.empty((T, case.num_heads, case.head_dim), dtype=case.q.dtype)
    case.v_new = np.empty_like(case.k_new)
    fill_normal_f16(case.k_new, case.seed, 4)
    fill_normal_f16(case.v_new, case.seed, 5)


def duplicate_prefix(case: DecodeCase) -> DecodeCase:
    """The same logical K/V with every shared block copied into private blocks.

    Each sequence that uses a block that another sequence also uses gets its
    own copy, appended to the pool; the result must give identical attention
    outputs ("vLLM 2026 推理引擎全解", §2.3: sharing changes storage, not the
    values a request sees).
    """
    tables = case.block_tables.copy()
    owners: dict[int, int] = {}
    extra = []
    next_id = case.num_blocks
    for s in range(case.num_seqs):
        for b in range(blocks_needed(case.context_lens[s], case.block_size)):
            phys = int(tables[s, b])
            if phys in owners:
                extra.append(phys)
                tables[s, b] = next_id
                next_id += 1
            else:
                owners[phys] = s
    if extra:
        idx = np.asarray(extra, dtype=np.int64)
        k_cache = np.concatenate([case.k_cache, case.k_cache[idx]], axis=0)
        v_cache = np.concatenate([case.v_cache, case.v_cache[idx]], axis=0)
    else:
        k_cache, v_cache = case.k_cache.copy(), case.v_cache.copy()
    return replace(case, name=case.name + "_dup", block_tables=tables,
                   k_cache=k_cache, v_cache=v_cache, shared_prefix_blocks=0)


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

WORKLOADS = ("tiny", "llama7b_b64", "cb_mix", "shared_prefix", "long_ctx", "cb_mix_1k",
             "cb_mix_4k", "shared_prefix_4k")


def make_workload(kind: str, seed: Optional[int] = None, **kw) -> DecodeCase:
    """The five synthetic decode workloads, by name.

    tiny          4 seqs, 4 heads, D 64, 64 physical blocks; ctx ~ U[1, 100];
                  the 64 ids are handed out from one seeded permutation.
    llama7b_b64   64 seqs, 32 heads, D 128 (a LLaMA-7B layer); ctx ~ U[128,
                  2048]; shuffled free list; plus one new token per sequence
                  for reshape_and_cache.
    cb_mix        256 seqs, 32 heads, D 128; ctx = U[16, 512] prompt +
                  min(Geometric(1/200), 1000) generated tokens (the pages'
                  mean-200 / max-1000 generation-length example).
    shared_prefix 128 seqs, 32 heads, D 128; every table starts with the same
                  32 physical blocks (a 512-token system prompt) followed by a
                  private suffix of U[16, 512] tokens.
    long_ctx      8 seqs, 32 heads, D 128, 32768 tokens each (2048 blocks).
    cb_mix_1k     cb_mix's length recipe at a serving batch of 1024 sequences
                  (32 heads, D 128; 7.8 GB of K/V).
    cb_mix_4k     the same recipe at 4096 sequences, with 8 heads of D 128 (the
                  K/V of a layer with 8 key/value heads; 7.8 GB of K/V).
    shared_prefix_4k  shared_prefix's recipe (one 512-token prompt, private
                  suffixes of U[16, 512] tokens) at 4096 sequences, 8 heads.
    """
    seeds = {"tiny": 1, "llama7b_b64": 2, "cb_mix": 3, "shared_prefix": 4, "long_ctx": 5,
             "cb_mix_1k": 6, "cb_mix_4k": 7, "shared_prefix_4k": 8}
    if kind not in seeds:
        raise KeyError(kind)
    seed = seeds[kind] if seed is None else seed
    rng = np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(0,)))
    if kind == "tiny":
        ctx = rng.integers(1, 100, size=4, endpoint=True)
        return build_case(kind, ctx, num_heads=4, head_dim=64, seed=seed,
                          num_blocks=64, max_blocks_per_seq=8, **kw)
    if kind == "llama7b_b64":
        ctx = rng.integers(128, 2048, size=64, endpoint=True)
        kw.setdefault("new_tokens", True)
        return build_case(kind, ctx, num_heads=32, head_dim=128, seed=seed,
                          max_blocks_per_seq=128, **kw)
    if kind == "cb_mix":
        prompt = rng.integers(16, 512, size=256, endpoint=True)
        gen = np.minimum(rng.geometric(1.0 / 200.0, size=256), 1000)
        return build_case(kind, prompt + gen, num_heads=32, head_dim=128, seed=seed,
                          max_blocks_per_seq=blocks_needed(512 + 1000), **kw)
    if kind in ("cb_mix_1k", "cb_mix_4k"):
        n, heads = (1024, 32) if kind == "cb_mix_1k" else (4096, 8)
        prompt = rng.integers(16, 512, size=n, endpoint=True)
        gen = np.minimum(rng.geometric(1.0 / 200.0, size=n), 1000)
        return build_case(kind, prompt + gen, num_heads=heads, head_dim=128, seed=seed,
                          max_blocks_per_seq=blocks_needed(512 + 1000), **kw)
    if kind in ("shared_prefix", "shared_prefix_4k"):
        n, heads = (128, 32) if kind == "shared_prefix" else (4096, 8)
        suffix = rng.integers(16, 512, size=n, endpoint=True)
        return build_case(kind, 512 + suffix, num_heads=heads, head_dim=128, seed=seed,
                          max_blocks_per_seq=64, shared_prefix_blocks=32, **kw)
    # long_ctx
    return build_case(kind, np.full(8, 32768), num_heads=32, head_dim=128, seed=seed,
                      max_blocks_per_seq=2048, **kw)


def kv_bytes_per_token(num_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """K plus V bytes one token occupies in one layer: 2 * H * D * dtype_size
    (mjmagnets.cn vLLM tutorial, §2; "vLLM 2026 推理引擎全解", §1.1)."""
    return 2 * num_heads * head_dim * dtype_bytes


def decode_algorithmic_bytes(case: DecodeCase) -> int:
    """Bytes a decode call must move at minimum.

    K and V of the ctx tokens of every sequence, each counted once per
    sequence that reads it, plus q, the output, the table entries used and the
    context lengths.  Shared prefix blocks count once per reader here; the
    unique-bytes figure is decode_unique_bytes().
    """
    S, H, D = case.num_seqs, case.num_heads, case.head_dim
    tokens = int(case.context_lens.astype(np.int64).sum())
    used_entries = int(case.blocks_used().sum())
    return (tokens * kv_bytes_per_token(H, D) + 2 * S * H * D * 2
            + used_entries * 4 + S * 4)


def decode_unique_bytes(case: DecodeCase) -> int:
    """Like decode_algorithmic_bytes but every distinct (block, slot) once."""
    S, H, D, B = case.num_seqs, case.num_heads, case.head_dim, case.block_size
    seen = {}
    for s in range(S):
        ctx = int(case.context_lens[s])
        for b in range(blocks_needed(ctx, B)):
            phys = int(case.block_tables[s, b])
            seen[phys] = max(seen.get(phys, 0), min(B, ctx - b * B))
    tokens = sum(seen.values())
    used_entries = int(case.blocks_used().sum())
    return (tokens * kv_bytes_per_token(H, D) + 2 * S * H * D * 2
            + used_entries * 4 + S * 4)


def reshape_algorithmic_bytes(case: DecodeCase) -> int:
    """reshape_and_cache moves each new token's K and V once in and once out."""
    T = case.num_new_tokens
    return 2 * T * kv_bytes_per_token(case.num_heads, case.head_dim) + T * 4
