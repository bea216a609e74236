"""Seeded synthetic decode workloads shaped like the pages' workloads.

This module only draws random numbers and lays them out through the host
block manager; it holds none of the attention arithmetic.  The same tensors
(as CPU bytes) feed both the CUDA path and the test oracle.

Workloads (all one decode query token per sequence, head dim 128):

* ``tiny``            5 sequences of 37/91/128/201/511 tokens (the worked
                      example of "PagedAttention and Online Inference"),
                      8 query heads = 8 KV heads, fp16, block size 16 or 32,
                      physical blocks drawn from a shuffled 64-block pool.
* ``gqa_batch``       64 sequences, context uniform on 512..4096, block 16,
                      32 query heads over 8 KV heads, bf16, shuffled pool of
                      1.2x the blocks needed; one new token per sequence is
                      written (kv_write) and attention covers context + 1.
* ``opt13b_like``     40 heads (MHA), fp16, block 16, 128 sequences whose
                      prompt / output lengths are log-normal (medians 160 and
                      340, sigma 1, total capped at 2048) and whose blocks
                      interleave in the pool in Poisson arrival order.
* ``long_context``    8 sequences of 32768 tokens, 32 query / 8 KV heads,
                      bf16, block 16, shuffled pool of exactly 16384 blocks.
* ``PrefixSharingScenario``  16 prompts x 8 samples sharing the prompt's
                      blocks through reference counts, block 32, 256 decode
                      steps; with a prompt length that is not a multiple of
                      the block size the shared partial block is copied on
                      write before each sample diverges.
* ``BeamSearchScenario``  beams of one prompt that fork and fall out of the
                      top-k every step, sharing blocks through refcounts.
* ``prefill_batch`` / ``build_prefill_step``  prompts (optionally after a
                      cached context) for causal paged prefill attention.

``gqa_batch`` takes a block size (8..128) for the block-size sweep.

Sizes of the K/V pools are [num_blocks, H_kv, B, d]; q is [S, H_q, d]; new
tokens are [S, H_kv, d]; slot mappings are int64; block tables and sequence
lengths are int32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from .block_manager import BlockManager

TORCH_DTYPES = {"float16": torch.float16, "bfloat16": torch.bfloat16}
HEAD_DIM = 128


@dataclass
class DecodeStep:
    """Inputs of one decode step: optional CoW copies, kv_write, attention."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    slot_mapping: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    cow_pairs: torch.Tensor
    scale: float
    k_cache: Optional[torch.Tensor] = None
    v_cache: Optional[torch.Tensor] = None
    meta: Dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    @property
    def kv_tokens(self) -> int:
        """Sum of attended lengths (tokens of K and V each query reads)."""
        return int(self.seq_lens.to(torch.int64).sum().item())


def _randn(shape, generator, dtype: str) -> torch.Tensor:
    return torch.randn(shape, generator=generator, dtype=torch.float32).to(TORCH_DTYPES[dtype])


def _fill_unreferenced(cache: torch.Tensor, manager: BlockManager, seq_ids, value: float) -> None:
    """Write ``value`` into every slot no sequence has filled (tests of masking)."""
    used = np.zeros(manager.num_blocks, dtype=bool)
    bs = manager.block_size
    for s in seq_ids:
        table = manager.tables[s]
        used[table] = True
        n = manager.lengths[s]
        if n % bs and table:
            cache[table[(n - 1) // bs], :, n % bs:, :] = value
    unused = torch.from_numpy(np.nonzero(~used)[0])
    if unused.numel():
        cache[unused] = value


def build_decode_step(name: str, context_lens: Sequence[int], num_q_heads: int,
                      num_kv_heads: int, block_size: int, dtype: str, seed: int,
                      pool_factor: float = 1.2, num_blocks: Optional[int] = None,
                      shuffle: bool = True, unfilled: Optional[float] = None,
                      head_dim: int = HEAD_DIM) -> DecodeStep:
    """Decode step over sequences whose caches hold ``context_lens`` tokens.

    Each sequence gets one new token (slot from the block manager, so a new
    block is allocated when the last one is full) and attention covers the
    context plus that token.  ``unfilled`` (e.g. NaN) overwrites every slot
    that no sequence uses, to check that such slots are never read.
    """
    g = torch.Generator().manual_seed(int(seed))
    context = [int(c) for c in context_lens]
    attended = [c + 1 for c in context]
    needed = sum(-(-n // block_size) for n in attended)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * needed))
    if num_blocks < needed:
        raise ValueError(f"pool of {num_blocks} blocks < {needed} needed")
    order = torch.randperm(num_blocks, generator=g).tolist() if shuffle else None
    manager = BlockManager(num_blocks, block_size, free_order=order)
    slots: List[int] = []
    for s, c in enumerate(context):
        manager.add_sequence(s, c)
        slot, cow = manager.append_slot(s)
        assert cow is None
        slots.append(slot)
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_cache = _randn(shape, g, dtype)
    v_cache = _randn(shape, g, dtype)
    S = len(context)
    q = _randn((S, num_q_heads, head_dim), g, dtype)
    k_new = _randn((S, num_kv_heads, head_dim), g, dtype)
    v_new = _randn((S, num_kv_heads, head_dim), g, dtype)
    seq_ids = list(range(S))
    if unfilled is not None:
        _fill_unreferenced(k_cache, manager, seq_ids, unfilled)
        _fill_unreferenced(v_cache, manager, seq_ids, unfilled)
    return DecodeStep(
        name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.tensor(slots, dtype=torch.int64),
        block_tables=torch.from_numpy(manager.block_table_array(seq_ids)),
        seq_lens=torch.from_numpy(manager.seq_lens_array(seq_ids)),
        cow_pairs=torch.zeros((0, 2), dtype=torch.int64), scale=1.0 / math.sqrt(head_dim),
        k_cache=k_cache, v_cache=v_cache,
        meta={"seed": int(seed), "num_blocks": num_blocks, "blocks_needed": needed})


# ---------------------------------------------------------------------------
# The five workloads.  Seeds are 242 + workload index unless given.
# ---------------------------------------------------------------------------
TINY_LENGTHS = (37, 91, 128, 201, 511)


def tiny(block_size: int = 16, seed: int = 243) -> DecodeStep:
    """Attended lengths 37/91/128/201/511; the last token is written by kv_write."""
    return build_decode_step(f"tiny_B{block_size}", [n - 1 for n in TINY_LENGTHS], 8, 8,
                             block_size, "float16", seed, num_blocks=64, shuffle=True)


def gqa_batch(seed: int = 244, num_seqs: int = 64, block_size: int = 16) -> DecodeStep:
    g = torch.Generator().manual_seed(seed)
    context = torch.randint(512, 4097, (num_seqs,), generator=g).tolist()
    return build_decode_step("gqa_batch" if block_size == 16 else f"gqa_batch_B{block_size}",
                             context, 32, 8, block_size, "bfloat16", seed + 1000,
                             pool_factor=1.2)


def long_context(seed: int = 246, num_seqs: int = 8, tokens: int = 32768) -> DecodeStep:
    blocks = num_seqs * (-(-tokens // 16))
    return build_decode_step("long_context", [tokens - 1] * num_seqs, 32, 8, 16, "bfloat16",
                             seed, num_blocks=blocks, shuffle=True)


def opt13b_like(seed: int = 245, num_seqs: int = 128, block_size: int = 16) -> DecodeStep:
    """MHA 40 x 128, fp16; log-normal lengths; Poisson-ordered pool interleaving.

    Prompt and output lengths: round(exp(ln(median) + N(0, 1))), at least 1,
    total capped at 2048.  Arrivals: a Poisson process of rate one request
    per decode iteration.  Replay: at its arrival iteration a request
    allocates its prompt's blocks from a FIFO free list; every later
    iteration each live request appends one token (a new block when the
    last is full) until it holds all but its final token.  The step itself
    then writes that final token for every sequence and attends over it.
    """
    g = torch.Generator().manual_seed(seed)
    prompt = torch.exp(math.log(160.0) + torch.randn(num_seqs, generator=g)).round().clamp(min=1)
    output = torch.exp(math.log(340.0) + torch.randn(num_seqs, generator=g)).round().clamp(min=1)
    total = torch.clamp(prompt + output, max=2048).to(torch.int64)
    total = torch.clamp(total, min=2)
    prompt = torch.minimum(prompt.to(torch.int64), total - 1)
    gaps = -torch.log(torch.rand(num_seqs, generator=g, dtype=torch.float64))
    arrival = torch.floor(torch.cumsum(gaps, 0)).to(torch.int64).tolist()
    total, prompt = total.tolist(), prompt.tolist()
    num_blocks = sum(-(-n // block_size) for n in total)
    manager = BlockManager(num_blocks, block_size)  # FIFO free list 0..NB-1
    live: List[int] = []
    nxt = 0
    it = 0
    while nxt < num_seqs or any(manager.lengths[s] < total[s] - 1 for s in live):
        for s in live:
            if manager.lengths[s] < total[s] - 1:
                manager.append_slot(s)
        while nxt < num_seqs and arrival[nxt] <= it:
            manager.add_sequence(nxt, prompt[nxt])
            live.append(nxt)
            nxt += 1
        it += 1
    slots = []
    for s in range(num_seqs):
        slot, cow = manager.append_slot(s)
        assert cow is None
        slots.append(slot)
    H, d = 40, HEAD_DIM
    shape = (num_blocks, H, block_size, d)
    k_cache = _randn(shape, g, "float16")
    v_cache = _randn(shape, g, "float16")
    q = _randn((num_seqs, H, d), g, "float16")
    k_new = _randn((num_seqs, H, d), g, "float16")
    v_new = _randn((num_seqs, H, d), g, "float16")
    seq_ids = list(range(num_seqs))
    return DecodeStep(
        name="opt13b_like", dtype="float16", num_q_heads=H, num_kv_heads=H, head_dim=d,
        block_size=block_size, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.tensor(slots, dtype=torch.int64),
        block_tables=torch.from_numpy(manager.block_table_array(seq_ids)),
        seq_lens=torch.from_numpy(manager.seq_lens_array(seq_ids)),
        cow_pairs=torch.zeros((0, 2), dtype=torch.int64), scale=1.0 / math.sqrt(d),
        k_cache=k_cache, v_cache=v_cache,
        meta={"seed": seed, "num_blocks": num_blocks, "iterations": it,
              "prompt": prompt, "total": total, "arrival": arrival})


class PrefixSharingScenario:
    """Parallel sampling over shared prompts with copy-on-write.

    ``num_prompts`` prompts of ``prompt_len`` tokens are prefilled once;
    each is forked into ``samples`` sequences that map the prompt's logical
    blocks onto the same physical blocks (reference count = samples).  Each
    decode step appends one token to every sample: a sample that writes into
    a block still shared gets a copy first (``cow_pairs``), as in "vLLM
    PagedAttention & continuous batching", sharing with reference counts and
    copy-on-write.  With ``prompt_len`` a multiple of the block size the
    first decode token opens a new private block and no copy happens.
    """

    def __init__(self, prompt_len: int = 1024, num_prompts: int = 16, samples: int = 8,
                 decode_steps: int = 256, block_size: int = 32, num_q_heads: int = 32,
                 num_kv_heads: int = 8, dtype: str = "bfloat16", seed: int = 247,
                 head_dim: int = HEAD_DIM) -> None:
        self.prompt_len, self.num_prompts, self.samples = prompt_len, num_prompts, samples
        self.decode_steps, self.block_size = decode_steps, block_size
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, num_kv_heads, head_dim
        self.dtype, self.seed = dtype, seed
        B = block_size
        prompt_blocks = -(-prompt_len // B)
        final_blocks = -(-(prompt_len + decode_steps) // B)
        copies = (samples - 1) if prompt_len % B else 0
        needed = num_prompts * (prompt_blocks + copies + samples * (final_blocks - prompt_blocks))
        self.num_blocks = math.ceil(1.2 * needed)
        g = torch.Generator().manual_seed(seed)
        order = torch.randperm(self.num_blocks, generator=g).tolist()
        self.manager = BlockManager(self.num_blocks, B, free_order=order)
        self.seq_ids = []
        for p in range(num_prompts):
            root = p * samples
            self.manager.add_sequence(root, prompt_len)
            self.seq_ids.append(root)
            for j in range(1, samples):
                self.manager.fork(root, root + j)
                self.seq_ids.append(root + j)
        shape = (self.num_blocks, num_kv_heads, B, head_dim)
        self.k_cache = _randn(shape, g, dtype)
        self.v_cache = _randn(shape, g, dtype)
        self.max_blocks = final_blocks
        self.step_index = 0
        self.total_copies = 0

    @property
    def num_seqs(self) -> int:
        return len(self.seq_ids)

    def unique_blocks_in_use(self) -> int:
        return int((self.manager.refcount > 0).sum())

    def logical_blocks_in_use(self) -> int:
        return sum(len(self.manager.tables[s]) for s in self.seq_ids)

    def next_step(self) -> DecodeStep:
        if self.step_index >= self.decode_steps:
            raise StopIteration
        t = self.step_index
        g = torch.Generator().manual_seed(self.seed * 1009 + t + 1)
        slots, pairs = [], []
        for s in self.seq_ids:
            slot, cow = self.manager.append_slot(s)
            slots.append(slot)
            if cow is not None:
                pairs.append(cow)
        self.total_copies += len(pairs)
        S = self.num_seqs
        q = _randn((S, self.num_q_heads, self.head_dim), g, self.dtype)
        k_new = _randn((S, self.num_kv_heads, self.head_dim), g, self.dtype)
        v_new = _randn((S, self.num_kv_heads, self.head_dim), g, self.dtype)
        self.step_index += 1
        return DecodeStep(
            name=f"prefix_sharing_step{t}", dtype=self.dtype, num_q_heads=self.num_q_heads,
            num_kv_heads=self.num_kv_heads, head_dim=self.head_dim, block_size=self.block_size,
            q=q, k_new=k_new, v_new=v_new, slot_mapping=torch.tensor(slots, dtype=torch.int64),
            block_tables=torch.from_numpy(
                self.manager.block_table_array(self.seq_ids, max_blocks=self.max_blocks)),
            seq_lens=torch.from_numpy(self.manager.seq_lens_array(self.seq_ids)),
            cow_pairs=torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2),
            scale=1.0 / math.sqrt(self.head_dim), meta={"step": t})


@dataclass
class PrefillStep:
    """Inputs of one prefill call: the prompt tokens' kv_write, then causal attention."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    q: torch.Tensor             # [total_q, H_q, d]
    cu_q: torch.Tensor          # int32 [S + 1]
    k_new: torch.Tensor         # [total_q, H_kv, d] keys of the prompt tokens
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # int64 [total_q]
    block_tables: torch.Tensor
    seq_lens: torch.Tensor      # cached context + prompt tokens
    scale: float
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    meta: Dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    @property
    def max_q_len(self) -> int:
        return int((self.cu_q[1:] - self.cu_q[:-1]).max().item()) if self.seq_lens.numel() else 0

    def causal_flops(self) -> int:
        """Useful flops: 4 * head_dim per (query head, visible key)."""
        total = 0
        for s in range(self.num_seqs):
            ql = int(self.cu_q[s + 1] - self.cu_q[s])
            ctx = int(self.seq_lens[s]) - ql
            total += ql * ctx + ql * (ql + 1) // 2
        return total * 4 * self.head_dim * self.num_q_heads


def build_prefill_step(name: str, ctx_lens: Sequence[int], q_lens: Sequence[int],
                       num_q_heads: int, num_kv_heads: int, block_size: int, dtype: str,
                       seed: int, pool_factor: float = 1.2,
                       head_dim: int = HEAD_DIM) -> PrefillStep:
    """Sequences with ``ctx_lens`` tokens already cached get ``q_lens`` prompt
    tokens: their slots come from the block manager (new blocks as the last
    fills), their keys / values are written with kv_write, and the prompt's
    queries attend causally over the context and the prompt so far."""
    g = torch.Generator().manual_seed(int(seed))
    ctx = [int(c) for c in ctx_lens]
    ql = [int(x) for x in q_lens]
    needed = sum(-(-(c + x) // block_size) for c, x in zip(ctx, ql))
    num_blocks = max(1, math.ceil(pool_factor * needed))
    order = torch.randperm(num_blocks, generator=g).tolist()
    manager = BlockManager(num_blocks, block_size, free_order=order)
    slots: List[int] = []
    for s, (c, x) in enumerate(zip(ctx, ql)):
        manager.add_sequence(s, c)
        for _ in range(x):
            slots.append(manager.append_slot(s)[0])
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_cache = _randn(shape, g, dtype)
    v_cache = _randn(shape, g, dtype)
    total = sum(ql)
    q = _randn((total, num_q_heads, head_dim), g, dtype)
    k_new = _randn((total, num_kv_heads, head_dim), g, dtype)
    v_new = _randn((total, num_kv_heads, head_dim), g, dtype)
    seq_ids = list(range(len(ctx)))
    cu = [0]
    for x in ql:
        cu.append(cu[-1] + x)
    return PrefillStep(
        name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, q=q, cu_q=torch.tensor(cu, dtype=torch.int32),
        k_new=k_new, v_new=v_new, slot_mapping=torch.tensor(slots, dtype=torch.int64),
        block_tables=torch.from_numpy(manager.block_table_array(seq_ids)),
        seq_lens=torch.from_numpy(manager.seq_lens_array(seq_ids)),
        scale=1.0 / math.sqrt(head_dim), k_cache=k_cache, v_cache=v_cache,
        meta={"seed": int(seed), "num_blocks": num_blocks})


def prefill_batch(seed: int = 249, num_seqs: int = 16) -> PrefillStep:
    """Prompts of 512..2048 tokens from an empty cache, 32 / 8 heads, bf16, block 16."""
    g = torch.Generator().manual_seed(seed)
    q_lens = torch.randint(512, 2049, (num_seqs,), generator=g).tolist()
    return build_prefill_step("prefill_batch", [0] * num_seqs, q_lens, 32, 8, 16, "bfloat16",
                              seed + 1000)


class BeamSearchScenario:
    """Beam search over one prompt, with blocks shared through reference counts.

    Every step, each live beam appends one token (a beam whose last block
    is still shared gets a copy first, ``cow_pairs``) and attends over its
    sequence.  Before the next step the search keeps ``width`` beams: a
    seeded number of beams falls out of the top-k and frees its references
    (blocks at count zero return to the pool) and a seeded surviving beam is
    forked into their places, sharing all of its blocks ("vLLM
    PagedAttention & continuous batching", sharing with reference counts and
    copy-on-write: beam search).  The kernels see only physical block ids.
    """

    def __init__(self, prompt_len: int = 100, width: int = 4, decode_steps: int = 24,
                 block_size: int = 16, num_q_heads: int = 32, num_kv_heads: int = 8,
                 dtype: str = "bfloat16", seed: int = 248, head_dim: int = HEAD_DIM) -> None:
        self.width, self.decode_steps, self.block_size = width, decode_steps, block_size
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, num_kv_heads, head_dim
        self.dtype, self.seed = dtype, seed
        per_beam = -(-(prompt_len + decode_steps) // block_size)
        self.num_blocks = width * (per_beam + 2) + 8
        self.rng = torch.Generator().manual_seed(seed)
        order = torch.randperm(self.num_blocks, generator=self.rng).tolist()
        self.manager = BlockManager(self.num_blocks, block_size, free_order=order)
        self.manager.add_sequence(0, prompt_len)
        for b in range(1, width):
            self.manager.fork(0, b)
        self.live = list(range(width))
        self.next_id = width
        self.max_blocks = per_beam + 1
        shape = (self.num_blocks, num_kv_heads, block_size, head_dim)
        self.k_cache = _randn(shape, self.rng, dtype)
        self.v_cache = _randn(shape, self.rng, dtype)
        self.step_index = 0
        self.total_copies = 0
        self.savings = []  # 1 - physical / logical blocks, per step

    def _prune_and_fork(self) -> None:
        drop = int(torch.randint(0, self.width, (1,), generator=self.rng))
        order = torch.randperm(len(self.live), generator=self.rng).tolist()
        dropped = [self.live[i] for i in order[:drop]]
        survivors = [s for s in self.live if s not in dropped]
        for s in dropped:
            self.manager.free(s)
        best = survivors[int(torch.randint(0, len(survivors), (1,), generator=self.rng))]
        for _ in dropped:
            self.manager.fork(best, self.next_id)
            survivors.append(self.next_id)
            self.next_id += 1
        self.live = survivors

    def next_step(self) -> DecodeStep:
        if self.step_index >= self.decode_steps:
            raise StopIteration
        if self.step_index > 0:
            self._prune_and_fork()
        slots, pairs = [], []
        for s in self.live:
            slot, cow = self.manager.append_slot(s)
            slots.append(slot)
            if cow is not None:
                pairs.append(cow)
        self.total_copies += len(pairs)
        logical = sum(len(self.manager.tables[s]) for s in self.live)
        physical = int((self.manager.refcount > 0).sum())
        self.savings.append(1.0 - physical / logical)
        S = len(self.live)
        g = torch.Generator().manual_seed(self.seed * 7919 + self.step_index)
        q = _randn((S, self.num_q_heads, self.head_dim), g, self.dtype)
        k_new = _randn((S, self.num_kv_heads, self.head_dim), g, self.dtype)
        v_new = _randn((S, self.num_kv_heads, self.head_dim), g, self.dtype)
        t = self.step_index
        self.step_index += 1
        return DecodeStep(
            name=f"beam_search_step{t}", dtype=self.dtype, num_q_heads=self.num_q_heads,
            num_kv_heads=self.num_kv_heads, head_dim=self.head_dim, block_size=self.block_size,
            q=q, k_new=k_new, v_new=v_new, slot_mapping=torch.tensor(slots, dtype=torch.int64),
            block_tables=torch.from_numpy(
                self.manager.block_table_array(self.live, max_blocks=self.max_blocks)),
            seq_lens=torch.from_numpy(self.manager.seq_lens_array(self.live)),
            cow_pairs=torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2),
            scale=1.0 / math.sqrt(self.head_dim), meta={"step": t, "live": list(self.live)})


def bits(t: torch.Tensor) -> np.ndarray:
    """16-bit tensor -> numpy uint16 bit patterns (same bytes, CPU)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
