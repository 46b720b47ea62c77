"""Seeded synthetic inputs for paged KV-cache attention.

This module only draws inputs: block tables, slot lists, sequence lengths and
N(0, 1) bf16 tensors.  It performs none of the attention arithmetic, and both
the CUDA library's tests and the CPU oracle's tests take their inputs from it.

Shapes follow the Qwen3-0.6B attention layer used throughout "大模型推理入门与
nano-vLLM 源码详解" (§11.5: 16 query heads, 8 KV heads, head_dim 128, bf16; the
per-layer cache view is [num_blocks, block_size, kv_heads, head_dim]).

Conventions:
* metadata (tables, lengths, slots) is drawn with numpy ``PCG64(seed)``;
* tensors are drawn with ``torch.Generator(device).manual_seed(seed)`` in fp32
  and rounded to bf16 (round-to-nearest-even) by torch;
* every cache row that holds no token, and every unused table entry, is
  poisoned (bf16 NaN, -1), so a kernel that reads outside the live context
  produces NaN;
* new-token q/k/v are column views of one fused [T, (Hq + 2*Hkv) * d] buffer,
  as the output of a fused QKV projection is, so token strides are not packed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HQ, HKV, HEAD_DIM = 16, 8, 128
SCALE = 1.0 / math.sqrt(HEAD_DIM)
BF16_NAN_BITS = 0x7FC0
SEED_BASE = 1100


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a bf16 tensor as a numpy uint16 array (copied to host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_from_values(values, device="cpu") -> torch.Tensor:
    """A bf16 tensor from exact values (test fixtures with small numbers)."""
    return torch.as_tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16).to(device)


# --------------------------------------------------------------------------- layout


@dataclass
class PagedLayout:
    """Block tables over one pool.  ``reserve_lens[b]`` positions are backed by
    blocks for sequence b; the first ``shared_prefix_blocks`` logical blocks
    of every sequence are the same physical blocks."""

    block_size: int
    num_blocks: int
    block_tables: np.ndarray  # int32 [B, max_blocks], -1 padded
    reserve_lens: np.ndarray  # int64 [B]
    shared_prefix_blocks: int = 0

    @property
    def num_seqs(self) -> int:
        return self.block_tables.shape[0]

    def slots(self, seq: int, positions) -> np.ndarray:
        """Pool rows of the given positions of one sequence (the generator's own
        bookkeeping for where each token lives)."""
        pos = np.asarray(positions, dtype=np.int64)
        blocks = self.block_tables[seq][pos // self.block_size].astype(np.int64)
        assert (blocks >= 0).all()
        return blocks * self.block_size + pos % self.block_size


def make_layout(seed: int, reserve_lens, block_size: int, num_blocks: int | None = None,
                shared_prefix_blocks: int = 0, table_width: int | None = None) -> PagedLayout:
    """Fully fragmented tables: the physical ids are a seeded permutation of
    the pool, handed out in sequence order."""
    r = rng(seed)
    reserve = np.asarray(reserve_lens, dtype=np.int64)
    need = -(-reserve // block_size)
    assert (need >= shared_prefix_blocks).all()
    total = shared_prefix_blocks + int((need - shared_prefix_blocks).sum())
    num_blocks = total if num_blocks is None else num_blocks
    assert num_blocks >= total, (num_blocks, total)
    ids = r.permutation(num_blocks)[:total].astype(np.int32)
    width = int(need.max()) if table_width is None else table_width
    assert width >= need.max()
    tables = np.full((len(reserve), max(width, 1)), -1, dtype=np.int32)
    shared = ids[:shared_prefix_blocks]
    nxt = shared_prefix_blocks
    for b, n in enumerate(need):
        tables[b, :shared_prefix_blocks] = shared
        own = int(n) - shared_prefix_blocks
        tables[b, shared_prefix_blocks:n] = ids[nxt:nxt + own]
        nxt += own
    return PagedLayout(block_size, num_blocks, tables, reserve, shared_prefix_blocks)


# --------------------------------------------------------------------------- tensors


def _randn_bf16(gen: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class NewTokens:
    qkv: torch.Tensor  # bf16 [T, (Hq + 2 Hkv) * d]
    q: torch.Tensor    # view [T, Hq, d]
    k: torch.Tensor    # view [T, Hkv, d]
    v: torch.Tensor    # view [T, Hkv, d]


def new_tokens(seed: int, num_tokens: int, num_heads=HQ, num_kv_heads=HKV, head_dim=HEAD_DIM,
               device="cpu") -> NewTokens:
    gen = torch.Generator(device=device).manual_seed(seed)
    width = (num_heads + 2 * num_kv_heads) * head_dim
    qkv = _randn_bf16(gen, (num_tokens, width), device)
    a, b = num_heads * head_dim, (num_heads + num_kv_heads) * head_dim
    q = qkv[:, :a].view(num_tokens, num_heads, head_dim)
    k = qkv[:, a:b].view(num_tokens, num_kv_heads, head_dim)
    v = qkv[:, b:].view(num_tokens, num_kv_heads, head_dim)
    return NewTokens(qkv, q, k, v)


def history_rows(layout: PagedLayout, history_lens) -> np.ndarray:
    """Pool rows that hold positions 0..history_lens[b]-1 of each sequence
    (shared prefix rows listed once)."""
    rows = []
    for b, n in enumerate(np.asarray(history_lens, dtype=np.int64)):
        rows.append(layout.slots(b, np.arange(n)))
    if not rows:
        return np.zeros(0, dtype=np.int64)
    return np.unique(np.concatenate(rows))


def make_pool(layout: PagedLayout, history_lens, seed: int, num_kv_heads=HKV, head_dim=HEAD_DIM,
              device="cpu", chunk_rows: int = 1 << 16):
    """(k_cache, v_cache) [NB, bs, Hkv, d] bf16: rows of the listed history are
    N(0,1), every other row is NaN."""
    nrows = layout.num_blocks * layout.block_size
    width = num_kv_heads * head_dim
    gen = torch.Generator(device=device).manual_seed(seed)
    live = torch.zeros(nrows, dtype=torch.bool, device=device)
    idx = history_rows(layout, history_lens)
    if idx.size:
        live[torch.as_tensor(idx, device=device)] = True
    caches = []
    for _ in range(2):
        c = torch.empty((nrows, width), dtype=torch.bfloat16, device=device)
        for r0 in range(0, nrows, chunk_rows):
            r1 = min(nrows, r0 + chunk_rows)
            c[r0:r1] = _randn_bf16(gen, (r1 - r0, width), device)
        c[~live] = float("nan")
        caches.append(c.view(layout.num_blocks, layout.block_size, num_kv_heads, head_dim))
    return caches[0], caches[1]


# --------------------------------------------------------------------------- batches


@dataclass
class PagedBatch:
    """One attention call's worth of inputs over a paged pool."""

    layout: PagedLayout
    context_lens: np.ndarray   # int32 [B]: keys visible to the last query of each seq
    query_lens: np.ndarray     # int32 [B]: new tokens (queries) per seq this call
    tokens: NewTokens          # q/k/v of the new tokens, packed by sequence
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    num_heads: int = HQ
    num_kv_heads: int = HKV
    head_dim: int = HEAD_DIM
    scale: float = SCALE
    extra: dict = field(default_factory=dict)

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.query_lens)]).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.context_lens)]).astype(np.int32)

    @property
    def slot_mapping(self) -> np.ndarray:
        parts = [self.layout.slots(b, np.arange(c - n, c))
                 for b, (c, n) in enumerate(zip(self.context_lens, self.query_lens))]
        return np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)

    @property
    def block_tables(self) -> np.ndarray:
        return self.layout.block_tables

    @property
    def positions(self) -> np.ndarray:
        """int32 [T]: the position of every new token within its sequence (the
        last query_lens[b] of context_lens[b] positions)."""
        parts = [np.arange(c - n, c) for c, n in zip(self.context_lens, self.query_lens)]
        return np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())


def paged_batch(seed: int, context_lens, query_lens, block_size: int, *, reserve_lens=None,
                num_blocks=None, shared_prefix_blocks=0, table_width=None, num_heads=HQ,
                num_kv_heads=HKV, head_dim=HEAD_DIM, device="cpu", scale=None) -> PagedBatch:
    """General builder: sequence b has context_lens[b] positions after this
    call, the last query_lens[b] of which are new (their K/V are inputs to the
    KV write, their Q are the queries); the earlier positions are already in
    the pool."""
    ctx = np.asarray(context_lens, dtype=np.int32)
    ql = np.asarray(query_lens, dtype=np.int32)
    assert ctx.shape == ql.shape and (ql <= ctx).all()
    reserve = ctx if reserve_lens is None else np.asarray(reserve_lens)
    layout = make_layout(seed, reserve, block_size, num_blocks, shared_prefix_blocks, table_width)
    k_cache, v_cache = make_pool(layout, ctx - ql, seed + 1, num_kv_heads, head_dim, device)
    toks = new_tokens(seed + 2, int(ql.sum()), num_heads, num_kv_heads, head_dim, device)
    return PagedBatch(layout, ctx, ql, toks, k_cache, v_cache, num_heads, num_kv_heads, head_dim,
                      SCALE if scale is None else scale)


# --------------------------------------------------------------------------- the five workloads

TINY_LENGTHS = (7, 33, 64, 100)
TINY_DECODE_STEPS = 8


def tiny_prefill(device="cpu") -> PagedBatch:
    """Tiny single-layer case: prompts of 7/33/64/100 tokens, block_size 16,
    a 64-block pool and tables drawn from a seeded permutation; blocks are
    reserved for the 8 decode steps that follow."""
    lens = np.array(TINY_LENGTHS)
    return paged_batch(SEED_BASE + 1, lens, lens, 16, reserve_lens=lens + TINY_DECODE_STEPS,
                       num_blocks=64, device=device)


def tiny_decode_tokens(step: int, device="cpu") -> NewTokens:
    """q/k/v of the one token each tiny sequence appends at decode step `step`."""
    return new_tokens(SEED_BASE + 1 + 100 * (step + 1), len(TINY_LENGTHS), device=device)


def decode_batch(device="cpu", num_seqs=256, seed=SEED_BASE + 2) -> PagedBatch:
    """Decode batch: context_lens U[100, 1024] (the count includes the token
    written this step), block_size 256, pool sized to fit."""
    ctx = rng(seed + 7).integers(100, 1024, size=num_seqs, endpoint=True)
    return paged_batch(seed, ctx, np.ones_like(ctx), 256, device=device)


def varlen_prefill_lengths(seed=SEED_BASE + 3, budget=16384):
    r = rng(seed + 7)
    lens, total = [], 0
    while True:
        n = int(r.integers(100, 1024, endpoint=True))
        if total + n > budget:
            return np.array(lens, dtype=np.int32)
        lens.append(n)
        total += n


def varlen_prefill(device="cpu") -> PagedBatch:
    """Packed prompts of U[100, 1024] tokens filling max_num_batched_tokens =
    16384, no cached prefix (cu_seqlens_q == cu_seqlens_k), block_size 256."""
    lens = varlen_prefill_lengths()
    return paged_batch(SEED_BASE + 3, lens, lens, 256, device=device)


PREFIX_LEN = 2048
PREFIX_SEQS = 32


def prefix_chunk(device="cpu"):
    """32 sequences sharing a resident 2048-token prefix (the same 8 block ids
    in every table) with U[128, 512] new suffix tokens each; sequence 0's
    suffix is split into two chunks at floor(s0 / 2).  Returns (call_a,
    call_b, suffix_lens): call_a holds every sequence with sequence 0 limited
    to its first chunk; call_b holds sequence 0's second chunk alone, over the
    same pool.  Both calls' new K/V are written to the pool by the KV write
    before their attention."""
    seed = SEED_BASE + 4
    suffix = rng(seed + 7).integers(128, 512, size=PREFIX_SEQS, endpoint=True).astype(np.int32)
    c1 = int(suffix[0] // 2)
    full_ctx = PREFIX_LEN + suffix
    ql_a = suffix.copy()
    ql_a[0] = c1
    ctx_a = full_ctx.copy()
    ctx_a[0] = PREFIX_LEN + c1
    a = paged_batch(seed, ctx_a, ql_a, 256, reserve_lens=full_ctx,
                    shared_prefix_blocks=PREFIX_LEN // 256, device=device)
    # history of call a is the shared prefix only (every query of call a is new)
    lay_b = PagedLayout(256, a.layout.num_blocks, a.layout.block_tables[:1].copy(),
                        full_ctx[:1], a.layout.shared_prefix_blocks)
    toks_b = new_tokens(seed + 3, int(suffix[0]) - c1, device=device)
    b = PagedBatch(lay_b, full_ctx[:1].astype(np.int32), np.array([suffix[0] - c1], np.int32),
                   toks_b, a.k_cache, a.v_cache)
    return a, b, suffix


def long_decode(device="cpu", num_seqs=512, seed=SEED_BASE + 5) -> PagedBatch:
    """Long-context max-batch decode: 512 sequences, context_lens U[1024,
    4096], block_size 256, fully fragmented tables over a pool of 16 blocks per
    sequence (8192 blocks, about 8.6 GB of K+V per layer, for 512; fewer
    sequences give the small case of the same shape that a profiler capture
    needs)."""
    ctx = rng(seed + 7).integers(1024, 4096, size=num_seqs, endpoint=True)
    return paged_batch(seed, ctx, np.ones_like(ctx), 256, num_blocks=16 * num_seqs, device=device)


# ----------------------------------------------------------------- head norm and RoPE inputs

ROPE_BASE = 1_000_000.0   # Qwen3's rope_theta
RMS_EPS = 1e-6            # Qwen3-0.6B's rms_norm_eps (a configuration value; the pages name the field only)
MAX_POSITIONS = 40_960    # Qwen3-0.6B's max_position_embeddings


def norm_weights(seed: int, head_dim=HEAD_DIM, device="cpu"):
    """(q_norm_weight, k_norm_weight): bf16 [head_dim] each, U[0.5, 1.5] (random
    initialisation in the range of trained norm weights; no checkpoint)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    w = (torch.rand((2, head_dim), generator=gen, dtype=torch.float32) + 0.5).to(torch.bfloat16)
    return w[0].contiguous().to(device), w[1].contiguous().to(device)
