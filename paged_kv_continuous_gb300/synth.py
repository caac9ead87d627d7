"""Seeded synthetic workloads for paged-KV attention.

This module only *creates inputs*: random context lengths, a shuffled
physical block pool, block tables, bf16 q/K/V values and the slot mapping of
the tokens stored in the step.  It contains none of the attention arithmetic
and imports nothing from the CUDA binding or from the oracle, so both the
oracle tests and the GPU tests can draw identical inputs from it.

Shapes follow the Qwen2.5-1.5B attention layer the pages build (12 query
heads, 2 KV heads, head_dim 128, 16-token blocks; koas-w "errors and
solutions", sections "模型层" and "KV Cache 管理").  Values are N(0, 1) drawn
in fp32 and rounded once to bf16 (round to nearest even).  Pool slots that
hold no key of any sequence are poisoned with bf16 NaN, so a kernel that
reads a slot it should not read produces a visible NaN.

Draw order inside one workload (one ``numpy.random.Generator`` seeded with
``seed``): context lengths -> block permutation -> q -> K -> V.  The new
tokens of the step (the last ``q_len`` positions of each sequence) are drawn
with K and V but are *not* placed in the pool: the store step places them
through ``slot_mapping``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
SEED_BASE = 20260000


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclass
class PagedWorkload:
    """One attention step over a paged KV pool (all arrays on the host)."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    q: np.ndarray               # uint16 [rows, Hq, D]; rows = sum(q_lens)
    cu_seqlens: np.ndarray      # int32 [B + 1]; prefix sums of q_lens
    context_lens: np.ndarray    # int32 [B]; keys seen by the last query of b
    block_tables: np.ndarray    # int32 [B, max_blocks]; -1 past each sequence's blocks
    k_cache: np.ndarray         # uint16 [num_blocks, bs, Hkv, D]; new tokens NOT yet stored
    v_cache: np.ndarray
    new_k: np.ndarray           # uint16 [rows, Hkv, D]; K of the step's new tokens
    new_v: np.ndarray
    slot_mapping: np.ndarray    # int32 [rows]; physical slot of each new token
    k_seq: list = field(default_factory=list)   # per sequence uint16 [ctx, Hkv, D]
    v_seq: list = field(default_factory=list)

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens).astype(np.int32)

    @property
    def positions(self) -> np.ndarray:
        """int32 [rows]: absolute position of each new token (the last q_len
        positions of its sequence, in order)."""
        ql = self.q_lens.astype(np.int64)
        first = np.repeat(self.context_lens.astype(np.int64) - ql, ql)
        within = np.arange(int(ql.sum()), dtype=np.int64) - np.repeat(
            self.cu_seqlens[:-1].astype(np.int64), ql)
        return (first + within).astype(np.int32)

    def stored_caches(self):
        """Copies of the pools with the step's new tokens already placed."""
        kc, vc = self.k_cache.copy(), self.v_cache.copy()
        flat_k = kc.reshape(-1, self.num_kv_heads, self.head_dim)
        flat_v = vc.reshape(-1, self.num_kv_heads, self.head_dim)
        ok = self.slot_mapping >= 0
        flat_k[self.slot_mapping[ok]] = self.new_k[ok]
        flat_v[self.slot_mapping[ok]] = self.new_v[ok]
        return kc, vc


def make_paged(rng: np.random.Generator, name: str, context_lens, q_lens, num_blocks: int,
               num_q_heads: int = 12, num_kv_heads: int = 2, head_dim: int = 128,
               block_size: int = 16, scale: float | None = None,
               max_blocks_per_seq: int | None = None, keep_seq: bool = True,
               poison: bool = True) -> PagedWorkload:
    """Build one paged workload; ``rng`` has already drawn the context lengths."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    B = ctx.shape[0]
    assert ql.shape == (B,) and np.all(ql <= ctx) and np.all(ql >= 0)
    nblk = (ctx + block_size - 1) // block_size
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, int(nblk.max()) if B else 1)
    assert int(nblk.sum()) <= num_blocks, "pool too small"
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((B, max_blocks_per_seq), -1, np.int32)
    off = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += int(nblk[b])
    rows = int(ql.sum())
    q = bf16_bits(rng.standard_normal((rows, num_q_heads, head_dim), dtype=np.float32))
    total = int(ctx.sum())
    K = bf16_bits(rng.standard_normal((total, num_kv_heads, head_dim), dtype=np.float32))
    V = bf16_bits(rng.standard_normal((total, num_kv_heads, head_dim), dtype=np.float32))

    fill = BF16_NAN if poison else np.uint16(0)
    k_cache = np.full((num_blocks, block_size, num_kv_heads, head_dim), fill, np.uint16)
    v_cache = np.full_like(k_cache, fill)
    flat_k = k_cache.reshape(-1, num_kv_heads, head_dim)
    flat_v = v_cache.reshape(-1, num_kv_heads, head_dim)

    # physical slot of every (sequence, position)
    seq_of = np.repeat(np.arange(B), ctx)
    starts = np.concatenate([[0], np.cumsum(ctx)[:-1]]).astype(np.int64)
    pos = np.arange(total, dtype=np.int64) - np.repeat(starts, ctx)
    slots = (tables[seq_of, pos // block_size].astype(np.int64) * block_size
             + pos % block_size)
    is_new = pos >= np.repeat(ctx - ql, ctx)
    old = ~is_new
    flat_k[slots[old]] = K[old]
    flat_v[slots[old]] = V[old]

    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(ql)
    new_k = np.ascontiguousarray(K[is_new])
    new_v = np.ascontiguousarray(V[is_new])
    slot_mapping = slots[is_new].astype(np.int32)

    k_seq, v_seq = [], []
    if keep_seq:
        for b in range(B):
            k_seq.append(K[starts[b]:starts[b] + ctx[b]])
            v_seq.append(V[starts[b]:starts[b] + ctx[b]])
    if scale is None:
        scale = 1.0 / float(np.sqrt(head_dim))
    return PagedWorkload(name, num_q_heads, num_kv_heads, head_dim, block_size, float(scale),
                         q, cu, ctx.astype(np.int32), tables, k_cache, v_cache, new_k, new_v,
                         slot_mapping, k_seq, v_seq)


# ---------------------------------------------------------------------------
# The five workloads.  Each takes its own seed (SEED_BASE + index) so that
# every config is reproducible on its own.
# ---------------------------------------------------------------------------

def tiny_decode(seed: int = SEED_BASE + 0) -> PagedWorkload:
    """2 sequences, context_lens [5, 37], 64-block pool placed by a seeded
    permutation, Hq 12 / Hkv 2 / D 128; the step stores the 2 new tokens
    (positions 4 and 36) and then decodes."""
    rng = np.random.default_rng(seed)
    return make_paged(rng, "tiny_decode_b2_ctx5_37", [5, 37], [1, 1], num_blocks=64)


def qwen_decode_b8(seed: int = SEED_BASE + 1) -> PagedWorkload:
    """Batch 8, context_lens uniform in [128, 4096], 4096-block shuffled pool."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(128, 4096, size=8, endpoint=True)
    return make_paged(rng, "qwen_decode_b8_ctx128_4096", ctx, np.ones(8, np.int64),
                      num_blocks=4096)


def cb_lengths(rng: np.random.Generator, batch: int = 64, median: float = 1024.0,
               sigma: float = 1.0, lo: int = 1, hi: int = 8192) -> np.ndarray:
    """Lognormal context lengths (median 1024, sigma 1.0) clipped to [1, 8192]."""
    x = np.exp(rng.normal(np.log(median), sigma, size=batch))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def cb_decode_b64(seed: int = SEED_BASE + 2, num_blocks: int = 40000,
                  keep_seq: bool = True) -> PagedWorkload:
    """Continuous-batching mix: batch 64, lognormal lengths, 40000-block pool;
    the step stores 64 new tokens, then decodes every sequence."""
    rng = np.random.default_rng(seed)
    ctx = cb_lengths(rng)
    return make_paged(rng, "cb_decode_b64_lognormal1024", ctx, np.ones(64, np.int64),
                      num_blocks=num_blocks, keep_seq=keep_seq)


def long_decode_b4(seed: int = SEED_BASE + 3, context: int = 32768,
                   num_blocks: int = 10240, keep_seq: bool = True) -> PagedWorkload:
    """Long-context split-K decode: batch 4 x 32768 keys, Hq 32 / Hkv 8."""
    rng = np.random.default_rng(seed)
    ctx = np.full(4, context, np.int64)
    return make_paged(rng, "long_decode_b4_ctx32768_h32_8", ctx, np.ones(4, np.int64),
                      num_blocks=num_blocks, num_q_heads=32, num_kv_heads=8,
                      keep_seq=keep_seq)


def varlen_prefill(seed: int = SEED_BASE + 4, chunk: int = 512, n_decode: int = 8,
                   n_chunk: int = 8, max_prefix: int = 2048,
                   keep_seq: bool = True) -> PagedWorkload:
    """Chunked prefill mix: 8 one-token rows and 8 chunks of 512 queries in a
    seeded order, each behind a paged prefix uniform in [0, 2048]."""
    rng = np.random.default_rng(seed)
    kinds = rng.permutation(np.array([1] * n_decode + [chunk] * n_chunk, np.int64))
    prefix = rng.integers(0, max_prefix, size=kinds.shape[0], endpoint=True)
    ctx = prefix + kinds
    need = int(((ctx + 15) // 16).sum())
    return make_paged(rng, "varlen_prefill_8x1_8x512", ctx, kinds,
                      num_blocks=int(need * 1.25) + 1, keep_seq=keep_seq)


def rope_tables(max_position: int, head_dim: int = 128, base: float = 1.0e6):
    """Rotary-embedding inputs: float32 cos / sin tables [max_position,
    head_dim / 2] of the angles p * base^(-2i / head_dim), evaluated in
    float64 and rounded once.  base 1e6 is the Qwen2.5 configuration value
    (the pages leave it open; any table is a valid input)."""
    inv = base ** (-np.arange(head_dim // 2, dtype=np.float64) * 2.0 / head_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


CONFIGS = {
    "tiny_decode": tiny_decode,
    "qwen_decode_b8": qwen_decode_b8,
    "cb_decode_b64": cb_decode_b64,
    "long_decode_b4": long_decode_b4,
    "varlen_prefill": varlen_prefill,
}
