"""Test helpers: build paged pools from contiguous per-sequence K/V, and a
brute-force fp64 attention over contiguous K/V (used only as a pin for the
oracle's paging, never as a reference for the GPU)."""
from __future__ import annotations

import numpy as np

from paged_kv_continuous_gb300.synth import BF16_NAN, bf16_bits, bf16_to_f64


def random_tables(rng, ctx, num_blocks, block_size=16, pad=-1):
    """Distinct physical blocks for every sequence, drawn by a permutation."""
    ctx = np.asarray(ctx)
    nblk = (ctx + block_size - 1) // block_size
    perm = rng.permutation(num_blocks)
    tables = np.full((len(ctx), max(1, int(nblk.max()))), pad, np.int32)
    off = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[off:off + n]
        off += n
    assert off <= num_blocks
    return tables


def scatter_pool(seqs, tables, num_blocks, block_size=16, fill=BF16_NAN):
    """Place seqs[b][j] (uint16 [Hkv, D]) at physical block tables[b][j // bs],
    row j % bs of a fresh pool filled with ``fill`` everywhere else."""
    Hkv, D = seqs[0].shape[1:]
    pool = np.full((num_blocks, block_size, Hkv, D), fill, np.uint16)
    for b, s in enumerate(seqs):
        for j in range(s.shape[0]):
            pool[tables[b, j // block_size], j % block_size] = s[j]
    return pool


def brute_attention(q_bits, k_bits, v_bits, scale, n_keys):
    """fp64 softmax(scale q K^T) V for one query head over the first n_keys
    rows of contiguous K/V (uint16 [n, D]).  Written independently of the
    oracle: numpy matmul + scipy-free exp."""
    q = bf16_to_f64(q_bits)
    K = bf16_to_f64(k_bits[:n_keys])
    V = bf16_to_f64(v_bits[:n_keys])
    if n_keys == 0:
        return np.zeros(q.shape[-1])
    s = scale * (K @ q)
    w = np.exp(s - s.max())
    return (w @ V) / w.sum()


def normal_bits(rng, shape):
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def const_bits(value, shape):
    return bf16_bits(np.full(shape, value, np.float32))
