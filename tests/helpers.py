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


def oracle_stored_caches(w):
    """Copies of the workload's pools after the step's store, placed by the
    oracle's store (every expected pool and every pool the oracle reads is
    built here, from oracle/ alone)."""
    import oracle
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.store_kv(w.new_k, w.new_v, kc, vc, w.slot_mapping)
    return kc, vc


def normal_bits(rng, shape):
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def const_bits(value, shape):
    return bf16_bits(np.full(shape, value, np.float32))


# ---------------------------------------------------------------------------
# GPU-side helpers (torch imported lazily so CPU tests never need CUDA)
# ---------------------------------------------------------------------------

def to_dev_bf16(bits):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 CUDA tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).cuda()


def to_dev_i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def bf16_dev_to_bits(t):
    """torch.bfloat16 CUDA tensor -> numpy uint16 bit patterns."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_to_f64(t):
    """GPU output (bf16 or fp32) -> float64 numpy, exactly."""
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_to_f64(bf16_dev_to_bits(t))
    return t.float().cpu().numpy().astype(np.float64)


ATOL = 2e-3
RTOL = 1e-2


def assert_attention_close(got, ref, what="", strict=False):
    """The attention tolerance (bf16 inputs, fp32 accumulation): every element
    within 2e-3 + 1e-2 |ref|.  With ``strict`` (fp32 outputs, where no output
    rounding is involved) also max-abs <= 2e-3 and max-rel <= 1e-2, the
    relative denominator floored at 1e-3."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} err {err[i]:.3e}")
    if strict:
        mabs, mrel = max_errors(got, ref)
        assert mabs <= ATOL, f"{what}: max abs error {mabs:.3e} > {ATOL}"
        assert mrel <= RTOL, f"{what}: max rel error {mrel:.3e} > {RTOL}"


def max_errors(got, ref):
    err = np.abs(np.asarray(got, np.float64) - ref)
    rel = err / np.maximum(np.abs(ref), 1e-3)
    return float(err.max(initial=0.0)), float(rel.max(initial=0.0))
