"""Pins for the CPU oracle: every oracle function is checked here against
something other than itself -- exact placement, brute force over contiguous
K/V built before paging, closed forms, invariants and the pages' own varlen
example.  Each test names the mistake it would catch."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_continuous_gb300 import synth
from paged_kv_continuous_gb300.synth import BF16_NAN, bf16_bits, bf16_to_f64
from tests.helpers import (brute_attention, const_bits, normal_bits, oracle_stored_caches,
                           random_tables, scatter_pool)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / math.sqrt(128.0)


# --------------------------------------------------------------------------
# store
# --------------------------------------------------------------------------

def test_store_exact_placement_and_untouched_slots():
    """Token t lands bit-for-bit at slot_mapping[t]; every other slot keeps
    its sentinel; negative slots are skipped (catches a logical-vs-physical
    slot mix-up and off-by-one block/row arithmetic)."""
    rng = np.random.default_rng(1)
    NB, bs, Hkv, D, T = 32, 16, 2, 128, 40
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    slots[[3, 17]] = -1
    k = normal_bits(rng, (T, Hkv, D))
    v = normal_bits(rng, (T, Hkv, D))
    kc = np.full((NB, bs, Hkv, D), 0x1234, np.uint16)
    vc = np.full((NB, bs, Hkv, D), 0x4321, np.uint16)
    oracle.store_kv(k, v, kc, vc, slots)
    fk, fv = kc.reshape(NB * bs, Hkv, D), vc.reshape(NB * bs, Hkv, D)
    ok = slots >= 0
    assert np.array_equal(fk[slots[ok]], k[ok])
    assert np.array_equal(fv[slots[ok]], v[ok])
    untouched = np.ones(NB * bs, bool)
    untouched[slots[ok]] = False
    assert np.all(fk[untouched] == 0x1234) and np.all(fv[untouched] == 0x4321)


def test_store_strided_views_of_fused_qkv():
    """K/V passed as views into a fused [T, (Hq + 2 Hkv), D] buffer give the
    same pool as contiguous copies (the strided-store bug on the pages)."""
    rng = np.random.default_rng(2)
    NB, bs, Hq, Hkv, D, T = 8, 16, 12, 2, 128, 20
    qkv = normal_bits(rng, (T, Hq + 2 * Hkv, D))
    k_view, v_view = qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    assert not k_view.flags.c_contiguous
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    a_k = np.zeros((NB, bs, Hkv, D), np.uint16); a_v = np.zeros_like(a_k)
    b_k = np.zeros_like(a_k); b_v = np.zeros_like(a_k)
    oracle.store_kv(k_view, v_view, a_k, a_v, slots)
    oracle.store_kv(np.ascontiguousarray(k_view), np.ascontiguousarray(v_view), b_k, b_v,
                    slots)
    assert np.array_equal(a_k, b_k) and np.array_equal(a_v, b_v)
    flat = a_k.reshape(-1, Hkv, D)
    assert np.array_equal(flat[slots], k_view)


def test_store_rejects_out_of_range_slot():
    k = np.zeros((1, 2, 128), np.uint16)
    kc = np.zeros((2, 16, 2, 128), np.uint16)
    with pytest.raises(ValueError):
        oracle.store_kv(k, k, kc, kc.copy(), np.array([32], np.int32))


# --------------------------------------------------------------------------
# decode: paging against brute force on contiguous K/V
# --------------------------------------------------------------------------

@pytest.mark.parametrize("ctx", [1, 15, 16, 17, 31, 32, 33, 100])
def test_decode_brute_force_contiguous(ctx):
    """Oracle decode through a shuffled block table equals fp64 attention over
    the contiguous K/V drawn before paging (catches any gather, table or
    head-map error)."""
    rng = np.random.default_rng(100 + ctx)
    Hq, Hkv, D, NB = 12, 2, 128, 64
    lens = [ctx, 37]
    ks = [normal_bits(rng, (n, Hkv, D)) for n in lens]
    vs = [normal_bits(rng, (n, Hkv, D)) for n in lens]
    tables = random_tables(rng, lens, NB)
    kc, vc = scatter_pool(ks, tables, NB), scatter_pool(vs, tables, NB)
    q = normal_bits(rng, (2, Hq, D))
    out = oracle.decode(q, kc, vc, tables, np.array(lens, np.int32), SCALE)
    for b, n in enumerate(lens):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ref = brute_attention(q[b, h], ks[b][:, g], vs[b][:, g], SCALE, n)
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)
    assert np.all(np.isfinite(out))  # NaN-poisoned slots never reach the result


@pytest.mark.parametrize("scale", [-4.0, -0.09, 0.0, 3.0])
def test_decode_and_prefill_any_sign_of_scale(scale):
    """Softmax scales of either sign and zero (the kernels accept any finite
    scale): decode and prefill equal fp64 attention over the contiguous K/V,
    and scale 0 gives the plain mean of the visible V rows (catches a scale
    dropped, applied with the wrong sign or clamped to positive values)."""
    rng = np.random.default_rng(700 + int(abs(scale) * 100))
    lens = [45, 3]
    ks = [normal_bits(rng, (n, 2, 128)) for n in lens]
    vs = [normal_bits(rng, (n, 2, 128)) for n in lens]
    t = random_tables(rng, lens, 16)
    kc, vc = scatter_pool(ks, t, 16), scatter_pool(vs, t, 16)
    q = normal_bits(rng, (2, 12, 128))
    out = oracle.decode(q, kc, vc, t, np.array(lens, np.int32), scale)
    for b, n in enumerate(lens):
        for h in range(12):
            ref = brute_attention(q[b, h], ks[b][:, h // 6], vs[b][:, h // 6], scale, n)
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)
            if scale == 0.0:
                mean = bf16_to_f64(vs[b][:n, h // 6]).mean(axis=0)
                np.testing.assert_allclose(out[b, h], mean, rtol=1e-12, atol=1e-13)
    # prefill: the last 5 positions of sequence 0 as a chunk behind a prefix of 40
    qp = normal_bits(rng, (5, 12, 128))
    cu = np.array([0, 5], np.int32)
    outp = oracle.prefill_varlen(qp, cu, kc, vc, t[:1], np.array([45], np.int32), scale)
    for i in range(5):
        for h in range(12):
            ref = brute_attention(qp[i, h], ks[0][:, h // 6], vs[0][:, h // 6], scale, 41 + i)
            np.testing.assert_allclose(outp[i, h], ref, rtol=1e-12, atol=1e-13)


def test_tiny_config_brute_force_after_store():
    """The 2-sequence workload: store the step's two tokens, then decode; the
    result equals brute force over the full contiguous sequences, so the
    query sees the key stored in the same step (the context_lens
    one-too-short bug on the pages)."""
    w = synth.tiny_decode()
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.store_kv(w.new_k, w.new_v, kc, vc, w.slot_mapping)
    out = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        n = int(w.context_lens[b])
        for h in range(w.num_q_heads):
            ref = brute_attention(w.q[b, h], w.k_seq[b][:, h // G], w.v_seq[b][:, h // G],
                                  w.scale, n)
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)
    # without the store, the newest key is NaN-poisoned and the output is not finite
    bad = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    assert not np.all(np.isfinite(bad))


def test_decode_permutation_invariance_bitwise():
    """Two different physical placements of the same logical K/V give
    bit-identical oracle output."""
    rng = np.random.default_rng(7)
    Hq, Hkv, D, NB = 12, 2, 128, 96
    lens = [70, 5, 33]
    ks = [normal_bits(rng, (n, Hkv, D)) for n in lens]
    vs = [normal_bits(rng, (n, Hkv, D)) for n in lens]
    q = normal_bits(rng, (3, Hq, D))
    outs = []
    for _ in range(2):
        t = random_tables(rng, lens, NB)
        outs.append(oracle.decode(q, scatter_pool(ks, t, NB), scatter_pool(vs, t, NB), t,
                                  np.array(lens, np.int32), SCALE))
    assert np.array_equal(outs[0], outs[1])


# --------------------------------------------------------------------------
# decode: closed forms
# --------------------------------------------------------------------------

def _single_seq(rng, k_rows, v_rows, q, NB=8):
    t = random_tables(rng, [k_rows.shape[0]], NB)
    return (scatter_pool([k_rows], t, NB), scatter_pool([v_rows], t, NB), t)


def test_single_key_returns_value_exactly():
    """One key: the weight is exactly 1, so o = v exactly."""
    rng = np.random.default_rng(11)
    k, v = normal_bits(rng, (1, 2, 128)), normal_bits(rng, (1, 2, 128))
    q = normal_bits(rng, (1, 12, 128))
    kc, vc, t = _single_seq(rng, k, v, q)
    out = oracle.decode(q, kc, vc, t, np.array([1], np.int32), SCALE)
    for h in range(12):
        assert np.array_equal(out[0, h], bf16_to_f64(v[0, h // 6]))


def test_equal_value_rows_return_that_row():
    """All V rows equal c: any convex combination is c."""
    rng = np.random.default_rng(12)
    n = 45
    c = normal_bits(rng, (2, 128))
    v = np.broadcast_to(c, (n, 2, 128)).copy()
    k = normal_bits(rng, (n, 2, 128))
    q = normal_bits(rng, (1, 12, 128))
    kc, vc, t = _single_seq(rng, k, v, q)
    out = oracle.decode(q, kc, vc, t, np.array([n], np.int32), SCALE)
    for h in range(12):
        np.testing.assert_allclose(out[0, h], bf16_to_f64(c[h // 6]), rtol=1e-14, atol=0)


def test_zero_query_gives_mean_of_values():
    """q = 0: every score is 0, weights are uniform, o = mean of V rows."""
    rng = np.random.default_rng(13)
    n = 29
    k, v = normal_bits(rng, (n, 2, 128)), normal_bits(rng, (n, 2, 128))
    q = np.zeros((1, 12, 128), np.uint16)
    kc, vc, t = _single_seq(rng, k, v, q)
    out = oracle.decode(q, kc, vc, t, np.array([n], np.int32), SCALE)
    for h in range(12):
        np.testing.assert_allclose(out[0, h], bf16_to_f64(v[:, h // 6]).mean(0), rtol=1e-13,
                                   atol=1e-15)


def test_two_keys_closed_form_weights():
    """Two keys with scaled scores 0 and delta = scale * x: the weight of the
    second key is the logistic function of delta (catches a missing or wrong
    scale, a base-2 exponent, or a dropped normaliser)."""
    rng = np.random.default_rng(14)
    D = 128
    x = 3.0                                   # bf16-exact
    q = np.zeros((1, 12, D), np.uint16)
    q[0, :, 0] = bf16_bits(np.float32([1.0]))[0]
    k = np.zeros((2, 2, D), np.uint16)
    k[1, :, 0] = bf16_bits(np.float32([x]))[0]
    v = normal_bits(rng, (2, 2, D))
    kc, vc, t = _single_seq(rng, k, v, q)
    out = oracle.decode(q, kc, vc, t, np.array([2], np.int32), SCALE)
    delta = SCALE * x
    w1 = 1.0 / (1.0 + math.exp(-delta))      # logistic(delta)
    for h in range(12):
        g = h // 6
        ref = (1 - w1) * bf16_to_f64(v[0, g]) + w1 * bf16_to_f64(v[1, g])
        np.testing.assert_allclose(out[0, h], ref, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("Hq,Hkv", [(12, 2), (32, 8), (8, 8), (8, 1)])
def test_gqa_head_map(Hq, Hkv):
    """V of kv head g is the constant g + 1: q head h must return
    h // (Hq / Hkv) + 1 (catches h % Hkv and other head maps)."""
    rng = np.random.default_rng(15)
    n, D = 20, 128
    k = normal_bits(rng, (n, Hkv, D))
    v = np.stack([const_bits(g + 1, (n, D)) for g in range(Hkv)], axis=1)
    q = normal_bits(rng, (1, Hq, D))
    kc, vc, t = _single_seq(rng, k, v, q)
    out = oracle.decode(q, kc, vc, t, np.array([n], np.int32), SCALE)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], h // (Hq // Hkv) + 1, rtol=1e-14)


def test_dominant_key_is_stable():
    """Scores near 1e4 (exp overflows without the max subtraction): the
    output is the value row of the largest score."""
    rng = np.random.default_rng(16)
    n, D = 40, 128
    q = np.zeros((1, 12, D), np.uint16)
    q[0, :, :] = bf16_bits(np.float32([64.0]))[0]
    k = np.zeros((n, 2, D), np.uint16)
    k[:, :, 0] = bf16_bits(np.linspace(1, 10, n).astype(np.float32))[:, None]
    k[17, :, :] = bf16_bits(np.float32([16.0]))[0]        # score 64*16*128*scale ~ 11585
    v = normal_bits(rng, (n, 2, D))
    kc, vc, t = _single_seq(rng, k, v, q)
    out = oracle.decode(q, kc, vc, t, np.array([n], np.int32), SCALE)
    assert np.all(np.isfinite(out))
    for h in range(12):
        np.testing.assert_allclose(out[0, h], bf16_to_f64(v[17, h // 6]), rtol=1e-12)


def test_zero_context_gives_zero_row():
    rng = np.random.default_rng(17)
    k, v = normal_bits(rng, (3, 2, 128)), normal_bits(rng, (3, 2, 128))
    q = normal_bits(rng, (2, 12, 128))
    t = np.array([[2, -1], [-1, -1]], np.int32)
    kc = scatter_pool([k], t[:1], 4)
    vc = scatter_pool([v], t[:1], 4)
    out, lse = oracle.decode(q, kc, vc, t, np.array([3, 0], np.int32), SCALE, with_lse=True)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(out[0]))


# --------------------------------------------------------------------------
# varlen prefill
# --------------------------------------------------------------------------

def test_cu_seqlens_example_from_the_pages():
    """The pages' example: chunks of 3, 1 and 2 tokens -> cu_seqlens
    [0, 3, 4, 6]; each token attends only inside its own sequence.  Values
    of sequence s are the constant s + 1, so row r must return the constant
    of the sequence that owns it."""
    g = json.load(open(os.path.join(GOLDEN, "cu_seqlens_batched_forward.json")))
    q_lens = np.array(g["q_lens"])
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    assert cu.tolist() == g["cu_seqlens"]
    rng = np.random.default_rng(18)
    prefix = np.array([5, 0, 19])
    ctx = prefix + q_lens
    ks = [normal_bits(rng, (n, 2, 128)) for n in ctx]
    vs = [const_bits(s + 1, (n, 2, 128)) for s, n in enumerate(ctx)]
    t = random_tables(rng, ctx, 16)
    out = oracle.prefill_varlen(normal_bits(rng, (6, 12, 128)), cu, scatter_pool(ks, t, 16),
                                scatter_pool(vs, t, 16), t, ctx.astype(np.int32), SCALE)
    for s, rows in enumerate(g["tokens_of_sequence"]):
        for r in rows:
            np.testing.assert_allclose(out[r], s + 1, rtol=1e-14)


def test_causal_boundary_closed_form():
    """q = 0 and V row j = j (bf16-exact): query i of a chunk behind a prefix
    of P keys sees keys 0..P+i, so o = (P + i) / 2 (catches an exclusive
    boundary, a missing prefix, or attention past the diagonal)."""
    rng = np.random.default_rng(19)
    P, L = 37, 21
    n = P + L
    k = normal_bits(rng, (n, 2, 128))
    v = np.stack([const_bits(j, (2, 128)) for j in range(n)])
    t = random_tables(rng, [n], 8)
    q = np.zeros((L, 12, 128), np.uint16)
    out = oracle.prefill_varlen(q, np.array([0, L], np.int32), scatter_pool([k], t, 8),
                                scatter_pool([v], t, 8), t, np.array([n], np.int32), SCALE)
    for i in range(L):
        np.testing.assert_allclose(out[i], (P + i) / 2.0, rtol=1e-14)


def test_prefill_brute_force_contiguous():
    rng = np.random.default_rng(20)
    q_lens = np.array([4, 1, 17])
    prefix = np.array([12, 40, 0])
    ctx = prefix + q_lens
    ks = [normal_bits(rng, (n, 2, 128)) for n in ctx]
    vs = [normal_bits(rng, (n, 2, 128)) for n in ctx]
    t = random_tables(rng, ctx, 32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = normal_bits(rng, (int(q_lens.sum()), 12, 128))
    out = oracle.prefill_varlen(q, cu, scatter_pool(ks, t, 32), scatter_pool(vs, t, 32), t,
                                ctx.astype(np.int32), SCALE)
    for s in range(3):
        for i in range(q_lens[s]):
            r = cu[s] + i
            for h in range(12):
                ref = brute_attention(q[r, h], ks[s][:, h // 6], vs[s][:, h // 6], SCALE,
                                      prefix[s] + i + 1)
                np.testing.assert_allclose(out[r, h], ref, rtol=1e-12, atol=1e-13)


def test_varlen_equals_per_sequence_bitwise():
    """The pages' equivalence: the flattened batch gives, row for row, what
    each sequence gives alone."""
    w = synth.varlen_prefill(chunk=24, n_decode=3, n_chunk=3, max_prefix=60)
    kc, vc = oracle_stored_caches(w)
    full = oracle.prefill_varlen(w.q, w.cu_seqlens, kc, vc, w.block_tables, w.context_lens,
                                 w.scale)
    for s in range(w.batch):
        a, b = w.cu_seqlens[s], w.cu_seqlens[s + 1]
        alone = oracle.prefill_varlen(w.q[a:b], np.array([0, b - a], np.int32), kc, vc,
                                      w.block_tables[s:s + 1], w.context_lens[s:s + 1],
                                      w.scale)
        assert np.array_equal(full[a:b], alone)


def test_decode_equals_prefill_with_one_query_bitwise():
    w = synth.tiny_decode()
    kc, vc = oracle_stored_caches(w)
    dec = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    pre = oracle.prefill_varlen(w.q, np.arange(w.batch + 1, dtype=np.int32), kc, vc,
                                w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(dec, pre)


# --------------------------------------------------------------------------
# split-K partials and the merge
# --------------------------------------------------------------------------

def test_merge_of_splits_equals_unsplit():
    """Partials over any cut of the key range, merged by log-sum-exp, equal
    attention over the whole range (the flash-decoding identity); an empty
    split (lse = -inf) carries no weight."""
    w = synth.qwen_decode_b8()
    kc, vc = oracle_stored_caches(w)
    full = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    rng = np.random.default_rng(21)
    S = 5
    cuts = np.sort(rng.integers(0, w.context_lens[:, None] + 1, size=(w.batch, S - 1)), 1)
    cuts[:, 0] = 0                               # first split empty for every sequence
    bounds = np.concatenate([np.zeros((w.batch, 1), int), cuts,
                             w.context_lens[:, None]], 1)
    po = np.zeros((w.batch, w.num_q_heads, S, w.head_dim))
    pl = np.zeros((w.batch, w.num_q_heads, S))
    for s in range(S):
        o, l = oracle.decode_range(w.q, kc, vc, w.block_tables, bounds[:, s], bounds[:, s + 1],
                                   w.scale)
        po[:, :, s], pl[:, :, s] = o, l
    assert np.all(np.isneginf(pl[:, :, 0]))
    merged = oracle.merge(po.reshape(-1, S, w.head_dim), pl.reshape(-1, S))
    np.testing.assert_allclose(merged.reshape(full.shape), full, rtol=1e-11, atol=1e-13)


def test_merge_single_split_is_identity_and_all_empty_is_zero():
    rng = np.random.default_rng(22)
    po = rng.standard_normal((7, 1, 128))
    pl = rng.standard_normal((7, 1))
    assert np.array_equal(oracle.merge(po, pl), po[:, 0])
    pl2 = np.full((3, 4), -np.inf)
    assert np.all(oracle.merge(rng.standard_normal((3, 4, 128)), pl2) == 0)


def test_decode_range_full_range_matches_decode_lse():
    w = synth.tiny_decode()
    kc, vc = oracle_stored_caches(w)
    o1, l1 = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                           with_lse=True)
    o2, l2 = oracle.decode_range(w.q, kc, vc, w.block_tables, np.zeros(w.batch, np.int32),
                                 w.context_lens, w.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # lse closed form for one sequence/head: log of the sum of exp(scores)
    G = w.num_q_heads // w.num_kv_heads
    K = bf16_to_f64(w.k_seq[0][:, 0])
    s = w.scale * (K @ bf16_to_f64(w.q[0, 0]))
    assert abs(l1[0, 0] - np.log(np.exp(s).sum())) < 1e-12
    assert G == 6


def test_synth_slot_mapping_places_new_token_at_last_position():
    """The step's new token of sequence b goes to the slot of position
    context_lens[b] - 1 through b's own block table row."""
    w = synth.cb_decode_b64()
    bs = w.block_size
    pos = w.context_lens - 1
    expect = w.block_tables[np.arange(w.batch), pos // bs] * bs + pos % bs
    assert np.array_equal(w.slot_mapping, expect)
    assert np.all(w.context_lens >= 1) and np.all(w.context_lens <= 8192)


# --------------------------------------------------------------------------
# rotary embedding (fused RoPE + store)
# --------------------------------------------------------------------------

def _rope_tables(max_pos, D, base=10000.0):
    """Standard RoPE angles theta_{p,i} = p * base^(-2i/D), as float32 tables."""
    inv = base ** (-np.arange(D // 2, dtype=np.float64) * 2.0 / D)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def test_rope_complex_form():
    """Rotate-half RoPE is multiplication of the complex numbers
    x_i + j x_{i+D/2} by c + j s ([EAS] day 4-5: the complex form the
    table-lookup version replaced).  Catches a sign error in either term,
    an interleaved (2i, 2i+1) pairing and a wrong table row or column."""
    rng = np.random.default_rng(31)
    T, H, D, P = 9, 3, 128, 64
    x = normal_bits(rng, (T, H, D))
    pos = rng.integers(0, P, T).astype(np.int32)
    cos_t = rng.uniform(-1, 1, (P, D // 2)).astype(np.float32)   # arbitrary angles,
    sin_t = rng.uniform(-1, 1, (P, D // 2)).astype(np.float32)   # not unit: any table
    out = oracle.rope(x, pos, cos_t, sin_t)
    xf = bf16_to_f64(x)
    z = xf[..., :D // 2] + 1j * xf[..., D // 2:]
    w = cos_t[pos].astype(np.float64) + 1j * sin_t[pos].astype(np.float64)
    r = z * w[:, None, :]
    assert np.allclose(out[..., :D // 2], r.real, rtol=1e-14, atol=1e-14)
    assert np.allclose(out[..., D // 2:], r.imag, rtol=1e-14, atol=1e-14)


def test_rope_position_zero_is_identity_and_norms_are_kept():
    """cos 1 / sin 0 returns the input exactly; unit (cos, sin) keeps the
    norm of every (i, i + D/2) pair (catches a scaled or mixed-up term)."""
    rng = np.random.default_rng(32)
    T, H, D = 6, 2, 128
    x = normal_bits(rng, (T, H, D))
    cos_t, sin_t = _rope_tables(4096, D)
    zero = np.zeros(T, np.int32)
    assert np.array_equal(oracle.rope(x, zero, cos_t, sin_t), bf16_to_f64(x))
    pos = rng.integers(0, 4096, T).astype(np.int32)
    out = oracle.rope(x, pos, cos_t, sin_t)
    xf = bf16_to_f64(x)
    n_in = xf[..., :D // 2] ** 2 + xf[..., D // 2:] ** 2
    n_out = out[..., :D // 2] ** 2 + out[..., D // 2:] ** 2
    unit = (cos_t[pos].astype(np.float64) ** 2 + sin_t[pos].astype(np.float64) ** 2)[:, None, :]
    assert np.allclose(n_out, n_in * unit, rtol=1e-12, atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    """The defining property of RoPE: <R(q, m), R(k, n)> depends on m - n
    alone.  With standard frequency tables, shifting both positions by the
    same amount leaves the score unchanged up to the float32 table rounding
    (catches using the token index instead of positions[t], and an angle
    applied with the wrong sign on one side)."""
    rng = np.random.default_rng(33)
    D = 128
    cos_t, sin_t = _rope_tables(8192, D)
    q = normal_bits(rng, (1, 1, D))
    k = normal_bits(rng, (1, 1, D))
    scores = []
    for shift in (0, 37, 1000, 5000):
        m, n = np.array([100 + shift], np.int32), np.array([60 + shift], np.int32)
        qr = oracle.rope(q, m, cos_t, sin_t)
        kr = oracle.rope(k, n, cos_t, sin_t)
        scores.append(float(np.sum(qr * kr)))
    mag = float(np.sum(np.abs(bf16_to_f64(q)) * np.abs(bf16_to_f64(k))))
    assert max(scores) - min(scores) < 1e-5 * mag
    # and the score does move with the offset itself
    qr = oracle.rope(q, np.array([100], np.int32), cos_t, sin_t)
    kr = oracle.rope(k, np.array([90], np.int32), cos_t, sin_t)
    assert abs(float(np.sum(qr * kr)) - scores[0]) > 1e-3 * mag


def test_rope_uses_each_tokens_position():
    """Tokens rotated in one call equal tokens rotated one at a time, and
    permuting the tokens (with their positions) permutes the output."""
    rng = np.random.default_rng(34)
    T, H, D = 8, 2, 128
    x = normal_bits(rng, (T, H, D))
    cos_t, sin_t = _rope_tables(512, D)
    pos = rng.integers(0, 512, T).astype(np.int32)
    full = oracle.rope(x, pos, cos_t, sin_t)
    for t in range(T):
        one = oracle.rope(x[t:t + 1], pos[t:t + 1], cos_t, sin_t)
        assert np.array_equal(one[0], full[t])
    perm = rng.permutation(T)
    assert np.array_equal(oracle.rope(np.ascontiguousarray(x[perm]), pos[perm], cos_t, sin_t),
                          full[perm])


def test_rope_store_places_rounded_rotated_k_and_plain_v():
    """The fused store: v lands bit-for-bit, k lands as its rotation rounded
    once to bf16 (checked against float32 arithmetic where it is exact),
    through slot_mapping with padding skipped; other slots untouched."""
    rng = np.random.default_rng(35)
    NB, bs, Hq, Hkv, D, T = 16, 16, 12, 2, 128, 24
    qkv = normal_bits(rng, (T, Hq + 2 * Hkv, D))
    q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    cos_t, sin_t = _rope_tables(2048, D)
    pos = rng.integers(0, 2048, T).astype(np.int32)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    slots[5] = -1
    kc = np.full((NB, bs, Hkv, D), 0x1234, np.uint16)
    vc = np.full((NB, bs, Hkv, D), 0x4321, np.uint16)
    q_rot, k_rot = oracle.rope_store_kv(q, k, v, pos, cos_t, sin_t, kc, vc, slots)
    assert np.array_equal(q_rot, oracle.rope(q, pos, cos_t, sin_t))
    fk, fv = kc.reshape(NB * bs, Hkv, D), vc.reshape(NB * bs, Hkv, D)
    ok = slots >= 0
    assert np.array_equal(fv[slots[ok]], v[ok])
    stored = bf16_to_f64(fk[slots[ok]])
    exact = k_rot[ok]
    # one rounding to nearest: within half a bf16 ulp (8 significant bits:
    # at most 2^-8 relative) and equal to the independent rounding below
    assert np.all(np.abs(stored - exact) <= np.abs(exact) * 2.0 ** -8)
    assert np.array_equal(fk[slots[ok]], oracle.round_to_bf16_bits(exact))
    untouched = np.ones(NB * bs, bool)
    untouched[slots[ok]] = False
    assert np.all(fk[untouched] == 0x1234) and np.all(fv[untouched] == 0x4321)


def test_round_to_bf16_bits_ties_and_carries():
    """Round-to-nearest-even at the halfway points, and the carry into the
    exponent; equal to float32 rounding where float32 holds the value."""
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -30,
                  -(1.0 + 2 ** -8), 2.0 - 2 ** -9, 3.0, 0.0])
    got = (oracle.round_to_bf16_bits(x).astype(np.uint32) << 16).view(np.float32)
    assert got.tolist() == [1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -1.0, 2.0, 3.0, 0.0]
    rng = np.random.default_rng(36)
    f = rng.standard_normal(1000).astype(np.float32)
    # float32 -> bf16 by integer rounding of the bit pattern (ties to even)
    u = f.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(oracle.round_to_bf16_bits(f.astype(np.float64)), ref)


# --------------------------------------------------------------------------
# FP8 (E4M3) KV cache
# --------------------------------------------------------------------------

def test_e4m3_values_closed_forms_and_library():
    """Closed forms of the format (largest finite 448, smallest subnormal
    2^-9, smallest normal 2^-6, one = 0x38, NaN = 0x7F) and agreement with
    torch's float8_e4m3fn widening on all 256 codes (an independent
    implementation of the same format)."""
    v = oracle.e4m3_values()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6 and v[0x38] == 1.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and v[0x80] == 0.0
    assert np.all(np.diff(v[:127]) > 0)           # codes 0..126 increase
    torch = pytest.importorskip("torch")
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    assert np.array_equal(np.nan_to_num(v, nan=7e7), np.nan_to_num(lib, nan=7e7))


def test_e4m3_encode_round_trip_ties_and_saturation():
    """Every finite code encodes back to itself; a value halfway between two
    codes goes to the even one; beyond 448 saturates; agreement with torch's
    float32 -> float8_e4m3fn rounding on random in-range values."""
    v = oracle.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(v[c]) and c != 0x80])
    assert np.array_equal(oracle.e4m3_encode(v[finite]), finite.astype(np.uint8))
    mids = (v[0:126] + v[1:127]) / 2.0
    got = oracle.e4m3_encode(mids)
    even = np.where(np.arange(126) % 2 == 0, np.arange(126), np.arange(1, 127))
    assert np.array_equal(got, even.astype(np.uint8))
    assert oracle.e4m3_encode(np.array([449.0, 500.0, 1e30]))[0] == 0x7E
    assert oracle.e4m3_encode(np.array([-1e30]))[0] == 0xFE
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(41)
    y = (rng.standard_normal(20000) * 50).astype(np.float32)
    y = y[np.abs(y) < 440]
    lib = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(y), lib)


def test_store_kv_fp8_layout_and_quantisation():
    """K codes land token-major at [block][row][h], V codes dim-major at
    [block][h][:][row]; codes are the rounding of x / scale[h] in float32;
    padding skipped; other slots untouched."""
    rng = np.random.default_rng(42)
    NB, bs, Hkv, D, T = 8, 16, 2, 128, 10
    k = normal_bits(rng, (T, Hkv, D))
    v = normal_bits(rng, (T, Hkv, D))
    ks = np.array([0.01, 0.02], np.float32)
    vs = np.array([0.015, 0.005], np.float32)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    slots[4] = -1
    kp = np.full((NB, bs, Hkv, D), 0x55, np.uint8)
    vp = np.full((NB, Hkv, D, bs), 0x66, np.uint8)
    oracle.store_kv_fp8(k, v, kp, vp, ks, vs, slots)
    for t in range(T):
        if slots[t] < 0:
            continue
        blk, row = divmod(int(slots[t]), bs)
        for h in range(Hkv):
            kf = bf16_to_f64(k[t, h]).astype(np.float32) / ks[h]
            vf = bf16_to_f64(v[t, h]).astype(np.float32) / vs[h]
            assert np.array_equal(kp[blk, row, h], oracle.e4m3_encode(kf))
            assert np.array_equal(vp[blk, h, :, row], oracle.e4m3_encode(vf))
    live = slots[slots >= 0]
    mask = np.ones(NB * bs, bool)
    mask[live] = False
    assert np.all(kp.reshape(NB * bs, Hkv, D)[mask] == 0x55)
    vflat = vp.transpose(0, 3, 1, 2).reshape(NB * bs, Hkv, D)
    assert np.all(vflat[mask] == 0x66)


def test_decode_fp8_equals_bf16_decode_on_exact_values():
    """With power-of-two scales every code * scale is exactly a bf16 value:
    the FP8 decode must then equal the (pinned) bf16 decode bit for bit over
    pools holding those values (catches a wrong scale, a wrong head's scale,
    or V read in the token-major order)."""
    rng = np.random.default_rng(43)
    NB, bs, Hq, Hkv, D = 24, 16, 12, 2, 128
    ctx = np.array([1, 17, 40, 100], np.int32)
    tables = random_tables(rng, ctx, NB)
    ks = np.array([0.125, 2.0], np.float32)
    vs = np.array([0.5, 0.0625], np.float32)
    v = oracle.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(v[c])], np.uint8)
    kp = rng.choice(finite, size=(NB, bs, Hkv, D)).astype(np.uint8)
    vp = rng.choice(finite, size=(NB, Hkv, D, bs)).astype(np.uint8)
    # the widened pools written out from the definition, head by head and row
    # by row (value of the code times its own kv head's scale; V dim-major)
    kf = np.empty((NB, bs, Hkv, D))
    vf = np.empty((NB, bs, Hkv, D))
    for h in range(Hkv):
        kf[:, :, h, :] = v[kp[:, :, h, :]] * float(ks[h])
        for r in range(bs):
            vf[:, r, h, :] = v[vp[:, h, :, r]] * float(vs[h])
    got_k, got_v = oracle.dequantize_pools_fp8(kp, vp, ks, vs)
    assert np.array_equal(got_k, kf) and np.array_equal(got_v, vf)
    kb, vb = bf16_bits(kf.astype(np.float32)), bf16_bits(vf.astype(np.float32))
    assert np.array_equal(bf16_to_f64(kb), kf) and np.array_equal(bf16_to_f64(vb), vf)
    q = normal_bits(rng, (len(ctx), Hq, D))
    a = oracle.decode(q, kb, vb, tables, ctx, SCALE)
    b = oracle.decode_fp8(q, kp, vp, ks, vs, tables, ctx, SCALE)
    assert np.array_equal(a, b)
    # and the V layout matters: reading V token-major gives something else
    wrong = oracle.decode_fp8(q, kp, np.ascontiguousarray(
        vp.transpose(0, 1, 3, 2)).reshape(NB, Hkv, D, bs), ks, vs, tables, ctx, SCALE)
    assert not np.allclose(wrong, a)
