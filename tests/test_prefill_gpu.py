"""GPU parity of pa_prefill_varlen (tcgen05 path) against the oracle.

The step's new tokens are first placed with pa_store_kv (on the GPU), then
the varlen prefill attends over each sequence's paged keys, as in a
chunked-prefill step.  Tolerance as for decode: every element within
2e-3 + 1e-2 |ref|; fp32 outputs also max-abs 2e-3 / max-rel 1e-2."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import (assert_attention_close, const_bits, dev_to_f64, normal_bits,
                           oracle_stored_caches, random_tables, scatter_pool, to_dev_bf16,
                           to_dev_i32)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


def gpu_prefill(ops, w, out_dtype=torch.float32, max_q_len=None, err=None, store=True):
    q = to_dev_bf16(w.q)
    if store:
        kc, vc = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
        ops.store_kv(to_dev_bf16(w.new_k), to_dev_bf16(w.new_v), kc, vc,
                     to_dev_i32(w.slot_mapping))
    else:
        kcn, vcn = w.stored_caches()
        kc, vc = to_dev_bf16(kcn), to_dev_bf16(vcn)
    mq = int(w.q_lens.max()) if max_q_len is None else max_q_len
    out = ops.prefill_varlen(q, to_dev_i32(w.cu_seqlens), kc, vc, to_dev_i32(w.block_tables),
                             to_dev_i32(w.context_lens), w.scale, mq, out_dtype=out_dtype,
                             error_flags=err)
    torch.cuda.synchronize()
    return out


def oracle_prefill(w):
    """The oracle over the whole launch, on pools placed by the oracle's store."""
    kc, vc = oracle_stored_caches(w)
    return oracle.prefill_varlen(w.q, w.cu_seqlens, kc, vc, w.block_tables, w.context_lens,
                                 w.scale)


@pytest.fixture(scope="module")
def full_mix():
    """The full 8 x 1 + 8 x 512 chunked-prefill mix (prefixes up to 2048) and
    the oracle's answer for every one of its 4104 rows."""
    w = synth.varlen_prefill(keep_seq=False)
    return w, oracle_prefill(w)


def test_prefill_reduced_mix_all_rows(ops):
    """8 one-token rows and 8 chunks of 200 queries behind prefixes up to
    600: every output row against the oracle, bf16 and fp32 outputs."""
    w = synth.varlen_prefill(chunk=200, max_prefix=600)
    ref = oracle_prefill(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = dev_to_f64(gpu_prefill(ops, w, torch.float32, err=err))
    assert int(err.item()) == 0
    assert_attention_close(got, ref, "prefill f32", strict=True)
    assert_attention_close(dev_to_f64(gpu_prefill(ops, w, torch.bfloat16)), ref, "prefill bf16")


def test_prefill_full_workload_all_sequences(ops, full_mix):
    """The full mix in the launch the bench times: all 16 sequences (every
    row, every head) against the oracle over the whole launch, fp32 output
    held to the strict rule, bf16 output to the elementwise rule."""
    w, ref = full_mix
    got = dev_to_f64(gpu_prefill(ops, w))
    for s in range(w.batch):
        a, b = int(w.cu_seqlens[s]), int(w.cu_seqlens[s + 1])
        assert_attention_close(got[a:b], ref[a:b], f"sequence {s} (q_len {b - a})", strict=True)
    assert_attention_close(dev_to_f64(gpu_prefill(ops, w, torch.bfloat16)), ref,
                           "full mix bf16")


def test_prefill_cu_seqlens_example_from_the_pages(ops):
    """cu_seqlens [0, 3, 4, 6]: chunks of 3, 1, 2 tokens; V of sequence s is
    the constant s + 1, so each row returns its own sequence's constant."""
    g = json.load(open(os.path.join(GOLDEN, "cu_seqlens_batched_forward.json")))
    q_lens = np.array(g["q_lens"])
    cu = np.array(g["cu_seqlens"], np.int32)
    rng = np.random.default_rng(61)
    prefix = np.array([5, 0, 19])
    ctx = prefix + q_lens
    ks = [normal_bits(rng, (n, 2, 128)) for n in ctx]
    vs = [const_bits(s + 1, (n, 2, 128)) for s, n in enumerate(ctx)]
    t = random_tables(rng, ctx, 16)
    q = to_dev_bf16(normal_bits(rng, (6, 12, 128)))
    out = ops.prefill_varlen(q, to_dev_i32(cu), to_dev_bf16(scatter_pool(ks, t, 16)),
                             to_dev_bf16(scatter_pool(vs, t, 16)), to_dev_i32(t),
                             to_dev_i32(ctx), 128 ** -0.5, 3, out_dtype=torch.float32)
    o = out.cpu().numpy()
    for s, rows in enumerate(g["tokens_of_sequence"]):
        for r in rows:
            np.testing.assert_allclose(o[r], s + 1, rtol=1e-5)  # hi+lo bf16 weights: ~2^-16


@pytest.mark.parametrize("hq,hkv", [(12, 2), (32, 8), (8, 1), (7, 1), (16, 4), (8, 8)])
def test_prefill_head_shapes_and_ragged_lengths(ops, hq, hkv):
    rng = np.random.default_rng(hq * 10 + hkv)
    q_lens = np.array([1, 17, 130, 5, 64])
    prefix = np.array([0, 300, 1, 129, 16])
    w = synth.make_paged(rng, "shapes", prefix + q_lens, q_lens, num_blocks=200,
                         num_q_heads=hq, num_kv_heads=hkv)
    got = dev_to_f64(gpu_prefill(ops, w))
    assert_attention_close(got, oracle_prefill(w), f"hq={hq} hkv={hkv}", strict=True)


@pytest.mark.parametrize("scale", [-3.0, -0.088, 0.0])
def test_prefill_scale_sign(ops, scale):
    """Negative softmax scales (the larger one gives near one-hot weights)
    and a zero one (every visible key weighs the same), on diagonal and
    ragged tiles, with the fused store too."""
    rng = np.random.default_rng(77 + int(abs(scale) * 1000))
    q_lens = np.array([1, 17, 130, 5, 64])
    prefix = np.array([0, 300, 1, 129, 16])
    w = synth.make_paged(rng, "scale", prefix + q_lens, q_lens, num_blocks=200,
                         num_q_heads=12, num_kv_heads=2, scale=scale)
    ref = oracle_prefill(w)
    assert_attention_close(dev_to_f64(gpu_prefill(ops, w)), ref, f"scale={scale}", strict=True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _, _ = fused_prefill(ops, w, err=err)
    assert int(err.item()) == 0
    assert_attention_close(dev_to_f64(out), ref, f"fused store, scale={scale}", strict=True)


def test_prefill_many_sequences_grid_order(ops):
    """More sequences than a CTA has threads (300 short chunks behind short
    prefixes, some empty): the CTAs take their tiles in grid order instead
    of the longest-first pick; every row against the oracle."""
    rng = np.random.default_rng(300)
    q_lens = rng.integers(0, 5, size=300)
    q_lens[0] = 4
    prefix = rng.integers(0, 40, size=300)
    w = synth.make_paged(rng, "many_seqs", prefix + q_lens, q_lens, num_blocks=1000,
                         num_q_heads=12, num_kv_heads=2)
    got = dev_to_f64(gpu_prefill(ops, w))
    assert_attention_close(got, oracle_prefill(w), "300 sequences", strict=True)


def test_prefill_varlen_equals_per_sequence_bitwise(ops):
    """The pages' equivalence: each sequence's rows of the batched call are
    bit-identical to a call with that sequence alone."""
    w = synth.varlen_prefill(chunk=150, max_prefix=300)
    full = gpu_prefill(ops, w, store=False).cpu().numpy()
    kcn, vcn = w.stored_caches()
    kc, vc = to_dev_bf16(kcn), to_dev_bf16(vcn)
    for s in range(w.batch):
        a, b = int(w.cu_seqlens[s]), int(w.cu_seqlens[s + 1])
        alone = ops.prefill_varlen(to_dev_bf16(w.q[a:b]), to_dev_i32([0, b - a]), kc, vc,
                                   to_dev_i32(w.block_tables[s:s + 1]),
                                   to_dev_i32(w.context_lens[s:s + 1]), w.scale, b - a,
                                   out_dtype=torch.float32).cpu().numpy()
        assert np.array_equal(full[a:b], alone)


def test_prefill_one_token_rows_match_decode(ops):
    """A sequence with q_len 1 is a decode row: same answer as pa_decode."""
    w = synth.cb_decode_b64()
    kcn, vcn = w.stored_caches()
    kc, vc = to_dev_bf16(kcn), to_dev_bf16(vcn)
    q = to_dev_bf16(w.q)
    tables, ctx = to_dev_i32(w.block_tables), to_dev_i32(w.context_lens)
    pre = ops.prefill_varlen(q, to_dev_i32(np.arange(w.batch + 1)), kc, vc, tables, ctx, w.scale,
                             1, out_dtype=torch.float32)
    dec = ops.decode(q, kc, vc, tables, ctx, w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_attention_close(dev_to_f64(pre), dev_to_f64(dec), "prefill q_len 1 vs decode",
                           strict=True)


def test_prefill_causal_closed_form(ops):
    """q = 0, V row j = j: query i behind a prefix of P keys returns (P+i)/2."""
    rng = np.random.default_rng(71)
    P, L = 150, 140
    n = P + L
    k = normal_bits(rng, (n, 2, 128))
    v = np.stack([const_bits(min(j, 255), (2, 128)) for j in range(n)])
    t = random_tables(rng, [n], 40)
    q = torch.zeros((L, 12, 128), dtype=torch.bfloat16, device="cuda")
    out = ops.prefill_varlen(q, to_dev_i32([0, L]), to_dev_bf16(scatter_pool([k], t, 40)),
                             to_dev_bf16(scatter_pool([v], t, 40)), to_dev_i32(t),
                             to_dev_i32([n]), 128 ** -0.5, L, out_dtype=torch.float32)
    vv = np.minimum(np.arange(n), 255).astype(np.float64)
    o = out.cpu().numpy()
    for i in range(L):
        np.testing.assert_allclose(o[i], vv[:P + i + 1].mean(), rtol=2e-3)


def test_prefill_shape_errors_are_reported(ops):
    """q_len > context (negative prefix) and q_len > max_q_len set
    PA_DEVERR_SHAPE without faulting."""
    w = synth.varlen_prefill(chunk=40, max_prefix=50)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_prefill(ops, w, max_q_len=20, err=err)
    assert int(err.item()) & ops.DEVERR_SHAPE
    bad = synth.varlen_prefill(chunk=40, max_prefix=50)
    bad.context_lens = bad.context_lens.copy()
    bad.context_lens[int(np.argmax(bad.q_lens))] = 3
    err.zero_()
    gpu_prefill(ops, bad, err=err, store=False)
    assert int(err.item()) & ops.DEVERR_SHAPE


# --------------------------------------------------------------------------
# pa_prefill_store_varlen: the chunks' store fused into the prefill
# --------------------------------------------------------------------------

def fused_prefill(ops, w, out_dtype=torch.float32, err=None):
    q = to_dev_bf16(w.q)
    kc, vc = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    out = ops.prefill_store_varlen(q, to_dev_bf16(w.new_k), to_dev_bf16(w.new_v),
                                   to_dev_i32(w.slot_mapping), to_dev_i32(w.cu_seqlens), kc, vc,
                                   to_dev_i32(w.block_tables), to_dev_i32(w.context_lens),
                                   w.scale, int(w.q_lens.max()), out_dtype=out_dtype,
                                   error_flags=err)
    torch.cuda.synchronize()
    return out, kc, vc


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("hq,hkv", [(12, 2), (32, 8), (8, 1), (16, 4)])
def test_prefill_store_equals_store_then_prefill(ops, hq, hkv):
    """Chunk pages read from the new rows, the page that straddles the
    prefix assembled from both (prefixes 0, 1, 16, 129, 300): the output
    equals pa_store_kv + pa_prefill_varlen bit for bit, the pools equal the
    oracle's store, and the result matches the oracle."""
    rng = np.random.default_rng(900 + hq * 10 + hkv)
    q_lens = np.array([1, 17, 130, 5, 64])
    prefix = np.array([0, 300, 1, 129, 16])
    w = synth.make_paged(rng, "fused_shapes", prefix + q_lens, q_lens, num_blocks=200,
                         num_q_heads=hq, num_kv_heads=hkv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_f, kc, vc = fused_prefill(ops, w, err=err)
    assert int(err.item()) == 0
    out_u = gpu_prefill(ops, w)
    assert torch.equal(out_f, out_u)
    kref, vref = oracle_stored_caches(w)
    assert np.array_equal(_bits(kc), kref) and np.array_equal(_bits(vc), vref)
    assert_attention_close(dev_to_f64(out_f), oracle_prefill(w), f"fused hq={hq} hkv={hkv}",
                           strict=True)


def test_prefill_store_full_workload(ops, full_mix):
    """The varlen_prefill workload (8 one-token rows + 8 chunks of 512):
    fused equals store + prefill bit for bit; pools as the oracle's store;
    every row against the oracle (bf16 output: elementwise rule; fp32
    output: strict)."""
    w, ref = full_mix
    out_f, kc, vc = fused_prefill(ops, w, out_dtype=torch.bfloat16)
    out_u = gpu_prefill(ops, w, out_dtype=torch.bfloat16)
    assert torch.equal(out_f.view(torch.int16), out_u.view(torch.int16))
    kref, vref = oracle_stored_caches(w)
    assert np.array_equal(_bits(kc), kref) and np.array_equal(_bits(vc), vref)
    assert_attention_close(dev_to_f64(out_f), ref, "fused full mix bf16")
    out_f32, _, _ = fused_prefill(ops, w, out_dtype=torch.float32)
    assert_attention_close(dev_to_f64(out_f32), ref, "fused full mix f32", strict=True)


def test_prefill_store_bad_slot_reported(ops):
    rng = np.random.default_rng(77)
    q_lens = np.array([20, 3])
    prefix = np.array([5, 40])
    w = synth.make_paged(rng, "fused_bad", prefix + q_lens, q_lens, num_blocks=40)
    w.slot_mapping[4] = w.num_blocks * 16 + 7
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fused_prefill(ops, w, err=err)
    assert int(err.item()) & ops.DEVERR_SLOT_INDEX
