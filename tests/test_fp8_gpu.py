"""GPU parity of the FP8 (E4M3) KV cache against the oracle.

pa_store_kv_fp8 must write the oracle's codes bit for bit (the quantised
code is an integer decided in float32: IEEE division, nearest even,
saturation).  pa_decode_fp8 is compared element by element with the oracle's
attention over the widened pools (code * scale), within 2e-3 + 1e-2 |ref|:
the codes widen exactly, q is exact in f16 for these magnitudes and P keeps
~22 bits (f16 hi + lo), so the bound of the bf16 path carries over."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import bf16_dev_to_bits, normal_bits, random_tables, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


def fp8_pools_from(w, ks, vs):
    """Quantise a workload's bf16 pools into the FP8 layouts.  Unused slots
    (bf16 NaN) get the NaN code 0x7F; only the live rows are quantised."""
    NB, bs, Hkv, D = w.k_cache.shape
    kf = w.k_cache.reshape(NB * bs, Hkv, D)
    vf = w.v_cache.reshape(NB * bs, Hkv, D)
    live = np.flatnonzero(np.any(kf.reshape(NB * bs, -1) != synth.BF16_NAN, axis=1))
    kq = np.full((NB * bs, Hkv, D), 0x7F, np.uint8)
    vq = np.full((NB * bs, Hkv, D), 0x7F, np.uint8)
    kq[live] = oracle.quantize_fp8(kf[live], ks)
    vq[live] = oracle.quantize_fp8(vf[live], vs)
    kp = kq.reshape(NB, bs, Hkv, D)
    vp = np.ascontiguousarray(vq.reshape(NB, bs, Hkv, D).transpose(0, 2, 3, 1))
    return kp, vp


def compact(kp, vp, tables):
    """The pools restricted to the blocks the tables reference, and the
    tables renumbered (the oracle's result does not depend on placement)."""
    used = np.unique(tables[tables >= 0])
    remap = np.full(kp.shape[0], -1, np.int64)
    remap[used] = np.arange(used.shape[0])
    t2 = np.where(tables >= 0, remap[np.maximum(tables, 0)], -1).astype(np.int32)
    return np.ascontiguousarray(kp[used]), np.ascontiguousarray(vp[used]), t2


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_step(ops, w, ks, vs, num_splits=0, out_dtype=torch.float32):
    kp, vp = fp8_pools_from(w, ks, vs)
    kref, vref = kp.copy(), vp.copy()
    oracle.store_kv_fp8(w.new_k, w.new_v, kref, vref, ks, vs, w.slot_mapping)
    kd, vd = dev_u8(kp), dev_u8(vp)
    ksd, vsd = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.store_kv_fp8(to_dev_bf16(w.new_k), to_dev_bf16(w.new_v), kd, vd, ksd, vsd,
                     to_dev_i32(w.slot_mapping), error_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(kd.cpu().numpy(), kref), "K codes differ from the oracle's"
    assert np.array_equal(vd.cpu().numpy(), vref), "V codes differ from the oracle's"
    out = ops.decode_fp8(to_dev_bf16(w.q), kd, vd, ksd, vsd, to_dev_i32(w.block_tables),
                         to_dev_i32(w.context_lens), w.scale, out_dtype=out_dtype,
                         num_splits=num_splits)
    torch.cuda.synchronize()
    kc, vc, t2 = compact(kref, vref, w.block_tables)
    ref = oracle.decode_fp8(w.q, kc, vc, ks, vs, t2, w.context_lens, w.scale)
    got = out.float().cpu().numpy().astype(np.float64)
    return got, ref


def assert_close(got, ref):
    err = np.abs(got - ref)
    bound = 2e-3 + 1e-2 * np.abs(ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= bound), f"max excess {float(np.max(err - bound))}"


@pytest.mark.parametrize("name", ["tiny_decode", "qwen_decode_b8", "cb_decode_b64"])
def test_fp8_store_and_decode_workloads(ops, name):
    w = synth.CONFIGS[name]()
    ks = np.array([0.011, 0.0095], np.float32)[:w.num_kv_heads]
    vs = np.array([0.0105, 0.012], np.float32)[:w.num_kv_heads]
    got, ref = run_step(ops, w, ks, vs)
    assert_close(got, ref)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (4, 4), (32, 8), (16, 2), (2, 2)])
@pytest.mark.parametrize("num_splits", [0, 7])
def test_fp8_gqa_shapes_and_splits(ops, Hq, Hkv, num_splits):
    """Every kv-head count, group sizes 1..8, the default split count and a
    small one (long sequences cut across splits: partials and merges)."""
    rng = np.random.default_rng(500 + Hq * 10 + Hkv + num_splits)
    ctx = rng.integers(1, 700, size=6)
    ctx[0], ctx[1] = 1, 16
    w = synth.make_paged(rng, "fp8_shape", ctx, np.ones(6, np.int64), num_blocks=400,
                         num_q_heads=Hq, num_kv_heads=Hkv)
    ks = rng.uniform(0.008, 0.012, Hkv).astype(np.float32)
    vs = rng.uniform(0.008, 0.012, Hkv).astype(np.float32)
    got, ref = run_step(ops, w, ks, vs, num_splits=num_splits)
    assert_close(got, ref)


@pytest.mark.parametrize("scale", [-3.0, 0.0])
@pytest.mark.parametrize("Hq,Hkv", [(12, 2), (32, 8)])
def test_fp8_softmax_scale_sign(ops, scale, Hq, Hkv):
    """A negative softmax scale (near one-hot weights at this size) and a zero
    one (every key weighs the same), with the K scale folded into it."""
    rng = np.random.default_rng(700 + Hq + int(abs(scale)))
    ctx = np.array([900, 1, 37, 260])
    w = synth.make_paged(rng, "fp8_scale", ctx, np.ones(4, np.int64), num_blocks=128,
                         num_q_heads=Hq, num_kv_heads=Hkv, scale=scale)
    ks = rng.uniform(0.008, 0.012, Hkv).astype(np.float32)
    vs = rng.uniform(0.008, 0.012, Hkv).astype(np.float32)
    got, ref = run_step(ops, w, ks, vs)
    assert_close(got, ref)


def test_fp8_saturating_scale_and_bf16_output(ops):
    """A scale small enough that many values saturate at +-448 codes, and a
    bf16 output (held to the elementwise rule)."""
    w = synth.qwen_decode_b8()
    ks = np.array([0.004, 0.003], np.float32)
    vs = np.array([0.0035, 0.005], np.float32)
    got, ref = run_step(ops, w, ks, vs, out_dtype=torch.bfloat16)
    assert_close(got, ref)


def test_fp8_store_padding_strides_and_bad_slot(ops):
    """Padding tokens skipped, strided fused-QKV views, a slot past the pool
    reported (PA_DEVERR_SLOT_INDEX) and skipped."""
    rng = np.random.default_rng(9)
    NB, Hq, Hkv, D, T = 20, 12, 2, 128, 100
    qkv_bits = normal_bits(rng, (T, Hq + 2 * Hkv, D))
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int32)
    slots[::9] = -1
    slots[5] = NB * 16 + 3
    ks = np.array([0.01, 0.02], np.float32)
    vs = np.array([0.015, 0.01], np.float32)
    kp0 = np.full((NB, 16, Hkv, D), 0x11, np.uint8)
    vp0 = np.full((NB, Hkv, D, 16), 0x22, np.uint8)
    kref, vref = kp0.copy(), vp0.copy()
    good = slots < NB * 16
    oracle.store_kv_fp8(qkv_bits[good][:, Hq:Hq + Hkv], qkv_bits[good][:, Hq + Hkv:], kref,
                        vref, ks, vs, slots[good])
    qkv = to_dev_bf16(qkv_bits)
    kd, vd = dev_u8(kp0), dev_u8(vp0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.store_kv_fp8(qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:], kd, vd,
                     torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(), to_dev_i32(slots),
                     error_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DEVERR_SLOT_INDEX
    assert np.array_equal(kd.cpu().numpy(), kref) and np.array_equal(vd.cpu().numpy(), vref)


def test_fp8_decode_empty_and_single_key_rows(ops):
    """Context 0 gives a zero row; a single key gives exactly that key's
    widened V row (rounded only by the f16 weight 1.0 and the output)."""
    rng = np.random.default_rng(10)
    NB, Hq, Hkv, D = 8, 12, 2, 128
    ctx = np.array([0, 1, 3], np.int32)
    tables = random_tables(rng, np.maximum(ctx, 1), NB)
    ks = np.array([0.01, 0.01], np.float32)
    vs = np.array([0.02, 0.03], np.float32)
    v = oracle.e4m3_values()
    finite = np.array([c for c in range(256) if not np.isnan(v[c])], np.uint8)
    kp = rng.choice(finite, size=(NB, 16, Hkv, D)).astype(np.uint8)
    vp = rng.choice(finite, size=(NB, Hkv, D, 16)).astype(np.uint8)
    q = normal_bits(rng, (3, Hq, D))
    out = ops.decode_fp8(to_dev_bf16(q), dev_u8(kp), dev_u8(vp), torch.from_numpy(ks).cuda(),
                         torch.from_numpy(vs).cuda(), to_dev_i32(tables), to_dev_i32(ctx),
                         1 / np.sqrt(128), out_dtype=torch.float32)
    got = out.cpu().numpy().astype(np.float64)
    ref = oracle.decode_fp8(q, kp, vp, ks, vs, tables, ctx, 1 / np.sqrt(128))
    assert np.all(got[0] == 0.0)
    assert_close(got, ref)


@pytest.mark.parametrize("name", ["tiny_decode", "qwen_decode_b8", "cb_decode_b64"])
@pytest.mark.parametrize("num_splits", [0, 5])
def test_fp8_store_decode_equals_store_then_decode(ops, name, num_splits):
    """pa_store_decode_fp8 (quantised store fused into the decode) leaves
    the same codes as pa_store_kv_fp8 and gives the same output bits as
    pa_store_kv_fp8 followed by pa_decode_fp8, and matches the oracle."""
    w = synth.CONFIGS[name]()
    ks = np.array([0.011, 0.0095], np.float32)[:w.num_kv_heads]
    vs = np.array([0.0105, 0.012], np.float32)[:w.num_kv_heads]
    kp, vp = fp8_pools_from(w, ks, vs)
    kref, vref = kp.copy(), vp.copy()
    oracle.store_kv_fp8(w.new_k, w.new_v, kref, vref, ks, vs, w.slot_mapping)
    ksd, vsd = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    q, nk, nv = to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)
    bt, cl, sm = to_dev_i32(w.block_tables), to_dev_i32(w.context_lens), to_dev_i32(w.slot_mapping)
    kf, vf = dev_u8(kp), dev_u8(vp)
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, num_splits, 128, "cuda")
    out_f = ops.store_decode_fp8(q, nk, nv, kf, vf, ksd, vsd, sm, bt, cl, w.scale,
                                 out_dtype=torch.float32, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) == 0
    assert np.array_equal(kf.cpu().numpy(), kref) and np.array_equal(vf.cpu().numpy(), vref)
    ku, vu = dev_u8(kp), dev_u8(vp)
    ops.store_kv_fp8(nk, nv, ku, vu, ksd, vsd, sm)
    out_u = ops.decode_fp8(q, ku, vu, ksd, vsd, bt, cl, w.scale, out_dtype=torch.float32,
                           num_splits=num_splits)
    torch.cuda.synchronize()
    assert torch.equal(out_f, out_u)
    kc, vc, t2 = compact(kref, vref, w.block_tables)
    ref = oracle.decode_fp8(w.q, kc, vc, ks, vs, t2, w.context_lens, w.scale)
    assert_close(out_f.cpu().numpy().astype(np.float64), ref)
