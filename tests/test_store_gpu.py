"""GPU parity of pa_store_kv against the oracle: bit-exact pools."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import bf16_dev_to_bits, normal_bits, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


def run_store(ops, k_bits, v_bits, kc_bits, vc_bits, slots, k_dev=None, v_dev=None):
    k = to_dev_bf16(k_bits) if k_dev is None else k_dev
    v = to_dev_bf16(v_bits) if v_dev is None else v_dev
    kc, vc = to_dev_bf16(kc_bits), to_dev_bf16(vc_bits)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.store_kv(k, v, kc, vc, to_dev_i32(slots), error_flags=err)
    torch.cuda.synchronize()
    return bf16_dev_to_bits(kc), bf16_dev_to_bits(vc), int(err.item())


@pytest.mark.parametrize("name", ["tiny_decode", "cb_decode_b64", "varlen_prefill"])
def test_store_configs_bit_exact(ops, name):
    w = synth.CONFIGS[name]()
    kc_ref, vc_ref = w.k_cache.copy(), w.v_cache.copy()
    oracle.store_kv(w.new_k, w.new_v, kc_ref, vc_ref, w.slot_mapping)
    kc, vc, err = run_store(ops, w.new_k, w.new_v, w.k_cache, w.v_cache, w.slot_mapping)
    assert err == 0
    assert np.array_equal(kc, kc_ref) and np.array_equal(vc, vc_ref)


def test_store_strided_fused_qkv_and_padding(ops):
    rng = np.random.default_rng(5)
    NB, Hq, Hkv, D, T = 40, 12, 2, 128, 300
    qkv_bits = normal_bits(rng, (T, Hq + 2 * Hkv, D))
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int32)
    slots[::7] = -1                                       # padding tokens
    kc0 = np.full((NB, 16, Hkv, D), 0x5555, np.uint16)
    vc0 = np.full((NB, 16, Hkv, D), 0x2222, np.uint16)
    kref, vref = kc0.copy(), vc0.copy()
    oracle.store_kv(qkv_bits[:, Hq:Hq + Hkv], qkv_bits[:, Hq + Hkv:], kref, vref, slots)
    qkv = to_dev_bf16(qkv_bits)
    kc, vc, err = run_store(ops, None, None, kc0, vc0, slots, k_dev=qkv[:, Hq:Hq + Hkv],
                            v_dev=qkv[:, Hq + Hkv:])
    assert err == 0
    assert np.array_equal(kc, kref) and np.array_equal(vc, vref)


def test_store_unaligned_strides_take_scalar_path(ops):
    """Token stride not a multiple of 8 elements: still bit-exact."""
    rng = np.random.default_rng(6)
    NB, Hkv, D, T = 8, 2, 128, 50
    buf = normal_bits(rng, (T, 2 * Hkv * D + 3))
    k_bits = np.lib.stride_tricks.as_strided(buf, (T, Hkv, D), (buf.strides[0], 2 * D, 2))
    v_bits = np.lib.stride_tricks.as_strided(buf[:, 3:], (T, Hkv, D),
                                             (buf.strides[0], 2 * D, 2))
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int32)
    kref = np.zeros((NB, 16, Hkv, D), np.uint16)
    vref = np.zeros_like(kref)
    oracle.store_kv(k_bits, v_bits, kref, vref, slots)
    dev = to_dev_bf16(buf)
    k_dev = dev.as_strided((T, Hkv, D), (dev.stride(0), D, 1))
    v_dev = dev[:, 3:].as_strided((T, Hkv, D), (dev.stride(0), D, 1), dev.storage_offset() + 3)
    kc, vc, err = run_store(ops, None, None, np.zeros_like(kref), np.zeros_like(vref), slots,
                            k_dev=k_dev, v_dev=v_dev)
    assert err == 0
    assert np.array_equal(kc, kref) and np.array_equal(vc, vref)


def test_store_out_of_range_slot_sets_error_and_skips(ops):
    rng = np.random.default_rng(7)
    NB, Hkv, D = 4, 2, 128
    k = normal_bits(rng, (3, Hkv, D))
    slots = np.array([5, NB * 16, 9], np.int32)          # middle one is past the pool
    kc0 = np.zeros((NB, 16, Hkv, D), np.uint16)
    kc, vc, err = run_store(ops, k, k, kc0, kc0, slots)
    assert err & ops.DEVERR_SLOT_INDEX
    flat = kc.reshape(-1, Hkv, D)
    assert np.array_equal(flat[5], k[0]) and np.array_equal(flat[9], k[2])
    mask = np.ones(NB * 16, bool)
    mask[[5, 9]] = False
    assert np.all(flat[mask] == 0)
