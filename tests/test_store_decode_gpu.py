"""pa_store_decode: the decode step's store fused into the decode kernel.

The pools after the call must equal the oracle's store bit for bit; the
output must equal, bit for bit, pa_store_kv followed by pa_decode with the
same split count (the patched tile holds exactly the stored row), and match
the oracle within 2e-3 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import bf16_dev_to_bits, oracle_stored_caches, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


def fused_vs_unfused(ops, w, slots=None, num_splits=0, pre_store=False):
    slots = w.slot_mapping if slots is None else slots
    kc0, vc0 = (oracle_stored_caches(w) if pre_store else (w.k_cache, w.v_cache))
    q, nk, nv = to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)
    bt, cl, sm = to_dev_i32(w.block_tables), to_dev_i32(w.context_lens), to_dev_i32(slots)
    # fused
    kf, vf = to_dev_bf16(kc0), to_dev_bf16(vc0)
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, num_splits, 128, "cuda")
    out_f = ops.store_decode(q, nk, nv, kf, vf, sm, bt, cl, w.scale, out_dtype=torch.float32,
                             num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    err = ops.read_error_word(ws)
    # unfused, with the slots the fused call accepted
    ku, vu = to_dev_bf16(kc0), to_dev_bf16(vc0)
    ops.store_kv(nk, nv, ku, vu, sm)
    out_u = ops.decode(q, ku, vu, bt, cl, w.scale, out_dtype=torch.float32,
                       num_splits=num_splits)
    torch.cuda.synchronize()
    return out_f, out_u, kf, vf, err


def check_oracle(w, out, kc_ref, vc_ref):
    ref = oracle.decode(w.q, kc_ref, vc_ref, w.block_tables, w.context_lens, w.scale)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref))


@pytest.mark.parametrize("name", ["tiny_decode", "qwen_decode_b8", "cb_decode_b64"])
@pytest.mark.parametrize("num_splits", [0, 5])
def test_store_decode_equals_store_then_decode(ops, name, num_splits):
    w = synth.CONFIGS[name]()
    out_f, out_u, kf, vf, err = fused_vs_unfused(ops, w, num_splits=num_splits)
    assert err == 0
    kref, vref = w.k_cache.copy(), w.v_cache.copy()
    oracle.store_kv(w.new_k, w.new_v, kref, vref, w.slot_mapping)
    assert np.array_equal(bf16_dev_to_bits(kf), kref)
    assert np.array_equal(bf16_dev_to_bits(vf), vref)
    assert torch.equal(out_f, out_u)
    check_oracle(w, out_f, kref, vref)


def test_store_decode_padding_and_wrong_slot(ops):
    """slot < 0: nothing stored, the pool row (already holding the token)
    is used; a slot that is not the new position's: error bit, nothing
    stored or patched, the pool row is used."""
    w = synth.qwen_decode_b8()
    slots = w.slot_mapping.copy()
    slots[1] = -1
    slots[4] = slots[4] + 1 if slots[4] % 16 != 15 else slots[4] - 1
    kc0, vc0 = oracle_stored_caches(w)    # the pool already holds every new token
    q, nk, nv = to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)
    kf, vf = to_dev_bf16(kc0), to_dev_bf16(vc0)
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, 0, 128, "cuda")
    out = ops.store_decode(q, nk, nv, kf, vf, to_dev_i32(slots), to_dev_i32(w.block_tables),
                           to_dev_i32(w.context_lens), w.scale, out_dtype=torch.float32,
                           workspace=ws)
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) & ops.DEVERR_SLOT_INDEX
    # the pools are unchanged (the valid tokens rewrite what they already held)
    assert np.array_equal(bf16_dev_to_bits(kf), kc0)
    assert np.array_equal(bf16_dev_to_bits(vf), vc0)
    check_oracle(w, out, kc0, vc0)
