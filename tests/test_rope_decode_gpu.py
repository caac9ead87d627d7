"""pa_rope_store_decode: rotary embedding, the store of the new tokens and
the decode of one step in one kernel.

The output must equal, bit for bit, pa_rope_store_kv (q rotated into q_out,
K rotated and stored with V) followed by pa_decode on q_out with the same
split count; the pools after the call must equal those pa_rope_store_kv
leaves; and the output must match the oracle (its RoPE and store, then its
decode on its own rounding of the rotated q) within 2e-3 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import bf16_dev_to_bits, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


def fused_and_two_calls(ops, w, positions, cos_t, sin_t, num_splits):
    q, nk, nv = to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)
    bt, cl, sm = to_dev_i32(w.block_tables), to_dev_i32(w.context_lens), to_dev_i32(w.slot_mapping)
    pd = to_dev_i32(positions)
    ct, st = torch.from_numpy(cos_t).cuda(), torch.from_numpy(sin_t).cuda()
    kf, vf = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, num_splits, 128, "cuda")
    q_before = q.clone()
    out_f = ops.rope_store_decode(q, nk, nv, kf, vf, sm, bt, cl, w.scale, pd, ct, st,
                                  out_dtype=torch.float32, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    err = ops.read_error_word(ws)
    assert torch.equal(q, q_before), "q must not be written"
    ku, vu = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    q_out = torch.zeros_like(q)
    ops.rope_store_kv(q, nk, nv, pd, ct, st, ku, vu, sm, q_out=q_out)
    out_u = ops.decode(q_out, ku, vu, bt, cl, w.scale, out_dtype=torch.float32,
                       num_splits=num_splits)
    torch.cuda.synchronize()
    return out_f, out_u, (kf, vf), (ku, vu), err


@pytest.mark.parametrize("name", ["tiny_decode", "qwen_decode_b8", "cb_decode_b64"])
@pytest.mark.parametrize("num_splits", [0, 5])
def test_rope_store_decode_equals_two_calls_and_oracle(ops, name, num_splits):
    w = synth.CONFIGS[name]()
    pos = w.positions
    cos_t, sin_t = synth.rope_tables(int(w.context_lens.max()) + 1)
    out_f, out_u, (kf, vf), (ku, vu), err = fused_and_two_calls(ops, w, pos, cos_t, sin_t,
                                                                num_splits)
    assert err == 0
    assert torch.equal(out_f, out_u)
    assert torch.equal(kf.view(torch.int16), ku.view(torch.int16))
    assert torch.equal(vf.view(torch.int16), vu.view(torch.int16))
    # the oracle: its rotation and store, then its decode on its rounded q
    kref, vref = w.k_cache.copy(), w.v_cache.copy()
    q_rot, _ = oracle.rope_store_kv(w.q, w.new_k, w.new_v, pos, cos_t, sin_t, kref, vref,
                                    w.slot_mapping)
    assert np.array_equal(bf16_dev_to_bits(vf), vref)
    ref = oracle.decode(oracle.round_to_bf16_bits(q_rot), kref, vref, w.block_tables,
                        w.context_lens, w.scale)
    got = out_f.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref))


def test_rope_store_decode_bad_position(ops):
    """A position outside the tables: PA_DEVERR_POSITION, that sequence's new
    row is neither stored nor patched, every other sequence is unaffected."""
    w = synth.qwen_decode_b8()
    pos = w.positions.copy()
    cos_t, sin_t = synth.rope_tables(int(w.context_lens.max()) + 1)
    bad = 1
    pos[bad] = cos_t.shape[0] + 5
    out_f, out_u, (kf, vf), (ku, vu), err = fused_and_two_calls(ops, w, pos, cos_t, sin_t, 0)
    assert err & ops.DEVERR_POSITION
    keep = np.arange(w.batch) != bad
    assert torch.equal(out_f[keep], out_u[keep])
    # the bad token's slot still holds the pool's old row, in both forms
    kb = bf16_dev_to_bits(kf).reshape(-1, w.num_kv_heads, 128)
    slot = int(w.slot_mapping[bad])
    assert np.array_equal(kb[slot], w.k_cache.reshape(-1, w.num_kv_heads, 128)[slot])
    assert torch.equal(kf.view(torch.int16), ku.view(torch.int16))
    assert torch.equal(vf.view(torch.int16), vu.view(torch.int16))
