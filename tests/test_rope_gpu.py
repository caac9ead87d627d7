"""GPU parity of pa_rope_store_kv (fused rotary embedding + slot_mapping
store) against the oracle.

v rows and every pool row the call must not touch are compared bit for bit.
Rotated values (q_out and the stored k rows) are compared element by element
with the exact fp64 rotation.  The kernel computes each x c -+ y s in fp32 (a
rounded product and one fused multiply-add, error <= 2^-23 (|x c| + |y s|))
and rounds once to bf16 (at most half an ulp: 2^-8 of the result), so the
bound written here is
    |gpu - exact| <= 2^-8 |exact| + 2^-21 (|x c| + |y s|),
and at least 99% of the values must equal the oracle's own single rounding
of the exact value (a kernel that truncated instead of rounding fails that).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from paged_kv_continuous_gb300.synth import bf16_to_f64
from tests.helpers import bf16_dev_to_bits, normal_bits, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


def rot_bound(x_bits, positions, cos_t, sin_t, exact):
    """Per-element tolerance of the fp32 rotation + one bf16 rounding."""
    x = bf16_to_f64(x_bits)
    D = x.shape[-1]
    c = np.abs(cos_t[positions].astype(np.float64))[:, None, :]
    s = np.abs(sin_t[positions].astype(np.float64))[:, None, :]
    mag = np.abs(x[..., :D // 2]) * c + np.abs(x[..., D // 2:]) * s
    mag = np.concatenate([mag, np.abs(x[..., D // 2:]) * c + np.abs(x[..., :D // 2]) * s], -1)
    return 2.0 ** -8 * np.abs(exact) + 2.0 ** -21 * mag


def check_rotated(got_bits, exact, bound):
    if got_bits.size == 0:      # e.g. every token of the case is padding
        return
    got = bf16_to_f64(got_bits)
    assert np.all(np.isfinite(got))
    err = np.abs(got - exact)
    assert np.all(err <= bound), f"max excess {float(np.max(err - bound))}"
    same = np.mean(got_bits == oracle.round_to_bf16_bits(exact))
    assert same >= 0.99, f"only {same:.4f} of the values equal the single rounding"


def run_case(ops, rng, T, Hq, Hkv, NB, max_pos=4096, pad_every=0, tables=None, in_place=False,
             tok_pad=0, bad_pos=()):
    D = 128
    W = (Hq + 2 * Hkv) * D + tok_pad
    qkv_bits = normal_bits(rng, (T, W))
    qv = qkv_bits[:, :Hq * D].reshape(T, Hq, D)
    kv = qkv_bits[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D)
    vv = qkv_bits[:, (Hq + Hkv) * D:(Hq + 2 * Hkv) * D].reshape(T, Hkv, D)
    cos_t, sin_t = tables if tables is not None else synth.rope_tables(max_pos)
    pos = rng.integers(0, cos_t.shape[0], T).astype(np.int32)
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int32)
    if pad_every:
        slots[::pad_every] = -1
    for t in bad_pos:
        pos[t] = cos_t.shape[0] + 3 if t % 2 else -1
    kc0 = np.full((NB, 16, Hkv, D), 0x1357, np.uint16)
    vc0 = np.full((NB, 16, Hkv, D), 0x2468, np.uint16)

    good = np.ones(T, bool)
    good[list(bad_pos)] = False
    kref, vref = kc0.copy(), vc0.copy()
    q_rot, k_rot = oracle.rope_store_kv(
        np.ascontiguousarray(qv[good]), np.ascontiguousarray(kv[good]),
        np.ascontiguousarray(vv[good]), pos[good], cos_t, sin_t, kref, vref, slots[good])

    qkv = to_dev_bf16(qkv_bits)
    q_d = qkv[:, :Hq * D].view(T, Hq, D) if tok_pad == 0 else \
        torch.as_strided(qkv, (T, Hq, D), (W, D, 1))
    k_d = torch.as_strided(qkv, (T, Hkv, D), (W, D, 1), Hq * D)
    v_d = torch.as_strided(qkv, (T, Hkv, D), (W, D, 1), (Hq + Hkv) * D)
    kc, vc = to_dev_bf16(kc0), to_dev_bf16(vc0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sentinel = torch.full((T, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    q_out = q_d if in_place else sentinel
    res = ops.rope_store_kv(q_d, k_d, v_d, to_dev_i32(pos), torch.from_numpy(cos_t).cuda(),
                            torch.from_numpy(sin_t).cuda(), kc, vc, to_dev_i32(slots),
                            q_out=q_out, error_flags=err)
    torch.cuda.synchronize()
    q_bits = bf16_dev_to_bits(res)
    kc_b, vc_b = bf16_dev_to_bits(kc), bf16_dev_to_bits(vc)

    check_rotated(q_bits[good], q_rot, rot_bound(qv[good], pos[good], cos_t, sin_t, q_rot))
    if not in_place:
        assert np.all(q_bits[~good] == np.uint16(0x40E0))   # skipped tokens: untouched (7.0)
    # pools: v bit-exact and untouched rows bit-exact; k rows rotated
    assert np.array_equal(vc_b, vref)
    fk, fr = kc_b.reshape(NB * 16, Hkv, D), kref.reshape(NB * 16, Hkv, D)
    stored = good & (slots >= 0)
    others = np.ones(NB * 16, bool)
    others[slots[stored]] = False
    assert np.array_equal(fk[others], fr[others])
    gk = kv[stored]
    kr = k_rot[(slots >= 0)[good]]
    check_rotated(fk[slots[stored]], kr, rot_bound(gk, pos[stored], cos_t, sin_t, kr))
    return int(err.item())


@pytest.mark.parametrize("T,Hq,Hkv", [(1, 12, 2), (64, 12, 2), (37, 32, 8), (300, 8, 1),
                                      (5, 1, 1)])
def test_rope_store_matches_oracle(ops, T, Hq, Hkv):
    rng = np.random.default_rng(100 + T + Hq)
    assert run_case(ops, rng, T, Hq, Hkv, NB=max(8, T // 8 + 4), pad_every=5) == 0


def test_rope_store_prefill_size_and_arbitrary_tables(ops):
    """4104 tokens (the varlen prefill workload) with tables that are not
    unit rotations: the kernel applies the tables as given."""
    rng = np.random.default_rng(7)
    tab = (rng.uniform(-1.5, 1.5, (1024, 64)).astype(np.float32),
           rng.uniform(-1.5, 1.5, (1024, 64)).astype(np.float32))
    assert run_case(ops, rng, 4104, 12, 2, NB=300, tables=tab) == 0


def test_rope_in_place_and_unaligned_strides(ops):
    """q rotated in place, and a token stride that is not a multiple of 8
    elements (the scalar path)."""
    rng = np.random.default_rng(8)
    assert run_case(ops, rng, 50, 12, 2, NB=16, in_place=True) == 0
    assert run_case(ops, rng, 50, 12, 2, NB=16, tok_pad=3) == 0


def test_rope_bad_position_reported_and_skipped(ops):
    rng = np.random.default_rng(9)
    err = run_case(ops, rng, 40, 12, 2, NB=16, max_pos=256, bad_pos=(3, 10))
    assert err & ops.DEVERR_POSITION


def test_rope_workload_positions_then_decode(ops):
    """The decode step of cb_decode_b64 with RoPE: the new tokens' q is
    rotated at their positions and k is rotated into the pool; decode over
    the result matches the oracle run on the oracle's rotated inputs."""
    w = synth.cb_decode_b64(keep_seq=False)
    cos_t, sin_t = synth.rope_tables(int(w.context_lens.max()) + 1)
    pos = w.positions
    kref, vref = w.k_cache.copy(), w.v_cache.copy()
    q_rot, _ = oracle.rope_store_kv(w.q, w.new_k, w.new_v, pos, cos_t, sin_t, kref, vref,
                                    w.slot_mapping)
    q_rot_bits = oracle.round_to_bf16_bits(q_rot)
    kc, vc = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    q_out = ops.rope_store_kv(to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v),
                              to_dev_i32(pos), torch.from_numpy(cos_t).cuda(),
                              torch.from_numpy(sin_t).cuda(), kc, vc, to_dev_i32(w.slot_mapping))
    torch.cuda.synchronize()
    # rotated q and pool agree with the oracle's single rounding almost everywhere
    assert np.mean(bf16_dev_to_bits(q_out) == q_rot_bits) >= 0.99
    assert np.array_equal(bf16_dev_to_bits(vc), vref)
    # decode on the GPU's rotated inputs vs the oracle decode on its own
    out = ops.decode(q_out, kc, vc, to_dev_i32(w.block_tables), to_dev_i32(w.context_lens),
                     w.scale, out_dtype=torch.float32)
    ref = oracle.decode(q_rot_bits, kref, vref, w.block_tables, w.context_lens, w.scale)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref))
