"""PA_LAUNCH_EARLY_KV: a chain of fused decode steps over several layers,
each call launched with programmatic dependent launch and requesting its
first K/V pages before the previous layer's kernel completes.

Every layer has its own pools, so the kernel before each call never writes
the pools that call reads (the flag's contract).  The chain must give, bit
for bit, the outputs and pools of the same chain without the flag and of
plain stream-ordered calls, also when captured in a CUDA graph and replayed;
every layer's output must match the oracle within 2e-3 + 1e-2 |ref|."""
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


def layer_inputs(w, n_layers):
    """Per-layer (q, new_k, new_v, k_pool, v_pool) as bf16 bit arrays: the
    workload's own, then sign-flipped and K/V-swapped variants (finite rows
    stay finite, the unused NaN rows stay NaN)."""
    flip = np.uint16(0x8000)
    base = (w.q, w.new_k, w.new_v, w.k_cache, w.v_cache)
    out = [base]
    if n_layers > 1:
        out.append(tuple(x ^ flip for x in base))
    if n_layers > 2:
        out.append((w.q[:, ::-1].copy(), w.new_v, w.new_k, w.v_cache, w.k_cache))
    return out[:n_layers]


def run_chain(ops, w, inputs, mode, num_splits, rounds=2):
    """mode: 'plain' (no PDL), 'pdl', 'early' (PDL + early K/V) or 'graph'
    (the 'early' chain captured once and replayed `rounds` times)."""
    bt, cl, sm = to_dev_i32(w.block_tables), to_dev_i32(w.context_lens), to_dev_i32(w.slot_mapping)
    dev = [tuple(to_dev_bf16(a) for a in x) for x in inputs]
    outs = [torch.empty((w.q.shape[0], w.num_q_heads, 128), dtype=torch.float32, device="cuda")
            for _ in inputs]
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, num_splits, 128, "cuda")
    pdl = mode != "plain"
    early = mode in ("early", "graph")

    def chain():
        for (q, nk, nv, kc, vc), o in zip(dev, outs):
            ops.store_decode(q, nk, nv, kc, vc, sm, bt, cl, w.scale, out=o,
                             num_splits=num_splits, workspace=ws, pdl=pdl, early_kv=early)

    if mode == "graph":
        chain()  # eager first: kernel attributes are set outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            chain()
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(rounds):
            g.replay()
    else:
        for _ in range(rounds):
            chain()
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) == 0
    return ([o.cpu() for o in outs],
            [(bf16_dev_to_bits(d[3]), bf16_dev_to_bits(d[4])) for d in dev])


@pytest.mark.parametrize("name", ["tiny_decode", "cb_decode_b64"])
@pytest.mark.parametrize("num_splits", [0, 7])
def test_early_kv_chain_equals_plain_chain(ops, name, num_splits):
    w = synth.CONFIGS[name]()
    inputs = layer_inputs(w, 3)
    ref_out, ref_pools = run_chain(ops, w, inputs, "plain", num_splits)
    for mode in ("pdl", "early", "graph"):
        out, pools = run_chain(ops, w, inputs, mode, num_splits)
        for l in range(len(inputs)):
            assert torch.equal(out[l], ref_out[l]), f"{mode}: layer {l} output differs"
            assert np.array_equal(pools[l][0], ref_pools[l][0]), f"{mode}: layer {l} K pool"
            assert np.array_equal(pools[l][1], ref_pools[l][1]), f"{mode}: layer {l} V pool"
    # every layer against the oracle (its store, then its decode)
    for l, (q, nk, nv, kc, vc) in enumerate(inputs):
        kref, vref = kc.copy(), vc.copy()
        oracle.store_kv(nk, nv, kref, vref, w.slot_mapping)
        assert np.array_equal(ref_pools[l][0], kref) and np.array_equal(ref_pools[l][1], vref)
        ref = oracle.decode(q, kref, vref, w.block_tables, w.context_lens, w.scale)
        got = ref_out[l].numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref)), f"layer {l}"


def finite_codes(rng, shape):
    """Random finite E4M3 codes of both signs (0x7F / 0xFF are NaN)."""
    mag = rng.integers(0, 0x7F, shape, dtype=np.uint8)
    return mag | (rng.integers(0, 2, shape, dtype=np.uint8) << 7)


def test_early_kv_fp8_chain_equals_plain_chain(ops):
    """The FP8 fused step with the flag, over two layers with their own
    pools and scales: same output bits and codes as without it."""
    w = synth.cb_decode_b64()
    rng = np.random.default_rng(31)
    NB = w.k_cache.shape[0]
    layers = []
    for l in range(2):
        kp = torch.from_numpy(finite_codes(rng, (NB, 16, 2, 128))).cuda()
        vp = torch.from_numpy(finite_codes(rng, (NB, 2, 128, 16))).cuda()
        ks = torch.tensor([0.011, 0.0095 + 0.001 * l], dtype=torch.float32, device="cuda")
        vs = torch.tensor([0.0105, 0.012 - 0.001 * l], dtype=torch.float32, device="cuda")
        layers.append((kp, vp, ks, vs))
    q, nk, nv = to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)
    bt, cl, sm = to_dev_i32(w.block_tables), to_dev_i32(w.context_lens), to_dev_i32(w.slot_mapping)
    ws = ops.decode_workspace(12, 2, 0, 128, "cuda")
    results = {}
    for mode in ("plain", "early"):
        pools = [(kp.clone(), vp.clone(), ks, vs) for kp, vp, ks, vs in layers]
        outs = []
        for _ in range(2):
            outs = [ops.store_decode_fp8(q, nk, nv, kp, vp, ks, vs, sm, bt, cl, w.scale,
                                         out_dtype=torch.float32, workspace=ws,
                                         pdl=mode == "early", early_kv=mode == "early")
                    for kp, vp, ks, vs in pools]
        torch.cuda.synchronize()
        assert ops.read_error_word(ws) == 0
        results[mode] = ([o.cpu() for o in outs], [(kp.cpu(), vp.cpu()) for kp, vp, _, _ in pools])
    for l in range(2):
        assert torch.equal(results["plain"][0][l], results["early"][0][l])
        assert torch.equal(results["plain"][1][l][0], results["early"][1][l][0])
        assert torch.equal(results["plain"][1][l][1], results["early"][1][l][1])


def test_early_kv_requires_pdl(ops):
    w = synth.tiny_decode()
    with pytest.raises(ops.PagedAttentionError):
        ops.store_decode(to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v),
                         to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache), to_dev_i32(w.slot_mapping),
                         to_dev_i32(w.block_tables), to_dev_i32(w.context_lens), w.scale,
                         early_kv=True)
