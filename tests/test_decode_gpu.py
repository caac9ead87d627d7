"""GPU parity of pa_decode (+ pa_decode_merge) against the oracle.

Tolerance: bf16 inputs, fp32 accumulation -- every element within
2e-3 + 1e-2 |ref|; fp32-output runs also meet max-abs 2e-3 / max-rel 1e-2."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import (assert_attention_close, bf16_dev_to_bits, const_bits, dev_to_f64,
                           normal_bits, oracle_stored_caches, random_tables, scatter_pool,
                           to_dev_bf16, to_dev_i32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


class Dev:
    """A workload's arrays on the device (pools with the step's tokens stored
    by the GPU store, so decode runs exactly as in a decode step)."""

    def __init__(self, ops, w, store_on_gpu=True):
        self.w = w
        self.q = to_dev_bf16(w.q)
        self.tables = to_dev_i32(w.block_tables)
        self.ctx = to_dev_i32(w.context_lens)
        if store_on_gpu:
            self.kc, self.vc = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
            ops.store_kv(to_dev_bf16(w.new_k), to_dev_bf16(w.new_v), self.kc, self.vc,
                         to_dev_i32(w.slot_mapping))
        else:
            kc, vc = w.stored_caches()
            self.kc, self.vc = to_dev_bf16(kc), to_dev_bf16(vc)

    def decode(self, ops, out_dtype=torch.bfloat16, num_splits=0):
        ws = ops.decode_workspace(self.w.num_q_heads, self.w.num_kv_heads, num_splits)
        out = ops.decode(self.q, self.kc, self.vc, self.tables, self.ctx, self.w.scale,
                         out_dtype=out_dtype, num_splits=num_splits, workspace=ws)
        torch.cuda.synchronize()
        assert ops.read_error_word(ws) == 0
        return out


def oracle_decode(w):
    kc, vc = oracle_stored_caches(w)
    return oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)


@pytest.mark.parametrize("name", ["tiny_decode", "qwen_decode_b8", "cb_decode_b64",
                                  "long_decode_b4"])
def test_decode_configs(ops, name):
    w = synth.CONFIGS[name]()
    ref = oracle_decode(w)
    d = Dev(ops, w)
    assert_attention_close(dev_to_f64(d.decode(ops)), ref, f"{name} bf16")
    assert_attention_close(dev_to_f64(d.decode(ops, torch.float32)), ref, f"{name} f32",
                           strict=True)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 500, 4096])
def test_decode_split_counts(ops, splits):
    """Any split count (one CTA for everything, many cut sequences, more
    splits than blocks) gives the same attention."""
    w = synth.cb_decode_b64()
    ref = oracle_decode(w)
    d = Dev(ops, w)
    assert_attention_close(dev_to_f64(d.decode(ops, torch.float32, splits)), ref,
                           f"splits={splits}", strict=True)


@pytest.mark.parametrize("hq,hkv", [(12, 2), (32, 8), (8, 1), (7, 1), (16, 4), (8, 8),
                                    (64, 8), (3, 1), (20, 4)])
@pytest.mark.parametrize("ctx", [[1, 15, 16, 17], [31, 32, 33, 100], [1000, 3, 0, 257]])
def test_decode_head_shapes_and_ragged_tails(ops, hq, hkv, ctx):
    rng = np.random.default_rng(hq * 100 + hkv + sum(ctx))
    w = synth.make_paged(rng, "shape", ctx, [1 if c > 0 else 0 for c in ctx], num_blocks=256,
                         num_q_heads=hq, num_kv_heads=hkv)
    # q rows exist for every sequence, also one with no key
    if w.q.shape[0] != len(ctx):
        w.q = normal_bits(rng, (len(ctx), hq, 128))
    ref = oracle.decode(w.q, *oracle_stored_caches(w), w.block_tables, w.context_lens, w.scale)
    d = Dev(ops, w, store_on_gpu=False)
    for splits in (0, 3):
        got = dev_to_f64(d.decode(ops, torch.float32, splits))
        assert_attention_close(got, ref, f"hq={hq} hkv={hkv} ctx={ctx} S={splits}",
                               strict=True)
        for b, c in enumerate(ctx):
            if c == 0:
                assert np.all(got[b] == 0)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 4)])
def test_decode_split_merge_path(ops, hq, hkv):
    """Few long sequences over many splits (4 or 8 kv heads, S >= 8 * batch):
    the decode kernel only writes the partials and a second kernel merges
    them.  The same inputs through that path (default S = one per SM, and
    S = 24), through the in-kernel merge (S = 23 < 8 * 3), and through
    pa_store_decode on the merge-kernel path (the new rows stored and
    attended in the decode kernel, the merge after it): every output against
    the oracle, the pools bit for bit."""
    rng = np.random.default_rng(4242 + hq)
    ctx = [3000, 17, 1500]
    w = synth.make_paged(rng, "split_merge", ctx, [1, 1, 1], num_blocks=512, num_q_heads=hq,
                         num_kv_heads=hkv)
    kref, vref = oracle_stored_caches(w)
    ref = oracle.decode(w.q, kref, vref, w.block_tables, w.context_lens, w.scale)
    d = Dev(ops, w, store_on_gpu=False)
    for splits in (0, 24, 23):
        assert_attention_close(dev_to_f64(d.decode(ops, torch.float32, splits)), ref,
                               f"hq={hq} hkv={hkv} S={splits}", strict=True)
    kc, vc = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    ws = ops.decode_workspace(hq, hkv, 0)
    out = ops.store_decode(to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v), kc, vc,
                           to_dev_i32(w.slot_mapping), d.tables, d.ctx, w.scale,
                           out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) == 0
    assert np.array_equal(bf16_dev_to_bits(kc), kref)
    assert np.array_equal(bf16_dev_to_bits(vc), vref)
    assert_attention_close(dev_to_f64(out), ref, f"store_decode hq={hq} hkv={hkv}", strict=True)


@pytest.mark.parametrize("scale", [-4.0, -0.09, 0.0, 2.5])
@pytest.mark.parametrize("hq,hkv,splits", [(12, 2, 0), (12, 2, 7), (32, 8, 0)])
def test_decode_scale_sign_and_size(ops, scale, hq, hkv, splits):
    """Softmax scales of either sign, zero (every key weighs the same) and
    large magnitudes (near one-hot weights, scaled scores spread over
    hundreds of base-2 units, so the reference max moves many times):
    against the oracle through the in-kernel merge, a small split count
    and the merge-kernel path."""
    rng = np.random.default_rng(900 + int(abs(scale) * 100) + hq + splits)
    ctx = [2100, 1, 16, 333, 47]
    w = synth.make_paged(rng, "scale", ctx, [1] * len(ctx), num_blocks=256, num_q_heads=hq,
                         num_kv_heads=hkv, scale=scale)
    kref, vref = oracle_stored_caches(w)
    ref = oracle.decode(w.q, kref, vref, w.block_tables, w.context_lens, w.scale)
    d = Dev(ops, w, store_on_gpu=False)
    assert_attention_close(dev_to_f64(d.decode(ops, torch.float32, splits)), ref,
                           f"scale={scale} hq={hq} hkv={hkv} S={splits}", strict=True)


def test_decode_deterministic_and_placement_invariant(ops):
    """Fixed split count: bit-identical across runs and across two physical
    placements of the same logical K/V."""
    rng = np.random.default_rng(31)
    lens = [700, 5, 1290, 33, 64]
    ks = [normal_bits(rng, (n, 2, 128)) for n in lens]
    vs = [normal_bits(rng, (n, 2, 128)) for n in lens]
    q = to_dev_bf16(normal_bits(rng, (5, 12, 128)))
    ctx = to_dev_i32(lens)
    outs = []
    for _ in range(2):
        t = random_tables(rng, lens, 300)
        kc = to_dev_bf16(scatter_pool(ks, t, 300))
        vc = to_dev_bf16(scatter_pool(vs, t, 300))
        for _ in range(2):
            o = ops.decode(q, kc, vc, to_dev_i32(t), ctx, 128 ** -0.5, num_splits=11,
                           out_dtype=torch.float32)
            outs.append(o.cpu().numpy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_decode_nan_poisoned_pool_stays_finite(ops):
    """Every pool slot outside the sequences' keys holds NaN (synth poisons
    them), block-table padding holds -1: outputs are finite and correct."""
    w = synth.qwen_decode_b8()
    d = Dev(ops, w)
    got = dev_to_f64(d.decode(ops, torch.float32, 37))
    assert np.all(np.isfinite(got))
    assert_attention_close(got, oracle_decode(w), "poisoned", strict=True)


def test_decode_sees_key_stored_same_step_over_several_steps(ops):
    """Store at position L, decode with context L+1, repeat: each step matches
    the oracle (the context_lens / seq_len timing bugs on the pages)."""
    rng = np.random.default_rng(41)
    lens0 = np.array([3, 16, 40, 129])
    steps = 5
    full = lens0 + steps
    ks = [normal_bits(rng, (n, 2, 128)) for n in full]
    vs = [normal_bits(rng, (n, 2, 128)) for n in full]
    t = random_tables(rng, full, 64)
    # pool holds only the first lens0 positions; the rest arrives step by step
    kpool = scatter_pool([k[:n] for k, n in zip(ks, lens0)], t, 64)
    vpool = scatter_pool([v[:n] for v, n in zip(vs, lens0)], t, 64)
    kc, vc = to_dev_bf16(kpool), to_dev_bf16(vpool)
    kref, vref = kpool.copy(), vpool.copy()
    tables = to_dev_i32(t)
    for s in range(steps):
        pos = lens0 + s
        slots = (t[np.arange(4), pos // 16] * 16 + pos % 16).astype(np.int32)
        nk = np.stack([k[p] for k, p in zip(ks, pos)])
        nv = np.stack([v[p] for v, p in zip(vs, pos)])
        ops.store_kv(to_dev_bf16(nk), to_dev_bf16(nv), kc, vc, to_dev_i32(slots))
        oracle.store_kv(nk, nv, kref, vref, slots)
        q = normal_bits(rng, (4, 12, 128))
        ctx = (pos + 1).astype(np.int32)
        got = ops.decode(to_dev_bf16(q), kc, vc, tables, to_dev_i32(ctx), 128 ** -0.5,
                         out_dtype=torch.float32, num_splits=5)
        ref = oracle.decode(q, kref, vref, t, ctx, 128 ** -0.5)
        assert_attention_close(dev_to_f64(got), ref, f"step {s}", strict=True)


def _pdl_chain(ops, kc, vc, tables, steps_in, ws, outs, num_splits):
    for (nk, nv, slots, q, ctx), out in zip(steps_in, outs):
        ops.store_kv(nk, nv, kc, vc, slots, pdl=True)
        ops.decode(q, kc, vc, tables, ctx, 128 ** -0.5, out=out, num_splits=num_splits,
                   workspace=ws, pdl=True)


def test_decode_pdl_chain_matches_oracle(ops):
    """store -> decode -> store -> decode ... all launched with PA_LAUNCH_PDL,
    back to back with no host synchronisation (each kernel may start while the
    one before finishes), eagerly and replayed from a CUDA graph: every step's
    rows match the oracle, and the graph replay gives the eager bits."""
    rng = np.random.default_rng(43)
    lens0 = np.array([100, 17, 300, 1, 230, 64])
    steps = 6
    full = lens0 + steps
    ks = [normal_bits(rng, (n, 2, 128)) for n in full]
    vs = [normal_bits(rng, (n, 2, 128)) for n in full]
    t = random_tables(rng, full, 160)
    kpool = scatter_pool([k[:n] for k, n in zip(ks, lens0)], t, 160)
    vpool = scatter_pool([v[:n] for v, n in zip(vs, lens0)], t, 160)
    kref, vref = kpool.copy(), vpool.copy()
    tables = to_dev_i32(t)
    B = len(lens0)
    steps_in, refs = [], []
    for s in range(steps):
        pos = lens0 + s
        slots = (t[np.arange(B), pos // 16] * 16 + pos % 16).astype(np.int32)
        nk = np.stack([k[p] for k, p in zip(ks, pos)])
        nv = np.stack([v[p] for v, p in zip(vs, pos)])
        q = normal_bits(rng, (B, 12, 128))
        ctx = (pos + 1).astype(np.int32)
        oracle.store_kv(nk, nv, kref, vref, slots)
        refs.append(oracle.decode(q, kref, vref, t, ctx, 128 ** -0.5))
        steps_in.append((to_dev_bf16(nk), to_dev_bf16(nv), to_dev_i32(slots), to_dev_bf16(q),
                         to_dev_i32(ctx)))
    splits = 7  # long sequences are cut: the chain exercises the in-kernel merges
    ws = ops.decode_workspace(12, 2, splits)
    # eager chain
    kc, vc = to_dev_bf16(kpool), to_dev_bf16(vpool)
    outs = [torch.empty((B, 12, 128), dtype=torch.float32, device="cuda") for _ in range(steps)]
    _pdl_chain(ops, kc, vc, tables, steps_in, ws, outs, splits)
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) == 0
    for s in range(steps):
        assert_attention_close(dev_to_f64(outs[s]), refs[s], f"pdl step {s}", strict=True)
    # the same chain captured in a graph and replayed on fresh pools
    kc2, vc2 = to_dev_bf16(kpool), to_dev_bf16(vpool)
    outs2 = [torch.empty_like(o) for o in outs]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _pdl_chain(ops, kc2, vc2, tables, steps_in, ws, outs2, splits)
    g.replay()
    torch.cuda.synchronize()
    for s in range(steps):
        assert torch.equal(outs2[s], outs[s]), f"graph replay step {s}"


def test_decode_closed_forms_on_gpu(ops):
    """Single key -> v exactly (up to output rounding); equal V rows -> that row;
    head-marked V -> kv head index."""
    rng = np.random.default_rng(51)
    hq, hkv = 12, 2
    lens = [1, 77, 300]
    ks = [normal_bits(rng, (n, hkv, 128)) for n in lens]
    vs = [normal_bits(rng, (1, hkv, 128)),
          np.broadcast_to(normal_bits(rng, (1, hkv, 128)), (77, hkv, 128)).copy(),
          np.stack([const_bits(g + 1, (300, 128)) for g in range(hkv)], axis=1)]
    t = random_tables(rng, lens, 40)
    q = to_dev_bf16(normal_bits(rng, (3, hq, 128)))
    out = ops.decode(q, to_dev_bf16(scatter_pool(ks, t, 40)), to_dev_bf16(scatter_pool(vs, t, 40)),
                     to_dev_i32(t), to_dev_i32(lens), 128 ** -0.5, out_dtype=torch.float32,
                     num_splits=4)
    o = out.cpu().numpy().astype(np.float64)
    from paged_kv_continuous_gb300.synth import bf16_to_f64
    for h in range(hq):
        np.testing.assert_array_equal(o[0, h], bf16_to_f64(vs[0][0, h // 6]))
        np.testing.assert_allclose(o[1, h], bf16_to_f64(vs[1][0, h // 6]), rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(o[2, h], h // 6 + 1, rtol=1e-6)


def test_decode_bad_block_index_sets_error_without_fault(ops):
    """A block-table entry outside the pool is reported in the error word and
    skipped; the call completes."""
    w = synth.tiny_decode()
    d = Dev(ops, w)
    bad = w.block_tables.copy()
    bad[1, 1] = w.num_blocks + 5
    bad[0, 0] = -3
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, 4)
    ops.decode(d.q, d.kc, d.vc, to_dev_i32(bad), d.ctx, w.scale, num_splits=4, workspace=ws)
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) & ops.DEVERR_BLOCK_INDEX


def _partition(lens, S, bs=16):
    """The documented split partition, restated: split c starts at
    floor(N W(c) / W(S)), every split weighing 4 except, with S >= 32 and
    N >= 4 S, the last four (3, 3, 3, 2)."""
    n = [(c + bs - 1) // bs if c > 0 else 0 for c in lens]
    P = np.concatenate([[0], np.cumsum(n)]).astype(np.int64)
    N = int(P[-1])
    tail = S >= 32 and N >= 4 * S
    w = [4] * S
    if tail:
        w[-4:] = [3, 3, 3, 2]
    W = np.concatenate([[0], np.cumsum(w)]).astype(np.int64)

    def begin(c):
        return int(N * W[c] // W[S])

    def split_of(x):
        # the largest c with begin(c) <= x, by search over the (few) splits
        return int(np.searchsorted([begin(c) for c in range(S + 1)], x, side="right") - 1)
    return n, P, N, begin, split_of


@pytest.mark.parametrize("S", [29, 64])
def test_merge_entry_point_against_oracle_partials(ops, S):
    """Fill the workspace with oracle partials laid out as the header
    documents, run pa_decode_merge alone, compare with the oracle (S = 64:
    the lighter shares of the last four splits)."""
    w = synth.qwen_decode_b8()
    kc, vc = oracle_stored_caches(w)
    n, P, N, begin, split_of = _partition(w.context_lens, S)
    Hq, D = w.num_q_heads, w.head_dim
    part_o = np.zeros((2, S, Hq, D), np.float32)         # [slot][split][head][dim]
    part_l = np.full((2, S, Hq), np.nan, np.float32)   # unused slots are poison
    cut = []
    for b in range(w.batch):
        c0, c1 = split_of(P[b]), split_of(P[b] + n[b] - 1)
        cut.append(c1 > c0)
        if c1 == c0:
            continue
        for c in range(c0, c1 + 1):
            lo_blk, hi_blk = max(begin(c), P[b]), min(begin(c + 1), P[b] + n[b])
            if hi_blk <= lo_blk:
                continue
            klo = (lo_blk - P[b]) * 16
            khi = min((hi_blk - P[b]) * 16, int(w.context_lens[b]))
            lo_arr = np.zeros(w.batch, np.int32)
            hi_arr = np.zeros(w.batch, np.int32)
            lo_arr[b], hi_arr[b] = klo, khi
            o, l = oracle.decode_range(w.q, kc, vc, w.block_tables, lo_arr, hi_arr, w.scale)
            slot = 1 if c == c0 else 0
            part_o[slot, c] = o[b]
            part_l[slot, c] = l[b]
    ws = ops.decode_workspace(Hq, w.num_kv_heads, S)
    hdr = 256 + 4 * 4096                      # error word + fixed counter area
    po_bytes = ((S * 2 * Hq * D * 4 + 255) // 256) * 256
    ws[hdr:hdr + part_o.nbytes].copy_(torch.from_numpy(part_o.view(np.uint8).reshape(-1)))
    ws[hdr + po_bytes:hdr + po_bytes + part_l.nbytes].copy_(
        torch.from_numpy(part_l.view(np.uint8).reshape(-1)))
    out = torch.full((w.batch, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ops.decode_merge(out, ws, to_dev_i32(w.context_lens), S)
    torch.cuda.synchronize()
    ref = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    got = out.cpu().numpy().astype(np.float64)
    cut = np.array(cut)
    assert cut.sum() >= 4
    assert_attention_close(got[cut], ref[cut], "merge", strict=True)
    assert np.all(np.isnan(got[~cut]))          # rows of uncut sequences untouched


def test_decode_reuses_one_workspace_across_calls(ops):
    """The in-kernel merge leaves its arrival counters at zero: one workspace
    serves many consecutive calls (different split counts, different
    batches) and every call matches the oracle."""
    ws = ops.decode_workspace(12, 2, 500)
    torch.cuda.synchronize()
    for name, splits in [("cb_decode_b64", 500), ("qwen_decode_b8", 97), ("cb_decode_b64", 31),
                         ("tiny_decode", 3), ("cb_decode_b64", 500)]:
        w = synth.CONFIGS[name]()
        d = Dev(ops, w, store_on_gpu=False)
        out = ops.decode(d.q, d.kc, d.vc, d.tables, d.ctx, w.scale, out_dtype=torch.float32,
                         num_splits=splits, workspace=ws)
        torch.cuda.synchronize()
        assert ops.read_error_word(ws) == 0
        assert_attention_close(dev_to_f64(out), oracle_decode(w), f"{name} S={splits}",
                               strict=True)
    counters = ws.view(torch.int32)[64:64 + 4096]      # bytes [256, 256 + 4 * 4096)
    assert int(counters.abs().sum().item()) == 0
