"""The decode step captured as one CUDA graph (koas-w "errors and
solutions", section "CUDA Graph": static index buffers updated in place,
one capture replayed every step).

Checks: a replay gives the same bits as the same calls made eagerly; after
the index buffers and the layers' new q / k / v are refilled for the next
token of every sequence, a second replay matches the oracle on that step."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from paged_kv_continuous_gb300.synth import BF16_NAN
from tests.helpers import bf16_dev_to_bits, normal_bits, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from paged_kv_continuous_gb300 import graph, ops
    return ops, graph


def make_layers(w, L, rng):
    """L layers over the same sequences (tables, lengths, slots); layer l > 0
    gets fresh values in every live pool slot and fresh new-token rows."""
    host = []
    for l in range(L):
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        if l:
            live = kc != BF16_NAN
            kc[live] = normal_bits(rng, int(live.sum()))
            vc[live] = normal_bits(rng, int(live.sum()))
        q = w.q if l == 0 else normal_bits(rng, w.q.shape)
        nk = w.new_k if l == 0 else normal_bits(rng, w.new_k.shape)
        nv = w.new_v if l == 0 else normal_bits(rng, w.new_v.shape)
        host.append(dict(q=q, k=nk, v=nv, k_cache=kc, v_cache=vc))
    return host


def to_dev(h):
    d = {k: to_dev_bf16(v) for k, v in h.items()}
    d["out"] = torch.empty(d["q"].shape, dtype=torch.bfloat16, device="cuda")
    return d


def oracle_step(h, w_tables, ctx, slots, scale, rope=None):
    """Store (with RoPE if given) then decode, on host copies of a layer."""
    kc, vc = h["k_cache"].copy(), h["v_cache"].copy()
    if rope is None:
        oracle.store_kv(h["k"], h["v"], kc, vc, slots)
        q = h["q"]
    else:
        pos, cos_t, sin_t = rope
        q_rot, _ = oracle.rope_store_kv(h["q"], h["k"], h["v"], pos, cos_t, sin_t, kc, vc, slots)
        q = oracle.round_to_bf16_bits(q_rot)
    return oracle.decode(q, kc, vc, w_tables, ctx, scale), kc, vc


def close(got_bits, ref):
    got = torch.from_numpy(got_bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    return np.all(np.abs(got.astype(np.float64) - ref) <= 2e-3 + 1e-2 * np.abs(ref))


@pytest.mark.parametrize("use_rope,fused", [(False, False), (True, False), (False, True),
                                            (True, True)])
def test_graph_replay_matches_eager_then_oracle_next_step(mods, use_rope, fused):
    """fused: one pa_store_decode per layer (early K/V requests behind the
    previous layer), which must give the bits of the two-call form."""
    ops, graph = mods
    w = synth.qwen_decode_b8()
    rng = np.random.default_rng(77)
    L = 3
    # one spare table column, so that every sequence can take a next token
    tables = np.concatenate([w.block_tables, np.full((w.batch, 1), -1, np.int32)], 1)
    host = make_layers(w, L, rng)
    rope = None
    extra = {}
    if use_rope:
        cos_t, sin_t = synth.rope_tables(int(w.context_lens.max()) + 64)
        rope = (w.positions, cos_t, sin_t)
        extra = dict(positions=to_dev_i32(w.positions), cos_table=torch.from_numpy(cos_t).cuda(),
                     sin_table=torch.from_numpy(sin_t).cuda())
    # eager reference run on separate copies
    eager = [to_dev(h) for h in host]
    splits = ops.default_splits(w.num_q_heads, w.num_kv_heads, torch.cuda.current_device())
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, splits, 128, "cuda")
    bt, cl, sm = to_dev_i32(tables), to_dev_i32(w.context_lens), to_dev_i32(w.slot_mapping)
    for x in eager:
        if use_rope:
            ops.rope_store_kv(x["q"], x["k"], x["v"], extra["positions"], extra["cos_table"],
                              extra["sin_table"], x["k_cache"], x["v_cache"], sm, q_out=x["q"])
        else:
            ops.store_kv(x["k"], x["v"], x["k_cache"], x["v_cache"], sm)
        ops.decode(x["q"], x["k_cache"], x["v_cache"], bt, cl, w.scale, out=x["out"],
                   num_splits=splits, workspace=ws)
    # the graph over fresh copies
    layers = [to_dev(h) for h in host]
    g = graph.DecodeStepGraph(layers, bt, cl, sm, w.scale, num_splits=splits, fused=fused,
                              **extra)
    assert g.launches_per_replay() == (1 if fused else 2) * L
    g.replay()
    torch.cuda.synchronize()
    assert g.read_error_word() == 0
    for x, e in zip(layers, eager):
        assert torch.equal(x["out"].view(torch.int16), e["out"].view(torch.int16))
        assert torch.equal(x["k_cache"].view(torch.int16), e["k_cache"].view(torch.int16))
    # step 1 against the oracle, and keep the oracle's pools for step 2
    ref_pools = []
    for l, (h, x) in enumerate(zip(host, layers)):
        ref, kc, vc = oracle_step(h, tables, w.context_lens, w.slot_mapping, w.scale, rope)
        assert close(bf16_dev_to_bits(x["out"]), ref), f"layer {l} step 1"
        ref_pools.append((kc, vc))

    # step 2: every sequence gains one token; a sequence whose new position
    # opens a block takes an unused physical block
    ctx2 = w.context_lens + 1
    pos2 = w.context_lens.copy()
    tables2 = tables.copy()
    used = set(int(b) for b in tables.ravel() if b >= 0)
    free = [b for b in range(w.num_blocks) if b not in used]
    for b in range(w.batch):
        if pos2[b] % 16 == 0:
            tables2[b, pos2[b] // 16] = free.pop()
    slots2 = (tables2[np.arange(w.batch), pos2 // 16].astype(np.int64) * 16
              + pos2 % 16).astype(np.int32)
    g.update(block_tables=to_dev_i32(tables2), context_lens=to_dev_i32(ctx2),
             slot_mapping=to_dev_i32(slots2),
             **({"positions": to_dev_i32(pos2)} if use_rope else {}))
    host2 = []
    for l, x in enumerate(layers):
        h2 = dict(q=normal_bits(rng, w.q.shape), k=normal_bits(rng, w.new_k.shape),
                  v=normal_bits(rng, w.new_v.shape), k_cache=ref_pools[l][0],
                  v_cache=ref_pools[l][1])
        x["q"].copy_(to_dev_bf16(h2["q"]))
        x["k"].copy_(to_dev_bf16(h2["k"]))
        x["v"].copy_(to_dev_bf16(h2["v"]))
        host2.append(h2)
    g.replay()
    torch.cuda.synchronize()
    assert g.read_error_word() == 0
    rope2 = (pos2, rope[1], rope[2]) if use_rope else None
    for l, (h2, x) in enumerate(zip(host2, layers)):
        ref, _, _ = oracle_step(h2, tables2, ctx2, slots2, w.scale, rope2)
        assert close(bf16_dev_to_bits(x["out"]), ref), f"layer {l} step 2"


def test_graph_update_rejects_shape_change(mods):
    ops, graph = mods
    w = synth.tiny_decode()
    layers = [to_dev(h) for h in make_layers(w, 1, np.random.default_rng(1))]
    g = graph.DecodeStepGraph(layers, to_dev_i32(w.block_tables), to_dev_i32(w.context_lens),
                              to_dev_i32(w.slot_mapping), w.scale)
    with pytest.raises(ops.PagedAttentionError):
        g.update(context_lens=to_dev_i32(np.ones(w.batch + 1, np.int32)))
    with pytest.raises(ops.PagedAttentionError):
        g.update(positions=to_dev_i32(np.zeros(w.batch, np.int32)))
