"""pa_copy (a byte copy as a kernel, between device memory and pinned host
memory) and the prepared pa_store_decode call of the binding."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import (assert_attention_close, dev_to_f64, oracle_stored_caches,
                           to_dev_bf16, to_dev_i32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from paged_kv_continuous_gb300 import ops as o
    return o


@pytest.mark.parametrize("nbytes", [16, 4096, 393728, 1000003])
def test_copy_pinned_host_to_device_and_back(ops, nbytes):
    rng = np.random.default_rng(nbytes)
    host = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    ops.copy(dev, host)
    ops.copy(back, dev, pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host) and torch.equal(back, host)


def test_copy_unaligned_bytes(ops):
    """Addresses off the 16-byte grid: at most 256 bytes, one by one."""
    src = torch.arange(300, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(300, dtype=torch.uint8, device="cuda")
    ops.copy(dst[3:203], src[1:201])
    torch.cuda.synchronize()
    assert torch.equal(dst[3:203], src[1:201]) and int(dst[:3].sum()) == 0
    assert int(dst[203:].sum()) == 0
    with pytest.raises(ops.PagedAttentionError):
        ops.copy(dst[1:299], src[2:300])        # 298 unaligned bytes: unsupported


def test_staged_step_chain_matches_oracle(ops):
    """A serving loop's step as a programmatic-launch chain of two kernels:
    pa_copy stages the NEXT step's q, block tables and context lengths from
    pinned host memory into one of three device buffers (bytes moved before
    its wait, next launch released at once), then the prepared
    pa_store_decode decodes this step's buffer and stores its output rows
    straight into pinned host memory.  Steps alternate between q and -q;
    five steps, each output against the oracle."""
    w = synth.qwen_decode_b8()
    kref, vref = oracle_stored_caches(w)
    qs = [w.q, w.q ^ np.uint16(0x8000)]  # bf16 bit patterns: q and -q
    refs = [oracle.decode(q, kref, vref, w.block_tables, w.context_lens, w.scale) for q in qs]
    B, Hq = w.batch, w.num_q_heads
    qb, tb, cb = B * Hq * 128 * 2, w.block_tables.size * 4, B * 4
    o_t, o_c = qb, qb + (tb + 15) // 16 * 16
    pack = o_c + (cb + 15) // 16 * 16
    host = []
    for q in qs:
        h = torch.zeros(pack, dtype=torch.uint8)
        h[:qb] = torch.from_numpy(np.ascontiguousarray(q).view(np.uint8).reshape(-1))
        h[o_t:o_t + tb] = torch.from_numpy(
            np.ascontiguousarray(w.block_tables, np.int32).view(np.uint8).reshape(-1))
        h[o_c:o_c + cb] = torch.from_numpy(
            np.ascontiguousarray(w.context_lens, np.int32).view(np.uint8).reshape(-1))
        host.append(h.pin_memory())
    bufs = [torch.empty(pack, dtype=torch.uint8, device="cuda") for _ in range(3)]
    kc, vc = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    nk, nv = to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)
    slots = to_dev_i32(w.slot_mapping)
    ws = ops.decode_workspace(Hq, w.num_kv_heads, 0, 128, "cuda")
    steps = 5
    host_out = [torch.full((B, Hq, 128), float("nan")).pin_memory() for _ in range(steps)]
    calls = []
    for n in range(steps):
        buf = bufs[n % 3]
        calls.append(ops.StoreDecodeCall(
            buf[:qb].view(torch.bfloat16).view(B, Hq, 128), nk, nv, kc, vc, slots,
            buf[o_t:o_t + tb].view(torch.int32).view(w.block_tables.shape),
            buf[o_c:o_c + cb].view(torch.int32), w.scale, host_out[n], workspace=ws,
            pdl=True))
    ops.copy(bufs[0], host[0])
    for n in range(steps):
        ops.copy(bufs[(n + 1) % 3], host[(n + 1) % 2], pdl=True, before_wait=True)
        calls[n]()
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) == 0
    for n in range(steps):
        assert_attention_close(host_out[n].numpy().astype(np.float64), refs[n % 2],
                               f"step {n}", strict=True)


def test_prepared_call_equals_store_decode(ops):
    w = synth.cb_decode_b64(keep_seq=False)
    args = [to_dev_bf16(w.q), to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)]
    idx = [to_dev_i32(w.block_tables), to_dev_i32(w.context_lens)]
    slots = to_dev_i32(w.slot_mapping)
    ka, va = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    kb, vb = to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    out_a = ops.store_decode(*args, ka, va, slots, *idx, w.scale, out_dtype=torch.float32)
    out_b = torch.empty_like(out_a)
    call = ops.StoreDecodeCall(*args, kb, vb, slots, *idx, w.scale, out_b)
    call()
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    # pools hold NaN in unused slots: compare bit patterns
    assert torch.equal(ka.view(torch.int16), kb.view(torch.int16))
    assert torch.equal(va.view(torch.int16), vb.view(torch.int16))
    assert_attention_close(dev_to_f64(out_b), dev_to_f64(out_a), "prepared", strict=True)
