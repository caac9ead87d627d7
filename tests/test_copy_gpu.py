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
    """A serving loop's step as a programmatic-launch chain: the inputs copied
    from pinned host memory by pa_copy before the wait, the prepared
    pa_store_decode, the output copied back by pa_copy; three steps in a row
    on two staging buffers, each output against the oracle."""
    w = synth.qwen_decode_b8()
    kc0, vc0 = w.k_cache, w.v_cache
    kref, vref = oracle_stored_caches(w)
    ref = oracle.decode(w.q, kref, vref, w.block_tables, w.context_lens, w.scale)
    host_q = torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).view(
        torch.bfloat16).pin_memory()
    kc, vc = to_dev_bf16(kc0), to_dev_bf16(vc0)
    nk, nv = to_dev_bf16(w.new_k), to_dev_bf16(w.new_v)
    tables, ctx, slots = (to_dev_i32(w.block_tables), to_dev_i32(w.context_lens),
                          to_dev_i32(w.slot_mapping))
    qbuf = [torch.empty_like(host_q, device="cuda") for _ in range(2)]
    outs = [torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
            for _ in range(2)]
    ws = ops.decode_workspace(w.num_q_heads, w.num_kv_heads, 0, 128, "cuda")
    calls = [ops.StoreDecodeCall(qbuf[i], nk, nv, kc, vc, slots, tables, ctx, w.scale, outs[i],
                                 workspace=ws, pdl=True) for i in range(2)]
    host_out = [torch.full((w.batch, w.num_q_heads, 128), float("nan")).pin_memory()
                for _ in range(3)]
    for step in range(3):
        i = step % 2
        ops.copy(qbuf[i], host_q, pdl=True, before_wait=step > 0)
        calls[i]()
        ops.copy(host_out[step], outs[i], pdl=True)
    torch.cuda.synchronize()
    assert ops.read_error_word(ws) == 0
    for step in range(3):
        assert_attention_close(host_out[step].numpy().astype(np.float64), ref,
                               f"step {step}", strict=True)


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
