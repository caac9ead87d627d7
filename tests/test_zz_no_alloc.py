"""pa_decode_noalloc, the decode entry point for callers that cannot
allocate device memory (its split partials live in a fixed array inside the
library), called through the C ABI: two calls in a row each match pa_decode
with a caller-provided workspace, and the oracle, within the attention
tolerance.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.  It also passes alone in a fresh
process (the first call on the device does the one-time address lookup)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_continuous_gb300 import synth
from tests.helpers import (assert_attention_close, dev_to_f64, oracle_stored_caches, to_dev_bf16,
                           to_dev_i32)

pytestmark = pytest.mark.gpu


def _call_noalloc(ops, q, kc, vc, tables, ctx, scale, out, splits, err, flags=0):
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = kc.shape
    P = ctypes.c_void_p
    return ops.lib.pa_decode_noalloc(
        P(out.data_ptr()), ops.PA_DTYPE_F32 if out.dtype == torch.float32 else ops.PA_DTYPE_BF16,
        P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()), NB, P(tables.data_ptr()),
        tables.stride(0), P(ctx.data_ptr()), B, Hq, Hkv, D, bs, float(scale), splits,
        P(err.data_ptr()) if err is not None else None, flags,
        P(torch.cuda.current_stream().cuda_stream))


def _workload(name):
    if name == "wide_h64_8":
        # 64 query heads over 8 kv heads: the default split count (one per SM)
        # needs more partials than the array holds, so the call lowers it
        rng = np.random.default_rng(64)
        ctx = [3000, 17, 900, 4096, 1]
        return synth.make_paged(rng, "wide_h64_8", ctx, [1] * len(ctx), num_blocks=600,
                                num_q_heads=64, num_kv_heads=8, keep_seq=False)
    fn = synth.CONFIGS[name]
    return fn(keep_seq=False) if name != "qwen_decode_b8" else fn()


@pytest.mark.parametrize("name,splits,flags,with_err", [
    ("cb_decode_b64", 0, 0, True),
    ("long_decode_b4", 0, 0, True),
    ("qwen_decode_b8", 37, 0, True),
    ("wide_h64_8", 0, 0, True),
    ("cb_decode_b64", 0, 0, False),          # no error word: the kernel skips its reports
    ("cb_decode_b64", 0, 3, True),           # PA_LAUNCH_PDL | PA_LAUNCH_EARLY_KV
])
def test_noalloc_matches_workspace_decode_twice(name, splits, flags, with_err):
    from paged_kv_continuous_gb300 import ops
    assert flags in (0, ops.PA_LAUNCH_PDL | ops.PA_LAUNCH_EARLY_KV)
    w = _workload(name)
    kc_np, vc_np = oracle_stored_caches(w)
    ref_oracle = oracle.decode(w.q, kc_np, vc_np, w.block_tables, w.context_lens, w.scale)
    q, kc, vc = to_dev_bf16(w.q), to_dev_bf16(kc_np), to_dev_bf16(vc_np)
    tables, ctx = to_dev_i32(w.block_tables), to_dev_i32(w.context_lens)
    ref = ops.decode(q, kc, vc, tables, ctx, w.scale, out_dtype=torch.float32,
                     num_splits=splits)
    ref_np = dev_to_f64(ref)
    assert_attention_close(ref_np, ref_oracle, f"{name} pa_decode", strict=True)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda") if with_err else None
        status = _call_noalloc(ops, q, kc, vc, tables, ctx, w.scale, out, splits, err, flags)
        assert status == ops.PA_OK, ops.lib.pa_status_string(status)
        torch.cuda.synchronize()
        if err is not None:
            assert int(err.item()) == 0
        got = dev_to_f64(out)
        assert_attention_close(got, ref_np, f"{name} call {call} vs pa_decode", strict=True)
        assert_attention_close(got, ref_oracle, f"{name} call {call} vs oracle", strict=True)


def test_noalloc_rejects_split_counts_beyond_its_array():
    from paged_kv_continuous_gb300 import ops
    w = synth.tiny_decode()
    q, kc, vc = to_dev_bf16(w.q), to_dev_bf16(w.k_cache), to_dev_bf16(w.v_cache)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = _call_noalloc(ops, q, kc, vc, to_dev_i32(w.block_tables),
                           to_dev_i32(w.context_lens), w.scale, out, 4000, err)
    assert status == 3   # PA_ERR_WORKSPACE, nothing launched
