"""The input generator's convenience store, pinned to the oracle's store.

``synth.PagedWorkload.stored_caches()`` places a workload's new tokens in
copies of its pools.  Some GPU tests use it to build pools that already hold
the step's tokens (their inputs); every expected pool and every pool the
oracle reads comes from ``oracle.store_kv``.  This pins the two together, bit
for bit, on the five workloads and on a workload with padding slots."""
import numpy as np
import pytest

import oracle
from paged_kv_continuous_gb300 import synth


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_synth_store_equals_oracle_store(name):
    fn = synth.CONFIGS[name]
    w = fn(keep_seq=False) if name not in ("tiny_decode", "qwen_decode_b8") else fn()
    kc, vc = w.stored_caches()
    ko, vo = w.k_cache.copy(), w.v_cache.copy()
    oracle.store_kv(w.new_k, w.new_v, ko, vo, w.slot_mapping)
    assert np.array_equal(kc, ko) and np.array_equal(vc, vo)
    # the store changed something: the pools held NaN at every new slot
    flat = w.k_cache.reshape(-1, w.num_kv_heads, w.head_dim)
    assert np.all(flat[w.slot_mapping] == synth.BF16_NAN)


def test_synth_store_skips_padding_like_the_oracle():
    w = synth.qwen_decode_b8()
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[[1, 5]] = -1
    kc, vc = w.stored_caches()
    ko, vo = w.k_cache.copy(), w.v_cache.copy()
    oracle.store_kv(w.new_k, w.new_v, ko, vo, w.slot_mapping)
    assert np.array_equal(kc, ko) and np.array_equal(vc, vo)
