"""GB300-native paged-KV attention: slot_mapping store, paged GQA decode with
split-K partials and merge, and varlen prefill over a paged prefix.

The compute lives in a C-ABI shared library built from ``csrc/`` for
sm_103a; ``paged_kv_continuous_gb300.ops`` is the thin binding over it.
Importing the package itself loads nothing, so the input generators in
``synth`` work on machines without a GPU.
"""
__all__ = ["synth", "ops"]
