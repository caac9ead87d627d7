"""Planted mistakes in copies of the oracle source must each fail the pins.

Each mutant is a one-line change a real implementation could plausibly
contain.  The copy is compiled on the CPU into a temporary directory and the
pin suite is run against it in a subprocess; the test passes only when the
pins reject the mutant.  The real oracle is never modified."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

MUTANTS = {
    "gqa_interleaved_head_map": ("g * group + hi;", "hi * num_kv_heads + g;"),
    "causal_boundary_exclusive": ("prefix + i + 1,", "prefix + i,"),
    "scale_dropped": ("double s = scale * dot;", "double s = dot;"),
    "max_not_subtracted": ("double p = exp(scores[j - lo] - m);",
                           "double p = exp(scores[j - lo]);"),
    "normaliser_dropped": ("o[d] = acc / l;", "o[d] = acc;"),
    "gather_row_off_by_one": ("int64_t row = j % block_size;",
                              "int64_t row = (j + 1) % block_size;"),
    "gather_logical_block": ("int64_t block = table_row[j / block_size];",
                             "int64_t block = j / block_size;"),
    "store_row_from_block": ("int64_t row = slot % block_size;",
                             "int64_t row = (slot / block_size) % block_size;"),
    "merge_unweighted": ("acc += exp(lse[s] - M) * part_o", "acc += part_o"),
    "lse_natural_log_dropped": ("return m + log(l);", "return m + log2(l);"),
    "rope_first_half_sign": ("o[i] = x1 * c - x2 * s;", "o[i] = x1 * c + x2 * s;"),
    "rope_second_half_sign": ("o[i + half] = x2 * c + x1 * s;",
                              "o[i + half] = x2 * c - x1 * s;"),
    "rope_token_index_as_position": ("int64_t p = positions[t];", "int64_t p = t;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    mutant = tmp_path / "pa_oracle_mutant.c"
    mutant.write_text(text.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-fopenmp", "-shared", str(mutant),
                    "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, PA_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins accepted mutant {name}:\n{r.stdout[-2000:]}"


# The FP8 functions of the oracle are NumPy code: a mutant is the function
# rebuilt from its own source with one change, put in place of the original
# for the duration of the test (monkeypatch restores it); the FP8 pins then
# run in this process and at least one must fail.
PY_MUTANTS = {
    "e4m3_subnormal_scale": ("e4m3_values", "sign * m * 2.0 ** -9", "sign * m * 2.0 ** -10"),
    "e4m3_exponent_bias": ("e4m3_values", "2.0 ** (e - 7)", "2.0 ** (e - 8)"),
    "e4m3_ties_away_from_zero": ("e4m3_encode", "np.where(lo % 2 == 0, lo, hi)", "hi"),
    "fp8_scale_multiplied": ("quantize_fp8", "y = xf / np.asarray(scale",
                             "y = xf * np.asarray(scale"),
    "fp8_v_widened_with_k_scale": ("dequantize_pools_fp8",
                                   "vf = vals[v_pool] * np.asarray(v_scale",
                                   "vf = vals[v_pool] * np.asarray(k_scale"),
    "fp8_k_scale_of_other_head": ("dequantize_pools_fp8",
                                  "np.asarray(k_scale, np.float32).astype(np.float64)[None",
                                  "np.asarray(k_scale, np.float32).astype(np.float64)[::-1][None"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_fp8_pins_reject_mutant(name, monkeypatch):
    import inspect
    import textwrap
    sys.path.insert(0, ROOT)
    import oracle
    from tests import test_oracle_pins as pins
    fname, old, new = PY_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fname)))
    assert src.count(old) == 1, f"mutation site for {name} not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, fname, ns[fname])
    failed = []
    for test in (pins.test_e4m3_values_closed_forms_and_library,
                 pins.test_e4m3_encode_round_trip_ties_and_saturation,
                 pins.test_store_kv_fp8_layout_and_quantisation,
                 pins.test_decode_fp8_equals_bf16_decode_on_exact_values):
        try:
            test()
        except AssertionError:
            failed.append(test.__name__)
    assert failed, f"the FP8 pins accepted mutant {name}"
