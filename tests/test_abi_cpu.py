"""The C-ABI library loads without a GPU and exports every entry point that
include/pa.h declares; argument checks that run before any CUDA call
return the documented statuses.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_continuous_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_five_operations():
    names = declared_functions()
    for op in ("pa_store_kv", "pa_rope_store_kv", "pa_decode", "pa_decode_merge",
               "pa_prefill_varlen"):
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in pa.h but not exported"


def test_binding_names_match_header():
    from paged_kv_continuous_gb300 import build
    build.build()
    from paged_kv_continuous_gb300 import ops
    assert sorted(ops.EXPORTED) == declared_functions()


def test_version_and_status_strings(lib):
    lib.pa_abi_version.restype = ctypes.c_int32
    assert lib.pa_abi_version() == 11
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [ctypes.c_int32]
    assert lib.pa_status_string(0) == b"ok"
    assert b"workspace" in lib.pa_status_string(3)
    assert lib.pa_status_string(99) == b"unknown status"


def test_workspace_size_formula(lib):
    f = lib.pa_decode_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int32] * 3

    def up(x):
        return (x + 255) // 256 * 256
    for S, H in [(1, 12), (152, 12), (152, 32), (7, 5)]:
        assert f(S, H, 128) == 256 + 4 * 4096 + up(S * 2 * H * 128 * 4) + up(S * 2 * H * 4)
    assert f(0, 12, 128) == 0 and f(4, 12, 64) == 0 and f(4097, 12, 128) == 0


def test_argument_checks_before_any_launch():
    """Shapes outside the supported set and malformed arguments are rejected
    on the host, before the library touches the device."""
    from paged_kv_continuous_gb300 import build
    build.build()
    from paged_kv_continuous_gb300 import ops
    L = ops.lib
    nul = None
    # unsupported head_dim / block size / group size
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 1, 12, 2, 64, 16, 0.1, 0, nul, 0,
                       0, nul) == 2
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 1, 12, 2, 128, 32, 0.1, 0, nul,
                       0, 0, nul) == 2
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 1, 18, 2, 128, 16, 0.1, 0, nul,
                       0, 0, nul) == 2          # group of 9
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 1, 12, 3, 128, 16, 0.1, 0, nul,
                       0, 0, nul) == 2          # 3 kv heads
    # bad dtype / negative batch / NaN scale / null pointers
    assert L.pa_decode(nul, 7, nul, nul, nul, 1, nul, 1, nul, 1, 12, 2, 128, 16, 0.1, 0, nul, 0,
                       0, nul) == 1
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, -1, 12, 2, 128, 16, 0.1, 0, nul,
                       0, 0, nul) == 1
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 1, 12, 2, 128, 16, float("nan"),
                       0, nul, 0, 0, nul) == 1
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 1, 12, 2, 128, 16, 0.1, 0, nul, 0,
                       0, nul) == 1
    # empty batch is a no-op
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 0, 12, 2, 128, 16, 0.1, 0, nul, 0,
                       0, nul) == 0
    assert L.pa_store_kv(nul, nul, 0, 0, 0, 0, 0, nul, nul, 1, 16, 2, 128, nul, nul, 0, nul) == 0
    assert L.pa_store_kv(nul, nul, 4, 0, 0, 0, 0, nul, nul, 1, 16, 2, 128, nul, nul, 0, nul) == 1
    assert L.pa_store_kv(nul, nul, 4, 0, 0, 0, 0, nul, nul, 1, 16, 2, 96, nul, nul, 0, nul) == 2
    # store launch flags other than PA_LAUNCH_PDL are rejected (PA_LAUNCH_EARLY_KV is decode-only)
    assert L.pa_store_kv(nul, nul, 4, 0, 0, 0, 0, nul, nul, 1, 16, 2, 128, nul, nul, 2, nul) == 1
    assert L.pa_store_kv(nul, nul, 4, 0, 0, 0, 0, nul, nul, 1, 16, 2, 128, nul, nul, 3, nul) == 1
    assert L.pa_decode(nul, 0, nul, nul, nul, 1, nul, 1, nul, 1, 12, 2, 128, 16, 0.1, 0, nul, 0,
                       4, nul) == 1
    assert L.pa_decode_merge(nul, 0, nul, 0, nul, 1, 12, 128, 16, 0, nul) == 1
    assert L.pa_decode_merge(nul, 0, nul, 0, nul, 1, 12, 128, 16, 4, nul) == 1


def test_rope_store_kv_argument_checks(lib):
    """pa_rope_store_kv validates before launching: empty is a no-op, null
    pointers and negative strides are invalid, other shapes unsupported,
    unknown flags rejected, misaligned tables rejected."""
    L = lib
    P, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    L.pa_rope_store_kv.restype = i32
    L.pa_rope_store_kv.argtypes = [P, i64, P, i64, P, i64, P, i64, i64, i32, i32, i32, P, P, P,
                                   i64, P, P, i64, i32, P, P, u32, P]
    nul = None
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: every case fails before a launch

    def call(T=4, Hq=12, Hkv=2, D=128, bs=16, q_tok=1536, flags=0, ptr=fake, tab=fake):
        return L.pa_rope_store_kv(ptr, q_tok, ptr, q_tok, ptr, 256, ptr, 256, T, Hq, Hkv, D,
                                  ptr, tab, tab, 4096, ptr, ptr, 64, bs, ptr, nul, flags, nul)

    assert call(T=0, ptr=nul, tab=nul) == 0
    assert call(ptr=nul) == 1
    assert call(q_tok=-1) == 1
    assert call(D=64) == 2
    assert call(bs=32) == 2
    assert call(Hkv=0) == 2
    assert call(flags=2) == 1
    assert call(tab=ctypes.c_void_p(0x10004)) == 1


def _bind(lib, name, argtypes):
    f = getattr(lib, name)
    f.restype = ctypes.c_int32
    f.argtypes = argtypes
    return f


def test_fused_and_fp8_entry_points_argument_checks(lib):
    """pa_store_decode, pa_store_decode_fp8, pa_decode_fp8, pa_store_kv_fp8
    and pa_prefill_store_varlen validate before any launch: empty batches are
    no-ops, missing pointers are invalid, other shapes unsupported, unknown
    flags rejected."""
    P, i32, i64, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t)
    nul = None
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: every case fails before a launch
    sd = _bind(lib, "pa_store_decode", [P, i32, P, P, P, i64, i64, P, P, P, i64, P, i32, P, i32,
                                        i32, i32, i32, i32, f32, i32, P, sz, u32, P])

    def store_decode(batch=4, new=fake, slots=fake, tok=256, hq=12, hkv=2, d=128, flags=0):
        return sd(fake, 0, fake, new, new, tok, tok, slots, fake, fake, 64, fake, 8, fake, batch,
                  hq, hkv, d, 16, 0.1, 0, nul, 0, flags, nul)
    assert store_decode(batch=0, new=nul, slots=nul) == 0
    assert store_decode(new=nul) == 1
    assert store_decode(slots=nul) == 1
    assert store_decode(d=64) == 2
    assert store_decode(hq=12, hkv=3) == 2
    assert store_decode(flags=2) == 1       # PA_LAUNCH_EARLY_KV needs PA_LAUNCH_PDL
    assert store_decode(flags=2, d=64) == 1
    assert store_decode(flags=3, d=64) == 2  # both flags accepted: the shape decides
    assert store_decode(flags=7) == 1

    df = _bind(lib, "pa_decode_fp8", [P, i32, P, P, P, P, P, i64, P, i32, P, i32, i32, i32, i32,
                                      i32, f32, i32, P, sz, u32, P])

    def decode_fp8(batch=4, scales=fake, d=128, flags=0):
        return df(fake, 0, fake, fake, fake, scales, scales, 64, fake, 8, fake, batch, 12, 2, d,
                  16, 0.1, 0, nul, 0, flags, nul)
    assert decode_fp8(batch=0, scales=nul) == 0
    assert decode_fp8(d=96) == 2
    assert decode_fp8(flags=8) == 1
    assert decode_fp8(flags=3, d=96) == 2

    sf = _bind(lib, "pa_store_kv_fp8", [P, P, i64, i64, i64, i64, i64, P, P, P, P, i64, i32, i32,
                                        i32, P, P, u32, P])

    def store_fp8(T=4, scales=fake, d=128, flags=0):
        return sf(fake, fake, T, 256, 128, 256, 128, fake, fake, scales, scales, 8, 16, 2, d,
                  fake, nul, flags, nul)
    assert store_fp8(T=0, scales=nul) == 0
    assert store_fp8(scales=nul) == 1
    assert store_fp8(d=64) == 2
    assert store_fp8(flags=4) == 1

    pf = _bind(lib, "pa_prefill_store_varlen", [P, i32, P, P, P, i64, i64, P, P, i32, i32, i32, P,
                                                P, i64, P, i32, P, i32, i32, i32, i32, f32, P, P])

    def prefill_store(T=10, new=fake, tok=256, d=128):
        return pf(fake, 0, fake, new, new, tok, tok, fake, fake, 2, T, 8, fake, fake, 64, fake, 8,
                  fake, 12, 2, d, 16, 0.1, nul, nul)
    assert prefill_store(T=0, new=nul) == 0
    assert prefill_store(new=nul) == 1
    assert prefill_store(tok=257) == 1      # token stride not a multiple of 8 elements
    assert prefill_store(d=64) == 2


def test_launch_flag_values_match_header():
    """The binding's launch-flag values are the header's, and early K/V
    requests without PDL are refused before any call."""
    from paged_kv_continuous_gb300 import build
    build.build()
    from paged_kv_continuous_gb300 import ops
    hdr = open(os.path.join(ROOT, "include", "pa.h")).read()
    vals = {m.group(1): int(m.group(2)) for m in
            re.finditer(r"#define (PA_LAUNCH_\w+) (\d+)u", hdr)}
    assert vals == {"PA_LAUNCH_PDL": ops.PA_LAUNCH_PDL,
                    "PA_LAUNCH_EARLY_KV": ops.PA_LAUNCH_EARLY_KV}
    assert ops._decode_flags(False, False) == 0
    assert ops._decode_flags(True, False) == ops.PA_LAUNCH_PDL
    assert ops._decode_flags(True, True) == ops.PA_LAUNCH_PDL | ops.PA_LAUNCH_EARLY_KV
    with pytest.raises(ops.PagedAttentionError):
        ops._decode_flags(False, True)


def test_rope_store_decode_argument_checks(lib):
    """pa_rope_store_decode: empty batch is a no-op; a missing position or
    table pointer, max_position < 1 and unaligned tables are invalid before
    any device query; other shapes unsupported; store-only flags rejected."""
    P, i32, i64, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t)
    nul = None
    fake = ctypes.c_void_p(0x10000)    # never dereferenced: every case fails before a launch
    odd = ctypes.c_void_p(0x10004)     # not 16-byte aligned
    fn = _bind(lib, "pa_rope_store_decode",
               [P, i32, P, P, P, i64, i64, P, P, P, i64, P, P, P, i64, P, i32, P, i32, i32, i32,
                i32, i32, f32, i32, P, sz, u32, P])

    def call(batch=4, pos=fake, cos=fake, sin=fake, maxp=64, d=128, hkv=2, flags=0):
        return fn(fake, 0, fake, fake, fake, 256, 256, pos, cos, sin, maxp, fake, fake, fake, 64,
                  fake, 8, fake, batch, 12, hkv, d, 16, 0.1, 0, nul, 0, flags, nul)
    assert call(batch=0, pos=nul, cos=nul, sin=nul) == 0
    assert call(pos=nul) == 1
    assert call(cos=nul) == 1
    assert call(sin=nul) == 1
    assert call(maxp=0) == 1
    assert call(cos=odd) == 1
    assert call(sin=odd) == 1
    assert call(d=64) == 2
    assert call(hkv=3) == 2
    assert call(flags=2) == 1
    assert call(flags=3, d=64) == 2


def test_decode_step_graph_argument_checks_before_any_device_work():
    """DecodeStepGraph rejects an empty layer list and rotary arguments given
    only in part before it touches a device."""
    from paged_kv_continuous_gb300 import build
    build.build()
    import torch
    from paged_kv_continuous_gb300 import graph, ops
    t = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ops.PagedAttentionError):
        graph.DecodeStepGraph([], t, t, t, 0.1)
    layer = {"q": torch.zeros((1, 12, 128), dtype=torch.bfloat16)}
    with pytest.raises(ops.PagedAttentionError):
        graph.DecodeStepGraph([layer], t, t, t, 0.1, positions=t)
    with pytest.raises(ops.PagedAttentionError):
        graph.DecodeStepGraph([layer], t, t, t, 0.1, positions=t,
                              cos_table=torch.zeros((4, 64)))


def test_device_error_readback_checks_pointers_first():
    """pa_get_device_error rejects null pointers before it enqueues anything
    (so it needs no device here)."""
    from paged_kv_continuous_gb300 import build
    build.build()
    from paged_kv_continuous_gb300 import ops
    L = ops.lib
    word = ctypes.c_int32(0)
    assert L.pa_get_device_error(None, ctypes.byref(word), 0, None) == 1
    assert L.pa_get_device_error(ctypes.c_void_p(16), None, 1, None) == 1


def test_copy_checks_arguments_before_any_launch():
    """pa_copy: bad flags, a negative size or a null pointer are rejected
    before anything is launched; a zero-byte copy launches nothing."""
    from paged_kv_continuous_gb300 import build
    build.build()
    from paged_kv_continuous_gb300 import ops
    L = ops.lib
    p = ctypes.c_void_p(16)
    assert L.pa_copy(p, p, 16, 8, None) == 1              # unknown flag bit
    assert L.pa_copy(p, p, 16, ops.PA_COPY_BEFORE_WAIT, None) == 1  # before-wait needs PDL
    assert L.pa_copy(p, p, -1, 0, None) == 1
    assert L.pa_copy(None, p, 16, 0, None) == 1
    assert L.pa_copy(p, None, 16, 0, None) == 1
    assert L.pa_copy(None, None, 0, 0, None) == 0
