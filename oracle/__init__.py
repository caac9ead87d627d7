"""CPU oracle for paged-KV attention (ctypes wrapper around pa_oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this package.  The product library in
``paged_kv_continuous_gb300`` never imports, links or executes anything here,
and this package imports nothing from it.

Each function returns float64 NumPy arrays computed by the plain definitions
in ``pa_oracle.c`` (see the header there for the passages each follows and
the readings taken where the pages are silent).  Inputs are bf16 bit patterns
held in ``np.uint16`` arrays and int32 index arrays, all on the host.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against brute force over contiguous K/V, closed forms and invariants (the
E4M3 codec also against torch's float8_e4m3fn conversions); none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpa_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (C11, fp64, OpenMP, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
           "-fopenmp", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PA_ORACLE_LIB points the wrapper at another build of pa_oracle.c;
            # the mutation tests use it to load deliberately broken copies.
            lib = ctypes.CDLL(os.environ.get("PA_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.pa_oracle_store_kv.argtypes = [P, P, i64, i64, i64, i64, i64, P, P, i64,
                                               i32, i32, i32, P]
            lib.pa_oracle_prefill_varlen.argtypes = [P, P, P, P, i32, P, P, i64, P, i64, P,
                                                     i32, i32, i32, i32, dbl, i32]
            lib.pa_oracle_decode.argtypes = [P, P, P, P, P, i64, P, i64, P, i32, i32, i32,
                                             i32, i32, dbl, i32]
            lib.pa_oracle_decode_range.argtypes = [P, P, P, P, P, i64, P, i64, P, P, i32,
                                                   i32, i32, i32, i32, dbl]
            lib.pa_oracle_merge.argtypes = [P, P, P, i64, i32, i32]
            lib.pa_oracle_merge.restype = None
            lib.pa_oracle_rope.argtypes = [P, P, i64, i64, i32, i32, P, P, P, i64]
            lib.pa_oracle_decode_f64.argtypes = [P, P, P, P, P, i64, P, i64, P, i32, i32, i32,
                                                 i32, i32, dbl]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().pa_oracle_max_threads())


def _check(rc: int, what: str):
    if rc != 0:
        names = {1: "bad argument", 2: "index out of range", 3: "out of memory"}
        raise ValueError(f"oracle {what}: {names.get(rc, rc)}")


def store_kv(k, v, k_cache, v_cache, slot_mapping, block_size=16):
    """Copy each token's K/V rows into the pool slots named by slot_mapping.

    ``k``/``v`` are uint16 arrays of shape [T, Hkv, D] (any strides);
    ``k_cache``/``v_cache`` are uint16 [num_blocks, block_size, Hkv, D] and are
    updated in place.
    """
    lib = _load()
    assert k.dtype == np.uint16 and v.dtype == np.uint16
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T, Hkv, D = k.shape
    isz = k.itemsize
    slots = _c(slot_mapping, np.int32)
    rc = lib.pa_oracle_store_kv(
        _ptr(k), _ptr(v), T, k.strides[0] // isz, k.strides[1] // isz,
        v.strides[0] // isz, v.strides[1] // isz, _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], block_size, Hkv, D, _ptr(slots))
    assert k.strides[2] == isz and v.strides[2] == isz
    _check(rc, "store_kv")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, num_threads=0,
           with_lse=False):
    """Paged GQA decode: one query per sequence over its context_lens keys.

    q: uint16 [B, Hq, D]; caches uint16 [NB, bs, Hkv, D]; block_tables int32
    [B, max_blocks]; context_lens int32 [B].  Returns float64 [B, Hq, D]
    (and the natural-log sum-exp [B, Hq] when ``with_lse``).
    """
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    assert D2 == D
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib.pa_oracle_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(_c(k_cache, np.uint16)),
                              _ptr(_c(v_cache, np.uint16)), NB, _ptr(bt), bt.shape[1],
                              _ptr(ctx), B, Hq, Hkv, D, bs, float(scale), int(num_threads))
    _check(rc, "decode")
    return (out, lse) if with_lse else out


def decode_range(q, k_cache, v_cache, block_tables, key_lo, key_hi, scale):
    """Decode query of each sequence over keys [key_lo[b], key_hi[b]) only.

    Returns (out float64 [B, Hq, D], lse float64 [B, Hq]).
    """
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    bt = _c(block_tables, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib.pa_oracle_decode_range(_ptr(out), _ptr(lse), _ptr(q),
                                    _ptr(_c(k_cache, np.uint16)), _ptr(_c(v_cache, np.uint16)),
                                    NB, _ptr(bt), bt.shape[1], _ptr(_c(key_lo, np.int32)),
                                    _ptr(_c(key_hi, np.int32)), B, Hq, Hkv, D, bs,
                                    float(scale))
    _check(rc, "decode_range")
    return out, lse


def prefill_varlen(q, cu_seqlens, k_cache, v_cache, block_tables, context_lens, scale,
                   num_threads=0, with_lse=False):
    """Varlen causal prefill over each sequence's paged keys.

    q: uint16 [T, Hq, D] (rows of sequence s are cu_seqlens[s]..cu_seqlens[s+1]-1);
    the chunk's own keys are read from the cache (they are stored before
    attention).  Returns float64 [T, Hq, D] (and lse [T, Hq]).
    """
    lib = _load()
    q = _c(q, np.uint16)
    T, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    cu = _c(cu_seqlens, np.int32)
    bt = _c(block_tables, np.int32)
    out = np.zeros((T, Hq, D), np.float64)
    lse = np.zeros((T, Hq), np.float64)
    rc = lib.pa_oracle_prefill_varlen(_ptr(out), _ptr(lse), _ptr(q), _ptr(cu), len(cu) - 1,
                                      _ptr(_c(k_cache, np.uint16)),
                                      _ptr(_c(v_cache, np.uint16)), NB, _ptr(bt),
                                      bt.shape[1], _ptr(_c(context_lens, np.int32)), Hq, Hkv,
                                      D, bs, float(scale), int(num_threads))
    _check(rc, "prefill_varlen")
    return (out, lse) if with_lse else out


def merge(part_o, part_lse):
    """Log-sum-exp merge of split partials.

    part_o float64 [R, S, D], part_lse float64 [R, S] -> float64 [R, D].
    """
    lib = _load()
    po = _c(part_o, np.float64)
    pl = _c(part_lse, np.float64)
    R, S, D = po.shape
    out = np.zeros((R, D), np.float64)
    lib.pa_oracle_merge(_ptr(out), _ptr(po), _ptr(pl), R, S, D)
    return out


def rope(x, positions, cos_table, sin_table):
    """Rotary embedding (table lookup, rotate-half pairs i and i + D/2).

    ``x`` uint16 (bf16 bits) [T, H, D], any token stride, heads contiguous;
    ``positions`` int32 [T]; ``cos_table``/``sin_table`` float32
    [max_position, D/2].  Returns float64 [T, H, D]; see ``pa_oracle_rope``.
    """
    lib = _load()
    assert x.dtype == np.uint16 and x.strides[2] == 2 and x.strides[1] == 2 * x.shape[2]
    T, H, D = x.shape
    cos_t = _c(cos_table, np.float32)
    sin_t = _c(sin_table, np.float32)
    assert cos_t.shape == sin_t.shape and cos_t.shape[1] == D // 2
    pos = _c(positions, np.int32)
    out = np.zeros((T, H, D), np.float64)
    rc = lib.pa_oracle_rope(_ptr(out), _ptr(x), T, x.strides[0] // 2, H, D, _ptr(pos),
                            _ptr(cos_t), _ptr(sin_t), cos_t.shape[0])
    _check(rc, "rope")
    return out


def round_to_bf16_bits(x):
    """float64 -> bf16 bit patterns, one rounding to nearest (ties to even).

    For finite values in the normal range, which is all the oracle produces:
    the significand is rounded to 8 bits in float64 (exact), then the value
    (now exactly representable in bf16, hence in float32) is truncated to its
    top 16 bits.
    """
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)                      # x = m 2^e, 0.5 <= |m| < 1
    y = np.ldexp(np.rint(m * 256.0) / 256.0, e)
    return (y.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rope_store_kv(q, k, v, positions, cos_table, sin_table, k_cache, v_cache, slot_mapping,
                  block_size=16):
    """Fused rotary embedding + slot_mapping store ([EAS] "自写 Triton Kernel",
    fused_rope_and_cache_store_kernel).

    q is rotated (returned as float64 [T, Hq, D]); k is rotated (returned as
    float64 [T, Hkv, D]) and, rounded once to bf16, stored with the unrotated
    v through slot_mapping exactly as ``store_kv`` does (pools updated in
    place).  Returns (q_rot, k_rot).
    """
    q_rot = rope(q, positions, cos_table, sin_table)
    k_rot = rope(k, positions, cos_table, sin_table)
    store_kv(round_to_bf16_bits(k_rot), v, k_cache, v_cache, slot_mapping, block_size)
    return q_rot, k_rot


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV cache with per-kv-head scales
#
# Reading of the pages: koas-w / PocketLLM, "cpp_engine Batching
# Implementation (Phase 3.1)", section "当前 KV cache 结构", keeps k_scale /
# v_scale tensors beside the caches "for FP8/INT8 quantisation" and says no
# more.  Taken here: E4M3 codes (1 sign bit, 4 exponent bits with bias 7, 3
# mantissa bits; exponent 0 subnormal; exponent 15 with mantissa 7 is NaN;
# largest finite 448; no infinities), one float32 scale per kv head for K and
# one for V, stored value = round_to_nearest_even(x / scale) saturated to
# +-448, read value = code value * scale.  K pages keep the bf16 layout
# [num_blocks][block_size][Hkv][D]; V pages are dim-major inside a block,
# [num_blocks][Hkv][D][block_size].
# ---------------------------------------------------------------------------

def e4m3_values():
    """float64 value of each of the 256 E4M3 codes, from the field formula."""
    vals = np.empty(256, np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        if e == 15 and m == 7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = sign * m * 2.0 ** -9           # 0.m * 2^(1 - 7)
        else:
            vals[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def e4m3_encode(y):
    """Nearest E4M3 code of each value (ties to the even code), magnitudes
    beyond 448 saturated to 448, NaN to 0x7F.  Codes 0..126 are the
    non-negative finite values in increasing order; the sign is bit 7."""
    y = np.asarray(y, np.float64)
    pos = e4m3_values()[:127]
    a = np.abs(y)
    hi = np.clip(np.searchsorted(pos, a), 1, 126)          # pos[hi-1] <= a <= pos[hi] (in range)
    lo = hi - 1
    d_lo, d_hi = a - pos[lo], pos[hi] - a
    code = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(a >= 448.0, 126, code)
    code = code.astype(np.uint8) | np.where(np.signbit(y), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(y), np.uint8(0x7F), code).astype(np.uint8)


def quantize_fp8(x_bits, scale):
    """bf16 rows [T, H, D] -> E4M3 codes of x / scale[h]; the division is
    IEEE float32 (the precision the stored code is decided in)."""
    xf = (x_bits.astype(np.uint32) << 16).view(np.float32)
    y = xf / np.asarray(scale, np.float32)[None, :, None]
    return e4m3_encode(y.astype(np.float32))


def store_kv_fp8(k, v, k_pool, v_pool, k_scale, v_scale, slot_mapping, block_size=16):
    """Quantise each token's K/V rows and place them at slot_mapping[t]
    (slot < 0 skipped): K at [block][row][h][:], V at [block][h][:][row]."""
    kq, vq = quantize_fp8(k, k_scale), quantize_fp8(v, v_scale)
    nslots = k_pool.shape[0] * block_size
    for t, slot in enumerate(np.asarray(slot_mapping, np.int64)):
        if slot < 0:
            continue
        if slot >= nslots:
            raise ValueError("oracle store_kv_fp8: index out of range")
        blk, row = divmod(int(slot), block_size)
        k_pool[blk, row] = kq[t]
        v_pool[blk, :, :, row] = vq[t]


def dequantize_pools_fp8(k_pool, v_pool, k_scale, v_scale):
    """float64 pools in the bf16 layout [NB][bs][Hkv][D]: code value * scale."""
    vals = e4m3_values()
    kf = vals[k_pool] * np.asarray(k_scale, np.float32).astype(np.float64)[None, None, :, None]
    vf = vals[v_pool] * np.asarray(v_scale, np.float32).astype(np.float64)[None, :, None, None]
    return kf, np.ascontiguousarray(vf.transpose(0, 3, 1, 2))


def decode_fp8(q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, scale,
               with_lse=False):
    """Paged GQA decode over FP8 pools: every code widened exactly and
    multiplied by its head's scale, then the same attention as ``decode``."""
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    kf, vf = dequantize_pools_fp8(k_pool, v_pool, k_scale, v_scale)
    NB, bs, Hkv, _ = kf.shape
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = lib.pa_oracle_decode_f64(_ptr(out), _ptr(lse), _ptr(q), _ptr(kf), _ptr(vf), NB,
                                  _ptr(bt), bt.shape[1], _ptr(ctx), B, Hq, Hkv, D, bs,
                                  float(scale))
    _check(rc, "decode_fp8")
    return (out, lse) if with_lse else out
