"""Thin Python binding over libpa_gb300.so (the C ABI in include/pa.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, checks shapes and dtypes, and passes raw device pointers,
element strides and the current CUDA stream to the C entry point of the same
name.  All arithmetic runs in the library's sm_103a kernels; there is no
fallback path.  Importing this module loads the library and raises if it has
not been built (``python -m paged_kv_continuous_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpa_gb300.so")

PA_OK = 0
PA_DTYPE_BF16 = 0
PA_DTYPE_F32 = 1
PA_LAUNCH_PDL = 1  # programmatic dependent launch (see include/pa.h)
PA_LAUNCH_EARLY_KV = 2  # decode: K/V pages requested before the previous kernel completes
PA_COPY_BEFORE_WAIT = 4  # pa_copy: the bytes move before the previous kernel completes
DEVERR_BLOCK_INDEX = 1
DEVERR_SLOT_INDEX = 2
DEVERR_WAIT_TIMEOUT = 4
DEVERR_SHAPE = 8
DEVERR_POSITION = 16

EXPORTED = (
    "pa_abi_version", "pa_status_string", "pa_store_kv", "pa_decode_workspace_size",
    "pa_decode_default_splits", "pa_decode", "pa_decode_merge", "pa_prefill_varlen",
    "pa_decode_noalloc", "pa_rope_store_kv", "pa_store_kv_fp8", "pa_decode_fp8",
    "pa_store_decode", "pa_store_decode_fp8", "pa_prefill_store_varlen",
    "pa_rope_store_decode", "pa_get_device_error", "pa_copy",
)


class PagedAttentionError(RuntimeError):
    pass


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise PagedAttentionError(
            f"{path} is missing: build it with `python -m paged_kv_continuous_gb300.build`")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz, u32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_float, ctypes.c_size_t, ctypes.c_uint32)
    lib.pa_abi_version.restype = i32
    lib.pa_abi_version.argtypes = []
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [i32]
    lib.pa_get_device_error.restype = i32
    lib.pa_get_device_error.argtypes = [P, P, i32, P]
    lib.pa_copy.restype = i32
    lib.pa_copy.argtypes = [P, P, i64, u32, P]
    lib.pa_store_kv.restype = i32
    lib.pa_store_kv.argtypes = [P, P, i64, i64, i64, i64, i64, P, P, i64, i32, i32, i32, P, P,
                                u32, P]
    lib.pa_rope_store_kv.restype = i32
    lib.pa_rope_store_kv.argtypes = [P, i64, P, i64, P, i64, P, i64, i64, i32, i32, i32, P, P,
                                     P, i64, P, P, i64, i32, P, P, u32, P]
    lib.pa_decode_workspace_size.restype = sz
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32]
    lib.pa_decode_default_splits.restype = i32
    lib.pa_decode_default_splits.argtypes = [i32, i32, i32]
    lib.pa_decode.restype = i32
    lib.pa_decode.argtypes = [P, i32, P, P, P, i64, P, i32, P, i32, i32, i32, i32, i32, f32,
                              i32, P, sz, u32, P]
    lib.pa_store_decode.restype = i32
    lib.pa_store_decode.argtypes = [P, i32, P, P, P, i64, i64, P, P, P, i64, P, i32, P, i32,
                                    i32, i32, i32, i32, f32, i32, P, sz, u32, P]
    lib.pa_rope_store_decode.restype = i32
    lib.pa_rope_store_decode.argtypes = [P, i32, P, P, P, i64, i64, P, P, P, i64, P, P, P, i64,
                                         P, i32, P, i32, i32, i32, i32, i32, f32, i32, P, sz,
                                         u32, P]
    lib.pa_store_decode_fp8.restype = i32
    lib.pa_store_decode_fp8.argtypes = [P, i32, P, P, P, i64, i64, P, P, P, P, P, i64, P, i32,
                                        P, i32, i32, i32, i32, i32, f32, i32, P, sz, u32, P]
    lib.pa_decode_fp8.restype = i32
    lib.pa_decode_fp8.argtypes = [P, i32, P, P, P, P, P, i64, P, i32, P, i32, i32, i32, i32,
                                  i32, f32, i32, P, sz, u32, P]
    lib.pa_store_kv_fp8.restype = i32
    lib.pa_store_kv_fp8.argtypes = [P, P, i64, i64, i64, i64, i64, P, P, P, P, i64, i32, i32,
                                    i32, P, P, u32, P]
    lib.pa_decode_merge.restype = i32
    lib.pa_decode_merge.argtypes = [P, i32, P, sz, P, i32, i32, i32, i32, i32, P]
    lib.pa_decode_noalloc.restype = i32
    lib.pa_decode_noalloc.argtypes = [P, i32, P, P, P, i64, P, i32, P, i32, i32, i32, i32, i32,
                                      f32, i32, P, u32, P]
    lib.pa_prefill_varlen.restype = i32
    lib.pa_prefill_varlen.argtypes = [P, i32, P, P, i32, i32, i32, P, P, i64, P, i32, P, i32,
                                      i32, i32, i32, f32, P, P]
    lib.pa_prefill_store_varlen.restype = i32
    lib.pa_prefill_store_varlen.argtypes = [P, i32, P, P, P, i64, i64, P, P, i32, i32, i32, P,
                                            P, i64, P, i32, P, i32, i32, i32, i32, f32, P, P]
    return lib


lib = load_library()


def _check(status: int, what: str):
    if status != PA_OK:
        raise PagedAttentionError(f"{what}: {lib.pa_status_string(status).decode()} ({status})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, dims=None):
    if not t.is_cuda:
        raise PagedAttentionError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise PagedAttentionError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise PagedAttentionError(f"{name} must have {dims} dims, got {tuple(t.shape)}")


def _out_code(dtype):
    if dtype == torch.bfloat16:
        return PA_DTYPE_BF16
    if dtype == torch.float32:
        return PA_DTYPE_F32
    raise PagedAttentionError(f"unsupported output dtype {dtype}")


def store_kv(k, v, k_cache, v_cache, slot_mapping, error_flags=None, stream=None, pdl=False):
    """pa_store_kv: k/v bf16 [T, Hkv, D] (any token/head strides, unit dim
    stride) into the pools at slot_mapping (int32 [T]).  pdl: launch with
    PA_LAUNCH_PDL."""
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    if k.stride(2) != 1 or v.stride(2) != 1:
        raise PagedAttentionError("k/v need a unit stride along head_dim")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise PagedAttentionError("pools must be contiguous")
    T, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise PagedAttentionError("shape mismatch between k/v and the pools")
    if slot_mapping.shape[0] != T:
        raise PagedAttentionError("slot_mapping must have one entry per token")
    _check(lib.pa_store_kv(_ptr(k), _ptr(v), T, k.stride(0), k.stride(1), v.stride(0),
                           v.stride(1), _ptr(k_cache), _ptr(v_cache), NB, bs, Hkv, D,
                           _ptr(slot_mapping), _ptr(error_flags),
                           PA_LAUNCH_PDL if pdl else 0, _stream(stream)),
           "pa_store_kv")


def rope_store_kv(q, k, v, positions, cos_table, sin_table, k_cache, v_cache, slot_mapping,
                  q_out=None, error_flags=None, stream=None, pdl=False):
    """pa_rope_store_kv: rotate q (bf16 [T, Hq, D]) into q_out (new tensor,
    or q itself for in place) and k (bf16 [T, Hkv, D]) by the rotary tables
    (float32 [max_position, D/2]) at positions (int32 [T]); store the rotated
    k and the plain v at slot_mapping.  q/k/v may be views of a fused QKV
    buffer (any token stride; heads contiguous).  Returns q_out."""
    for t, n, d in ((q, "q", 3), (k, "k", 3), (v, "v", 3)):
        _need(t, torch.bfloat16, n, d)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise PagedAttentionError(f"{n} needs contiguous heads ([T, H, D], unit dim stride)")
    _need(positions, torch.int32, "positions", 1)
    _need(cos_table, torch.float32, "cos_table", 2)
    _need(sin_table, torch.float32, "sin_table", 2)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise PagedAttentionError("pools must be contiguous")
    if not (cos_table.is_contiguous() and sin_table.is_contiguous()):
        raise PagedAttentionError("rotary tables must be contiguous")
    T, Hq, D = q.shape
    _, Hkv, _ = k.shape
    NB, bs, Hkv2, D2 = k_cache.shape
    if k.shape != (T, Hkv, D) or v.shape != k.shape or (Hkv2, D2) != (Hkv, D) or \
            v_cache.shape != k_cache.shape:
        raise PagedAttentionError("shape mismatch between q/k/v and the pools")
    if cos_table.shape != sin_table.shape or cos_table.shape[1] != D // 2:
        raise PagedAttentionError("rotary tables must be [max_position, head_dim / 2]")
    if positions.shape[0] != T or slot_mapping.shape[0] != T:
        raise PagedAttentionError("positions and slot_mapping need one entry per token")
    if q_out is None:
        q_out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q.device)
    _need(q_out, torch.bfloat16, "q_out", 3)
    if q_out.shape != q.shape or q_out.stride(2) != 1 or q_out.stride(1) != D:
        raise PagedAttentionError("q_out must be [T, Hq, D] with contiguous heads")
    _check(lib.pa_rope_store_kv(_ptr(q), q.stride(0), _ptr(q_out), q_out.stride(0), _ptr(k),
                                k.stride(0), _ptr(v), v.stride(0), T, Hq, Hkv, D,
                                _ptr(positions), _ptr(cos_table), _ptr(sin_table),
                                cos_table.shape[0], _ptr(k_cache), _ptr(v_cache), NB, bs,
                                _ptr(slot_mapping), _ptr(error_flags),
                                PA_LAUNCH_PDL if pdl else 0, _stream(stream)),
           "pa_rope_store_kv")
    return q_out


def _device_index(device=None) -> int:
    if device is None:
        return torch.cuda.current_device()
    if isinstance(device, torch.device):
        return device.index if device.index is not None else torch.cuda.current_device()
    if isinstance(device, str):
        return _device_index(torch.device(device))
    return int(device)


def default_splits(num_q_heads: int, num_kv_heads: int, device=None) -> int:
    return int(lib.pa_decode_default_splits(_device_index(device), num_q_heads, num_kv_heads))


def decode_workspace(num_q_heads: int, num_kv_heads: int, num_splits: int = 0,
                     head_dim: int = 128, device=None):
    """A zeroed workspace for pa_decode (error word and counters start at zero)."""
    s = num_splits if num_splits > 0 else default_splits(num_q_heads, num_kv_heads, device)
    n = int(lib.pa_decode_workspace_size(s, num_q_heads, head_dim))
    if n == 0:
        raise PagedAttentionError("bad workspace request")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _decode_flags(pdl, early_kv):
    """Launch flags of the decode entry points.  early_kv (with pdl): the
    kernel requests its first K/V pages before the kernel launched just
    before it completes, so that kernel must not write the pools."""
    if early_kv and not pdl:
        raise PagedAttentionError("early_kv needs pdl")
    return (PA_LAUNCH_PDL if pdl else 0) | (PA_LAUNCH_EARLY_KV if early_kv else 0)


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
           out_dtype=torch.bfloat16, num_splits=0, workspace=None, stream=None, pdl=False,
           early_kv=False):
    """pa_decode: q bf16 [B, Hq, D] over the paged pools; returns out [B, Hq, D].
    pdl: launch with PA_LAUNCH_PDL (context_lens and block_tables must then
    not be written by the kernel launched just before).  early_kv (with pdl):
    PA_LAUNCH_EARLY_KV, the first K/V pages are requested before that kernel
    completes, so it must not write k_cache / v_cache either."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if not q.is_contiguous():
        raise PagedAttentionError("q must be contiguous")
    if block_tables.stride(1) != 1:
        raise PagedAttentionError("block_tables rows must be contiguous")
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = decode_workspace(Hq, Hkv, num_splits, D, q.device)
    _check(lib.pa_decode(_ptr(out), _out_code(out.dtype), _ptr(q), _ptr(k_cache),
                         _ptr(v_cache), NB, _ptr(block_tables), block_tables.stride(0),
                         _ptr(context_lens), B, Hq, Hkv, D, bs, float(scale), int(num_splits),
                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                         _decode_flags(pdl, early_kv), _stream(stream)), "pa_decode")
    return out


def store_decode(q, new_k, new_v, k_cache, v_cache, slot_mapping, block_tables, context_lens,
                 scale, out=None, out_dtype=torch.bfloat16, num_splits=0, workspace=None,
                 stream=None, pdl=False, early_kv=False):
    """pa_store_decode: one decode step in one kernel -- each sequence's new
    token (new_k / new_v bf16 [B, Hkv, D], heads contiguous) is stored at
    slot_mapping[b] and attended with the rest of the pool.  Returns out."""
    _need(q, torch.bfloat16, "q", 3)
    _need(new_k, torch.bfloat16, "new_k", 3)
    _need(new_v, torch.bfloat16, "new_v", 3)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if not q.is_contiguous():
        raise PagedAttentionError("q must be contiguous")
    for t, n in ((new_k, "new_k"), (new_v, "new_v")):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise PagedAttentionError(f"{n} needs contiguous heads")
    if block_tables.stride(1) != 1:
        raise PagedAttentionError("block_tables rows must be contiguous")
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if tuple(new_k.shape) != (B, Hkv, D) or new_v.shape != new_k.shape or \
            slot_mapping.shape[0] != B:
        raise PagedAttentionError("new_k / new_v / slot_mapping need one row per sequence")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = decode_workspace(Hq, Hkv, num_splits, D, q.device)
    _check(lib.pa_store_decode(_ptr(out), _out_code(out.dtype), _ptr(q), _ptr(new_k),
                               _ptr(new_v), new_k.stride(0), new_v.stride(0), _ptr(slot_mapping),
                               _ptr(k_cache), _ptr(v_cache), NB, _ptr(block_tables),
                               block_tables.stride(0), _ptr(context_lens), B, Hq, Hkv, D, bs,
                               float(scale), int(num_splits), _ptr(workspace),
                               workspace.numel() * workspace.element_size(),
                               _decode_flags(pdl, early_kv), _stream(stream)),
           "pa_store_decode")
    return out


class StoreDecodeCall:
    """A prepared pa_store_decode: the tensors are checked once and the
    marshalled arguments kept, so each call is one foreign call.  The caller
    updates the tensors' contents in place between calls (as with the static
    buffers of a captured step) and keeps them alive; ``call(stream)`` then
    enqueues the step on ``stream`` (default: the current stream)."""

    def __init__(self, q, new_k, new_v, k_cache, v_cache, slot_mapping, block_tables,
                 context_lens, scale, out, num_splits=0, workspace=None, pdl=False,
                 early_kv=False):
        _need(q, torch.bfloat16, "q", 3)
        _need(new_k, torch.bfloat16, "new_k", 3)
        _need(new_v, torch.bfloat16, "new_v", 3)
        _need(k_cache, torch.bfloat16, "k_cache", 4)
        _need(v_cache, torch.bfloat16, "v_cache", 4)
        _need(slot_mapping, torch.int32, "slot_mapping", 1)
        _need(block_tables, torch.int32, "block_tables", 2)
        _need(context_lens, torch.int32, "context_lens", 1)
        if not q.is_contiguous():
            raise PagedAttentionError("q must be contiguous")
        for t, n in ((new_k, "new_k"), (new_v, "new_v")):
            if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
                raise PagedAttentionError(f"{n} needs contiguous heads")
        if block_tables.stride(1) != 1:
            raise PagedAttentionError("block_tables rows must be contiguous")
        B, Hq, D = q.shape
        NB, bs, Hkv, _ = k_cache.shape
        if tuple(new_k.shape) != (B, Hkv, D) or new_v.shape != new_k.shape or \
                slot_mapping.shape[0] != B:
            raise PagedAttentionError("new_k / new_v / slot_mapping need one row per sequence")
        if out.shape != (B, Hq, D) or not out.is_contiguous():
            raise PagedAttentionError("out must be a contiguous [B, Hq, D] tensor")
        if workspace is None:
            workspace = decode_workspace(Hq, Hkv, num_splits, D, q.device)
        self._keep = (q, new_k, new_v, k_cache, v_cache, slot_mapping, block_tables,
                      context_lens, out, workspace)
        c = ctypes
        self._args = (
            c.c_void_p(out.data_ptr()), c.c_int32(_out_code(out.dtype)), c.c_void_p(q.data_ptr()),
            c.c_void_p(new_k.data_ptr()), c.c_void_p(new_v.data_ptr()),
            c.c_int64(new_k.stride(0)), c.c_int64(new_v.stride(0)),
            c.c_void_p(slot_mapping.data_ptr()), c.c_void_p(k_cache.data_ptr()),
            c.c_void_p(v_cache.data_ptr()), c.c_int64(NB), c.c_void_p(block_tables.data_ptr()),
            c.c_int32(block_tables.stride(0)), c.c_void_p(context_lens.data_ptr()), c.c_int32(B),
            c.c_int32(Hq), c.c_int32(Hkv), c.c_int32(D), c.c_int32(bs), c.c_float(scale),
            c.c_int32(num_splits), c.c_void_p(workspace.data_ptr()),
            c.c_size_t(workspace.numel() * workspace.element_size()),
            c.c_uint32(_decode_flags(pdl, early_kv)))
        self.out = out
        self.workspace = workspace

    def __call__(self, stream=None):
        st = lib.pa_store_decode(*self._args, _stream(stream))
        if st != PA_OK:
            _check(st, "pa_store_decode")
        return self.out


class CopyCall:
    """A prepared pa_copy (dst <- src, checked once, as ``copy`` checks)."""

    def __init__(self, dst, src, pdl=False, before_wait=False):
        nbytes, flags = _copy_check(dst, src, pdl, before_wait)
        self._keep = (dst, src)
        self._args = (ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()),
                      ctypes.c_int64(nbytes), ctypes.c_uint32(flags))

    def __call__(self, stream=None):
        st = lib.pa_copy(*self._args, _stream(stream))
        if st != PA_OK:
            _check(st, "pa_copy")


def _copy_check(dst, src, pdl, before_wait):
    for t, n in ((dst, "dst"), (src, "src")):
        if not (t.is_cuda or t.is_pinned()):
            raise PagedAttentionError(f"{n} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous():
            raise PagedAttentionError(f"{n} must be contiguous")
    nbytes = dst.numel() * dst.element_size()
    if nbytes != src.numel() * src.element_size():
        raise PagedAttentionError("dst and src differ in size")
    if before_wait and not pdl:
        raise PagedAttentionError("before_wait needs pdl")
    return nbytes, (PA_LAUNCH_PDL if pdl else 0) | (PA_COPY_BEFORE_WAIT if before_wait else 0)


def copy(dst, src, pdl=False, before_wait=False, stream=None):
    """pa_copy: dst <- src (tensors of the same byte size, contiguous; each on
    the GPU or in pinned host memory).  pdl: launch with PA_LAUNCH_PDL;
    before_wait (with pdl): PA_COPY_BEFORE_WAIT, the bytes move before the
    kernel launched just before completes (it must not write src nor touch
    dst)."""
    nbytes, flags = _copy_check(dst, src, pdl, before_wait)
    _check(lib.pa_copy(_ptr(dst), _ptr(src), nbytes, flags, _stream(stream)), "pa_copy")


def rope_store_decode(q, new_k, new_v, k_cache, v_cache, slot_mapping, block_tables,
                      context_lens, scale, positions, cos_table, sin_table, out=None,
                      out_dtype=torch.bfloat16, num_splits=0, workspace=None, stream=None,
                      pdl=False, early_kv=False):
    """pa_rope_store_decode: store_decode with the rotary embedding of q and
    the new K rows at positions (int32 [B]) from cos_table / sin_table
    (float32 [max_position, D/2]).  q is not written.  Returns out."""
    _need(q, torch.bfloat16, "q", 3)
    _need(new_k, torch.bfloat16, "new_k", 3)
    _need(new_v, torch.bfloat16, "new_v", 3)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    _need(positions, torch.int32, "positions", 1)
    _need(cos_table, torch.float32, "cos_table", 2)
    _need(sin_table, torch.float32, "sin_table", 2)
    if not q.is_contiguous():
        raise PagedAttentionError("q must be contiguous")
    for t, n in ((new_k, "new_k"), (new_v, "new_v")):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise PagedAttentionError(f"{n} needs contiguous heads")
    if block_tables.stride(1) != 1:
        raise PagedAttentionError("block_tables rows must be contiguous")
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if tuple(new_k.shape) != (B, Hkv, D) or new_v.shape != new_k.shape or \
            slot_mapping.shape[0] != B or positions.shape[0] != B:
        raise PagedAttentionError(
            "new_k / new_v / slot_mapping / positions need one row per sequence")
    if cos_table.shape != sin_table.shape or cos_table.shape[1] != D // 2 or \
            not cos_table.is_contiguous() or not sin_table.is_contiguous():
        raise PagedAttentionError("cos_table / sin_table must be contiguous [max_position, D/2]")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = decode_workspace(Hq, Hkv, num_splits, D, q.device)
    _check(lib.pa_rope_store_decode(_ptr(out), _out_code(out.dtype), _ptr(q), _ptr(new_k),
                                    _ptr(new_v), new_k.stride(0), new_v.stride(0),
                                    _ptr(positions), _ptr(cos_table), _ptr(sin_table),
                                    cos_table.shape[0], _ptr(slot_mapping), _ptr(k_cache),
                                    _ptr(v_cache), NB, _ptr(block_tables),
                                    block_tables.stride(0), _ptr(context_lens), B, Hq, Hkv, D, bs,
                                    float(scale), int(num_splits), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _decode_flags(pdl, early_kv), _stream(stream)),
           "pa_rope_store_decode")
    return out


def fp8_pools(num_blocks, num_kv_heads, head_dim=128, block_size=16, device=None):
    """Empty FP8 pools: K uint8 [NB, bs, Hkv, D] (token-major), V uint8
    [NB, Hkv, D, bs] (dim-major inside a block)."""
    k = torch.empty((num_blocks, block_size, num_kv_heads, head_dim), dtype=torch.uint8,
                    device=device)
    v = torch.empty((num_blocks, num_kv_heads, head_dim, block_size), dtype=torch.uint8,
                    device=device)
    return k, v


def _need_fp8_pools(k_cache, v_cache, k_scale, v_scale):
    _need(k_cache, torch.uint8, "k_cache", 4)
    _need(v_cache, torch.uint8, "v_cache", 4)
    _need(k_scale, torch.float32, "k_scale", 1)
    _need(v_scale, torch.float32, "v_scale", 1)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise PagedAttentionError("pools must be contiguous")
    NB, bs, Hkv, D = k_cache.shape
    if tuple(v_cache.shape) != (NB, Hkv, D, bs):
        raise PagedAttentionError("FP8 V pool must be [num_blocks, Hkv, D, block_size]")
    if k_scale.shape[0] != Hkv or v_scale.shape[0] != Hkv:
        raise PagedAttentionError("k_scale / v_scale need one entry per kv head")
    return NB, bs, Hkv, D


def store_kv_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, error_flags=None,
                 stream=None, pdl=False):
    """pa_store_kv_fp8: quantise k/v bf16 [T, Hkv, D] (any token/head
    strides) into the FP8 pools (see fp8_pools) at slot_mapping."""
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    if k.stride(2) != 1 or v.stride(2) != 1:
        raise PagedAttentionError("k/v need a unit stride along head_dim")
    NB, bs, Hkv, D = _need_fp8_pools(k_cache, v_cache, k_scale, v_scale)
    T = k.shape[0]
    if tuple(k.shape) != (T, Hkv, D) or v.shape != k.shape or slot_mapping.shape[0] != T:
        raise PagedAttentionError("shape mismatch between k/v, the pools and slot_mapping")
    _check(lib.pa_store_kv_fp8(_ptr(k), _ptr(v), T, k.stride(0), k.stride(1), v.stride(0),
                               v.stride(1), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                               _ptr(v_scale), NB, bs, Hkv, D, _ptr(slot_mapping),
                               _ptr(error_flags), PA_LAUNCH_PDL if pdl else 0, _stream(stream)),
           "pa_store_kv_fp8")


def decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
               out=None, out_dtype=torch.bfloat16, num_splits=0, workspace=None, stream=None,
               pdl=False, early_kv=False):
    """pa_decode_fp8: q bf16 [B, Hq, D] over the FP8 pools with per-kv-head
    scales; returns out [B, Hq, D]."""
    _need(q, torch.bfloat16, "q", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if not q.is_contiguous():
        raise PagedAttentionError("q must be contiguous")
    if block_tables.stride(1) != 1:
        raise PagedAttentionError("block_tables rows must be contiguous")
    NB, bs, Hkv, _ = _need_fp8_pools(k_cache, v_cache, k_scale, v_scale)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = decode_workspace(Hq, Hkv, num_splits, D, q.device)
    _check(lib.pa_decode_fp8(_ptr(out), _out_code(out.dtype), _ptr(q), _ptr(k_cache),
                             _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), NB,
                             _ptr(block_tables), block_tables.stride(0), _ptr(context_lens), B,
                             Hq, Hkv, D, bs, float(scale), int(num_splits), _ptr(workspace),
                             workspace.numel() * workspace.element_size(),
                             _decode_flags(pdl, early_kv), _stream(stream)), "pa_decode_fp8")
    return out


def store_decode_fp8(q, new_k, new_v, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                     block_tables, context_lens, scale, out=None, out_dtype=torch.bfloat16,
                     num_splits=0, workspace=None, stream=None, pdl=False,
                     early_kv=False):
    """pa_store_decode_fp8: store_decode over FP8 pools (see fp8_pools)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(new_k, torch.bfloat16, "new_k", 3)
    _need(new_v, torch.bfloat16, "new_v", 3)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if not q.is_contiguous():
        raise PagedAttentionError("q must be contiguous")
    for t, n in ((new_k, "new_k"), (new_v, "new_v")):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise PagedAttentionError(f"{n} needs contiguous heads")
    if block_tables.stride(1) != 1:
        raise PagedAttentionError("block_tables rows must be contiguous")
    NB, bs, Hkv, _ = _need_fp8_pools(k_cache, v_cache, k_scale, v_scale)
    B, Hq, D = q.shape
    if tuple(new_k.shape) != (B, Hkv, D) or new_v.shape != new_k.shape or \
            slot_mapping.shape[0] != B:
        raise PagedAttentionError("new_k / new_v / slot_mapping need one row per sequence")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if workspace is None:
        workspace = decode_workspace(Hq, Hkv, num_splits, D, q.device)
    _check(lib.pa_store_decode_fp8(_ptr(out), _out_code(out.dtype), _ptr(q), _ptr(new_k),
                                   _ptr(new_v), new_k.stride(0), new_v.stride(0),
                                   _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(k_scale), _ptr(v_scale), NB, _ptr(block_tables),
                                   block_tables.stride(0), _ptr(context_lens), B, Hq, Hkv, D, bs,
                                   float(scale), int(num_splits), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(),
                                   _decode_flags(pdl, early_kv), _stream(stream)),
           "pa_store_decode_fp8")
    return out


def decode_merge(out, workspace, context_lens, num_splits, block_size=16, stream=None):
    """pa_decode_merge over a workspace filled by pa_decode (or by hand)."""
    B, Hq, D = out.shape
    _check(lib.pa_decode_merge(_ptr(out), _out_code(out.dtype), _ptr(workspace),
                               workspace.numel() * workspace.element_size(),
                               _ptr(context_lens), B, Hq, D, block_size, int(num_splits),
                               _stream(stream)), "pa_decode_merge")
    return out


def prefill_varlen(q, cu_seqlens, k_cache, v_cache, block_tables, context_lens, scale,
                   max_q_len, out=None, out_dtype=torch.bfloat16, error_flags=None,
                   stream=None):
    """pa_prefill_varlen: q bf16 [T, Hq, D] packed by cu_seqlens (int32 [N+1])."""
    _need(q, torch.bfloat16, "q", 3)
    _need(cu_seqlens, torch.int32, "cu_seqlens", 1)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    T, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((T, Hq, D), dtype=out_dtype, device=q.device)
    _check(lib.pa_prefill_varlen(_ptr(out), _out_code(out.dtype), _ptr(q), _ptr(cu_seqlens),
                                 cu_seqlens.shape[0] - 1, T, int(max_q_len), _ptr(k_cache),
                                 _ptr(v_cache), NB, _ptr(block_tables), block_tables.stride(0),
                                 _ptr(context_lens), Hq, Hkv, D, bs, float(scale),
                                 _ptr(error_flags), _stream(stream)), "pa_prefill_varlen")
    return out


def prefill_store_varlen(q, new_k, new_v, slot_mapping, cu_seqlens, k_cache, v_cache,
                         block_tables, context_lens, scale, max_q_len, out=None,
                         out_dtype=torch.bfloat16, error_flags=None, stream=None):
    """pa_prefill_store_varlen: the chunks' K/V rows (new_k / new_v bf16
    [T, Hkv, D], heads contiguous) stored at slot_mapping (int32 [T]) and
    attended, in one kernel; otherwise as prefill_varlen."""
    _need(q, torch.bfloat16, "q", 3)
    _need(new_k, torch.bfloat16, "new_k", 3)
    _need(new_v, torch.bfloat16, "new_v", 3)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    _need(cu_seqlens, torch.int32, "cu_seqlens", 1)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    for t, n in ((new_k, "new_k"), (new_v, "new_v")):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise PagedAttentionError(f"{n} needs contiguous heads")
    T, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if tuple(new_k.shape) != (T, Hkv, D) or new_v.shape != new_k.shape or \
            slot_mapping.shape[0] != T:
        raise PagedAttentionError("new_k / new_v / slot_mapping need one row per token")
    if out is None:
        out = torch.empty((T, Hq, D), dtype=out_dtype, device=q.device)
    _check(lib.pa_prefill_store_varlen(_ptr(out), _out_code(out.dtype), _ptr(q), _ptr(new_k),
                                       _ptr(new_v), new_k.stride(0), new_v.stride(0),
                                       _ptr(slot_mapping), _ptr(cu_seqlens),
                                       cu_seqlens.shape[0] - 1, T, int(max_q_len), _ptr(k_cache),
                                       _ptr(v_cache), NB, _ptr(block_tables),
                                       block_tables.stride(0), _ptr(context_lens), Hq, Hkv, D, bs,
                                       float(scale), _ptr(error_flags), _stream(stream)),
           "pa_prefill_store_varlen")
    return out


def read_error_word(buf, clear=False, stream=None) -> int:
    """The int32 error word at the start of ``buf`` (a decode workspace or an
    error_flags tensor), read through pa_get_device_error: the copy is
    enqueued on ``stream`` and the stream synchronised; ``clear`` resets the
    word to 0 after the copy."""
    if not buf.is_cuda or buf.numel() * buf.element_size() < 4:
        raise PagedAttentionError("error word must be a CUDA tensor of at least 4 bytes")
    flags = ctypes.c_int32(0)
    _check(lib.pa_get_device_error(_ptr(buf), ctypes.byref(flags), 1 if clear else 0,
                                   _stream(stream)), "pa_get_device_error")
    return int(flags.value)
