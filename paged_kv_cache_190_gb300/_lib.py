"""ctypes binding of libpagedattn (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(PKG, "libpagedattn.so")

PA_F32, PA_BF16 = 0, 1
PA_OK = 0
PA_ERR_OUT_OF_BLOCKS = -3
PA_ERR_SWAPPED = -8
PA_DEVERR_BAD_BLOCK, PA_DEVERR_BAD_LENGTH, PA_DEVERR_BAD_SLOT, PA_DEVERR_TIMEOUT = 1, 2, 4, 8

# Every function include/pa.h declares (checked by the tests).
EXPORTED_SYMBOLS = [
    "pa_get_error_string", "pa_reshape_and_cache", "pa_copy_blocks", "pa_decode_chunk_tokens",
    "pa_decode_workspace_size", "pa_decode", "pa_decode_noalloc", "pa_debug_set_wait_limit",
    "pa_read_device_errors", "pa_reshape_and_cache_fp8", "pa_decode_fp8", "pa_swap_blocks",
    "pa_decode_multi", "pa_decode_cascade", "pa_decode_cascade_workspace_size",
    "pa_cascade_groups",
    "pa_bm_create", "pa_bm_destroy", "pa_bm_add_seq", "pa_bm_append_slot", "pa_bm_fork",
    "pa_bm_free", "pa_bm_block_table", "pa_bm_refcount", "pa_bm_num_free", "pa_bm_free_list",
    "pa_bm_stats", "pa_bm_append_slots", "pa_bm_build_block_tables", "pa_bm_enable_swap",
    "pa_bm_swap_out", "pa_bm_swap_in", "pa_bm_num_free_host", "pa_bm_host_free_list",
]

_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_pi32 = ctypes.POINTER(ctypes.c_int32)
_pi64 = ctypes.POINTER(ctypes.c_int64)

_SIGNATURES = {
    "pa_get_error_string": (ctypes.c_char_p, [_i32]),
    "pa_reshape_and_cache": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                    _vp, _vp]),
    "pa_copy_blocks": (_i32, [_vp, _vp, _vp, _i32, _sz, _i32, _vp, _vp]),
    "pa_decode_chunk_tokens": (_i32, [_i32, _i32, _i32, _i32]),
    "pa_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_decode": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _i32, _i32, _i32, _i32,
                         _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "pa_decode_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _i32, _i32, _i32,
                                 _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pa_reshape_and_cache_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                        _i32, _i32, _vp, _vp]),
    "pa_decode_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _i32, _i32,
                             _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "pa_swap_blocks": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _sz, _i32, _i32, _vp, _vp]),
    "pa_decode_multi": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _i32, _i32, _i32,
                               _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _vp,
                               _vp]),
    "pa_decode_cascade": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, ctypes.c_float,
                                 _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz,
                                 _vp, _vp]),
    "pa_decode_cascade_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_cascade_groups": (_i32, [_pi32, _pi32, _i32, _i32, _i32, _pi32, _pi32,
                                 ctypes.POINTER(_i32)]),
    "pa_debug_set_wait_limit": (_i32, [_i32]),
    "pa_read_device_errors": (_i32, [_vp, _pi32, _i32, _vp]),
    "pa_bm_create": (_i32, [_i32, _i32, _pi32, ctypes.POINTER(_vp)]),
    "pa_bm_destroy": (None, [_vp]),
    "pa_bm_add_seq": (_i32, [_vp, _i64]),
    "pa_bm_append_slot": (_i32, [_vp, _i64, _pi64, _pi64, _pi64]),
    "pa_bm_fork": (_i32, [_vp, _i64, _i64]),
    "pa_bm_free": (_i32, [_vp, _i64]),
    "pa_bm_block_table": (_i32, [_vp, _i64, _pi32, _i32, _pi32, _pi32]),
    "pa_bm_refcount": (_i32, [_vp, ctypes.c_int32]),
    "pa_bm_num_free": (_i32, [_vp]),
    "pa_bm_free_list": (_i32, [_vp, _pi32, _i32]),
    "pa_bm_stats": (_i32, [_vp, _pi64]),
    "pa_bm_append_slots": (_i32, [_vp, _pi64, _i32, _pi64, _pi64, _pi32, _pi32]),
    "pa_bm_build_block_tables": (_i32, [_vp, _pi64, _i32, _pi32, _i32, _pi32]),
    "pa_bm_enable_swap": (_i32, [_vp, _i32, _pi32]),
    "pa_bm_swap_out": (_i32, [_vp, _i64, _pi64, _i32, _pi32]),
    "pa_bm_swap_in": (_i32, [_vp, _i64, _pi64, _i32, _pi32]),
    "pa_bm_num_free_host": (_i32, [_vp]),
    "pa_bm_host_free_list": (_i32, [_vp, _pi32, _i32]),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def library():
    """Load libpagedattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                    "g.build()\"` (needs nvcc); there is no fallback implementation")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class PaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {pa_get_error_string(status)} (status {status})")


class OutOfBlocks(PaError):
    pass


class Swapped(PaError):
    pass


def _check(rc: int, what: str):
    if rc != PA_OK:
        if rc == PA_ERR_OUT_OF_BLOCKS:
            raise OutOfBlocks(rc, what)
        if rc == PA_ERR_SWAPPED:
            raise Swapped(rc, what)
        raise PaError(rc, what)


def pa_get_error_string(status: int) -> str:
    return library().pa_get_error_string(int(status)).decode()


# ---------------------------------------------------------------- marshalling
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    import torch
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported element type {t.dtype}")


def _need_cuda_contig(name, t):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


class PreparedCall:
    """One C-ABI call with its arguments marshalled once.  Calling it enqueues
    the same call again -- same pointers, sizes and stream -- so the tensors it
    was made from must stay alive and in place.  The device-op wrappers below
    return one instead of calling when given ``prepare=True``: for loops that
    issue the same step over and over with no per-call argument checks."""

    __slots__ = ("name", "fn", "args")

    def __init__(self, name, args):
        self.name, self.fn, self.args = name, getattr(library(), name), args

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != PA_OK:
            _check(rc, self.name)


# ----------------------------------------------------------------- device ops
def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, device_errors=None, stream=None,
                         prepare=False):
    """k, v [T, Hkv, D]; caches [NB, Hkv, bs, D]; slot_mapping int64 [T] (see pa.h)."""
    import torch
    for n, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("slot_mapping", slot_mapping)):
        _need_cuda_contig(n, t)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    NB, Hkv, bs, D = k_cache.shape
    call = PreparedCall("pa_reshape_and_cache", (
        _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), int(k.shape[0]),
        int(Hkv), int(D), int(bs), int(NB), _dtype_code(k_cache), _ptr(device_errors),
        _stream(stream, k_cache.device)))
    if prepare:
        return call
    call()


def pa_copy_blocks(k_cache, v_cache, src_dst_pairs, device_errors=None, stream=None,
                   prepare=False):
    """src_dst_pairs int64 [P, 2] on the device (see pa.h)."""
    import torch
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("src_dst_pairs", src_dst_pairs)):
        _need_cuda_contig(n, t)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    NB = k_cache.shape[0]
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    call = PreparedCall("pa_copy_blocks", (_ptr(k_cache), _ptr(v_cache), _ptr(src_dst_pairs),
                                  int(src_dst_pairs.shape[0]), block_bytes, int(NB),
                                  _ptr(device_errors), _stream(stream, k_cache.device)))
    if prepare:
        return call
    call()


def pa_swap_blocks(src_k, src_v, dst_k, dst_v, src_dst_pairs, device_errors=None, stream=None):
    """dst[d] = src[s] for each (s, d) row of src_dst_pairs (int64 [P, 2] on the
    device), K and V; pools [blocks, ...] of equal block size, each in device
    memory or pinned host memory (see pa.h)."""
    import torch
    for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v)):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must be a contiguous CUDA tensor or pinned host tensor")
    _need_cuda_contig("src_dst_pairs", src_dst_pairs)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    block_bytes = src_k[0].numel() * src_k.element_size()
    if dst_k[0].numel() * dst_k.element_size() != block_bytes:
        raise ValueError("the two pools have different block sizes")
    device = src_dst_pairs.device
    rc = library().pa_swap_blocks(_ptr(src_k), _ptr(src_v), _ptr(dst_k), _ptr(dst_v),
                                  _ptr(src_dst_pairs), int(src_dst_pairs.shape[0]), block_bytes,
                                  int(src_k.shape[0]), int(dst_k.shape[0]), _ptr(device_errors),
                                  _stream(stream, device))
    _check(rc, "pa_swap_blocks")


def pa_decode_chunk_tokens(num_seqs, num_kv_heads, block_size, max_context_len) -> int:
    rc = library().pa_decode_chunk_tokens(int(num_seqs), int(num_kv_heads), int(block_size),
                                          int(max_context_len))
    if rc < 0:
        _check(rc, "pa_decode_chunk_tokens")
    return rc


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_context_len, chunk_tokens=0) -> int:
    return int(library().pa_decode_workspace_size(int(num_seqs), int(num_q_heads),
                                                  int(num_kv_heads), int(head_dim),
                                                  int(block_size), int(max_context_len),
                                                  int(chunk_tokens)))


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
              max_context_len, workspace=None, chunk_tokens=0, device_errors=None, stream=None,
              prepare=False):
    """out, q [B, Hq, D]; caches [NB, Hkv, bs, D]; block_tables int32 [B, max_blocks];
    context_lens int32 [B] (see pa.h).  ``workspace``: a uint8 CUDA tensor of at
    least pa_decode_workspace_size() bytes; allocated here when None."""
    import torch
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(n, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if int(Hkv) != int(num_kv_heads):
        raise ValueError("num_kv_heads does not match the cache shape")
    if workspace is None:
        nbytes = pa_decode_workspace_size(B, Hq, Hkv, D, bs, max_context_len, chunk_tokens)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    call = PreparedCall("pa_decode", (
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), int(num_kv_heads), int(B), int(Hq), int(D), int(bs), int(NB),
        int(block_tables.shape[1]), int(max_context_len), _dtype_code(q), int(chunk_tokens),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(device_errors),
        _stream(stream, q.device)))
    if prepare:
        return call
    call()
    return out


def pa_decode_multi(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                    max_context_len, workspace=None, chunk_tokens=0, device_errors=None,
                    stream=None, prepare=False):
    """Causal paged attention for q_len new tokens per sequence: out, q
    [B, q_len, Hq, D]; the rest as pa_decode (see pa.h)."""
    import torch
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(n, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    B, q_len, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if int(Hkv) != int(num_kv_heads):
        raise ValueError("num_kv_heads does not match the cache shape")
    if workspace is None:
        nbytes = pa_decode_workspace_size(B, q_len * Hq, Hkv, D, bs, max_context_len, chunk_tokens)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    call = PreparedCall("pa_decode_multi", (
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), int(num_kv_heads), int(B), int(Hq), int(q_len), int(D), int(bs), int(NB),
        int(block_tables.shape[1]), int(max_context_len), _dtype_code(q), int(chunk_tokens),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(device_errors),
        _stream(stream, q.device)))
    if prepare:
        return call
    call()
    return out


def pa_decode_cascade_workspace_size(num_seqs, num_groups, num_q_heads, num_kv_heads, head_dim,
                                     block_size, max_context_len, chunk_tokens=0):
    n = library().pa_decode_cascade_workspace_size(
        int(num_seqs), int(num_groups), int(num_q_heads), int(num_kv_heads), int(head_dim),
        int(block_size), int(max_context_len), int(chunk_tokens))
    if n == 0 and num_seqs > 0:
        raise PaError(PA_ERR_UNSUPPORTED, "pa_decode_cascade_workspace_size: unsupported sizes")
    return n


def pa_cascade_groups(block_tables, context_lens, block_size):
    """Groups of sequences sharing leading pages (see pa.h), from host int32
    arrays block_tables [B, max_blocks] and context_lens [B].  Returns numpy
    int32 (group_start [G + 1], shared_lens [G])."""
    import numpy as np
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = int(lens.shape[0])
    if tables.ndim != 2 or tables.shape[0] != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    starts = np.zeros(B + 1, np.int32)
    shared = np.zeros(max(B, 1), np.int32)
    n = _i32(0)
    rc = library().pa_cascade_groups(
        tables.ctypes.data_as(_pi32), lens.ctypes.data_as(_pi32), B, int(tables.shape[1]),
        int(block_size), starts.ctypes.data_as(_pi32), shared.ctypes.data_as(_pi32),
        ctypes.byref(n))
    _check(rc, "pa_cascade_groups")
    return starts[:n.value + 1].copy(), shared[:n.value].copy()


def pa_decode_cascade(out, q, k_cache, v_cache, block_tables, context_lens, group_start,
                      shared_lens, scale, num_kv_heads, max_context_len, workspace=None,
                      chunk_tokens=0, device_errors=None, stream=None, prepare=False):
    """Shared-prefix decode (see pa.h): pa_decode's arguments plus group_start
    int32 [groups + 1] and shared_lens int32 [groups] (device tensors); bf16."""
    import torch
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens),
                 ("group_start", group_start), ("shared_lens", shared_lens)):
        _need_cuda_contig(n, t)
    for n, t in (("block_tables", block_tables), ("context_lens", context_lens),
                 ("group_start", group_start), ("shared_lens", shared_lens)):
        if t.dtype != torch.int32:
            raise TypeError(f"{n} must be int32")
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    G = shared_lens.numel()
    if group_start.numel() != G + 1:
        raise ValueError("group_start must have one more entry than shared_lens")
    if int(Hkv) != int(num_kv_heads):
        raise ValueError("num_kv_heads does not match the cache shape")
    if workspace is None:
        nbytes = pa_decode_cascade_workspace_size(B, G, Hq, Hkv, D, bs, max_context_len,
                                                  chunk_tokens)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    call = PreparedCall("pa_decode_cascade", (
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(group_start), _ptr(shared_lens), int(G), float(scale), int(num_kv_heads), int(B),
        int(Hq), int(D), int(bs), int(NB), int(block_tables.shape[1]), int(max_context_len),
        int(chunk_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(device_errors), _stream(stream, q.device)))
    if prepare:
        return call
    call()
    return out


PA_NOALLOC_SCRATCH_BYTES = 96 << 20


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                      max_context_len, chunk_tokens=0, device_errors=None, stream=None):
    """pa_decode without a workspace, for callers that cannot allocate device
    memory: the library's static scratch array (PA_NOALLOC_SCRATCH_BYTES) is used
    instead.  Calls share that array, so calls that could overlap on the GPU must
    be serialised; the first call on a device looks the array up and should come
    before any stream capture."""
    import torch
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _need_cuda_contig(n, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if int(Hkv) != int(num_kv_heads):
        raise ValueError("num_kv_heads does not match the cache shape")
    rc = library().pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), int(num_kv_heads), int(B), int(Hq), int(D), int(bs), int(NB),
        int(block_tables.shape[1]), int(max_context_len), _dtype_code(q), int(chunk_tokens),
        _ptr(device_errors), _stream(stream, q.device))
    _check(rc, "pa_decode_noalloc")
    return out


def _need_fp8_pool(name, t):
    _need_cuda_contig(name, t)
    if t.element_size() != 1:
        raise TypeError(f"{name} must hold one-byte e4m3 codes (uint8 or float8_e4m3fn)")


def _need_scales(k_scale, v_scale, num_kv_heads):
    import torch
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need_cuda_contig(n, t)
        if t.dtype != torch.float32 or t.numel() != num_kv_heads:
            raise TypeError(f"{n} must be float32 [num_kv_heads]")


def pa_reshape_and_cache_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale,
                             device_errors=None, stream=None, prepare=False):
    """k, v bf16 [T, Hkv, 128]; caches one-byte e4m3 [NB, Hkv, bs, 128];
    k_scale, v_scale float32 [Hkv] (see pa.h)."""
    import torch
    for n, t in (("k", k), ("v", v), ("slot_mapping", slot_mapping)):
        _need_cuda_contig(n, t)
    _need_fp8_pool("k_cache", k_cache)
    _need_fp8_pool("v_cache", v_cache)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("k and v must be bf16")
    NB, Hkv, bs, D = k_cache.shape
    _need_scales(k_scale, v_scale, Hkv)
    call = PreparedCall("pa_reshape_and_cache_fp8", (
        _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), _ptr(k_scale),
        _ptr(v_scale), int(k.shape[0]), int(Hkv), int(D), int(bs), int(NB), _ptr(device_errors),
        _stream(stream, k_cache.device)))
    if prepare:
        return call
    call()


def pa_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                  num_kv_heads, max_context_len, workspace=None, chunk_tokens=0,
                  device_errors=None, stream=None, prepare=False):
    """pa_decode over e4m3 pools: out, q bf16 [B, Hq, 128]; caches one-byte
    [NB, Hkv, bs, 128]; k_scale, v_scale float32 [Hkv] (see pa.h)."""
    import torch
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables),
                 ("context_lens", context_lens)):
        _need_cuda_contig(n, t)
    _need_fp8_pool("k_cache", k_cache)
    _need_fp8_pool("v_cache", v_cache)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("q and out must be bf16")
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if int(Hkv) != int(num_kv_heads):
        raise ValueError("num_kv_heads does not match the cache shape")
    _need_scales(k_scale, v_scale, Hkv)
    if workspace is None:
        nbytes = pa_decode_workspace_size(B, Hq, Hkv, D, bs, max_context_len, chunk_tokens)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    call = PreparedCall("pa_decode_fp8", (
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), _ptr(k_scale), _ptr(v_scale), int(num_kv_heads), int(B), int(Hq), int(D),
        int(bs), int(NB), int(block_tables.shape[1]), int(max_context_len), int(chunk_tokens),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(device_errors),
        _stream(stream, q.device)))
    if prepare:
        return call
    call()
    return out


def pa_debug_set_wait_limit(polls: int) -> None:
    """Test hook: bound every decode pipeline wait to `polls` polls (< 0: normal)."""
    _check(library().pa_debug_set_wait_limit(int(polls)), "pa_debug_set_wait_limit")


def pa_read_device_errors(device_errors, clear=True, stream=None) -> int:
    """Synchronise the stream and return (and optionally clear) the error bits."""
    flags = ctypes.c_int32(0)
    rc = library().pa_read_device_errors(_ptr(device_errors), ctypes.byref(flags), int(clear),
                                         _stream(stream, device_errors.device))
    _check(rc, "pa_read_device_errors")
    return int(flags.value)


# -------------------------------------------------------------- block manager
def _i64p(a):
    return a.ctypes.data_as(_pi64)


def _i32p(a):
    return a.ctypes.data_as(_pi32)


class BlockManager:
    """Host block manager (C++ in the library): LIFO free list, reference
    counts, fork and copy-on-write -- see pa.h for the exact rules."""

    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        lib = library()
        self._lib = lib
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        handle = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            self._order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
            order = _i32p(self._order)
        _check(lib.pa_bm_create(self.num_blocks, self.block_size, order, ctypes.byref(handle)),
               "pa_bm_create")
        self._h = handle

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add_seq(self, seq_id: int):
        _check(self._lib.pa_bm_add_seq(self._h, int(seq_id)), "pa_bm_add_seq")

    def append_slot(self, seq_id: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.pa_bm_append_slot(self._h, int(seq_id), ctypes.byref(slot),
                                           ctypes.byref(src), ctypes.byref(dst)),
               "pa_bm_append_slot")
        return slot.value, src.value, dst.value

    def fork(self, parent: int, child: int):
        _check(self._lib.pa_bm_fork(self._h, int(parent), int(child)), "pa_bm_fork")

    def free(self, seq_id: int):
        _check(self._lib.pa_bm_free(self._h, int(seq_id)), "pa_bm_free")

    def block_table(self, seq_id: int):
        n, length = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.pa_bm_block_table(self._h, int(seq_id), None, 0, ctypes.byref(n),
                                           ctypes.byref(length)), "pa_bm_block_table")
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        _check(self._lib.pa_bm_block_table(self._h, int(seq_id), _i32p(out), n.value,
                                           ctypes.byref(n), ctypes.byref(length)),
               "pa_bm_block_table")
        return out[:n.value].tolist(), length.value

    def refcount(self, block: int) -> int:
        rc = self._lib.pa_bm_refcount(self._h, int(block))
        if rc < 0:
            _check(rc, "pa_bm_refcount")
        return rc

    def num_free(self) -> int:
        return self._lib.pa_bm_num_free(self._h)

    def free_list(self):
        n = self._lib.pa_bm_free_list(self._h, None, 0)
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._lib.pa_bm_free_list(self._h, _i32p(out), n)
        return out[:n].tolist()

    def stats(self):
        out = np.zeros(4, dtype=np.int64)
        _check(self._lib.pa_bm_stats(self._h, _i64p(out)), "pa_bm_stats")
        return tuple(int(x) for x in out)

    def append_slots(self, seq_ids):
        """One decode step: returns (slots int64 [n], cow_pairs int64 [P, 2])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        slots = np.zeros(max(n, 1), dtype=np.int64)
        pairs = np.zeros((max(n, 1), 2), dtype=np.int64)
        num_cow, done = ctypes.c_int(), ctypes.c_int()
        rc = self._lib.pa_bm_append_slots(self._h, _i64p(ids), n, _i64p(slots), _i64p(pairs),
                                          ctypes.byref(num_cow), ctypes.byref(done))
        _check(rc, "pa_bm_append_slots")
        return slots[:n], pairs[:num_cow.value]

    # swapping to a host pool
    def enable_swap(self, num_host_blocks: int, initial_host_order=None):
        order = None
        if initial_host_order is not None:
            self._host_order = np.ascontiguousarray(initial_host_order, dtype=np.int32)
            order = _i32p(self._host_order)
        _check(self._lib.pa_bm_enable_swap(self._h, int(num_host_blocks), order),
               "pa_bm_enable_swap")
        self.num_host_blocks = int(num_host_blocks)

    def _swap(self, fn, seq_id, what):
        # a sequence holds at most every block of the pool it moves from
        cap = max(self.num_blocks, getattr(self, "num_host_blocks", 0))
        pairs = np.zeros((cap, 2), dtype=np.int64)
        n = ctypes.c_int()
        _check(fn(self._h, int(seq_id), _i64p(pairs), cap, ctypes.byref(n)), what)
        return pairs[:n.value]

    def swap_out(self, seq_id: int):
        """Returns int64 [pages, 2] (device page, host block), table order."""
        return self._swap(self._lib.pa_bm_swap_out, seq_id, "pa_bm_swap_out")

    def swap_in(self, seq_id: int):
        """Returns int64 [pages, 2] (host block, device page), table order."""
        return self._swap(self._lib.pa_bm_swap_in, seq_id, "pa_bm_swap_in")

    def num_free_host(self) -> int:
        return self._lib.pa_bm_num_free_host(self._h)

    def host_free_list(self):
        n = self._lib.pa_bm_host_free_list(self._h, None, 0)
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._lib.pa_bm_host_free_list(self._h, _i32p(out), n)
        return out[:n].tolist()

    def build_block_tables(self, seq_ids, max_blocks: int):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        tables = np.zeros((max(n, 1), max_blocks), dtype=np.int32)
        lens = np.zeros(max(n, 1), dtype=np.int32)
        _check(self._lib.pa_bm_build_block_tables(self._h, _i64p(ids), n, _i32p(tables),
                                                  int(max_blocks), _i32p(lens)),
               "pa_bm_build_block_tables")
        return tables[:n], lens[:n]
