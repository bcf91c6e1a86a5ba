"""ctypes front end of the C oracle (``pa_oracle.c``) -- test infrastructure only.

The C file holds the arithmetic; this module only compiles it with gcc (plain
``-O2``, no fast-math, no FMA contraction, so the fp64 result is the same on x86
and Arm) and marshals numpy arrays into it.
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
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "bf16": 1, "fp8": 2}


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
            lib.oracle_decode_f64.restype = ctypes.c_int
            lib.oracle_decode_f64.argtypes = [
                vp, vp, vp, vp, i32p, i32p, ctypes.c_double,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int]
            lib.oracle_decode_kv8_f64.restype = ctypes.c_int
            lib.oracle_decode_kv8_f64.argtypes = [
                vp, vp, vp, vp, i32p, i32p, ctypes.c_double, vp, vp,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int]
            lib.oracle_widen.restype = None
            lib.oracle_widen.argtypes = [vp, vp, ctypes.c_long, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _storage(a: np.ndarray, dtype: str) -> np.ndarray:
    want = {"bf16": np.uint16, "f32": np.float32, "fp8": np.uint8}[dtype]
    if a.dtype != want:
        raise TypeError(f"{dtype} data must be stored as {want.__name__}, got {a.dtype}")
    return np.ascontiguousarray(a)


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored elements (float32, or bf16 bit patterns as uint16) -> float64."""
    src = _storage(a, dtype)
    out = np.empty(src.shape, dtype=np.float64)
    _load().oracle_widen(out.ctypes.data, src.ctypes.data, src.size, DTYPE_CODES[dtype])
    return out


def decode_f64(q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
               dtype: str, rows=None, threads: int = 0) -> np.ndarray:
    """fp64 paged decode attention, the plain definition (see ``pa_oracle.c``).

    q [B, Hq, D], k_cache/v_cache [NB, Hkv, bs, D] as float32 or uint16 (bf16 bits),
    block_tables int32 [B, max_blocks], context_lens int32 [B].
    Returns float64 [B, Hq, D], or [len(rows), D] when ``rows`` lists (b, i) pairs.
    """
    q = _storage(q, dtype)
    k_cache = _storage(k_cache, dtype)
    v_cache = _storage(v_cache, dtype)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or Hkv != num_kv_heads:
        raise ValueError("shape mismatch between q and the caches")
    if bt.ndim != 2 or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    if rows is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rows_arr, nrows = None, 0
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        nrows = rows_arr.shape[0]
        out = np.zeros((nrows, D), dtype=np.float64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    rc = _load().oracle_decode_f64(
        out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
        bt.ctypes.data_as(i32p), cl.ctypes.data_as(i32p), float(scale),
        B, Hq, num_kv_heads, D, bs, bt.shape[1], NB, DTYPE_CODES[dtype],
        rows_arr.ctypes.data_as(i32p) if rows_arr is not None else None, nrows, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_decode_f64 refused the input (status {rc})")
    return out


def decode_kv8_f64(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                   rows=None, threads: int = 0) -> np.ndarray:
    """fp64 paged decode with float8 e4m3 caches: K = code * k_scale[h],
    V = code * v_scale[h] for kv head h; q is bf16 (uint16 bits)."""
    q = _storage(q, "bf16")
    k_cache = _storage(k_cache, "fp8")
    v_cache = _storage(v_cache, "fp8")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    ks = np.ascontiguousarray(k_scale, dtype=np.float64)
    vs = np.ascontiguousarray(v_scale, dtype=np.float64)
    if D2 != D or v_cache.shape != k_cache.shape or ks.shape != (Hkv,) or vs.shape != (Hkv,):
        raise ValueError("shape mismatch")
    if rows is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rows_arr, nrows = None, 0
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        nrows = rows_arr.shape[0]
        out = np.zeros((nrows, D), dtype=np.float64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    rc = _load().oracle_decode_kv8_f64(
        out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
        bt.ctypes.data_as(i32p), cl.ctypes.data_as(i32p), float(scale), ks.ctypes.data,
        vs.ctypes.data, B, Hq, Hkv, D, bs, bt.shape[1], NB,
        rows_arr.ctypes.data_as(i32p) if rows_arr is not None else None, nrows, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_decode_kv8_f64 refused the input (status {rc})")
    return out


def decode_multi_f64(q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads,
                     dtype: str, rows=None, threads: int = 0) -> np.ndarray:
    """fp64 paged attention for q_len new tokens per sequence, causal.

    q [B, q_len, Hq, D]; context_lens counts all q_len new tokens, so query token
    j of sequence b sits at position L_b - q_len + j and attends to positions
    0 .. L_b - q_len + j of its own sequence (each new token sees the prefix and
    the new tokens before it, itself included).  That is the single-token decode
    of a sequence cut at that position, so this is written as exactly that:
    one decode row per (b, j) over the same block table with length
    L_b - q_len + j + 1 (rows with no key return zeros).
    Returns float64 [B, q_len, Hq, D], or [len(rows), D] for (b, j, i) triples.
    """
    q = np.asarray(q)
    B, q_len, Hq, D = q.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.asarray(context_lens, dtype=np.int64)
    vlens = (cl[:, None] - q_len + np.arange(q_len)[None, :] + 1).clip(min=0).astype(np.int32)
    vq = np.ascontiguousarray(q.reshape(B * q_len, Hq, D))
    vbt = np.ascontiguousarray(np.repeat(bt, q_len, axis=0))
    if rows is None:
        out = decode_f64(vq, k_cache, v_cache, vbt, vlens.reshape(-1), scale, num_kv_heads, dtype,
                         threads=threads)
        return out.reshape(B, q_len, Hq, D)
    trip = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    vrows = np.stack([trip[:, 0] * q_len + trip[:, 1], trip[:, 2]], axis=1)
    return decode_f64(vq, k_cache, v_cache, vbt, vlens.reshape(-1), scale, num_kv_heads, dtype,
                      rows=vrows, threads=threads)

