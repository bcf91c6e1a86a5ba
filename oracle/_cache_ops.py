"""Oracle cache write and page copy -- test infrastructure only.

Both are plain element copies on numpy arrays (float32, or bf16 bit patterns as
uint16), so they are exact by construction and compared byte for byte.
"""
from __future__ import annotations

import numpy as np


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping) -> None:
    """Write token t's K/V rows into slot ``slot_mapping[t]``, in place.

    "PagedAttention原理" §3.3.4 (append_token): a new token's K/V goes into the
    next free position of the sequence's last page; a global slot number names
    that position as physical_page * page_size + offset.  A negative slot marks a
    padding token and writes nothing.

    k, v [T, Hkv, D]; k_cache, v_cache [NB, Hkv, bs, D]; slot_mapping int64 [T].
    """
    T = k.shape[0]
    NB, Hkv, bs, D = k_cache.shape
    if k.shape != (T, Hkv, D) or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    for t in range(T):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        page, offset = divmod(slot, bs)
        if page >= NB:
            raise ValueError(f"slot {slot} is outside the pool")
        for h in range(Hkv):
            k_cache[page, h, offset, :] = k[t, h, :]
            v_cache[page, h, offset, :] = v[t, h, :]


def copy_blocks(k_cache, v_cache, src_dst_pairs) -> None:
    """Copy whole pages, all heads, K and V: cache[dst] = cache[src] for each pair.

    "mlx-paged-attention" feature 2 (memory sharing and copy-on-write): a shared
    page is duplicated only when one of its holders is about to modify it.
    Pairs are applied in order; callers give distinct destinations that are not
    also sources, which makes the order irrelevant.
    """
    pairs = np.asarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2)
    NB = k_cache.shape[0]
    for src, dst in pairs:
        if not (0 <= src < NB and 0 <= dst < NB):
            raise ValueError(f"pair ({src}, {dst}) is outside the pool")
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]


def copy_pages(src_k, src_v, dst_k, dst_v, src_dst_pairs) -> None:
    """Copy whole pages between two pools: dst[d] = src[s] for each pair, K and V.

    "PagedAttention MLX：为Apple Silicon打造的高吞吐量LLM推理引擎" (dynamic
    scheduling; physical KV pool): pages of inactive requests are swapped out to
    CPU memory and back.  A swap is this copy from the device pool to a host pool
    (or back) for the pairs the block manager hands out.
    """
    pairs = np.asarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2)
    for src, dst in pairs:
        if not (0 <= src < src_k.shape[0] and 0 <= dst < dst_k.shape[0]):
            raise ValueError(f"pair ({src}, {dst}) is outside a pool")
        dst_k[dst] = src_k[src]
        dst_v[dst] = src_v[src]


# ------------------------------------------------------------------ float8 e4m3
def e4m3_value(code: int) -> float:
    """Value of an e4m3 code: 1 sign bit, 4 exponent bits (bias 7), 3 fraction
    bits; exponent 0 is subnormal (fraction * 2^-9); 0x7F / 0xFF are NaN."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_POS = np.array([e4m3_value(c) for c in range(0x7F)])     # codes 0..126, increasing


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> e4m3 codes: the nearest representable value, ties to
    the even code; magnitudes past the largest finite value (448) saturate to
    it; NaN -> 0x7F.  The sign bit follows the input's sign."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    code = np.where(d_hi < d_lo, hi, lo)
    tie = d_hi == d_lo
    code = np.where(tie & (hi != lo), np.where(hi % 2 == 0, hi, lo), code)
    code = np.where(a >= _E4M3_POS[126], 126, code)            # saturate (incl. +-inf)
    code = code.astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def reshape_and_cache_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale) -> None:
    """The cache write with float8 e4m3 pools: each element of token t, kv head
    h is stored as e4m3(k / k_scale[h]) (the division in float32), likewise v.
    k, v: bf16 bits (uint16) [T, Hkv, D]; caches uint8 [NB, Hkv, bs, D]."""
    from ._decode import widen
    T = k.shape[0]
    NB, Hkv, bs, D = k_cache.shape
    ks = np.asarray(k_scale, dtype=np.float32).reshape(1, Hkv, 1)
    vs = np.asarray(v_scale, dtype=np.float32).reshape(1, Hkv, 1)
    kq = e4m3_encode(widen(k, "bf16").astype(np.float32) / ks)
    vq = e4m3_encode(widen(v, "bf16").astype(np.float32) / vs)
    reshape_and_cache(kq, vq, k_cache, v_cache, slot_mapping)
