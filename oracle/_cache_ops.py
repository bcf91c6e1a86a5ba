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
