"""CPU oracle for paged-KV decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm may import this package.  The product (``paged_kv_cache_190_gb300``)
never imports it and shares no code with it; the two meet only through the
seeded input generators in ``pa_inputs``.

Contents, each written from the pages (cited in the modules):
  * ``decode_f64``         -- fp64 gather-then-attend over the block table (plain C).
  * ``decode_multi_f64``   -- the same for q_len new tokens per sequence, causal.
  * ``reshape_and_cache``  -- byte copy of each new token's K/V into its slot.
  * ``copy_blocks``        -- byte copy of whole pages for copy-on-write.
  * ``e4m3_encode`` / ``decode_kv8_f64`` / ``reshape_and_cache_fp8`` -- the same
                              path with float8 e4m3 pools and per-kv-head scales.
  * ``RefBlockManager``    -- the teaching allocator of "PagedAttention原理" §3.3.4
                              with the reference counts of §3.3.3, copy-on-write and
                              swapping whole sequences to a host pool.
  * ``copy_pages``         -- byte copy of pages between two pools (the swap copy).
"""
from ._decode import (build, decode_f64, decode_kv8_f64, decode_multi_f64, library_path,
                      max_threads, widen)
from ._cache_ops import (copy_blocks, copy_pages, e4m3_encode, e4m3_value, reshape_and_cache,
                         reshape_and_cache_fp8)
from .ref_block_manager import OutOfBlocks, RefBlockManager, Swapped

__all__ = [
    "build", "decode_f64", "decode_kv8_f64", "decode_multi_f64", "library_path", "max_threads",
    "widen",
    "copy_blocks", "copy_pages", "e4m3_encode", "e4m3_value", "reshape_and_cache",
    "reshape_and_cache_fp8", "OutOfBlocks", "RefBlockManager", "Swapped",
]
