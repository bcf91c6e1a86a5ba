"""The bench's algorithmic byte counts on the CPU: the shared-prefix step from
the oracle's block manager, counted per child (pa_decode) and once per family
(the shared-prefix decode)."""
import numpy as np

import bench
import oracle
import pa_inputs


def test_shared_prefix_step_bytes():
    s = pa_inputs.shared_prefix_script(scale_parents=3, scale_children=4, prompt_len=200,
                                       tail=(0, 4))
    case, pairs = pa_inputs.shared_prefix_step(
        oracle.RefBlockManager(s.num_blocks, s.block_size, s.initial_free_order), s)
    Hkv, D, bs = s.num_kv_heads, s.head_dim, s.block_size
    row = 2 * Hkv * D * 2                                # K and V of one token, bf16
    L = case.context_lens.astype(np.int64)
    # every child: the parent's prompt plus its own new token
    assert np.array_equal(L, np.repeat(s.prefix_lens.astype(np.int64) + 1, 4))
    # copy-on-write: all but the last child of each family copy the partial page
    assert len(pairs) == 3 * 3
    plain = bench.shared_prefix_bytes(case, pairs)
    assert plain["kv"] == int(L.sum()) * row
    assert plain["copy"] == 2 * 2 * len(pairs) * Hkv * bs * D * 2
    starts = np.arange(0, 13, 4)
    shared = s.prefix_lens.astype(np.int64) // bs * bs
    casc = bench.shared_prefix_bytes(case, pairs, starts, shared)
    own = int(L.sum()) - 4 * int(shared.sum())
    assert casc["kv"] == (int(shared.sum()) + own) * row
    assert casc["kv_logical"] == plain["kv"]
    assert casc["decode"] - casc["kv"] == plain["decode"] - plain["kv"]   # q, out, tables
    assert casc["step"] - casc["decode"] == plain["step"] - plain["decode"]
