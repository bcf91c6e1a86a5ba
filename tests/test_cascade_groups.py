"""Host grouping for the shared-prefix decode (pa_cascade_groups, C++), on the CPU:
a hand-worked example, the forked families of the shared-prefix script, and the
defining properties on random batches built by sharing pages."""
import numpy as np
import pytest

import pa_inputs
import paged_kv_cache_190_gb300 as pa


def test_worked_example():
    # seqs 0-2 share pages 1, 2 (seq 1's third page differs); seq 3 alone; seqs 4
    # and 5 share page 9, but seq 4 has only 10 tokens: no whole page below them
    t = np.array([[1, 2, 3, -1], [1, 2, 4, -1], [1, 2, 3, 5], [7, 8, -1, -1], [9, -1, -1, -1],
                  [9, 10, -1, -1]], np.int32)
    lens = np.array([40, 40, 60, 20, 10, 20], np.int32)
    starts, shared = pa.pa_cascade_groups(t, lens, 16)
    assert starts.tolist() == [0, 3, 6] and shared.tolist() == [32, 0]
    # the shortest member keeps one token of its own: 32 tokens -> 1 shared page
    lens[1] = 32
    starts, shared = pa.pa_cascade_groups(t, lens, 16)
    assert starts.tolist() == [0, 3, 6] and shared.tolist() == [16, 0]


def test_forked_families_are_the_groups():
    s = pa_inputs.shared_prefix_script(scale_parents=4, scale_children=3, prompt_len=100,
                                       tail=(0, 4))
    bm = pa.BlockManager(s.num_blocks, s.block_size, s.initial_free_order)
    pa_inputs.shared_prefix_prefill(bm, s)
    _, children = pa_inputs.shared_prefix_ids(s)
    bm.append_slots(children)              # copy-on-write of each family's partial page
    mb = max(len(bm.block_table(c)[0]) for c in children)
    tables, lens = bm.build_block_tables(children, mb)
    starts, shared = pa.pa_cascade_groups(tables, lens, s.block_size)
    C = s.children_per_parent
    assert starts.tolist() == list(range(0, len(children) + 1, C))
    assert shared.tolist() == [int(n) // s.block_size * s.block_size for n in s.prefix_lens]


@pytest.mark.parametrize("seed", range(6))
def test_random_batches_have_maximal_valid_groups(seed):
    rng = np.random.default_rng(seed)
    bs, B, mb = 16, 40, 12
    tables = np.full((B, mb), -1, np.int32)
    lens = rng.integers(0, mb * bs + 1, size=B).astype(np.int32)
    nxt = 0
    for b in range(B):
        n = (int(lens[b]) + bs - 1) // bs
        tables[b, :n] = np.arange(nxt, nxt + n)
        nxt += n
        if b and rng.random() < 0.6 and lens[b - 1] > 0 and n > 0:
            k = int(rng.integers(0, min(n, (int(lens[b - 1]) + bs - 1) // bs) + 1))
            tables[b, :k] = tables[b - 1, :k]              # fork from the previous sequence
    starts, shared = pa.pa_cascade_groups(tables, lens, bs)
    assert starts[0] == 0 and starts[-1] == B and np.all(np.diff(starts) > 0)
    for f in range(len(shared)):
        g0, g1, sl = int(starts[f]), int(starts[f + 1]), int(shared[f])
        assert sl % bs == 0 and sl >= 0
        if sl == 0:
            continue
        npg = sl // bs
        assert g1 - g0 >= 2
        for b in range(g0, g1):
            assert lens[b] > sl                            # one own token at least
            assert np.array_equal(tables[b, :npg], tables[g0, :npg])
        # maximal: one more page is not common to all, or not below every length
        more_common = all(tables[b, npg] == tables[g0, npg] >= 0 for b in range(g0, g1)) \
            if npg < mb else False
        more_fits = all(lens[b] > sl + bs for b in range(g0, g1))
        assert not (more_common and more_fits)


def test_empty_batch_and_bad_arguments():
    starts, shared = pa.pa_cascade_groups(np.zeros((0, 4), np.int32), np.zeros(0, np.int32), 16)
    assert starts.tolist() == [0] and shared.tolist() == []
    with pytest.raises(pa.PaError):
        pa.pa_cascade_groups(np.zeros((2, 4), np.int32), np.array([5, -1], np.int32), 16)
