"""Pins of the oracle block manager (CPU only): the hand traces of the teaching
allocator and of shared pages / copy-on-write, plus invariants over seeded
random operation sequences and exhaustive short ones."""
import copy
import itertools

import pytest

import oracle
import pa_inputs
from bm_trace import check_invariants, load_trace, replay


class _Adapter:
    """Gives the oracle manager the refcount() query the invariant checker uses."""

    def __init__(self, bm):
        self.bm = bm
        self.block_size = bm.block_size

    def __getattr__(self, name):
        return getattr(self.bm, name)

    def refcount(self, page):
        return self.bm.refcount[page]


def _is_oom(fn):
    try:
        fn()
    except oracle.OutOfBlocks:
        return True
    return False


@pytest.mark.parametrize("name", ["bm_teaching_trace.txt", "bm_refcount_cow_trace.txt"])
def test_hand_trace(name):
    header, steps = load_trace(name)
    bm = oracle.RefBlockManager(header["num_pages"], header["page_size"])
    replay(bm, steps, _is_oom)


def _apply(bm, op, live):
    kind, a, b = op
    try:
        if kind == "add":
            if a in live:
                return "skip"
            bm.add_seq(a)
            live.add(a)
        elif kind == "append":
            if a not in live:
                return "skip"
            bm.append_slot(a)
        elif kind == "fork":
            if a not in live or b in live:
                return "skip"
            bm.fork(a, b)
            live.add(b)
        elif kind == "free":
            if a not in live:
                return "skip"
            bm.free(a)
            live.discard(a)
    except oracle.OutOfBlocks:
        return "oom"
    return "ok"


@pytest.mark.parametrize("seed", range(12))
def test_random_ops_keep_counts_consistent(seed):
    num_blocks, bs = 9, 2
    bm = oracle.RefBlockManager(num_blocks, bs)
    live = set()
    for op in pa_inputs.random_bm_ops(seed, 300):
        before = copy.deepcopy(bm.__dict__)
        status = _apply(bm, op, live)
        if status == "oom":
            assert bm.__dict__ == before, "a failed allocation changed the state"
        check_invariants(_Adapter(bm), num_blocks, live)
    for s in sorted(live):
        bm.free(s)
    assert sorted(bm.free_list()) == list(range(num_blocks))
    assert all(r == 0 for r in bm.refcount)


def test_exhaustive_short_sequences():
    """Every sequence of 6 operations over two sequence ids on a 3-page pool."""
    alphabet = [("add", 0, 0), ("add", 1, 1), ("append", 0, 0), ("append", 1, 1),
                ("fork", 0, 1), ("fork", 1, 0), ("free", 0, 0), ("free", 1, 1)]
    count = 0
    for ops in itertools.product(alphabet, repeat=6):
        bm = oracle.RefBlockManager(3, 2)
        live = set()
        for op in ops:
            _apply(bm, op, live)
        check_invariants(_Adapter(bm), 3, live)
        for s in sorted(live):
            bm.free(s)
        assert sorted(bm.free_list()) == [0, 1, 2]
        count += 1
    assert count == 8 ** 6


def test_cow_last_holder_writes_in_place():
    bm = oracle.RefBlockManager(40, 16)
    bm.add_seq(0)
    for _ in range(20):
        bm.append_slot(0)
    for c in range(1, 5):
        bm.fork(0, c)
    bm.free(0)
    pairs = [bm.append_slot(c) for c in range(1, 5)]
    cows = [(s, d) for _, s, d in pairs if s >= 0]
    assert len(cows) == 3                                  # 4 holders: 3 copy, the last writes in place
    assert len({d for _, d in cows}) == 3
    shared_partial = bm.block_table(4)[0][1]
    assert bm.refcount[shared_partial] == 1 and all(s == shared_partial for s, _ in cows)
