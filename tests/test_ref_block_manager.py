"""Pins of the oracle block manager (CPU only): the hand traces of the teaching
allocator and of shared pages / copy-on-write, plus invariants over seeded
random operation sequences and exhaustive short ones."""
import copy
import itertools

import numpy as np
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


def _is_swapped(fn):
    try:
        fn()
    except oracle.Swapped:
        return True
    return False


@pytest.mark.parametrize("name", ["bm_teaching_trace.txt", "bm_refcount_cow_trace.txt",
                                  "bm_swap_trace.txt"])
def test_hand_trace(name):
    header, steps = load_trace(name)
    bm = oracle.RefBlockManager(header["num_pages"], header["page_size"])
    if "host_blocks" in header:
        bm.enable_swap(header["host_blocks"])
    replay(bm, steps, _is_oom, _is_swapped)


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


# ------------------------------------------------------------------ swapping
def _apply_swap(bm, op, resident, swapped):
    kind, a, b = op
    try:
        if kind == "add":
            if a in resident or a in swapped:
                return "skip"
            bm.add_seq(a)
            resident.add(a)
        elif kind == "append":
            if a not in resident:
                return "skip"
            bm.append_slot(a)
        elif kind == "fork":
            if a not in resident or b in resident or b in swapped:
                return "skip"
            bm.fork(a, b)
            resident.add(b)
        elif kind == "free":
            if a not in resident and a not in swapped:
                return "skip"
            bm.free(a)
            resident.discard(a)
            swapped.discard(a)
        elif kind == "swapout":
            if a not in resident:
                return "skip"
            bm.swap_out(a)
            resident.discard(a)
            swapped.add(a)
        elif kind == "swapin":
            if a not in swapped:
                return "skip"
            bm.swap_in(a)
            swapped.discard(a)
            resident.add(a)
    except oracle.OutOfBlocks:
        return "oom"
    return "ok"


@pytest.mark.parametrize("seed", range(12))
def test_random_ops_with_swapping_keep_counts_consistent(seed):
    """Device refcounts equal the resident tables holding each page; the host
    free list holds exactly the host blocks no swapped sequence holds; a failed
    swap changes nothing; a swapped sequence keeps its length."""
    num_blocks, num_host, bs = 9, 7, 2
    bm = oracle.RefBlockManager(num_blocks, bs)
    bm.enable_swap(num_host)
    resident, swapped = set(), set()
    for op in pa_inputs.random_bm_ops(seed, 400, swap=True):
        before = copy.deepcopy(bm.__dict__)
        lengths = dict(bm.lengths)
        status = _apply_swap(bm, op, resident, swapped)
        if status == "oom":
            assert bm.__dict__ == before, "a failed operation changed the state"
        if op[0] in ("swapout", "swapin") and status == "ok":
            assert bm.lengths == lengths
        check_invariants(_Adapter(bm), num_blocks, resident)
        held = [h for s in swapped for h in bm.swapped[s]]
        assert len(held) == len(set(held))
        assert sorted(held + bm.host_free_list()) == list(range(num_host))
    for s in sorted(resident | swapped):
        bm.free(s)
    assert sorted(bm.free_list()) == list(range(num_blocks))
    assert sorted(bm.host_free_list()) == list(range(num_host))


def test_swapped_sequence_is_refused_growth_and_fork():
    bm = oracle.RefBlockManager(8, 4)
    bm.enable_swap(4)
    bm.add_seq(1)
    bm.swap_out(1)
    for fn in (lambda: bm.append_slot(1), lambda: bm.fork(1, 2), lambda: bm.block_table(1)):
        with pytest.raises(oracle.Swapped):
            fn()
    with pytest.raises(KeyError):
        bm.add_seq(1)


def test_swap_round_trip_preserves_the_attention_output():
    """Swap every other sequence out (page copies into a host pool), let other
    sequences take the freed pages and overwrite them, swap back in to fresh
    pages: the decode of the swapped sequences is bit-identical (the result
    depends on the logical sequence only -- vLLM ch. 3 §3.4)."""
    rng = np.random.default_rng(21)
    NB, NH, Hkv, bs, D, Hq = 40, 24, 2, 4, 8, 4
    bm = oracle.RefBlockManager(NB, bs, rng.permutation(NB).tolist())
    bm.enable_swap(NH, rng.permutation(NH).tolist())
    kc = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    vc = rng.standard_normal((NB, Hkv, bs, D)).astype(np.float32)
    hk = np.full((NH, Hkv, bs, D), np.nan, np.float32)
    hv = np.full((NH, Hkv, bs, D), np.nan, np.float32)
    lens = [9, 14, 3, 17]
    for s, L in enumerate(lens):
        bm.add_seq(s)
        for _ in range(L):
            bm.append_slot(s)
    q = rng.standard_normal((len(lens), Hq, D)).astype(np.float32)

    def decode(ids):
        tables = np.full((len(ids), 8), -1, np.int32)
        cl = np.zeros(len(ids), np.int32)
        for j, s in enumerate(ids):
            t, L = bm.block_table(s)
            tables[j, :len(t)] = t
            cl[j] = L
        return oracle.decode_f64(q[list(ids)], kc, vc, tables, cl, 0.35, Hkv, "f32")

    before = decode([1, 3])
    for s in (1, 3):
        oracle.copy_pages(kc, vc, hk, hv, bm.swap_out(s))
    bm.add_seq(7)                                        # reuses freed pages
    for _ in range(20):
        slot, _, _ = bm.append_slot(7)
        page, off = divmod(slot, bs)
        kc[page, :, off] = -99.0                          # and overwrites them
        vc[page, :, off] = 99.0
    for s in (3, 1):
        oracle.copy_pages(hk, hv, kc, vc, bm.swap_in(s))
    after = decode([1, 3])
    np.testing.assert_array_equal(after, before)

