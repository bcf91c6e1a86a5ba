"""The library's C++ block manager against the oracle's (CPU only): the hand
traces, seeded random operation sequences (every result and the whole state
compared after each step), the batched step call, and the shared-prefix script
run to the end with every page back on the free list."""
import pytest

import numpy as np

import oracle
import pa_inputs
import paged_kv_cache_190_gb300 as pa
from bm_trace import check_invariants, load_trace, replay


def _is_oom(fn):
    try:
        fn()
    except pa.OutOfBlocks:
        return True
    return False


def _is_swapped(fn):
    try:
        fn()
    except pa.Swapped:
        return True
    return False


@pytest.mark.parametrize("name", ["bm_teaching_trace.txt", "bm_refcount_cow_trace.txt",
                                  "bm_swap_trace.txt"])
def test_hand_trace(name):
    header, steps = load_trace(name)
    bm = pa.BlockManager(header["num_pages"], header["page_size"])
    if "host_blocks" in header:
        bm.enable_swap(header["host_blocks"])
    replay(bm, steps, _is_oom, _is_swapped)


def _state(bm, nb, live, refcount):
    tables = {s: bm.block_table(s) for s in sorted(live)}
    return tables, list(bm.free_list()), [refcount(p) for p in range(nb)]


def _do(bm, op, errors):
    kind, a, b = op
    try:
        if kind == "add":
            bm.add_seq(a)
            return "ok"
        if kind == "append":
            return bm.append_slot(a)
        if kind == "fork":
            bm.fork(a, b)
            return "ok"
        if kind == "free":
            bm.free(a)
            return "ok"
    except errors as e:
        return type(e).__name__
    raise ValueError(kind)


@pytest.mark.parametrize("seed", range(20))
@pytest.mark.parametrize("nb,bs", [(7, 2), (12, 4), (30, 16)])
def test_matches_oracle_on_random_operations(seed, nb, bs):
    prod = pa.BlockManager(nb, bs, np.random.default_rng(seed).permutation(nb))
    ref = oracle.RefBlockManager(nb, bs, np.random.default_rng(seed).permutation(nb))
    live = set()
    for op in pa_inputs.random_bm_ops(seed * 7 + nb, 400):
        kind, a, b = op
        # only issue operations whose preconditions hold; the errors compared are OOM
        if kind == "add" and a in live:
            continue
        if kind in ("append", "free") and a not in live:
            continue
        if kind == "fork" and (a not in live or b in live):
            continue
        r_prod = _do(prod, op, (pa.OutOfBlocks,))
        r_ref = _do(ref, op, (oracle.OutOfBlocks,))
        if r_ref == "OutOfBlocks":
            assert r_prod == "OutOfBlocks", op
        else:
            assert r_prod == r_ref, (op, r_prod, r_ref)
            if kind in ("add",):
                live.add(a)
            elif kind == "fork":
                live.add(b)
            elif kind == "free":
                live.discard(a)
        assert _state(prod, nb, live, prod.refcount) == _state(ref, nb, live,
                                                                lambda p: ref.refcount[p]), op
        assert prod.stats() == ref.stats()
    check_invariants(prod, nb, live)
    for s in sorted(live):
        prod.free(s)
    assert sorted(prod.free_list()) == list(range(nb))
    assert all(prod.refcount(p) == 0 for p in range(nb))


def test_batched_step_equals_single_calls():
    nb, bs = 64, 4
    a = pa.BlockManager(nb, bs)
    b = oracle.RefBlockManager(nb, bs)
    for s in range(5):
        a.add_seq(s), b.add_seq(s)
        for _ in range(s * 3 + 1):
            a.append_slot(s), b.append_slot(s)
    a.fork(2, 7), b.fork(2, 7)
    a.fork(4, 8), b.fork(4, 8)
    ids = [0, 2, 7, 4, 8, 1]
    slots, pairs = a.append_slots(ids)
    want = [b.append_slot(s) for s in ids]
    assert slots.tolist() == [w[0] for w in want]
    assert [tuple(p) for p in pairs.tolist()] == [(w[1], w[2]) for w in want if w[1] >= 0]
    tables, lens = a.build_block_tables(ids, 8)
    for j, s in enumerate(ids):
        t, L = b.block_table(s)
        assert tables[j, :len(t)].tolist() == t and all(tables[j, len(t):] == -1)
        assert lens[j] == L


def test_out_of_blocks_leaves_state_unchanged():
    bm = pa.BlockManager(3, 2)
    bm.add_seq(0)
    bm.fork(0, 1)                  # page 2 shared by sequences 0 and 1
    bm.add_seq(2)
    bm.add_seq(3)                  # free list now empty
    before = (bm.free_list(), bm.block_table(0), bm.block_table(1), bm.stats())
    with pytest.raises(pa.OutOfBlocks):
        bm.append_slot(1)          # needs a copy of the shared page: none free
    with pytest.raises(pa.OutOfBlocks):
        bm.add_seq(9)
    assert (bm.free_list(), bm.block_table(0), bm.block_table(1), bm.stats()) == before


def test_unknown_and_duplicate_ids():
    bm = pa.BlockManager(4, 2)
    bm.add_seq(1)
    with pytest.raises(pa.PaError):
        bm.add_seq(1)
    with pytest.raises(pa.PaError):
        bm.append_slot(5)
    with pytest.raises(pa.PaError):
        bm.fork(1, 1)
    with pytest.raises(pa.PaError):
        bm.free(3)


def _run_script(bm, script, after_step=None):
    prefix_slots = pa_inputs.shared_prefix_prefill(bm, script)
    _, children = pa_inputs.shared_prefix_ids(script)
    trace = [[s.tolist() for s in prefix_slots]]
    slots, pairs = bm.append_slots(children) if hasattr(bm, "append_slots") else (None, None)
    if slots is None:
        res = [bm.append_slot(c) for c in children]
        slots = [r[0] for r in res]
        pairs = [(r[1], r[2]) for r in res if r[1] >= 0]
    trace.append((list(map(int, slots)), [tuple(map(int, p)) for p in pairs]))
    if after_step is not None:
        after_step(bm, children)
    # finish: every child generates its tail, then leaves in the scripted order
    remaining = {c: int(script.tails[c]) for c in children}
    step = 0
    order = pa_inputs.shared_prefix_finish_order(script)
    while remaining:
        active = [c for c in children if c in remaining and remaining[c] > step]
        if active:
            res = [bm.append_slot(c) for c in active]
            trace.append([tuple(map(int, r)) for r in res])
        for c in order:
            if c in remaining and remaining[c] == step:
                bm.free(c)
                del remaining[c]
        step += 1
    return trace


def test_shared_prefix_script_matches_oracle_and_returns_every_page():
    script = pa_inputs.shared_prefix_script(scale_parents=3, scale_children=5, prompt_len=100,
                                            tail=(0, 40))
    prod = pa.BlockManager(script.num_blocks, script.block_size, script.initial_free_order)
    ref = oracle.RefBlockManager(script.num_blocks, script.block_size, script.initial_free_order)
    t_prod = _run_script(prod, script)
    t_ref = _run_script(ref, script)
    assert t_prod == t_ref
    # the step's copies: in each family all but the last child copy the partial page
    cows = t_prod[1][1]
    assert len(cows) == script.num_parents * (script.children_per_parent - 1)
    assert prod.num_free() == script.num_blocks
    assert sorted(prod.free_list()) == list(range(script.num_blocks))
    assert all(prod.refcount(p) == 0 for p in range(script.num_blocks))


def test_shared_prefix_script_full_size():
    """The shared-prefix workload at its stated size: 8 parents of 2048 + g_p
    tokens fork 16 children each, every child writes one token (copy-on-write of
    its family's partial page), then generates its tail of U{0..512} tokens and
    leaves in the scripted random order.  Library and oracle managers agree on
    every slot and copy; right after the step the reference counts are what the
    sharing implies; at the end every page is back on the free list."""
    script = pa_inputs.shared_prefix_script()
    P, C, bs = script.num_parents, script.children_per_parent, script.block_size
    assert (P, C) == (8, 16) and all(2049 <= n <= 2063 for n in script.prefix_lens)

    def after_step(bm, children):
        rc = (lambda p: bm.refcount[p]) if isinstance(bm.refcount, list) else bm.refcount
        for p in range(P):
            fam = children[p * C:(p + 1) * C]
            tables = [bm.block_table(c)[0] for c in fam]
            full = int(script.prefix_lens[p]) // bs
            shared = tables[-1][:full]
            for t in tables:                       # the full prompt pages stay shared by all
                assert t[:full] == shared
            assert all(rc(page) == C for page in shared)
            # the partial page: C - 1 children copied it, the last wrote in place
            last = [t[full] for t in tables]
            assert len(set(last)) == C and all(rc(page) == 1 for page in last)
        used = sum(1 for page in range(script.num_blocks) if rc(page) > 0)
        assert used + bm.num_free() == script.num_blocks

    prod = pa.BlockManager(script.num_blocks, bs, script.initial_free_order)
    ref = oracle.RefBlockManager(script.num_blocks, bs, script.initial_free_order)
    t_prod = _run_script(prod, script, after_step)
    t_ref = _run_script(ref, script, after_step)
    assert t_prod == t_ref
    assert len(t_prod[1][1]) == P * (C - 1)
    assert len(t_prod) - 2 == int(script.tails.max())          # one trace entry per later step
    for bm in (prod, ref):
        assert bm.num_free() == script.num_blocks
        assert sorted(bm.free_list()) == list(range(script.num_blocks))
    assert all(prod.refcount(p) == 0 for p in range(script.num_blocks))
    assert all(r == 0 for r in ref.refcount)


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("nb,nh,bs", [(7, 5, 2), (20, 9, 4)])
def test_swapping_matches_oracle_on_random_operations(seed, nb, nh, bs):
    """Swap-out / swap-in mixed into the random operations: the copy pairs, the
    refusals, both free lists and the resident tables match the oracle's."""
    rng = np.random.default_rng(seed)
    order, host_order = rng.permutation(nb), rng.permutation(nh)
    prod, ref = pa.BlockManager(nb, bs, order), oracle.RefBlockManager(nb, bs, order.tolist())
    prod.enable_swap(nh, host_order)
    ref.enable_swap(nh, host_order.tolist())
    resident, swapped = set(), set()
    for kind, a, b in pa_inputs.random_bm_ops(seed * 11 + nb, 500, swap=True):
        if kind == "add" and (a in resident or a in swapped):
            continue
        if kind == "fork" and (b in resident or b in swapped):
            continue
        if kind in ("append", "fork", "free", "swapout") and a not in resident | swapped:
            continue
        if kind == "swapin" and a not in resident | swapped:
            continue
        results = []
        for bm, errs in ((prod, (pa.OutOfBlocks, pa.Swapped, pa.PaError)),
                         (ref, (oracle.OutOfBlocks, oracle.Swapped, KeyError))):
            try:
                if kind == "add":
                    bm.add_seq(a); r = "ok"
                elif kind == "append":
                    r = tuple(bm.append_slot(a))
                elif kind == "fork":
                    bm.fork(a, b); r = "ok"
                elif kind == "free":
                    bm.free(a); r = "ok"
                elif kind == "swapout":
                    r = [tuple(int(x) for x in p) for p in bm.swap_out(a)]
                else:
                    r = [tuple(int(x) for x in p) for p in bm.swap_in(a)]
            except errs as e:
                r = {"Swapped": "swapped", "OutOfBlocks": "oom"}.get(type(e).__name__, "refused")
            results.append(r)
        r_prod, r_ref = results
        assert r_prod == r_ref, (kind, a, b, r_prod, r_ref)
        if r_ref not in ("oom", "swapped", "refused"):
            if kind == "add":
                resident.add(a)
            elif kind == "fork":
                resident.add(b)
            elif kind == "free":
                resident.discard(a); swapped.discard(a)
            elif kind == "swapout":
                resident.discard(a); swapped.add(a)
            elif kind == "swapin":
                swapped.discard(a); resident.add(a)
        assert list(prod.free_list()) == ref.free_list()
        assert list(prod.host_free_list()) == ref.host_free_list()
        for q in sorted(resident):
            got, L = prod.block_table(q)
            assert (list(got), L) == ref.block_table(q)
        assert prod.stats() == ref.stats()
    for q in sorted(resident | swapped):
        prod.free(q)
    assert sorted(prod.free_list()) == list(range(nb))
    assert sorted(prod.host_free_list()) == list(range(nh))

