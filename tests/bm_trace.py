"""Reader and replayer of the hand-written block-manager traces in tests/golden/.

A trace line reads ``op args -> result ; SEQ=[pages] ; free=[pages]``, with an
optional ``; host=[blocks]`` (the host free list) for swap traces.  The replayer
drives any manager with the oracle's method names (add_seq, append_slot, fork,
free, swap_out, swap_in, block_table, free_list, host_free_list) and compares
each result.
"""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _ids(text):
    text = text.strip()[1:-1].strip()
    return [int(x) for x in text.split(",")] if text else []


def load_trace(name):
    header, steps = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if "->" not in line:
                key, value = line.split()
                header[key] = int(value)
                continue
            lhs, rhs = line.split("->")
            op = lhs.split()
            parts = [part.strip() for part in rhs.split(";")]
            result, table, free = parts[:3]
            host = _ids(parts[3].split("=", 1)[1]) if len(parts) > 3 else None
            steps.append((op, result, table, _ids(free.split("=", 1)[1]), host))
    return header, steps


def _pairs(text):
    return [tuple(int(x) for x in p.split(":")) for p in text.split(",")] if text else []


def replay(manager, steps, is_oom, is_swapped=None):
    """``is_oom(callable)`` runs an operation and says whether it reported an
    out-of-blocks error (raising anything else); ``is_swapped(callable)`` likewise
    for the refusal of an operation on a swapped-out sequence."""
    names = {}

    def sid(name):
        return names.setdefault(name, len(names) + 10)

    for op, result, table, free, host in steps:
        kind = op[0]
        if result == "swapped":
            args = [sid(x) for x in op[1:]]
            fn = {"append": manager.append_slot, "fork": manager.fork}[kind]
            assert is_swapped(lambda: fn(*args)), op
        elif kind in ("swapout", "swapin") and result == "oom":
            fn = manager.swap_out if kind == "swapout" else manager.swap_in
            assert is_oom(lambda: fn(sid(op[1]))), op
        elif kind in ("swapout", "swapin"):
            fn = manager.swap_out if kind == "swapout" else manager.swap_in
            got = [tuple(int(x) for x in p) for p in fn(sid(op[1]))]
            assert got == _pairs(result), (op, got, result)
        elif kind == "add":
            if result == "oom":
                assert is_oom(lambda: manager.add_seq(sid(op[1]))), op
            else:
                manager.add_seq(sid(op[1]))
        elif kind == "append":
            slot, src, dst = manager.append_slot(sid(op[1]))
            parts = result.split()
            assert slot == int(parts[0]), (op, slot, result)
            if len(parts) > 1:
                assert parts[1] == "cow" and (src, dst) == (int(parts[2]), int(parts[3])), (op, src, dst)
            else:
                assert (src, dst) == (-1, -1), (op, src, dst)
        elif kind == "fork":
            manager.fork(sid(op[1]), sid(op[2]))
        elif kind == "free":
            manager.free(sid(op[1]))
        else:
            raise ValueError(kind)
        if table != "-":
            seq, pages = table.split("=")
            got, _ = manager.block_table(sid(seq))
            assert list(got) == _ids(pages), (op, got, pages)
        assert list(manager.free_list()) == free, (op, manager.free_list(), free)
        if host is not None:
            assert list(manager.host_free_list()) == host, (op, manager.host_free_list(), host)


def check_invariants(manager, num_blocks, live):
    """Reference counts equal the number of live tables holding each page; the
    free list holds exactly the pages with count zero, each once."""
    holders = [0] * num_blocks
    for s in live:
        pages, length = manager.block_table(s)
        for p in pages:
            holders[p] += 1
        bs = manager.block_size
        assert (len(pages) - 1) * bs <= length <= len(pages) * bs or (length == 0 and len(pages) == 1)
    for p in range(num_blocks):
        assert manager.refcount(p) == holders[p], (p, manager.refcount(p), holders[p])
    free = list(manager.free_list())
    assert len(free) == len(set(free))
    assert set(free) == {p for p in range(num_blocks) if holders[p] == 0}


