"""Pins of the oracle's cache write and page copies to facts outside themselves
(CPU only).

* hand traces of where each new token lands (``golden/reshape_slots_trace.txt``)
  and of what every page holds after a copy (``golden/copy_blocks_trace.txt``),
  with NaN canaries in every cell that must stay untouched;
* the float8 write with power-of-two scales stores codes whose value times the
  head's scale is the input exactly;
* composition: slots from the oracle block manager, written by the oracle cache
  write, decoded by the (already pinned) oracle decode, equal dense fp64 SDPA on
  each sequence's logical K/V -- so a token written to the wrong cell changes a
  decode that a library routine fixes;
* copy-on-write: after the page copy of a shared partial page and one append,
  every sharer's decode is unchanged and every writer's equals dense SDPA on its
  own logical sequence;
* planted mistakes in copies of ``oracle/_cache_ops.py`` each fail one of the above.
"""
import importlib.util
import math
import os

import numpy as np
import pytest
import torch

import oracle
import pa_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ORACLE_OPS = os.path.join(os.path.dirname(oracle.__file__), "_cache_ops.py")


def _read_golden(name):
    head, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key in ("token",):
                rows.append(rest)
            else:
                head[key] = rest
    return head, rows


def _pairs(text):
    return np.array([[int(x) for x in p.split()] for p in text.split(";")], np.int64)


# ------------------------------------------------------------ the pin checks
# Each takes the module under test (the oracle's, or a planted-mistake copy).
def check_reshape_trace(ops):
    head, rows = _read_golden("reshape_slots_trace.txt")
    bs, NB = int(head["page_size"]), int(head["num_pages"])
    Hkv, D = int(head["num_kv_heads"]), int(head["head_dim"])
    T = len(rows)
    t_ = np.arange(T)[:, None, None]
    h_ = np.arange(Hkv)[None, :, None]
    d_ = np.arange(D)[None, None, :]
    k = (10 * t_ + 2 * h_ + d_ + 1).astype(np.float32)
    v = -k
    slots = np.zeros(T, np.int64)
    expect = []                                             # (token, page, offset)
    for r in rows:
        lhs, rhs = r.split("->")
        tok, _, slot = lhs.split()
        slots[int(tok)] = int(slot)
        rhs = rhs.split()
        if rhs[0] != "none":
            expect.append((int(tok), int(rhs[1]), int(rhs[3])))
    kc = np.full((NB, Hkv, bs, D), np.nan, np.float32)
    vc = np.full((NB, Hkv, bs, D), np.nan, np.float32)
    ops.reshape_and_cache(k, v, kc, vc, slots)
    written = np.zeros((NB, bs), bool)
    for tok, page, off in expect:
        np.testing.assert_array_equal(kc[page, :, off, :], k[tok])
        np.testing.assert_array_equal(vc[page, :, off, :], v[tok])
        written[page, off] = True
    # every other cell is still NaN (nothing written anywhere else)
    assert np.all(np.isnan(kc[~written[:, None, :, None].repeat(Hkv, 1).repeat(D, 3)
                             .reshape(NB, Hkv, bs, D)]))
    assert np.all(np.isnan(vc[~written[:, None, :, None].repeat(Hkv, 1).repeat(D, 3)
                             .reshape(NB, Hkv, bs, D)]))


def _coded_pool(NB, Hkv, bs, D):
    p = np.arange(NB)[:, None, None, None]
    h = np.arange(Hkv)[None, :, None, None]
    o = np.arange(bs)[None, None, :, None]
    d = np.arange(D)[None, None, None, :]
    k = (1000 * p + 100 * h + 10 * o + d + 1).astype(np.float32)
    return k, -k


def check_copy_trace(ops):
    head, _ = _read_golden("copy_blocks_trace.txt")
    bs, NB = int(head["page_size"]), int(head["num_pages"])
    Hkv, D = int(head["num_kv_heads"]), int(head["head_dim"])
    k0, v0 = _coded_pool(NB, Hkv, bs, D)
    kc, vc = k0.copy(), v0.copy()
    ops.copy_blocks(kc, vc, _pairs(head["pairs"]))
    for i, src in enumerate(int(x) for x in head["k_sources"].split()):
        np.testing.assert_array_equal(kc[i], k0[src])
    for i, src in enumerate(int(x) for x in head["v_sources"].split()):
        np.testing.assert_array_equal(vc[i], v0[src])
    # between two pools
    ky = np.full_like(k0, np.nan)
    vy = np.full_like(v0, np.nan)
    kx, vx = k0.copy(), v0.copy()
    ops.copy_pages(kx, vx, ky, vy, _pairs(head["pool_pairs"]))
    np.testing.assert_array_equal(kx, k0)                  # the source pool is only read
    np.testing.assert_array_equal(vx, v0)
    for i, src in enumerate(head["y_sources"].split()):
        if src == "nan":
            assert np.all(np.isnan(ky[i])) and np.all(np.isnan(vy[i]))
        else:
            np.testing.assert_array_equal(ky[i], k0[int(src)])
            np.testing.assert_array_equal(vy[i], v0[int(src)])


def _code_values(codes):
    """Values of e4m3 codes, one Python int at a time."""
    codes = np.asarray(codes)
    return np.array([oracle.e4m3_value(int(c)) for c in codes.ravel()]).reshape(codes.shape)


def check_fp8_write_exact(ops):
    """Inputs that are e4m3 values times a power-of-two scale are stored as the
    code of that value: code value x scale == input, bit for bit."""
    Hkv, D, bs, NB, T = 3, 8, 4, 5, 6
    k_scale = np.array([0.5, 2.0, 0.125], np.float32)
    v_scale = np.array([4.0, 0.25, 1.0], np.float32)
    rng = np.random.default_rng(3)
    # finite, non-NaN codes whose values stay in bf16's exact range after scaling
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.int64)
    kcode = rng.choice(codes, size=(T, Hkv, D)).astype(np.uint8)
    vcode = rng.choice(codes, size=(T, Hkv, D)).astype(np.uint8)
    kval = _code_values(kcode) * k_scale[None, :, None]
    vval = _code_values(vcode) * v_scale[None, :, None]
    k = pa_inputs.to_storage(kval.astype(np.float32), "bf16")
    v = pa_inputs.to_storage(vval.astype(np.float32), "bf16")
    assert np.array_equal(oracle.widen(k, "bf16"), kval)   # exact in bf16 too
    slots = np.array([0, 5, 19, -1, 9, 14], np.int64)
    kc = np.full((NB, Hkv, bs, D), 0x7F, np.uint8)
    vc = np.full((NB, Hkv, bs, D), 0x7F, np.uint8)
    ops.reshape_and_cache_fp8(k, v, kc, vc, slots, k_scale, v_scale)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        page, off = s // bs, s % bs
        got_k = _code_values(kc[page, :, off, :]) * k_scale[:, None]
        got_v = _code_values(vc[page, :, off, :]) * v_scale[:, None]
        np.testing.assert_array_equal(got_k, kval[t])
        np.testing.assert_array_equal(got_v, vval[t])


def _torch_widen(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(torch.float64)


def _dense(q_row, k_log, v_log, scale, G):
    """Dense fp64 SDPA of one sequence: q [Hq, D], k/v [L, Hkv, D] (stored form)."""
    qt = _torch_widen(q_row, "bf16")[:, None, :]
    kt = _torch_widen(k_log, "bf16").permute(1, 0, 2).repeat_interleave(G, dim=0)
    vt = _torch_widen(v_log, "bf16").permute(1, 0, 2).repeat_interleave(G, dim=0)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[:, 0].numpy()


def _tables(bm, seqs):
    rows = [bm.block_table(s) for s in seqs]
    mb = max(len(t) for t, _ in rows)
    tables = np.full((len(seqs), mb), -1, np.int32)
    lens = np.zeros(len(seqs), np.int32)
    for j, (t, L) in enumerate(rows):
        tables[j, :len(t)] = t
        lens[j] = L
    return tables, lens


def check_bm_write_decode_equals_dense(ops):
    """Slots from the block manager, K/V written token by token in decode steps
    (with a padding token in every batch), then the decode equals dense SDPA on
    the tokens in the order each sequence produced them."""
    dtype, Hq, Hkv, D, bs, NB = "bf16", 4, 2, 16, 4, 24
    G = Hq // Hkv
    rng = np.random.default_rng(11)
    bm = oracle.RefBlockManager(NB, bs, rng.permutation(NB).tolist())
    target = {0: 9, 1: 4, 2: 14}
    logs = {s: ([], []) for s in target}
    kc = pa_inputs.nan_fill((NB, Hkv, bs, D), dtype)
    vc = pa_inputs.nan_fill((NB, Hkv, bs, D), dtype)
    for s in target:
        bm.add_seq(s)
    step = 0
    while any(len(logs[s][0]) < target[s] for s in target):
        live = [s for s in target if len(logs[s][0]) < target[s]]
        slots = [bm.append_slot(s)[0] for s in live] + [-1]
        k = pa_inputs.to_storage(rng.standard_normal((len(slots), Hkv, D), dtype=np.float32), dtype)
        v = pa_inputs.to_storage(rng.standard_normal((len(slots), Hkv, D), dtype=np.float32), dtype)
        for j, s in enumerate(live):
            logs[s][0].append(k[j])
            logs[s][1].append(v[j])
        ops.reshape_and_cache(k, v, kc, vc, np.array(slots, np.int64))
        step += 1
    seqs = sorted(target)
    tables, lens = _tables(bm, seqs)
    q = pa_inputs.to_storage(rng.standard_normal((len(seqs), Hq, D), dtype=np.float32), dtype)
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode_f64(q, kc, vc, tables, lens, scale, Hkv, dtype)
    for j, s in enumerate(seqs):
        want = _dense(q[j], np.stack(logs[s][0]), np.stack(logs[s][1]), scale, G)
        np.testing.assert_allclose(got[j], want, rtol=0, atol=1e-12)


def check_copy_on_write_decode(ops):
    """A parent with a partial last page is forked twice; each holder then
    appends one token.  The two children copy the shared page before writing
    (the parent, the last holder, writes in place).  Afterwards every sequence's
    decode equals dense SDPA on its own logical tokens, and a decode of the
    parent's old length is what it was before the copies."""
    dtype, Hq, Hkv, D, bs, NB = "bf16", 4, 2, 16, 4, 12
    G = Hq // Hkv
    rng = np.random.default_rng(12)
    bm = oracle.RefBlockManager(NB, bs, rng.permutation(NB).tolist())
    kc = pa_inputs.nan_fill((NB, Hkv, bs, D), dtype)
    vc = pa_inputs.nan_fill((NB, Hkv, bs, D), dtype)
    bm.add_seq(0)
    pk = pa_inputs.to_storage(rng.standard_normal((6, Hkv, D), dtype=np.float32), dtype)
    pv = pa_inputs.to_storage(rng.standard_normal((6, Hkv, D), dtype=np.float32), dtype)
    for t in range(6):                                      # 2 pages, the second half full
        slot = bm.append_slot(0)[0]
        ops.reshape_and_cache(pk[t:t + 1], pv[t:t + 1], kc, vc, np.array([slot], np.int64))
    bm.fork(0, 1)
    bm.fork(0, 2)
    scale = 1.0 / math.sqrt(D)
    q = pa_inputs.to_storage(rng.standard_normal((3, Hq, D), dtype=np.float32), dtype)
    t_before, l_before = _tables(bm, [0])
    before = oracle.decode_f64(q[:1], kc, vc, t_before, l_before, scale, Hkv, dtype)
    nk = pa_inputs.to_storage(rng.standard_normal((3, Hkv, D), dtype=np.float32), dtype)
    nv = pa_inputs.to_storage(rng.standard_normal((3, Hkv, D), dtype=np.float32), dtype)
    order = [1, 2, 0]
    copies = 0
    for s in order:
        slot, src, dst = bm.append_slot(s)
        if src >= 0:
            ops.copy_blocks(kc, vc, np.array([[src, dst]], np.int64))
            copies += 1
        ops.reshape_and_cache(nk[s:s + 1], nv[s:s + 1], kc, vc, np.array([slot], np.int64))
        if s == 1:
            # the parent still reads its shared pages unchanged
            np.testing.assert_array_equal(
                oracle.decode_f64(q[:1], kc, vc, t_before, l_before, scale, Hkv, dtype), before)
    assert copies == 2
    tables, lens = _tables(bm, [0, 1, 2])
    got = oracle.decode_f64(q, kc, vc, tables, lens, scale, Hkv, dtype)
    for s in (0, 1, 2):
        want = _dense(q[s], np.concatenate([pk, nk[s:s + 1]]), np.concatenate([pv, nv[s:s + 1]]),
                      scale, G)
        np.testing.assert_allclose(got[s], want, rtol=0, atol=1e-12)


CHECKS = [check_reshape_trace, check_copy_trace, check_fp8_write_exact,
          check_bm_write_decode_equals_dense, check_copy_on_write_decode]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_oracle_cache_ops_pin(check):
    from oracle import _cache_ops
    check(_cache_ops)


# ------------------------------------------------------------ planted mistakes
MUTANTS = {
    "slot offset off by one": ("page, offset = divmod(slot, bs)\n",
                               "page, offset = divmod(slot, bs)\n        offset = (offset + 1) % bs\n"),
    "V written from K": ("v_cache[page, h, offset, :] = v[t, h, :]",
                         "v_cache[page, h, offset, :] = k[t, h, :]"),
    "padding slot written": ("if slot < 0:\n            continue", "if slot < -1:\n            continue"),
    "kv heads crossed": ("k_cache[page, h, offset, :] = k[t, h, :]",
                         "k_cache[page, h, offset, :] = k[t, Hkv - 1 - h, :]"),
    "page copy V from K": ("v_cache[dst] = v_cache[src]", "v_cache[dst] = k_cache[src]"),
    "page copy reversed": ("k_cache[dst] = k_cache[src]\n        v_cache[dst] = v_cache[src]",
                           "k_cache[src] = k_cache[dst]\n        v_cache[src] = v_cache[dst]"),
    "pool copy V from K": ("dst_v[dst] = src_v[src]", "dst_v[dst] = src_k[src]"),
    "pool copy to the source index": ("dst_k[dst] = src_k[src]", "dst_k[src] = src_k[src]"),
    "fp8 V divided by K's scale": ('vq = e4m3_encode(widen(v, "bf16").astype(np.float32) / vs)',
                                   'vq = e4m3_encode(widen(v, "bf16").astype(np.float32) / ks)'),
}


def _load_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    with open(ORACLE_OPS) as f:
        src = f.read()
    assert src.count(old) == 1, name
    path = tmp_path / "_cache_ops_mutant.py"
    path.write_text(src.replace(old, new))
    # a submodule of the oracle package, so its relative import resolves
    spec = importlib.util.spec_from_file_location("oracle._cache_ops_mutant", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_cache_pins_catch_planted_mistake(name, tmp_path):
    mod = _load_mutant(name, tmp_path)
    failed = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mod)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"planted mistake '{name}' was not caught by any cache pin"
