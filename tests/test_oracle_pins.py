"""Pins of the CPU decode oracle to facts outside itself (CPU only).

* bf16 widening against hand-decoded bit patterns and against torch's cast;
* a decode example solved by hand;
* equality with a library routine (torch fp64 scaled_dot_product_attention) on
  logically contiguous K/V that the test scatters into pages itself;
* closed forms (one token returns V exactly, constant V, identical keys);
* invariants of paging (page permutation, block size 16 vs 32, shared pages
  equal private copies);
* planted mistakes in a copy of the oracle's C source are caught.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import pa_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _scatter_into_pool(k_log, v_log, tables, lens, num_blocks, block_size, dtype, fill=None):
    """Test-side placement: token t of sequence b goes to page tables[b][t // bs],
    offset t % bs.  k_log[b] is [L_b, Hkv, D] storage."""
    Hkv, D = k_log[0].shape[1], k_log[0].shape[2]
    k_pool = pa_inputs.nan_fill((num_blocks, Hkv, block_size, D), dtype)
    v_pool = pa_inputs.nan_fill((num_blocks, Hkv, block_size, D), dtype)
    for b, L in enumerate(lens):
        for t in range(L):
            page = tables[b][t // block_size]
            k_pool[page, :, t % block_size, :] = k_log[b][t]
            v_pool[page, :, t % block_size, :] = v_log[b][t]
    return k_pool, v_pool


def _random_logical(seed, lens, Hq, Hkv, D, dtype, std=1.0):
    rng = _rng(seed)
    k_log = [pa_inputs.to_storage(rng.standard_normal((L, Hkv, D), dtype=np.float32) * std, dtype)
             for L in lens]
    v_log = [pa_inputs.to_storage(rng.standard_normal((L, Hkv, D), dtype=np.float32) * std, dtype)
             for L in lens]
    q = pa_inputs.to_storage(rng.standard_normal((len(lens), Hq, D), dtype=np.float32) * std, dtype)
    return rng, k_log, v_log, q


def _tables_from_perm(perm, lens, block_size, max_blocks):
    tables = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    cur = 0
    for b, L in enumerate(lens):
        n = (L + block_size - 1) // block_size
        tables[b, :n] = perm[cur:cur + n]
        cur += n
    return tables


def _torch_widen(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(torch.float64)


# ---------------------------------------------------------------- bf16 widening
def test_bf16_widen_matches_hand_decoded_patterns():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                bits, value = line.split()
                rows.append((int(bits, 16), float(value)))
    bits = np.array([r[0] for r in rows], dtype=np.uint16)
    got = oracle.widen(bits, "bf16")
    for (b, want), g in zip(rows, got):
        assert g == want and math.copysign(1.0, g) == math.copysign(1.0, want), hex(b)


def test_bf16_widen_matches_torch_cast():
    rng = _rng(7)
    bits = rng.integers(0, 1 << 16, size=20000).astype(np.uint16)
    exp_all_ones = (bits & 0x7F80) == 0x7F80
    bits = bits[~exp_all_ones]  # drop Inf/NaN patterns
    got = oracle.widen(bits, "bf16")
    want = _torch_widen(bits, "bf16").numpy()
    np.testing.assert_array_equal(got, want)


# ------------------------------------------------------------- worked example
def test_decode_worked_example_by_hand():
    with open(os.path.join(GOLDEN, "decode_worked_example.txt")) as f:
        line = [l for l in f if l.startswith("out")][0]
    want = np.array([float(x) for x in line.split()[1:]])
    k = np.full((3, 1, 2, 2), np.nan, dtype=np.float32)
    v = np.full((3, 1, 2, 2), np.nan, dtype=np.float32)
    k[2, 0, 0] = [0, 0]; v[2, 0, 0] = [1, 0]
    k[2, 0, 1] = [1, 0]; v[2, 0, 1] = [0, 1]
    k[0, 0, 0] = [2, 0]; v[0, 0, 0] = [1, 1]
    q = np.array([[[1.0, 0.0]]], dtype=np.float32)
    out = oracle.decode_f64(q, k, v, np.array([[2, 0]], np.int32), np.array([3], np.int32),
                            1.0, 1, "f32")
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-15)


# ------------------------------------------------ library routine: dense SDPA
def _sdpa_reference(q, k_log, v_log, lens, scale, Hkv, dtype):
    B, Hq, D = q.shape
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b, L in enumerate(lens):
        if L == 0:
            continue
        qt = _torch_widen(q[b], dtype)[:, None, :]                      # [Hq, 1, D]
        kt = _torch_widen(k_log[b], dtype).permute(1, 0, 2)             # [Hkv, L, D]
        vt = _torch_widen(v_log[b], dtype).permute(1, 0, 2)
        kt = kt.repeat_interleave(G, dim=0)                            # q head i -> kv head i // G
        vt = vt.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out


DENSE_CASES = [
    # dtype, B, Hq, Hkv, D, bs
    ("f32", 3, 4, 4, 64, 16),
    ("f32", 3, 8, 2, 64, 32),
    ("bf16", 4, 8, 2, 128, 16),
    ("bf16", 2, 8, 1, 128, 32),
    ("bf16", 3, 4, 4, 64, 16),
]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,D,bs", DENSE_CASES)
def test_oracle_equals_dense_sdpa(dtype, B, Hq, Hkv, D, bs):
    lens = [1, 17, 70][:B] + [33] * max(0, B - 3)
    rng, k_log, v_log, q = _random_logical(11 + B + D + bs, lens, Hq, Hkv, D, dtype)
    mb = max((L + bs - 1) // bs for L in lens)
    NB = sum((L + bs - 1) // bs for L in lens) + 3
    tables = _tables_from_perm(rng.permutation(NB).astype(np.int32), lens, bs, mb)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, lens, NB, bs, dtype)
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode_f64(q, kp, vp, tables, np.array(lens, np.int32), scale, Hkv, dtype)
    want = _sdpa_reference(q, k_log, v_log, lens, scale, Hkv, dtype)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# --------------------------------------------------------------- closed forms
def test_single_token_returns_v_exactly():
    dtype, Hq, Hkv, D, bs = "bf16", 8, 2, 128, 16
    rng, k_log, v_log, q = _random_logical(21, [1, 1], Hq, Hkv, D, dtype, std=30.0)
    tables = np.array([[5], [2]], np.int32)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, [1, 1], 7, bs, dtype)
    out = oracle.decode_f64(q, kp, vp, tables, np.array([1, 1], np.int32), 0.088, Hkv, dtype)
    for b in range(2):
        for i in range(Hq):
            np.testing.assert_array_equal(out[b, i], oracle.widen(v_log[b][0, i // (Hq // Hkv)], dtype))


def test_constant_values_give_that_value():
    dtype, Hq, Hkv, D, bs, L = "f32", 4, 4, 64, 16, 100
    rng, k_log, v_log, q = _random_logical(22, [L], Hq, Hkv, D, dtype)
    c = rng.standard_normal((Hkv, D)).astype(np.float32)
    v_log = [np.broadcast_to(c, (L, Hkv, D)).copy()]
    tables = np.array([rng.permutation(9)[:7]], np.int32)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, [L], 9, bs, dtype)
    out = oracle.decode_f64(q, kp, vp, tables, np.array([L], np.int32), 0.125, Hkv, dtype)
    np.testing.assert_allclose(out[0], c.astype(np.float64), rtol=1e-14, atol=1e-14)


def test_identical_keys_give_mean_of_values():
    dtype, Hq, Hkv, D, bs, L = "f32", 4, 2, 64, 32, 77
    rng, k_log, v_log, q = _random_logical(23, [L], Hq, Hkv, D, dtype)
    k_log = [np.broadcast_to(k_log[0][0], (L, Hkv, D)).copy()]
    tables = np.array([[4, 0, 2]], np.int32)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, [L], 5, bs, dtype)
    out = oracle.decode_f64(q, kp, vp, tables, np.array([L], np.int32), 0.125, Hkv, dtype)
    mean_v = v_log[0].astype(np.float64).mean(axis=0)            # [Hkv, D]
    for i in range(Hq):
        np.testing.assert_allclose(out[0, i], mean_v[i // 2], rtol=0, atol=1e-14)


def test_zero_length_row_is_zero():
    dtype = "f32"
    rng, k_log, v_log, q = _random_logical(24, [5, 0], 2, 2, 64, dtype)
    tables = np.array([[1], [-1]], np.int32)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, [5, 0], 3, 16, dtype)
    out = oracle.decode_f64(q, kp, vp, tables, np.array([5, 0], np.int32), 0.125, 2, dtype)
    assert np.all(out[1] == 0.0) and np.all(np.isfinite(out[0]))


# ---------------------------------------------------------- paging invariants
def test_page_permutation_leaves_output_bit_identical():
    dtype, Hq, Hkv, D, bs = "bf16", 8, 2, 128, 16
    lens = [200, 45, 16]
    rng, k_log, v_log, q = _random_logical(25, lens, Hq, Hkv, D, dtype)
    NB = 40
    outs = []
    for s in range(3):
        perm = _rng(100 + s).permutation(NB).astype(np.int32)
        tables = _tables_from_perm(perm, lens, bs, 13)
        kp, vp = _scatter_into_pool(k_log, v_log, tables, lens, NB, bs, dtype)
        outs.append(oracle.decode_f64(q, kp, vp, tables, np.array(lens, np.int32), 0.088, Hkv, dtype))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


def test_block_size_16_and_32_agree():
    dtype, Hq, Hkv, D = "bf16", 8, 2, 64
    lens = [100, 33]
    rng, k_log, v_log, q = _random_logical(26, lens, Hq, Hkv, D, dtype)
    outs = []
    for bs in (16, 32):
        mb = max((L + bs - 1) // bs for L in lens)
        NB = 20
        tables = _tables_from_perm(rng.permutation(NB).astype(np.int32), lens, bs, mb)
        kp, vp = _scatter_into_pool(k_log, v_log, tables, lens, NB, bs, dtype)
        outs.append(oracle.decode_f64(q, kp, vp, tables, np.array(lens, np.int32), 0.125, Hkv, dtype))
    np.testing.assert_array_equal(outs[0], outs[1])


def test_shared_pages_equal_private_copies():
    """N sequences whose tables point at the same prefix pages give the same
    output as N sequences each holding a private copy of those pages."""
    dtype, Hq, Hkv, D, bs, N = "bf16", 4, 1, 64, 16, 5
    prefix = 48
    rng = _rng(27)
    pk = pa_inputs.to_storage(rng.standard_normal((prefix, Hkv, D), dtype=np.float32), dtype)
    pv = pa_inputs.to_storage(rng.standard_normal((prefix, Hkv, D), dtype=np.float32), dtype)
    tails = [3, 0, 16, 9, 1]
    k_log, v_log = [], []
    for n in tails:
        tk = pa_inputs.to_storage(rng.standard_normal((n, Hkv, D), dtype=np.float32), dtype)
        tv = pa_inputs.to_storage(rng.standard_normal((n, Hkv, D), dtype=np.float32), dtype)
        k_log.append(np.concatenate([pk, tk]))
        v_log.append(np.concatenate([pv, tv]))
    lens = [prefix + n for n in tails]
    q = pa_inputs.to_storage(rng.standard_normal((N, Hq, D), dtype=np.float32), dtype)
    ctx = np.array(lens, np.int32)
    # private: every sequence has its own pages
    NB = 64
    tables_p = _tables_from_perm(rng.permutation(NB).astype(np.int32), lens, bs, 5)
    kp, vp = _scatter_into_pool(k_log, v_log, tables_p, lens, NB, bs, dtype)
    out_private = oracle.decode_f64(q, kp, vp, tables_p, ctx, 0.125, Hkv, dtype)
    # shared: the 3 prefix pages are the same physical pages in every table
    tables_s = np.full((N, 5), -1, np.int32)
    shared_ids = [7, 3, 11]
    free_ids = [i for i in range(NB) if i not in shared_ids]
    cur = 0
    for b, L in enumerate(lens):
        n = (L + bs - 1) // bs
        tables_s[b, :3] = shared_ids
        tables_s[b, 3:n] = free_ids[cur:cur + n - 3]
        cur += n - 3
    kp, vp = _scatter_into_pool(k_log, v_log, tables_s, lens, NB, bs, dtype)
    out_shared = oracle.decode_f64(q, kp, vp, tables_s, ctx, 0.125, Hkv, dtype)
    np.testing.assert_array_equal(out_private, out_shared)


def test_row_subset_matches_full_output():
    case = pa_inputs.scaled_workload("gqa_bf16", 6)
    oracle.reshape_and_cache(case.k_new, case.v_new, case.k_cache, case.v_cache, case.slot_mapping)
    args = (case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens, case.scale,
            case.num_kv_heads, case.dtype)
    full = oracle.decode_f64(*args)
    rows = [(0, 0), (5, 31), (2, 17), (3, 4)]
    sub = oracle.decode_f64(*args, rows=rows)
    for r, (b, i) in enumerate(rows):
        np.testing.assert_array_equal(sub[r], full[b, i])


def test_oracle_refuses_out_of_range_block():
    q = np.zeros((1, 1, 64), np.float32)
    k = np.zeros((2, 1, 16, 64), np.float32)
    with pytest.raises(ValueError):
        oracle.decode_f64(q, k, k, np.array([[2]], np.int32), np.array([3], np.int32), 1.0, 1, "f32")
    with pytest.raises(ValueError):
        oracle.decode_f64(q, k, k, np.array([[0]], np.int32), np.array([17], np.int32), 1.0, 1, "f32")


# ------------------------------------------------------------ planted mistakes
MUTANTS = {
    "scale dropped": ("s[t] = scale * dot;", "s[t] = dot;"),
    "head mapping i % Hkv": ("const int h = i / G;", "const int h = i % num_kv_heads;"),
    "slot offset off by one": ("const int offset = t % block_size;",
                               "const int offset = (t + 1) % block_size;"),
    "no normalisation": ("p[t] = p[t] / z;", "p[t] = p[t];"),
    "K read from the V pool": ("K[(size_t)t * D + d] = load_elem(k_cache,",
                               "K[(size_t)t * D + d] = load_elem(v_cache,"),
    "table row stride": ("block_tables[(size_t)b * max_blocks_per_seq + logical_page]",
                         "block_tables[(size_t)b * block_size + logical_page]"),
    "values read in reverse token order": ("out_row[d] += p[t] * V[(size_t)t * D + d];",
                                           "out_row[d] += p[t] * V[(size_t)(L - 1 - t) * D + d];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")).read()
    assert src.count(old) == 1, name
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(mutant_c), "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_decode_f64.restype = ctypes.c_int
    # the dense-SDPA pin on a GQA bf16 case with several pages and a ragged tail
    dtype, Hq, Hkv, D, bs = "bf16", 8, 2, 64, 16
    lens = [37, 70]
    rng, k_log, v_log, q = _random_logical(31, lens, Hq, Hkv, D, dtype)
    tables = _tables_from_perm(rng.permutation(12).astype(np.int32), lens, bs, 5)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, lens, 12, bs, dtype)
    # fill unused slots with finite values so a wrong slot reads data, not NaN
    kp[np.isnan(oracle.widen(kp, dtype))] = 0x3F80
    vp[np.isnan(oracle.widen(vp, dtype))] = 0x3F80
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((2, Hq, D))
    ctx = np.array(lens, np.int32)
    i32p = ctypes.POINTER(ctypes.c_int32)
    rc = lib.oracle_decode_f64(
        ctypes.c_void_p(out.ctypes.data), ctypes.c_void_p(q.ctypes.data),
        ctypes.c_void_p(kp.ctypes.data), ctypes.c_void_p(vp.ctypes.data),
        tables.ctypes.data_as(i32p), ctx.ctypes.data_as(i32p), ctypes.c_double(scale),
        2, Hq, Hkv, D, bs, tables.shape[1], 12, 1, None, 0, 1)
    want = _sdpa_reference(q, k_log, v_log, lens, scale, Hkv, dtype)
    caught = rc != 0 or not np.all(np.isfinite(out)) or np.max(np.abs(out - want)) > 1e-6
    assert caught, f"planted mistake '{name}' was not caught by the dense pin"


# ------------------------------------- q_len > 1: causal attention over the pages
def _causal_sdpa_reference(q, k_log, v_log, lens, scale, Hkv, dtype):
    """Dense fp64 SDPA with an explicit mask: query token j of sequence b (at
    position L_b - q_len + j) attends to keys t <= L_b - q_len + j."""
    B, q_len, Hq, D = q.shape
    G = Hq // Hkv
    out = np.zeros((B, q_len, Hq, D))
    for b, L in enumerate(lens):
        qt = _torch_widen(q[b], dtype).permute(1, 0, 2)                 # [Hq, q_len, D]
        kt = _torch_widen(k_log[b], dtype).permute(1, 0, 2).repeat_interleave(G, dim=0)
        vt = _torch_widen(v_log[b], dtype).permute(1, 0, 2).repeat_interleave(G, dim=0)
        pos = torch.arange(q_len)[:, None] + (L - q_len)
        mask = torch.arange(L)[None, :] <= pos                          # [q_len, L]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        out[b] = o.permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("dtype,q_len,Hq,Hkv,bs", [("f32", 4, 4, 4, 16), ("bf16", 2, 8, 2, 16),
                                                   ("bf16", 8, 2, 2, 32), ("f32", 3, 8, 4, 16)])
def test_multi_token_oracle_equals_causal_dense_sdpa(dtype, q_len, Hq, Hkv, bs):
    lens = [q_len, 19, 70]
    D = 64
    rng, k_log, v_log, _ = _random_logical(41 + q_len, lens, Hq, Hkv, D, dtype)
    q = pa_inputs.to_storage(rng.standard_normal((len(lens), q_len, Hq, D), dtype=np.float32), dtype)
    mb = max((L + bs - 1) // bs for L in lens)
    NB = sum((L + bs - 1) // bs for L in lens) + 2
    tables = _tables_from_perm(rng.permutation(NB).astype(np.int32), lens, bs, mb)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, lens, NB, bs, dtype)
    got = oracle.decode_multi_f64(q, kp, vp, tables, np.array(lens, np.int32), 0.125, Hkv, dtype)
    want = _causal_sdpa_reference(q, k_log, v_log, lens, 0.125, Hkv, dtype)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    rows = [(1, q_len - 1, Hq - 1), (2, 0, 0), (0, q_len - 1, 0)]
    sel = oracle.decode_multi_f64(q, kp, vp, tables, np.array(lens, np.int32), 0.125, Hkv, dtype,
                                  rows=rows)
    np.testing.assert_array_equal(sel, np.stack([got[b, j, i] for b, j, i in rows]))


def test_multi_token_with_one_token_is_decode():
    dtype, Hq, Hkv, D, bs = "bf16", 8, 2, 128, 16
    lens = [5, 40]
    rng, k_log, v_log, q = _random_logical(47, lens, Hq, Hkv, D, dtype)
    tables = _tables_from_perm(rng.permutation(6).astype(np.int32), lens, bs, 3)
    kp, vp = _scatter_into_pool(k_log, v_log, tables, lens, 6, bs, dtype)
    cl = np.array(lens, np.int32)
    multi = oracle.decode_multi_f64(q[:, None], kp, vp, tables, cl, 0.09, Hkv, dtype)
    np.testing.assert_array_equal(multi[:, 0], oracle.decode_f64(q, kp, vp, tables, cl, 0.09, Hkv, dtype))
