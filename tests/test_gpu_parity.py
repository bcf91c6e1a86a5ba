"""GPU parity: the library (through its C ABI) against the CPU oracle on the same
seeded inputs.

Bars: cache write, page copy and block management bit-exact; decode with fp32
inputs max |err| <= 1e-4; decode with bf16 inputs max |err| <= 2e-2 and mean
|err| <= 2e-3 (fp32 accumulation; the bf16 output rounding, <= 2^-9 relative,
is inside the bar).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import (DEV, DeviceCase, check_tolerance, oracle_step, out_as_f64,
                         storage_to_host, to_dev)

pytestmark = pytest.mark.gpu


def _bits(a):
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


# ------------------------------------------------------------------ cache write
@pytest.mark.parametrize("dtype,D,bs", [("bf16", 128, 16), ("bf16", 64, 32), ("f32", 64, 16),
                                        ("f32", 128, 32)])
def test_reshape_and_cache_bit_exact(dtype, D, bs):
    rng = np.random.default_rng(5)
    NB, Hkv, T = 37, 4, 50
    kc = pa_inputs.nan_fill((NB, Hkv, bs, D), dtype)
    vc = pa_inputs.nan_fill((NB, Hkv, bs, D), dtype)
    k = pa_inputs.to_storage(rng.standard_normal((T, Hkv, D), dtype=np.float32), dtype)
    v = pa_inputs.to_storage(rng.standard_normal((T, Hkv, D), dtype=np.float32), dtype)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[::7] = -1                                    # padding tokens
    bf = dtype == "bf16"
    dkc, dvc = to_dev(kc, bf), to_dev(vc, bf)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_reshape_and_cache(to_dev(k, bf), to_dev(v, bf), dkc, dvc, to_dev(slots),
                            device_errors=errs)
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    np.testing.assert_array_equal(_bits(storage_to_host(dkc, dtype)), _bits(kc))
    np.testing.assert_array_equal(_bits(storage_to_host(dvc, dtype)), _bits(vc))
    assert pa.pa_read_device_errors(errs) == 0


def test_reshape_out_of_pool_slot_is_flagged_and_skipped():
    NB, Hkv, bs, D = 4, 2, 16, 64
    kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, Hkv, D), dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([NB * bs, 3], dtype=torch.int64, device=DEV)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_reshape_and_cache(k, k, kc, vc, slots, device_errors=errs)
    assert pa.pa_read_device_errors(errs) == pa.PA_DEVERR_BAD_SLOT
    assert float(kc.float().sum()) == Hkv * D                # only slot 3 was written


# -------------------------------------------------------------------- page copy
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_copy_blocks_bit_exact(dtype):
    rng = np.random.default_rng(6)
    NB, Hkv, bs, D = 50, 8, 16, 128
    kc = pa_inputs.to_storage(rng.standard_normal((NB, Hkv, bs, D), dtype=np.float32), dtype)
    vc = pa_inputs.to_storage(rng.standard_normal((NB, Hkv, bs, D), dtype=np.float32), dtype)
    ids = rng.permutation(NB)
    pairs = np.stack([ids[:12], ids[12:24]], axis=1).astype(np.int64)
    bf = dtype == "bf16"
    dkc, dvc = to_dev(kc, bf), to_dev(vc, bf)
    pa.pa_copy_blocks(dkc, dvc, to_dev(pairs))
    oracle.copy_blocks(kc, vc, pairs)
    np.testing.assert_array_equal(_bits(storage_to_host(dkc, dtype)), _bits(kc))
    np.testing.assert_array_equal(_bits(storage_to_host(dvc, dtype)), _bits(vc))


def test_copy_blocks_out_of_pool_pair_is_flagged():
    kc = torch.zeros((4, 1, 16, 64), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_copy_blocks(kc, vc, torch.tensor([[0, 4]], dtype=torch.int64, device=DEV),
                      device_errors=errs)
    assert pa.pa_read_device_errors(errs) == pa.PA_DEVERR_BAD_BLOCK


# ----------------------------------------------------- decode: the workloads
SCALED = [("tiny_fp32", 4), ("mha_bf16", 6), ("gqa_bf16", 24), ("long128k_bf16", 1)]


@pytest.mark.parametrize("name,B", SCALED)
def test_decode_workloads_at_oracle_size(name, B):
    over = {}
    if name == "long128k_bf16":
        over = dict(lens=("fixed", 20000))              # several chunks and a ragged tail
    case = pa_inputs.workload(name) if name == "tiny_fp32" else pa_inputs.scaled_workload(name, B, **over)
    dc = DeviceCase(case)
    got = out_as_f64(dc.step())
    assert dc.device_errors() == 0
    want = oracle_step(case)
    check_tolerance(got, want, case.dtype, case.name)


@pytest.mark.parametrize("name", ["mha_bf16", "gqa_bf16", "long128k_bf16"])
def test_decode_full_size_every_row(name):
    """Full-size workload in the bench's launch configuration (automatic split:
    the chunk the library picks for 152 SMs, up to 256 chunks per sequence of
    the long-context workload), every output row against the oracle, so the
    mean-error bar is judged on the whole output."""
    case = pa_inputs.workload(name)
    dc = DeviceCase(case)
    out = dc.step()
    assert dc.device_errors() == 0
    got = out_as_f64(out)
    want = oracle_step(case)
    assert got.shape == want.shape
    check_tolerance(got, want, case.dtype, case.name)


def _shared_prefix_step_parity(script, cascade):
    dtype, bs = script.dtype, script.block_size
    Hkv, D = script.num_kv_heads, script.head_dim
    results = []
    for side in ("library", "oracle"):
        bm = (pa.BlockManager if side == "library" else oracle.RefBlockManager)(
            script.num_blocks, bs, script.initial_free_order)
        prefix_slots = pa_inputs.shared_prefix_prefill(bm, script)
        _, children = pa_inputs.shared_prefix_ids(script)
        kc = pa_inputs.nan_fill((script.num_blocks, Hkv, bs, D), dtype)
        vc = pa_inputs.nan_fill((script.num_blocks, Hkv, bs, D), dtype)
        for p, slots in enumerate(prefix_slots):
            pa_inputs.place_at_slots(kc, slots, script.prefix_k[p], bs)
            pa_inputs.place_at_slots(vc, slots, script.prefix_v[p], bs)
        if side == "library":
            slots, pairs = bm.append_slots(children)
            mb = max(len(bm.block_table(c)[0]) for c in children)
            tables, lens = bm.build_block_tables(children, mb)
        else:
            res = [bm.append_slot(c) for c in children]
            slots = np.array([r[0] for r in res], np.int64)
            pairs = np.array([(r[1], r[2]) for r in res if r[1] >= 0], np.int64).reshape(-1, 2)
            mb = max(len(bm.block_table(c)[0]) for c in children)
            tables = np.full((len(children), mb), -1, np.int32)
            lens = np.zeros(len(children), np.int32)
            for j, c in enumerate(children):
                t, L = bm.block_table(c)
                tables[j, :len(t)] = t
                lens[j] = L
        results.append((slots, pairs, tables, lens, kc, vc))
    (s_l, p_l, t_l, l_l, kc, vc), (s_o, p_o, t_o, l_o, kc_o, vc_o) = results
    np.testing.assert_array_equal(s_l, s_o)
    np.testing.assert_array_equal(p_l, p_o)
    np.testing.assert_array_equal(t_l, t_o)
    np.testing.assert_array_equal(l_l, l_o)
    assert len(p_l) == script.num_parents * (script.children_per_parent - 1)
    # library side on the GPU
    bf = dtype == "bf16"
    dkc, dvc = to_dev(kc, bf), to_dev(vc, bf)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_copy_blocks(dkc, dvc, to_dev(p_l), device_errors=errs)
    pa.pa_reshape_and_cache(to_dev(script.k_new, bf), to_dev(script.v_new, bf), dkc, dvc,
                            to_dev(s_l), device_errors=errs)
    q = to_dev(script.q, bf)
    out = torch.empty_like(q)
    pa.pa_decode(out, q, dkc, dvc, to_dev(t_l), to_dev(l_l), script.scale, Hkv, int(l_l.max()),
                 device_errors=errs)
    outs = {"pa_decode": out}
    if cascade:
        starts, shared = pa.pa_cascade_groups(t_l, l_l, bs)
        C = script.children_per_parent
        assert list(starts) == list(range(0, len(l_l) + 1, C))      # one group per family
        assert list(shared) == [int(n) // bs * bs for n in script.prefix_lens]
        outs["pa_decode_cascade"] = torch.full_like(q, float("nan"))
        pa.pa_decode_cascade(outs["pa_decode_cascade"], q, dkc, dvc, to_dev(t_l), to_dev(l_l),
                             to_dev(starts), to_dev(shared), script.scale, Hkv, int(l_l.max()),
                             device_errors=errs)
    assert pa.pa_read_device_errors(errs) == 0
    # oracle side on the CPU
    oracle.copy_blocks(kc_o, vc_o, p_o)
    oracle.reshape_and_cache(script.k_new, script.v_new, kc_o, vc_o, s_o)
    want = oracle.decode_f64(script.q, kc_o, vc_o, t_o, l_o, script.scale, Hkv, dtype)
    for what, o in outs.items():
        check_tolerance(out_as_f64(o), want, dtype, f"shared prefix, {what}")
    # the caches themselves agree byte for byte after the copies and the write
    np.testing.assert_array_equal(storage_to_host(dkc, dtype), kc_o)
    np.testing.assert_array_equal(storage_to_host(dvc, dtype), vc_o)


def test_decode_shared_prefix_workload():
    """The shared-prefix step at a reduced size: copy-on-write of each family's
    partial page, the new tokens' write, then decode -- tables and copies from
    the library's block manager, checked against the oracle running its own
    block manager."""
    _shared_prefix_step_parity(
        pa_inputs.shared_prefix_script(scale_parents=2, scale_children=6, prompt_len=300), False)


def test_decode_shared_prefix_workload_full_size():
    """The shared-prefix step at its stated size -- 8 parents of 2048 + g_p
    tokens, 16 children each -- in the bench's order (copies, write, decode),
    every row of both pa_decode and pa_decode_cascade against the oracle, and
    the pools byte for byte against the oracle's copies and write."""
    _shared_prefix_step_parity(pa_inputs.shared_prefix_script(), True)


# ------------------------------------------------------ decode: every variant
VARIANTS = [(dt, D, G, bs) for dt in ("bf16", "f32") for D in (64, 128) for G in (1, 2, 4, 8)
            for bs in (16, 32)]


@pytest.mark.parametrize("dtype,D,G,bs", VARIANTS)
def test_decode_every_instantiation(dtype, D, G, bs):
    Hkv = 2
    case = pa_inputs.make_decode_case(
        f"v-{dtype}-{D}-{G}-{bs}", seed=300 + D + G + bs, dtype=dtype, num_seqs=5,
        num_q_heads=Hkv * G, num_kv_heads=Hkv, head_dim=D, block_size=bs,
        lens=("list", [1, 15, 16, 17, 700]))
    dc = DeviceCase(case)
    got = out_as_f64(dc.step(chunk_tokens=64 if bs == 16 else 128))
    assert dc.device_errors() == 0
    check_tolerance(got, oracle_step(case), dtype, case.name)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_sizes_agree(dtype):
    """One chunk per sequence vs several chunks merged by log-sum-exp."""
    case = pa_inputs.make_decode_case("split", seed=41, dtype=dtype, num_seqs=3, num_q_heads=8,
                                      num_kv_heads=2, head_dim=128, block_size=16,
                                      lens=("list", [512, 300, 77]))
    outs = {}
    for chunk in (512, 128, 64, 16):
        dc = DeviceCase(case)
        outs[chunk] = out_as_f64(dc.step(chunk_tokens=chunk))
        assert dc.device_errors() == 0
    want = oracle_step(case)
    for chunk, got in outs.items():
        check_tolerance(got, want, dtype, f"chunk {chunk}")
    if dtype == "f32":
        for chunk in (128, 64, 16):
            assert np.max(np.abs(outs[chunk] - outs[512])) <= 1e-5


def test_single_token_context_returns_v_bits():
    case = pa_inputs.make_decode_case("one", seed=42, dtype="bf16", num_seqs=4, num_q_heads=32,
                                      num_kv_heads=8, head_dim=128, block_size=16,
                                      lens=("fixed", 1), std=20.0)
    dc = DeviceCase(case)
    out = dc.step()
    got = storage_to_host(out, "bf16")
    for b in range(case.num_seqs):
        for i in range(case.num_q_heads):
            np.testing.assert_array_equal(got[b, i], case.v_new[b, i // 4])


def test_zero_length_rows_are_zero():
    case = pa_inputs.make_decode_case("zero", seed=43, dtype="bf16", num_seqs=3, num_q_heads=8,
                                      num_kv_heads=8, head_dim=64, block_size=16,
                                      lens=("list", [0, 40, 0]))
    dc = DeviceCase(case)
    out = out_as_f64(dc.step())
    assert dc.device_errors() == 0
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    check_tolerance(out, oracle_step(case), "bf16", "zero-length")


def test_no_work_listed_leaves_zero_rows():
    """Every length zero but a positive length bound: the plan lists no work
    and zeroes every row, and the decode kernel leaves at once."""
    case = pa_inputs.make_decode_case("nowork", seed=46, dtype="bf16", num_seqs=3, num_q_heads=8,
                                      num_kv_heads=8, head_dim=64, block_size=16,
                                      lens=("list", [40, 40, 40]))
    dc = DeviceCase(case)
    lens = torch.zeros_like(dc.lens)
    out = torch.full(dc.q.shape, float("nan"), dtype=dc.tdt, device=DEV)
    pa.pa_decode(out, dc.q, dc.k_cache, dc.v_cache, dc.tables, lens, case.scale,
                 case.num_kv_heads, case.max_context_len, device_errors=dc.errs)
    torch.cuda.synchronize()
    assert dc.device_errors() == 0
    assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("num_seqs", [300, 600, 1500])
def test_plan_block_sizes(num_seqs):
    """The plan runs with the smallest block (128, 256, 512 or 1024 threads)
    that takes the batch, 1024 at a time past that: batches in each range,
    short lengths (several chunks for some), a few empty sequences."""
    rng = np.random.default_rng(500 + num_seqs)
    lens = [int(x) for x in rng.integers(0, 160, size=num_seqs)]
    case = pa_inputs.make_decode_case(f"plan-{num_seqs}", seed=500 + num_seqs, dtype="bf16",
                                      num_seqs=num_seqs, num_q_heads=8, num_kv_heads=2,
                                      head_dim=64, block_size=16, lens=("list", lens))
    dc = DeviceCase(case)
    got = out_as_f64(dc.step(chunk_tokens=64))
    assert dc.device_errors() == 0
    check_tolerance(got, oracle_step(case), "bf16", case.name)


def test_decode_is_deterministic():
    case = pa_inputs.scaled_workload("gqa_bf16", 32)
    dc = DeviceCase(case)
    a = dc.step()
    b = dc.step(write=False)
    c = dc.step(write=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_bad_block_id_is_flagged_not_read():
    case = pa_inputs.make_decode_case("badblock", seed=44, dtype="bf16", num_seqs=2,
                                      num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                      lens=("list", [40, 40]))
    case.block_tables[1, 1] = case.num_blocks + 5
    dc = DeviceCase(case)
    dc.step()
    assert dc.device_errors() & pa.PA_DEVERR_BAD_BLOCK


def test_length_beyond_bound_is_flagged_and_clamped():
    case = pa_inputs.make_decode_case("badlen", seed=45, dtype="bf16", num_seqs=2,
                                      num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                      lens=("list", [64, 64]))
    dc = DeviceCase(case)
    dc.lens[1] = 100                                    # beyond max_context_len = 64
    dc.step()
    assert dc.device_errors() & pa.PA_DEVERR_BAD_LENGTH
