"""GPU parity of the float8 e4m3 pools: the library (through its C ABI) against
the CPU oracle on the same seeded inputs.

Bars: the fp8 cache write bit-exact (the same e4m3 codes as the oracle's
nearest-even encoder with saturation); decode with e4m3 pools and bf16 q/out
max |err| <= 2e-2 and mean |err| <= 2e-3 against the fp64 oracle that
dequantises each code exactly (code * scale of its kv head).
"""
import numpy as np
import pytest
import torch

import oracle
import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import (DEV, DeviceCase, check_tolerance, oracle_step, out_as_f64,
                         storage_to_host, to_dev)

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    return pa_inputs.to_storage(np.asarray(x, dtype=np.float32), "bf16")


def _hard_values(rng, n):
    """bf16 values that exercise every branch of the encoder at scale 1: exact
    codes, midpoints between neighbouring codes (ties), the subnormal range,
    signed zeros, the saturation region and infinities."""
    codes = np.arange(0x7F)
    vals = np.array([oracle.e4m3_value(int(c)) for c in codes])
    mids = (vals[:-1] + vals[1:]) / 2                    # exact ties (bf16 holds them)
    special = np.array([0.0, -0.0, 448.0, 449.0, 464.0, 465.0, 1e4, np.inf, -np.inf,
                        2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 2.0 ** -12])
    pool = np.concatenate([vals, -vals, mids, -mids, special, -special])
    return rng.choice(pool, size=n)


@pytest.mark.parametrize("bs", [16, 32])
def test_reshape_and_cache_fp8_bit_exact(bs):
    rng = np.random.default_rng(15)
    NB, Hkv, D, T = 23, 4, 128, 40
    x = rng.standard_normal((2, T, Hkv, D)).astype(np.float32) * 3.0
    x[0, :8] = _hard_values(rng, 8 * Hkv * D).reshape(8, Hkv, D)
    x[1, :8] = _hard_values(rng, 8 * Hkv * D).reshape(8, Hkv, D)
    k, v = _bf16_bits(x[0]), _bf16_bits(x[1])
    ks = np.array([1.0, 0.0173, 0.5, 3.25], dtype=np.float32)      # head 0: unscaled
    vs = np.array([1.0, 0.021, 0.75, 2.0], dtype=np.float32)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[5::9] = -1                                                 # padding tokens
    kc = pa_inputs.nan_fill((NB, Hkv, bs, D), "fp8")
    vc = pa_inputs.nan_fill((NB, Hkv, bs, D), "fp8")
    dkc, dvc = to_dev(kc), to_dev(vc)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_reshape_and_cache_fp8(to_dev(k, True), to_dev(v, True), dkc, dvc, to_dev(slots),
                                to_dev(ks), to_dev(vs), device_errors=errs)
    oracle.reshape_and_cache_fp8(k, v, kc, vc, slots, ks, vs)
    np.testing.assert_array_equal(storage_to_host(dkc, "fp8"), kc)
    np.testing.assert_array_equal(storage_to_host(dvc, "fp8"), vc)
    assert pa.pa_read_device_errors(errs) == 0


def test_reshape_fp8_out_of_pool_slot_is_flagged_and_skipped():
    NB, Hkv, bs, D = 4, 2, 16, 128
    kc = torch.zeros((NB, Hkv, bs, D), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, Hkv, D), dtype=torch.bfloat16, device=DEV)
    sc = torch.ones(Hkv, dtype=torch.float32, device=DEV)
    slots = torch.tensor([NB * bs, 3], dtype=torch.int64, device=DEV)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_reshape_and_cache_fp8(k, k, kc, vc, slots, sc, sc, device_errors=errs)
    assert pa.pa_read_device_errors(errs) == pa.PA_DEVERR_BAD_SLOT
    # only slot 3 was written: 1.0 is code 0x38
    assert int((kc != 0).sum()) == Hkv * D
    assert bool((kc[0, :, 3] == 0x38).all())


# ----------------------------------------------------- decode: the workloads
SCALED = [("mha_fp8", 6, {}), ("gqa_fp8", 24, {}),
          ("long128k_fp8", 1, dict(lens=("fixed", 20000)))]


@pytest.mark.parametrize("name,B,over", SCALED)
def test_decode_fp8_workloads_at_oracle_size(name, B, over):
    case = pa_inputs.scaled_workload(name, B, **over)
    dc = DeviceCase(case)
    got = out_as_f64(dc.step())
    assert dc.device_errors() == 0
    check_tolerance(got, oracle_step(case), case.dtype, case.name)


@pytest.mark.parametrize("name", ["mha_fp8", "gqa_fp8", "long128k_fp8"])
def test_decode_fp8_full_size_every_row(name):
    """Full-size fp8 workload in the bench's launch configuration, every output
    row against the oracle (the mean-error bar on the whole output)."""
    case = pa_inputs.workload(name)
    dc = DeviceCase(case)
    got = out_as_f64(dc.step())
    assert dc.device_errors() == 0
    want = oracle_step(case)
    assert got.shape == want.shape
    check_tolerance(got, want, case.dtype, case.name)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_decode_fp8_every_group(G, bs):
    Hkv = 2
    case = pa_inputs.make_decode_case(
        f"fp8-{G}-{bs}", seed=500 + G + bs, dtype="fp8", num_seqs=5, num_q_heads=Hkv * G,
        num_kv_heads=Hkv, head_dim=128, block_size=bs, lens=("list", [1, 15, 16, 17, 700]))
    dc = DeviceCase(case)
    got = out_as_f64(dc.step(chunk_tokens=64 if bs == 16 else 128))
    assert dc.device_errors() == 0
    check_tolerance(got, oracle_step(case), "fp8", case.name)


@pytest.mark.parametrize("Hkv,G", [(3, 2), (6, 1), (4, 4)])
def test_decode_fp8_head_pairs_and_odd_head_counts(Hkv, G):
    """16-token pages: an even number of kv heads runs items over head pairs
    (one 32-row copy per page and pool, each row masked to its own head, each
    head with its own scales); an odd number runs single-head items."""
    case = pa_inputs.make_decode_case(
        f"fp8-pairs-{Hkv}-{G}", seed=540 + Hkv + G, dtype="fp8", num_seqs=4,
        num_q_heads=Hkv * G, num_kv_heads=Hkv, head_dim=128, block_size=16,
        lens=("list", [2, 31, 48, 333]))
    dc = DeviceCase(case)
    got = out_as_f64(dc.step(chunk_tokens=64))
    assert dc.device_errors() == 0
    check_tolerance(got, oracle_step(case), "fp8", case.name)


def test_decode_fp8_split_sizes_agree():
    case = pa_inputs.make_decode_case("fp8-split", seed=51, dtype="fp8", num_seqs=3,
                                      num_q_heads=8, num_kv_heads=2, head_dim=128,
                                      block_size=16, lens=("list", [512, 300, 77]))
    want = oracle_step(case)
    for chunk in (512, 128, 64, 16):
        dc = DeviceCase(case)
        got = out_as_f64(dc.step(chunk_tokens=chunk))
        assert dc.device_errors() == 0
        check_tolerance(got, want, "fp8", f"chunk {chunk}")


def test_decode_fp8_large_scores():
    """Wide logits (std 4 inputs): the softmax is nearly one-hot, so an error in
    the score scale or in which token a score belongs to shows at once."""
    case = pa_inputs.make_decode_case("fp8-wide", seed=52, dtype="fp8", num_seqs=4,
                                      num_q_heads=16, num_kv_heads=4, head_dim=128,
                                      block_size=16, lens=("list", [33, 250, 1000, 2]),
                                      std=4.0)
    dc = DeviceCase(case)
    got = out_as_f64(dc.step())
    assert dc.device_errors() == 0
    want = oracle_step(case)
    # outputs scale with the value std (4): the bars scale with it
    err = np.abs(got - want)
    assert err.max() <= 4 * 2e-2 and err.mean() <= 4 * 2e-3, (err.max(), err.mean())


def test_decode_fp8_zero_length_rows_are_zero():
    case = pa_inputs.make_decode_case("fp8-zero", seed=53, dtype="fp8", num_seqs=3,
                                      num_q_heads=8, num_kv_heads=8, head_dim=128,
                                      block_size=16, lens=("list", [0, 40, 0]))
    dc = DeviceCase(case)
    out = out_as_f64(dc.step())
    assert dc.device_errors() == 0
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    check_tolerance(out, oracle_step(case), "fp8", "fp8 zero-length")


def test_decode_fp8_is_deterministic():
    case = pa_inputs.scaled_workload("gqa_fp8", 32)
    dc = DeviceCase(case)
    a = dc.step()
    b = dc.step(write=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decode_fp8_bad_block_id_is_flagged():
    case = pa_inputs.make_decode_case("fp8-badblock", seed=54, dtype="fp8", num_seqs=2,
                                      num_q_heads=8, num_kv_heads=2, head_dim=128,
                                      block_size=16, lens=("list", [40, 40]))
    case.block_tables[1, 1] = case.num_blocks + 5
    dc = DeviceCase(case)
    dc.step()
    assert dc.device_errors() & pa.PA_DEVERR_BAD_BLOCK


def test_decode_fp8_rejects_other_head_dims():
    q = torch.zeros((1, 2, 64), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((2, 2, 16, 64), dtype=torch.uint8, device=DEV)
    sc = torch.ones(2, dtype=torch.float32, device=DEV)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    cl = torch.ones(1, dtype=torch.int32, device=DEV)
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_fp8(torch.empty_like(q), q, kc, kc, bt, cl, 0.125, sc, sc, 2, 1)
    assert "unsupported" in str(e.value)
