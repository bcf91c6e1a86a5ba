"""Pins of the oracle's float8 e4m3 pieces (CPU only): code values against
hand-decoded patterns and torch's float8_e4m3fn; the encoder against torch's
cast inside the finite range, with ties to even and saturation past 448; and
fp8-pool decode against the already-pinned fp32 decode on the same values."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import pa_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "e4m3_values.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            rows.append((int(c, 16), float(v)))
    return rows


def _same(a, b):
    if math.isnan(b):
        return math.isnan(a)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def test_code_values_match_hand_decoded_patterns():
    rows = _golden()
    codes = np.array([c for c, _ in rows], dtype=np.uint8)
    widened = oracle.widen(codes, "fp8")                    # the C decoder
    for (c, want), got in zip(rows, widened):
        assert _same(got, want), hex(c)
        assert _same(oracle.e4m3_value(c), want), hex(c)    # the encoder's table


def test_all_codes_match_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.widen(codes, "fp8")
    for c in range(256):
        assert _same(got[c], want[c]), hex(c)


def test_encoder_matches_torch_cast_in_the_finite_range():
    rng = np.random.default_rng(8)
    finite = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (finite[:-1] + finite[1:]) / 2                    # exact ties
    x = np.concatenate([
        rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01,
        rng.uniform(-463.9, 463.9, 5000), mids, -mids, finite, -finite,
    ]).astype(np.float32)
    got = oracle.e4m3_encode(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, want)


def test_encoder_saturates_past_448():
    x = np.array([464.0, 480.0, 1e6, np.inf, -464.0, -np.inf, 447.99, np.nan], np.float32)
    got = oracle.e4m3_encode(x)
    np.testing.assert_array_equal(got, np.array([0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7E, 0x7F],
                                                np.uint8))


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    values = oracle.widen(codes, "fp8").astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(values), codes)


@pytest.mark.parametrize("G", [1, 4])
def test_fp8_pool_decode_equals_fp32_decode_of_the_same_values(G):
    """Codes times per-head scales (powers of two, so the products are exact in
    fp32) fed to the fp32 path must give the same result as the fp8 path."""
    rng = np.random.default_rng(12 + G)
    Hkv, D, bs, NB = 2, 64, 16, 12
    Hq = Hkv * G
    lens = np.array([1, 40, 100], np.int32)
    k8 = rng.integers(0, 256, size=(NB, Hkv, bs, D)).astype(np.uint8)
    v8 = rng.integers(0, 256, size=(NB, Hkv, bs, D)).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x38                           # no NaN codes
    v8[(v8 & 0x7F) == 0x7F] = 0x38
    ks = np.array([2.0 ** -6, 2.0 ** -3])
    vs = np.array([2.0 ** -4, 0.5])
    tables = np.array([rng.permutation(NB)[:7] for _ in range(3)], np.int32)
    q = pa_inputs.to_storage(rng.standard_normal((3, Hq, D)).astype(np.float32), "bf16")
    got = oracle.decode_kv8_f64(q, k8, v8, tables, lens, 0.125, ks, vs)
    kf = (oracle.widen(k8, "fp8") * ks.reshape(1, Hkv, 1, 1)).astype(np.float32)
    vf = (oracle.widen(v8, "fp8") * vs.reshape(1, Hkv, 1, 1)).astype(np.float32)
    qf = oracle.widen(q, "bf16").astype(np.float32)
    want = oracle.decode_f64(qf, kf, vf, tables, lens, 0.125, Hkv, "f32")
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    swapped = oracle.decode_kv8_f64(q, k8, v8, tables, lens, 0.125, ks[::-1].copy(), vs)
    assert np.max(np.abs(swapped - want)) > 1e-3            # the head's own scale is used
