"""GPU parity of paged attention for q_len new tokens per sequence (causal among
them): the library (through its C ABI) against the CPU oracle, which computes
each new token as the decode of its sequence cut at that token."""
import numpy as np
import pytest
import torch

import oracle
import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import DEV, check_tolerance, out_as_f64, to_dev

pytestmark = pytest.mark.gpu


def _multi_case(name, seed, dtype, num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
                block_size, lens):
    """A decode case whose last q_len positions are the step's new tokens: the
    prefill draws fill positions 0 .. L-1 (all in the pool, as after the cache
    write of the step) and q holds q_len rows per sequence."""
    case = pa_inputs.make_decode_case(name, seed=seed, dtype=dtype, num_seqs=num_seqs,
                                      num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                                      head_dim=head_dim, block_size=block_size,
                                      lens=("list", [L + 1 for L in lens]))
    # drop the extra position the single-token case reserves for its new token
    case.context_lens = np.asarray(lens, np.int32)
    rng = np.random.default_rng(seed + 7)
    q = pa_inputs.to_storage(rng.standard_normal((num_seqs, q_len, num_q_heads, head_dim),
                                                 dtype=np.float32), dtype)
    return case, q


def _run(case, q, q_len, chunk_tokens=0):
    bf = case.dtype == "bf16"
    kc, vc = to_dev(case.k_cache, bf), to_dev(case.v_cache, bf)
    dq = to_dev(q, bf)
    out = torch.empty(dq.shape, dtype=dq.dtype, device=DEV)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_decode_multi(out, dq, kc, vc, to_dev(case.block_tables), to_dev(case.context_lens),
                       case.scale, case.num_kv_heads, int(case.context_lens.max()),
                       chunk_tokens=chunk_tokens, device_errors=errs)
    return out, pa.pa_read_device_errors(errs)


def _want(case, q):
    return oracle.decode_multi_f64(q, case.k_cache, case.v_cache, case.block_tables,
                                   case.context_lens, case.scale, case.num_kv_heads, case.dtype)


# (dtype, q_len, Hq, Hkv, D, bs): rows per item = q_len * group in {2, 4, 8}
VARIANTS = [("bf16", 2, 8, 8, 128, 16), ("bf16", 4, 8, 8, 128, 16), ("bf16", 8, 4, 4, 128, 32),
            ("bf16", 2, 8, 2, 128, 16), ("bf16", 2, 16, 4, 128, 16), ("bf16", 4, 4, 2, 64, 16),
            ("f32", 4, 4, 4, 64, 16), ("f32", 2, 8, 2, 128, 32), ("f32", 8, 2, 2, 64, 16)]


@pytest.mark.parametrize("dtype,q_len,Hq,Hkv,D,bs", VARIANTS)
@pytest.mark.parametrize("chunk", [0, 64])
def test_multi_token_matches_oracle(dtype, q_len, Hq, Hkv, D, bs, chunk):
    # lengths put the causal boundary at a chunk edge, just past one, inside a
    # short last chunk, and at L = q_len
    lens = [q_len, 64 + 1, 64 * 2 + q_len - 1, 300, 129]
    if chunk and chunk % bs:
        pytest.skip("chunk must be a multiple of the page")
    case, q = _multi_case(f"multi-{dtype}-{q_len}-{Hq}-{Hkv}", 900 + q_len + Hq + D + bs, dtype,
                          len(lens), q_len, Hq, Hkv, D, bs, lens)
    out, flags = _run(case, q, q_len, chunk)
    assert flags == 0
    got = out_as_f64(out)
    check_tolerance(got.reshape(-1, D), _want(case, q).reshape(-1, D), dtype, case.name)


def test_multi_token_with_one_token_equals_decode():
    case, q = _multi_case("multi-1", 950, "bf16", 4, 1, 32, 8, 128, 16, [17, 300, 1, 64])
    out, flags = _run(case, q, 1)
    assert flags == 0
    single = torch.empty((4, 32, 128), dtype=torch.bfloat16, device=DEV)
    pa.pa_decode(single, to_dev(q[:, 0], True), to_dev(case.k_cache, True),
                 to_dev(case.v_cache, True), to_dev(case.block_tables),
                 to_dev(case.context_lens), case.scale, 8, 300)
    assert torch.equal(out[:, 0].view(torch.int16), single.view(torch.int16))


def test_length_below_q_len_is_flagged_and_rows_without_keys_are_zero():
    case, q = _multi_case("multi-short", 951, "bf16", 2, 4, 4, 4, 128, 16, [2, 40])
    out, flags = _run(case, q, 4)
    assert flags & pa.PA_DEVERR_BAD_LENGTH
    got = out_as_f64(out)
    assert np.all(got[0, :2] == 0)                       # tokens at positions -2, -1
    want = _want(case, q)
    check_tolerance(got[:, 2:].reshape(-1, 128), want[:, 2:].reshape(-1, 128), "bf16", "short")
    check_tolerance(got[1].reshape(-1, 128), want[1].reshape(-1, 128), "bf16", "short")


def test_unsupported_row_counts_are_refused():
    case, q = _multi_case("multi-bad", 952, "bf16", 2, 4, 16, 4, 128, 16, [40, 40])
    with pytest.raises(pa.PaError) as e:
        _run(case, q, 4)                                  # 4 tokens x group 4 = 16 rows
    assert "unsupported" in str(e.value)
