"""GPU parity of swapping pages to a pinned host pool and back: the library's
page copy (through its C ABI) against the oracle's byte copy, with the copy
pairs handed out by the library's block manager; and the decode of swapped
sequences after they come back, bit-identical to the decode before."""
import numpy as np
import pytest
import torch

import oracle
import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import DEV, DeviceCase, out_as_f64, storage_to_host, to_dev

pytestmark = pytest.mark.gpu


def _pinned(shape, dtype):
    return torch.zeros(shape, dtype=dtype).pin_memory()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_swap_out_and_in_are_byte_copies(dtype):
    rng = np.random.default_rng(31)
    NB, NH, Hkv, bs, D = 48, 40, 4, 16, 128
    if dtype == "fp8":
        kc = rng.integers(0, 256, size=(NB, Hkv, bs, D), dtype=np.uint8)
        vc = rng.integers(0, 256, size=(NB, Hkv, bs, D), dtype=np.uint8)
        tdt = torch.uint8
    else:
        kc = pa_inputs.to_storage(rng.standard_normal((NB, Hkv, bs, D), dtype=np.float32), "bf16")
        vc = pa_inputs.to_storage(rng.standard_normal((NB, Hkv, bs, D), dtype=np.float32), "bf16")
        tdt = torch.bfloat16
    bf = dtype == "bf16"
    dk, dv = to_dev(kc, bf), to_dev(vc, bf)
    hk, hv = _pinned((NH, Hkv, bs, D), tdt), _pinned((NH, Hkv, bs, D), tdt)
    ok_host_k, ok_host_v = np.zeros_like(kc[:NH]), np.zeros_like(vc[:NH])
    bm = pa.BlockManager(NB, bs, rng.permutation(NB))
    bm.enable_swap(NH, rng.permutation(NH))
    for s, L in enumerate([40, 17, 64, 1, 90]):
        bm.add_seq(s)
        for _ in range(L):
            bm.append_slot(s)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_pairs = np.concatenate([bm.swap_out(s) for s in (0, 2, 4)])
    pa.pa_swap_blocks(dk, dv, hk, hv, to_dev(out_pairs), device_errors=errs)
    oracle.copy_pages(kc, vc, ok_host_k, ok_host_v, out_pairs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(storage_to_host(hk, dtype), ok_host_k[:NH])
    np.testing.assert_array_equal(storage_to_host(hv, dtype), ok_host_v[:NH])
    # the freed device pages get other data, then the sequences come back
    dk.view(torch.uint8).fill_(0xEE)
    dv.view(torch.uint8).fill_(0xEE)
    kc2, vc2 = storage_to_host(dk, dtype), storage_to_host(dv, dtype)
    in_pairs = np.concatenate([bm.swap_in(s) for s in (4, 0, 2)])
    pa.pa_swap_blocks(hk, hv, dk, dv, to_dev(in_pairs), device_errors=errs)
    oracle.copy_pages(ok_host_k, ok_host_v, kc2, vc2, in_pairs)
    np.testing.assert_array_equal(storage_to_host(dk, dtype), kc2)
    np.testing.assert_array_equal(storage_to_host(dv, dtype), vc2)
    assert pa.pa_read_device_errors(errs) == 0


def test_decode_after_swap_round_trip_is_bit_identical():
    """Sequences swapped out, their pages reused and overwritten by others, and
    swapped back into different pages decode to the same bits."""
    case = pa_inputs.scaled_workload("gqa_bf16", 24)
    dc = DeviceCase(case)
    before = dc.step()                                   # writes the new tokens, decodes
    NB, Hkv, bs, D = case.k_cache.shape
    used = set()
    for b in range(case.num_seqs):
        used.update(int(p) for p in case.block_tables[b] if p >= 0)
    # every other sequence leaves for the host pool (pairs in table order)
    victims = list(range(0, case.num_seqs, 2))
    host_pages = sum(int((case.block_tables[b] >= 0).sum()) for b in victims)
    hk = _pinned((host_pages, Hkv, bs, D), torch.bfloat16)
    hv = _pinned((host_pages, Hkv, bs, D), torch.bfloat16)
    out_pairs, h = [], 0
    for b in victims:
        for p in case.block_tables[b]:
            if p >= 0:
                out_pairs.append((int(p), h))
                h += 1
    out_pairs = np.array(out_pairs, np.int64)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_swap_blocks(dc.k_cache, dc.v_cache, hk, hv, to_dev(out_pairs), device_errors=errs)
    # overwrite every page the victims held with NaN, then bring them back into
    # the pages no table uses (and the victims' own, permuted)
    freed = out_pairs[:, 0]
    dc.k_cache[torch.from_numpy(freed).to(DEV)] = float("nan")
    dc.v_cache[torch.from_numpy(freed).to(DEV)] = float("nan")
    spare = np.array(sorted(set(range(NB)) - (used - set(freed.tolist()))), np.int64)
    dest = np.random.default_rng(5).permutation(spare)[:host_pages]
    in_pairs = np.stack([out_pairs[:, 1], dest], axis=1)
    pa.pa_swap_blocks(hk, hv, dc.k_cache, dc.v_cache, to_dev(in_pairs), device_errors=errs)
    tables = case.block_tables.copy()
    h = 0
    for b in victims:
        for j, p in enumerate(tables[b]):
            if p >= 0:
                tables[b, j] = dest[h]
                h += 1
    dc.tables = to_dev(tables)
    after = dc.step(write=False)
    assert pa.pa_read_device_errors(errs) == 0
    assert dc.device_errors() == 0
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))
    assert np.all(np.isfinite(out_as_f64(after)))


def test_swap_out_of_pool_pair_is_flagged_and_skipped():
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device=DEV)
    hk = _pinned((2, 2, 16, 64), torch.bfloat16)
    pairs = torch.tensor([[1, 5], [7, 0], [2, 1]], dtype=torch.int64, device=DEV)
    kc[2] = 3.0
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_swap_blocks(kc, kc, hk, hk, pairs, device_errors=errs)
    assert pa.pa_read_device_errors(errs) == pa.PA_DEVERR_BAD_BLOCK
    assert bool((hk[1].float() == 3.0).all()) and bool((hk[0].float() == 0.0).all())
