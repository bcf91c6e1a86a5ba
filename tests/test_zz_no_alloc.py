"""The allocation-free decode entry point, for callers that cannot allocate
device memory (code inside a runtime that owns every device allocation, or a
decode loop that must not allocate between steps).  Through the C ABI it must
match the oracle within the decode tolerance and give bit for bit the output of
pa_decode with a caller workspace, call after call; it must not allocate on the
device once set up; and it must refuse problems bigger than its static scratch
before enqueueing anything.

Kept in a file that runs last so a failure here cannot hide any other test.
"""
import numpy as np
import pytest
import torch

import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import DEV, DeviceCase, check_tolerance, oracle_step, out_as_f64

pytestmark = pytest.mark.gpu


def _noalloc(dc, out):
    c = dc.case
    pa.pa_decode_noalloc(out, dc.q, dc.k_cache, dc.v_cache, dc.tables, dc.lens, c.scale,
                         c.num_kv_heads, c.max_context_len, device_errors=dc.errs)


CASES = [
    # several chunks per sequence of the GQA workload's length mix
    ("gqa_bf16", 16, {}),
    # the long-context workload cut to 20 000 tokens: a dozen chunks per
    # sequence and a ragged tail, so the split partials and the merge use the scratch
    ("long128k_bf16", 2, dict(lens=("fixed", 20000))),
]


@pytest.mark.parametrize("name,B,over", CASES)
def test_noalloc_matches_oracle_and_pa_decode_on_two_calls_in_a_row(name, B, over):
    case = pa_inputs.scaled_workload(name, B, **over)
    dc = DeviceCase(case)
    ref = dc.step()                          # cache write + pa_decode with its own workspace
    want = oracle_step(case)
    outs = [torch.full(dc.q.shape, float("nan"), dtype=dc.tdt, device=DEV) for _ in range(3)]
    _noalloc(dc, outs[0])                    # set-up call (looks the scratch address up)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    alloc_before = torch.cuda.memory_allocated()
    for out in outs[1:]:                     # two more calls in a row
        _noalloc(dc, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed across calls"
    assert torch.cuda.memory_allocated() == alloc_before
    assert dc.device_errors() == 0
    for k, out in enumerate(outs):
        check_tolerance(out_as_f64(out), want, case.dtype, f"{case.name} call {k}")
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"{case.name} call {k}: differs from pa_decode"


def test_noalloc_after_a_different_problem():
    # the shared scratch keeps the previous call's contents; a call on another
    # shape must not be affected by them
    small = DeviceCase(pa_inputs.workload("tiny_fp32"))
    big = DeviceCase(pa_inputs.scaled_workload("mha_bf16", 4))
    ref_small, ref_big = small.step(), big.step()
    want_small, want_big = oracle_step(small.case), oracle_step(big.case)
    for dc, ref, want in ((big, ref_big, want_big), (small, ref_small, want_small),
                          (big, ref_big, want_big)):
        out = torch.empty(dc.q.shape, dtype=dc.tdt, device=DEV)
        _noalloc(dc, out)
        check_tolerance(out_as_f64(out), want, dc.case.dtype, dc.case.name)
        assert torch.equal(out, ref)
    assert small.device_errors() == 0 and big.device_errors() == 0


def test_noalloc_refuses_problems_larger_than_its_scratch():
    B, Hq, Hkv, D, bs, L = 4096, 32, 8, 128, 32, 131072
    need = pa.pa_decode_workspace_size(B, Hq, Hkv, D, bs, L)
    assert need > pa.PA_NOALLOC_SCRATCH_BYTES
    t = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    rc = pa.library().pa_decode_noalloc(
        t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(),
        1.0, Hkv, B, Hq, D, bs, 10, L // bs, L, pa.PA_BF16, 0, None, None)
    assert rc == -7            # PA_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
