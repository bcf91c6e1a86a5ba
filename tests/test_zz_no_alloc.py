"""The allocation-free decode entry point, for callers that cannot allocate
device memory (code inside a runtime that owns every device allocation, or a
decode loop that must not allocate between steps): through the C ABI it must
give the same output as pa_decode with a caller workspace, call after call,
and refuse problems bigger than its static scratch before enqueueing anything.

Kept in a file that runs last so a failure here cannot hide any other test.
"""
import numpy as np
import pytest
import torch

import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import DEV, DeviceCase, check_tolerance, out_as_f64

pytestmark = pytest.mark.gpu


def _noalloc(dc, out):
    c = dc.case
    pa.pa_decode_noalloc(out, dc.q, dc.k_cache, dc.v_cache, dc.tables, dc.lens, c.scale,
                         c.num_kv_heads, c.max_context_len, device_errors=dc.errs)


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    # several chunks per sequence, so the split partials and the merge use the scratch
    case = pa_inputs.scaled_workload("gqa_bf16", 16)
    dc = DeviceCase(case)
    want = out_as_f64(dc.step())                 # cache write + pa_decode with its own workspace
    for _ in range(2):
        out = torch.full(dc.q.shape, float("nan"), dtype=dc.tdt, device=DEV)
        _noalloc(dc, out)
        torch.cuda.synchronize()
        got = out_as_f64(out)
        check_tolerance(got, want, case.dtype, "pa_decode_noalloc vs pa_decode")
    assert dc.device_errors() == 0


def test_noalloc_after_a_different_problem():
    # the shared scratch keeps the previous call's contents; a call on another
    # shape must not be affected by them
    small = DeviceCase(pa_inputs.workload("tiny_fp32"))
    big = DeviceCase(pa_inputs.scaled_workload("mha_bf16", 4))
    want_small = out_as_f64(small.step())
    want_big = out_as_f64(big.step())
    for dc, want in ((big, want_big), (small, want_small), (big, want_big)):
        out = torch.empty(dc.q.shape, dtype=dc.tdt, device=DEV)
        _noalloc(dc, out)
        check_tolerance(out_as_f64(out), want, dc.case.dtype, dc.case.name)
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
