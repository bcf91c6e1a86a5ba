"""Failure path of the decode kernel, without a GPU fault: every pipeline wait is
bounded, and when one expires the kernel reports PA_DEVERR_TIMEOUT through the
device error word, waits for its own copies in flight and returns.  The test
hook pa_debug_set_wait_limit shortens the bound so that waits expire; the next
call with the normal bound must be correct again (the context stays usable)."""
import numpy as np
import pytest
import torch

import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import DeviceCase, check_tolerance, oracle_step, out_as_f64

pytestmark = pytest.mark.gpu

CASES = [
    ("gqa_bf16", dict(B=12)),          # tensor-core consumer, tensor-map copies
    ("tiny_fp32", dict()),             # CUDA-core consumer, bulk copies
    ("gqa_fp8", dict(B=12)),           # e4m3 pools: f16 tensor-core consumer
]


def _case(name, B=None):
    return pa_inputs.workload(name) if B is None else pa_inputs.scaled_workload(name, B)


@pytest.mark.parametrize("name,kw", CASES)
def test_expired_waits_report_timeout_and_leave_the_context_usable(name, kw):
    case = _case(name, kw.get("B"))
    dc = DeviceCase(case)
    try:
        pa.pa_debug_set_wait_limit(0)          # every wait gives up at once
        dc.step()
        flags = dc.device_errors()             # synchronises: the kernel returned
    finally:
        pa.pa_debug_set_wait_limit(-1)
    assert flags & pa.PA_DEVERR_TIMEOUT
    assert flags & ~pa.PA_DEVERR_TIMEOUT == 0
    got = out_as_f64(dc.step(write=False))     # normal bound again
    assert dc.device_errors() == 0
    check_tolerance(got, oracle_step(case), case.dtype, case.name)


@pytest.mark.parametrize("name,kw", CASES)
def test_waits_expiring_mid_pipeline_drain_their_copies(name, kw):
    """With a short bound the pipeline gets partway (copies in flight) before a
    wait expires; the kernel must still return and the next call be exact."""
    case = _case(name, kw.get("B"))
    dc = DeviceCase(case)
    try:
        pa.pa_debug_set_wait_limit(64)
        for _ in range(3):
            dc.step(write=False)
        flags = dc.device_errors()
    finally:
        pa.pa_debug_set_wait_limit(-1)
    assert flags & ~pa.PA_DEVERR_TIMEOUT == 0
    got = out_as_f64(dc.step())
    assert dc.device_errors() == 0
    check_tolerance(got, oracle_step(case), case.dtype, case.name)
