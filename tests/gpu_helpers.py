"""Shared plumbing of the GPU tests: numpy <-> torch transfers and the two sides
of a decode step (the library through its C ABI; the oracle on the CPU)."""
import numpy as np
import torch

import oracle
import paged_kv_cache_190_gb300 as pa

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def to_dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if bf16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(DEV)


def storage_to_host(t, dtype):
    """Device tensor -> numpy storage form (float32, bf16 bits as uint16, or
    e4m3 codes as uint8)."""
    t = t.detach().cpu().contiguous()
    if dtype == "fp8":
        return t.view(torch.uint8).numpy()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def out_as_f64(t):
    return t.detach().float().cpu().double().numpy()


class DeviceCase:
    """A pa_inputs.DecodeCase moved to the device."""

    def __init__(self, case):
        self.case = case
        self.fp8 = case.dtype == "fp8"           # e4m3 pools, bf16 q / new token / out
        bf = case.dtype in ("bf16", "fp8")
        self.bf16 = bf
        self.tdt = torch.bfloat16 if bf else torch.float32
        self.k_cache = to_dev(case.k_cache, bf and not self.fp8)
        self.v_cache = to_dev(case.v_cache, bf and not self.fp8)
        self.k_new = to_dev(case.k_new, bf)
        self.v_new = to_dev(case.v_new, bf)
        self.q = to_dev(case.q, bf)
        if self.fp8:
            self.k_scale = to_dev(case.extra["k_scale"])
            self.v_scale = to_dev(case.extra["v_scale"])
        self.slots = to_dev(case.slot_mapping)
        self.tables = to_dev(case.block_tables)
        self.lens = to_dev(case.context_lens)
        self.errs = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step(self, chunk_tokens=0, write=True):
        c = self.case
        if self.fp8:
            if write:
                pa.pa_reshape_and_cache_fp8(self.k_new, self.v_new, self.k_cache, self.v_cache,
                                            self.slots, self.k_scale, self.v_scale,
                                            device_errors=self.errs)
            out = torch.empty(self.q.shape, dtype=self.tdt, device=DEV)
            pa.pa_decode_fp8(out, self.q, self.k_cache, self.v_cache, self.tables, self.lens,
                             c.scale, self.k_scale, self.v_scale, c.num_kv_heads,
                             c.max_context_len, chunk_tokens=chunk_tokens,
                             device_errors=self.errs)
            return out
        if write:
            pa.pa_reshape_and_cache(self.k_new, self.v_new, self.k_cache, self.v_cache, self.slots,
                                    device_errors=self.errs)
        out = torch.empty(self.q.shape, dtype=self.tdt, device=DEV)
        pa.pa_decode(out, self.q, self.k_cache, self.v_cache, self.tables, self.lens, c.scale,
                     c.num_kv_heads, c.max_context_len, chunk_tokens=chunk_tokens,
                     device_errors=self.errs)
        return out

    def device_errors(self):
        return pa.pa_read_device_errors(self.errs)


def oracle_step(case, rows=None, threads=0):
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    if case.dtype == "fp8":
        ks, vs = case.extra["k_scale"], case.extra["v_scale"]
        oracle.reshape_and_cache_fp8(case.k_new, case.v_new, kc, vc, case.slot_mapping, ks, vs)
        return oracle.decode_kv8_f64(case.q, kc, vc, case.block_tables, case.context_lens,
                                     case.scale, ks, vs, rows=rows, threads=threads)
    oracle.reshape_and_cache(case.k_new, case.v_new, kc, vc, case.slot_mapping)
    return oracle.decode_f64(case.q, kc, vc, case.block_tables, case.context_lens, case.scale,
                             case.num_kv_heads, case.dtype, rows=rows, threads=threads)


def check_tolerance(got, want, dtype, what=""):
    """fp32 inputs: max |err| <= 1e-4.  bf16 outputs (bf16 or e4m3 pools): max <= 2e-2,
    mean <= 2e-3."""
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    if dtype == "f32":
        assert err.max() <= 1e-4, f"{what}: max |err| {err.max():.3e}"
    else:
        assert err.max() <= 2e-2, f"{what}: max |err| {err.max():.3e}"
        assert err.mean() <= 2e-3, f"{what}: mean |err| {err.mean():.3e}"
    return float(err.max()), float(err.mean())
