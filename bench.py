"""Benchmark: one decode step of the paged-KV path per timed step.

A step is the hot path over one batch: the new tokens' cache write
(pa_reshape_and_cache; for the shared-prefix workload the copy-on-write page
copies first) followed by paged decode attention (pa_decode: plan, persistent
decode kernel, split-K merge).  Inputs are seeded synthetic data
(pa_inputs) already resident in HBM; the K/V working set of the default
workload (2.4 GB) is far larger than L2, so no flush is needed between steps.

Prints one JSON line.  `value` is KV-read GB/s: the algorithmic bytes of the
step (valid tokens' K and V, q, out, block-table entries, lengths, and the
cache write) divided by the device time of the step, summed over ranks.

`--impl reference` times the CPU oracle (fp64, OpenMP on the host cores) on a
bounded sample of the same workload and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import pa_inputs  # noqa: E402

METRIC = "paged decode KV-read GB/s (% of GB300 HBM peak); decode steps/s, µs/step"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "mha_bf16"   # Llama-2-7B-shaped MHA decode, bf16, batch 64
DECODE_SOURCES = ["paged_decode.cuh", "decode_launch.cu", "decode_instances.cuh", "pa_device.cuh",
                  "pa_internal.h"]
CASCADE_SOURCES = DECODE_SOURCES + ["cascade.cu"]


# ------------------------------------------------------------------ helpers
def element_sizes(case):
    """(cache element bytes, q / out / new-token element bytes)."""
    return {"f32": (4, 4), "bf16": (2, 2), "fp8": (1, 2)}[case.dtype]


def algorithmic_bytes(case) -> dict:
    kv_elt, act_elt = element_sizes(case)
    L = case.context_lens.astype(np.int64)
    B, Hq, Hkv, D, bs = (case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim,
                         case.block_size)
    T = B * case.q_len                                   # new tokens (query rows per head)
    kv = int(L.sum()) * 2 * Hkv * D * kv_elt
    q = T * Hq * D * act_elt
    out = T * Hq * D * act_elt
    tables = 4 * (int(((L + bs - 1) // bs).sum()) + B)
    scales = 2 * 4 * Hkv if case.dtype == "fp8" else 0
    decode = kv + q + out + tables + scales
    # read the new k/v, write them into the pool, the slots (and the scales)
    write = 2 * T * Hkv * D * (act_elt + kv_elt) + 8 * T + scales
    return dict(kv=kv, decode=decode, write=write, step=decode + write)


def unique_kv_bytes(case, group_start, shared_lens) -> int:
    """K/V bytes a shared-prefix decode must read: each group's shared tokens
    once, every sequence's own tokens once."""
    kv_elt, _ = element_sizes(case)
    sizes = np.diff(np.asarray(group_start, np.int64))
    shared = np.asarray(shared_lens, np.int64)
    own = int(case.context_lens.astype(np.int64).sum() - np.repeat(shared, sizes).sum())
    return (int(shared.sum()) + own) * 2 * case.num_kv_heads * case.head_dim * kv_elt


def shared_prefix_bytes(case, pairs, group_start=None, shared_lens=None) -> dict:
    """algorithmic_bytes of the shared-prefix step: plus the copy-on-write page
    copies; with groups (the cascade decode), K/V counted once per group."""
    b = algorithmic_bytes(case)
    kv_elt, _ = element_sizes(case)
    b["copy"] = 2 * 2 * len(pairs) * case.num_kv_heads * case.block_size * case.head_dim * kv_elt
    b["step"] += b["copy"]
    if group_start is not None:
        unique = unique_kv_bytes(case, group_start, shared_lens)
        b["kv_logical"] = b["kv"]
        b["decode"] += unique - b["kv"]
        b["step"] += unique - b["kv"]
        b["kv"] = unique
    return b


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            data = json.load(open(path))

            def find(d):
                if isinstance(d, dict):
                    for k, v in d.items():
                        if isinstance(v, (int, float)) and "hbm" in k.lower() and "gb" in k.lower():
                            return float(v)
                        r = find(v)
                        if r:
                            return r
                return None
            v = find(data)
            if v:
                return v, "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def source_digest(names) -> str:
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "paged_kv_cache_190_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per decode call (the decode kernel's launch; for the cascade
    the prefix and merge kernels') from the committed ncu summary, or None when
    the kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}_traffic.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    sources = CASCADE_SOURCES if "cascade" in workload else DECODE_SOURCES
    if fields.get("source_digest") != source_digest(sources):
        return None
    try:
        return int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""
    QUERY = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        else:
            self.lines = []

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, flag in zip(names, parts[2:6]):
                if flag.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, device, world: int) -> float:
    """The slowest rank's value (every rank gets it); `device` is where the
    process group's backend reduces (a CUDA device for NCCL, the CPU for gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, world: int, seconds_per_step: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_step_per_rank / seconds_per_step / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------- GPU workload
class GpuStep:
    """Device-resident inputs of one workload and the step that runs on them."""

    def __init__(self, name: str, device, torch, pa, chunk_tokens: int = 0, num_seqs: int = 0):
        self.torch, self.pa, self.device = torch, pa, device
        self.chunk_tokens = chunk_tokens
        self.name = name
        self.reduced = bool(num_seqs)
        self.cascade = name == "shared_prefix_cascade_bf16"
        if name in ("shared_prefix_bf16", "shared_prefix_cascade_bf16"):
            self._init_shared_prefix(num_seqs)
        elif num_seqs:
            self._init_decode(pa_inputs.scaled_workload(name, num_seqs))
        else:
            self._init_decode(pa_inputs.workload(name))

    def _t(self, a, bf16=False):
        t = self.torch.from_numpy(np.ascontiguousarray(a))
        if bf16:
            t = t.view(self.torch.int16).view(self.torch.bfloat16)
        return t.to(self.device)

    def _init_decode(self, case, finish=True):
        torch = self.torch
        self.fp8 = case.dtype == "fp8"            # e4m3 pools; q, new token, out bf16
        bf = case.dtype in ("bf16", "fp8")
        self.case = case
        self.k_cache = self._t(case.k_cache, bf and not self.fp8)
        self.v_cache = self._t(case.v_cache, bf and not self.fp8)
        if self.fp8:
            self.k_scale = self._t(case.extra["k_scale"])
            self.v_scale = self._t(case.extra["v_scale"])
        self.k_new, self.v_new = self._t(case.k_new, bf), self._t(case.v_new, bf)
        self.q = self._t(case.q, bf)
        self.slots = self._t(case.slot_mapping)
        self.tables = self._t(case.block_tables)
        self.lens = self._t(case.context_lens)
        self.pairs = None
        self.out = torch.empty(self.q.shape, dtype=self.q.dtype, device=self.device)
        self.max_len = case.max_context_len
        self.Hkv = case.num_kv_heads
        self.scale = case.scale
        self.bytes = algorithmic_bytes(case)
        self.host_inputs = dict(q=case.q, k_new=case.k_new, v_new=case.v_new,
                                slots=case.slot_mapping, tables=case.block_tables,
                                lens=case.context_lens)
        self.bf16 = bf
        if finish:
            self._finish_init()

    def _init_shared_prefix(self, num_parents=0):
        """Shared-prefix step: the library's block manager forks each parent's
        pages to its children; the step copies the partial shared page for all
        but the last child of each family, writes the new tokens, decodes."""
        pa = self.pa
        s = pa_inputs.shared_prefix_script(scale_parents=num_parents or None)
        bm = pa.BlockManager(s.num_blocks, s.block_size, s.initial_free_order)
        prefix_slots = pa_inputs.shared_prefix_prefill(bm, s)
        _, children = pa_inputs.shared_prefix_ids(s)
        kc = pa_inputs.nan_fill((s.num_blocks, s.num_kv_heads, s.block_size, s.head_dim), s.dtype)
        vc = pa_inputs.nan_fill(kc.shape, s.dtype)
        for p, sl in enumerate(prefix_slots):
            pa_inputs.place_at_slots(kc, sl, s.prefix_k[p], s.block_size)
            pa_inputs.place_at_slots(vc, sl, s.prefix_v[p], s.block_size)
        slots, pairs = bm.append_slots(children)
        mb = max(len(bm.block_table(c)[0]) for c in children)
        tables, lens = bm.build_block_tables(children, mb)
        case = pa_inputs.DecodeCase(
            name="shared_prefix_bf16", dtype=s.dtype, num_seqs=len(children),
            num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads, head_dim=s.head_dim,
            block_size=s.block_size, num_blocks=s.num_blocks, scale=s.scale, context_lens=lens,
            block_tables=tables, slot_mapping=slots, k_cache=kc, v_cache=vc, k_new=s.k_new,
            v_new=s.v_new, q=s.q)
        self._init_decode(case, finish=False)
        self.pairs = self._t(pairs)
        self.host_inputs["pairs"] = pairs
        if self.cascade:
            # groups from the host tables (the library's grouping); the decode then
            # needs each family's shared pages once, each child's own tokens once
            starts, shared = pa.pa_cascade_groups(tables, lens, s.block_size)
            self.group_start, self.shared_lens = self._t(starts), self._t(shared)
            self.host_inputs["group_start"], self.host_inputs["shared_lens"] = starts, shared
            self.bytes = shared_prefix_bytes(case, pairs, starts, shared)
            self.groups = len(shared)
        else:
            self.bytes = shared_prefix_bytes(case, pairs)
        self._finish_init()

    def _finish_init(self):
        torch, pa = self.torch, self.pa
        c = self.case
        if self.cascade:
            self.ws_bytes = pa.pa_decode_cascade_workspace_size(
                c.num_seqs, self.groups, c.num_q_heads, c.num_kv_heads, c.head_dim,
                c.block_size, self.max_len, self.chunk_tokens)
        else:
            self.ws_bytes = pa.pa_decode_workspace_size(c.num_seqs, c.q_len * c.num_q_heads,
                                                        c.num_kv_heads, c.head_dim,
                                                        c.block_size, self.max_len,
                                                        self.chunk_tokens)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8,
                                     device=self.device)
        self.errs = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.chunk = self.chunk_tokens or pa.pa_decode_chunk_tokens(
            c.num_seqs, c.num_kv_heads, c.block_size, self.max_len)
        # kernels of ours per step: [copy_blocks] + reshape + plan + decode [+ merge];
        # the cascade adds the prefix kernel and always merges
        self.launches_per_step = (1 if self.pairs is not None else 0) + 3 + (
            1 if self.max_len > self.chunk else 0)
        if self.cascade:
            self.launches_per_step = (1 if self.pairs is not None else 0) + 5

    def write(self, prepare=False):
        """Enqueue the step's page copies and cache write; with ``prepare`` return
        them as prepared C-ABI calls instead."""
        pa, calls = self.pa, []
        if self.pairs is not None:
            calls.append(pa.pa_copy_blocks(self.k_cache, self.v_cache, self.pairs,
                                           device_errors=self.errs, prepare=prepare))
        if self.fp8:
            calls.append(pa.pa_reshape_and_cache_fp8(self.k_new, self.v_new, self.k_cache,
                                                     self.v_cache, self.slots, self.k_scale,
                                                     self.v_scale, device_errors=self.errs,
                                                     prepare=prepare))
        else:
            calls.append(pa.pa_reshape_and_cache(self.k_new, self.v_new, self.k_cache,
                                                 self.v_cache, self.slots, device_errors=self.errs,
                                                 prepare=prepare))
        return calls

    def decode(self, prepare=False):
        """Enqueue the step's decode call (or return it prepared)."""
        pa = self.pa
        common = dict(workspace=self.workspace, chunk_tokens=self.chunk_tokens,
                      device_errors=self.errs, prepare=prepare)
        if self.cascade:
            return [pa.pa_decode_cascade(self.out, self.q, self.k_cache, self.v_cache, self.tables,
                                         self.lens, self.group_start, self.shared_lens,
                                         self.scale, self.Hkv, self.max_len, **common)]
        if self.case.q_len > 1:
            return [pa.pa_decode_multi(self.out, self.q, self.k_cache, self.v_cache, self.tables,
                                       self.lens, self.scale, self.Hkv, self.max_len, **common)]
        if self.fp8:
            return [pa.pa_decode_fp8(self.out, self.q, self.k_cache, self.v_cache, self.tables,
                                     self.lens, self.scale, self.k_scale, self.v_scale, self.Hkv,
                                     self.max_len, **common)]
        return [pa.pa_decode(self.out, self.q, self.k_cache, self.v_cache, self.tables, self.lens,
                             self.scale, self.Hkv, self.max_len, **common)]

    def dtype_text(self):
        if self.fp8:
            return ("e4m3 K/V codes (e4m3 tensor-core products, q and P split into e4m3 hi + lo, "
                    "fp32 accumulate), bf16 q/out")
        return "bf16" if self.bf16 else "f32"

    def unique_kv_bytes(self):
        """K/V bytes of the distinct physical pages the step's tables touch."""
        c = self.case
        pages = set()
        for b in range(c.num_seqs):
            n = (int(c.context_lens[b]) + c.block_size - 1) // c.block_size
            pages.update(c.block_tables[b, :n].tolist())
        kv_elt, _ = element_sizes(c)
        return len(pages) * 2 * c.num_kv_heads * c.block_size * c.head_dim * kv_elt

    def cascade_summary(self, dec_ms):
        b = self.bytes
        return {"unique_kv_bytes": b["kv"], "logical_kv_bytes": b["kv_logical"],
                "logical_decode_gbs": round((b["decode"] - b["kv"] + b["kv_logical"])
                                            / (dec_ms * 1e-3) / 1e9, 1)}

    def step(self):
        self.write()
        self.decode()

    def prepared_step(self):
        """The whole step as prepared C-ABI calls, in order."""
        return self.write(prepare=True) + self.decode(prepare=True)


# Measured after the headline workload in a default single-GPU run, each with its
# own timing, roofline and clocks: the GQA batch and the 128K-context decode,
# the shared-prefix step (with pa_decode, and with the shared-prefix decode), and
# the float8 pools.
EXTRA_WORKLOADS = ("gqa_bf16", "long128k_bf16", "shared_prefix_bf16",
                   "shared_prefix_cascade_bf16", "mha_fp8", "gqa_fp8", "long128k_fp8")


def time_steps(ws, K, warmup, torch, pa, device, stream, barrier):
    """W untimed steps, then K steps timed with CUDA events on the launching
    stream (around the whole region and around each step's write and decode),
    clocks sampled meanwhile."""
    for _ in range(warmup):
        ws.step()
    torch.cuda.synchronize(device)
    flags = pa.pa_read_device_errors(ws.errs)
    if flags:
        raise RuntimeError(f"{ws.name}: device error bits {flags} during warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    # the step's C-ABI calls with their arguments marshalled once, so that the
    # timed loop enqueues work as fast as the library takes it
    write_calls, decode_calls = ws.write(prepare=True), ws.decode(prepare=True)
    barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            for call in write_calls:
                call()
            ev[i][1].record(stream)
            for call in decode_calls:
                call()
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(device)
        # keep the sampler running for a moment so short regions still get a sample
        if K * 0.5e-3 < 0.3:
            time.sleep(0.3)
    barrier()
    flags = pa.pa_read_device_errors(ws.errs)
    if flags:
        raise RuntimeError(f"{ws.name}: device error bits {flags} during the timed steps")
    return {"total_ms": t_start.elapsed_time(t_end),
            "decode_ms": [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)],
            "write_ms": [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)],
            "clocks": clocks.summary()}


def roofline(ws, dec_avg_ms, peak, peak_src):
    b = ws.bytes
    achieved = b["decode"] / (dec_avg_ms * 1e-3) / 1e9
    kernel = ("pa_decode_cascade call (plan + prefix kernel + paged_decode_kernel + merge)"
              if ws.cascade else "pa_decode call (plan + paged_decode_kernel + merge)")
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": None if ws.reduced else ncu_traffic(ws.name),
            "kernel": kernel + ", CUDA events", "algorithmic_bytes_per_launch": b["decode"],
            "avg_launch_us": round(dec_avg_ms * 1e3, 2),
            "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json hbm_gbs' if peak_src == 'measured' else 'profiling recipe fallback 6.8 TB/s'})"}


def l2_note(ws):
    kv = ws.bytes["kv"]
    if kv > 1e9:
        return "no flush: the step reads %.2f GB of K/V, far above the 129 MB L2" % (kv / 1e9)
    return ("no flush: the step's %.0f MB of distinct K/V pages can sit in the 129 MB L2, so its "
            "GB/s is not a DRAM rate" % (ws.unique_kv_bytes() / 1e6))


def workload_entry(ws, m, e2e, world, peak, peak_src):
    """Summary of one extra workload for the JSON line."""
    K = len(m["decode_ms"])
    ms_per_step = m["total_ms"] / K
    dec_ms = statistics.mean(m["decode_ms"])
    c = ws.case
    entry = {
        "value": round(whole_job_gbs(ws.bytes["step"], world, ms_per_step * 1e-3), 2),
        "unit": "GB/s", "steps": K, "us_per_step": round(ms_per_step * 1e3, 2),
        "steps_per_s": round(1e3 / ms_per_step, 1),
        "dtype": ws.dtype_text(),
        "config": {"num_seqs": c.num_seqs, "num_q_heads": c.num_q_heads,
                   "num_kv_heads": c.num_kv_heads, "head_dim": c.head_dim,
                   "block_size": c.block_size, "mean_context": float(c.context_lens.mean()),
                   "max_context": ws.max_len, "chunk_tokens": ws.chunk, "l2": l2_note(ws),
                   "algorithmic_bytes_per_step": ws.bytes["step"]},
        "roofline": roofline(ws, dec_ms, peak, peak_src),
        "write_avg_us": round(statistics.mean(m["write_ms"]) * 1e3, 2),
        "e2e": e2e, "gpu_launches": ws.launches_per_step * K, "clocks": m["clocks"],
    }
    if ws.cascade:
        entry["config"]["groups"] = ws.groups
        entry["cascade"] = ws.cascade_summary(dec_ms)
    return entry


def run_gpu(args, world, rank, local):
    import torch
    import paged_kv_cache_190_gb300 as pa
    pa.library()
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    ws = GpuStep(args.workload, device, torch, pa, args.chunk_tokens, args.num_seqs)
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    K = args.steps
    m = time_steps(ws, K, args.warmup, torch, pa, device, stream, barrier)
    ms_per_step = max_over_ranks(m["total_ms"] / K, device, world)

    # end to end through the C ABI with host buffers
    e2e = run_e2e(ws, K, args.warmup, torch, device, stream, barrier, world)

    peak, peak_src = hbm_peak()
    extras = {}
    if world == 1 and args.extra_workloads and not args.num_seqs:
        # the other configurations the target is stated on, measured the same way
        names = [w for w in args.extra_workloads.split(",") if w and w != args.workload]
        host_ms = {}
        for name in names:
            t0 = time.perf_counter()
            xs = GpuStep(name, device, torch, pa, 0)
            xK, xW = max(K, args.extra_steps), max(args.warmup, 5)
            xm = time_steps(xs, xK, xW, torch, pa, device, stream, barrier)
            xe = run_e2e(xs, xK, xW, torch, device, stream, barrier, world)
            extras[name] = workload_entry(xs, xm, xe, world, peak, peak_src)
            host_ms[name] = round((time.perf_counter() - t0) * 1e3, 1)
            del xs
            torch.cuda.empty_cache()
    if rank != 0:
        return None
    b = ws.bytes
    value = whole_job_gbs(b["step"], world, ms_per_step * 1e-3)
    dec_avg_ms = statistics.mean(m["decode_ms"])
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "steps_per_s": round(world * 1e3 / ms_per_step, 1),
        "hbm_frac_step": round(value / world / peak, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ws.dtype_text(), "data": "synthetic (seeded pa_inputs; no dataset or weights)",
        "config": {
            "workload": args.workload + (f"[reduced: {args.num_seqs}]" if args.num_seqs else ""),
            "num_seqs": ws.case.num_seqs,
            "num_q_heads": ws.case.num_q_heads, "num_kv_heads": ws.case.num_kv_heads,
            "head_dim": ws.case.head_dim, "block_size": ws.case.block_size,
            "num_blocks": ws.case.num_blocks, "mean_context": float(ws.case.context_lens.mean()),
            "max_context": ws.max_len, "chunk_tokens": ws.chunk,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": l2_note(ws),
            "step": ("copy_blocks + " if ws.pairs is not None else "")
            + "reshape_and_cache + decode (plan, persistent decode, split-K merge)",
            "algorithmic_bytes_per_step": b["step"],
        },
        "roofline": roofline(ws, dec_avg_ms, peak, peak_src),
        "write_avg_us": round(statistics.mean(m["write_ms"]) * 1e3, 2),
        "host_block_manager": host_block_manager_time(ws.case, pa),
        "e2e": e2e,
        "gpu_launches": ws.launches_per_step * K,
        "clocks": m["clocks"],
    }
    if ws.cascade:
        # algorithmic bytes above count each family's shared pages once; the same
        # call measured against every child's whole context, for comparison with
        # pa_decode on the same batch
        result["config"]["step"] = ("copy_blocks + reshape_and_cache + cascade decode (plan, "
                                    "shared-prefix kernel, persistent decode over each "
                                    "sequence's own pages, merge)")
        result["config"]["groups"] = ws.groups
        result["cascade"] = ws.cascade_summary(dec_avg_ms)
    if extras:
        result["workloads"] = extras
        result["workloads_note"] = (
            "each measured after the headline in the same process: its own warm-up, "
            f"max(steps, {args.extra_steps}) timed steps, CUDA-event decode time, roofline "
            "against the same peak, clocks and e2e; host seconds to build each: "
            + ", ".join(f"{k} {v / 1e3:.1f}" for k, v in host_ms.items()))
    if not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(ws.case, budget_s=args.cpu_budget,
                                              step_bytes=b["step"])
    return result


SWAP_METRIC = "page swap GB/s (device pool <-> pinned host pool, out + in)"


def host_link_peak(torch, device, nbytes=1 << 30, reps=5):
    """Measured copy-engine rate of one large pinned <-> device copy each way
    (GB/s): the denominator of the swap roofline."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    rates = {}
    for name, (dst, src) in (("d2h", (h, d)), ("h2d", (d, h))):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize(device)
        rates[name] = nbytes * reps / (a.elapsed_time(b) * 1e-3) / 1e9
    del h, d
    return rates


def run_swap(args, world, rank, local):
    """Swap a quarter of the GQA workload's sequences (every 4th) out to a
    pinned host pool and back into their pages, every step: one pa_swap_blocks
    call each way, plus the host block manager's swap bookkeeping for the same
    sequences timed separately."""
    import torch
    import paged_kv_cache_190_gb300 as pa
    pa.library()
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if rank != 0:
        return None
    case = pa_inputs.workload("gqa_bf16")
    NB, Hkv, bs, D = case.k_cache.shape
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    kc, vc = to(case.k_cache), to(case.v_cache)
    victims = list(range(0, case.num_seqs, 4))
    pages = [int(p) for b in victims for p in case.block_tables[b] if p >= 0]
    H = len(pages)
    hk = torch.empty((H, Hkv, bs, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((H, Hkv, bs, D), dtype=torch.bfloat16).pin_memory()
    out_pairs = torch.tensor([[p, h] for h, p in enumerate(pages)], dtype=torch.int64, device=device)
    in_pairs = out_pairs[:, [1, 0]].contiguous()
    errs = torch.zeros(1, dtype=torch.int32, device=device)
    block_bytes = Hkv * bs * D * 2
    bytes_step = 2 * 2 * H * block_bytes                  # K and V, out and in
    stream = torch.cuda.current_stream(device)

    def step():
        pa.pa_swap_blocks(kc, vc, hk, hv, out_pairs, device_errors=errs)
        pa.pa_swap_blocks(hk, hv, kc, vc, in_pairs, device_errors=errs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    K = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        for i in range(K):
            ev[i][0].record(stream)
            pa.pa_swap_blocks(kc, vc, hk, hv, out_pairs, device_errors=errs)
            ev[i][1].record(stream)
            pa.pa_swap_blocks(hk, hv, kc, vc, in_pairs, device_errors=errs)
            ev[i][2].record(stream)
        torch.cuda.synchronize(device)
    flags = pa.pa_read_device_errors(errs)
    if flags:
        raise RuntimeError(f"device error bits {flags}")
    out_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    in_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(K))
    ms = out_ms + in_ms
    peak = host_link_peak(torch, device)
    half = bytes_step / 2
    out_gbs, in_gbs = half / (out_ms * 1e-3) / 1e9, half / (in_ms * 1e-3) / 1e9
    # host bookkeeping: swap the same sequences out and in through the C++ manager
    bm = pa.BlockManager(NB, bs)
    bm.enable_swap(H + 1)
    lens = case.context_lens
    for b in victims:
        bm.add_seq(b)
        for _ in range(int(lens[b])):
            bm.append_slot(b)
    t0 = time.perf_counter()
    for b in victims:
        bm.swap_out(b)
    t1 = time.perf_counter()
    for b in victims:
        bm.swap_in(b)
    t2 = time.perf_counter()
    bm.close()
    return {
        "metric": SWAP_METRIC, "value": round(bytes_step / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bytes",
        "data": "synthetic (seeded pa_inputs; no dataset or weights)",
        "config": {"workload": "swap_gqa", "sequences_swapped": len(victims), "pages": H,
                   "page_bytes_per_pool": block_bytes, "bytes_per_step": bytes_step,
                   "host_pool": "pinned host memory, addressed by the kernel over the host link"},
        "roofline": {"bound": "host-link", "achieved": round(min(out_gbs, in_gbs), 1),
                     "peak": round(min(peak["d2h"], peak["h2d"]), 1), "unit": "GB/s",
                     "frac": round(min(out_gbs / peak["d2h"], in_gbs / peak["h2d"]), 4),
                     "traffic": None, "out_gbs": round(out_gbs, 1), "in_gbs": round(in_gbs, 1),
                     "peak_source": "measured in this run: one 1 GiB pinned<->device copy each way "
                                    f"(d2h {peak['d2h']:.1f}, h2d {peak['h2d']:.1f} GB/s)"},
        "host_block_manager": {"swap_out_all_us": round((t1 - t0) * 1e6, 1),
                               "swap_in_all_us": round((t2 - t1) * 1e6, 1),
                               "sequences": len(victims)},
        "gpu_launches": 2 * K, "clocks": clocks.summary(),
    }


def host_block_manager_time(case, pa, repeats: int = 100):
    """Host cost of the block manager for this batch, after the sequences have
    been grown to the workload's lengths: one decode step (every sequence takes
    its next slot -- a new page at page boundaries -- and the step's tables and
    lengths are exported), and a fork plus a free of every sequence (the
    shared-prefix and finish paths).  Medians over `repeats`."""
    B, bs = case.num_seqs, case.block_size
    lens = case.context_lens.astype(np.int64)
    pages = (lens + bs - 1) // bs
    mb = int(pages.max()) + repeats // bs + 2
    bm = pa.BlockManager(int(pages.sum()) + B * (repeats // bs + 3), bs)
    ids = np.arange(B, dtype=np.int64)
    for b in range(B):
        bm.add_seq(b)
    for t in range(int(lens.max())):
        active = ids[lens > t]
        if active.size:
            bm.append_slots(active)
    step_us, fork_free_us = [], []
    for _ in range(repeats):
        t0 = time.perf_counter()
        bm.append_slots(ids)
        bm.build_block_tables(ids, mb)
        step_us.append((time.perf_counter() - t0) * 1e6)
    for _ in range(max(3, repeats // 10)):
        t0 = time.perf_counter()
        for b in range(B):
            bm.fork(b, B + b)
        for b in range(B):
            bm.free(B + b)
        fork_free_us.append((time.perf_counter() - t0) * 1e6)
    bm.close()
    return {"step_append_slots_and_tables_us": round(statistics.median(step_us), 1),
            "fork_and_free_all_us": round(statistics.median(fork_free_us), 1),
            "num_seqs": B, "note": "host C++ block manager via ctypes; outside the device timing"}


def run_e2e(ws, steps, warmup, torch, device, stream, barrier, world):
    """End to end through the C ABI with host buffers.  The step's inputs (q,
    new k/v, slots, tables, lengths, and the copy pairs or groups where the
    workload has them) sit packed in one pinned host buffer; every step copies
    it into one device buffer whose views are the step's device inputs, runs the
    step's C-ABI calls (prepared once: the same pointers every step), copies the
    output back into pinned host memory and synchronises the stream."""
    spans, off = {}, 0
    for name, a in ws.host_inputs.items():
        nbytes = np.ascontiguousarray(a).nbytes
        spans[name] = (off, nbytes)
        off += (nbytes + 255) // 256 * 256
    host = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev = torch.empty(off, dtype=torch.uint8, device=device)
    host_np = host.numpy()
    for name, a in ws.host_inputs.items():
        o, nbytes = spans[name]
        host_np[o:o + nbytes] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
        old = getattr(ws, name)                       # rebind the input as a view of `dev`
        setattr(ws, name, dev[o:o + nbytes].view(old.dtype).view(old.shape))
    calls = ws.prepared_step()
    out_host = torch.empty(ws.out.shape, dtype=ws.out.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()

    def one():
        dev.copy_(host, non_blocking=True)
        for call in calls:
            call()
        out_host.copy_(ws.out, non_blocking=True)
        stream.synchronize()

    for _ in range(max(3, warmup // 4)):
        one()
    n = max(10, min(steps, 500))
    barrier()
    t0 = time.perf_counter()
    for _ in range(n):
        one()
    t1 = time.perf_counter()
    barrier()
    sec = max_over_ranks((t1 - t0) / n, device, world)
    return {"value": round(whole_job_gbs(ws.bytes["step"], world, sec), 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(off), "d2h_bytes_per_step": int(d2h),
            "us_per_step": round(sec * 1e6, 2), "steps": n,
            "copies_per_step": "1 H2D (packed inputs) + 1 D2H (out), stream synchronised"}


# -------------------------------------------------------------- CPU oracle
def _oracle_sample(case, n_rows, rng):
    if case.q_len > 1:                                   # (sequence, new token, query head)
        rows = [(int(rng.integers(case.num_seqs)), int(rng.integers(case.q_len)),
                 int(rng.integers(case.num_q_heads))) for _ in range(n_rows)]
    else:
        rows = [(int(rng.integers(case.num_seqs)), int(rng.integers(case.num_q_heads)))
                for _ in range(n_rows)]
    elt, act_elt = element_sizes(case)
    D = case.head_dim
    # bytes the sampled rows stand for: each row reads its sequence's K and V for
    # one head (shared by the GQA group, counted once per group member here is
    # avoided by dividing by the group size), plus its q and out row
    G = case.num_q_heads // case.num_kv_heads
    nbytes = sum(int(case.context_lens[r[0]]) * 2 * D * elt / G / case.q_len + 2 * D * act_elt
                 for r in rows)
    return rows, nbytes


def _oracle_write(case, kc, vc):
    import oracle
    if case.dtype == "fp8":
        oracle.reshape_and_cache_fp8(case.k_new, case.v_new, kc, vc, case.slot_mapping,
                                     case.extra["k_scale"], case.extra["v_scale"])
    else:
        oracle.reshape_and_cache(case.k_new, case.v_new, kc, vc, case.slot_mapping)


def _oracle_decode(case, kc, vc, rows=None):
    import oracle
    if case.q_len > 1:
        return oracle.decode_multi_f64(case.q, kc, vc, case.block_tables, case.context_lens,
                                       case.scale, case.num_kv_heads, case.dtype, rows=rows)
    if case.dtype == "fp8":
        return oracle.decode_kv8_f64(case.q, kc, vc, case.block_tables, case.context_lens,
                                     case.scale, case.extra["k_scale"], case.extra["v_scale"],
                                     rows=rows)
    return oracle.decode_f64(case.q, kc, vc, case.block_tables, case.context_lens, case.scale,
                             case.num_kv_heads, case.dtype, rows=rows)


def cpu_baseline(case, budget_s=15.0, kind="oracle", step_bytes=None):
    """The oracle, as it stands, on the host cores: whole decode steps of the
    workload (cache write + every (sequence, query head) row) repeated until
    about `budget_s` seconds have passed, or a random subset of rows when one
    step alone would take longer.  The rate counts the GPU arm's algorithmic
    bytes of a step (`step_bytes`), pro rata for a subset of rows."""
    import oracle
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    threads = oracle.max_threads()
    rng = np.random.default_rng(9)
    all_rows = case.num_seqs * case.q_len * case.num_q_heads
    # calibrate on a few rows
    rows, _ = _oracle_sample(case, 8, rng)
    t0 = time.perf_counter()
    _oracle_decode(case, kc, vc, rows=rows)
    per_row = (time.perf_counter() - t0) / 8
    if step_bytes is None:
        step_bytes = algorithmic_bytes(case)["step"]
    if per_row * all_rows <= budget_s:
        steps, elapsed = 0, 0.0
        while steps == 0 or elapsed < budget_s:
            t0 = time.perf_counter()
            _oracle_write(case, kc, vc)
            _oracle_decode(case, kc, vc)
            elapsed += time.perf_counter() - t0
            steps += 1
        nbytes, sample = steps * step_bytes, f"{steps} whole {case.name} steps"
    else:
        n = int(max(8, budget_s / max(per_row, 1e-9)))
        rows, _ = _oracle_sample(case, n, rng)
        t0 = time.perf_counter()
        _oracle_decode(case, kc, vc, rows=rows)
        elapsed = time.perf_counter() - t0
        nbytes = step_bytes * n / all_rows
        sample = f"{n} random (sequence, query head) rows of the {case.name} step"
    return {"value": round(nbytes / elapsed / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": kind, "sample": f"{sample}, fp64 gather-then-attend, {elapsed:.1f} s",
            "seconds": round(elapsed, 2)}


def run_reference_swap(args, world):
    """The oracle's page copy (numpy) on the swap_gqa pages: out to a host pool
    and back, every step."""
    import oracle
    case = pa_inputs.workload("gqa_bf16")
    NB, Hkv, bs, D = case.k_cache.shape
    victims = list(range(0, case.num_seqs, 4))
    pages = [int(p) for b in victims for p in case.block_tables[b] if p >= 0]
    out_pairs = np.array([[p, h] for h, p in enumerate(pages)], np.int64)
    in_pairs = out_pairs[:, ::-1].copy()
    hk = np.empty((len(pages), Hkv, bs, D), case.k_cache.dtype)
    hv = np.empty_like(hk)
    kc, vc = case.k_cache, case.v_cache
    bytes_step = 2 * 2 * len(pages) * Hkv * bs * D * 2
    for _ in range(min(args.warmup, 2)):
        oracle.copy_pages(kc, vc, hk, hv, out_pairs)
        oracle.copy_pages(hk, hv, kc, vc, in_pairs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.copy_pages(kc, vc, hk, hv, out_pairs)
        oracle.copy_pages(hk, hv, kc, vc, in_pairs)
    sec = (time.perf_counter() - t0) / args.steps
    value = bytes_step / sec / 1e9
    return {"metric": SWAP_METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bytes",
            "data": "synthetic (seeded pa_inputs)", "impl": "reference",
            "config": {"workload": "swap_gqa", "pages": len(pages)},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": "every step whole (numpy page copies)"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle on a bounded sample per step."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    if args.workload == "swap_gqa":
        return run_reference_swap(args, world)
    pairs = None
    if args.workload in ("shared_prefix_bf16", "shared_prefix_cascade_bf16"):
        # the same step the GPU arm times, from the oracle's block manager; the
        # oracle decodes every child over its whole context (sharing changes only
        # where the bytes live), the rate counts the GPU arm's bytes
        s = pa_inputs.shared_prefix_script()
        case, pairs = pa_inputs.shared_prefix_step(
            oracle.RefBlockManager(s.num_blocks, s.block_size, s.initial_free_order), s)
        if args.workload == "shared_prefix_cascade_bf16":
            C = s.children_per_parent
            starts = np.arange(0, case.num_seqs + 1, C)
            shared = (s.prefix_lens.astype(np.int64) // s.block_size) * s.block_size
            step_bytes = shared_prefix_bytes(case, pairs, starts, shared)["step"]
        else:
            step_bytes = shared_prefix_bytes(case, pairs)["step"]
    else:
        case = pa_inputs.workload(args.workload)
        step_bytes = algorithmic_bytes(case)["step"]
    all_rows = case.num_seqs * case.q_len * case.num_q_heads
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    threads = oracle.max_threads()
    rng = np.random.default_rng(11)
    # size a step so K + W steps take about two minutes
    rows, _ = _oracle_sample(case, 4, rng)
    t0 = time.perf_counter()
    _oracle_decode(case, kc, vc, rows=rows)
    per_row = (time.perf_counter() - t0) / 4
    total_steps = args.steps + args.warmup
    n_rows = int(max(1, min(4 * threads, 120.0 / max(total_steps, 1) / max(per_row, 1e-6))))
    samples = [_oracle_sample(case, n_rows, rng) for _ in range(args.steps + args.warmup)]
    elapsed, nbytes_total = 0.0, 0.0
    for i, (rows, _) in enumerate(samples):
        t0 = time.perf_counter()
        if pairs is not None:
            oracle.copy_blocks(kc, vc, pairs)
        _oracle_write(case, kc, vc)
        _oracle_decode(case, kc, vc, rows=rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            elapsed += dt
            nbytes_total += step_bytes * len(rows) / all_rows
    value = nbytes_total / elapsed / 1e9
    ms = elapsed / args.steps * 1e3
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded pa_inputs)", "impl": "reference",
            "config": {"workload": args.workload, "num_seqs": case.num_seqs,
                       "rows_per_step": n_rows},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"{n_rows} random (sequence, query head) rows per step"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def replica_command(n, argv, port):
    """The command that runs this benchmark as n ranks, one process per GPU."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
            os.path.abspath(__file__), *argv]


def launch_replicas(n, argv) -> int:
    """`--gpus N` without a launcher: start N ranks (one per GPU) and pass their
    output through; rank 0 prints the JSON line.  Returns the launcher's status."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    return subprocess.call(replica_command(n, argv, port))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(pa_inputs.WORKLOADS) + ["shared_prefix_bf16",
                                                         "shared_prefix_cascade_bf16", "swap_gqa"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--chunk-tokens", type=int, default=0,
                    help="split size for pa_decode (0: the library's automatic choice)")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="a reduced case: the workload's shapes and draws with this many "
                         "sequences (parents for the shared-prefix workloads); 0: full size")
    ap.add_argument("--extra-workloads", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads measured after the headline one in a "
                         "single-GPU run (empty: none)")
    ap.add_argument("--extra-steps", type=int, default=300,
                    help="at least this many timed steps for each extra workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    world, rank, local = dist_env()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: relaunch this command under torch.distributed.run
        sys.exit(launch_replicas(args.gpus, sys.argv[1:] if argv is None else list(argv)))
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    elif args.workload == "swap_gqa":
        res = run_swap(args, world, rank, local)
    else:
        res = run_gpu(args, world, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
