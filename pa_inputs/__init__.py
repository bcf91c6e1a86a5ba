"""Seeded synthetic inputs for paged-KV decode.

This module serves both the CUDA path and the CPU oracle.  It draws random
numbers and lays them out; it holds none of the attention arithmetic and makes
no block-management decision (no free list, no reference counts, no
copy-on-write) -- those belong to the two implementations under test.

Everything comes from ``numpy.random.Generator(PCG64(seed))``.  Draw order for a
decode case: context lengths -> pool permutation -> prefill K/V -> new-token
K/V -> q.  Values are drawn in float32 and, for bf16 cases, rounded to bf16 with
round-to-nearest-even (torch's ``.to(torch.bfloat16)``); bf16 data is carried as
its uint16 bit patterns.

Pool layout: ``[num_blocks][num_kv_heads][block_size][head_dim]`` for K and for V.
Slots that hold no token are filled with NaN so that any read of them by an
implementation shows up in its output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16_NAN = np.uint16(0x7FC0)

# The five workloads: decode over a paged pool, by name.
WORKLOADS = {
    "tiny_fp32": dict(seed=1001, dtype="f32", num_seqs=4, num_q_heads=8, num_kv_heads=8,
                      head_dim=64, block_size=16, lens=("uniform", 17, 200), num_blocks=64,
                      std=1.0),
    "mha_bf16": dict(seed=1002, dtype="bf16", num_seqs=64, num_q_heads=32, num_kv_heads=32,
                     head_dim=128, block_size=16, lens=("uniform", 512, 4096), std=1.0),
    "gqa_bf16": dict(seed=1003, dtype="bf16", num_seqs=256, num_q_heads=32, num_kv_heads=8,
                     head_dim=128, block_size=16, lens=("lognormal", 1024, 1.0, 16, 8192),
                     std=1.0),
    "long128k_bf16": dict(seed=1004, dtype="bf16", num_seqs=4, num_q_heads=32, num_kv_heads=8,
                          head_dim=128, block_size=32, lens=("fixed", 131072), std=0.5),
}

# The same decode workloads with float8 e4m3 K/V pools (q and the new token bf16).
for _name in ("mha_bf16", "gqa_bf16", "long128k_bf16"):
    WORKLOADS[_name.replace("bf16", "fp8")] = dict(WORKLOADS[_name], dtype="fp8")

# Speculative-verify steps: q_len new (draft) tokens per sequence, causal.
WORKLOADS["spec4_mha_bf16"] = dict(WORKLOADS["mha_bf16"], q_len=4)
WORKLOADS["spec2_gqa_bf16"] = dict(WORKLOADS["gqa_bf16"], q_len=2)

SHARED_PREFIX = dict(seed=1005, dtype="bf16", num_parents=8, children_per_parent=16,
                     prompt_len=2048, parent_extra=(1, 15), tail=(0, 512), num_q_heads=32,
                     num_kv_heads=8, head_dim=128, block_size=16, std=1.0)


def to_storage(x: np.ndarray, dtype: str, scale=None) -> np.ndarray:
    """float32 samples -> stored form: float32; bf16 bits as uint16 (RNE); or,
    for "fp8", e4m3 codes of x / scale[h] (scale per kv head, axis 1 of x),
    through torch's float8_e4m3fn cast on values kept inside +-448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    import torch
    if dtype == "fp8":
        sc = np.asarray(scale, dtype=np.float32).reshape((1, -1) + (1,) * (x.ndim - 2))
        y = np.clip(x / sc, -448.0, 448.0)
        return torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def storage_dtype(dtype: str):
    return {"bf16": np.uint16, "f32": np.float32, "fp8": np.uint8}[dtype]


FP8_NAN = np.uint8(0x7F)


def nan_fill(shape, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return np.full(shape, BF16_NAN, dtype=np.uint16)
    if dtype == "fp8":
        return np.full(shape, FP8_NAN, dtype=np.uint8)
    return np.full(shape, np.nan, dtype=np.float32)


def fp8_scales(num_kv_heads: int, std: float) -> np.ndarray:
    """Per-kv-head dequantisation scales of the fp8 workloads: 8 standard
    deviations map to 448, slightly different for every head."""
    h = np.arange(num_kv_heads, dtype=np.float64)
    return (std * 8.0 / 448.0 * (1.0 + h / 16.0)).astype(np.float32)


def draw_lengths(rng: np.random.Generator, spec, num_seqs: int) -> np.ndarray:
    kind = spec[0]
    if kind == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=num_seqs).astype(np.int32)
    if kind == "lognormal":
        median, sigma, lo, hi = spec[1:]
        raw = rng.lognormal(mean=math.log(median), sigma=sigma, size=num_seqs)
        return np.clip(np.rint(raw), lo, hi).astype(np.int32)
    if kind == "fixed":
        return np.full(num_seqs, spec[1], dtype=np.int32)
    if kind == "list":
        return np.asarray(spec[1], dtype=np.int32)
    raise ValueError(kind)


@dataclass
class DecodeCase:
    """One decode step's inputs.  ``context_lens`` counts the new tokens: the
    last q_len positions L_b - q_len .. L_b - 1 are written by the step's cache
    write, positions before them are already in the pool (q_len = 1: a plain
    decode step)."""
    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    context_lens: np.ndarray      # int32 [B]
    block_tables: np.ndarray      # int32 [B, max_blocks], -1 past each sequence's pages
    slot_mapping: np.ndarray      # int64 [B * q_len], slots of the new positions (-1: none)
    k_cache: np.ndarray           # [NB, Hkv, bs, D] storage
    v_cache: np.ndarray
    k_new: np.ndarray             # [B * q_len, Hkv, D] storage
    v_new: np.ndarray
    q: np.ndarray                 # [B, Hq, D] storage; [B, q_len, Hq, D] when q_len > 1
    extra: dict = field(default_factory=dict)
    q_len: int = 1

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    def kv_bytes(self) -> int:
        """Bytes of K and V of the valid tokens (what one decode step must read)."""
        elt = {"bf16": 2, "f32": 4, "fp8": 1}[self.dtype]
        return int(self.context_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_dim * elt


def _draw_normal(rng, shape, std):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def make_decode_case(name="custom", *, seed, dtype, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, lens, std=1.0, num_blocks=None, slack=0.10,
                     scale=None, max_blocks_per_seq=None, q_len=1) -> DecodeCase:
    """Build a seeded decode case; ``lens`` is a length spec (see ``draw_lengths``).
    With q_len > 1 the step writes and attends with q_len new tokens per
    sequence (lengths below q_len are raised to q_len)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, Hq, Hkv, D, bs = num_seqs, num_q_heads, num_kv_heads, head_dim, block_size
    # fp8 cases: e4m3 pools with per-kv-head scales; q and the new token in bf16
    kv_dtype, act_dtype = dtype, ("bf16" if dtype == "fp8" else dtype)
    ksc = fp8_scales(Hkv, std) if dtype == "fp8" else None
    vsc = ksc * np.float32(1.25) if dtype == "fp8" else None
    L = draw_lengths(rng, lens, B)
    if q_len > 1:
        L = np.maximum(L, q_len).astype(np.int32)
    pages = [(int(l) + bs - 1) // bs for l in L]
    need = int(sum(pages))
    NB = int(num_blocks) if num_blocks is not None else max(1, int(math.ceil((1.0 + slack) * need)))
    if need > NB:
        raise ValueError(f"pool of {NB} blocks cannot hold {need} pages")
    perm = rng.permutation(NB).astype(np.int32)
    mb = max_blocks_per_seq if max_blocks_per_seq is not None else max(1, max(pages) if pages else 1)
    tables = np.full((B, mb), -1, dtype=np.int32)
    # physical pages are dealt from the end of the permutation, one sequence after another
    cursor = NB
    for b in range(B):
        tables[b, :pages[b]] = perm[cursor - pages[b]:cursor][::-1]
        cursor -= pages[b]

    k_cache = nan_fill((NB, Hkv, bs, D), kv_dtype)
    v_cache = nan_fill((NB, Hkv, bs, D), kv_dtype)
    for b in range(B):
        n_old = max(int(L[b]) - q_len, 0)
        if n_old == 0:
            continue
        kb = to_storage(_draw_normal(rng, (n_old, Hkv, D), std), kv_dtype, ksc)
        vb = to_storage(_draw_normal(rng, (n_old, Hkv, D), std), kv_dtype, vsc)
        _lay_out_prefix(k_cache, tables[b], kb, bs)
        _lay_out_prefix(v_cache, tables[b], vb, bs)
    k_new = to_storage(_draw_normal(rng, (B * q_len, Hkv, D), std), act_dtype)
    v_new = to_storage(_draw_normal(rng, (B * q_len, Hkv, D), std), act_dtype)
    q_shape = (B, Hq, D) if q_len == 1 else (B, q_len, Hq, D)
    q = to_storage(_draw_normal(rng, q_shape, std), act_dtype)
    slots = np.full(B * q_len, -1, dtype=np.int64)
    for b in range(B):
        for j in range(q_len):
            pos = int(L[b]) - q_len + j
            if pos >= 0:
                slots[b * q_len + j] = int(tables[b, pos // bs]) * bs + pos % bs
    return DecodeCase(name=name, dtype=dtype, num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv,
                      head_dim=D, block_size=bs, num_blocks=NB,
                      scale=float(scale) if scale is not None else 1.0 / math.sqrt(D),
                      context_lens=L, block_tables=tables, slot_mapping=slots,
                      k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new, q=q,
                      extra={} if ksc is None else {"k_scale": ksc, "v_scale": vsc},
                      q_len=q_len)


def _lay_out_prefix(pool, table_row, rows, bs):
    """Put rows[t] (shape [T, Hkv, D]) at logical position t of the sequence whose
    pages are ``table_row``: page table_row[t // bs], offset t % bs."""
    T = rows.shape[0]
    full = T // bs
    if full:
        blk = rows[:full * bs].reshape(full, bs, rows.shape[1], rows.shape[2]).transpose(0, 2, 1, 3)
        pool[table_row[:full]] = blk
    rem = T - full * bs
    if rem:
        pool[table_row[full], :, :rem, :] = rows[full * bs:].transpose(1, 0, 2)


def share_leading_pages(case: DecodeCase, group_sizes, shared_pages) -> DecodeCase:
    """The case with its sequences cut into consecutive groups (sizes
    ``group_sizes``) whose members read their group leader's first
    ``shared_pages[f]`` pages instead of their own (as forked sequences do; a
    member's own first pages are left unused).  Only the tables change; the
    new-token slots lie past the shared pages.  Returns the new case and the
    int32 (group_start, shared_lens) arrays."""
    tables = case.block_tables.copy()
    starts, shared = [0], []
    for size, npg in zip(group_sizes, shared_pages):
        g0 = starts[-1]
        for b in range(g0 + 1, g0 + size):
            tables[b, :npg] = tables[g0, :npg]
        starts.append(g0 + size)
        shared.append(npg * case.block_size)
    if starts[-1] != case.num_seqs:
        raise ValueError("group sizes must add up to the batch")
    out = DecodeCase(**{**case.__dict__, "block_tables": tables})
    return out, np.asarray(starts, np.int32), np.asarray(shared, np.int32)


def place_at_slots(pool, slots, rows, block_size):
    """Put rows[t] (shape [T, Hkv, D]) at global slot slots[t] (prefill of a pool
    whose slots were handed out by a block manager)."""
    slots = np.asarray(slots, dtype=np.int64)
    pool[slots // block_size, :, slots % block_size, :] = rows


def workload(name: str, **overrides) -> DecodeCase:
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    return make_decode_case(name, **spec)


def scaled_workload(name: str, num_seqs: int, seed_offset: int = 0, **overrides) -> DecodeCase:
    """The named workload's shapes and distributions with fewer sequences (for the
    oracle to finish in seconds)."""
    spec = dict(WORKLOADS[name])
    spec["num_seqs"] = num_seqs
    spec["seed"] = spec["seed"] + seed_offset
    if "num_blocks" in spec and name != "tiny_fp32":
        spec.pop("num_blocks")
    spec.update(overrides)
    return make_decode_case(f"{name}[B={num_seqs}]", **spec)


# --------------------------------------------------------------------------
# Shared-prefix / beam workload: the random draws only.  The block manager
# under test turns the script into page tables, slots and copy pairs.
# --------------------------------------------------------------------------
@dataclass
class SharedPrefixScript:
    dtype: str
    num_parents: int
    children_per_parent: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    prefix_lens: np.ndarray          # int32 [P]  tokens each parent holds when it forks
    tails: np.ndarray                # int32 [P * C]  further tokens each child generates
    prefix_k: list                   # P arrays [prefix_len, Hkv, D] storage
    prefix_v: list
    k_new: np.ndarray                # [P * C, Hkv, D] storage (the step's new token)
    v_new: np.ndarray
    q: np.ndarray                    # [P * C, Hq, D]
    finish_keys: np.ndarray          # float64 [P * C]: ties among children finishing together
    initial_free_order: np.ndarray   # int32 [NB]: a seeded permutation of the pool

    @property
    def num_children(self) -> int:
        return self.num_parents * self.children_per_parent


def shared_prefix_script(scale_parents=None, scale_children=None, seed=None,
                         prompt_len=None, tail=None) -> SharedPrefixScript:
    spec = dict(SHARED_PREFIX)
    if seed is not None:
        spec["seed"] = seed
    P = scale_parents or spec["num_parents"]
    C = scale_children or spec["children_per_parent"]
    prompt = prompt_len if prompt_len is not None else spec["prompt_len"]
    t_lo, t_hi = tail if tail is not None else spec["tail"]
    Hq, Hkv, D, bs = spec["num_q_heads"], spec["num_kv_heads"], spec["head_dim"], spec["block_size"]
    dtype, std = spec["dtype"], spec["std"]
    rng = np.random.Generator(np.random.PCG64(spec["seed"]))
    g_lo, g_hi = spec["parent_extra"]
    extra = rng.integers(g_lo, g_hi + 1, size=P)
    prefix_lens = (prompt + extra).astype(np.int32)
    tails = rng.integers(t_lo, t_hi + 1, size=P * C).astype(np.int32)
    # pool: shared pages once per family, plus every private page the run can need
    shared_pages = sum((int(n) + bs - 1) // bs for n in prefix_lens)
    private = 0
    for p in range(P):
        for c in range(C):
            total = int(prefix_lens[p]) + 1 + int(tails[p * C + c])
            private += (total + bs - 1) // bs - int(prefix_lens[p]) // bs
    NB = int(math.ceil(1.10 * (shared_pages + private)))
    free_order = rng.permutation(NB).astype(np.int32)
    prefix_k, prefix_v = [], []
    for p in range(P):
        n = int(prefix_lens[p])
        prefix_k.append(to_storage(_draw_normal(rng, (n, Hkv, D), std), dtype))
        prefix_v.append(to_storage(_draw_normal(rng, (n, Hkv, D), std), dtype))
    k_new = to_storage(_draw_normal(rng, (P * C, Hkv, D), std), dtype)
    v_new = to_storage(_draw_normal(rng, (P * C, Hkv, D), std), dtype)
    q = to_storage(_draw_normal(rng, (P * C, Hq, D), std), dtype)
    finish_keys = rng.random(P * C)
    return SharedPrefixScript(dtype=dtype, num_parents=P, children_per_parent=C,
                              num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                              num_blocks=NB, scale=1.0 / math.sqrt(D), prefix_lens=prefix_lens,
                              tails=tails, prefix_k=prefix_k, prefix_v=prefix_v, k_new=k_new,
                              v_new=v_new, q=q, finish_keys=finish_keys,
                              initial_free_order=free_order)


def random_bm_ops(seed: int, num_ops: int, max_seqs: int = 6, swap: bool = False):
    """A seeded random sequence of block-manager operations (names and operands
    only; whether each succeeds is up to the manager under test).  With ``swap``
    the mix includes swapping sequences out to the host pool and back in."""
    rng = np.random.Generator(np.random.PCG64(seed))
    kinds = ["add", "append", "append", "append", "fork", "free"]
    if swap:
        kinds += ["swapout", "swapin"]
    ops = []
    for _ in range(num_ops):
        kind = kinds[int(rng.integers(0, len(kinds)))]
        a = int(rng.integers(0, max_seqs))
        b = int(rng.integers(0, max_seqs))
        ops.append((kind, a, b))
    return ops


# --------------------------------------------------------------------------
# Driving a block manager through the shared-prefix script.  Every decision
# (which page, whether to copy) is the manager's; this only issues the calls.
# --------------------------------------------------------------------------
def shared_prefix_ids(script: SharedPrefixScript):
    P, C = script.num_parents, script.children_per_parent
    parents = [1_000_000 + p for p in range(P)]
    children = [p * C + c for p in range(P) for c in range(C)]
    return parents, children


def shared_prefix_prefill(manager, script: SharedPrefixScript):
    """Parents take their prompt plus generated tokens, fork their children and
    leave.  Returns per-parent slot arrays (where the prefix rows go)."""
    parents, _ = shared_prefix_ids(script)
    C = script.children_per_parent
    prefix_slots = []
    for p, pid in enumerate(parents):
        manager.add_seq(pid)
        slots = [manager.append_slot(pid)[0] for _ in range(int(script.prefix_lens[p]))]
        prefix_slots.append(np.asarray(slots, dtype=np.int64))
        for c in range(C):
            manager.fork(pid, p * C + c)
        manager.free(pid)
    return prefix_slots


def shared_prefix_step(manager, script: SharedPrefixScript):
    """The timed step of the shared-prefix workload, on any block manager with
    the oracle's method names: the prefill (parents fork their children and
    leave), then one new token per child in id order (its slot; a copy pair when
    it writes into a page it still shares).  Returns the DecodeCase (pools holding
    the prefill, the step's tables and lengths, new tokens and q) and the int64
    copy pairs [P, 2]."""
    s = script
    prefix_slots = shared_prefix_prefill(manager, s)
    _, children = shared_prefix_ids(s)
    kc = nan_fill((s.num_blocks, s.num_kv_heads, s.block_size, s.head_dim), s.dtype)
    vc = nan_fill(kc.shape, s.dtype)
    for p, sl in enumerate(prefix_slots):
        place_at_slots(kc, sl, s.prefix_k[p], s.block_size)
        place_at_slots(vc, sl, s.prefix_v[p], s.block_size)
    slots, pairs = [], []
    for c in children:
        slot, src, dst = manager.append_slot(c)
        slots.append(slot)
        if src >= 0:
            pairs.append((src, dst))
    rows = [manager.block_table(c) for c in children]
    mb = max(len(pages) for pages, _ in rows)
    tables = np.full((len(children), mb), -1, np.int32)
    for i, (pages, _) in enumerate(rows):
        tables[i, :len(pages)] = pages
    lens = np.asarray([length for _, length in rows], np.int32)
    case = DecodeCase(name="shared_prefix_bf16", dtype=s.dtype, num_seqs=len(children),
                      num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads, head_dim=s.head_dim,
                      block_size=s.block_size, num_blocks=s.num_blocks, scale=s.scale,
                      context_lens=lens, block_tables=tables,
                      slot_mapping=np.asarray(slots, np.int64), k_cache=kc, v_cache=vc,
                      k_new=s.k_new, v_new=s.v_new, q=s.q)
    return case, np.asarray(pairs, np.int64).reshape(-1, 2)


def shared_prefix_finish_order(script: SharedPrefixScript):
    """Step at which each child finishes (after its tail) and the order of the
    children finishing at the same step."""
    _, children = shared_prefix_ids(script)
    order = sorted(children, key=lambda c: (int(script.tails[c]), float(script.finish_keys[c])))
    return order
