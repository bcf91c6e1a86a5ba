"""GPU parity of the shared-prefix (cascade) decode: the library, through its C
ABI, against the CPU oracle's plain decode over each sequence's whole context
(sharing pages changes where the keys are read from, not what is computed)."""
import numpy as np
import pytest
import torch

import oracle
import pa_inputs
import paged_kv_cache_190_gb300 as pa
from gpu_helpers import DEV, check_tolerance, out_as_f64, to_dev

pytestmark = pytest.mark.gpu


def _grouped_case(name, seed, Hq, Hkv, D, bs, lens, group_sizes, shared_tokens):
    case = pa_inputs.make_decode_case(name, seed=seed, dtype="bf16", num_seqs=len(lens),
                                      num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                      block_size=bs, lens=("list", lens))
    return pa_inputs.share_leading_pages(case, group_sizes, [t // bs for t in shared_tokens])


def _cascade(case, starts, shared, chunk_tokens=0, write=True):
    """Cache write of the step's new tokens, then the cascade decode."""
    kc, vc = to_dev(case.k_cache, True), to_dev(case.v_cache, True)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    if write:
        pa.pa_reshape_and_cache(to_dev(case.k_new, True), to_dev(case.v_new, True), kc, vc,
                                to_dev(case.slot_mapping), device_errors=errs)
    out = torch.full((case.num_seqs, case.num_q_heads, case.head_dim), float("nan"),
                     dtype=torch.bfloat16, device=DEV)
    pa.pa_decode_cascade(out, to_dev(case.q, True), kc, vc, to_dev(case.block_tables),
                         to_dev(case.context_lens), to_dev(starts), to_dev(shared), case.scale,
                         case.num_kv_heads, case.max_context_len, chunk_tokens=chunk_tokens,
                         device_errors=errs)
    return out, pa.pa_read_device_errors(errs), (kc, vc)


def _oracle(case, write=True):
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    if write:
        oracle.reshape_and_cache(case.k_new, case.v_new, kc, vc, case.slot_mapping)
    return oracle.decode_f64(case.q, kc, vc, case.block_tables, case.context_lens, case.scale,
                             case.num_kv_heads, "bf16")


# groups of 5, 1, 3 and 4 sequences sharing 160 tokens (two full 64-token
# stages of the prefix kernel and a ragged one), nothing, 384 (six full stages)
# and 64; the own suffixes run from one token (L = shared + 1, attended to in
# the merge) to several decode-kernel chunks
LENS = [161, 300, 200, 225, 500, 77, 385, 700, 390, 65, 90, 1000, 66]
GROUPS = [5, 1, 3, 4]
SHARED = [160, 0, 384, 64]

# every (group, head_dim) instance of the merge: groups 1, 2, 4, 8 at head_dim 128 and 64
VARIANTS = [(32, 8, 128, 16), (8, 8, 128, 16), (16, 2, 128, 32), (8, 4, 64, 16), (4, 4, 64, 32),
            (16, 16, 64, 16), (16, 8, 128, 16), (16, 4, 64, 16), (16, 2, 64, 32)]


@pytest.mark.parametrize("Hq,Hkv,D,bs", VARIANTS)
@pytest.mark.parametrize("chunk", [0, 64])
def test_cascade_matches_oracle(Hq, Hkv, D, bs, chunk):
    case, starts, shared = _grouped_case(f"cascade-{Hq}-{Hkv}-{D}-{bs}", 1200 + Hq + Hkv + D + bs,
                                         Hq, Hkv, D, bs, LENS, GROUPS, SHARED)
    out, flags, _ = _cascade(case, starts, shared, chunk)
    assert flags == 0
    check_tolerance(out_as_f64(out), _oracle(case), "bf16", case.name)


def test_cascade_close_to_plain_decode():
    """The same batch through pa_decode: both within the tolerance of the oracle
    and of each other (they add the same terms in another order)."""
    case, starts, shared = _grouped_case("cascade-vs-decode", 1250, 32, 8, 128, 16, LENS, GROUPS,
                                         SHARED)
    out, flags, (kc, vc) = _cascade(case, starts, shared)
    plain = torch.empty_like(out)
    pa.pa_decode(plain, to_dev(case.q, True), kc, vc, to_dev(case.block_tables),
                 to_dev(case.context_lens), case.scale, case.num_kv_heads, case.max_context_len)
    assert flags == 0
    diff = np.abs(out_as_f64(out) - out_as_f64(plain))
    assert diff.max() <= 2e-2 and diff.mean() <= 1e-3


def test_long_prefix_with_the_most_pieces():
    """A 4096-token shared prefix (64 stages) cut into the most pieces a group
    may have (32), then 64-token decode chunks of the own suffixes: up to 47
    partials per row."""
    lens = [4096 + 70, 4096 + 1, 4096 + 300, 5000]
    case, starts, shared = _grouped_case("cascade-long", 1260, 16, 4, 128, 16, lens, [4],
                                         [4096])
    out, flags, _ = _cascade(case, starts, shared, chunk_tokens=64)
    assert flags == 0
    check_tolerance(out_as_f64(out), _oracle(case), "bf16", case.name)


def test_shared_prefix_script_through_the_block_manager():
    """Forked families from the library's block manager (copy-on-write of each
    family's partial page), grouped by pa_cascade_groups: every family is one
    group sharing its parent's full pages."""
    s = pa_inputs.shared_prefix_script(scale_parents=3, scale_children=5, prompt_len=300,
                                       tail=(0, 8))
    bm = pa.BlockManager(s.num_blocks, s.block_size, s.initial_free_order)
    prefix_slots = pa_inputs.shared_prefix_prefill(bm, s)
    _, children = pa_inputs.shared_prefix_ids(s)
    shape = (s.num_blocks, s.num_kv_heads, s.block_size, s.head_dim)
    kc, vc = pa_inputs.nan_fill(shape, s.dtype), pa_inputs.nan_fill(shape, s.dtype)
    for p, sl in enumerate(prefix_slots):
        pa_inputs.place_at_slots(kc, sl, s.prefix_k[p], s.block_size)
        pa_inputs.place_at_slots(vc, sl, s.prefix_v[p], s.block_size)
    slots, pairs = bm.append_slots(children)
    mb = max(len(bm.block_table(c)[0]) for c in children)
    tables, lens = bm.build_block_tables(children, mb)
    starts, shared = pa.pa_cascade_groups(tables, lens, s.block_size)
    C = s.children_per_parent
    assert list(starts) == list(range(0, len(children) + 1, C))
    assert list(shared) == [int(n) // s.block_size * s.block_size for n in s.prefix_lens]
    dk, dv = to_dev(kc, True), to_dev(vc, True)
    errs = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_copy_blocks(dk, dv, to_dev(pairs), device_errors=errs)
    pa.pa_reshape_and_cache(to_dev(s.k_new, True), to_dev(s.v_new, True), dk, dv, to_dev(slots),
                            device_errors=errs)
    out = torch.empty((len(children), s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device=DEV)
    pa.pa_decode_cascade(out, to_dev(s.q, True), dk, dv, to_dev(tables), to_dev(lens),
                         to_dev(starts), to_dev(shared), s.scale, s.num_kv_heads,
                         int(lens.max()), device_errors=errs)
    assert pa.pa_read_device_errors(errs) == 0
    oracle.copy_blocks(kc, vc, pairs)
    oracle.reshape_and_cache(s.k_new, s.v_new, kc, vc, slots)
    want = oracle.decode_f64(s.q, kc, vc, tables, lens, s.scale, s.num_kv_heads, "bf16")
    check_tolerance(out_as_f64(out), want, "bf16", "shared-prefix script")


def test_bad_shared_lengths_are_flagged_and_decoded_without_sharing():
    """A shared length that is not a whole number of pages (group 0), or not
    below a member's length (group 1): PA_DEVERR_BAD_LENGTH, and the rows are
    still the plain decode (those sequences read their own pages)."""
    lens = [100, 120, 90, 64, 200]
    case, starts, shared = _grouped_case("cascade-badlen", 1270, 8, 4, 128, 16, lens, [3, 2],
                                         [64, 64])
    shared = np.array([40, 64], np.int32)                 # 40: not a whole page; 64 = L of seq 3
    out, flags, _ = _cascade(case, starts, shared)
    assert flags == pa.PA_DEVERR_BAD_LENGTH
    check_tolerance(out_as_f64(out), _oracle(case), "bf16", case.name)


def test_member_reading_other_pages_is_flagged():
    """A member whose table does not hold the leader's pages over the shared
    length: PA_DEVERR_BAD_BLOCK; the other groups are unaffected."""
    lens = [300, 310, 280, 150, 170]
    case, starts, shared = _grouped_case("cascade-badblock", 1280, 8, 4, 128, 16, lens, [3, 2],
                                         [256, 128])
    case.block_tables[1, 3] = case.block_tables[1, 10]   # page 3 of member 1 differs
    out, flags, _ = _cascade(case, starts, shared)
    assert flags == pa.PA_DEVERR_BAD_BLOCK
    want = _oracle(case)
    check_tolerance(out_as_f64(out)[3:], want[3:], "bf16", case.name)


def test_zero_length_and_single_token_sequences():
    """Sequences of length 0 (zero rows) and 1 in a group that shares nothing,
    next to a sharing group."""
    lens = [0, 1, 33, 200, 250]
    case, starts, shared = _grouped_case("cascade-short", 1290, 8, 8, 128, 16, lens, [3, 2],
                                         [0, 192])
    case.slot_mapping[0] = -1                             # nothing to write for length 0
    out, flags, _ = _cascade(case, starts, shared)
    assert flags == 0
    got = out_as_f64(out)
    assert np.all(got[0] == 0)
    check_tolerance(got[1:], _oracle(case)[1:], "bf16", case.name)


def test_host_refusals():
    case, starts, shared = _grouped_case("cascade-refuse", 1300, 16, 1, 128, 16, [40, 40], [2],
                                         [32])
    q = to_dev(case.q, True)
    kc = to_dev(case.k_cache, True)
    out = torch.empty_like(q)
    args = (to_dev(case.block_tables), to_dev(case.context_lens))
    with pytest.raises(pa.PaError) as e:                  # 16 query heads per kv head
        pa.pa_decode_cascade(out, q, kc, kc, *args, to_dev(starts), to_dev(shared), case.scale,
                             1, 40)
    assert "unsupported" in str(e.value)
    with pytest.raises(ValueError):                       # group_start must have G + 1 entries
        pa.pa_decode_cascade(out, q, kc, kc, *args, to_dev(shared), to_dev(shared), case.scale,
                             1, 40)


@pytest.mark.parametrize("Hq,Hkv,members", [(16, 4, 24), (16, 2, 17), (8, 8, 70)])
def test_groups_wider_than_one_row_set(Hq, Hkv, members):
    """More than 64 rows in a group (members x query heads per kv head): the
    prefix work is split into several row sets (96, 136 and 70 rows here),
    the last one partial."""
    rng = np.random.default_rng(1310 + members)
    shared = 320                                          # 5 stages of 64 tokens
    lens = [shared + int(x) for x in rng.integers(1, 90, size=members)] + [150, 60]
    case, starts, shared_lens = _grouped_case(f"cascade-wide-{Hq}-{Hkv}-{members}", 1310 + members,
                                              Hq, Hkv, 128, 16, lens, [members, 2], [shared, 48])
    out, flags, _ = _cascade(case, starts, shared_lens)
    assert flags == 0
    check_tolerance(out_as_f64(out), _oracle(case), "bf16", case.name)


def test_more_groups_than_the_plan_caches():
    """2100 groups (the plan keeps at most 2048 in shared memory): pairs of
    sequences sharing one page, and singles."""
    rng = np.random.default_rng(1320)
    sizes = [2 if i % 3 == 0 else 1 for i in range(2100)]
    lens = []
    for s in sizes:
        lens += [16 + int(x) for x in rng.integers(1, 40, size=s)]
    case, starts, shared = _grouped_case("cascade-many-groups", 1320, 8, 8, 64, 16, lens, sizes,
                                         [16 if s == 2 else 0 for s in sizes])
    out, flags, _ = _cascade(case, starts, shared)
    assert flags == 0
    check_tolerance(out_as_f64(out), _oracle(case), "bf16", case.name)


@pytest.mark.parametrize("num_seqs", [129, 257, 513])
def test_plan_block_sizes(num_seqs):
    """The plan runs with the smallest block (128, 256, 512 or 1024 threads)
    that takes every sequence and group in one pass: batches just past each
    step, in groups of eight sharing two pages, the last group partial."""
    rng = np.random.default_rng(1330 + num_seqs)
    sizes = [8] * (num_seqs // 8) + ([num_seqs % 8] if num_seqs % 8 else [])
    lens = [32 + int(x) for x in rng.integers(1, 40, size=num_seqs)]
    case, starts, shared = _grouped_case(f"cascade-plan-{num_seqs}", 1330 + num_seqs, 8, 4, 64, 16,
                                         lens, sizes, [32] * len(sizes))
    out, flags, _ = _cascade(case, starts, shared)
    assert flags == 0
    check_tolerance(out_as_f64(out), _oracle(case), "bf16", case.name)


@pytest.mark.parametrize("limit", [0, 64])
def test_expired_waits_in_the_prefix_kernel_leave_the_context_usable(limit):
    """The shared-prefix kernel's pipeline waits (TMA rings, tensor-core
    completions, tensor-memory hand-overs) are bounded: with the bound cut to
    `limit` polls they expire, the call reports PA_DEVERR_TIMEOUT and returns
    (tensor memory released, copies drained), and the next call with the normal
    bound is exact."""
    case, starts, shared = _grouped_case("cascade-timeout", 1280, 32, 8, 128, 16, LENS, GROUPS,
                                         SHARED)
    try:
        pa.pa_debug_set_wait_limit(limit)
        _, flags, _ = _cascade(case, starts, shared)
    finally:
        pa.pa_debug_set_wait_limit(-1)
    assert flags & ~pa.PA_DEVERR_TIMEOUT == 0
    if limit == 0:
        assert flags & pa.PA_DEVERR_TIMEOUT
    out, flags, _ = _cascade(case, starts, shared)
    assert flags == 0
    check_tolerance(out_as_f64(out), _oracle(case), "bf16", case.name)
