"""GPU parity of pa_decode_shared_prefix (groups of sequences sharing prefix blocks)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import DeviceBatch, compare, oracle_scatter, run_decode, run_scatter, sampled_oracle_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


def family_groups(b):
    """group_start / shared blocks of the agentic families (forks share floor(0.96 * blocks))."""
    starts, shared = [0], []
    for fam in b.families:
        assert fam == list(range(starts[-1], starts[-1] + len(fam)))
        nb = -(-int(b.seq_lens[fam[0]]) // b.block_size)
        shared.append(int(np.floor(0.96 * nb)) if len(fam) > 1 else 0)
        starts.append(starts[-1] + len(fam))
    return np.array(starts, np.int32), np.array(shared, np.int32)


def run_shared(pa, db, starts, shared, max_group=8, partition_size=0):
    b = db.b
    out = torch.empty_like(db.q)
    ws = pa.workspace_tensor(pa.pa_decode_shared_prefix_workspace_size(
        b.num_seqs, len(shared), b.num_q_heads, b.num_kv_heads, b.head_size, b.max_seq_len, b.block_size,
        partition_size), DEV)
    pa.pa_decode_shared_prefix(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws,
                               torch.from_numpy(starts).to(DEV), torch.from_numpy(shared).to(DEV), max_group,
                               db.k_scale, db.v_scale, partition_size)
    return out


def _parity(pa, b, starts, shared, partition_size=0, max_group=8):
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    out = run_shared(pa, db, starts, shared, max_group, partition_size)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, b.kv_dtype, b.block_tables, b.seq_lens, b.block_size,
                              b.scale, b.k_scale, b.v_scale)
    compare(out, ref, b.kv_dtype, where=b.name)
    plain = run_decode(pa, db, partition_size)
    return out, plain


@pytest.mark.parametrize("part", [0, 32, 160])
def test_agentic_families_scaled_down(pa, part):
    b = workloads.agentic(seed=7, host_cache=True, scale_lengths=1 / 400.0)
    starts, shared = family_groups(b)
    out, plain = _parity(pa, b, starts, shared, part)
    assert (out.double() - plain.double()).abs().max().item() < 1e-2


@pytest.mark.parametrize("kv,per_head", [("fp8_e4m3", False), ("fp8_e5m2", False), ("fp8_e4m3", True)])
def test_fp8_groups_and_clamped_share(pa, kv, per_head):
    # two groups of 3 declaring 5 shared blocks and one singleton; the last member of
    # group 1 holds only 3 full blocks, so that group's shared length is clamped to 3
    lens = [300, 300, 300, 200, 210, 100, 77]
    shared_map = {1: (0, 5), 2: (0, 5), 4: (3, 5), 5: (3, 3)}
    scales = [0.011, 2.0 ** -6, 0.3, 2.0 ** -2, 0.05, 1.0, 2.0 ** -9, 0.0071] if per_head else 2.0 ** -6
    b = workloads.build("fp8grp", 21, lens, [1] * 7, 32, 8, 128, 32, kv, shared=shared_map, fp8_scale=scales)
    starts = np.array([0, 3, 6, 7], np.int32)
    shared = np.array([5, 5, 0], np.int32)
    _parity(pa, b, starts, shared, 64)


def test_groups_larger_than_bound_share_nothing(pa):
    b = workloads.agentic(seed=9, host_cache=True, scale_lengths=1 / 400.0)
    starts, shared = family_groups(b)
    out, plain = _parity(pa, b, starts, shared, 64, max_group=4)  # families of 5 exceed the bound
    assert torch.equal(out, plain) or (out.double() - plain.double()).abs().max().item() < 1e-2


def _unused_blocks(b, n, rng):
    used = set(int(x) for x in b.block_tables.ravel() if x >= 0)
    free = np.array([p for p in range(b.num_blocks) if p not in used], np.int64)
    assert len(free) >= n
    return [int(x) for x in rng.choice(free, size=n, replace=False)]


def _repoint(b, seq, blocks, rng):
    """Point `seq`'s entries for the given logical blocks at unused physical blocks (a
    copy-on-write that the group declaration does not know about); the cache there
    holds other values, so the output changes."""
    for j, p in zip(blocks, _unused_blocks(b, len(blocks), rng)):
        b.block_tables[seq, j] = p


def _stale_parity(pa, b, starts, shared, partition_size, max_group=8):
    """Values against the oracle, which reads every sequence's own table; the call sets
    only the diagnostic bit."""
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    out = run_shared(pa, db, starts, shared, max_group, partition_size)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == pa.PA_ERRFLAG_SHARED_MISMATCH
    k_ref, v_ref = oracle_scatter(b)
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, b.kv_dtype, b.block_tables, b.seq_lens, b.block_size,
                              b.scale, b.k_scale, b.v_scale)
    compare(out, ref, b.kv_dtype, where=b.name)
    plain = run_decode(pa, db, partition_size)
    torch.cuda.synchronize()
    assert (out.double() - plain.double()).abs().max().item() < 1e-2


@pytest.mark.parametrize("part", [0, 64])
def test_stale_and_wrong_share_declarations_bf16(pa, part):
    """[AGENTIC] "統一分頁 + 共用池": shared blocks are copied on write, so a group's
    declaration can be stale.  Family 0: one fork copied the last two declared blocks;
    family 1: one fork copied a block in the middle and another fork the first; family
    2: one fork shares nothing (every declared entry differs)."""
    b = workloads.agentic(seed=7, host_cache=True, scale_lengths=1 / 400.0)
    starts, shared = family_groups(b)
    rng = np.random.default_rng(5)
    f0, f1, f2 = b.families[0], b.families[1], b.families[2]
    _repoint(b, f0[2], [int(shared[0]) - 2, int(shared[0]) - 1], rng)
    _repoint(b, f1[4], [int(shared[1]) // 2], rng)
    _repoint(b, f1[1], [0], rng)
    _repoint(b, f2[3], list(range(int(shared[2]))), rng)
    _stale_parity(pa, b, starts, shared, part)


@pytest.mark.parametrize("kv", ["fp8_e4m3", "nvfp4"])
def test_stale_share_declarations_scaled_caches(pa, kv):
    """The member-warp shared-prefix kernel (FP8 and NVFP4 caches) under the same
    stale and wrong declarations: a group of 3 declaring 5 shared blocks where the
    last member copied blocks 1 and 4, and a group of 3 whose middle member shares
    nothing."""
    lens = [300, 300, 300, 260, 280, 290, 77]
    shared_map = {1: (0, 5), 2: (0, 5), 4: (3, 5), 5: (3, 5)}
    b = workloads.build("stale_" + kv, 25, lens, [1] * 7, 32, 8, 128, 32, kv, shared=shared_map)
    rng = np.random.default_rng(6)
    _repoint(b, 2, [1, 4], rng)
    _repoint(b, 4, [0, 1, 2, 3, 4], rng)
    starts = np.array([0, 3, 6, 7], np.int32)
    shared = np.array([5, 5, 0], np.int32)
    _stale_parity(pa, b, starts, shared, 64)


def test_declared_share_that_is_not_shared(pa):
    """Sequences 0 and 1 share nothing in truth but are declared to share 4 blocks."""
    b = workloads.build("liar", 23, [200, 200, 64], [1] * 3, 16, 2, 128, 16, "bf16")
    starts = np.array([0, 2, 3], np.int32)
    shared = np.array([4, 0], np.int32)
    _stale_parity(pa, b, starts, shared, 64, max_group=4)


@pytest.mark.slow
def test_agentic_full_size_sampled(pa):
    b = workloads.agentic()
    starts, shared = family_groups(b)
    db = DeviceBatch(b, DEV)
    seqs = [b.families[0][0], b.families[1][2], b.families[2][4], b.families[3][0]]
    outs = []

    def gpu():
        run_scatter(pa, db)
        outs.append(run_shared(pa, db, starts, shared))

    k, v, tables = sampled_oracle_inputs(db, seqs, gpu)
    assert pa.pa_get_error_flags() == 0
    ref = oracle.paged_decode(b.q, b.q_dtype, k, v, b.kv_dtype, tables, b.seq_lens, b.block_size, b.scale,
                              seqs=seqs)
    compare(outs[0], ref, b.kv_dtype, rows=seqs, where="agentic shared prefix")


@pytest.mark.parametrize("part", [32, 0])
def test_many_groups_more_items_than_ctas(pa, part):
    """40 groups of 1-4 sequences with random lengths and shares: with 32-token
    partitions there are far more (group, KV head, partition) items than resident
    CTAs, so each CTA of the shared tiles runs many items of different sizes in turn
    (and skips the items of singleton groups and past each group's share)."""
    rng = np.random.default_rng(77)
    lens, shared_map, starts, shared = [], {}, [0], []
    for _ in range(40):
        size = int(rng.integers(1, 5))
        base = len(lens)
        L = int(rng.integers(50, 400))
        nsh = int(rng.integers(0, L // 16 + 1))
        for m in range(size):
            lens.append(L + int(rng.integers(0, 40)) if m else L)
            if m:
                shared_map[base + m] = (base, nsh)
        starts.append(len(lens))
        shared.append(nsh if size > 1 else 0)
    b = workloads.build("many_groups", 79, lens, [1] * len(lens), 16, 4, 128, 16, "bf16", shared=shared_map)
    _parity(pa, b, np.array(starts, np.int32), np.array(shared, np.int32), part, max_group=4)


@pytest.mark.parametrize("offsets", [[1], [2], [0, 1], [3, 4], [6, 7], [5]], ids=lambda o: "at_" + "_".join(map(str, o)))
def test_stale_block_at_each_position_of_a_block_pair(pa, offsets):
    """The bf16 tiles take whole shared blocks two at a time; a block a member copied
    on write (read as stages of its own) can fall first or second in a pair, or end
    an item of odd length.  Groups of 3 over 8-block partitions (128 tokens), the
    stale blocks at the given offsets of each partition of the last member."""
    lens = [600, 600, 600, 555]
    shared_map = {1: (0, 35), 2: (0, 35)}  # 35 blocks: the last partition holds 3
    b = workloads.build("pair_" + "_".join(map(str, offsets)), 31, lens, [1] * 4, 16, 2, 128, 16, "bf16",
                        shared=shared_map)
    rng = np.random.default_rng(7)
    stale = [8 * z + o for z in range(35 // 8 + 1) for o in offsets if 8 * z + o < 35]
    _repoint(b, 2, stale, rng)
    starts = np.array([0, 3, 4], np.int32)
    shared = np.array([35, 0], np.int32)
    _stale_parity(pa, b, starts, shared, 128)
