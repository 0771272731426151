"""GPU parity of the scatter and PagedAttention decode against the fp64 oracle.

Every test calls the CUDA library through its C ABI (Python binding) and compares
element by element with the oracle run on the same seeded inputs.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import (DeviceBatch, compare, oracle_scatter, run_decode, run_scatter,
                     sampled_oracle_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


DEV = "cuda:0"


def _full_parity(pa, b, partition_size=0):
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    out = run_decode(pa, db, partition_size)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    assert np.array_equal(workloads.torch_to_bits(db.kc, b.kv_dtype), k_ref), "K cache bytes"
    assert np.array_equal(workloads.torch_to_bits(db.vc, b.kv_dtype), v_ref), "V cache bytes"
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, b.kv_dtype, b.block_tables, b.seq_lens,
                              b.block_size, b.scale, b.k_scale, b.v_scale)
    return compare(out, ref, b.kv_dtype, where=b.name)


def test_tiny_workload(pa):
    _full_parity(pa, workloads.tiny())


RAGGED = [1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 511, 1000]

CASES = [
    # (name, kv dtype, Hq, Hkv, d, bs, lens, partition)
    ("bf16_g4_d128_bs16", "bf16", 32, 8, 128, 16, RAGGED, 0),
    ("bf16_g4_split64", "bf16", 32, 8, 128, 16, RAGGED, 64),
    ("bf16_g8_split16", "bf16", 16, 2, 128, 16, RAGGED, 16),
    ("bf16_g1_d64", "bf16", 4, 4, 64, 16, RAGGED, 128),
    ("bf16_g16_two_groups", "bf16", 32, 2, 128, 16, RAGGED, 256),
    ("bf16_g6_bs32", "bf16", 12, 2, 128, 32, RAGGED, 64),
    ("bf16_d64_bs32", "bf16", 8, 2, 64, 32, RAGGED, 0),
    ("f16_g4_d128", "f16", 32, 8, 128, 16, RAGGED, 96),
    ("f32_g4_generic", "f32", 16, 4, 128, 16, RAGGED, 64),
    ("f32_d96_generic", "f32", 6, 3, 96, 8, RAGGED, 24),
    ("bf16_d256_generic", "bf16", 8, 2, 256, 16, RAGGED[:8], 0),
    ("fp8_g4_bs32", "fp8_e4m3", 32, 8, 128, 32, RAGGED, 64),
    ("fp8_g8_bs16", "fp8_e4m3", 16, 2, 128, 16, RAGGED, 0),
    ("fp8_f16q", "fp8_e4m3", 8, 2, 128, 32, RAGGED, 32),
    ("fp8e5m2_g4_bs32", "fp8_e5m2", 32, 8, 128, 32, RAGGED, 64),
    ("fp8e5m2_g8_bs16", "fp8_e5m2", 16, 2, 128, 16, RAGGED, 0),
    ("fp8e5m2_f32q_generic", "fp8_e5m2", 8, 2, 128, 16, RAGGED, 48),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_parity(pa, case):
    name, kv, hq, hkv, d, bs, lens, part = case
    q_dtype = {"fp8_f16q": "f16", "fp8e5m2_f32q_generic": "f32"}.get(name)
    b = workloads.build(name, 100 + len(name), lens, [1] * len(lens), hq, hkv, d, bs, kv, q_dtype=q_dtype,
                        src_dtype=q_dtype)
    _full_parity(pa, b, part)


def test_fp8_scatter_matches_cuda_conversion(pa):
    """Quantisation of ties, subnormals and out-of-range values: oracle == CUDA's e4m3 conversion."""
    mags = oracle.e4m3_table()[:127]
    vals = np.concatenate([mags, (mags[:-1] + mags[1:]) / 2, [500.0, 1e6, 464.0, 463.9, 2.0 ** -10, 3e-4]])
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    n = -(-vals.size // 128) * 128
    x = np.zeros(n, np.float32)
    x[: vals.size] = vals
    tokens = n // 128
    for scale in (1.0, 0.37):
        key = torch.from_numpy(x.reshape(tokens, 1, 128)).to(DEV)
        kc = torch.zeros((tokens, 1, 16, 128), dtype=torch.uint8, device=DEV)
        vc = torch.zeros_like(kc)
        slots = torch.arange(tokens, dtype=torch.int64, device=DEV) * 16 + 3
        sc = torch.tensor([scale], dtype=torch.float32, device=DEV)
        pa.pa_reshape_and_cache(key, key, kc, vc, slots, sc, sc)
        got = kc[:, 0, 3, :].cpu().numpy().reshape(-1)
        ref = oracle.quantize_e4m3(x.astype(np.float64), scale)
        assert np.array_equal(got, ref), f"scale {scale}: {np.count_nonzero(got != ref)} codes differ"


def test_fp8_e5m2_scatter_matches_cuda_conversion(pa):
    """e5m2 quantisation of ties, subnormals and out-of-range values: oracle == CUDA's conversion."""
    mags = oracle.e5m2_table()[:124]
    vals = np.concatenate([mags, (mags[:-1] + mags[1:]) / 2, [61440.0, 1e9, 60000.0, 2.0 ** -18, 3e-6]])
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    n = -(-vals.size // 128) * 128
    x = np.zeros(n, np.float32)
    x[: vals.size] = vals
    tokens = n // 128
    for scale in (1.0, 0.37):
        key = torch.from_numpy(x.reshape(tokens, 1, 128)).to(DEV)
        kc = torch.zeros((tokens, 1, 16, 128), dtype=torch.float8_e5m2, device=DEV)
        vc = torch.zeros_like(kc)
        slots = torch.arange(tokens, dtype=torch.int64, device=DEV) * 16 + 3
        sc = torch.tensor([scale], dtype=torch.float32, device=DEV)
        pa.pa_reshape_and_cache(key, key, kc, vc, slots, sc, sc)
        got = kc[:, 0, 3, :].view(torch.uint8).cpu().numpy().reshape(-1)
        ref = oracle.quantize_e5m2(x.astype(np.float64), scale)
        assert np.array_equal(got, ref), f"scale {scale}: {np.count_nonzero(got != ref)} codes differ"


def test_scatter_padding_and_bad_slot_flag(pa):
    b = workloads.build("pad", 7, [40, 3], [2, 1], 8, 2, 64, 16, "bf16")
    db = DeviceBatch(b, DEV)
    slots = db.slots.clone()
    slots[0] = -1
    slots[1] = b.num_blocks * b.block_size + 5  # out of range: skipped and flagged
    before_k = workloads.torch_to_bits(db.kc, "bf16").copy()
    pa.pa_reshape_and_cache(db.key, db.value, db.kc, db.vc, slots)
    flags = pa.pa_get_error_flags()
    assert flags == pa.PA_ERRFLAG_SLOT
    after = workloads.torch_to_bits(db.kc, "bf16")
    s2 = int(b.slot_mapping[2])
    assert np.array_equal(after[s2 // 16, :, s2 % 16], b.key[2])
    changed = np.argwhere(np.any(after != before_k, axis=-1))
    assert len(changed) == b.num_kv_heads  # only token 2's rows


def test_block_permutation_invariance_on_gpu(pa):
    """Same logical K/V under two physical placements -> bitwise identical outputs."""
    b = workloads.build("perm", 9, [300, 45, 700], [1, 1, 1], 32, 8, 128, 16, "bf16", pool_factor=3.0)
    db = DeviceBatch(b, DEV)
    out1 = run_decode(pa, db, 64)
    perm = np.random.default_rng(1).permutation(b.num_blocks)
    inv = np.argsort(perm)
    kc2 = db.kc[torch.from_numpy(perm).to(DEV)]
    vc2 = db.vc[torch.from_numpy(perm).to(DEV)]
    tables2 = b.block_tables.copy()
    m = tables2 >= 0
    tables2[m] = inv[tables2[m]]
    db2 = DeviceBatch(b, DEV, cache=(kc2.contiguous(), vc2.contiguous()))
    db2.tables = torch.from_numpy(tables2).to(DEV)
    out2 = run_decode(pa, db2, 64)
    assert torch.equal(out1, out2)


def test_shared_blocks_give_identical_outputs(pa):
    b = workloads.agentic(seed=3, host_cache=True, scale_lengths=1 / 500.0)
    fam = b.families[0]
    b.q[fam[1]] = b.q[fam[0]]
    b.block_tables[fam[1]] = b.block_tables[fam[0]]
    db = DeviceBatch(b, DEV)
    out = run_decode(pa, db, 32)
    assert torch.equal(out[fam[0]], out[fam[1]])
    assert pa.pa_get_error_flags() == 0


def test_bad_block_table_entry_is_flagged_not_read(pa):
    b = workloads.build("badtab", 5, [100, 50], [1, 1], 8, 2, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    t = db.tables.clone()
    t[0, 2] = b.num_blocks + 1000
    t[1, 0] = -7
    db.tables = t
    run_decode(pa, db, 32)
    assert pa.pa_get_error_flags() & pa.PA_ERRFLAG_BLOCK_TABLE


def test_bad_seq_len_zero_row_and_flag(pa):
    b = workloads.build("badlen", 5, [100, 50, 20], [1, 1, 1], 8, 2, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    db.lens = torch.tensor([100, 0, 20], dtype=torch.int32, device=DEV)
    out = run_decode(pa, db)
    assert pa.pa_get_error_flags() & pa.PA_ERRFLAG_SEQ_LEN
    assert torch.count_nonzero(out[1]) == 0
    ref = oracle.paged_decode(b.q, "bf16", b.k_cache, b.v_cache, "bf16", b.block_tables, [100, 1, 20], 16,
                              b.scale, seqs=[0, 2])
    compare(out, ref, "bf16", rows=[0, 2], where="bad seq_len")


def test_host_side_argument_errors(pa):
    b = workloads.build("args", 5, [10], [1], 8, 2, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    out = torch.empty_like(db.q)
    ws = pa.workspace_tensor(256, DEV)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    big = pa.workspace_tensor(1 << 20, DEV)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, big,
                     partition_size=24)  # not a multiple of block_size
    assert e.value.status == pa.PA_ERR_INVALID_ARG


# ------------------------------------------------------------ full-size workloads (sampled rows)

def _sampled_full_size(pa, b, seqs):
    db = DeviceBatch(b, DEV)
    outs = []

    def gpu():
        run_scatter(pa, db)
        outs.append(run_decode(pa, db))

    k, v, tables = sampled_oracle_inputs(db, seqs, gpu)
    assert pa.pa_get_error_flags() == 0
    ref = oracle.paged_decode(b.q, b.q_dtype, k, v, b.kv_dtype, tables, b.seq_lens, b.block_size, b.scale,
                              b.k_scale, b.v_scale, seqs=seqs)
    return compare(outs[0], ref, b.kv_dtype, rows=seqs, where=b.name)


def _spread_by_length(b, n):
    """n sequences spread evenly over the batch's length ranks, the shortest and the
    longest included."""
    order = np.argsort(b.seq_lens, kind="stable")
    picks = np.unique(np.round(np.linspace(0, len(order) - 1, n)).astype(int))
    return sorted(int(order[i]) for i in picks)


@pytest.mark.slow
def test_llama_full_size_every_row(pa):
    """Every one of the 64 sequences of the full-size Llama-shaped batch, with the
    default partitioning the bench uses, against the oracle."""
    b = workloads.llama()
    _sampled_full_size(pa, b, list(range(b.num_seqs)))


@pytest.mark.slow
def test_agentic_full_size_sampled(pa):
    b = workloads.agentic()
    fam = b.families
    _sampled_full_size(pa, b, [fam[0][0], fam[0][3], fam[3][0]])


@pytest.mark.slow
def test_fp8_full_size_sampled(pa):
    """16 of the 256 sequences of the full-size FP8 batch, spread over the length range
    from the shortest to the longest."""
    b = workloads.fp8()
    seqs = _spread_by_length(b, 16)
    lens = b.seq_lens[seqs]
    assert len(seqs) == 16 and lens.min() == b.seq_lens.min() and lens.max() == b.seq_lens.max()
    _sampled_full_size(pa, b, seqs)


@pytest.mark.slow
def test_fp8_e5m2_full_size_sampled(pa):
    b = workloads.fp8_e5m2()
    _sampled_full_size(pa, b, [1, 128, 254])


PER_HEAD = [0.011, 2.0 ** -6, 0.3, 2.0 ** -2, 0.05, 1.0, 2.0 ** -9, 0.0071]


@pytest.mark.parametrize("kv,q_dtype", [("fp8_e4m3", None), ("fp8_e5m2", None), ("fp8_e4m3", "f32")])
def test_per_head_fp8_scales(pa, kv, q_dtype):
    """One scale per KV head (scatter codes and decode) on the tensor-core and generic paths."""
    b = workloads.build("phs_" + kv, 131, RAGGED, [1] * len(RAGGED), 32, 8, 128, 32, kv, q_dtype=q_dtype,
                        src_dtype=q_dtype, fp8_scale=PER_HEAD)
    assert np.ndim(b.k_scale) == 1
    _full_parity(pa, b, 64)
