"""GPU parity of the flattened variable-length (chunked prefill + decode) attention."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import (DeviceBatch, compare, oracle_scatter, run_decode, run_scatter, run_varlen,
                     sampled_oracle_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


def _varlen_parity(pa, b, partition_size=0, causal=True):
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    out = run_varlen(pa, db, partition_size, causal)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    assert np.array_equal(workloads.torch_to_bits(db.kc, b.kv_dtype), k_ref)
    assert np.array_equal(workloads.torch_to_bits(db.vc, b.kv_dtype), v_ref)
    ref = oracle.paged_varlen(b.q, b.q_dtype, k_ref, v_ref, b.kv_dtype, b.block_tables, b.query_start_loc,
                              b.seq_lens, b.block_size, b.scale, causal, b.k_scale, b.v_scale)
    return compare(out, ref, b.kv_dtype, where=b.name)


VARLEN_CASES = [
    # (name, kv, Hq, Hkv, d, bs, lens, q_lens, partition, causal)
    ("mixed_bf16", "bf16", 32, 8, 128, 16, [700, 37, 1, 300, 90], [64, 1, 1, 300, 17], 64, True),
    ("mixed_bf16_default_part", "bf16", 32, 8, 128, 16, [700, 37, 1, 300, 90], [64, 1, 1, 300, 17], 0, True),
    ("prefill_only_g8", "bf16", 16, 2, 128, 16, [129, 200, 33], [129, 50, 33], 32, True),
    ("non_causal", "bf16", 8, 2, 128, 16, [100, 40], [30, 40], 32, False),
    ("empty_requests", "bf16", 8, 2, 64, 16, [10, 50, 7, 70], [0, 5, 0, 1], 16, True),
    ("f16_bs32", "f16", 12, 4, 128, 32, [400, 33, 65], [100, 1, 65], 64, True),
    ("f32_generic", "f32", 8, 2, 64, 16, [200, 17, 64], [40, 1, 64], 48, True),
    ("fp8_mixed", "fp8_e4m3", 32, 8, 128, 32, [500, 64, 33], [70, 1, 33], 64, True),
    ("prefill_g16_two_groups", "bf16", 32, 2, 128, 16, [300, 80], [150, 80], 64, True),
    ("prefill_g3_padded", "bf16", 6, 2, 128, 32, [200, 45], [100, 45], 32, True),
    ("prefill_g1_d64", "bf16", 4, 4, 64, 16, [130, 66], [70, 66], 0, True),
    ("prefill_ragged_tiles", "bf16", 32, 8, 128, 16, [97, 33, 1000], [97, 31, 45], 48, True),
    ("prefill_split_k_default", "bf16", 16, 4, 128, 16, [20000, 17000, 40], [100, 33, 1], 0, True),
    ("non_causal_g8", "f16", 16, 2, 128, 16, [250, 90], [60, 90], 64, False),
    ("prefill_bs64", "bf16", 16, 4, 128, 64, [300, 129, 64], [150, 129, 1], 128, True),
    ("prefill_bs64_d64_f16", "f16", 8, 2, 64, 64, [513, 70], [200, 70], 0, True),
    ("prefill_part_not_chunk_multiple", "bf16", 8, 2, 128, 32, [1000, 161], [230, 161], 96, True),
    ("fp8_prefill_split_default", "fp8_e4m3", 32, 8, 128, 16, [20000, 3000, 40], [300, 129, 1], 0, True),
    ("fp8_prefill_ragged_part48", "fp8_e4m3", 32, 8, 128, 16, [97, 33, 1000], [97, 31, 45], 48, True),
    ("fp8_prefill_noncausal_bs64", "fp8_e4m3", 16, 2, 128, 64, [250, 90], [60, 90], 64, False),
    ("fp8e5m2_prefill_mixed", "fp8_e5m2", 32, 8, 128, 16, [2000, 33, 700, 1], [300, 1, 64, 1], 0, True),
    # more (item, KV head) tiles than the first persistent grid has CTAs, beside decode rows
    ("mha_g1_many_tiles", "bf16", 8, 8, 128, 16, [1000, 700, 600, 520, 800, 900, 515, 640, 300, 1],
     [512, 512, 512, 512, 512, 512, 512, 512, 1, 1], 0, True),
    ("g2_f16_bs32", "f16", 8, 4, 128, 32, [513, 90, 1200], [257, 90, 1], 64, True),
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=[c[0] for c in VARLEN_CASES])
def test_varlen_parity(pa, case):
    name, kv, hq, hkv, d, bs, lens, q_lens, part, causal = case
    b = workloads.build(name, 300 + len(name), lens, q_lens, hq, hkv, d, bs, kv, causal=causal)
    _varlen_parity(pa, b, part, causal)


def test_fp8_prefill_with_f16_queries(pa):
    b = workloads.build("fp8_f16q_pf", 71, [700, 37, 300], [64, 1, 300], 32, 8, 128, 32, "fp8_e4m3",
                        q_dtype="f16", src_dtype="f16")
    _varlen_parity(pa, b, 64, True)


def test_varlen_single_tokens_equals_decode(pa):
    lens = [1, 17, 300, 1000, 64]
    b = workloads.build("eq", 77, lens, [1] * len(lens), 32, 8, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    a = run_decode(pa, db, 64)
    v = run_varlen(pa, db, 64)
    assert torch.equal(a, v)


def test_mixed_workload_scaled_down(pa):
    """The mixed continuous-batching step with every length scaled by 1/64 (same structure)."""
    b = workloads.mixed(seed=3, host_cache=True, scale_lengths=1 / 64.0, chunk=64, n_decode=32)
    _varlen_parity(pa, b)


def test_bad_query_start_loc_flagged(pa):
    b = workloads.build("badq", 3, [40, 30], [5, 3], 8, 2, 64, 16, "bf16")
    db = DeviceBatch(b, DEV)
    db.qsl = torch.tensor([0, 5, 8], dtype=torch.int32, device=DEV)
    db.lens = torch.tensor([40, 2], dtype=torch.int32, device=DEV)  # q_len 3 > seq_len 2
    run_varlen(pa, db, 16)
    assert pa.pa_get_error_flags() & pa.PA_ERRFLAG_QUERY


@pytest.mark.slow
@pytest.mark.parametrize("kind", ["mixed", "mixed_fp8", "mixed_nvfp4"])
def test_mixed_full_size_sampled(pa, kind):
    b = workloads.NAMED[kind]()
    db = DeviceBatch(b, DEV)
    qsl = b.query_start_loc
    rng = np.random.default_rng(0)
    # every prefill request's first, last and a few random rows; a few decode rows
    rows, seqs = [], [0, 1, 2, 3, 4, 50, 131]
    for r in range(4):
        lo, hi = int(qsl[r]), int(qsl[r + 1])
        rows += [lo, hi - 1] + [int(x) for x in rng.integers(lo, hi, 3)]
    rows += [int(qsl[r]) for r in (4, 50, 131)]
    outs = []

    def gpu():
        run_scatter(pa, db)
        outs.append(run_varlen(pa, db))

    k, v, tables = sampled_oracle_inputs(db, seqs, gpu)
    assert pa.pa_get_error_flags() == 0
    ref = oracle.paged_varlen(b.q, b.q_dtype, k, v, b.kv_dtype, tables, b.query_start_loc, b.seq_lens,
                              b.block_size, b.scale, True, b.k_scale, b.v_scale, rows=rows)
    compare(outs[0], ref, b.kv_dtype, rows=sorted(set(rows)), where=b.name + " full size")


@pytest.mark.parametrize("kv", ["fp8_e4m3", "fp8_e5m2"])
def test_fp8_prefill_per_head_scales(pa, kv):
    scales = [0.011, 2.0 ** -6, 0.3, 2.0 ** -2, 0.05, 1.0, 2.0 ** -9, 0.0071]
    b = workloads.build("phs_pf_" + kv, 72, [700, 37, 300, 1], [64, 1, 300, 1], 32, 8, 128, 16, kv,
                        fp8_scale=scales)
    _varlen_parity(pa, b, 0, True)
