"""GPU parity at the edges of the supported sizes.

The agentic workload's context lengths are clipped to [32K, 256K] tokens
([AGENTIC] "Agentic 工作負載長什麼樣": input median about 142K tokens), so the
longest context the workloads produce is 262,144 tokens.  These tests run decode
and a chunked-prefill step at exactly that length (block-aligned and one token
short of it), with the default partitions and with 16-token partitions (16,384
partial states per row for the merge), FP8 codes at the same length, a batch of
4,096 one-token sequences (the degenerate case: the output is the new value),
and the scatter into the pool's first and last slots.  Every comparison is
against the oracle on the same inputs: sampled rows where the whole batch is too
large for it, every row otherwise.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import (DeviceBatch, compare, oracle_scatter, run_decode, run_scatter, run_varlen,
                     sampled_oracle_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LONGEST = 262144  # the agentic length distribution's upper clip, in tokens


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


def _decode_sampled(pa, b, seqs, partition_size=0):
    db = DeviceBatch(b, DEV)
    outs = []

    def gpu():
        run_scatter(pa, db)
        outs.append(run_decode(pa, db, partition_size))

    k, v, tables = sampled_oracle_inputs(db, seqs, gpu)
    assert pa.pa_get_error_flags() == 0
    ref = oracle.paged_decode(b.q, b.q_dtype, k, v, b.kv_dtype, tables, b.seq_lens, b.block_size, b.scale,
                              b.k_scale, b.v_scale, seqs=seqs)
    return compare(outs[0], ref, b.kv_dtype, rows=seqs, where=f"{b.name} part {partition_size}")


@pytest.mark.slow
@pytest.mark.parametrize("part", [0, 16])
def test_decode_at_the_longest_context(pa, part):
    # block-aligned, one token short of it (a one-token tail block), and a one-token sequence
    b = workloads.build("longest", 61, [LONGEST, LONGEST - 1, 1], [1, 1, 1], 16, 2, 128, 16, "bf16",
                        host_cache=False)
    assert b.max_blocks_per_seq == LONGEST // 16
    _decode_sampled(pa, b, [0, 1, 2], part)


@pytest.mark.slow
def test_fp8_decode_at_the_longest_context(pa):
    b = workloads.build("longest_fp8", 62, [LONGEST, 40000, LONGEST - 33], [1, 1, 1], 8, 2, 128, 32,
                        "fp8_e4m3", host_cache=False)
    _decode_sampled(pa, b, [0, 1, 2])


@pytest.mark.slow
def test_prefill_chunk_ending_at_the_longest_context(pa):
    """A 512-token chunk whose last token sits at position 262,143, beside decode rows."""
    b = workloads.build("longest_varlen", 63, [LONGEST, 3000, LONGEST - 1], [512, 1, 1], 16, 2, 128, 16,
                        "bf16", host_cache=False)
    db = DeviceBatch(b, DEV)
    qsl = b.query_start_loc
    rng = np.random.default_rng(5)
    rows = [0, 1, 255, 256, 511] + [int(x) for x in rng.integers(0, 512, 4)] + [int(qsl[1]), int(qsl[2])]
    outs = []

    def gpu():
        run_scatter(pa, db)
        outs.append(run_varlen(pa, db))

    k, v, tables = sampled_oracle_inputs(db, [0, 1, 2], gpu)
    assert pa.pa_get_error_flags() == 0
    ref = oracle.paged_varlen(b.q, b.q_dtype, k, v, b.kv_dtype, tables, b.query_start_loc, b.seq_lens,
                              b.block_size, b.scale, True, b.k_scale, b.v_scale, rows=rows)
    compare(outs[0], ref, b.kv_dtype, rows=sorted(set(rows)), where="longest varlen")


def test_many_one_token_sequences(pa):
    """4,096 sequences of one token each: every output row is that token's own value."""
    n = 4096
    b = workloads.build("one_token", 64, [1] * n, [1] * n, 32, 8, 128, 16, "bf16", pool_factor=1.0)
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    out = run_decode(pa, db)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    assert np.array_equal(workloads.torch_to_bits(db.kc, b.kv_dtype), k_ref)
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, b.kv_dtype, b.block_tables, b.seq_lens,
                              b.block_size, b.scale)
    compare(out, ref, b.kv_dtype, where="one-token sequences")
    # closed form: a single key takes the whole weight, so head h returns value row h // G
    v64 = oracle.decode_bits(b.value, b.src_dtype)                      # [n][Hkv][d]
    want = np.repeat(v64, b.num_q_heads // b.num_kv_heads, axis=1)      # [n][Hq][d]
    assert np.array_equal(out.double().cpu().numpy(), want)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "nvfp4"])
def test_scatter_into_the_first_and_last_slots(pa, kv):
    b = workloads.build("edge_slots_" + kv, 65, [40, 3, 17], [2, 1, 1], 8, 2, 128, 16, kv)
    last = b.num_blocks * b.block_size - 1
    b.slot_mapping[:] = [0, last, -1, last - b.block_size]
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    assert np.array_equal(workloads.torch_to_bits(db.kc, b.kv_dtype), k_ref)
    assert np.array_equal(workloads.torch_to_bits(db.vc, b.kv_dtype), v_ref)
