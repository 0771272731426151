"""GPU parity of sliding-window attention (pa_decode_windowed, pa_varlen_attn_windowed).

Block-table entries of blocks wholly before a request's window are set to -1, as a
cache manager that has already released them would leave them: the kernels must
neither read nor flag them."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import DeviceBatch, compare, oracle_scatter, run_scatter

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


def _release_before_window(b, window):
    """Block tables with every block wholly before the first query's window set to -1."""
    tables = b.block_tables.copy()
    for r in range(b.num_seqs):
        q_len = int(b.query_start_loc[r + 1] - b.query_start_loc[r])
        first = max(0, int(b.seq_lens[r]) - q_len - window + 1)
        tables[r, : first // b.block_size] = -1
    return tables


def _decode(pa, db, window, part, tables):
    b = db.b
    out = torch.empty_like(db.q)
    ws = pa.workspace_tensor(pa.pa_decode_workspace_size(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_size,
                                                         b.max_seq_len, b.block_size, part), DEV)
    pa.pa_decode(out, db.q, db.kc, db.vc, torch.from_numpy(tables).to(DEV), db.lens, b.max_seq_len, b.scale, ws,
                 db.k_scale, db.v_scale, part, window=window)
    return out


def _varlen(pa, db, window, part, tables, causal=True):
    b = db.b
    out = torch.empty_like(db.q)
    ws = pa.workspace_tensor(pa.pa_varlen_workspace_size(b.num_seqs, b.total_q, b.max_query_len, b.num_q_heads,
                                                         b.num_kv_heads, b.head_size, b.max_seq_len, b.block_size,
                                                         part), DEV)
    pa.pa_varlen_attn(out, db.q, db.kc, db.vc, torch.from_numpy(tables).to(DEV), db.qsl, db.lens, b.max_query_len,
                      b.max_seq_len, b.scale, ws, causal, db.k_scale, db.v_scale, part, window=window)
    return out


DECODE_CASES = [
    # (name, kv, Hq, Hkv, d, bs, lens, window, partition)
    ("bf16_w100_split", "bf16", 32, 8, 128, 16, [700, 37, 1, 300, 4000], 100, 64),
    ("bf16_w_block", "bf16", 32, 8, 128, 16, [700, 37, 1, 300, 4000], 16, 0),
    ("bf16_w1", "bf16", 16, 2, 128, 32, [700, 37, 1, 300], 1, 64),
    ("bf16_w_long_default", "bf16", 32, 8, 128, 16, [9000, 5000, 70], 4096, 0),
    ("fp8_w300_bs32", "fp8_e4m3", 32, 8, 128, 32, [1000, 37, 301, 3000], 300, 128),
    ("f32_generic_w50", "f32", 8, 2, 64, 16, [200, 17, 64, 90], 50, 32),
    ("bf16_d64_w77", "bf16", 8, 2, 64, 16, [500, 80], 77, 48),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_decode_window_parity(pa, case):
    name, kv, hq, hkv, d, bs, lens, window, part = case
    b = workloads.build(name, 400 + len(name), lens, [1] * len(lens), hq, hkv, d, bs, kv)
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    tables = _release_before_window(b, window)
    out = _decode(pa, db, window, part, tables)
    assert pa.pa_get_error_flags(clear=True) == 0
    k_ref, v_ref = oracle_scatter(b)
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, kv, tables, b.seq_lens, bs, b.scale, b.k_scale,
                              b.v_scale, window=window)
    compare(out, ref, kv, where=name)


VARLEN_CASES = [
    # (name, kv, Hq, Hkv, d, bs, lens, q_lens, window, partition)
    ("mixed_bf16_w128", "bf16", 32, 8, 128, 16, [700, 37, 1, 300, 900], [64, 1, 1, 300, 17], 128, 64),
    ("prefill_long_w1000_default", "bf16", 16, 4, 128, 16, [20000, 3000, 40], [300, 129, 1], 1000, 0),
    ("prefill_w_below_chunk", "bf16", 8, 2, 128, 32, [1000, 161], [230, 161], 40, 96),
    ("fp8_prefill_w200", "fp8_e4m3", 32, 8, 128, 16, [2000, 33, 700], [300, 1, 64], 200, 0),
    ("f16_d64_bs64_w70", "f16", 8, 2, 64, 64, [513, 70], [200, 70], 70, 0),
    ("f32_generic_w33", "f32", 8, 2, 64, 16, [200, 17, 64], [40, 1, 64], 33, 48),
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=[c[0] for c in VARLEN_CASES])
def test_varlen_window_parity(pa, case):
    name, kv, hq, hkv, d, bs, lens, q_lens, window, part = case
    b = workloads.build(name, 500 + len(name), lens, q_lens, hq, hkv, d, bs, kv)
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    tables = _release_before_window(b, window)
    out = _varlen(pa, db, window, part, tables)
    assert pa.pa_get_error_flags(clear=True) == 0
    k_ref, v_ref = oracle_scatter(b)
    ref = oracle.paged_varlen(b.q, b.q_dtype, k_ref, v_ref, kv, tables, b.query_start_loc, b.seq_lens, bs, b.scale,
                              True, b.k_scale, b.v_scale, window=window)
    compare(out, ref, kv, where=name)


def test_window_covering_every_context_equals_full_attention(pa):
    b = workloads.build("wfull", 81, [700, 37, 300], [64, 1, 300], 32, 8, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    full = _varlen(pa, db, 0, 64, b.block_tables)
    wide = _varlen(pa, db, 10000, 64, b.block_tables)
    assert torch.equal(full.view(torch.int16), wide.view(torch.int16))
    b1 = workloads.build("wfull1", 82, [700, 37, 4000], [1, 1, 1], 32, 8, 128, 16, "bf16")
    db1 = DeviceBatch(b1, DEV)
    run_scatter(pa, db1)
    assert torch.equal(_decode(pa, db1, 0, 0, b1.block_tables).view(torch.int16),
                       _decode(pa, db1, 5000, 0, b1.block_tables).view(torch.int16))


def test_window_needs_causal_and_non_negative(pa):
    b = workloads.build("wbad", 83, [100, 40], [30, 40], 8, 2, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    with pytest.raises(pa.PAError):
        _varlen(pa, db, 16, 32, b.block_tables, causal=False)
    bd = workloads.build("wbad1", 84, [100, 40], [1, 1], 8, 2, 128, 16, "bf16")
    dbd = DeviceBatch(bd, DEV)
    with pytest.raises(pa.PAError):
        _decode(pa, dbd, -1, 0, bd.block_tables)
