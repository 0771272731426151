"""pa_decode_static_workspace: decode for callers that cannot allocate device memory.

Some callers cannot allocate device memory where attention runs (a runtime whose
memory planner only provides the tensors it planned, a plug-in that must not call
cudaMalloc on the serving path).  This entry point takes inputs and outputs only
and keeps its split-K scratch in a fixed array inside the library.  These tests
call it through the C ABI (ctypes, no Python wrapper) and compare its output with
pa_decode's, which uses a caller-provided workspace, on consecutive calls, and with
the fp64 oracle.
"""

import ctypes
import importlib.util
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import TOL, TOL_FP8, DeviceBatch, compare, run_decode

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = os.path.join(ROOT, "paged_kv_cache_pagedattention_gb300", "libpa.so")
    if not os.path.exists(path):
        spec = importlib.util.spec_from_file_location(
            "_pa_build", os.path.join(ROOT, "paged_kv_cache_pagedattention_gb300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
    import paged_kv_cache_pagedattention_gb300 as pa

    c = ctypes.CDLL(pa.LIB_PATH)
    fn = c.pa_decode_static_workspace
    fn.restype, fn.argtypes = pa.SIGNATURES["pa_decode_static_workspace"]
    return pa, fn


def _call_static(fn, pa, db, partition_size=0):
    b = db.b
    out = torch.full_like(db.q, float("nan"))
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    st = fn(out.data_ptr(), db.q.data_ptr(), db.kc.data_ptr(), db.vc.data_ptr(), b.num_blocks,
            db.tables.data_ptr(), b.max_blocks_per_seq, db.lens.data_ptr(), b.num_seqs, b.max_seq_len,
            b.num_q_heads, b.num_kv_heads, b.head_size, b.block_size, b.scale, pa.dtype_code(db.q),
            pa.dtype_code(db.kc), ptr(db.k_scale), ptr(db.v_scale), partition_size,
            torch.cuda.current_stream().cuda_stream)
    return st, out


def _check_close(a, b, kv_dtype):
    tol = TOL_FP8 if kv_dtype in workloads.FP8 else TOL
    err = (a.double() - b.double()).abs()
    assert torch.isfinite(a.double()).all()
    assert err.max().item() <= tol["max"] and err.mean().item() <= tol["mean"], (err.max().item(), err.mean().item())


def test_static_workspace_matches_decode_on_consecutive_calls(lib):
    pa, fn = lib
    cases = [
        # split-K with many partitions (the scratch holds partial states)
        (workloads.build("nz1", 41, [1, 17, 300, 1000, 777], [1] * 5, 32, 8, 128, 16, "bf16"), 64),
        # a different batch right after: FP8 cache, default partitioning
        (workloads.build("nz2", 42, [5000, 33, 2048], [1] * 3, 16, 2, 128, 32, "fp8_e4m3"), 0),
        # the first batch again, after the scratch holds the second call's contents
        (workloads.build("nz1", 41, [1, 17, 300, 1000, 777], [1] * 5, 32, 8, 128, 16, "bf16"), 64),
    ]
    for b, part in cases:
        db = DeviceBatch(b, DEV)
        st, got = _call_static(fn, pa, db, part)
        assert st == pa.PA_OK, pa.pa_status_string(st)
        ref = run_decode(pa, db, part)
        torch.cuda.synchronize()
        assert pa.pa_get_error_flags() == 0
        _check_close(got, ref, b.kv_dtype)
        # and with the oracle on the same cache contents (nothing was scattered)
        expect = oracle.paged_decode(b.q, b.q_dtype, b.k_cache, b.v_cache, b.kv_dtype, b.block_tables,
                                     b.seq_lens, b.block_size, b.scale, b.k_scale, b.v_scale)
        compare(got, expect, b.kv_dtype, where=f"static workspace {b.name}")


def test_static_workspace_coarsens_the_default_partitioning(lib):
    """A few short sequences under a large max_seq_len hint with 64 query heads per KV
    head: the default partitioning needs more partial states than the fixed array
    holds, so the call doubles the partition size until they fit.  Checked against
    pa_decode at the partition size the doubling reaches, and against the oracle."""
    pa, fn = lib
    b = workloads.build("nz4", 44, [100, 2000, 37, 5000], [1] * 4, 64, 1, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    hint = 200000
    cap = 32 << 20
    need = lambda part: pa.pa_decode_workspace_size(b.num_seqs, 64, 1, 128, hint, 16, part)  # noqa: E731
    part = pa.pa_default_partition_size(b.num_seqs, 1, hint, 16)
    assert need(part) > cap  # the coarsening loop runs
    while part < hint and need(part) > cap:
        part *= 2
    assert need(part) <= cap
    out = torch.full_like(db.q, float("nan"))
    st = fn(out.data_ptr(), db.q.data_ptr(), db.kc.data_ptr(), db.vc.data_ptr(), b.num_blocks,
            db.tables.data_ptr(), b.max_blocks_per_seq, db.lens.data_ptr(), b.num_seqs, hint, 64, 1, 128, 16,
            b.scale, pa.PA_BF16, pa.PA_BF16, None, None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_OK, pa.pa_status_string(st)
    ref = torch.empty_like(db.q)
    ws = pa.workspace_tensor(need(part), DEV)
    pa.pa_decode(ref, db.q, db.kc, db.vc, db.tables, db.lens, hint, b.scale, ws, None, None, part)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
    _check_close(out, ref, b.kv_dtype)
    expect = oracle.paged_decode(b.q, b.q_dtype, b.k_cache, b.v_cache, b.kv_dtype, b.block_tables, b.seq_lens,
                                 b.block_size, b.scale)
    compare(out, expect, b.kv_dtype, where="static workspace, coarsened")


def test_static_workspace_reports_invalid_arguments_first(lib):
    """Invalid arguments on a problem too large for the array give the argument error
    (as pa_decode does), not PA_ERR_WORKSPACE."""
    pa, fn = lib
    b = workloads.build("nz5", 45, [40], [1], 8, 2, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    s = torch.cuda.current_stream().cuda_stream
    args = lambda hq, hkv, part: (db.q.data_ptr(), db.q.data_ptr(), db.kc.data_ptr(), db.vc.data_ptr(),  # noqa
                                  b.num_blocks, db.tables.data_ptr(), b.max_blocks_per_seq, db.lens.data_ptr(),
                                  4096, 100000, hq, hkv, 128, 16, b.scale, pa.PA_BF16, pa.PA_BF16, None, None,
                                  part, s)
    assert fn(*args(63, 8, 16)) == pa.PA_ERR_INVALID_ARG  # query heads not a multiple of KV heads
    assert fn(*args(64, 8, 24)) == pa.PA_ERR_INVALID_ARG  # partition not a multiple of the block
    assert fn(*args(64, 8, 16)) == pa.PA_ERR_WORKSPACE    # valid, but too large for the array
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0


def test_static_workspace_rejects_problems_beyond_its_size(lib):
    pa, fn = lib
    b = workloads.build("nz3", 43, [40], [1], 8, 2, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    need = pa.pa_decode_workspace_size(4096, 64, 8, 128, 100000, 16, 16)
    assert need > (32 << 20)
    # 4096 sequences x 64 heads x 6250 partitions of partial states cannot fit: rejected before any launch
    st = fn(db.q.data_ptr(), db.q.data_ptr(), db.kc.data_ptr(), db.vc.data_ptr(), b.num_blocks,
            db.tables.data_ptr(), b.max_blocks_per_seq, db.lens.data_ptr(), 4096, 100000, 64, 8, 128, 16,
            b.scale, pa.PA_BF16, pa.PA_BF16, None, None, 16, torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
