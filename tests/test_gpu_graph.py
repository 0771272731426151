"""The library's calls can be captured into a CUDA graph (they neither synchronise
nor allocate): scatter + attention captured once and replayed give the same bytes
as eager calls, for decode, shared-prefix decode (side-stream fork/join) and varlen."""

import numpy as np
import pytest
import torch

import workloads
from harness import DeviceBatch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


def _graph_vs_eager(pa, db, call):
    """Run `call` eagerly, then capture it and replay twice; outputs must be equal."""
    eager = call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = call()
    for _ in range(2):
        captured.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(captured.view(torch.int16), eager.view(torch.int16))
    assert pa.pa_get_error_flags(clear=True) == 0


def test_decode_step_in_a_graph(pa):
    b = workloads.build("g_dec", 61, [700, 33, 1, 4000], [1, 1, 1, 1], 32, 8, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    ws = pa.workspace_tensor(pa.pa_decode_workspace_size(b.num_seqs, 32, 8, 128, b.max_seq_len, 16, 256), DEV)
    out = torch.empty_like(db.q)

    def call():
        s = torch.cuda.current_stream()
        pa.pa_reshape_and_cache(db.key, db.value, db.kc, db.vc, db.slots, None, None, s)
        pa.pa_decode(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws, None, None, 256, s)
        return out

    _graph_vs_eager(pa, db, call)


def test_shared_prefix_step_in_a_graph(pa):
    b = workloads.agentic(seed=7, host_cache=True, scale_lengths=1 / 64.0)
    db = DeviceBatch(b, DEV)
    starts, shared = [0], []
    for fam in b.families:
        starts.append(starts[-1] + len(fam))
        nb = -(-int(b.seq_lens[fam[0]]) // b.block_size)
        shared.append(int(np.floor(0.96 * nb)) if len(fam) > 1 else 0)
    gstart = torch.tensor(starts, dtype=torch.int32, device=DEV)
    gshared = torch.tensor(shared, dtype=torch.int32, device=DEV)
    ws = pa.workspace_tensor(pa.pa_decode_shared_prefix_workspace_size(
        b.num_seqs, len(shared), b.num_q_heads, b.num_kv_heads, b.head_size, b.max_seq_len, b.block_size, 0), DEV)
    out = torch.empty_like(db.q)
    max_group = max(len(f) for f in b.families)

    def call():
        s = torch.cuda.current_stream()
        pa.pa_reshape_and_cache(db.key, db.value, db.kc, db.vc, db.slots, None, None, s)
        pa.pa_decode_shared_prefix(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws,
                                   gstart, gshared, max_group, None, None, 0, s)
        return out

    _graph_vs_eager(pa, db, call)


def test_varlen_step_in_a_graph(pa):
    b = workloads.build("g_var", 62, [700, 37, 1, 300, 90], [64, 1, 1, 300, 17], 32, 8, 128, 16, "bf16")
    db = DeviceBatch(b, DEV)
    ws = pa.workspace_tensor(pa.pa_varlen_workspace_size(b.num_seqs, b.total_q, b.max_query_len, 32, 8, 128,
                                                         b.max_seq_len, 16, 64), DEV)
    out = torch.empty_like(db.q)

    def call():
        s = torch.cuda.current_stream()
        pa.pa_reshape_and_cache(db.key, db.value, db.kc, db.vc, db.slots, None, None, s)
        pa.pa_varlen_attn(out, db.q, db.kc, db.vc, db.tables, db.qsl, db.lens, b.max_query_len, b.max_seq_len,
                          b.scale, ws, True, None, None, 64, s)
        return out

    _graph_vs_eager(pa, db, call)
