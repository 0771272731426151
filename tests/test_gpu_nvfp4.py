"""GPU parity of the NVFP4 cache format (E2M1 codes + E4M3 block scales + fp32
scale) on every path: the scatter's bytes against the oracle exactly, decode
(tensor-core and generic kernels), sliding windows, shared-prefix decode, the
varlen step and the block copy within the FP8 bar."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import (DeviceBatch, compare, oracle_scatter, run_decode, run_scatter, run_varlen,
                     sampled_oracle_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
RAGGED = [1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 511, 1000]
PER_HEAD = [0.011, 2.0 ** -6, 0.3, 2.0 ** -2, 0.05, 1.0, 2.0 ** -9, 0.0071]


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


def _special_rows():
    """f32 rows of 128 (8 groups of 16) that hit every rounding decision: E2M1
    midpoints (ties) under an exact block scale, saturation of the codes and of the
    block scale, small negatives (negative zero codes), all-zero and vanishing groups,
    and N(0,1) groups."""
    rng = np.random.default_rng(17)
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    groups = []
    for sb in (1.0, 0.5, 3.0, 2.0 ** -5):
        g = [6.0 * sb] + [m * sb for m in mids] + [-m * sb for m in mids] + [-0.01 * sb]
        groups.append(g)
    groups.append([0.0] * 16)
    groups.append([1e-30] * 8 + [-1e-30] * 8)
    groups.append([6.0 * 448.0 * 9.0] + [1.0] * 15)          # block scale saturates at 448
    groups.append([7.0, -6.5] + [6.2] * 14)
    while len(groups) % 8:
        groups.append(list(rng.standard_normal(16)))
    for _ in range(40):
        groups.append(list(rng.standard_normal(16) * 10.0 ** rng.uniform(-3, 3)))
    return np.array(groups, np.float32).reshape(-1, 128)


@pytest.mark.parametrize("scale", [1.0, 0.37, 2.0 ** -10])
def test_scatter_codes_and_block_scales_bit_exact(pa, scale):
    rows = _special_rows()
    tokens = rows.shape[0]
    key = torch.from_numpy(rows.reshape(tokens, 1, 128)).to(DEV)
    value = torch.from_numpy(-rows.reshape(tokens, 1, 128)).to(DEV)
    tile = workloads.nvfp4_tile_bytes(16, 128)
    kc = torch.zeros((tokens, 1, tile), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    slot_np = np.arange(tokens, dtype=np.int64) * 16 + 5
    sc = torch.tensor([scale], dtype=torch.float32, device=DEV)
    pa.pa_reshape_and_cache(key, value, kc, vc, torch.from_numpy(slot_np).to(DEV), sc, sc)
    assert pa.pa_get_error_flags() == 0
    k_ref = np.zeros((tokens, 1, tile), np.uint8)
    v_ref = np.zeros_like(k_ref)
    kbits = rows.reshape(tokens, 1, 128).view(np.uint32)
    vbits = (-rows).reshape(tokens, 1, 128).view(np.uint32)
    oracle.reshape_and_cache(kbits, vbits, k_ref, v_ref, slot_np, 16, "f32", "nvfp4", scale, scale)
    got_k, got_v = kc.cpu().numpy(), vc.cpu().numpy()
    assert np.array_equal(got_k, k_ref), f"K: {np.count_nonzero(got_k != k_ref)} bytes differ"
    assert np.array_equal(got_v, v_ref), f"V: {np.count_nonzero(got_v != v_ref)} bytes differ"


def _full_parity(pa, b, partition_size=0, window=0):
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    if window:
        out = torch.empty_like(db.q)
        ws = pa.workspace_tensor(pa.pa_decode_workspace_size(b.num_seqs, b.num_q_heads, b.num_kv_heads,
                                                             b.head_size, b.max_seq_len, b.block_size,
                                                             partition_size), DEV)
        pa.pa_decode(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws, db.k_scale,
                     db.v_scale, partition_size, window=window)
    else:
        out = run_decode(pa, db, partition_size)
    torch.cuda.synchronize()
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    assert np.array_equal(workloads.torch_to_bits(db.kc, "nvfp4"), k_ref), "K cache bytes"
    assert np.array_equal(workloads.torch_to_bits(db.vc, "nvfp4"), v_ref), "V cache bytes"
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, "nvfp4", b.block_tables, b.seq_lens, b.block_size,
                              b.scale, b.k_scale, b.v_scale, window=window)
    return compare(out, ref, "nvfp4", where=b.name)


DECODE = [
    # (name, Hq, Hkv, d, bs, lens, partition, q dtype)
    ("g4_bs32_split64", 32, 8, 128, 32, RAGGED, 64, None),
    ("g8_bs16", 16, 2, 128, 16, RAGGED, 0, None),
    ("g16_two_groups", 32, 2, 128, 16, RAGGED, 256, None),
    ("f16q_bs32", 8, 2, 128, 32, RAGGED, 32, "f16"),
    ("f32q_generic", 8, 2, 128, 16, RAGGED, 48, "f32"),
    ("d64_generic", 8, 2, 64, 16, RAGGED, 0, None),
]


@pytest.mark.parametrize("case", DECODE, ids=[c[0] for c in DECODE])
def test_decode_parity(pa, case):
    name, hq, hkv, d, bs, lens, part, q_dtype = case
    b = workloads.build("nvfp4_" + name, 300 + len(name), lens, [1] * len(lens), hq, hkv, d, bs, "nvfp4",
                        q_dtype=q_dtype, src_dtype=q_dtype)
    _full_parity(pa, b, part)


def test_per_head_scales(pa):
    b = workloads.build("nvfp4_ph", 331, RAGGED, [1] * len(RAGGED), 32, 8, 128, 32, "nvfp4", nvfp4_scale=PER_HEAD)
    assert np.ndim(b.k_scale) == 1
    _full_parity(pa, b, 64)


@pytest.mark.parametrize("window,part", [(100, 64), (16, 0), (1000, 128)])
def test_sliding_window(pa, window, part):
    b = workloads.build("nvfp4_w", 341, [700, 37, 1, 300, 4000], [1] * 5, 32, 8, 128, 16, "nvfp4")
    _full_parity(pa, b, part, window)


VARLEN = [
    # (name, Hq, Hkv, bs, lens, q_lens, partition, causal, q dtype) -- multi-token rows on the
    # tcgen05 prefill tiles (NVFP4 tiles staged by bulk copies, widened by the converters)
    ("mixed_bs16_split64", 32, 8, 16, [700, 37, 1, 300, 900], [64, 1, 1, 300, 17], 64, True, None),
    ("bs32_default", 32, 8, 32, [2000, 33, 700], [300, 1, 64], 0, True, None),
    ("bs64_g8_f16q", 16, 2, 64, [1500, 513], [257, 200], 0, True, "f16"),
    ("non_causal_bs16", 8, 2, 16, [400, 90], [130, 17], 96, False, None),
]


@pytest.mark.parametrize("case", VARLEN, ids=[c[0] for c in VARLEN])
def test_varlen_parity(pa, case):
    name, hq, hkv, bs, lens, q_lens, part, causal, q_dtype = case
    b = workloads.build("nvfp4_v_" + name, 351 + len(name), lens, q_lens, hq, hkv, 128, bs, "nvfp4",
                        q_dtype=q_dtype, src_dtype=q_dtype, causal=causal)
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    out = run_varlen(pa, db, part, causal)
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    ref = oracle.paged_varlen(b.q, b.q_dtype, k_ref, v_ref, "nvfp4", b.block_tables, b.query_start_loc,
                              b.seq_lens, bs, b.scale, causal, b.k_scale, b.v_scale)
    compare(out, ref, "nvfp4", where="nvfp4 varlen " + name)


def test_varlen_window_and_per_head_scales(pa):
    b = workloads.build("nvfp4_vw", 391, [2000, 33, 700], [300, 1, 64], 32, 8, 128, 16, "nvfp4",
                        nvfp4_scale=PER_HEAD)
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    tables = b.block_tables.copy()
    for r in range(b.num_seqs):   # blocks wholly before the window: released
        q_len = int(b.query_start_loc[r + 1] - b.query_start_loc[r])
        tables[r, : max(0, int(b.seq_lens[r]) - q_len - 200 + 1) // 16] = -1
    out = torch.empty_like(db.q)
    ws = pa.workspace_tensor(pa.pa_varlen_workspace_size(b.num_seqs, b.total_q, b.max_query_len, 32, 8, 128,
                                                         b.max_seq_len, 16, 0), DEV)
    pa.pa_varlen_attn(out, db.q, db.kc, db.vc, torch.from_numpy(tables).to(DEV), db.qsl, db.lens, b.max_query_len,
                      b.max_seq_len, b.scale, ws, True, db.k_scale, db.v_scale, 0, window=200)
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    ref = oracle.paged_varlen(b.q, b.q_dtype, k_ref, v_ref, "nvfp4", tables, b.query_start_loc, b.seq_lens, 16,
                              b.scale, True, b.k_scale, b.v_scale, window=200)
    compare(out, ref, "nvfp4", where="nvfp4 varlen window per-head")


def test_shared_prefix_groups(pa):
    lens = [300, 300, 300, 200, 210, 100, 77]
    shared_map = {1: (0, 5), 2: (0, 5), 4: (3, 5), 5: (3, 3)}
    b = workloads.build("nvfp4_grp", 361, lens, [1] * 7, 32, 8, 128, 32, "nvfp4", shared=shared_map)
    db = DeviceBatch(b, DEV)
    run_scatter(pa, db)
    starts = torch.tensor([0, 3, 6, 7], dtype=torch.int32, device=DEV)
    shared = torch.tensor([5, 5, 0], dtype=torch.int32, device=DEV)
    out = torch.empty_like(db.q)
    ws = pa.workspace_tensor(pa.pa_decode_shared_prefix_workspace_size(7, 3, 32, 8, 128, b.max_seq_len, 32, 64),
                             DEV)
    pa.pa_decode_shared_prefix(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws, starts,
                               shared, 8, db.k_scale, db.v_scale, 64)
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = oracle_scatter(b)
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, "nvfp4", b.block_tables, b.seq_lens, 32, b.scale,
                              b.k_scale, b.v_scale)
    compare(out, ref, "nvfp4", where="nvfp4 shared prefix")


def test_copy_blocks_bit_exact(pa):
    rng = np.random.default_rng(43)
    nb = 40
    kb = workloads.nvfp4_random_cache(rng, nb, 8, 16, 128)
    vb = workloads.nvfp4_random_cache(rng, nb, 8, 16, 128)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:12], perm[12:24]], 1).astype(np.int64)
    kc, vc = torch.from_numpy(kb).to(DEV), torch.from_numpy(vb).to(DEV)
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).to(DEV))
    assert pa.pa_get_error_flags() == 0
    k_ref, v_ref = kb.copy(), vb.copy()
    assert oracle.copy_blocks(k_ref, v_ref, pairs) == []
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)


def test_shape_rules(pa):
    b = workloads.build("nvfp4_args", 371, [40], [1], 8, 2, 128, 16, "nvfp4")
    db = DeviceBatch(b, DEV)
    out = torch.empty_like(db.q)
    ws = pa.workspace_tensor(1 << 20, DEV)
    with pytest.raises(pa.PAError) as e:   # NVFP4 needs its fp32 scales
        pa.pa_decode(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    bad = torch.zeros((4, 1, 9 * 8 * 16 // 16), dtype=torch.uint8, device=DEV)  # block 8 x head 16: 72-byte tiles
    key = torch.zeros((1, 1, 16), dtype=torch.float32, device=DEV)
    sc = torch.ones(1, dtype=torch.float32, device=DEV)
    with pytest.raises(pa.PAError) as e:
        pa.pa_reshape_and_cache(key, key, bad, bad.clone(), torch.zeros(1, dtype=torch.int64, device=DEV), sc, sc)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


@pytest.mark.slow
def test_full_size_sampled(pa):
    """The FP8 decode shapes with an NVFP4 cache, full size: sampled rows against the oracle."""
    b = workloads.nvfp4()
    db = DeviceBatch(b, DEV)
    outs = []

    def gpu():
        run_scatter(pa, db)
        outs.append(run_decode(pa, db))

    seqs = [0, 100, 255]
    k, v, tables = sampled_oracle_inputs(db, seqs, gpu)
    assert pa.pa_get_error_flags() == 0
    ref = oracle.paged_decode(b.q, b.q_dtype, k, v, "nvfp4", tables, b.seq_lens, b.block_size, b.scale,
                              b.k_scale, b.v_scale, seqs=seqs)
    compare(outs[0], ref, "nvfp4", rows=seqs, where=b.name)
