"""GPU parity of the copy-on-write block copy (pa_copy_blocks): byte-exact against
the oracle, and a fork that copies its shared tail block before writing."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
_BITS = {"bf16": np.uint16, "f16": np.uint16, "f32": np.uint32, "fp8_e4m3": np.uint8, "fp8_e5m2": np.uint8}


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pagedattention_gb300 as lib
    lib.pa_get_error_flags(clear=True)
    return lib


def _pairs(rng, nb, n, extra=()):
    """n (src, dst) pairs with distinct destinations that are never sources."""
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:n], perm[n:2 * n]], 1).astype(np.int64)
    return np.concatenate([pairs, np.asarray(extra, np.int64).reshape(-1, 2)]) if len(extra) else pairs


@pytest.mark.parametrize("dtype,shape", [("bf16", (64, 8, 16, 128)), ("fp8_e4m3", (48, 8, 32, 128)),
                                         ("f32", (20, 2, 16, 64)), ("f16", (30, 3, 32, 64)),
                                         ("fp8_e5m2", (40, 8, 16, 128))])
def test_copy_blocks_bit_exact(pa, dtype, shape):
    rng = np.random.default_rng(41)
    hi = np.iinfo(_BITS[dtype]).max
    kb = rng.integers(0, hi, size=shape, dtype=_BITS[dtype], endpoint=True)
    vb = rng.integers(0, hi, size=shape, dtype=_BITS[dtype], endpoint=True)
    nb = shape[0]
    pairs = _pairs(rng, nb - 1, nb // 3)
    # a self-copy of the one block no pair uses, and two out-of-range pairs
    pairs = np.concatenate([pairs, [[nb - 1, nb - 1], [-1, 3], [2, nb]]]).astype(np.int64)
    kc, vc = workloads.bits_to_torch(kb, dtype, DEV), workloads.bits_to_torch(vb, dtype, DEV)
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).to(DEV))
    flags = pa.pa_get_error_flags(clear=True)
    k_ref, v_ref = kb.copy(), vb.copy()
    assert oracle.copy_blocks(k_ref, v_ref, pairs) == [len(pairs) - 2, len(pairs) - 1]
    assert flags == pa.PA_ERRFLAG_BLOCK_TABLE
    assert np.array_equal(workloads.torch_to_bits(kc, dtype), k_ref)
    assert np.array_equal(workloads.torch_to_bits(vc, dtype), v_ref)


def test_no_pairs_is_a_no_op(pa):
    kc = torch.randn(4, 2, 16, 64, device=DEV).to(torch.bfloat16)
    before = kc.clone()
    pa.pa_copy_blocks(kc, kc.clone(), torch.zeros(0, 2, dtype=torch.int64, device=DEV))
    assert pa.pa_get_error_flags(clear=True) == 0
    assert torch.equal(kc, before)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_copy_on_write_fork_on_device(pa, kv):
    """A parent of 1000 tokens and a fork share every block; the fork copies the shared
    tail block (8 of 16 slots used) into a free block, repoints its table, then both
    append a token at position 1000 and decode.  Device and oracle run the same steps."""
    L, bs = 1000, 16
    b = workloads.build("cow", 51, [L + 1, L + 1], [1, 1], 32, 8, 128, bs, kv, min_pool=160)
    nlog = -(-(L + 1) // bs)
    tables = b.block_tables.copy()
    tables[1, :nlog] = tables[0, :nlog]                       # the fork shares every block
    used = set(int(x) for x in tables[0, :nlog])
    fresh = next(x for x in range(b.num_blocks) if x not in used)
    tail = int(tables[0, L // bs])
    pairs = np.array([[tail, fresh]], np.int64)
    fork_tables = tables.copy()
    fork_tables[1, L // bs] = fresh
    slots = np.array([tail * bs + L % bs, fresh * bs + L % bs], np.int64)

    # oracle: the history is the builder's cache; copy, append both tokens, decode
    k_ref, v_ref = b.k_cache.copy(), b.v_cache.copy()
    assert oracle.copy_blocks(k_ref, v_ref, pairs) == []
    oracle.reshape_and_cache(b.key, b.value, k_ref, v_ref, slots, bs, b.src_dtype, kv, b.k_scale, b.v_scale)
    ref = oracle.paged_decode(b.q, b.q_dtype, k_ref, v_ref, kv, fork_tables, b.seq_lens, bs, b.scale,
                              b.k_scale, b.v_scale)

    kc = workloads.bits_to_torch(b.k_cache, kv, DEV)
    vc = workloads.bits_to_torch(b.v_cache, kv, DEV)
    fp8 = kv in workloads.FP8
    ks = torch.tensor([b.k_scale], dtype=torch.float32, device=DEV) if fp8 else None
    vs = torch.tensor([b.v_scale], dtype=torch.float32, device=DEV) if fp8 else None
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).to(DEV))
    key = workloads.bits_to_torch(b.key, b.src_dtype, DEV)
    value = workloads.bits_to_torch(b.value, b.src_dtype, DEV)
    pa.pa_reshape_and_cache(key, value, kc, vc, torch.from_numpy(slots).to(DEV), ks, vs)
    q = workloads.bits_to_torch(b.q, b.q_dtype, DEV)
    out = torch.empty_like(q)
    ws = pa.workspace_tensor(pa.pa_decode_workspace_size(2, 32, 8, 128, L + 1, bs, 64), DEV)
    pa.pa_decode(out, q, kc, vc, torch.from_numpy(fork_tables).to(DEV), torch.from_numpy(b.seq_lens).to(DEV),
                 L + 1, b.scale, ws, ks, vs, 64)
    assert pa.pa_get_error_flags(clear=True) == 0
    assert np.array_equal(workloads.torch_to_bits(kc, kv), k_ref)
    assert np.array_equal(workloads.torch_to_bits(vc, kv), v_ref)
    compare(out, ref, kv, where=f"copy-on-write fork {kv}")


def test_copy_blocks_full_pool_properties(pa):
    """A Llama-sized pool (18,432 blocks of 8 x 16 x 128 bf16, 1.2 GB for K and V) and
    4,096 pairs: every destination equals its source's bytes from before the call and
    a sample of the other blocks is unchanged."""
    nb = 18432
    g = torch.Generator(device=DEV).manual_seed(7)
    kc = torch.randn(nb, 8, 16, 128, device=DEV, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, 8, 16, 128, device=DEV, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(43)
    pairs = _pairs(rng, nb, 4096)
    src = torch.from_numpy(pairs[:, 0]).to(DEV)
    dst = torch.from_numpy(pairs[:, 1]).to(DEV)
    k_src, v_src = kc[src].clone(), vc[src].clone()
    others = torch.from_numpy(np.setdiff1d(rng.choice(nb, 2048, replace=False), pairs[:, 1])).to(DEV)
    k_oth, v_oth = kc[others].clone(), vc[others].clone()
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).to(DEV))
    assert pa.pa_get_error_flags(clear=True) == 0
    assert torch.equal(kc[dst].view(torch.int16), k_src.view(torch.int16))
    assert torch.equal(vc[dst].view(torch.int16), v_src.view(torch.int16))
    assert torch.equal(kc[others].view(torch.int16), k_oth.view(torch.int16))
    assert torch.equal(vc[others].view(torch.int16), v_oth.view(torch.int16))
