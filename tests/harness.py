"""Helpers shared by the GPU parity tests: move a workload to the device, run the
library through its binding, run the oracle on the same inputs, compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Parity bars: max-abs 1e-2 and mean-abs 1e-3 for fp32/fp16/bf16 caches, max-abs
# 5e-2 for FP8 caches (the oracle reads the same stored FP8 codes).  NVFP4 caches
# take the FP8 bar: the oracle reads the same stored codes and block scales, and
# the kernels widen them exactly, so the arithmetic left is that of the FP8 path.
TOL = {"max": 1e-2, "mean": 1e-3}
TOL_FP8 = {"max": 5e-2, "mean": 1e-3}


def tol_for(kv_dtype):
    return TOL_FP8 if kv_dtype in workloads.SCALED else TOL


class DeviceBatch:
    """A PagedBatch's tensors on one device."""

    def __init__(self, b: workloads.PagedBatch, dev, cache=None):
        self.b = b
        self.dev = dev
        self.kc, self.vc = cache if cache is not None else workloads.device_cache(b, dev)
        self.key = workloads.bits_to_torch(b.key, b.src_dtype, dev)
        self.value = workloads.bits_to_torch(b.value, b.src_dtype, dev)
        self.slots = torch.from_numpy(b.slot_mapping).to(dev)
        self.q = workloads.bits_to_torch(b.q, b.q_dtype, dev)
        self.tables = torch.from_numpy(b.block_tables).to(dev)
        self.lens = torch.from_numpy(b.seq_lens).to(dev)
        self.qsl = torch.from_numpy(b.query_start_loc).to(dev)
        scaled = b.kv_dtype in workloads.SCALED
        # one scale per tensor, or one per KV head
        self.k_scale = torch.tensor(np.atleast_1d(b.k_scale), dtype=torch.float32, device=dev) if scaled else None
        self.v_scale = torch.tensor(np.atleast_1d(b.v_scale), dtype=torch.float32, device=dev) if scaled else None


def run_scatter(pa, db: DeviceBatch):
    pa.pa_reshape_and_cache(db.key, db.value, db.kc, db.vc, db.slots, db.k_scale, db.v_scale)


def run_decode(pa, db: DeviceBatch, partition_size=0, out=None):
    b = db.b
    out = torch.empty_like(db.q) if out is None else out
    ws = pa.workspace_tensor(pa.pa_decode_workspace_size(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_size,
                                                         b.max_seq_len, b.block_size, partition_size), db.dev)
    pa.pa_decode(out, db.q, db.kc, db.vc, db.tables, db.lens, b.max_seq_len, b.scale, ws,
                 db.k_scale, db.v_scale, partition_size)
    return out


def run_varlen(pa, db: DeviceBatch, partition_size=0, causal=True, out=None):
    b = db.b
    out = torch.empty_like(db.q) if out is None else out
    ws = pa.workspace_tensor(pa.pa_varlen_workspace_size(b.num_seqs, b.total_q, b.max_query_len, b.num_q_heads,
                                                         b.num_kv_heads, b.head_size, b.max_seq_len,
                                                         b.block_size, partition_size), db.dev)
    pa.pa_varlen_attn(out, db.q, db.kc, db.vc, db.tables, db.qsl, db.lens, b.max_query_len, b.max_seq_len,
                      b.scale, ws, causal, db.k_scale, db.v_scale, partition_size)
    return out


def oracle_scatter(b: workloads.PagedBatch):
    """Host caches after the oracle's scatter of the batch's new tokens."""
    k_ref, v_ref = b.k_cache.copy(), b.v_cache.copy()
    oracle.reshape_and_cache(b.key, b.value, k_ref, v_ref, b.slot_mapping, b.block_size, b.src_dtype,
                             b.kv_dtype, b.k_scale, b.v_scale)
    return k_ref, v_ref


def compare(got: torch.Tensor, ref: np.ndarray, kv_dtype: str, rows=None, where=""):
    """Element-wise comparison of GPU output rows with the oracle; returns (max, mean)."""
    g = got.double().cpu().numpy()
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert np.all(np.isfinite(g)), f"{where}: non-finite GPU output"
    err = np.abs(g - ref)
    t = tol_for(kv_dtype)
    assert err.max() <= t["max"], f"{where}: max_abs {err.max():.4g} > {t['max']}"
    assert err.mean() <= t["mean"], f"{where}: mean_abs {err.mean():.4g} > {t['mean']}"
    return float(err.max()), float(err.mean())


def gather_request_blocks(db: DeviceBatch, seqs):
    """Host copy of the cache blocks the given sequences use, remapped to a compact pool.

    Returns (k_bits, v_bits, compact_tables, remap) so the oracle can run on a few
    sequences of a full-size workload without copying the whole cache.
    """
    b = db.b
    used = []
    for s in seqs:
        n = -(-int(b.seq_lens[s]) // b.block_size)
        used.extend(int(x) for x in b.block_tables[s, :n])
    uniq = sorted(set(used))
    remap = {p: i for i, p in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.long, device=db.dev)
    k = workloads.torch_to_bits(db.kc.index_select(0, idx), b.kv_dtype)
    v = workloads.torch_to_bits(db.vc.index_select(0, idx), b.kv_dtype)
    tables = np.full_like(b.block_tables, -1)
    for s in seqs:
        n = -(-int(b.seq_lens[s]) // b.block_size)
        tables[s, :n] = [remap[int(x)] for x in b.block_tables[s, :n]]
    return k, v, tables, remap


def sampled_oracle_inputs(db: DeviceBatch, seqs, run_gpu):
    """Oracle inputs for a few sequences of a full-size workload, none taken from the CUDA path.

    Snapshots the blocks of ``seqs`` BEFORE ``run_gpu()`` (which scatters and
    attends), applies the oracle's own scatter of those sequences' new tokens to
    the snapshot, and checks the GPU's post-scatter blocks equal it byte for byte.
    Returns (k_bits, v_bits, compact_tables) after the oracle's scatter.
    """
    b = db.b
    k, v, tables, remap = gather_request_blocks(db, seqs)
    run_gpu()
    torch.cuda.synchronize()
    k_after, v_after, _, _ = gather_request_blocks(db, seqs)
    toks, slots = [], []
    for s in seqs:
        for t in range(int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])):
            slot = int(b.slot_mapping[t])
            toks.append(t)
            slots.append(remap[slot // b.block_size] * b.block_size + slot % b.block_size)
    toks = np.array(toks, dtype=np.int64)
    oracle.reshape_and_cache(b.key[toks], b.value[toks], k, v, np.array(slots, np.int64), b.block_size,
                             b.src_dtype, b.kv_dtype, b.k_scale, b.v_scale)
    assert np.array_equal(k_after, k), "K cache bytes after scatter"
    assert np.array_equal(v_after, v), "V cache bytes after scatter"
    return k, v, tables
