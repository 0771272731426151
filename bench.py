"""Benchmark of the paged KV cache hot path on GB300 (one JSON line on stdout).

A step is one pass of the hot path over one batch: the scatter of every
sequence's new token into the paged cache (pa_reshape_and_cache), then
PagedAttention decode over the whole batch (pa_decode: split-K attention kernel
+ partial merge).  The default workload is the long-context agentic decode
(batch 16 = 3 families of parent + 4 forks sharing 96% of their blocks + 1 lone
parent, lengths log-normal around 142K tokens, 64 query / 8 KV heads, head 128,
bf16, block 16).  Its KV working set (~2.7 GB unique) is far larger than L2, so
consecutive steps do not hit in L2 across iterations.

metric: attended KV tokens per second (sum of seq_lens per step / step time),
whole job over all ranks.  Multi-GPU (torchrun): each rank runs its own
independent batch (weak scaling, no collective on the data path).

`--impl reference` times the fp64 CPU oracle instead (the reference arm), on the
host cores, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attended KV tokens/sec and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOADS = ("agentic", "llama", "fp8", "fp8_e5m2", "nvfp4", "mixed", "mixed_fp8", "mixed_nvfp4", "tiny")


# ----------------------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(x: float, device) -> float:
    """Max of a float over all ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch of the same shape (weak scaling)."""
    return base + 7919 * rank


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_sustained():
    """Sustained dense bf16 TFLOP/s (a kernel timed inside a long loop of steps)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def varlen_split(b) -> dict:
    """Bytes of the single-token rows and FLOPs of the multi-token rows of a varlen batch.

    Prefill FLOPs count 2 multiply-adds (QK and PV) x 2 flops x head_size per
    (query row, query head, attended key), with the causal key count."""
    import workloads

    kv_tok = 2 * b.num_kv_heads * b.head_size * workloads.ELEM_BYTES[b.kv_dtype]
    qb = workloads.ELEM_BYTES[b.q_dtype]
    dec_bytes, flops, pf_kv_bytes = 0, 0, 0
    for r in range(b.num_seqs):
        ql = int(b.query_start_loc[r + 1] - b.query_start_loc[r])
        L = int(b.seq_lens[r])
        if ql == 1:
            dec_bytes += L * kv_tok + 2 * b.num_q_heads * b.head_size * qb + 4 * (-(-L // b.block_size))
        elif ql > 1:
            keys = sum(L - ql + j + 1 for j in range(ql)) if b.causal else ql * L
            flops += 4 * b.head_size * b.num_q_heads * keys
            pf_kv_bytes += L * kv_tok
    return {"decode_bytes": dec_bytes, "prefill_flops": flops, "prefill_kv_bytes": pf_kv_bytes}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        import tempfile

        self.path = tempfile.mktemp(prefix="pa_clocks_", suffix=".csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.bus_id and not self.bus_id.endswith(parts[1].lower()[-12:]) and \
                        not parts[1].lower().endswith(self.bus_id[-12:]):
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def unique_kv_tokens(b) -> int:
    """Token slots that hold data some sequence reads, shared blocks counted once."""
    import numpy as np

    valid = {}
    for s in range(b.num_seqs):
        n = int(b.seq_lens[s])
        nb = -(-n // b.block_size)
        for j in range(nb):
            cnt = min(b.block_size, n - j * b.block_size)
            p = int(b.block_tables[s, j])
            if cnt > valid.get(p, 0):
                valid[p] = cnt
    return int(np.sum(list(valid.values()), dtype=np.int64))


KERNEL_SOURCES = {"decode_mma_kernel": ("attn_decode.cu", "pa_common.cuh"),
                  "varlen_span": ("attn_decode.cu", "attn_prefill_tc.cu", "pa_common.cuh"),
                  "shared_prefix_span": ("attn_decode.cu", "attn_prefill.cu", "pa_common.cuh"),
                  "prefill_tc_kernel": ("attn_prefill_tc.cu", "pa_common.cuh")}


def decode_source_hash(kernel: str = "decode_mma_kernel") -> str:
    """Hash of the sources a profiled kernel is built from (stale ncu numbers are dropped)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_cache_pagedattention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "decode_mma_kernel"):
    """DRAM bytes per launch of a kernel from the committed ncu summary, if it was
    captured on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_per_launch_bytes\s*=\s*([0-9.eE+]+)", text)
    h = re.search(r"source_hash\s*=\s*([0-9a-f]+)", text)
    if not m or not h or kernel not in KERNEL_SOURCES or h.group(1) != decode_source_hash(kernel):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------- workload

def make_workload(name: str, seed: int, length_scale: float = 1.0):
    import workloads

    if name == "agentic":
        return workloads.agentic(seed=seed, scale_lengths=length_scale)
    if name == "llama":
        return workloads.llama(seed=seed)
    if name == "fp8":
        return workloads.fp8(seed=seed, scale_lengths=length_scale)
    if name == "mixed":
        return workloads.mixed(seed=seed, scale_lengths=length_scale)
    if name == "fp8_e5m2":
        return workloads.fp8_e5m2(seed=seed, scale_lengths=length_scale)
    if name == "mixed_fp8":
        return workloads.mixed_fp8(seed=seed, scale_lengths=length_scale)
    if name == "nvfp4":
        return workloads.nvfp4(seed=seed, scale_lengths=length_scale)
    if name == "mixed_nvfp4":
        return workloads.mixed_nvfp4(seed=seed, scale_lengths=length_scale)
    if name == "tiny":
        return workloads.tiny(seed=seed)
    raise ValueError(name)


BASE_SEEDS = {"agentic": 2, "llama": 1, "fp8": 4, "fp8_e5m2": 4, "nvfp4": 4, "mixed": 3, "mixed_fp8": 3, "mixed_nvfp4": 3, "tiny": 0}


def prefix_groups(b):
    """Groups of consecutive sequences and the leading blocks they share (the
    scheduler's knowledge of its forks): (group_start [G+1], shared_blocks [G]) or None."""
    import numpy as np

    if not b.families or all(len(f) == 1 for f in b.families):
        return None
    starts, shared = [0], []
    for fam in b.families:
        if fam != list(range(starts[-1], starts[-1] + len(fam))):
            return None
        n = min(int(b.seq_lens[i]) for i in fam)
        common = n // b.block_size
        for i in fam[1:]:
            eq = b.block_tables[i, :common] == b.block_tables[fam[0], :common]
            common = int(np.argmin(eq)) if not eq.all() else common
        shared.append(common if len(fam) > 1 else 0)
        starts.append(starts[-1] + len(fam))
    return np.array(starts, np.int32), np.array(shared, np.int32)


def shared_split_bytes(b, groups) -> dict:
    """KV bytes read by the shared-prefix kernel (each group's prefix once) and by the
    private-part decode kernel (each sequence's remaining tokens)."""
    import workloads

    kv_tok = 2 * b.num_kv_heads * b.head_size * workloads.ELEM_BYTES[b.kv_dtype]
    starts, shared = groups
    shared_tok, private_tok = 0, 0
    for g in range(len(shared)):
        mem = range(int(starts[g]), int(starts[g + 1]))
        S = 0
        if len(mem) > 1:
            S = min([int(shared[g])] + [int(b.seq_lens[m]) // b.block_size for m in mem]) * b.block_size
        shared_tok += S
        private_tok += sum(int(b.seq_lens[m]) - S for m in mem)
    return {"shared": shared_tok * kv_tok, "private": private_tok * kv_tok}


def window_tokens(b, window: int) -> list:
    """Keys each decode sequence attends: all of them, or the last `window`."""
    return [min(int(n), window) if window > 0 else int(n) for n in b.seq_lens]


def algorithmic_bytes(b, window: int = 0) -> dict:
    """Bytes the attention must move at least (per call), and the logical total.
    With a sliding window (decode) only the window's keys and block-table entries."""
    import workloads

    kv_tok = 2 * b.num_kv_heads * b.head_size * workloads.ELEM_BYTES[b.kv_dtype]
    qb = workloads.ELEM_BYTES[b.q_dtype]
    q_out = 2 * b.total_q * b.num_q_heads * b.head_size * qb
    bs = b.block_size
    spans = [int(n) - (max(0, int(n) - window) // bs * bs if window > 0 else 0) for n in b.seq_lens]
    tables = sum(-(-sp // bs) for sp in spans) * 4 + 4 * b.num_seqs
    logical = int(sum(window_tokens(b, window))) * kv_tok
    unique = logical if window > 0 else unique_kv_tokens(b) * kv_tok
    return {"kv_token_bytes": kv_tok, "logical_kv": logical, "unique_kv": unique,
            "algorithmic": unique + q_out + tables, "logical_total": logical + q_out + tables}


def qk_pairs(b, window: int = 0) -> int:
    """(query token, key token) pairs the attention scores per call: request r's query j
    sits at position p = seq_len - q_len + j and attends keys 0..p when causal (the
    last `window` of them with a sliding window), all seq_len keys otherwise."""
    import numpy as np

    qsl = np.asarray(b.query_start_loc, dtype=np.int64)
    total = 0
    for r, n in enumerate(b.seq_lens):
        n, q = int(n), int(qsl[r + 1] - qsl[r])
        if q <= 0:
            continue
        if not b.causal:
            total += q * n
            continue
        keys = np.arange(n - q, n, dtype=np.int64) + 1
        total += int(np.minimum(keys, window).sum() if window > 0 else keys.sum())
    return total


# ----------------------------------------------------------------------------- oracle (CPU) arm

# The oracle's sample: the first ORACLE_SAMPLE_TOKENS tokens of the workload's
# median-length sequence, one decode query per worker process, each worker on its own
# copy.  The main arm's cpu_baseline and the reference arm time this same sample.
ORACLE_SAMPLE_TOKENS = 32768
REFERENCE_BUDGET_S = 240.0

_CPU_SAMPLE = {}


def _cpu_worker_init(shape):
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    name, seed, length, hq, hkv, d, bs, kv = shape
    import torch

    torch.set_num_threads(1)
    import workloads

    # one sequence with the workload's head shape, dtype and block size
    _CPU_SAMPLE["b"] = workloads.build(name + "_cpu_sample", seed, [length], [1], hq, hkv, d, bs, kv)


def _cpu_worker_run(_):
    import oracle

    b = _CPU_SAMPLE["b"]
    t0 = time.time()
    oracle.paged_decode(b.q, b.q_dtype, b.k_cache, b.v_cache, b.kv_dtype, b.block_tables, b.seq_lens,
                        b.block_size, b.scale, b.k_scale, b.v_scale)
    t1 = time.time()
    return t0, t1, int(b.seq_lens[0])


class OracleSampler:
    """The fp64 oracle timed on host cores: W worker processes (spawned, one BLAS
    thread each), each running the oracle on one decode sequence with the
    workload's head shape, dtype and block size: the first `tokens` tokens of the
    median-length sequence.  Rate = attended tokens / wall time of a step."""

    def __init__(self, b, workers: int, tokens: int = ORACLE_SAMPLE_TOKENS):
        self.b = b
        self.workers = workers
        L = int(sorted(b.seq_lens)[len(b.seq_lens) // 2])  # median-length sequence
        self.full_length = L
        self.length = min(L, int(tokens))
        shape = (b.name, 11, self.length, b.num_q_heads, b.num_kv_heads, b.head_size, b.block_size, b.kv_dtype)
        ctx = mp.get_context("spawn")
        env_keep = os.environ.get("OPENBLAS_NUM_THREADS")
        os.environ["OPENBLAS_NUM_THREADS"] = "1"
        os.environ["OMP_NUM_THREADS"] = "1"
        self.pool = ctx.Pool(workers, initializer=_cpu_worker_init, initargs=(shape,))
        if env_keep is None:
            os.environ.pop("OPENBLAS_NUM_THREADS", None)

    def step(self):
        res = self.pool.map(_cpu_worker_run, range(self.workers), chunksize=1)
        t0 = min(r[0] for r in res)
        t1 = max(r[1] for r in res)
        tokens = sum(r[2] for r in res)
        wall = t1 - t0
        return tokens / wall, wall

    def describe(self):
        which = ("the whole median-length sequence" if self.length == self.full_length else
                 f"the first {self.length} tokens of a median-length ({self.full_length}-token) sequence")
        return (f"{self.workers} processes x 1 decode query over {which}, "
                f"{self.b.num_q_heads}/{self.b.num_kv_heads} heads, head {self.b.head_size}, "
                f"{self.b.kv_dtype}, block {self.b.block_size}, per step")

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_workers():
    n = os.cpu_count() or 1
    return max(1, min(8, n))


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    b = make_workload(args.workload, BASE_SEEDS[args.workload])
    sampler = OracleSampler(b, cpu_workers())
    # The same sample as the main arm's cpu_baseline; shortened only when the whole
    # run (warm-up + timed steps) would not end within the budget.
    _, first = sampler.step()
    if first * (args.steps + args.warmup) > REFERENCE_BUDGET_S:
        tokens = max(256, int(sampler.length * REFERENCE_BUDGET_S / (first * (args.steps + args.warmup))))
        sampler.close()
        sampler = OracleSampler(b, cpu_workers(), tokens)
    for _ in range(max(0, args.warmup - 1)):
        sampler.step()
    rates, walls = [], []
    for _ in range(args.steps):
        r, w = sampler.step()
        rates.append(r)
        walls.append(w)
    sampler.close()
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.median(walls),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(b, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": sampler.workers, "kind": "oracle",
                         "sample": sampler.describe()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(b, args, api=None):
    if api is None:
        api = ("pa_varlen_attn" if b.max_query_len > 1 else
               "pa_decode" if (args.no_shared_prefix or not b.families) else "pa_decode_shared_prefix")
    return {"workload": b.name, "num_seqs": b.num_seqs, "total_context_tokens": int(sum(int(n) for n in b.seq_lens)),
            "max_seq_len": b.max_seq_len, "num_q_heads": b.num_q_heads, "num_kv_heads": b.num_kv_heads,
            "head_size": b.head_size, "block_size": b.block_size, "kv_dtype": b.kv_dtype,
            "q_dtype": b.q_dtype, "new_tokens_per_step": b.total_q,
            "partition_size": args.partition_size or "auto",
            "decode_api": api,
            "length_scale": args.length_scale,
            "sliding_window": args.window or None,
            "l2": "inputs larger than L2 (KV working set >> 129 MB)" if b.name != "tiny" else "tiny (fits L2)"}


# ----------------------------------------------------------------------------- GPU arm

def device_inputs(b, dev) -> dict:
    """The batch's tensors on the device: caches, new K/V, slots, q, tables, lengths."""
    import torch

    import workloads

    kc, vc = workloads.device_cache(b, dev)
    T = workloads.bits_to_torch
    scaled = b.kv_dtype in workloads.SCALED
    d = {"kc": kc, "vc": vc, "key": T(b.key, b.src_dtype, dev), "val": T(b.value, b.src_dtype, dev),
         "slots": torch.from_numpy(b.slot_mapping).to(dev), "q": T(b.q, b.q_dtype, dev),
         "tables": torch.from_numpy(b.block_tables).to(dev), "lens": torch.from_numpy(b.seq_lens).to(dev),
         "qsl": torch.from_numpy(b.query_start_loc).to(dev),
         "ks": torch.tensor([b.k_scale], dtype=torch.float32, device=dev) if scaled else None,
         "vs": torch.tensor([b.v_scale], dtype=torch.float32, device=dev) if scaled else None}
    d["out"] = torch.empty_like(d["q"])
    return d


class Runner:
    """One step of the hot path on a prepared batch: the scatter of the new tokens, then
    the attention call of `mode` -- "varlen" (pa_varlen_attn), "shared"
    (pa_decode_shared_prefix with the batch's fork groups) or "decode" (pa_decode,
    windowed when `window` > 0)."""

    def __init__(self, pa, b, d, dev, mode, part=0, window=0):
        import torch

        self.pa, self.b, self.d, self.dev = pa, b, d, dev
        self.mode, self.part, self.window = mode, part, window
        self.groups = prefix_groups(b) if mode == "shared" else None
        if mode == "shared" and self.groups is None:
            raise ValueError("shared-prefix mode needs a batch of fork families")
        if mode == "varlen":
            wsb = pa.pa_varlen_workspace_size(b.num_seqs, b.total_q, b.max_query_len, b.num_q_heads,
                                              b.num_kv_heads, b.head_size, b.max_seq_len, b.block_size, part)
        elif mode == "shared":
            wsb = pa.pa_decode_shared_prefix_workspace_size(b.num_seqs, len(self.groups[1]), b.num_q_heads,
                                                            b.num_kv_heads, b.head_size, b.max_seq_len,
                                                            b.block_size, part)
            self.gstart = torch.from_numpy(self.groups[0]).to(dev)
            self.gshared = torch.from_numpy(self.groups[1]).to(dev)
            self.max_group = int(max(self.groups[0][1:] - self.groups[0][:-1]))
        else:
            wsb = pa.pa_decode_workspace_size(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_size,
                                              b.max_seq_len, b.block_size, part)
        self.ws = pa.workspace_tensor(wsb, dev)

    def inputs(self) -> list:
        """The per-step inputs a caller copies in (the e2e leg's host-to-device bytes)."""
        d = self.d
        srcs = [d["q"], d["key"], d["val"], d["slots"], d["tables"], d["lens"]]
        if self.mode == "varlen":
            srcs.append(d["qsl"])
        if self.mode == "shared":
            srcs += [self.gstart, self.gshared]
        return srcs

    def step(self, srcs=None, out=None):
        import torch

        pa, b, d = self.pa, self.b, self.d
        q, key, val, slots, tables, lens = (srcs or self.inputs())[:6]
        out = d["out"] if out is None else out
        stream = torch.cuda.current_stream(self.dev)  # the capture stream while a graph is recorded
        pa.pa_reshape_and_cache(key, val, d["kc"], d["vc"], slots, d["ks"], d["vs"], stream)
        if self.mode == "varlen":
            qsl = srcs[6] if srcs else d["qsl"]
            pa.pa_varlen_attn(out, q, d["kc"], d["vc"], tables, qsl, lens, b.max_query_len, b.max_seq_len, b.scale,
                              self.ws, True, d["ks"], d["vs"], self.part, stream)
        elif self.mode == "shared":
            gs, gb = (srcs[-2], srcs[-1]) if srcs else (self.gstart, self.gshared)
            pa.pa_decode_shared_prefix(out, q, d["kc"], d["vc"], tables, lens, b.max_seq_len, b.scale, self.ws,
                                       gs, gb, self.max_group, d["ks"], d["vs"], self.part, stream)
        else:
            pa.pa_decode(out, q, d["kc"], d["vc"], tables, lens, b.max_seq_len, b.scale, self.ws, d["ks"], d["vs"],
                         self.part, stream, window=self.window)


def timed_regions(run, steps, stream, barrier, dev, min_total_ms):
    """Milliseconds per step of K = `steps` calls of `run`, each region bracketed by a
    barrier (and a device synchronise) on both sides and timed with CUDA events on
    the launching stream, maximum over ranks.  The region is repeated until about
    `min_total_ms` of device time has passed (so that a clock sampler running beside
    it sees the GPU under load); returns the per-step times of every repeat."""
    import torch

    out = []
    total = 0.0
    while True:
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1), dev)
        out.append(ms / steps)
        total += ms
        if total >= min_total_ms or len(out) >= 400:
            return out


def traced_eager(pa, run, steps, stream, barrier, dev):
    """One eager K-step region with the library's event tracing on: milliseconds per
    step, and per kernel kind (launches, total ms)."""
    import torch

    pa.pa_trace_read(0, reset=True)
    pa.pa_trace_enable(True)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    barrier()
    pa.pa_trace_enable(False)
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / steps
    return ms, {name: pa.pa_trace_read(k) for k, name in enumerate(pa.TRACE_KINDS)}


def capture(run):
    """The step captured once into a CUDA graph (the library's calls neither
    synchronise nor allocate), returned as its replay function."""
    import torch

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    return graph.replay


def roofline_of(b, runner, trace, ms_per_step, wl, window=0):
    """Roofline of the dominant kernel (or fork-join span) of one measured workload
    (`wl`: its workload key, which names its ncu summary under profiles/)."""
    import workloads

    nbytes = algorithmic_bytes(b, window)
    n_att, ms_att = trace["attention"]
    att_ms = ms_att / max(n_att, 1)
    peak, peak_kind = measured_peaks()
    kernel_ms = {k: (v[1] / v[0] if v[0] else 0.0) for k, v in trace.items()}
    src = f"{peak_kind} MEASURED_PEAKS.json hbm_gbs"
    if runner.mode == "shared":
        # the shared-prefix tiles and the private-remainder decode run concurrently:
        # their fork -> join span is the unit measured against HBM
        sb = shared_split_bytes(b, runner.groups)
        span_ms = kernel_ms.get("shared_span", 0.0)
        achieved = nbytes["algorithmic"] / (span_ms / 1000.0) / 1e9 if span_ms else 0.0
        logical_gbs = nbytes["logical_total"] / (span_ms / 1000.0) / 1e9 if span_ms else 0.0
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profiled_traffic(wl, "shared_prefix_span"),
                "kernel": "shared_prefix_tile_kernel || decode_mma_kernel (one fork-join span)",
                "peak_source": src, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                "byte_basis": "unique physical bytes: each shared prefix block counted once (the "
                              "prefix-sharing decode reads it once per family)",
                "algorithmic_bytes_per_launch": nbytes["algorithmic"],
                "shared_kv_bytes": sb["shared"], "private_kv_bytes": sb["private"],
                "logical_bytes_per_launch": nbytes["logical_total"],
                "logical_kv_bytes_per_launch": nbytes["logical_kv"], "logical_gbs": logical_gbs,
                "logical_over_peak": logical_gbs / peak,
                "logical_note": "logical bytes (every sequence's whole context, shared blocks once per "
                                "member) / span: above 1 because shared blocks are read once, not HBM bandwidth",
                "kernel_ms": span_ms,
                "overlapped_kernel_ms": {"shared_prefix_tile_kernel": kernel_ms.get("shared_prefix", 0.0),
                                         "decode_mma_kernel": att_ms}}
    if runner.mode == "decode":
        achieved = nbytes["algorithmic"] / (att_ms / 1000.0) / 1e9
        shared_blocks = nbytes["unique_kv"] != nbytes["logical_kv"]
        line = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "kernel": "decode_mma_kernel" if b.kv_dtype != "f32" else "attn_generic_kernel",
                "peak_source": src, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                "byte_basis": ("unique physical bytes (shared blocks once; L2 serves the repeats)" if shared_blocks
                               else "logical KV + q + out + block tables"),
                "algorithmic_bytes_per_launch": nbytes["algorithmic"],
                "logical_bytes_per_launch": nbytes["logical_total"],
                "logical_kv_bytes_per_launch": nbytes["logical_kv"],
                "logical_gbs": nbytes["logical_total"] / (att_ms / 1000.0) / 1e9,
                "kernel_ms": att_ms, "merge_ms": kernel_ms.get("merge", 0.0),
                "scatter_ms": kernel_ms.get("reshape_and_cache", 0.0)}
        prof = wl + "_pa_decode" if shared_blocks else wl
        line["traffic"] = profiled_traffic(prof)
        return line
    # varlen: the single-token rows (HBM-bound decode kernel) and the multi-token rows
    # (tensor-bound prefill tiles) run concurrently: their fork -> join span is the
    # unit, measured against HBM for all the bytes both must move, and against the
    # tensor peak for the prefill FLOPs
    vsplit = varlen_split(b)
    span_ms = kernel_ms.get("varlen_span", 0.0)
    qb = workloads.ELEM_BYTES[b.q_dtype]
    pf_rows = int(sum(int(b.query_start_loc[r + 1] - b.query_start_loc[r]) for r in range(b.num_seqs)
                      if int(b.query_start_loc[r + 1] - b.query_start_loc[r]) > 1))
    span_bytes = vsplit["decode_bytes"] + vsplit["prefill_kv_bytes"] + 2 * pf_rows * b.num_q_heads * b.head_size * qb
    achieved = span_bytes / (span_ms / 1000.0) / 1e9 if span_ms else 0.0
    pf_tflops = vsplit["prefill_flops"] / (span_ms / 1000.0) / 1e12 if span_ms else 0.0
    tpeak, tkind = measured_bf16_sustained()
    kernel_name = "decode_mma_kernel || prefill_tc_kernel (one fork-join span)"
    # per step: the prefill tiles launch twice when decode rows run beside them
    n_span = max(trace["varlen_span"][0], 1)
    overlapped = {"decode_mma_kernel": att_ms, "prefill_tc_kernel": trace["prefill_tiles"][1] / n_span}
    traffic = profiled_traffic(wl, "varlen_span")
    hbm_line = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "kernel": kernel_name, "peak_source": src,
                "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                "algorithmic_bytes_per_launch": span_bytes, "kernel_ms": span_ms,
                "overlapped_kernel_ms": overlapped}
    tensor_line = {"bound": "tensor", "achieved": pf_tflops, "peak": tpeak, "unit": "TFLOP/s",
                   "frac": pf_tflops / tpeak, "kernel": kernel_name, "kernel_ms": span_ms,
                   "algorithmic_flops_per_launch": vsplit["prefill_flops"], "traffic": traffic,
                   "peak_source": f"{tkind} MEASURED_PEAKS.json bf16_tflops_sustained",
                   "overlapped_kernel_ms": overlapped}
    # the binding resource: the larger of the two lower bounds on the span
    main, other = ((hbm_line, tensor_line) if hbm_line["frac"] >= tensor_line["frac"] else (tensor_line, hbm_line))
    return dict(main, secondary={k: v for k, v in other.items() if k != "overlapped_kernel_ms"})


def e2e_pipelined(runner, steps, stream, barrier, dev, use_graph):
    """The step end to end through the public API from pinned host memory, pipelined.

    Every input of a step (q, new K/V, slots, block tables, lengths, query_start_loc,
    prefix groups) sits in one pinned host buffer at 256-byte aligned offsets and
    moves with one host-to-device copy; the output returns with one device-to-host
    copy.  Two device input buffers and two outputs alternate between steps: a copy
    stream moves step i+1's inputs in while step i computes, and step i's output out
    while step i+1 computes.  Copy i+1 waits for step i-1 to finish with that input
    buffer; step i+2 waits (through copy i+2, behind it on the copy stream) for
    output i to have left.  Every copy of every step is inside the timed region."""
    import torch

    srcs = runner.inputs()
    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()

    def carve(buf, t, o):
        return buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for t, o in zip(srcs, offs):
        carve(hbuf, t, o).copy_(t)
    dbufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [[carve(db, t, o) for t, o in zip(srcs, offs)] for db in dbufs]
    outs = [torch.empty_like(runner.d["out"]) for _ in range(2)]
    houts = [torch.empty(outs[0].shape, dtype=outs[0].dtype).pin_memory() for _ in range(2)]
    computes = [lambda p=p: runner.step(views[p], outs[p]) for p in range(2)]
    launch, capture_error = "eager", None
    if use_graph:
        try:
            computes = [capture(c) for c in computes]
            launch = "cuda_graph_replay (compute) + copies on a second stream"
        except RuntimeError as ex:  # time the eager step instead, and say why
            capture_error = str(ex).splitlines()[0][:200]
            torch.cuda.synchronize(dev)
    cs = torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def run_k(k):
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            dbufs[0].copy_(hbuf, non_blocking=True)
            h2d_done[0].record(cs)
        for i in range(k):
            c, n = i % 2, 1 - i % 2
            if i + 1 < k:
                with torch.cuda.stream(cs):
                    cs.wait_event(comp_done[n])  # step i-1 is done with input buffer n
                    dbufs[n].copy_(hbuf, non_blocking=True)
                    h2d_done[n].record(cs)
            stream.wait_event(h2d_done[c])
            computes[c]()
            comp_done[c].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(comp_done[c])
                houts[c].copy_(outs[c], non_blocking=True)
        stream.wait_stream(cs)

    run_k(3)  # warm-up (and first use of the copy stream)
    barrier()
    t0 = time.perf_counter()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    run_k(steps)
    f1.record(stream)
    barrier()
    wall_ms = (time.perf_counter() - t0) * 1000.0
    e2e_ms = max_over_ranks(max(f0.elapsed_time(f1), wall_ms), dev) / steps
    # the copied inputs are the device-resident ones: the output read back must equal
    # the device-resident step's
    torch.cuda.synchronize(dev)
    runner.step()
    torch.cuda.synchronize(dev)
    same = bool(torch.equal(houts[(steps - 1) % 2], runner.d["out"].cpu()))
    line = {"ms_per_step": e2e_ms, "h2d_bytes_per_step": total,
            "d2h_bytes_per_step": houts[0].numel() * houts[0].element_size(),
            "copies_per_step": {"h2d": 1, "d2h": 1}, "step_launch": launch, "pipelined": True,
            "output_equals_device_step": same}
    if capture_error:
        line["capture_error"] = capture_error
    return line


def measure(pa, b, d, dev, mode, args, wl, stream, barrier, steps, warmup, min_total_ms, window=0, e2e=False):
    """Warm-up, one traced eager K-step region, then repeated graph-replayed K-step
    regions (eager with --no-graph); the roofline of the dominant kernel."""
    runner = Runner(pa, b, d, dev, mode, args.partition_size, window)
    for _ in range(warmup):
        runner.step()
    torch_sync(dev)
    flags = pa.pa_get_error_flags()
    if flags:
        raise RuntimeError(f"{b.name}: device error flags {flags:#x} during warm-up")
    ms_eager, trace = traced_eager(pa, runner.step, steps, stream, barrier, dev)
    run = runner.step
    if not args.no_graph:
        run = capture(runner.step)
        for _ in range(3):
            run()
    per_step = timed_regions(run, steps, stream, barrier, dev, min_total_ms)
    ms = statistics.median(per_step)
    res = {"runner": runner, "trace": trace, "ms_per_step": ms, "ms_per_step_eager": ms_eager,
           "repeats": len(per_step), "ms_per_step_min": min(per_step), "ms_per_step_max": max(per_step),
           "step_launch": "eager" if args.no_graph else "cuda_graph_replay",
           "launches": sum(n for name, (n, _) in trace.items() if not name.endswith("_span"))}
    res["roofline"] = roofline_of(b, runner, trace, ms, wl, window)
    if e2e:
        res["e2e"] = e2e_pipelined(runner, steps, stream, barrier, dev, not args.no_graph)
    flags = pa.pa_get_error_flags()
    if flags:
        raise RuntimeError(f"{b.name}: device error flags {flags:#x} during the timed region")
    return res


def torch_sync(dev):
    import torch

    torch.cuda.synchronize(dev)


# The other configurations of the path, measured in the same run as the headline:
# (entry name, workload, attention call).
CONFIG_LEGS = (("tiny", "tiny", "decode"), ("llama", "llama", "decode"), ("mixed", "mixed", "varlen"),
               ("fp8", "fp8", "decode"), ("agentic_pa_decode", "agentic", "decode"),
               ("mixed_fp8", "mixed_fp8", "varlen"), ("nvfp4", "nvfp4", "decode"),
               ("fp8_e5m2", "fp8_e5m2", "decode"), ("mixed_nvfp4", "mixed_nvfp4", "varlen"))


def compact(res, b, window=0) -> dict:
    """The fields of one measured configuration that the bench line reports."""
    rl = res["roofline"]
    ctx = int(sum(window_tokens(b, window)))
    keep = ("bound", "achieved", "peak", "unit", "frac", "kernel", "kernel_ms", "byte_basis", "traffic",
            "algorithmic_bytes_per_launch", "algorithmic_flops_per_launch", "logical_gbs", "merge_ms", "scatter_ms",
            "overlapped_kernel_ms")
    out = {"workload": b.name, "decode_api": {"decode": "pa_decode", "varlen": "pa_varlen_attn",
                                              "shared": "pa_decode_shared_prefix"}[res["runner"].mode],
           "ms_per_step": res["ms_per_step"], "ms_per_step_eager": res["ms_per_step_eager"],
           "timed_repeats": res["repeats"], "value": ctx / (res["ms_per_step"] / 1000.0), "unit": UNIT,
           "gpu_launches": res["launches"], "roofline": {k: rl[k] for k in keep if k in rl}}
    if "secondary" in rl:
        out["roofline"]["secondary"] = {k: rl["secondary"][k] for k in keep if k in rl["secondary"]}
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    import paged_kv_cache_pagedattention_gb300 as pa

    b = make_workload(args.workload, rank_seed(BASE_SEEDS[args.workload], rank), args.length_scale)
    varlen = b.max_query_len > 1
    if args.window and varlen:
        raise SystemExit("--window applies to the decode workloads (llama, fp8, agentic)")
    mode = ("varlen" if varlen else
            "shared" if (not args.no_shared_prefix and not args.window and prefix_groups(b) is not None) else
            "decode")
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    d = device_inputs(b, dev)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus) if rank == 0 else None
    if sampler:
        sampler.start()
    head = measure(pa, b, d, dev, mode, args, args.workload, stream, barrier, args.steps, args.warmup, args.min_timed_ms,
                   window=args.window, e2e=not args.no_e2e)
    clocks = sampler.stop() if sampler else None
    ms_per_step = head["ms_per_step"]
    ctx_tokens = int(sum(window_tokens(b, args.window)))
    tok_s = ctx_tokens * world / (ms_per_step / 1000.0)
    qk = qk_pairs(b, args.window)
    roofline = head["roofline"]
    e2e = None
    if "e2e" in head:
        e2e = dict(head["e2e"], value=ctx_tokens * world / (head["e2e"]["ms_per_step"] / 1000.0), unit=UNIT)
    if clocks and clocks.get("sm_mhz"):
        clocks["ms_per_step_x_median_sm_mhz"] = ms_per_step * clocks["sm_mhz"]

    # ---- every other configuration of the path, measured in this run (one GPU)
    configs = None
    if world == 1 and not args.no_configs and not args.window and args.length_scale == 1.0:
        configs = {}
        for name, wl, leg_mode in CONFIG_LEGS:
            if wl == args.workload and leg_mode == mode:
                continue  # the headline itself
            # the headline's batch is reused; any other workload's tensors are freed after its leg
            bb = b if wl == args.workload else make_workload(wl, BASE_SEEDS[wl])
            dd = d if wl == args.workload else device_inputs(bb, dev)
            res = measure(pa, bb, dd, dev, leg_mode, args, wl, stream, barrier, args.steps, args.warmup,
                          args.min_timed_ms / 4)
            configs[name] = compact(res, bb)
            del res, dd
            torch.cuda.synchronize(dev)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.window:
        sampler_cpu = OracleSampler(b, cpu_workers())
        rates, walls = [], []
        for _ in range(3):
            r, w = sampler_cpu.step()
            rates.append(r)
            walls.append(w)
        sampler_cpu.close()
        cpu = {"value": statistics.median(rates), "unit": UNIT, "cores": sampler_cpu.workers, "kind": "oracle",
               "sample": sampler_cpu.describe() + " (median of 3 steps)", "wall_s": statistics.median(walls)}

    if world > 1:
        dist.barrier()
    if rank == 0:
        trace = head["trace"]
        kernel_ms = {k: (v[1] / v[0] if v[0] else 0.0) for k, v in trace.items()}
        line = {"metric": METRIC, "value": tok_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if b.kv_dtype == "bf16" else b.kv_dtype,
                "data": "synthetic (seeded N(0,1) values, seeded block placement)",
                "config": workload_config(b, args, {"varlen": "pa_varlen_attn", "shared": "pa_decode_shared_prefix",
                                                    "decode": "pa_decode"}[mode]),
                "hbm_gbs": roofline["achieved"] if roofline["unit"] == "GB/s" else
                roofline.get("secondary", {}).get("achieved"),
                "qk_pairs_per_step": qk, "qk_pairs_per_s": qk * world / (ms_per_step / 1000.0),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "step_launch": head["step_launch"],
                "timed_repeats": head["repeats"],
                "timed_repeats_note": "each repeat times exactly `steps` steps between barriers; ms_per_step "
                                      "is the median over repeats",
                "ms_per_step_min": head["ms_per_step_min"], "ms_per_step_max": head["ms_per_step_max"],
                "ms_per_step_eager": head["ms_per_step_eager"],
                "gpu_launches": head["launches"],
                "launches_by_kernel": {k: v[0] for k, v in trace.items() if v[0] and not k.endswith("_span")},
                "kernel_ms_by_kind": {k: v for k, v in kernel_ms.items() if v},
                "clocks": clocks, "configs": configs}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_copy_blocks(args):
    """Copy-on-write block copy measured alone: a Llama-sized bf16 pool (18,432
    blocks of 8 KV heads x 16 slots x 128 dims) and 4,096 disjoint (src, dst) pairs
    per step, two pair sets alternating (each step moves 537 MB: > L2)."""
    import numpy as np
    import torch

    import paged_kv_cache_pagedattention_gb300 as pa

    rank, local_rank, world = dist_env()
    if world > 1 and rank != 0:
        return 0  # one GPU's kernel; further ranks would only repeat it
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    nb, hkv, bs, d, npairs = 18432, 8, 16, 128, 4096
    g = torch.Generator(device=dev).manual_seed(11)
    kc = torch.randn(nb, hkv, bs, d, device=dev, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d, device=dev, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(12)
    maps = []
    for _ in range(2):
        perm = rng.permutation(nb)
        maps.append(np.stack([perm[:npairs], perm[npairs:2 * npairs]], 1).astype(np.int64))
    dmaps = [torch.from_numpy(m).to(dev) for m in maps]
    stream = torch.cuda.current_stream(dev)
    block_bytes = hkv * bs * d * 2
    moved = 2 * 2 * block_bytes * npairs  # K and V, each read once and written once
    for i in range(args.warmup):
        pa.pa_copy_blocks(kc, vc, dmaps[i % 2], stream)
    torch.cuda.synchronize(dev)
    if pa.pa_get_error_flags():
        raise RuntimeError("device error flags during warm-up")
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus)
    sampler.start()
    pa.pa_trace_read(0, reset=True)
    pa.pa_trace_enable(True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        pa.pa_copy_blocks(kc, vc, dmaps[i % 2], stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    pa.pa_trace_enable(False)
    clocks = sampler.stop()
    n_copy, ms_copy = pa.pa_trace_read(7)
    ms_per_step = e0.elapsed_time(e1) / args.steps
    gbs = moved / (ms_per_step / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    kern_ms = ms_copy / n_copy if n_copy else ms_per_step
    achieved = moved / (kern_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": None, "kernel": "copy_blocks_kernel", "kernel_ms": kern_ms,
                "algorithmic_bytes_per_launch": moved, "peak_source": f"{peak_kind} MEASURED_PEAKS.json hbm_gbs"}
    e2e = None
    if not args.no_e2e:
        hmaps = [torch.from_numpy(m).pin_memory() for m in maps]
        dmap = torch.empty_like(dmaps[0])
        hflags = torch.empty(1, dtype=torch.int32).pin_memory()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            dmap.copy_(hmaps[i % 2], non_blocking=True)
            pa.pa_copy_blocks(kc, vc, dmap, stream)
            hflags.copy_(dmap[0, :1].to(torch.int32), non_blocking=True)  # completion read-back
        t1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = t0.elapsed_time(t1) / args.steps
        e2e = {"value": moved / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": maps[0].nbytes,
               "d2h_bytes_per_step": 4, "ms_per_step": e2e_ms}
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        # the oracle copying 64 pairs of host blocks of the same shape
        kh = np.random.default_rng(13).integers(0, 2 ** 16, size=(256, hkv, bs, d), dtype=np.uint16)
        vh = kh.copy()
        pairs = np.stack([np.arange(64), np.arange(64, 128)], 1)
        t = time.perf_counter()
        reps = 0
        while time.perf_counter() - t < 2.0:
            oracle.copy_blocks(kh, vh, pairs)
            reps += 1
        dt = time.perf_counter() - t
        cpu = {"value": reps * 64 * 4 * block_bytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{reps} x 64 block pairs (8 x 16 x 128 bf16) in 2 s"}
    line = {"metric": "copy-on-write block copy: HBM GB/s (bytes read + written)", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "replicas only", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) cache, seeded disjoint pairs)",
            "config": {"workload": "copy_blocks", "num_blocks": nb, "num_kv_heads": hkv, "block_size": bs,
                       "head_size": d, "pairs_per_step": npairs, "l2": "537 MB moved per step (> L2)"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n_copy, "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="agentic")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of replaying the step captured in a CUDA graph")
    ap.add_argument("--window", type=int, default=0,
                    help="decode workloads: sliding-window attention over the last W keys (pa_decode_windowed)")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="agentic: call pa_decode instead of pa_decode_shared_prefix")
    ap.add_argument("--op", choices=("attention", "copy_blocks"), default="attention",
                    help="copy_blocks: time the copy-on-write block copy alone")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure the headline workload only (skip the other configurations of the path)")
    ap.add_argument("--min-timed-ms", type=float, default=1500.0,
                    help="repeat the K-step timed region until about this much device time has passed")
    ap.add_argument("--length-scale", type=float, default=1.0,
                    help="shrink every sequence length (profiling captures only; 1.0 = the named workload)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "copy_blocks":
        return run_copy_blocks(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
