"""Seeded synthetic inputs for the paged KV cache hot path.

This module only produces inputs: sequence lengths, block tables with a
shuffled physical placement, slot mappings, queries, new keys/values and cache
contents.  It holds none of the method's arithmetic (no attention, no
quantisation rule of its own: casts go through torch's library casts) and is
the one module both the oracle-side tests and the CUDA-side tests/bench use.

Every array of element values is held as raw bits (uint32 for f32, uint16 for
f16/bf16, uint8 for FP8 e4m3) so that both sides read exactly the same inputs.

Workloads (shapes and distributions from the serving pages' workloads):

* ``tiny``    4 sequences {17, 64, 129, 200}, 8 q heads / 2 KV heads, d 64, fp32,
              block 16, 64 physical blocks in a seeded permutation, scale 1/8.
* ``llama``   Llama-3-8B-shaped decode layer: batch 64, lengths U[512, 4096],
              32/8 heads, d 128, bf16, block 16, pool of 2x the needed blocks.
* ``agentic`` long-context decode: batch 16 = 3 families of (parent + 4 forks)
              + 1 lone parent, family length log-normal (median 142,000, sigma
              0.5) clipped to [32768, 262144]; forks share the first 96% of their
              parent's block-table entries; 64/8 heads, d 128, bf16, block 16.
* ``mixed``   flattened varlen step: 4 prefill chunks of 512 tokens on cached
              prefixes U[8192, 65536] + 128 decodes with context U[1024, 32768];
              32/8 heads, d 128, bf16, block 16; 2,176 new tokens.
* ``fp8``     batch 256, lengths U[1024, 32768], 32/8 heads, d 128, FP8 e4m3
              K/V with per-tensor scale 2^-6, bf16 q/out, block 32.
* ``nvfp4``   the ``fp8`` decode shapes with an NVFP4 cache (4-bit E2M1 codes,
              one E4M3 scale per 16 elements, per-tensor fp32 scale 0.375).

NVFP4 caches are ``[num_blocks][num_kv_heads][tile_bytes]`` bytes: a (block, KV
head) tile holds block_size rows of head_size/2 code bytes, then block_size rows
of head_size/16 block-scale bytes.  Their history is drawn as random bits, not
quantised from values (this module has no quantiser): uniform E2M1 codes, and
block-scale codes uniform over the E4M3 codes 0x20..0x47 (values 0.125 .. 3.75),
so that code x block scale x 0.375 spans about +-8 with a mean magnitude near
0.6.  New tokens' keys and values are N(0,1) as for every other cache type; the
scatter under test quantises them.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# bytes per stored element; NVFP4: half a byte of code plus a sixteenth of a scale byte
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1, "fp8_e5m2": 1, "nvfp4": 0.5625}
BITS_NP = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "fp8_e4m3": np.uint8, "fp8_e5m2": np.uint8,
           "nvfp4": np.uint8}
FP8 = ("fp8_e4m3", "fp8_e5m2")
NVFP4 = "nvfp4"
SCALED = FP8 + (NVFP4,)  # cache types that carry fp32 scales
# largest finite magnitude of each FP8 format: torch's casts do not saturate
FP8_MAX = {"fp8_e4m3": 448.0, "fp8_e5m2": 57344.0}


@dataclasses.dataclass
class PagedBatch:
    """One step's worth of inputs for scatter + attention over a paged KV cache."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    q_dtype: str                 # dtype of q and of the attention output
    kv_dtype: str                # dtype stored in the cache
    src_dtype: str               # dtype of the new keys / values given to the scatter
    scale: float                 # softmax scale
    k_scale: float
    v_scale: float
    causal: bool
    seq_lens: np.ndarray         # int32 [B], context incl. the new tokens
    query_start_loc: np.ndarray  # int32 [B+1]
    block_tables: np.ndarray     # int32 [B][max_blocks_per_seq], unused entries -1
    slot_mapping: np.ndarray     # int64 [T_new]
    q: np.ndarray                # bits [T_q][Hq][d] of q_dtype
    key: np.ndarray              # bits [T_new][Hkv][d] of src_dtype
    value: np.ndarray            # bits [T_new][Hkv][d] of src_dtype
    k_cache: Optional[np.ndarray]  # bits [nb][Hkv][bs][d] of kv_dtype, or None (filled on device)
    v_cache: Optional[np.ndarray]
    cache_seed: int
    families: Optional[list] = None  # agentic: list of lists of sequence indices

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max())

    @property
    def max_query_len(self) -> int:
        return int(np.diff(self.query_start_loc).max())

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


# --------------------------------------------------------------------------
# value generation (torch library casts; no rounding rule of our own)
# --------------------------------------------------------------------------

def normal_bits(rng: np.random.Generator, shape, dtype: str, scale: float = 1.0) -> np.ndarray:
    """N(0,1) fp32 values cast to ``dtype`` (torch casts), returned as raw bits.

    For FP8 the value stored is x / scale cast by torch to float8_e4m3fn (e5m2)
    after clamping to +-448 (+-57344): torch's casts do not saturate.
    """
    import torch

    x = torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32))
    return _cast_bits(x, dtype, scale)


def _cast_bits(x, dtype: str, scale: float = 1.0) -> np.ndarray:
    import torch

    if dtype == "f32":
        return x.to(torch.float32).contiguous().view(torch.int32).numpy().view(np.uint32)
    if dtype == "f16":
        return x.to(torch.float16).contiguous().view(torch.int16).numpy().view(np.uint16)
    if dtype == "bf16":
        return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)
    if dtype in FP8:
        m = FP8_MAX[dtype]
        sc = torch.as_tensor(np.asarray(scale, dtype=np.float32))
        if sc.dim() == 1:  # one scale per KV head of a [blocks][heads][slots][dim] cache
            sc = sc.view(1, -1, 1, 1)
        y = (x.to(torch.float32) / sc).clamp(-m, m).to(torch_dtype(dtype))
        return y.contiguous().view(torch.uint8).numpy()
    raise ValueError(dtype)


def nvfp4_tile_bytes(block_size: int, head_size: int) -> int:
    """Storage size of one (block, KV head) tile of an NVFP4 cache."""
    return block_size * head_size // 2 + block_size * head_size // 16


def nvfp4_random_cache(rng: np.random.Generator, num_blocks: int, num_kv_heads: int, block_size: int,
                       head_size: int) -> np.ndarray:
    """Random NVFP4 cache bytes: uniform code bytes, block-scale codes in 0x20..0x47."""
    codes = rng.integers(0, 256, size=(num_blocks, num_kv_heads, block_size * head_size // 2), dtype=np.uint8)
    scales = rng.integers(0x20, 0x48, size=(num_blocks, num_kv_heads, block_size * head_size // 16),
                          dtype=np.uint8)
    return np.concatenate([codes, scales], axis=2)


def torch_dtype(dtype: str):
    import torch

    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
            "fp8_e4m3": torch.float8_e4m3fn, "fp8_e5m2": torch.float8_e5m2}[dtype]


def bits_to_torch(bits: np.ndarray, dtype: str, device=None):
    """Raw bits -> torch tensor of the element type (FP8 e4m3 as uint8 codes, e5m2 as
    torch.float8_e5m2 so the format travels with the tensor)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits))
    if dtype == "f32":
        t = t.view(torch.int32).view(torch.float32)
    elif dtype in ("f16", "bf16"):
        t = t.view(torch.int16).view(torch_dtype(dtype))
    elif dtype in ("fp8_e4m3", "nvfp4"):
        t = t.view(torch.uint8)
    elif dtype == "fp8_e5m2":
        t = t.view(torch.uint8).view(torch.float8_e5m2)
    if device is not None:
        t = t.to(device)
    return t


def torch_to_bits(t, dtype: str) -> np.ndarray:
    """torch tensor (any device) -> raw bits numpy array."""
    import torch

    t = t.detach().contiguous().cpu()
    if dtype == "f32":
        return t.view(torch.int32).numpy().view(np.uint32)
    if dtype in ("f16", "bf16"):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


# --------------------------------------------------------------------------
# layout construction
# --------------------------------------------------------------------------

def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _assign_blocks(rng, seq_lens, block_size, pool_factor=2.0, min_pool=0,
                   shared=None):
    """Block tables for ``seq_lens`` drawn from a shuffled pool of physical blocks.

    ``shared`` optionally maps a sequence index to (source sequence, number of
    leading entries to copy): those entries reuse the source's physical blocks.
    Returns (block_tables int32 [B][max_blocks] with -1 padding, num_blocks).
    """
    nblk = [_ceil_div(int(n), block_size) for n in seq_lens]
    shared = shared or {}
    fresh = sum(nb - shared.get(i, (None, 0))[1] for i, nb in enumerate(nblk))
    pool = max(int(np.ceil(pool_factor * fresh)), fresh, min_pool)
    order = rng.permutation(pool).astype(np.int32)
    max_blocks = max(nblk)
    table = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    nxt = 0
    for i, nb in enumerate(nblk):
        src, nshare = shared.get(i, (None, 0))
        if nshare:
            table[i, :nshare] = table[src, :nshare]
        take = nb - nshare
        table[i, nshare:nb] = order[nxt: nxt + take]
        nxt += take
    return table, pool


def _slots_for(table, seq_lens, q_lens, block_size):
    """Flat slots of each request's last q_len positions (phys * block_size + offset)."""
    slots = []
    for i, (n, ql) in enumerate(zip(seq_lens, q_lens)):
        for pos in range(int(n) - int(ql), int(n)):
            slots.append(int(table[i, pos // block_size]) * block_size + pos % block_size)
    return np.array(slots, dtype=np.int64)


def build(name, seed, seq_lens, q_lens, num_q_heads, num_kv_heads, head_size,
          block_size, kv_dtype, q_dtype=None, src_dtype=None, scale=None,
          fp8_scale=2.0 ** -6, pool_factor=2.0, min_pool=0, shared=None,
          host_cache=True, causal=True, families=None, nvfp4_scale=0.375) -> PagedBatch:
    """Generic builder: lengths, placement, slots, q / new K,V and (optionally) cache bits.

    ``fp8_scale`` (FP8) / ``nvfp4_scale`` (NVFP4) is the caches' fp32 scale: a float,
    or one value per KV head (K uses them in order, V reversed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    q_dtype = q_dtype or ("bf16" if kv_dtype in SCALED else kv_dtype)
    src_dtype = src_dtype or q_dtype
    if scale is None:
        scale = 1.0 / float(np.sqrt(head_size))
    table, nb = _assign_blocks(rng, seq_lens, block_size, pool_factor, min_pool, shared)
    qsl = np.zeros(len(seq_lens) + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    slots = _slots_for(table, seq_lens, q_lens, block_size)
    tq = int(qsl[-1])
    q = normal_bits(rng, (tq, num_q_heads, head_size), q_dtype)
    key = normal_bits(rng, (tq, num_kv_heads, head_size), src_dtype)
    value = normal_bits(rng, (tq, num_kv_heads, head_size), src_dtype)
    sc = fp8_scale if kv_dtype in FP8 else nvfp4_scale if kv_dtype == NVFP4 else 1.0
    ks = vs = sc
    if kv_dtype in SCALED and np.ndim(sc):  # one scale per KV head
        ks = np.asarray(sc, dtype=np.float32)
        vs = ks[::-1].copy()
        assert ks.shape == (num_kv_heads,)
    k_cache = v_cache = None
    cache_seed = int(rng.integers(0, 2**31 - 1))
    if host_cache:
        crng = np.random.Generator(np.random.PCG64(cache_seed))
        if kv_dtype == NVFP4:
            k_cache = nvfp4_random_cache(crng, nb, num_kv_heads, block_size, head_size)
            v_cache = nvfp4_random_cache(crng, nb, num_kv_heads, block_size, head_size)
        else:
            shape = (nb, num_kv_heads, block_size, head_size)
            k_cache = normal_bits(crng, shape, kv_dtype, ks)
            v_cache = normal_bits(crng, shape, kv_dtype, vs)
    return PagedBatch(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                      head_size=head_size, block_size=block_size, num_blocks=nb,
                      q_dtype=q_dtype, kv_dtype=kv_dtype, src_dtype=src_dtype,
                      scale=float(scale), k_scale=ks if np.ndim(ks) else float(ks),
                      v_scale=vs if np.ndim(vs) else float(vs),
                      causal=causal, seq_lens=seq_lens, query_start_loc=qsl,
                      block_tables=table, slot_mapping=slots, q=q, key=key, value=value,
                      k_cache=k_cache, v_cache=v_cache, cache_seed=cache_seed,
                      families=families)


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------

def tiny(seed: int = 0) -> PagedBatch:
    lens = [17, 64, 129, 200]
    return build("tiny", seed, lens, [1] * 4, 8, 2, 64, 16, "f32", scale=1.0 / 8.0,
                 pool_factor=0.0, min_pool=64)


def llama(seed: int = 1, host_cache: bool = False) -> PagedBatch:
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    return build("llama3_8b_decode", seed, lens, [1] * 64, 32, 8, 128, 16, "bf16",
                 host_cache=host_cache)


def agentic_lengths(seed: int):
    """Family lengths: log-normal, median 142,000, sigma 0.5, clipped to [32768, 262144]."""
    rng = np.random.Generator(np.random.PCG64(seed + 2000))
    L = np.exp(rng.normal(np.log(142000.0), 0.5, size=4))
    return np.clip(np.round(L), 32768, 262144).astype(np.int64)


def agentic(seed: int = 2, host_cache: bool = False, scale_lengths: float = 1.0) -> PagedBatch:
    """3 families of (parent + 4 forks) + 1 lone parent; forks share 96% of the blocks.

    ``scale_lengths`` < 1 shrinks every length (same structure) for oracle-sized runs.
    """
    bs = 16
    fam_len = agentic_lengths(seed)
    if scale_lengths != 1.0:
        fam_len = np.maximum(np.round(fam_len * scale_lengths).astype(np.int64), 2 * bs)
    lens, shared, families = [], {}, []
    for f in range(3):
        parent = len(lens)
        members = [parent]
        L = int(fam_len[f])
        lens.append(L)
        nshare = int(np.floor(0.96 * _ceil_div(L, bs)))
        for _ in range(4):
            shared[len(lens)] = (parent, nshare)
            members.append(len(lens))
            lens.append(L)
        families.append(members)
    families.append([len(lens)])
    lens.append(int(fam_len[3]))
    return build("agentic_long_context_decode", seed, lens, [1] * 16, 64, 8, 128, bs, "bf16",
                 shared=shared, families=families, host_cache=host_cache)


def mixed(seed: int = 3, host_cache: bool = False, scale_lengths: float = 1.0,
          chunk: int = 512, n_prefill: int = 4, n_decode: int = 128, kv_dtype: str = "bf16") -> PagedBatch:
    """Flattened chunked-prefill + decode step; prefill requests first."""
    rng = np.random.Generator(np.random.PCG64(seed + 3000))
    prefix = rng.integers(8192, 65536, size=n_prefill, endpoint=True)
    ctx = rng.integers(1024, 32768, size=n_decode, endpoint=True)
    if scale_lengths != 1.0:
        prefix = np.maximum(np.round(prefix * scale_lengths).astype(np.int64), 1)
        ctx = np.maximum(np.round(ctx * scale_lengths).astype(np.int64), 1)
    lens = [int(p) + chunk for p in prefix] + [int(c) for c in ctx]
    q_lens = [chunk] * n_prefill + [1] * n_decode
    if kv_dtype == "bf16":
        return build("mixed_chunked_prefill_decode", seed, lens, q_lens, 32, 8, 128, 16, "bf16",
                     host_cache=host_cache)
    return build("mixed_chunked_prefill_decode_" + kv_dtype, seed, lens, q_lens, 32, 8, 128, 16, kv_dtype,
                 q_dtype="bf16", src_dtype="bf16", host_cache=host_cache)


def mixed_nvfp4(seed: int = 3, host_cache: bool = False, scale_lengths: float = 1.0) -> PagedBatch:
    """The mixed step with an NVFP4 cache (tensor scale 0.375)."""
    return mixed(seed, host_cache, scale_lengths, kv_dtype=NVFP4)


def mixed_fp8(seed: int = 3, host_cache: bool = False, scale_lengths: float = 1.0) -> PagedBatch:
    """The mixed step with an FP8 e4m3 cache (per-tensor scales 2^-6)."""
    return mixed(seed, host_cache, scale_lengths, kv_dtype="fp8_e4m3")


def fp8(seed: int = 4, host_cache: bool = False, batch: int = 256,
        scale_lengths: float = 1.0, kv_dtype: str = "fp8_e4m3") -> PagedBatch:
    rng = np.random.Generator(np.random.PCG64(seed + 4000))
    lens = rng.integers(1024, 32768, size=batch, endpoint=True)
    if scale_lengths != 1.0:
        lens = np.maximum(np.round(lens * scale_lengths).astype(np.int64), 1)
    name = {"fp8_e4m3": "fp8_kv_decode", "fp8_e5m2": "fp8_e5m2_kv_decode", NVFP4: "nvfp4_kv_decode"}[kv_dtype]
    return build(name, seed, lens, [1] * batch, 32, 8, 128, 32, kv_dtype,
                 q_dtype="bf16", src_dtype="bf16", host_cache=host_cache)


def fp8_e5m2(seed: int = 4, host_cache: bool = False, scale_lengths: float = 1.0) -> PagedBatch:
    """The FP8 decode workload with an e5m2 cache."""
    return fp8(seed, host_cache, scale_lengths=scale_lengths, kv_dtype="fp8_e5m2")


def nvfp4(seed: int = 4, host_cache: bool = False, scale_lengths: float = 1.0) -> PagedBatch:
    """The FP8 decode shapes with an NVFP4 cache."""
    return fp8(seed, host_cache, scale_lengths=scale_lengths, kv_dtype=NVFP4)


NAMED = {"tiny": tiny, "llama": llama, "agentic": agentic, "mixed": mixed, "fp8": fp8, "mixed_fp8": mixed_fp8,
         "fp8_e5m2": fp8_e5m2, "nvfp4": nvfp4, "mixed_nvfp4": mixed_nvfp4}


# --------------------------------------------------------------------------
# device-side cache fill for full-size workloads
# --------------------------------------------------------------------------

def device_cache(batch: PagedBatch, device, chunk_elems: int = 1 << 28):
    """Allocate k_cache / v_cache on ``device`` and fill them from ``batch.cache_seed``.

    Host-built batches are copied; otherwise the values are N(0,1) drawn with a
    seeded torch generator on the device and cast with torch's casts (FP8:
    x / scale clamped to +-448, then float8_e4m3fn).  Deterministic for a given
    seed, shape and torch build.
    """
    import torch

    shape = (batch.num_blocks, batch.num_kv_heads, batch.block_size, batch.head_size)
    if batch.k_cache is not None:
        return (bits_to_torch(batch.k_cache, batch.kv_dtype, device),
                bits_to_torch(batch.v_cache, batch.kv_dtype, device))
    if batch.kv_dtype == NVFP4:
        # uniform code bytes, block-scale bytes in 0x20..0x47 (as nvfp4_random_cache)
        gen = torch.Generator(device=device)
        gen.manual_seed(batch.cache_seed)
        ncode = batch.block_size * batch.head_size // 2
        tile = nvfp4_tile_bytes(batch.block_size, batch.head_size)
        caches = []
        for _ in range(2):
            c = torch.empty((batch.num_blocks, batch.num_kv_heads, tile), dtype=torch.uint8, device=device)
            step = max(1, chunk_elems // (batch.num_kv_heads * tile))
            for lo in range(0, batch.num_blocks, step):
                hi = min(lo + step, batch.num_blocks)
                c[lo:hi, :, :ncode] = torch.randint(0, 256, (hi - lo, batch.num_kv_heads, ncode), generator=gen,
                                                    device=device, dtype=torch.int32).to(torch.uint8)
                c[lo:hi, :, ncode:] = torch.randint(0x20, 0x48, (hi - lo, batch.num_kv_heads, tile - ncode),
                                                    generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
            caches.append(c)
        return caches[0], caches[1]
    tdt = torch_dtype(batch.kv_dtype) if batch.kv_dtype != "fp8_e4m3" else torch.uint8
    if batch.kv_dtype == "fp8_e5m2":
        tdt = torch.float8_e5m2
    gen = torch.Generator(device=device)
    gen.manual_seed(batch.cache_seed)
    caches = []
    for sc in (batch.k_scale, batch.v_scale):
        c = torch.empty(shape, dtype=tdt, device=device)
        flat = c.view(-1)
        for lo in range(0, flat.numel(), chunk_elems):
            hi = min(lo + chunk_elems, flat.numel())
            x = torch.randn(hi - lo, generator=gen, device=device, dtype=torch.float32)
            if batch.kv_dtype == "fp8_e4m3":
                flat[lo:hi] = (x / sc).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            elif batch.kv_dtype == "fp8_e5m2":
                flat[lo:hi] = (x / sc).clamp_(-57344.0, 57344.0).to(torch.float8_e5m2)
            else:
                flat[lo:hi] = x.to(tdt)
            del x
        caches.append(c)
    return caches[0], caches[1]
