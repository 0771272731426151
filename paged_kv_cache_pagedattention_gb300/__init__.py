"""Python binding of libpa.so, the paged KV cache attention library for GB300.

Argument marshalling only: every function takes torch tensors, checks that they
are contiguous CUDA tensors of the expected shapes, and passes raw device
pointers, sizes and the current CUDA stream to the C ABI declared in
``include/pa.h``.  All computation happens in the library's CUDA kernels; there
is no fallback.  Importing this package raises ImportError when libpa.so has
not been built (``python paged_kv_cache_pagedattention_gb300/build.py``).

Cache tensors have shape ``[num_blocks][num_kv_heads][block_size][head_size]``;
FP8 e4m3 caches are uint8 tensors of codes with per-tensor fp32 scales passed as
one-element float32 CUDA tensors (one value per KV head selects per-head scales).
NVFP4 caches are 3-D uint8 tensors ``[num_blocks][num_kv_heads][tile_bytes]``,
``tile_bytes = 9 * block_size * head_size / 16`` (codes, then block scales; see
``include/pa.h``); their head size is taken from the query or key tensor.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libpa.so not found at {LIB_PATH}; build it with "
                      "`python paged_kv_cache_pagedattention_gb300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_BOUNDS, \
    PA_ERR_TIMEOUT, PA_ERR_CUDA = range(7)
PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3, PA_FP8_E5M2, PA_FP8_E4M3_PER_HEAD, PA_FP8_E5M2_PER_HEAD, PA_NVFP4, \
    PA_NVFP4_PER_HEAD = range(9)
PA_ERRFLAG_BLOCK_TABLE, PA_ERRFLAG_SLOT, PA_ERRFLAG_SEQ_LEN, PA_ERRFLAG_QUERY, PA_ERRFLAG_TIMEOUT = \
    0x1, 0x2, 0x4, 0x8, 0x10
# diagnostic only: a declared shared block differed for some member (the output is unaffected)
PA_ERRFLAG_SHARED_MISMATCH = 0x20

# Names of the kernel kinds reported by pa_trace_read.
TRACE_KINDS = ("reshape_and_cache", "attention", "merge", "varlen_plan", "prefill_tiles", "shared_prefix",
               "shared_span", "copy_blocks", "varlen_span")

# Every symbol include/pa.h declares, with its ctypes signature.
_P, _I32, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pa_version": (_I32, []),
    "pa_reshape_and_cache": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32,
                                            ctypes.c_int, ctypes.c_int, _P, _P, _P]),
    "pa_copy_blocks": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, ctypes.c_int, _P]),
    "pa_default_partition_size": (_I32, [_I32, _I32, _I32, _I32]),
    "pa_decode_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "pa_decode": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                 _I32, _F, ctypes.c_int, ctypes.c_int, _P, _P, _I32, _P, _SZ, _P]),
    "pa_decode_windowed": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                          _I32, _F, _I32, ctypes.c_int, ctypes.c_int, _P, _P, _I32, _P, _SZ, _P]),
    "pa_decode_shared_prefix_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "pa_decode_shared_prefix": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                               _I32, _F, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _I32,
                                               _I32, _I32, _P, _SZ, _P]),
    "pa_decode_static_workspace": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                                  _I32, _I32, _F, ctypes.c_int, ctypes.c_int, _P, _P, _I32, _P]),
    "pa_varlen_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "pa_varlen_attn": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                      _I32, _I32, _I32, _I32, _F, _I32, ctypes.c_int, ctypes.c_int,
                                      _P, _P, _I32, _P, _SZ, _P]),
    "pa_varlen_attn_windowed": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                               _I32, _I32, _I32, _I32, _F, _I32, _I32, ctypes.c_int, ctypes.c_int,
                                               _P, _P, _I32, _P, _SZ, _P]),
    "pa_get_error_flags": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _I32, _P]),
    "pa_trace_enable": (ctypes.c_int, [_I32]),
    "pa_trace_read": (ctypes.c_int, [_I32, ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_double), _I32]),
}
for _name, (_res, _args) in SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.pa_status_string(status).decode()}")


def _check(status: int, where: str) -> None:
    if status != PA_OK:
        raise PAError(status, where)


# FP8 caches: uint8 codes are e4m3; torch's float8 dtypes name their format
_DT = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.uint8: PA_FP8_E4M3,
       torch.float8_e4m3fn: PA_FP8_E4M3, torch.float8_e5m2: PA_FP8_E5M2}


def dtype_code(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported tensor dtype {t.dtype}") from None


def is_nvfp4(cache: torch.Tensor) -> bool:
    """NVFP4 caches are the 3-D uint8 tensors [num_blocks][num_kv_heads][tile_bytes]."""
    return cache.dim() == 3 and cache.dtype == torch.uint8


def kv_code(cache: torch.Tensor, k_scale=None) -> int:
    """Cache dtype code; scales holding more than one value (one per KV head, the
    cache's dimension 1) select the per-head format."""
    code = PA_NVFP4 if is_nvfp4(cache) else dtype_code(cache)
    if code in (PA_FP8_E4M3, PA_FP8_E5M2, PA_NVFP4) and k_scale is not None and k_scale.numel() > 1:
        if k_scale.numel() != cache.shape[1]:
            raise ValueError("scales: one per tensor or one per KV head")
        return {PA_FP8_E4M3: PA_FP8_E4M3_PER_HEAD, PA_FP8_E5M2: PA_FP8_E5M2_PER_HEAD,
                PA_NVFP4: PA_NVFP4_PER_HEAD}[code]
    return code


def cache_geometry(k_cache: torch.Tensor, v_cache: torch.Tensor, head_size: int):
    """(num_blocks, num_kv_heads, block_size, head_size) of a K/V cache pair; the
    head size of an NVFP4 cache comes from the caller's query or key tensor."""
    if tuple(v_cache.shape) != tuple(k_cache.shape) or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must match")
    if is_nvfp4(k_cache):
        nb, hkv, tile = k_cache.shape
        if head_size < 1 or (16 * tile) % (9 * head_size):
            raise ValueError("NVFP4 cache: tile_bytes must be 9 * block_size * head_size / 16")
        return nb, hkv, 16 * tile // (9 * head_size), head_size
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks][num_kv_heads][block_size][head_size]")
    return tuple(k_cache.shape)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def pa_status_string(status: int) -> str:
    return _lib.pa_status_string(status).decode()


def pa_version() -> int:
    return _lib.pa_version()


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None,
                         stream=None) -> None:
    """Write key/value [T][Hkv][d] into the paged caches at slot_mapping (int64 [T])."""
    nb, hkv, bs, d = cache_geometry(k_cache, v_cache, key.shape[-1])
    if key.dim() != 3 or tuple(key.shape[1:]) != (hkv, d) or key.shape != value.shape:
        raise ValueError("key/value must be [num_tokens][num_kv_heads][head_size]")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != key.shape[0]:
        raise ValueError("slot_mapping must be int64 [num_tokens]")
    _check(_lib.pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(slot_mapping), key.shape[0], nb, hkv, d, bs,
                                     dtype_code(key), kv_code(k_cache, k_scale), _ptr(k_scale), _ptr(v_scale),
                                     _stream(stream)), "pa_reshape_and_cache")


def pa_copy_blocks(k_cache, v_cache, block_mapping, stream=None) -> None:
    """Copy whole physical blocks: block_mapping is int64 [num_pairs][2] of (src, dst)."""
    if is_nvfp4(k_cache):
        # only the tile size matters for a copy: any (block_size, head_size) with
        # 9 * block_size * head_size / 16 == tile_bytes names it
        nb, hkv, bs, d = cache_geometry(k_cache, v_cache, k_cache.shape[2] // 9)
    else:
        nb, hkv, bs, d = cache_geometry(k_cache, v_cache, 0)
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be int64 [num_pairs][2]")
    if not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be contiguous")
    n = block_mapping.shape[0]
    _check(_lib.pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_mapping) if n else None, n, nb, hkv, d,
                               bs, kv_code(k_cache), _stream(stream)), "pa_copy_blocks")


def pa_default_partition_size(num_seqs, num_kv_heads, max_seq_len, block_size) -> int:
    return _lib.pa_default_partition_size(num_seqs, num_kv_heads, max_seq_len, block_size)


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, max_seq_len, block_size,
                             partition_size=0) -> int:
    return _lib.pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, max_seq_len,
                                         block_size, partition_size)


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale, workspace,
              k_scale=None, v_scale=None, partition_size=0, stream=None, window=0) -> None:
    """PagedAttention decode; out/q [B][Hq][d], block_tables int32 [B][max_blocks], seq_lens int32 [B].
    window > 0: sliding-window attention (pa_decode_windowed)."""
    nb, hkv, bs, d = cache_geometry(k_cache, v_cache, q.shape[-1])
    b, hq = q.shape[0], q.shape[1]
    if q.dim() != 3 or q.shape[2] != d or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q/out must be [num_seqs][num_q_heads][head_size] of one dtype")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be int32 [num_seqs][max_blocks_per_seq]")
    if seq_lens.dtype != torch.int32 or seq_lens.numel() != b:
        raise ValueError("seq_lens must be int32 [num_seqs]")
    _check(_lib.pa_decode_windowed(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                   block_tables.shape[1], _ptr(seq_lens), b, int(max_seq_len), hq, hkv, d, bs,
                                   float(scale), int(window), dtype_code(q), kv_code(k_cache, k_scale), _ptr(k_scale),
                                   _ptr(v_scale), int(partition_size), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)), "pa_decode")


def pa_decode_shared_prefix_workspace_size(num_seqs, num_groups, num_q_heads, num_kv_heads, head_size,
                                           max_seq_len, block_size, partition_size=0) -> int:
    return _lib.pa_decode_shared_prefix_workspace_size(num_seqs, num_groups, num_q_heads, num_kv_heads,
                                                       head_size, max_seq_len, block_size, partition_size)


def pa_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale, workspace,
                            group_start, group_shared_blocks, max_group_size, k_scale=None, v_scale=None,
                            partition_size=0, stream=None) -> None:
    """pa_decode where groups of consecutive sequences share leading blocks.

    group_start int32 [G+1] (device), group_shared_blocks int32 [G] (device)."""
    nb, hkv, bs, d = cache_geometry(k_cache, v_cache, q.shape[-1])
    b, hq = q.shape[0], q.shape[1]
    if q.dim() != 3 or q.shape[2] != d or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q/out must be [num_seqs][num_q_heads][head_size] of one dtype")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be int32 [num_seqs][max_blocks_per_seq]")
    if group_start.dtype != torch.int32 or group_shared_blocks.dtype != torch.int32 or \
            group_start.numel() != group_shared_blocks.numel() + 1:
        raise ValueError("group_start int32 [G+1], group_shared_blocks int32 [G]")
    _check(_lib.pa_decode_shared_prefix(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                        block_tables.shape[1], _ptr(seq_lens), b, int(max_seq_len), hq, hkv, d,
                                        bs, float(scale), dtype_code(q), kv_code(k_cache, k_scale), _ptr(k_scale),
                                        _ptr(v_scale), _ptr(group_start), _ptr(group_shared_blocks),
                                        group_shared_blocks.numel(), int(max_group_size), int(partition_size),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "pa_decode_shared_prefix")


def pa_decode_static_workspace(out, q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale,
                               k_scale=None, v_scale=None, partition_size=0, stream=None) -> None:
    """pa_decode with the library's fixed scratch array instead of a workspace: for
    callers that cannot allocate device memory where attention runs.  See pa.h."""
    nb, hkv, bs, d = cache_geometry(k_cache, v_cache, q.shape[-1])
    b, hq = q.shape[0], q.shape[1]
    if q.dim() != 3 or q.shape[2] != d or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q/out must be [num_seqs][num_q_heads][head_size] of one dtype")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be int32 [num_seqs][max_blocks_per_seq]")
    if seq_lens.dtype != torch.int32 or seq_lens.numel() != b:
        raise ValueError("seq_lens must be int32 [num_seqs]")
    _check(_lib.pa_decode_static_workspace(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), nb,
                                           _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), b,
                                           int(max_seq_len), hq, hkv, d, bs, float(scale), dtype_code(q),
                                           kv_code(k_cache, k_scale), _ptr(k_scale), _ptr(v_scale),
                                           int(partition_size), _stream(stream)),
           "pa_decode_static_workspace")


def pa_varlen_workspace_size(num_seqs, total_q_tokens, max_query_len, num_q_heads, num_kv_heads,
                             head_size, max_seq_len, block_size, partition_size=0) -> int:
    return _lib.pa_varlen_workspace_size(num_seqs, total_q_tokens, max_query_len, num_q_heads,
                                         num_kv_heads, head_size, max_seq_len, block_size, partition_size)


def pa_varlen_attn(out, q, k_cache, v_cache, block_tables, query_start_loc, seq_lens, max_query_len,
                   max_seq_len, scale, workspace, causal=True, k_scale=None, v_scale=None,
                   partition_size=0, stream=None, window=0) -> None:
    """Attention of a flattened varlen batch; out/q [T][Hq][d], query_start_loc int32 [B+1].
    window > 0: sliding-window attention (pa_varlen_attn_windowed)."""
    nb, hkv, bs, d = cache_geometry(k_cache, v_cache, q.shape[-1])
    t, hq = q.shape[0], q.shape[1]
    b = seq_lens.numel()
    if q.dim() != 3 or q.shape[2] != d or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q/out must be [total_q_tokens][num_q_heads][head_size] of one dtype")
    if query_start_loc.dtype != torch.int32 or query_start_loc.numel() != b + 1:
        raise ValueError("query_start_loc must be int32 [num_seqs+1]")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be int32 [num_seqs][max_blocks_per_seq]")
    _check(_lib.pa_varlen_attn_windowed(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                               block_tables.shape[1], _ptr(query_start_loc), _ptr(seq_lens), b, t,
                               int(max_query_len), int(max_seq_len), hq, hkv, d, bs, float(scale), int(window),
                               1 if causal else 0, dtype_code(q), kv_code(k_cache, k_scale), _ptr(k_scale),
                               _ptr(v_scale), int(partition_size), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)),
           "pa_varlen_attn")


def pa_get_error_flags(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return the device error word (PA_ERRFLAG_* bits)."""
    flags = ctypes.c_uint32(0)
    st = _lib.pa_get_error_flags(ctypes.byref(flags), 1 if clear else 0, _stream(stream))
    if st not in (PA_OK, PA_ERR_BOUNDS, PA_ERR_TIMEOUT):
        _check(st, "pa_get_error_flags")
    return int(flags.value)


def pa_trace_enable(on: bool) -> None:
    _check(_lib.pa_trace_enable(1 if on else 0), "pa_trace_enable")


def pa_trace_read(kind: int, reset: bool = False):
    """(launches, total device ms) of one kernel kind since the last reset."""
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(_lib.pa_trace_read(kind, ctypes.byref(n), ctypes.byref(ms), 1 if reset else 0), "pa_trace_read")
    return int(n.value), float(ms.value)


def workspace_tensor(nbytes: int, device=None) -> torch.Tensor:
    """A device byte buffer suitable as `workspace` (torch allocations are 256-byte aligned)."""
    return torch.empty(int(nbytes), dtype=torch.uint8, device=device or "cuda")
