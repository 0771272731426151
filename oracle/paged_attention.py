"""fp64 reference definitions of the paged KV cache hot path (test infrastructure).

Each function restates one step the pages describe, in the plainest form that
reaches the defined result: the block table is resolved into a contiguous K/V,
then textbook softmax attention runs on it.  Source keys ([AGENTIC], [NOTES],
[LINEAGE], [ARCH]) are listed in ``oracle/__init__.py``.

Storage convention (the data the CUDA path reads and writes, restated here
independently):

* a KV cache is two arrays ``k_cache``, ``v_cache`` of raw element bits with
  shape ``[num_blocks][num_kv_heads][block_size][head_size]``;
* a token written to flat slot ``s`` lands in physical block ``s // block_size``
  at offset ``s % block_size``; a negative slot is a padding token;
* query head ``h`` reads KV head ``h // (num_q_heads // num_kv_heads)``;
* the ``q_len`` new tokens of a request are the last ``q_len`` positions of its
  ``seq_len`` tokens; a query at position ``p`` attends keys ``0..p`` when causal.

Element types are named by strings: ``"f32"``, ``"f16"``, ``"bf16"``,
``"fp8_e4m3"``, ``"fp8_e5m2"``, ``"nvfp4"``.  Arrays of bits use uint32 /
uint16 / uint16 / uint8 / uint8.  An ``"nvfp4"`` cache is the exception to the
shape above: ``[num_blocks][num_kv_heads][tile_bytes]`` bytes, each (block, KV
head) tile holding the packed 4-bit codes of its ``block_size`` token rows
followed by their block scales (``nvfp4_tile_bytes``).
"""

from __future__ import annotations

import math

import numpy as np

DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1, "fp8_e5m2": 1}
_BITS = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "fp8_e4m3": np.uint8, "fp8_e5m2": np.uint8}

# Largest finite FP8 e4m3 magnitude: exponent field 15, mantissa 6 -> 1.75 * 2^8.
E4M3_MAX = 448.0
# Largest finite FP8 e5m2 magnitude: exponent field 30, mantissa 3 -> 1.75 * 2^15.
E5M2_MAX = 57344.0


# --------------------------------------------------------------------------
# Block arithmetic and byte counts
# --------------------------------------------------------------------------

def blocks_needed(num_tokens: int, block_size: int) -> int:
    """Number of fixed-size blocks that hold ``num_tokens`` tokens.

    [ARCH] Part 1, allocate_slots: the count of blocks is the token count
    divided by the block size, rounded up (17 new tokens at block size 16 take
    2 blocks).  Written as integer ceiling division.
    """
    if num_tokens < 0 or block_size <= 0:
        raise ValueError("num_tokens must be >= 0 and block_size > 0")
    return (num_tokens + block_size - 1) // block_size


def bytes_per_block(block_size: int, num_kv_heads: int, head_size: int,
                    dtype_bytes: int) -> int:
    """Bytes one physical KV block occupies for one transformer layer.

    [ARCH] Part 1, KV cache manager: 2 x block_size x num_kv_heads x head_size
    x dtype_bytes (the 2 counts K and V).
    """
    return 2 * block_size * num_kv_heads * head_size * dtype_bytes


def kv_cache_bytes(num_layers: int, dtype_bytes: int, num_kv_heads: int,
                   head_dim: int, seq_lens) -> int:
    """Total KV bytes of a set of requests.

    [LINEAGE] "KV Cache：动态批处理把显存变成主资源", the M_KV equation:
    M_KV = 2 * L * b * H_kv * d_h * sum_i T_i, the factor 2 counting K and V.
    """
    return 2 * num_layers * dtype_bytes * num_kv_heads * head_dim * int(sum(int(t) for t in seq_lens))


# --------------------------------------------------------------------------
# Element codecs
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Value of one FP8 e4m3 code, from its bit fields.

    Lower-precision KV is the [NOTES] engine-argument ``--kv-cache-dtype``
    (附录：参数速查).  Format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent field 0 holds subnormals m/8 * 2^-6; S.1111.111 is NaN;
    there is no infinity.
    """
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return math.nan
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** -6
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


def e4m3_table() -> np.ndarray:
    """float64 value of every one of the 256 e4m3 codes."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


_E4M3 = e4m3_table()
# Non-negative finite magnitudes, codes 0..126, strictly increasing.
_E4M3_POS = _E4M3[:127]


def _fp8_encode(x, pos_mags: np.ndarray, vmax: float) -> np.ndarray:
    """Nearest FP8 code, ties to even, saturating at ``vmax``; ``pos_mags`` are the
    non-negative finite magnitudes in code order (strictly increasing)."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    top = len(pos_mags) - 1
    for i, v in enumerate(flat):
        if math.isnan(v):
            out[i] = 0x7F
            continue
        a = abs(v)
        if a >= vmax:
            code = top
        else:
            hi = int(np.searchsorted(pos_mags, a, side="right"))  # first magnitude > a
            lo = hi - 1                                           # magnitude <= a
            d_lo = a - pos_mags[lo]
            d_hi = pos_mags[hi] - a
            if d_lo < d_hi:
                code = lo
            elif d_hi < d_lo:
                code = hi
            else:
                code = lo if lo % 2 == 0 else hi
        out[i] = code | (0x80 if math.copysign(1.0, v) < 0 else 0)
    return out.reshape(x.shape)


def e4m3_encode(x) -> np.ndarray:
    """Round float64 values to FP8 e4m3 codes: nearest, ties to even, saturating.

    For each |x| the two neighbouring representable magnitudes are found and
    the nearer one is taken; on an exact tie the code with an even (zero)
    least-significant mantissa bit wins.  Magnitudes at or above 448 give 448
    (saturation to the largest finite value).  The sign is kept, so small
    negative values give negative zero (0x80).  NaN gives 0x7F.
    """
    return _fp8_encode(x, _E4M3_POS, E4M3_MAX)


def e5m2_value(code: int) -> float:
    """Value of one FP8 e5m2 code, from its bit fields.

    The second FP8 cache format of the [NOTES] ``--kv-cache-dtype`` knob: 1 sign
    bit, 5 exponent bits (bias 15), 2 mantissa bits; exponent field 0 holds
    subnormals m/4 * 2^-14; exponent field 31 is infinity (mantissa 0) or NaN.
    """
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp_field = (code >> 2) & 0x1F
    mant = code & 0x3
    if exp_field == 0x1F:
        return sign * math.inf if mant == 0 else math.nan
    if exp_field == 0:
        return sign * (mant / 4.0) * 2.0 ** -14
    return sign * (1.0 + mant / 4.0) * 2.0 ** (exp_field - 15)


def e5m2_table() -> np.ndarray:
    """float64 value of every one of the 256 e5m2 codes."""
    return np.array([e5m2_value(c) for c in range(256)], dtype=np.float64)


_E5M2 = e5m2_table()
# Non-negative finite magnitudes, codes 0..123 (0x7B = 57344), strictly increasing.
_E5M2_POS = _E5M2[:124]


def e5m2_encode(x) -> np.ndarray:
    """Round float64 values to FP8 e5m2 codes: nearest, ties to even, saturating
    to +-57344 (no infinity is produced); NaN gives 0x7F."""
    return _fp8_encode(x, _E5M2_POS, E5M2_MAX)


def _scale64(scale) -> np.ndarray:
    """An fp32 scale (a scalar, or one per KV head: shape [Hkv] becomes [Hkv][1] so it
    broadcasts over [..][Hkv][d] element arrays) as float64."""
    s = np.asarray(scale, dtype=np.float32).astype(np.float64)
    return s.reshape(-1, 1) if s.ndim == 1 else s


def quantize_e4m3(x64, scale) -> np.ndarray:
    """FP8 code stored for a value ``x`` with an fp32 scale (per tensor, or per KV head).

    The stored code is the e4m3 rounding of the fp32 quotient x / scale.  The
    quotient is formed in float64 and rounded once to float32; since float64
    has more than 2*24+2 significand bits this equals the correctly rounded
    float32 quotient.  The float32 is then rounded to e4m3 (``e4m3_encode``).
    """
    q32 = (np.asarray(x64, dtype=np.float64) / _scale64(scale)).astype(np.float32)
    return e4m3_encode(q32.astype(np.float64))


def quantize_e5m2(x64, scale) -> np.ndarray:
    """As ``quantize_e4m3`` for the e5m2 format: e5m2 rounding of the fp32 quotient."""
    q32 = (np.asarray(x64, dtype=np.float64) / _scale64(scale)).astype(np.float32)
    return e5m2_encode(q32.astype(np.float64))


# --------------------------------------------------------------------------
# NVFP4: 4-bit KV with block scales
# --------------------------------------------------------------------------
#
# [DSV41] "三、第二招：把能合的内核全合成一个" (MegaAttention + NVFP4 compressed
# KV): an NVFP4 KV format 45% smaller than the FP8 KV cache.  The page names the
# format only; it is
# read here as NVIDIA's NVFP4: 4-bit E2M1 elements, one E4M3 scale for every 16
# consecutive elements of a row, and one fp32 scale per tensor (4.5 bits per
# element, 1 - 4.5/8 = 43.75% below FP8).

# Largest E2M1 magnitude: exponent field 3, mantissa 1 -> 1.5 * 2^2.
E2M1_MAX = 6.0
# Elements that share one E4M3 block scale.
NVFP4_GROUP = 16


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code, from its bit fields: 1 sign bit (bit 3),
    2 exponent bits (bias 1), 1 mantissa bit; exponent field 0 holds the
    subnormal m/2 (0 or 0.5).  There is no infinity or NaN."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp_field = (code >> 1) & 0x3
    mant = code & 0x1
    if exp_field == 0:
        return sign * (mant / 2.0)
    return sign * (1.0 + mant / 2.0) * 2.0 ** (exp_field - 1)


def e2m1_table() -> np.ndarray:
    """float64 value of every one of the 16 E2M1 codes."""
    return np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


_E2M1 = e2m1_table()


def e2m1_encode(x) -> np.ndarray:
    """Round values to E2M1 codes: nearest, ties to the even code (mantissa bit
    0), saturating at +-6; the sign is kept (small negatives give 0x8).  NaN gives
    0x7 (the largest positive code)."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    pos = _E2M1[:8]  # 0, 0.5, 1, 1.5, 2, 3, 4, 6
    for i, v in enumerate(flat):
        if math.isnan(v):
            out[i] = 0x7
            continue
        a = abs(v)
        if a >= E2M1_MAX:
            code = 7
        else:
            hi = int(np.searchsorted(pos, a, side="right"))
            lo = hi - 1
            d_lo, d_hi = a - pos[lo], pos[hi] - a
            code = lo if d_lo < d_hi else hi if d_hi < d_lo else (lo if lo % 2 == 0 else hi)
        out[i] = code | (0x8 if math.copysign(1.0, v) < 0 else 0)
    return out.reshape(x.shape)


def nvfp4_tile_bytes(block_size: int, head_size: int) -> int:
    """Bytes of one (block, KV head) tile of an NVFP4 cache: block_size rows of
    head_size/2 code bytes, then block_size rows of head_size/16 scale bytes."""
    return block_size * head_size // 2 + block_size * head_size // NVFP4_GROUP


def nvfp4_quantize_row(x64, scale: float):
    """NVFP4 codes and block scales of one (token, KV head) row.

    For each group of 16 consecutive elements with largest magnitude a, in fp32:
    the block scale is the E4M3 code of a / (6 * scale) (the group's largest
    element maps to the largest E2M1 magnitude), and each element x is stored as
    the E2M1 code of x / (scale * b), b the block scale's value.  A group whose
    block scale is zero stores zero codes.  Every product and quotient is one
    IEEE fp32 operation (numpy float32 arithmetic is correctly rounded).
    Returns (codes: uint8 [d], one code per element; scales: uint8 [d/16]).
    """
    x32 = np.asarray(x64, dtype=np.float64).astype(np.float32)
    s32 = np.float32(scale)
    d = x32.shape[0]
    codes = np.zeros(d, dtype=np.uint8)
    scales = np.zeros(d // NVFP4_GROUP, dtype=np.uint8)
    six_s = np.float32(np.float32(6.0) * s32)
    for g in range(d // NVFP4_GROUP):
        xs = x32[g * NVFP4_GROUP:(g + 1) * NVFP4_GROUP]
        amax = np.float32(np.max(np.abs(xs)))
        sb = e4m3_encode(np.float64(np.float32(amax / six_s)))
        scales[g] = sb
        b = np.float32(_E4M3[int(sb)])
        if b == 0:
            continue
        denom = np.float32(s32 * b)
        codes[g * NVFP4_GROUP:(g + 1) * NVFP4_GROUP] = e2m1_encode((xs / denom).astype(np.float64))
    return codes, scales


def nvfp4_pack(codes) -> np.ndarray:
    """Two E2M1 codes per byte: element 2i in the low nibble of byte i, element
    2i+1 in the high nibble."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, 2)
    return (c[:, 0] | (c[:, 1] << 4)).astype(np.uint8)


def nvfp4_rows(cache, phys, off, block_size: int, scale=1.0) -> np.ndarray:
    """float64 values ``[n][num_kv_heads][head_size]`` of token rows (phys[i], off[i])
    of an NVFP4 cache ``[num_blocks][num_kv_heads][tile_bytes]``: code value x
    block-scale value x the tensor's (or the KV head's) fp32 scale."""
    cache = np.asarray(cache)
    tile = cache.shape[2]
    d = tile * NVFP4_GROUP // (9 * block_size)
    phys = np.asarray(phys, dtype=np.int64)
    off = np.asarray(off, dtype=np.int64)
    tiles = cache[phys]                                               # [n][Hkv][tile]
    code_bytes = tiles[:, :, :block_size * d // 2].reshape(len(phys), -1, block_size, d // 2)
    scale_bytes = tiles[:, :, block_size * d // 2:].reshape(len(phys), -1, block_size, d // NVFP4_GROUP)
    n = np.arange(len(phys))
    cb = code_bytes[n, :, off, :]                                     # [n][Hkv][d/2]
    sb = scale_bytes[n, :, off, :]                                    # [n][Hkv][d/16]
    codes = np.stack([cb & 0xF, cb >> 4], axis=-1).reshape(cb.shape[0], cb.shape[1], d)
    vals = _E2M1[codes] * np.repeat(_E4M3[sb], NVFP4_GROUP, axis=-1)
    return vals * _scale64(scale)


def decode_bits(bits, dtype: str, scale: float = 1.0) -> np.ndarray:
    """Exact float64 value of stored elements given as raw bits.

    fp32 / fp16 widen exactly; bf16 is the upper half of an fp32 and widens
    exactly; FP8 e4m3 / e5m2 is looked up from its bit fields and multiplied by
    the scale in float64 (per tensor, or per KV head for [..][Hkv][d] arrays).
    """
    b = np.asarray(bits)
    if dtype == "f32":
        return b.astype(np.uint32).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return b.astype(np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp8_e4m3":
        return _E4M3[b.astype(np.uint8)] * _scale64(scale)
    if dtype == "fp8_e5m2":
        return _E5M2[b.astype(np.uint8)] * _scale64(scale)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# KV write: reshape_and_cache
# --------------------------------------------------------------------------

def reshape_and_cache(key_bits, value_bits, k_cache, v_cache, slot_mapping,
                      block_size: int, src_dtype: str, cache_dtype: str,
                      k_scale=1.0, v_scale=1.0) -> None:
    """Write each new token's K and V into its slot of the paged cache, in place.

    [NOTES] "Prefill 与 Decode": prefill stores K/V for every prompt token and
    each decode step appends the new token's K/V.  [ARCH] Part 1, forward pass:
    input preparation builds ``slot_mapping``, one flat slot per new token.
    Slot s lands in block s // block_size, offset s % block_size; a negative
    slot is padding and is skipped.  With the same element type the bits are
    copied; with an FP8 cache each value is quantised (``quantize_e4m3`` /
    ``quantize_e5m2``) with the tensor's scale, or its KV head's when the scales
    are given one per head; with an NVFP4 cache each (token, KV head) row is
    quantised by ``nvfp4_quantize_row`` and stored in its tile's code and scale
    rows.
    """
    key_bits = np.asarray(key_bits)
    value_bits = np.asarray(value_bits)
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        if cache_dtype == src_dtype:
            k_cache[blk, :, off, :] = key_bits[t]
            v_cache[blk, :, off, :] = value_bits[t]
        elif cache_dtype in ("fp8_e4m3", "fp8_e5m2"):
            quant = quantize_e4m3 if cache_dtype == "fp8_e4m3" else quantize_e5m2
            k_cache[blk, :, off, :] = quant(decode_bits(key_bits[t], src_dtype), k_scale)
            v_cache[blk, :, off, :] = quant(decode_bits(value_bits[t], src_dtype), v_scale)
        elif cache_dtype == "nvfp4":
            for cache, bits, sc in ((k_cache, key_bits, k_scale), (v_cache, value_bits, v_scale)):
                x = decode_bits(bits[t], src_dtype)                   # [Hkv][d]
                hkv, d = x.shape
                per_head = np.broadcast_to(np.asarray(sc, dtype=np.float32).reshape(-1), (hkv,))
                for h in range(hkv):
                    codes, scales = nvfp4_quantize_row(x[h], per_head[h])
                    cache[blk, h, off * d // 2:(off + 1) * d // 2] = nvfp4_pack(codes)
                    s0 = block_size * d // 2 + off * d // NVFP4_GROUP
                    cache[blk, h, s0:s0 + d // NVFP4_GROUP] = scales
        else:
            raise ValueError(f"unsupported {src_dtype} -> {cache_dtype}")


# --------------------------------------------------------------------------
# Copy-on-write block copy
# --------------------------------------------------------------------------

def copy_blocks(k_cache, v_cache, block_mapping) -> list:
    """Copy whole physical blocks, K and V, in place: ``cache[dst] = cache[src]``.

    [AGENTIC] "統一分頁 + 共用池" (reference counting + copy-on-write): forked
    sequences point their block tables at the same physical blocks and a block
    is duplicated only when shared content must change.  [LINEAGE] "Prefix
    reuse": a shared block that is not yet full must be copied before either
    branch writes its next token into it, or one branch would overwrite the
    other's history.  ``block_mapping`` is ``[num_pairs][2]`` (src, dst); a pair
    with an index outside ``[0, num_blocks)`` is skipped.  The caller keeps every
    dst distinct and never also a src, so the pairs are independent.  Returns the
    indices of the skipped pairs.
    """
    num_blocks = k_cache.shape[0]
    skipped = []
    for i, (src, dst) in enumerate(np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2)):
        src, dst = int(src), int(dst)
        if not (0 <= src < num_blocks and 0 <= dst < num_blocks):
            skipped.append(i)
            continue
        k_cache[dst] = k_cache[src].copy()
        v_cache[dst] = v_cache[src].copy()
    return skipped


# --------------------------------------------------------------------------
# Block-table resolution and attention
# --------------------------------------------------------------------------

def gather_kv(cache_bits, block_table_row, num_tokens: int, block_size: int,
              dtype: str, scale: float = 1.0, first: int = 0) -> np.ndarray:
    """Contiguous float64 K (or V) ``[num_tokens][num_kv_heads][head_size]`` of one request.

    [LINEAGE] "PagedAttention：把逻辑连续与物理连续分开": (sequence, logical
    block) maps to a physical block; the kernel reads K/V through the block
    table.  [AGENTIC] "統一分頁 + 共用池": physical blocks need not be
    contiguous.  Position ``pos`` lives in physical block
    ``block_table_row[pos // block_size]`` at offset ``pos % block_size``.
    Positions ``first .. num_tokens-1`` are gathered (row 0 = position ``first``).
    """
    pos = np.arange(first, num_tokens, dtype=np.int64)
    phys = np.asarray(block_table_row, dtype=np.int64)[pos // block_size]
    off = pos % block_size
    if dtype == "nvfp4":
        return nvfp4_rows(cache_bits, phys, off, block_size, scale)
    return decode_bits(np.asarray(cache_bits)[phys, :, off, :], dtype, scale)


def query_positions(seq_len: int, q_len: int) -> np.ndarray:
    """Positions of a request's new query tokens: the last ``q_len`` of ``seq_len``.

    [ARCH] Part 1, forward pass: all sequences are flattened into one long
    sequence and position indices plus a mask keep each token to its own
    sequence; [LINEAGE] "Chunked prefill": a chunk's tokens follow the already
    cached prefix.  Query j sits at position seq_len - q_len + j.
    """
    if not (1 <= q_len <= seq_len):
        raise ValueError("need 1 <= q_len <= seq_len")
    return np.arange(seq_len - q_len, seq_len, dtype=np.int64)


def softmax_weights(scores) -> np.ndarray:
    """Normalised softmax weights exp(s_i - max s) / sum_j exp(s_j - max s)."""
    s = np.asarray(scores, dtype=np.float64)
    w = np.exp(s - s.max())
    return w / w.sum()


def attend(q64, K64, V64, positions, scale: float, causal: bool = True, window: int = 0,
           key_offset: int = 0) -> np.ndarray:
    """Textbook softmax attention of one request's queries over its contiguous K/V.

    q64 ``[n][Hq][d]``, K64 / V64 ``[T][Hkv][d]`` (float64), ``positions[n]``.
    For query j and head h with KV head g = h // (Hq // Hkv):
    s_t = scale * <q_j,h , k_t,g> for t = 0..p_j (or 0..T-1 when not causal),
    out = sum_t exp(s_t - max s) v_t,g / sum_t exp(s_t - max s).
    [AGENTIC] "Online softmax 到底在幹嘛" gives the weighted average
    sum exp(score) * value / sum exp(score) and the max shift before exp.
    With ``window`` W > 0 (causal only) query j attends t = max(0, p_j - W + 1)
    .. p_j: [AGENTIC] "為什麼需要「分頁」記憶體管理", sliding-window attention
    only looks at the most recent fixed range.  Row 0 of K64 / V64 holds
    position ``key_offset``.
    """
    q64 = np.asarray(q64, dtype=np.float64)
    n, hq, d = q64.shape
    hkv = K64.shape[1]
    if hq % hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = hq // hkv
    out = np.empty((n, hq, d), dtype=np.float64)
    if window and not causal:
        raise ValueError("a sliding window needs causal attention")
    for j in range(n):
        last = int(positions[j]) if causal else key_offset + K64.shape[0] - 1
        first = max(0, last - window + 1) if window else 0
        if first < key_offset:
            raise ValueError("keys before key_offset are needed")
        for g in range(hkv):
            heads = slice(g * group, (g + 1) * group)
            k = K64[first - key_offset: last - key_offset + 1, g, :]     # [L][d]
            v = V64[first - key_offset: last - key_offset + 1, g, :]
            s = scale * (k @ q64[j, heads, :].T)              # [L][group]
            w = np.exp(s - s.max(axis=0, keepdims=True))
            out[j, heads, :] = (w.T @ v) / w.sum(axis=0)[:, None]
    return out


def paged_varlen(q_bits, q_dtype: str, k_cache, v_cache, kv_dtype: str,
                 block_tables, query_start_loc, seq_lens, block_size: int,
                 scale: float, causal: bool = True, k_scale: float = 1.0,
                 v_scale: float = 1.0, rows=None, window: int = 0) -> np.ndarray:
    """Attention of a flattened variable-length batch over a paged KV cache.

    Request r owns query rows query_start_loc[r] .. query_start_loc[r+1]-1 and
    has seq_lens[r] tokens of context including its new tokens.  [ARCH] Part 1
    (flattened super-sequence; V1 mixes prefill chunks and decodes in one
    step); [LINEAGE] "静态 batching" (per-step token budget sum q_i <= K with
    q_i = 1 for a decode).  Returns float64 ``[total_q][Hq][d]``; when ``rows``
    lists flattened query rows only those are computed and the rest are NaN.
    With a sliding ``window`` only positions some query of the request attends
    are read through the block table: entries of blocks that lie wholly before
    the first query's window may be released (any value).
    """
    q64 = decode_bits(q_bits, q_dtype)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    lens = np.asarray(seq_lens, dtype=np.int64)
    out = np.full(q64.shape, np.nan, dtype=np.float64)
    wanted = None if rows is None else set(int(r) for r in rows)
    for r in range(len(lens)):
        lo, hi = int(qsl[r]), int(qsl[r + 1])
        if hi <= lo:
            continue
        sel = [j for j in range(lo, hi) if wanted is None or j in wanted]
        if not sel:
            continue
        L = int(lens[r])
        pos = query_positions(L, hi - lo)
        first = max(0, int(pos[0]) - window + 1) if window else 0
        K = gather_kv(k_cache, block_tables[r], L, block_size, kv_dtype, k_scale, first)
        V = gather_kv(v_cache, block_tables[r], L, block_size, kv_dtype, v_scale, first)
        idx = np.array(sel, dtype=np.int64)
        out[idx] = attend(q64[idx], K, V, pos[idx - lo], scale, causal, window, first)
    return out


def paged_decode(q_bits, q_dtype: str, k_cache, v_cache, kv_dtype: str,
                 block_tables, seq_lens, block_size: int, scale: float,
                 k_scale: float = 1.0, v_scale: float = 1.0, seqs=None, window: int = 0) -> np.ndarray:
    """PagedAttention decode: one new query token per sequence, at its last position.

    [NOTES] "Prefill 与 Decode": the new token's Q attends the K/V of all
    cached tokens.  This is ``paged_varlen`` with q_len = 1 for every request.
    ``seqs`` optionally restricts the computation to some sequences (others NaN).
    """
    b = len(seq_lens)
    qsl = np.arange(b + 1, dtype=np.int64)
    return paged_varlen(q_bits, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                        qsl, seq_lens, block_size, scale, True, k_scale, v_scale,
                        rows=seqs, window=window)


# --------------------------------------------------------------------------
# Partial softmax states and their merge (split-K / context-parallel algebra)
# --------------------------------------------------------------------------

def softmax_partial(scores, values):
    """Partial state (m, l, acc) of one slice of keys.

    m = max score, l = sum exp(s - m), acc = sum exp(s - m) * v.  [AGENTIC]
    "Online softmax 到底在幹嘛": each part hands over a weighted sum and a
    weight sum, after subtracting its own local maximum.
    """
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    m = float(s.max())
    w = np.exp(s - m)
    return m, float(w.sum()), w @ v


def merge_partials(parts):
    """Merge partial states: rescale each by exp(m_j - m) to the global max, then add.

    [AGENTIC] "Online softmax 到底在幹嘛": the parts' weighted sums and weight
    sums are added and divided once; the local maxima are brought to the global
    maximum with a correction factor first.
    """
    m = max(p[0] for p in parts)
    l = sum(p[1] * math.exp(p[0] - m) for p in parts)
    acc = sum(np.asarray(p[2], dtype=np.float64) * math.exp(p[0] - m) for p in parts)
    return m, l, acc


def finalize_partial(part):
    """Output of a (merged) partial state: acc / l."""
    return np.asarray(part[2], dtype=np.float64) / part[1]
