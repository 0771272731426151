"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each ``check_*`` function measures one pin against an implementation passed in
(the real oracle by default), so ``test_planted_mistakes_are_caught`` can feed
deliberately broken copies and show that some pin fails for each mistake.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- block math

def test_block_count_golden():
    for n, bs, nb in _golden_rows("block_count.txt"):
        assert oracle.blocks_needed(int(n), int(bs)) == int(nb)


def test_internal_waste_below_one_block():
    # [LINEAGE] PagedAttention section: internal waste of a sequence is < P_b slots.
    for bs in (1, 16, 32):
        for n in range(0, 2000):
            waste = oracle.blocks_needed(n, bs) * bs - n
            assert 0 <= waste < bs


@pytest.mark.parametrize("factory", [workloads.tiny,
                                     lambda: workloads.build("x", 5, [40, 3], [1, 1], 8, 8, 128, 16, "bf16"),
                                     lambda: workloads.build("y", 6, [70, 64], [1, 1], 32, 8, 128, 32, "fp8_e4m3")])
def test_bytes_per_block_matches_allocated_tensors(factory):
    b = factory()
    per_block = (b.k_cache.nbytes + b.v_cache.nbytes) // b.num_blocks
    assert per_block == oracle.bytes_per_block(b.block_size, b.num_kv_heads, b.head_size,
                                               oracle.DTYPE_BYTES[b.kv_dtype])


def test_per_block_bytes_of_the_named_configs():
    # tiny fp32, Llama bf16 block 16, FP8 block 32: the allocations the workloads make.
    assert oracle.bytes_per_block(16, 2, 64, 4) == 2 * 16 * 2 * 64 * 4 == 16384
    assert np.zeros((1, 8, 16, 128), np.uint16).nbytes * 2 == oracle.bytes_per_block(16, 8, 128, 2)
    assert np.zeros((1, 8, 32, 128), np.uint8).nbytes * 2 == oracle.bytes_per_block(32, 8, 128, 1)


def test_byte_count_golden():
    rows = _golden_rows("byte_counts.txt")
    for heads, pos, dim, eb, k_only in rows[:2]:
        total = oracle.kv_cache_bytes(1, int(eb), int(heads), int(dim), [int(pos)])
        assert total // 2 == int(k_only)  # M_KV counts K and V; the page counts K only
    L, hkv, d, eb, bs, budget, tokens, ttok, tmb = rows[2]
    per_block_all_layers = int(L) * oracle.bytes_per_block(int(bs), int(hkv), int(d), int(eb))
    assert (int(budget) // per_block_all_layers) * int(bs) == int(tokens)
    transfer = oracle.blocks_needed(int(ttok), int(bs)) * per_block_all_layers
    assert abs(transfer / 2**20 - float(tmb)) < 6e-4


# ---------------------------------------------------------------- FP8 codec

def test_e4m3_decode_exhaustive_vs_torch():
    ours = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def _encode_sweep():
    mags = oracle.e4m3_table()[:127]
    mids = (mags[:-1] + mags[1:]) / 2                       # exact ties
    pts = np.concatenate([mags, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf)])
    rng = np.random.default_rng(7)
    pts = np.concatenate([pts, rng.uniform(0, 463.9, 4000), rng.uniform(0, 2 ** -6, 2000),
                          np.float64(2.0) ** rng.uniform(-12, 8.8, 2000)])
    pts = pts[pts < 464.0].astype(np.float32).astype(np.float64)  # values an fp32 quotient can take
    return np.concatenate([pts, -pts, [0.0, -0.0]])


def check_e4m3_encode(encode):
    x = _encode_sweep()
    ours = encode(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return int(np.count_nonzero(ours != ref))


def test_e4m3_encode_vs_torch_in_range():
    assert check_e4m3_encode(oracle.e4m3_encode) == 0


def test_e4m3_encode_saturates_and_nan():
    codes = oracle.e4m3_encode(np.array([448.0, 463.99, 464.0, 1e6, np.inf, -1e6, -np.inf, np.nan]))
    assert list(codes) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_e5m2_decode_exhaustive_vs_torch():
    ours = oracle.e5m2_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert ours[0x7B] == 57344.0 and ours[0x01] == 2.0 ** -16 and ours[0x7C] == np.inf


def test_e5m2_encode_vs_torch_in_range():
    mags = oracle.e5m2_table()[:124]
    mids = (mags[:-1] + mags[1:]) / 2                       # exact ties
    rng = np.random.default_rng(8)
    pts = np.concatenate([mags, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
                          rng.uniform(0, 57000, 4000), np.float64(2.0) ** rng.uniform(-18, 15.7, 4000)])
    pts = pts[pts < 57344.0].astype(np.float32).astype(np.float64)
    x = np.concatenate([pts, -pts, [0.0, -0.0]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.count_nonzero(oracle.e5m2_encode(x) != ref) == 0


def test_e5m2_encode_saturates_and_nan():
    codes = oracle.e5m2_encode(np.array([57344.0, 61439.0, 61440.0, 1e9, np.inf, -1e9, -np.inf, np.nan]))
    assert list(codes) == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0xFB, 0x7F]


def test_quantize_with_non_power_of_two_scale_vs_torch():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(5000).astype(np.float32)
    scale = np.float32(0.0123)
    ref_q = torch.from_numpy(x) / torch.tensor(scale)          # IEEE fp32 division
    keep = (ref_q.abs() < 464).numpy()
    ref = ref_q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = oracle.quantize_e4m3(x.astype(np.float64), float(scale))
    assert np.array_equal(ours[keep], ref[keep])


@pytest.mark.parametrize("kv", ["fp8_e4m3", "fp8_e5m2"])
def test_per_head_scales(kv):
    """One scale per KV head: equal scales reproduce the per-tensor result, and each
    head of a per-head run equals a one-head run with that head's scale."""
    b = workloads.build("phs", 35, [300, 37, 129], [1, 1, 1], 8, 4, 128, 16, "bf16")
    x64 = oracle.decode_bits(b.k_cache, "bf16")                         # [nb][Hkv][bs][d]
    x64 = x64.transpose(0, 2, 1, 3)                                     # [nb][bs][Hkv][d]
    quant = oracle.quantize_e4m3 if kv == "fp8_e4m3" else oracle.quantize_e5m2
    scales = np.array([2.0 ** -6, 0.011, 2.0 ** -3, 0.37], np.float32)
    kc = quant(x64, scales).transpose(0, 2, 1, 3).copy()
    vc = quant(-x64, scales[::-1].copy()).transpose(0, 2, 1, 3).copy()
    same = quant(x64, np.full(4, scales[0], np.float32)).transpose(0, 2, 1, 3)
    assert np.array_equal(same, quant(x64, scales[0]).transpose(0, 2, 1, 3))
    out = oracle.paged_decode(b.q, "bf16", kc, vc, kv, b.block_tables, b.seq_lens, 16, b.scale,
                              scales, scales[::-1].copy())
    for h in range(4):
        one = oracle.paged_decode(b.q[:, 2 * h: 2 * h + 2], "bf16", kc[:, h: h + 1], vc[:, h: h + 1], kv,
                                  b.block_tables, b.seq_lens, 16, b.scale, float(scales[h]),
                                  float(scales[::-1][h]))
        assert np.array_equal(out[:, 2 * h: 2 * h + 2], one)


def test_decode_bits_vs_torch_casts():
    rng = np.random.default_rng(1)
    x = torch.from_numpy(rng.standard_normal(1000).astype(np.float32) * 100)
    for dt, tdt in (("f32", torch.float32), ("f16", torch.float16), ("bf16", torch.bfloat16)):
        bits = workloads.torch_to_bits(x.to(tdt), dt)
        assert np.array_equal(oracle.decode_bits(bits, dt), x.to(tdt).to(torch.float64).numpy())


# ---------------------------------------------------------------- scatter

def test_scatter_round_trip_and_padding():
    b = workloads.build("s", 11, [5, 33, 16], [5, 2, 1], 4, 2, 64, 16, "bf16")
    k0, v0 = b.k_cache.copy(), b.v_cache.copy()
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    slots = b.slot_mapping.copy()
    slots[3] = -1                                           # a padding token
    oracle.reshape_and_cache(b.key, b.value, kc, vc, slots, 16, "bf16", "bf16")
    touched = np.zeros(kc.shape[0] * 16, bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        touched[s] = True
        assert np.array_equal(kc[s // 16, :, s % 16, :], b.key[t])
        assert np.array_equal(vc[s // 16, :, s % 16, :], b.value[t])
    # every other slot is unchanged
    flat_k = kc.transpose(0, 2, 1, 3).reshape(-1, 2, 64)
    flat_k0 = k0.transpose(0, 2, 1, 3).reshape(-1, 2, 64)
    assert np.array_equal(flat_k[~touched], flat_k0[~touched])
    assert np.array_equal(vc.transpose(0, 2, 1, 3).reshape(-1, 2, 64)[~touched],
                          v0.transpose(0, 2, 1, 3).reshape(-1, 2, 64)[~touched])


def test_scatter_fp8_codes_are_nearest():
    b = workloads.build("s8", 12, [40, 7], [3, 1], 8, 2, 128, 32, "fp8_e4m3")
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    oracle.reshape_and_cache(b.key, b.value, kc, vc, b.slot_mapping, 32, "bf16", "fp8_e4m3",
                             b.k_scale, b.v_scale)
    table = oracle.e4m3_table()
    mags = table[:127]
    for t, s in enumerate(b.slot_mapping):
        x = oracle.decode_bits(b.key[t], "bf16") / b.k_scale
        got = table[kc[s // 32, :, s % 32, :]]
        # nearest representable magnitude (brute force over the table)
        dist = np.abs(np.abs(x)[..., None] - mags)
        best = dist.min(axis=-1)
        assert np.all(np.abs(np.abs(got) - np.abs(x)) <= best + 0.0)
        assert np.all((got == 0) | (np.sign(got) == np.sign(x)))


# ---------------------------------------------------------------- NVFP4

_E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3_torch(codes):
    """E4M3 code -> value through torch's float8_e4m3fn (pinned independently)."""
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e2m1_values_are_the_two_bit_significand_floats():
    """E2M1 magnitudes are 0 and the multiples of 0.5 up to 6 whose significand has
    at most two bits (odd part 1 or 3), found by enumeration; negative codes are the
    sign-flipped magnitudes; every value is exact in E4M3 (torch's cast)."""
    mags = [0.0]
    for k in range(1, 13):
        odd = k
        while odd % 2 == 0:
            odd //= 2
        if odd in (1, 3):
            mags.append(k / 2)
    assert mags == _E2M1_MAGS
    t = oracle.e2m1_table()
    assert list(t[:8]) == mags
    assert np.array_equal(t[8:], -t[:8]) and all(math.copysign(1.0, v) < 0 for v in t[8:])
    tt = torch.tensor(t, dtype=torch.float32)
    assert torch.equal(tt.to(torch.float8_e4m3fn).to(torch.float32), tt)


def check_e2m1_encode(encode):
    """Brute force over y = k/32 in [-8, 8] and -0: the code is a nearest E2M1 value,
    an exact tie goes to the code with mantissa bit 0, |y| >= 6 saturates, the sign
    bit follows y.  Returns the number of violations."""
    ys = np.concatenate([np.arange(-256, 257) / 32.0, [-0.0]])
    codes = np.asarray(encode(ys))
    bad = 0
    for y, c in zip(ys, codes):
        a = abs(float(y))
        dist = [abs(a - m) for m in _E2M1_MAGS]
        near = [i for i, dd in enumerate(dist) if dd == min(dist)]
        want = near[0] if len(near) == 1 else [i for i in near if i % 2 == 0][0]
        if a >= 6.0:
            want = 7
        want |= 0x8 if math.copysign(1.0, float(y)) < 0 else 0
        bad += int(c) != want
    return bad


def test_e2m1_encode_nearest_even_saturating():
    assert check_e2m1_encode(oracle.e2m1_encode) == 0
    assert oracle.e2m1_encode([np.nan])[0] == 0x7


def check_nvfp4_round_trip(quantize):
    """Rows made of E2M1 values x normal E4M3 block scales x a power-of-two tensor
    scale, with one +-6 in every group (so the group maximum fixes its block scale
    exactly), are stored back as exactly those codes and scales.  Returns the
    number of mismatching codes."""
    rng = np.random.default_rng(5)
    bad = 0
    for _ in range(40):
        st = float(2.0 ** int(rng.integers(-8, 3)))
        d = 64
        sb = rng.integers(0x08, 0x77, size=d // 16).astype(np.uint8)       # normal E4M3 codes
        codes = rng.integers(0, 16, size=d).astype(np.uint8)
        for g in range(d // 16):
            codes[g * 16 + int(rng.integers(16))] = int(rng.choice([0x7, 0xF]))
        vals = np.array([(-1.0 if c & 8 else 1.0) * _E2M1_MAGS[c & 7] for c in codes])
        x = vals * np.repeat(_e4m3_torch(sb), 16) * st
        got_c, got_s = quantize(x, st)
        bad += int(np.sum(np.asarray(got_s) != sb)) + int(np.sum(np.asarray(got_c) != codes))
    return bad


def test_nvfp4_exact_rows_round_trip():
    assert check_nvfp4_round_trip(oracle.nvfp4_quantize_row) == 0


def test_nvfp4_quantisation_error_bound():
    """N(0,1) rows, tensor scale 0.0123: each block scale is the E4M3 rounding of
    amax / (6 s) (relative error <= 2^-4 for normal values), and each element's error
    is at most half the E2M1 spacing at its scaled magnitude, saturation included."""
    rng = np.random.default_rng(6)
    st = np.float32(0.0123)
    for _ in range(30):
        x = rng.standard_normal(128).astype(np.float32).astype(np.float64)
        codes, scales = oracle.nvfp4_quantize_row(x, float(st))
        b = _e4m3_torch(scales)
        for g in range(8):
            q = np.max(np.abs(x[g * 16:(g + 1) * 16])) / (6.0 * float(st))
            assert abs(b[g] - q) <= q * 2.0 ** -4 * 1.0001
            unit = float(st) * b[g]
            for i in range(g * 16, (g + 1) * 16):
                c = int(codes[i])
                deq = (-1.0 if c & 8 else 1.0) * _E2M1_MAGS[c & 7] * unit
                y = abs(x[i]) / unit
                half_gap = 0.25 if y < 2 else 0.5 if y < 4 else 1.0
                assert abs(deq - x[i]) <= half_gap * unit * 1.0001


def test_nvfp4_zero_and_vanishing_groups():
    st = 1.0
    x = np.zeros(32)
    x[16:] = 1e-6                     # amax / 6 rounds to E4M3 zero
    codes, scales = oracle.nvfp4_quantize_row(x, st)
    assert np.all(codes == 0) and np.all(scales == 0)
    x[16] = 6.0 * 448.0 * 4           # beyond the largest block scale: saturates
    codes, scales = oracle.nvfp4_quantize_row(x, st)
    assert scales[1] == 0x7E and (codes[16] & 7) == 7
    assert np.all(codes[17:] == 0)


def test_nvfp4_power_of_two_rescaling_keeps_codes():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(128)
    c0, s0 = oracle.nvfp4_quantize_row(x, 0.0123)
    c1, s1 = oracle.nvfp4_quantize_row(x * 8.0, 0.0123 * 8.0)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)


def test_nvfp4_is_about_45_percent_smaller_than_fp8():
    # [DSV41] "三、第二招": the NVFP4 KV format is 45% smaller than the FP8 KV cache.
    fp8_tile = 16 * 128 * oracle.DTYPE_BYTES["fp8_e4m3"]
    saving = 1.0 - oracle.nvfp4_tile_bytes(16, 128) / fp8_tile
    assert saving == 0.4375 and abs(saving - 0.45) < 0.02


def _golden_nvfp4_tile():
    """A tile of block 2, head 32, built byte by byte from the layout: code rows
    (16 bytes each, element 2i in the low nibble of byte i), then scale rows (2
    bytes each).  Expected values with tensor scale 0.5, worked by hand."""
    tile = np.zeros(36, np.uint8)
    tile[0], tile[1] = 0x21, 0xF7          # row 0: 0.5, 1.0, 6, -6, then zeros
    tile[16] = 0x3A                        # row 1: -1.0, 1.5, then 0.5 everywhere
    tile[17:32] = 0x11
    tile[32:36] = [0x38, 0x40, 0x30, 0x3C]  # scales 1.0, 2.0 | 0.5, 1.5
    want = np.zeros((2, 32))
    want[0, :4] = [0.25, 0.5, 3.0, -3.0]
    want[1, 0], want[1, 1] = -0.25, 0.375
    want[1, 2:16] = 0.125
    want[1, 16:] = 0.375
    return tile, want


def check_nvfp4_rows_golden(rows_impl):
    tile, want = _golden_nvfp4_tile()
    cache = np.zeros((3, 1, 36), np.uint8)
    cache[2, 0] = tile
    got = rows_impl(cache, [2, 2], [0, 1], 2, 0.5)[:, 0, :]
    return float(np.abs(got - want).max())


def test_nvfp4_rows_golden_tile():
    assert check_nvfp4_rows_golden(oracle.nvfp4_rows) == 0.0


def test_nvfp4_scatter_writes_the_quantised_row_in_its_tile():
    b = workloads.build("s4", 13, [40, 7], [3, 1], 8, 2, 128, 16, "nvfp4")
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    k0 = kc.copy()
    oracle.reshape_and_cache(b.key, b.value, kc, vc, b.slot_mapping, 16, "bf16", "nvfp4", b.k_scale, b.v_scale)
    for t, s in enumerate(b.slot_mapping):
        got = oracle.nvfp4_rows(kc, [s // 16], [s % 16], 16, b.k_scale)[0]
        for h in range(2):
            codes, scales = oracle.nvfp4_quantize_row(oracle.decode_bits(b.key[t, h], "bf16"), b.k_scale)
            vals = np.array([(-1.0 if c & 8 else 1.0) * _E2M1_MAGS[c & 7] for c in codes])
            assert np.array_equal(got[h], vals * np.repeat(_e4m3_torch(scales), 16) * b.k_scale)
    # bytes of other slots are untouched
    written = set(int(s) for s in b.slot_mapping)
    for blk in range(kc.shape[0]):
        for off in range(16):
            if blk * 16 + off in written:
                continue
            assert np.array_equal(kc[blk, :, off * 64:(off + 1) * 64], k0[blk, :, off * 64:(off + 1) * 64])
            assert np.array_equal(kc[blk, :, 1024 + off * 8:1024 + (off + 1) * 8],
                                  k0[blk, :, 1024 + off * 8:1024 + (off + 1) * 8])


def test_nvfp4_attention_is_placement_invariant_and_matches_sdpa():
    """Decode over an NVFP4 cache: the same logical blocks under a second placement
    give identical outputs, and both equal torch SDPA on the dequantised rows."""
    b = workloads.build("p4", 14, [70, 33, 16], [1, 1, 1], 8, 2, 128, 16, "nvfp4")
    out = oracle.paged_decode(b.q, "bf16", b.k_cache, b.v_cache, "nvfp4", b.block_tables, b.seq_lens, 16,
                              b.scale, b.k_scale, b.v_scale)
    perm = np.random.default_rng(3).permutation(b.num_blocks)
    inv = np.argsort(perm)
    kc2, vc2 = b.k_cache[perm], b.v_cache[perm]               # new block i holds old block perm[i]
    tables2 = np.where(b.block_tables >= 0, inv[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode(b.q, "bf16", kc2, vc2, "nvfp4", tables2, b.seq_lens, 16, b.scale, b.k_scale,
                               b.v_scale)
    assert np.array_equal(out, out2)
    q64 = oracle.decode_bits(b.q, "bf16")
    for r, n in enumerate(b.seq_lens):
        pos = np.arange(n)
        phys = b.block_tables[r][pos // 16]
        K = torch.from_numpy(oracle.nvfp4_rows(b.k_cache, phys, pos % 16, 16, b.k_scale))   # [n][2][d]
        V = torch.from_numpy(oracle.nvfp4_rows(b.v_cache, phys, pos % 16, 16, b.v_scale))
        q = torch.from_numpy(q64[r]).view(2, 4, 1, 128)                                    # [Hkv][G][1][d]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, K.permute(1, 0, 2)[:, None], V.permute(1, 0, 2)[:, None], scale=b.scale)
        assert np.allclose(out[r], ref.reshape(8, 128).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- softmax merge

def check_merge_golden(partial, merge, finalize):
    rows = _golden_rows("online_softmax_merge.txt")
    parts = []
    err = 0.0
    for tag, w, v, ws, wsum in rows[:2]:
        w = [float(a) for a in w.split(",")]
        v = [[float(a)] for a in v.split(",")]
        m, l, acc = partial(np.log(w), v)
        # undo the local max shift to compare with the page's un-shifted sums
        err = max(err, abs(acc[0] * math.exp(m) - float(ws)), abs(l * math.exp(m) - float(wsum)))
        parts.append((m, l, acc))
    _, total_ws, total_w, result = rows[2]
    merged = merge(parts)
    err = max(err, abs(merged[2][0] * math.exp(merged[0]) - float(total_ws)),
              abs(merged[1] * math.exp(merged[0]) - float(total_w)),
              abs(finalize(merged)[0] - float(result)))
    return err


def test_online_softmax_merge_golden():
    assert check_merge_golden(oracle.softmax_partial, oracle.merge_partials,
                              oracle.finalize_partial) < 1e-9


def test_merge_of_any_split_equals_whole():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(300) * 4
    v = rng.standard_normal((300, 7))
    whole = oracle.finalize_partial(oracle.softmax_partial(s, v))
    for cuts in ([150], [1, 2, 299], [10, 20, 30, 200]):
        edges = [0] + cuts + [300]
        parts = [oracle.softmax_partial(s[a:b], v[a:b]) for a, b in zip(edges[:-1], edges[1:])]
        assert np.allclose(oracle.finalize_partial(oracle.merge_partials(parts)), whole,
                           atol=1e-13, rtol=0)
    assert np.allclose(whole, oracle.softmax_weights(s) @ v, atol=1e-13)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(9)
    for n in (1, 2, 17, 1000):
        s = rng.standard_normal(n) * 30
        w = oracle.softmax_weights(s)
        assert abs(w.sum() - 1.0) < 1e-12 and np.all(w >= 0)
        assert np.allclose(oracle.softmax_weights(s + 1234.5), w, atol=1e-15)


# ---------------------------------------------------------------- attention

def _contiguous_case(seed, T, hq, hkv, d, q_len, bs=4):
    """One request whose blocks are stored in order (identity block table), fp32."""
    rng = np.random.default_rng(seed)
    nb = -(-T // bs)
    kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    q = rng.standard_normal((q_len, hq, d)).astype(np.float32)
    table = np.arange(nb, dtype=np.int32)[None, :]
    return q, kc, vc, table


def _run_varlen(attend_impl, gather_impl, q, kc, vc, table, lens, q_lens, bs, scale, causal=True):
    """Oracle's paged_varlen with its inner steps replaceable (for planted mistakes)."""
    qsl = np.concatenate([[0], np.cumsum(q_lens)])
    out = np.zeros(q.shape, np.float64)
    for r in range(len(lens)):
        L = int(lens[r])
        K = gather_impl(kc.view(np.uint32), table[r], L, bs, "f32")
        V = gather_impl(vc.view(np.uint32), table[r], L, bs, "f32")
        pos = oracle.query_positions(L, int(q_lens[r]))
        out[qsl[r]:qsl[r + 1]] = attend_impl(q[qsl[r]:qsl[r + 1]].astype(np.float64), K, V, pos,
                                             scale, causal)
    return out


def check_sdpa(attend_impl=oracle.attend, gather_impl=oracle.gather_kv):
    """Identity placement, one request: equals torch SDPA in fp64 (GQA by repeat_interleave)."""
    err = 0.0
    for seed, T, hq, hkv, d, q_len in ((0, 37, 8, 2, 16, 5), (1, 9, 4, 4, 8, 1), (2, 64, 6, 3, 32, 64)):
        q, kc, vc, table = _contiguous_case(seed, T, hq, hkv, d, q_len)
        scale = 0.3
        ours = _run_varlen(attend_impl, gather_impl, q, kc, vc, table, [T], [q_len], 4, scale)
        K = torch.from_numpy(kc.transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :T].astype(np.float64))
        V = torch.from_numpy(vc.transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :T].astype(np.float64))
        K = K.repeat_interleave(hq // hkv, dim=0)
        V = V.repeat_interleave(hq // hkv, dim=0)
        Q = torch.from_numpy(q.astype(np.float64)).transpose(0, 1)          # [hq][q_len][d]
        pos = torch.arange(T - q_len, T)
        mask = torch.arange(T)[None, :] <= pos[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        err = max(err, float(np.abs(ours - ref.transpose(0, 1).numpy()).max()))
    return err


def test_identity_placement_equals_library_sdpa():
    assert check_sdpa() < 1e-12


def _brute_force(q, kc, vc, table, lens, q_lens, bs, scale, group):
    """Pure-Python loops over lists, math.exp; tiny inputs only."""
    out = []
    start = 0
    for r, (L, ql) in enumerate(zip(lens, q_lens)):
        for j in range(ql):
            p = L - ql + j
            row = []
            for h in range(q.shape[1]):
                g = h // group
                keys, vals = [], []
                for t in range(p + 1):
                    blk = int(table[r][t // bs])
                    keys.append([float(x) for x in kc[blk, g, t % bs]])
                    vals.append([float(x) for x in vc[blk, g, t % bs]])
                qv = [float(x) for x in q[start + j, h]]
                sc = [scale * sum(a * b for a, b in zip(qv, k)) for k in keys]
                mx = max(sc)
                w = [math.exp(s - mx) for s in sc]
                tot = sum(w)
                row.append([sum(w[t] * vals[t][i] for t in range(len(w))) / tot
                            for i in range(len(qv))])
            out.append(row)
        start += ql
    return np.array(out)


def check_brute_force(attend_impl=oracle.attend, gather_impl=oracle.gather_kv):
    rng = np.random.default_rng(21)
    bs, hq, hkv, d = 2, 4, 2, 4
    lens, q_lens = [5, 3, 6], [2, 1, 6]
    nb = 12
    kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((3, 3), -1, np.int32)
    table[0, :3], table[1, :2], table[2, :3] = perm[:3], perm[3:5], perm[5:8]
    q = rng.standard_normal((sum(q_lens), hq, d)).astype(np.float32)
    ours = _run_varlen(attend_impl, gather_impl, q, kc, vc, table, lens, q_lens, bs, 0.7)
    ref = _brute_force(q, kc, vc, table, lens, q_lens, bs, 0.7, hq // hkv)
    return float(np.abs(ours - ref).max())


def test_brute_force_tiny():
    assert check_brute_force() < 1e-12


def test_closed_forms():
    rng = np.random.default_rng(4)
    d, hq, hkv, bs = 8, 4, 2, 4
    # constant V -> output equals that constant row, whatever the scores
    T = 11
    kc = rng.standard_normal((3, hkv, bs, d)).astype(np.float32)
    vc = np.broadcast_to(rng.standard_normal((1, hkv, 1, d)), (3, hkv, bs, d)).astype(np.float32).copy()
    q = rng.standard_normal((1, hq, d)).astype(np.float32)
    out = oracle.paged_decode(q.view(np.uint32), "f32", kc.view(np.uint32), vc.view(np.uint32), "f32",
                              np.array([[2, 0, 1]], np.int32), [T], bs, 1.0)
    for h in range(hq):
        assert np.allclose(out[0, h], vc[0, h // 2, 0], atol=1e-14)
    # q = 0 -> uniform weights -> mean of V over positions 0..p
    q0 = np.zeros((1, hq, d), np.float32)
    vc = rng.standard_normal((3, hkv, bs, d)).astype(np.float32)
    out = oracle.paged_decode(q0.view(np.uint32), "f32", kc.view(np.uint32), vc.view(np.uint32), "f32",
                              np.array([[2, 0, 1]], np.int32), [T], bs, 1.0)
    V = vc[[2, 0, 1]].transpose(1, 0, 2, 3).reshape(hkv, -1, d)[:, :T].astype(np.float64)
    for h in range(hq):
        assert np.allclose(out[0, h], V[h // 2].mean(axis=0), atol=1e-14)
    # seq_len 1 -> output is v_0
    out = oracle.paged_decode(q.view(np.uint32), "f32", kc.view(np.uint32), vc.view(np.uint32), "f32",
                              np.array([[1, -1, -1]], np.int32), [1], bs, 1.0)
    for h in range(hq):
        assert np.array_equal(out[0, h], vc[1, h // 2, 0].astype(np.float64))


def check_permutation_invariance(attend_impl=oracle.attend, gather_impl=oracle.gather_kv):
    """The same logical K/V stored under two placements gives identical outputs."""
    rng = np.random.default_rng(8)
    bs, hq, hkv, d = 4, 8, 2, 16
    lens, q_lens = [13, 29, 4], [1, 3, 4]
    need = [-(-n // bs) for n in lens]
    logical_k = [rng.standard_normal((n, hkv, bs, d)).astype(np.float32) for n in need]
    logical_v = [rng.standard_normal((n, hkv, bs, d)).astype(np.float32) for n in need]
    q = rng.standard_normal((sum(q_lens), hq, d)).astype(np.float32)
    outs = []
    for placement_seed in (0, 1):
        prng = np.random.default_rng(placement_seed)
        nb = 2 * sum(need)
        order = prng.permutation(nb) if placement_seed else np.arange(nb)
        kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)   # garbage elsewhere
        vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float32)
        table = np.full((3, max(need)), -1, np.int32)
        nxt = 0
        for r, n in enumerate(need):
            table[r, :n] = order[nxt:nxt + n]
            kc[order[nxt:nxt + n]] = logical_k[r]
            vc[order[nxt:nxt + n]] = logical_v[r]
            nxt += n
        outs.append(_run_varlen(attend_impl, gather_impl, q, kc, vc, table, lens, q_lens, bs, 0.25))
    return float(np.abs(outs[0] - outs[1]).max())


def test_block_permutation_invariance():
    assert check_permutation_invariance() == 0.0


def test_shared_prefix_blocks_equal_private_copies():
    b = workloads.agentic(seed=5, host_cache=True, scale_lengths=1 / 2000.0)
    fam = b.families[0]
    parent, child = fam[0], fam[1]
    nb = -(-int(b.seq_lens[child]) // b.block_size)
    nshare = int(np.floor(0.96 * nb))
    assert np.array_equal(b.block_tables[parent, :nshare], b.block_tables[child, :nshare])
    assert not set(b.block_tables[child, nshare:nb]) & set(b.block_tables[parent, :nb])
    # an unshared copy of the child: copy its shared blocks into fresh physical blocks
    kc = np.concatenate([b.k_cache, b.k_cache[b.block_tables[child, :nshare]]])
    vc = np.concatenate([b.v_cache, b.v_cache[b.block_tables[child, :nshare]]])
    table = b.block_tables.copy()
    table[child, :nshare] = np.arange(b.num_blocks, b.num_blocks + nshare)
    common = dict(q_bits=b.q, q_dtype="bf16", kv_dtype="bf16", seq_lens=b.seq_lens,
                  block_size=b.block_size, scale=b.scale, seqs=[child])
    shared = oracle.paged_decode(k_cache=b.k_cache, v_cache=b.v_cache, block_tables=b.block_tables, **common)
    private = oracle.paged_decode(k_cache=kc, v_cache=vc, block_tables=table, **common)
    assert np.array_equal(shared[child], private[child])
    # two sequences with identical (q, blocks, len) give identical outputs
    q2 = b.q.copy()
    q2[fam[2]] = q2[parent]
    t2 = b.block_tables.copy()
    t2[fam[2]] = t2[parent]
    both = oracle.paged_decode(q2, "bf16", b.k_cache, b.v_cache, "bf16", t2, b.seq_lens, b.block_size,
                               b.scale, seqs=[parent, fam[2]])
    assert np.array_equal(both[parent], both[fam[2]])


# ---------------------------------------------------------------- copy-on-write

def test_copy_blocks_copies_whole_blocks_and_nothing_else():
    rng = np.random.default_rng(31)
    kc = rng.integers(0, 2 ** 16, size=(12, 2, 16, 64), dtype=np.uint16)
    vc = rng.integers(0, 2 ** 16, size=(12, 2, 16, 64), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[3, 7], [0, 11], [5, 5], [2, 12], [-1, 4]], np.int64)
    assert oracle.copy_blocks(kc, vc, pairs) == [3, 4]      # out-of-range pairs skipped
    for src, dst in ((3, 7), (0, 11), (5, 5)):
        assert np.array_equal(kc[dst], k0[src]) and np.array_equal(vc[dst], v0[src])
    rest = [b for b in range(12) if b not in (7, 11)]
    assert np.array_equal(kc[rest], k0[rest]) and np.array_equal(vc[rest], v0[rest])
    assert oracle.copy_blocks(kc, vc, np.zeros((0, 2), np.int64)) == []


def _fork_appends(cow: bool):
    """A parent of 40 tokens (block 16: the third block holds 8) and a fork sharing all
    three blocks each append a different token at position 40.  Returns the paged
    decode of both and, for each, SDPA on its own dense history (fp64, torch)."""
    rng = np.random.default_rng(32)
    bs, hkv, hq, d, L, nb = 16, 2, 4, 32, 40, 8
    hist_k = rng.standard_normal((L, hkv, d)).astype(np.float32)
    hist_v = rng.standard_normal((L, hkv, d)).astype(np.float32)
    new_k = rng.standard_normal((2, hkv, d)).astype(np.float32)    # parent's, fork's
    new_v = rng.standard_normal((2, hkv, d)).astype(np.float32)
    q = rng.standard_normal((2, hq, d)).astype(np.float32)
    kc = np.zeros((nb, hkv, bs, d), np.uint32)
    vc = np.zeros((nb, hkv, bs, d), np.uint32)
    table = np.array([[4, 1, 6, 0], [4, 1, 6, 0]], np.int32)
    slots = np.array([table[0, t // bs] * bs + t % bs for t in range(L)], np.int64)
    oracle.reshape_and_cache(hist_k.view(np.uint32), hist_v.view(np.uint32), kc, vc, slots, bs, "f32", "f32")
    if cow:   # the fork takes a private copy of the shared, not yet full tail block
        assert oracle.copy_blocks(kc, vc, [[6, 7]]) == []
        table[1, 2] = 7
    for r in (0, 1):
        slot = [table[r, L // bs] * bs + L % bs]
        oracle.reshape_and_cache(new_k[r:r + 1].view(np.uint32), new_v[r:r + 1].view(np.uint32), kc, vc,
                                 slot, bs, "f32", "f32")
    scale = 0.3
    out = oracle.paged_decode(q.view(np.uint32), "f32", kc, vc, "f32", table, [L + 1, L + 1], bs, scale)
    refs = []
    for r in (0, 1):
        K = torch.from_numpy(np.concatenate([hist_k, new_k[r:r + 1]])).double()    # [L+1][hkv][d]
        V = torch.from_numpy(np.concatenate([hist_v, new_v[r:r + 1]])).double()
        K = K.permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)                 # [hq][L+1][d]
        V = V.permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
        qq = torch.from_numpy(q[r]).double()[:, None, :]                           # [hq][1][d]
        refs.append(torch.nn.functional.scaled_dot_product_attention(qq, K, V, scale=scale)[:, 0, :].numpy())
    return out, refs


def test_copy_on_write_keeps_each_branch_history():
    out, (ref_parent, ref_fork) = _fork_appends(cow=True)
    assert np.abs(out[0] - ref_parent).max() < 1e-12
    assert np.abs(out[1] - ref_fork).max() < 1e-12


def test_without_copy_on_write_the_fork_overwrites_the_parent():
    # [LINEAGE] "Prefix reuse": skipping the copy lets the later writer replace the
    # other branch's token in the shared tail block.
    out, (ref_parent, ref_fork) = _fork_appends(cow=False)
    assert np.abs(out[0] - ref_parent).max() > 1e-3
    assert np.abs(out[1] - ref_fork).max() < 1e-12


# ---------------------------------------------------------------- sliding window

def _windowed_batch(seed=33):
    return workloads.build("win", seed, [300, 37, 129, 1000], [40, 1, 129, 7], 8, 2, 64, 16, "f32")


def _varlen(b, window, tables=None):
    return oracle.paged_varlen(b.q, b.q_dtype, b.k_cache, b.v_cache, b.kv_dtype,
                               b.block_tables if tables is None else tables, b.query_start_loc, b.seq_lens,
                               b.block_size, b.scale, True, window=window)


def test_window_covering_the_context_is_full_attention():
    b = _windowed_batch()
    assert np.array_equal(_varlen(b, 0), _varlen(b, 5000))


def test_window_of_one_returns_the_own_value():
    b = _windowed_batch()
    out = _varlen(b, 1)
    group = b.num_q_heads // b.num_kv_heads
    for r in range(b.num_seqs):
        q0, q1, L = int(b.query_start_loc[r]), int(b.query_start_loc[r + 1]), int(b.seq_lens[r])
        for j in range(q0, q1):
            pos = L - (q1 - q0) + (j - q0)
            blk, off = int(b.block_tables[r, pos // 16]), pos % 16
            v = oracle.decode_bits(b.v_cache[blk, :, off, :], "f32")      # [Hkv][d]
            assert np.array_equal(out[j], np.repeat(v, group, axis=0))


def test_window_matches_sdpa_with_a_band_mask():
    # identity placement, one request with a 300-token prefix and 40 new tokens, window 100
    b = workloads.build("winsdpa", 34, [340], [40], 8, 2, 64, 16, "f32")
    W = 100
    out = _varlen(b, W)
    L, n = 340, 40
    K = torch.from_numpy(oracle.gather_kv(b.k_cache, b.block_tables[0], L, 16, "f32"))
    V = torch.from_numpy(oracle.gather_kv(b.v_cache, b.block_tables[0], L, 16, "f32"))
    q = torch.from_numpy(oracle.decode_bits(b.q, "f32"))                    # [n][Hq][d]
    pos = torch.arange(L - n, L)[:, None]
    keys = torch.arange(L)[None, :]
    band = (keys <= pos) & (keys > pos - W)                                  # [n][L]
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2), K.permute(1, 0, 2).repeat_interleave(4, 0), V.permute(1, 0, 2).repeat_interleave(4, 0),
        attn_mask=band, scale=b.scale).permute(1, 0, 2).numpy()
    assert np.abs(out - ref).max() < 1e-12


def test_released_blocks_before_the_window_are_never_read():
    # [AGENTIC] "為什麼需要「分頁」記憶體管理": blocks that leave the window are
    # reclaimed at once; their table entries may then hold anything.
    b = _windowed_batch()
    W = 64
    tables = b.block_tables.copy()
    for r in range(b.num_seqs):
        q_len = int(b.query_start_loc[r + 1] - b.query_start_loc[r])
        first = max(0, int(b.seq_lens[r]) - q_len - W + 1)
        tables[r, : first // 16] = -1
    assert (tables == -1).sum() > 0
    assert np.array_equal(_varlen(b, W), _varlen(b, W, tables))


def test_chunked_prefill_equals_single_chunk():
    """Queries of a prompt give the same output whether processed in one chunk or two."""
    q, kc, vc, table = _contiguous_case(13, 23, 8, 2, 16, 23)
    whole = _run_varlen(oracle.attend, oracle.gather_kv, q, kc, vc, table, [23], [23], 4, 0.2)
    first = _run_varlen(oracle.attend, oracle.gather_kv, q[:9], kc, vc, table, [9], [9], 4, 0.2)
    second = _run_varlen(oracle.attend, oracle.gather_kv, q[9:], kc, vc, table, [23], [14], 4, 0.2)
    assert np.array_equal(np.concatenate([first, second]), whole)


def test_varlen_with_single_tokens_equals_decode():
    b = workloads.build("v", 17, [30, 1, 64], [1, 1, 1], 8, 2, 64, 16, "f16")
    dec = oracle.paged_decode(b.q, "f16", b.k_cache, b.v_cache, "f16", b.block_tables, b.seq_lens, 16, b.scale)
    var = oracle.paged_varlen(b.q, "f16", b.k_cache, b.v_cache, "f16", b.block_tables,
                              b.query_start_loc, b.seq_lens, 16, b.scale)
    assert np.array_equal(dec, var)


def test_non_causal_attends_whole_context():
    q, kc, vc, table = _contiguous_case(14, 12, 4, 4, 8, 3)
    full = _run_varlen(oracle.attend, oracle.gather_kv, q, kc, vc, table, [12], [3], 4, 0.5, causal=False)
    last = _run_varlen(oracle.attend, oracle.gather_kv, q[2:], kc, vc, table, [12], [1], 4, 0.5)
    assert np.array_equal(full[2:], last)                 # the last query sees everything anyway
    first_causal = _run_varlen(oracle.attend, oracle.gather_kv, q, kc, vc, table, [12], [3], 4, 0.5)
    assert not np.allclose(full[0], first_causal[0])


# ---------------------------------------------------------------- workloads

def test_tiny_workload_shape():
    b = workloads.tiny()
    assert list(b.seq_lens) == [17, 64, 129, 200] and b.num_blocks == 64
    used = [int(x) for x in b.block_tables.ravel() if x >= 0]
    assert len(used) == 2 + 4 + 9 + 13 == len(set(used)) and max(used) < 64
    assert b.scale == 1 / 8 and b.kv_dtype == "f32" and b.block_tables.shape[1] == 13


def test_agentic_lengths_and_families():
    lens = workloads.agentic_lengths(2)
    assert np.all((lens >= 32768) & (lens <= 262144))
    b = workloads.agentic(seed=2, host_cache=False)
    assert b.num_seqs == 16 and [len(f) for f in b.families] == [5, 5, 5, 1]
    for fam in b.families[:3]:
        assert len({int(b.seq_lens[i]) for i in fam}) == 1


# ---------------------------------------------------------------- planted mistakes

def _attend_gqa_modulo(q64, K64, V64, positions, scale, causal=True):
    n, hq, d = q64.shape
    hkv = K64.shape[1]
    out = np.empty((n, hq, d))
    for j in range(n):
        last = int(positions[j]) if causal else K64.shape[0] - 1
        for h in range(hq):
            g = h % hkv                                   # wrong head map
            s = scale * (K64[: last + 1, g] @ q64[j, h])
            w = np.exp(s - s.max())
            out[j, h] = w @ V64[: last + 1, g] / w.sum()
    return out


def _attend_off_by_one(q64, K64, V64, positions, scale, causal=True):
    pos = np.maximum(np.asarray(positions) - 1, 0)        # drops the diagonal key
    return oracle.attend(q64, K64, V64, pos, scale, causal)


def _attend_no_scale(q64, K64, V64, positions, scale, causal=True):
    return oracle.attend(q64, K64, V64, positions, 1.0, causal)


def _gather_wrong_offset(cache_bits, row, n, bs, dtype, scale=1.0):
    pos = np.arange(n)
    phys = np.asarray(row, dtype=np.int64)[pos // bs]
    off = (bs - 1) - pos % bs                             # reversed within a block
    return oracle.decode_bits(np.asarray(cache_bits)[phys, :, off, :], dtype, scale)


def _gather_logical_as_physical(cache_bits, row, n, bs, dtype, scale=1.0):
    pos = np.arange(n)
    return oracle.decode_bits(np.asarray(cache_bits)[pos // bs, :, pos % bs, :], dtype, scale)


def _merge_no_rescale(parts):
    return 0.0, sum(p[1] for p in parts), sum(np.asarray(p[2]) for p in parts)


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    mags = oracle.e4m3_table()[:127]
    out = []
    for v in x:
        a = abs(v)
        code = int(np.argmin(np.abs(mags - a) - 1e-30 * mags))  # ties go to the larger
        out.append(code | (0x80 if math.copysign(1, v) < 0 else 0))
    return np.array(out, np.uint8)


def _e2m1_ties_away(x):
    out = []
    for v in np.asarray(x, dtype=np.float64):
        a = min(abs(v), 6.0)
        code = int(np.argmin(np.abs(np.array(_E2M1_MAGS) - a) - 1e-30 * np.array(_E2M1_MAGS)))
        out.append(code | (0x8 if math.copysign(1, v) < 0 else 0))
    return np.array(out, np.uint8)


def _nvfp4_amax_over_four(x64, scale):
    # a plausible slip: block scale from amax / 4 instead of amax / 6
    return oracle.nvfp4_quantize_row(np.asarray(x64) * 1.5, scale)


def _nvfp4_rows_nibbles_swapped(cache, phys, off, bs, scale=1.0):
    c = np.asarray(cache).copy()
    d = c.shape[2] * 16 // (9 * bs)
    codes = c[:, :, :bs * d // 2]
    c[:, :, :bs * d // 2] = (codes >> 4) | ((codes & 0xF) << 4)
    return oracle.nvfp4_rows(c, phys, off, bs, scale)


def test_planted_mistakes_are_caught():
    assert check_e2m1_encode(_e2m1_ties_away) > 0
    assert check_nvfp4_round_trip(_nvfp4_amax_over_four) > 0
    assert check_nvfp4_rows_golden(_nvfp4_rows_nibbles_swapped) > 0
    assert check_sdpa(attend_impl=_attend_gqa_modulo) > 1e-3
    assert check_brute_force(attend_impl=_attend_off_by_one) > 1e-3
    assert check_sdpa(attend_impl=_attend_no_scale) > 1e-3
    assert check_brute_force(gather_impl=_gather_wrong_offset) > 1e-3
    assert check_permutation_invariance(gather_impl=_gather_logical_as_physical) > 1e-3
    assert check_merge_golden(oracle.softmax_partial, _merge_no_rescale, oracle.finalize_partial) > 1e-3
    assert check_e4m3_encode(_encode_ties_away) > 0
