"""CPU-side checks of the C ABI: the library builds, loads, and exports every
symbol include/pa.h declares; host-only entry points behave as documented.
No compute call is made here (there may be no GPU)."""

import ctypes
import importlib.util
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def _lib_path():
    spec = importlib.util.spec_from_file_location(
        "_pa_build", os.path.join(ROOT, "paged_kv_cache_pagedattention_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(scope="module")
def pa():
    _lib_path()
    import paged_kv_cache_pagedattention_gb300 as lib
    return lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_hot_path_calls():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_varlen_attn"):
        assert n in names


def test_library_exports_every_declared_symbol(pa):
    lib = ctypes.CDLL(pa.LIB_PATH)
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(pa.SIGNATURES) == names


def test_status_strings_and_version(pa):
    for s in range(7):
        assert pa.pa_status_string(s).startswith("PA_")
    assert pa.pa_status_string(99) == "unknown pa_status"
    assert pa.pa_version() >= 100


def test_workspace_sizes(pa):
    a = pa.pa_decode_workspace_size(64, 32, 8, 128, 4096, 16)
    assert a >= 256 and a % 256 == 0
    # more context or more sequences never needs less workspace
    assert pa.pa_decode_workspace_size(64, 32, 8, 128, 8192, 16, 512) >= pa.pa_decode_workspace_size(
        64, 32, 8, 128, 4096, 16, 512)
    assert pa.pa_decode_workspace_size(128, 32, 8, 128, 4096, 16, 512) >= pa.pa_decode_workspace_size(
        64, 32, 8, 128, 4096, 16, 512)
    # explicit partition: partial rows = B * ceil(max_len / part); each row Hq*(8 + 4d) bytes
    exp = 256 + (64 * 8 * 32 * 8 + 255) // 256 * 256 + (64 * 8 * 32 * 128 * 4 + 255) // 256 * 256
    assert pa.pa_decode_workspace_size(64, 32, 8, 128, 4096, 16, 512) == exp
    assert pa.pa_varlen_workspace_size(132, 2176, 512, 32, 8, 128, 66048, 16) >= 256
    assert pa.pa_decode_workspace_size(0, 32, 8, 128, 4096, 16) == 256


def test_default_partition_is_a_block_multiple(pa):
    for bs in (16, 32, 48):
        for b, hkv, L in ((4, 2, 200), (64, 8, 4096), (16, 8, 262144), (256, 8, 32768), (1, 1, 10 ** 7)):
            part = pa.pa_default_partition_size(b, hkv, L, bs)
            assert part % bs == 0 and part >= bs
            assert -(-L // part) <= 65535


def test_host_validation_rejects_null_pointers_without_a_gpu(pa):
    lib = ctypes.CDLL(pa.LIB_PATH)
    for name, (res, args) in pa.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    st = lib.pa_decode(None, None, None, None, 10, None, 4, None, 2, 64, 8, 2, 128, 16, 1.0, 2, 2, None, None,
                       0, None, 0, None)
    assert st == pa.PA_ERR_INVALID_ARG
    st = lib.pa_varlen_attn(None, None, None, None, 10, None, 4, None, None, 2, 5, 4, 64, 8, 2, 128, 16, 1.0, 1,
                            2, 2, None, None, 0, None, 0, None)
    assert st == pa.PA_ERR_INVALID_ARG
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 10, 2, 128, 16, 2, 2, None, None,
                                    None) == pa.PA_OK  # nothing to write
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 3, 10, 2, 128, 16, 2, 2, None, None,
                                    None) == pa.PA_ERR_INVALID_ARG
    # zero sequences: a no-op that succeeds before touching any pointer
    assert lib.pa_decode(None, None, None, None, 10, None, 4, None, 0, 64, 8, 2, 128, 16, 1.0, 2, 2, None, None,
                         0, None, 0, None) == pa.PA_OK


def test_non_positive_scale_rejected_without_a_gpu(pa):
    lib = ctypes.CDLL(pa.LIB_PATH)
    fn = lib.pa_decode
    fn.restype, fn.argtypes = pa.SIGNATURES["pa_decode"]
    fake = 1 << 20  # aligned, never dereferenced: the checks return first
    for scale in (0.0, -0.125, float("inf"), float("nan")):
        st = fn(fake, fake, fake, fake, 10, fake, 4, fake, 2, 64, 8, 2, 128, 16, scale, 2, 2, None, None, 0,
                fake, 1 << 30, None)
        assert st == pa.PA_ERR_INVALID_ARG, scale


def test_copy_blocks_host_validation_without_a_gpu(pa):
    lib = ctypes.CDLL(pa.LIB_PATH)
    fn = lib.pa_copy_blocks
    fn.restype, fn.argtypes = pa.SIGNATURES["pa_copy_blocks"]
    assert fn(None, None, None, 0, 10, 2, 128, 16, pa.PA_BF16, None) == pa.PA_OK      # nothing to copy
    assert fn(None, None, None, 3, 10, 2, 128, 16, pa.PA_BF16, None) == pa.PA_ERR_INVALID_ARG
    assert fn(None, None, None, -1, 10, 2, 128, 16, pa.PA_BF16, None) == pa.PA_ERR_INVALID_ARG
    fake = 1 << 20  # aligned, never dereferenced: the checks return first
    assert fn(fake, fake, fake, 3, 10, 2, 128, 16, 99, None) == pa.PA_ERR_UNSUPPORTED  # unknown dtype
    # NVFP4 tiles must be whole 16-byte pieces: block 8 x head 16 is 72 bytes
    assert fn(fake, fake, fake, 3, 10, 2, 16, 8, pa.PA_NVFP4, None) == pa.PA_ERR_UNSUPPORTED
    assert fn(fake, fake, fake, 3, 10, 2, 4, 16, pa.PA_F16, None) == pa.PA_ERR_UNSUPPORTED  # 8-byte rows
    assert fn(fake + 8, fake, fake, 3, 10, 2, 128, 16, pa.PA_BF16, None) == pa.PA_ERR_INVALID_ARG


def test_nvfp4_host_validation_without_a_gpu(pa):
    """NVFP4 caches need their fp32 scales and whole tiles (head a multiple of 16,
    block x head a multiple of 256): checked before anything is launched."""
    lib = ctypes.CDLL(pa.LIB_PATH)
    fn = lib.pa_decode
    fn.restype, fn.argtypes = pa.SIGNATURES["pa_decode"]
    fake = 1 << 20
    st = fn(fake, fake, fake, fake, 10, fake, 4, fake, 2, 64, 8, 2, 128, 16, 0.1, pa.PA_BF16, pa.PA_NVFP4,
            None, None, 0, fake, 1 << 30, None)
    assert st == pa.PA_ERR_INVALID_ARG                                   # scales missing
    st = fn(fake, fake, fake, fake, 10, fake, 4, fake, 2, 64, 8, 2, 24, 16, 0.1, pa.PA_BF16, pa.PA_NVFP4,
            fake, fake, 0, fake, 1 << 30, None)
    assert st == pa.PA_ERR_UNSUPPORTED                                   # head 24: partial groups
    rc = lib.pa_reshape_and_cache
    rc.restype, rc.argtypes = pa.SIGNATURES["pa_reshape_and_cache"]
    assert rc(fake, fake, fake, fake, fake, 3, 10, 2, 16, 8, pa.PA_BF16, pa.PA_NVFP4, fake, fake,
              None) == pa.PA_ERR_UNSUPPORTED                             # 72-byte tiles
    assert rc(fake, fake, fake, fake, fake, 3, 10, 2, 128, 16, pa.PA_BF16, pa.PA_NVFP4_PER_HEAD, None, None,
              None) == pa.PA_ERR_INVALID_ARG                             # scales missing


def test_static_workspace_host_validation_without_a_gpu(pa):
    """The no-workspace decode rejects bad sizes, and does nothing for an empty batch,
    before it looks up its device array."""
    lib = ctypes.CDLL(pa.LIB_PATH)
    fn = lib.pa_decode_static_workspace
    fn.restype, fn.argtypes = pa.SIGNATURES["pa_decode_static_workspace"]
    fake = 1 << 20  # never dereferenced: the checks return first
    args = [fake, fake, fake, fake, 10, fake, 4, fake, 2, 64, 8, 2, 128, 16, 0.1, pa.PA_BF16, pa.PA_BF16, None, None,
            0, None]
    assert fn(*args[:8], 0, *args[9:]) == pa.PA_OK                      # no sequences: nothing to do
    assert fn(*args[:8], -1, *args[9:]) == pa.PA_ERR_INVALID_ARG         # negative batch
    assert fn(*args[:13], 0, *args[14:]) == pa.PA_ERR_INVALID_ARG        # block size 0
    assert fn(*args[:9], 0, *args[10:]) == pa.PA_ERR_INVALID_ARG         # max_seq_len 0
    assert fn(*args[:19], -16, None) == pa.PA_ERR_INVALID_ARG            # negative partition size
