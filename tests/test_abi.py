"""The C-ABI library builds, loads, exports every declared entry point, and
rejects bad arguments on the host before touching a device (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_123_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"^PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    for want in ("pa_compute_slot_mapping", "pa_reshape_and_cache", "pa_decode_attention",
                 "pa_copy_blocks", "pa_decode_workspace_bytes", "pa_get_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_123_gb300 import _lib
    names = declared_symbols()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"


def test_status_strings(lib):
    from paged_kv_cache_123_gb300 import _lib
    for code in _lib.STATUS_NAMES:
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(12345) == b"unknown status"
    assert lib.pa_abi_version() >= 1


def test_host_side_rejections_need_no_device(lib):
    # unsupported head size / group / block size are rejected before any CUDA call
    bad = [
        (64, 32, 32, 96, 16, 100),    # head_size 96
        (64, 32, 3, 128, 16, 100),    # 32 % 3 != 0
        (64, 48, 3, 128, 16, 100),    # group 16
        (64, 32, 32, 128, 12, 100),   # block 12 not a power of two
        (64, 32, 32, 128, 512, 100),  # block 512 too large
    ]
    for args in bad:
        assert lib.pa_decode_workspace_bytes(*args, 0) == -2, args
    p = ctypes.c_void_p(16)
    # decode: max_seq_len beyond the table capacity
    st = lib.pa_decode_attention(p, p, p, p, 4, p, 2, 4, 4, 64, 4, 8, 0, 1.0, 17, 0, p, None, 0, None)
    assert st == -5
    # decode: null q
    st = lib.pa_decode_attention(None, p, p, p, 4, p, 2, 4, 4, 64, 4, 8, 0, 1.0, 16, 0, p, None, 0, None)
    assert st == -1
    # decode: unknown dtype
    st = lib.pa_decode_attention(p, p, p, p, 4, p, 2, 4, 4, 64, 4, 8, 7, 1.0, 16, 0, p, None, 0, None)
    assert st == -3
    # decode: misaligned pointer
    q = ctypes.c_void_p(24)
    st = lib.pa_decode_attention(q, p, p, p, 4, p, 2, 4, 4, 64, 4, 8, 0, 1.0, 16, 0, p, None, 0, None)
    assert st == -8
    # reshape_and_cache: row not a multiple of 16 bytes, null pointers
    assert lib.pa_reshape_and_cache(p, p, 1, 1, 6, 1, p, p, p, 4, 4, None) == -2
    assert lib.pa_reshape_and_cache(None, p, 1, 1, 64, 1, p, p, p, 4, 4, None) == -1
    # slot mapping: bad block size, nothing to do
    assert lib.pa_compute_slot_mapping(p, 1, p, 1, p, 4, 0, p, None) == -2
    assert lib.pa_compute_slot_mapping(None, 0, None, 0, None, 0, 4, None, None) == 0


def test_copy_blocks_host_alias_and_range_checks(lib):
    p = ctypes.c_void_p(16)
    arr = (ctypes.c_void_p * 1)(16)

    def run(pairs, nb=8, block_bytes=256):
        flat = (ctypes.c_int64 * (2 * len(pairs)))(*[x for pr in pairs for x in pr])
        return lib.pa_copy_blocks(arr, arr, 1, p, flat, len(pairs), nb, block_bytes, None)

    assert run([(0, 1), (2, 1)]) == -7          # repeated destination
    assert run([(0, 1), (1, 2)]) == -7          # destination is also a source
    assert run([(0, 9)]) == -5                  # outside the pool
    assert run([(0, 1)], block_bytes=26) == -2  # not a multiple of 4
    assert lib.pa_copy_blocks(arr, arr, 1, p, None, 0, 8, 256, None) == 0  # no pairs


def test_map_to_kernel_blocks_host_checks(lib):
    p = ctypes.c_void_p(16)
    assert lib.pa_map_to_kernel_blocks(p, 2, 3, 3, 0, p, 6, None) == -2     # r < 1
    assert lib.pa_map_to_kernel_blocks(p, 2, 3, 3, 2, p, 5, None) == -2     # stride too small
    assert lib.pa_map_to_kernel_blocks(None, 2, 3, 3, 2, p, 6, None) == -1
    assert lib.pa_map_to_kernel_blocks(p, 0, 3, 3, 2, p, 6, None) == 0      # nothing to do


def test_fp8_and_multi_query_host_checks(lib):
    p = ctypes.c_void_p(16)
    f = ctypes.c_float
    # fp8 write: bad scale, head size not a multiple of 16, unknown dtype
    assert lib.pa_reshape_and_cache_fp8(p, p, 1, 1, 64, 1, p, p, p, 4, 4, f(0.0), f(1.0), None) == -2
    assert lib.pa_reshape_and_cache_fp8(p, p, 1, 1, 72, 1, p, p, p, 4, 4, f(1.0), f(1.0), None) == -2
    assert lib.pa_reshape_and_cache_fp8(p, p, 1, 1, 64, 9, p, p, p, 4, 4, f(1.0), f(1.0), None) == -3
    # fp8 decode: negative scale, table too short
    st = lib.pa_decode_attention_fp8(p, p, p, p, 4, p, 2, 4, 4, 64, 4, 8, 1, f(1.0), f(-1.0),
                                     f(1.0), 16, 0, p, None, 0, None)
    assert st == -2
    st = lib.pa_decode_attention_fp8(p, p, p, p, 4, p, 2, 4, 4, 64, 4, 8, 1, f(1.0), f(1.0),
                                     f(1.0), 17, 0, p, None, 0, None)
    assert st == -5
    # multi-query: fp32 refused, block size below 8 refused, nothing to do
    args = lambda dt, B, mq: (p, p, 2, 4, p, p, p, 4, p, 4, 4, 64, B, 8, dt, f(1.0), mq, 16, 0,
                              p, None, 0, None)
    assert lib.pa_multi_query_attention(*args(0, 16, 2)) == -2
    assert lib.pa_multi_query_attention(*args(1, 4, 2)) == -2
    assert lib.pa_multi_query_attention(*args(1, 16, 0)) == 0
    assert lib.pa_multi_query_workspace_bytes(8, 2, 48, 3, 128, 16, 4, 100, 0) == -2


def test_even_schedule_query_on_the_host(lib):
    # invalid arguments are refused, and calls that cannot take the even
    # schedule answer 0, before any device is touched
    q = lib.pa_decode_even_ctas
    assert q(8, 64, 8, 128, 16, 2, 3, 4000, 1000, 0) == -2       # kv_format 3
    assert q(8, 64, 8, 128, 16, 7, 0, 4000, 1000, 0) == -3       # dtype 7
    assert q(8, 64, 8, 96, 16, 2, 0, 4000, 1000, 0) == -2        # head size 96
    assert q(8, 64, 8, 128, 16, 2, 0, 4000, -1, 0) == -2         # window < 0
    assert q(8, 64, 8, 128, 16, 2, 0, 4000, 0, 0) == 0           # no window
    assert q(8, 64, 8, 128, 16, 2, 0, 4000, 4000, 0) == 0        # window covers all
    assert q(8, 64, 8, 128, 16, 2, 0, 4000, 1000, 256) == 0      # fixed partitions asked
    assert q(8, 64, 8, 64, 16, 2, 0, 4000, 1000, 0) == 0         # head size 64
    assert q(8, 64, 8, 128, 16, 0, 0, 4000, 1000, 0) == 0        # fp32 queries
    assert q(8, 8, 8, 128, 16, 2, 0, 4000, 1000, 0) == 0         # 16-bit pools, group 1
    assert q(8, 64, 8, 128, 4, 2, 1, 4000, 1000, 0) == 0         # blocks of 4 tokens
    assert q(9000, 64, 8, 128, 16, 2, 0, 4000, 1000, 0) == 0     # more than 8192 sequences
