"""ctypes binding to libpagedattn.so (include/pagedattn.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the C ABI. Torch supplies device memory and the current
stream. There is no fallback: if the library is missing or a call fails, an
exception says so.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedattn.so")

PA_OK = 0
STATUS_NAMES = {
    0: "PA_OK", -1: "PA_ERR_NULL", -2: "PA_ERR_SHAPE", -3: "PA_ERR_DTYPE",
    -4: "PA_ERR_WORKSPACE", -5: "PA_ERR_OUT_OF_RANGE", -6: "PA_ERR_CUDA",
    -7: "PA_ERR_ALIAS", -8: "PA_ERR_ALIGN", -9: "PA_ERR_DEVICE", -10: "PA_ERR_TIMEOUT",
}
DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

_c_i32, _c_i64, _c_p, _c_f = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
SIGNATURES = {
    "pa_status_string": ([_c_i32], ctypes.c_char_p),
    "pa_abi_version": ([], _c_i32),
    "pa_compute_slot_mapping": ([_c_p, _c_i32, _c_p, _c_i64, _c_p, _c_i64, _c_i32, _c_p, _c_p], _c_i32),
    "pa_reshape_and_cache": ([_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_p,
                              _c_i64, _c_i32, _c_p], _c_i32),
    "pa_decode_workspace_bytes": ([_c_i32] * 7, _c_i64),
    "pa_decode_partitioning": ([_c_i32] * 6 + [_c_p, _c_p], _c_i32),
    "pa_decode_window_partitioning": ([_c_i32] * 7 + [_c_p, _c_p], _c_i32),
    "pa_decode_fp8_partitioning": ([_c_i32] * 9 + [_c_p, _c_p], _c_i32),
    "pa_decode_even_ctas": ([_c_i32] * 10, _c_i32),
    "pa_decode_attention": ([_c_p, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32, _c_i32,
                             _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_i32, _c_i32, _c_p,
                             _c_p, _c_i64, _c_p], _c_i32),
    "pa_decode_attention_static": ([_c_p, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32,
                                    _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_i32,
                                    _c_i32, _c_p, _c_p], _c_i32),
    "pa_multi_query_attention": ([_c_p, _c_p, _c_i32, _c_i64, _c_p, _c_p, _c_p, _c_i64, _c_p,
                                  _c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_f,
                                  _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_i64, _c_p], _c_i32),
    "pa_multi_query_workspace_bytes": ([_c_i64] + [_c_i32] * 8, _c_i64),
    "pa_reshape_and_cache_fp8": ([_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_p,
                                  _c_i64, _c_i32, _c_f, _c_f, _c_p], _c_i32),
    "pa_decode_attention_fp8": ([_c_p, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32, _c_i32,
                                 _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_f, _c_f, _c_i32,
                                 _c_i32, _c_p, _c_p, _c_i64, _c_p], _c_i32),
    "pa_decode_window_workspace_bytes": ([_c_i32] * 8, _c_i64),
    "pa_decode_fp8_workspace_bytes": ([_c_i32] * 9, _c_i64),
    "pa_decode_attention_window": ([_c_p, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32,
                                    _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_i32,
                                    _c_i32, _c_i32, _c_p, _c_p, _c_i64, _c_p], _c_i32),
    "pa_decode_attention_fp8_window": ([_c_p, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32,
                                        _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_f,
                                        _c_f, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_i64,
                                        _c_p], _c_i32),
    "pa_reshape_and_cache_fp8_scaled": ([_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_p, _c_p,
                                         _c_p, _c_p, _c_p, _c_i64, _c_i32, _c_p], _c_i32),
    "pa_decode_attention_fp8_scaled": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_p,
                                        _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_i32,
                                        _c_f, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_i64, _c_p],
                                       _c_i32),
    "pa_copy_blocks": ([_c_p, _c_p, _c_i32, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p], _c_i32),
    "pa_get_device_error": ([_c_p, _c_p], _c_i32),
    "pa_selftest_bounded_wait": ([_c_p, ctypes.c_longlong, _c_p], _c_i32),
    "pa_map_to_kernel_blocks": ([_c_p, _c_i64, _c_i64, _c_i64, _c_i32, _c_p, _c_i64, _c_p],
                                _c_i32),
}

_lock = threading.Lock()
_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        try:
            msg = lib().pa_status_string(status).decode()
        except Exception:  # pragma: no cover
            msg = "?"
        super().__init__(f"{func} returned {name}: {msg}")


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it first "
                        "(python -c 'import __graft_entry__ as g; g.build()')")
                h = ctypes.CDLL(LIB_PATH)
                for name, (args, res) in SIGNATURES.items():
                    fn = getattr(h, name)
                    fn.argtypes = args
                    fn.restype = res
                _lib = h
    return _lib


def check(func: str, status: int) -> None:
    if status != PA_OK:
        raise PagedAttnError(func, status)


def ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def stream_handle(stream=None) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream
