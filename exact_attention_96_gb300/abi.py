"""ctypes view of the C ABI in include/fa.h (libfa_gb300.so).

Argument marshalling only: every function here forwards to the same-named C entry point.
Loading fails loudly when the library has not been built; there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_float = ctypes.c_float
_c_size_t = ctypes.c_size_t

# name -> (restype, argtypes), in the order include/fa.h declares them
SIGNATURES = {
    "fa_fwd": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                        _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_void_p]),
    "fa_fwd_fp8": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_void_p, _c_void_p,
                            _c_int, _c_int, _c_int, _c_int, _c_float, _c_float, _c_float, _c_float,
                            _c_int, _c_void_p]),
    "fa_e4m3_descale": (_c_int, [_c_void_p, ctypes.c_longlong, _c_void_p, _c_void_p]),
    "fa_quantize_e4m3": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_void_p, _c_void_p]),
    "fa_fwd_splitkv_workspace_bytes": (_c_size_t, [_c_int] * 6),
    "fa_fwd_splitkv_num_splits": (_c_int, [_c_int] * 6),
    "fa_fwd_splitkv": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                                _c_void_p, _c_size_t, _c_void_p]),
    "fa_fwd_partial": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_void_p]),
    "fa_merge_partials": (_c_int, [_c_void_p, _c_void_p, _c_int, ctypes.c_longlong, _c_int,
                                   _c_void_p, _c_void_p, _c_void_p]),
    "fa_bwd_workspace_bytes": (_c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "fa_bwd": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                        _c_void_p, _c_void_p, _c_void_p,
                        _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                        _c_void_p, _c_size_t, _c_void_p]),
    "fa_bwd_accumulate": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                   _c_void_p, _c_void_p, _c_void_p,
                                   _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                                   _c_void_p, _c_size_t, _c_void_p]),
    "fa_convert_f32_to_bf16": (_c_int, [_c_void_p, _c_void_p, ctypes.c_longlong, _c_void_p]),
    "fa_fwd_dropout": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                                ctypes.c_double, ctypes.c_ulonglong, _c_void_p]),
    "fa_bwd_dropout": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                _c_void_p, _c_void_p, _c_void_p,
                                _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                                ctypes.c_double, ctypes.c_ulonglong,
                                _c_void_p, _c_size_t, _c_void_p]),
    "fa_bwd_noalloc": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                _c_void_p, _c_void_p, _c_void_p,
                                _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_void_p]),
    "fa_step_host_workspace_bytes": (_c_size_t, [_c_int] * 5),
    "fa_step_host": (_c_int, [_c_void_p] * 18 + [_c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int,
                                                 _c_void_p, _c_size_t, _c_void_p]),
    "fa_status_check": (_c_int, [_c_void_p]),
    "fa_status_string": (ctypes.c_char_p, [_c_int]),
    "fa_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "fa_profile_next_bwd_main": (_c_int, [_c_void_p, _c_void_p]),
    "fa_test_withhold_kv_tile": (_c_int, [_c_int]),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status_string(status)} ({status})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libfa_gb300.so (once) and declares every entry point's signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(
            f"{path} is missing: build it with `python -m exact_attention_96_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().fa_status_string(status).decode()


def check(fn: str, status: int) -> None:
    if status != FA_OK:
        raise FAError(fn, status)


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    return load().fa_fwd(q, k, v, o, lse, B, H, N, d, scale, int(causal), stream)


def fa_fwd_fp8(q8, k8, vt8, ldv, o, lse, B, H, N, d, scale, q_descale, k_descale, v_descale, causal,
               stream) -> int:
    return load().fa_fwd_fp8(q8, k8, vt8, ldv, o, lse, B, H, N, d, scale, q_descale, k_descale,
                             v_descale, int(causal), stream)


def fa_e4m3_descale(x, n, descale, stream) -> int:
    return load().fa_e4m3_descale(x, n, descale, stream)


def fa_quantize_e4m3(x, out8, B, H, N, d, transpose, ld, descale, stream) -> int:
    return load().fa_quantize_e4m3(x, out8, B, H, N, d, int(transpose), ld, descale, stream)


def fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits) -> int:
    return load().fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)


def fa_fwd_splitkv_num_splits(B, H, Nq, Nk, d, num_splits) -> int:
    return load().fa_fwd_splitkv_num_splits(B, H, Nq, Nk, d, num_splits)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, num_splits, ws, ws_bytes, stream) -> int:
    return load().fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, num_splits, ws, ws_bytes, stream)


def fa_fwd_partial(q, k, v, o_part, lse_part, B, H, Nq, Nk, d, scale, causal, stream) -> int:
    return load().fa_fwd_partial(q, k, v, o_part, lse_part, B, H, Nq, Nk, d, scale, int(causal), stream)


def fa_merge_partials(o_parts, lse_parts, num_parts, rows, d, o, lse, stream) -> int:
    return load().fa_merge_partials(o_parts, lse_parts, num_parts, rows, d, o, lse, stream)


def fa_bwd_workspace_bytes(B, H, N, d) -> int:
    return load().fa_bwd_workspace_bytes(B, H, N, d)


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, causal, ws, ws_bytes, stream) -> int:
    return load().fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, int(causal),
                         ws, ws_bytes, stream)


def fa_bwd_accumulate(q, k, v, o, do, lse, dq_acc, dk_acc, dv_acc, B, H, N, d, scale, causal, ws, ws_bytes,
                      stream) -> int:
    return load().fa_bwd_accumulate(q, k, v, o, do, lse, dq_acc, dk_acc, dv_acc, B, H, N, d, scale, int(causal),
                                    ws, ws_bytes, stream)


def fa_convert_f32_to_bf16(src, dst, n, stream) -> int:
    return load().fa_convert_f32_to_bf16(src, dst, n, stream)


def fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, dropout_p, seed, stream) -> int:
    return load().fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, scale, int(causal), float(dropout_p),
                                 int(seed) & 0xFFFFFFFFFFFFFFFF, stream)


def fa_bwd_dropout(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, causal, dropout_p, seed,
                   ws, ws_bytes, stream) -> int:
    return load().fa_bwd_dropout(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, int(causal),
                                 float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF, ws, ws_bytes, stream)


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, causal, stream) -> int:
    return load().fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, int(causal), stream)


def fa_step_host_workspace_bytes(B, H, N, d, num_chunks) -> int:
    return load().fa_step_host_workspace_bytes(B, H, N, d, num_chunks)


def fa_step_host(host_ptrs, dev_ptrs, B, H, N, d, scale, causal, num_chunks, ws, ws_bytes, stream) -> int:
    """host_ptrs: (q, k, v, do, o, lse, dq, dk, dv); dev_ptrs: (q, k, v, do, o, lse, dq, dk, dv)."""
    return load().fa_step_host(*host_ptrs, *dev_ptrs, B, H, N, d, scale, int(causal), num_chunks, ws, ws_bytes,
                               stream)


def fa_status_check(stream) -> int:
    return load().fa_status_check(stream)


def fa_set_wait_limit_ns(ns: int) -> int:
    return load().fa_set_wait_limit_ns(ns)


def fa_profile_next_bwd_main(start_event, stop_event) -> int:
    return load().fa_profile_next_bwd_main(start_event, stop_event)


def fa_test_withhold_kv_tile(tile: int) -> int:
    return load().fa_test_withhold_kv_tile(tile)
