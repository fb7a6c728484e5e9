"""ctypes binding of libpace (argument marshalling only; every step of the path runs in the library).

Loading fails loudly when the compiled library is missing: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpace.so")

PACE_OK, PACE_ERR_INVALID_ARG, PACE_ERR_UNSUPPORTED, PACE_ERR_STATE, PACE_ERR_CUDA, PACE_ERR_TIMEOUT = range(6)
PACE_STATE_QUANT, PACE_STATE_FP32, PACE_STATE_BF16, PACE_STATE_BF16_BUF = 0, 1, 2, 3
PACE_BUF_INT8, PACE_BUF_MIXED, PACE_BUF_FP32 = 0, 1, 2
PACE_IO_BF16, PACE_IO_F32 = 0, 1
PACE_MAX_HEADS = 256
PACE_MAX_DP = 32
PACE_VALIDATE_N = 6
PACE_GUARD_BYTES = 256
_STATUS_NAMES = {0: "PACE_OK", 1: "PACE_ERR_INVALID_ARG", 2: "PACE_ERR_UNSUPPORTED", 3: "PACE_ERR_STATE",
                 4: "PACE_ERR_CUDA", 5: "PACE_ERR_TIMEOUT"}


class pace_config(C.Structure):
    _fields_ = [("n_heads", C.c_int), ("d_k", C.c_int), ("d_v", C.c_int), ("max_batch", C.c_int),
                ("dP", C.c_int), ("group", C.c_int), ("zero_point", C.c_int), ("buf_mode", C.c_int),
                ("state_mode", C.c_int), ("prefill_chunk", C.c_int), ("io_dtype", C.c_int), ("key_heads", C.c_int)]


class pace_layout(C.Structure):
    _fields_ = [("codes4", C.c_size_t), ("codes8", C.c_size_t), ("scale", C.c_size_t), ("zp", C.c_size_t),
                ("buf_k", C.c_size_t), ("buf_v", C.c_size_t), ("buf_s", C.c_size_t), ("m", C.c_size_t),
                ("S", C.c_size_t), ("status", C.c_size_t), ("total_bytes", C.c_size_t), ("H4", C.c_int), ("H8", C.c_int),
                ("head_slot", C.c_int * PACE_MAX_HEADS), ("head_is_int8", C.c_uint8 * PACE_MAX_HEADS)]


class PaceError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None
_VP, _SZ, _I, _F, _D = C.c_void_p, C.c_size_t, C.c_int, C.c_float, C.c_double
_PF = C.POINTER(C.c_float)
_PU8 = C.POINTER(C.c_uint8)

_SIGS = {
    "pace_version": (_I, []),
    "pace_last_error": (C.c_char_p, []),
    "pace_state_bytes": (_I, [C.POINTER(pace_config), _PU8, C.POINTER(_SZ)]),
    "pace_state_alloc": (_I, [C.POINTER(pace_config), _PU8, _VP, _SZ, _I, _VP, C.POINTER(_VP)]),
    "pace_state_free": (None, [_VP]),
    "pace_state_get_layout": (_I, [_VP, C.POINTER(pace_layout)]),
    "pace_prefill_chunk": (_I, [_VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "pace_decode_step": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "pace_flush": (_I, [_VP, _VP]),
    "pace_assign_heads": (_I, [_PF, _PF, _I, _I, _F, _PU8]),
    "pace_quantize_state": (_I, [_VP, _VP, _VP]),
    "pace_dequantize_state": (_I, [_VP, _VP, _VP]),
    "pace_calib_error_energy": (_I, [_VP, _I, _I, _I, _VP, _VP]),
    "pace_calib_error_energy_axis": (_I, [_VP, _I, _I, _I, _I, _VP, _VP]),
    "pace_state_export": (_I, [_VP, _VP, _SZ, _VP]),
    "pace_state_import": (_I, [_VP, _VP, _SZ, _VP]),
    "pace_resident_bits": (_D, [C.POINTER(pace_config), _PU8, _I]),
    "pace_get_status": (_I, [_VP, _I, C.POINTER(C.c_int), _VP]),
    "pace_test_wait_probe": (_I, [_VP, C.c_uint32]),
    "pace_validate_state": (_I, [_VP, C.POINTER(C.c_int64), _VP]),
}


def lib() -> C.CDLL:
    """The loaded library. Raises if libpace.so has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m bit_gated_delta_gb300.build` "
                               "or __graft_entry__.build(); there is no fallback implementation")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGS)


def check(status: int) -> None:
    if status != PACE_OK:
        raise PaceError(status, lib().pace_last_error().decode())
