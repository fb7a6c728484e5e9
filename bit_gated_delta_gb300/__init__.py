"""PACE decode hot path for GB300: Python binding of libpace.

The functions below carry the names of the C ABI (include/pace.h) and only marshal arguments:
torch tensors become device pointers, torch streams become cudaStream_t handles. PyTorch is used
for device memory and streams; every step of the path runs in the CUDA library.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from ._lib import (PACE_BUF_FP32, PACE_BUF_INT8, PACE_BUF_MIXED, PACE_ERR_STATE, PACE_ERR_TIMEOUT, PACE_IO_BF16,
                   PACE_IO_F32, PACE_MAX_DP, PACE_MAX_HEADS, PACE_STATE_BF16, PACE_STATE_BF16_BUF, PACE_STATE_FP32,
                   PACE_STATE_QUANT, PACE_GUARD_BYTES, PACE_VALIDATE_N, PaceError, check, lib, pace_config, pace_layout)

__all__ = [
    "pace_config", "make_config", "pace_state_bytes", "pace_state_alloc", "pace_state_free",
    "pace_state_get_layout", "pace_prefill_chunk", "pace_decode_step", "pace_flush", "pace_assign_heads",
    "pace_quantize_state", "pace_dequantize_state", "pace_calib_error_energy", "pace_calib_error_energy_axis",
    "pace_state_export",
    "pace_state_import", "pace_resident_bits", "pace_get_status", "pace_test_wait_probe", "pace_validate_state",
    "pace_last_error", "pace_version", "VALIDATE_FIELDS",
    "PaceState", "PaceError", "PACE_ERR_TIMEOUT", "PACE_ERR_STATE",
    "PACE_STATE_QUANT", "PACE_STATE_FP32", "PACE_STATE_BF16", "PACE_STATE_BF16_BUF", "PACE_BUF_INT8", "PACE_BUF_MIXED",
    "PACE_BUF_FP32", "PACE_IO_BF16", "PACE_IO_F32", "PACE_MAX_HEADS", "PACE_MAX_DP", "PACE_GUARD_BYTES",
    "PACE_VALIDATE_N",
]


def make_config(n_heads: int, d: int, max_batch: int, dP: int = 8, group: int = 64, zero_point: int = 0,
                buf_mode: int = PACE_BUF_INT8, state_mode: int = PACE_STATE_QUANT, io_dtype: int = PACE_IO_BF16,
                prefill_chunk: int = 256, key_heads: int = 0) -> pace_config:
    return pace_config(n_heads, d, d, max_batch, dP, group, zero_point, buf_mode, state_mode, prefill_chunk,
                       io_dtype, key_heads)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _mask(head_is_int8):
    if head_is_int8 is None:
        return None, None
    m = np.ascontiguousarray(np.asarray(head_is_int8, dtype=np.uint8))
    return m, m.ctypes.data_as(C.POINTER(C.c_uint8))


def pace_version() -> int:
    return lib().pace_version()


def pace_last_error() -> str:
    return lib().pace_last_error().decode()


def pace_state_bytes(cfg: pace_config, head_is_int8=None) -> int:
    keep, mp = _mask(head_is_int8)
    out = C.c_size_t()
    check(lib().pace_state_bytes(C.byref(cfg), mp, C.byref(out)))
    return out.value


def pace_state_alloc(cfg: pace_config, head_is_int8, device_mem, nbytes: int, batch: int, stream=None) -> int:
    keep, mp = _mask(head_is_int8)
    h = C.c_void_p()
    check(lib().pace_state_alloc(C.byref(cfg), mp, _ptr(device_mem), nbytes, batch, _stream(stream), C.byref(h)))
    return h.value


def pace_state_free(handle) -> None:
    if handle:
        lib().pace_state_free(handle)


def pace_state_get_layout(handle) -> pace_layout:
    out = pace_layout()
    check(lib().pace_state_get_layout(handle, C.byref(out)))
    return out


def pace_prefill_chunk(handle, n_tokens: int, q, k, v, a, beta, o, stream=None) -> None:
    check(lib().pace_prefill_chunk(handle, n_tokens, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(o),
                                   _stream(stream)))


def pace_decode_step(handle, q, k, v, a, beta, o, stream=None) -> None:
    check(lib().pace_decode_step(handle, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(o), _stream(stream)))


def pace_flush(handle, stream=None) -> None:
    check(lib().pace_flush(handle, _stream(stream)))


def pace_assign_heads(e_h, a_h, dP: int, frac: float = 0.25) -> np.ndarray:
    e = np.ascontiguousarray(e_h, dtype=np.float32)
    a = np.ascontiguousarray(a_h, dtype=np.float32)
    out = np.zeros(e.size, np.uint8)
    check(lib().pace_assign_heads(e.ctypes.data_as(C.POINTER(C.c_float)), a.ctypes.data_as(C.POINTER(C.c_float)),
                                  e.size, dP, frac, out.ctypes.data_as(C.POINTER(C.c_uint8))))
    return out


def pace_quantize_state(handle, S, stream=None) -> None:
    check(lib().pace_quantize_state(handle, _ptr(S), _stream(stream)))


def pace_dequantize_state(handle, S_out, stream=None) -> None:
    check(lib().pace_dequantize_state(handle, _ptr(S_out), _stream(stream)))


def pace_calib_error_energy(handle, bits: int, group: int, zero_point: int, e_out, stream=None) -> None:
    check(lib().pace_calib_error_energy(handle, bits, group, zero_point, _ptr(e_out), _stream(stream)))


def pace_calib_error_energy_axis(handle, bits: int, group: int, zero_point: int, axis: int, e_out,
                                 stream=None) -> None:
    check(lib().pace_calib_error_energy_axis(handle, bits, group, zero_point, axis, _ptr(e_out), _stream(stream)))


def pace_state_export(handle, dst, nbytes: int, stream=None) -> None:
    check(lib().pace_state_export(handle, _ptr(dst), nbytes, _stream(stream)))


def pace_state_import(handle, src, nbytes: int, stream=None) -> None:
    check(lib().pace_state_import(handle, _ptr(src), nbytes, _stream(stream)))


def pace_get_status(handle, clear: bool = False, stream=None) -> int:
    """Reads the state's device status word (synchronises the stream); raises PaceError on a timeout bit."""
    out = C.c_int()
    check(lib().pace_get_status(handle, int(clear), C.byref(out), _stream(stream)))
    return out.value


def pace_test_wait_probe(handle, ns: int) -> None:
    """Failure-detection hook: the state's tensor-core prefill launches first wait at most ns nanoseconds on a
    barrier that nothing signals and report the timeout; 0 turns it off."""
    check(lib().pace_test_wait_probe(handle, int(ns)))


VALIDATE_FIELDS = ("bad_counters", "bad_scales_or_values", "bad_zero_points", "unused_level_codes",
                   "bad_buffer_values", "changed_guard_bytes")


def pace_validate_state(handle, stream=None) -> dict:
    """Debug check of a state (synchronises the stream): the counts of pace_validate_state by name. A non-zero
    count is reported in the dict, not raised; other errors raise PaceError."""
    out = (C.c_int64 * PACE_VALIDATE_N)()
    st = lib().pace_validate_state(handle, out, _stream(stream))
    if st != PACE_ERR_STATE:
        check(st)
    return dict(zip(VALIDATE_FIELDS, (int(x) for x in out)))


def pace_resident_bits(cfg: pace_config, head_is_int8=None, literal_formula: bool = True) -> float:
    keep, mp = _mask(head_is_int8)
    return float(lib().pace_resident_bits(C.byref(cfg), mp, int(literal_formula)))


class PaceState:
    """Owns a device region (a torch uint8 tensor) bound to a libpace state handle."""

    def __init__(self, cfg: pace_config, batch: int, head_is_int8=None, device="cuda", stream=None):
        import torch
        self.cfg = cfg
        self.batch = batch
        self.head_is_int8 = None if head_is_int8 is None else np.asarray(head_is_int8, np.uint8).copy()
        self.nbytes = pace_state_bytes(cfg, head_is_int8)
        self.mem = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        self.base = (self.mem.data_ptr() + 255) // 256 * 256
        self.handle = pace_state_alloc(cfg, head_is_int8, self.base, self.nbytes, batch, stream)
        self.layout = pace_state_get_layout(self.handle)

    def region(self):
        """The state's bytes as a uint8 tensor view (total_bytes long)."""
        off = self.base - self.mem.data_ptr()
        return self.mem[off:off + self.layout.total_bytes]

    def decode_step(self, q, k, v, a, beta, o, stream=None):
        pace_decode_step(self.handle, q, k, v, a, beta, o, stream)

    def prefill_chunk(self, q, k, v, a, beta, o, stream=None):
        pace_prefill_chunk(self.handle, int(a.shape[-1]), q, k, v, a, beta, o, stream)

    def flush(self, stream=None):
        pace_flush(self.handle, stream)

    def validate(self, stream=None) -> dict:
        return pace_validate_state(self.handle, stream)

    def close(self):
        if getattr(self, "handle", None):
            pace_state_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
