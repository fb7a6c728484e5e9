"""ctypes wrapper of the plain CPU oracle (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package. It never imports the CUDA library and the CUDA library never imports it; the two
meet only through the seeded input generator in ``synth.py``.

The arithmetic lives in ``pace_oracle.c``; this module only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pace_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")

BUF_INT8, BUF_MIXED, BUF_FP32 = 0, 1, 2
STATE_QUANT, STATE_FP32, STATE_BF16, STATE_BF16_BUF = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction; OpenMP only for the batched timing call)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-fopenmp", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


class _Cfg(C.Structure):
    _fields_ = [("d_k", C.c_int), ("d_v", C.c_int), ("g", C.c_int), ("bits", C.c_int),
                ("zero_point", C.c_int), ("dP", C.c_int), ("buf_mode", C.c_int), ("state_mode", C.c_int)]


_P_I32 = C.POINTER(C.c_int32)
_P_F32 = C.POINTER(C.c_float)
_P_F64 = C.POINTER(C.c_double)


class _Unit(C.Structure):
    _fields_ = [("code", _P_I32), ("scale", _P_F32), ("zp", _P_I32), ("S", _P_F64), ("m", C.c_int),
                ("bk", _P_I32), ("bv", _P_I32), ("bsk", _P_F32), ("bsv", _P_F32), ("bkf", _P_F32),
                ("bvf", _P_F32), ("ba", _P_F32), ("bb", _P_F32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        L = _lib
        L.orc_bf16_rn.restype = C.c_float
        L.orc_bf16_rn.argtypes = [C.c_float]
        L.orc_error_energy.restype = C.c_double
        L.orc_error_energy_axis.restype = C.c_double
        L.orc_retained_error.restype = C.c_double
        L.orc_retained_error.argtypes = [C.c_double, C.c_double, C.c_int]
        L.orc_payload_bits.restype = C.c_double
        L.orc_payload_bits.argtypes = [C.c_int, C.c_int, C.c_int]
        L.orc_buffer_bits.restype = C.c_double
        L.orc_buffer_bits.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_double, C.c_int, C.c_int]
        L.orc_assign_heads.argtypes = [_P_F64, _P_F64, C.c_int, C.c_int, C.c_double, C.POINTER(C.c_uint8)]
        L.orc_max_threads.restype = C.c_int
    return _lib


def _p(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.POINTER(ct))


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32)


@dataclass
class Cfg:
    d_k: int
    d_v: int
    g: int = 64
    bits: int = 4
    zero_point: int = 0
    dP: int = 8
    buf_mode: int = BUF_INT8
    state_mode: int = STATE_QUANT

    def c(self) -> _Cfg:
        return _Cfg(self.d_k, self.d_v, self.g, self.bits, self.zero_point, self.dP, self.buf_mode,
                    self.state_mode)

    @property
    def n_groups(self) -> int:
        return self.d_k // self.g


class Unit:
    """One (sequence, head) of resident oracle state: codes/scales/zero points, or an fp64 state,
    plus the decode buffer. Starts at zero with an empty buffer."""

    def __init__(self, cfg: Cfg):
        dk, dv, P = cfg.d_k, cfg.d_v, cfg.dP
        self.cfg = cfg
        self.code = np.zeros((dk, dv), np.int32)
        self.scale = np.zeros((cfg.n_groups, dv), np.float32)
        self.zp = np.zeros((cfg.n_groups, dv), np.int32)
        self.S = np.zeros((dk, dv), np.float64)
        self.m = 0
        self.bk = np.zeros((P, dk), np.int32)
        self.bv = np.zeros((P, dv), np.int32)
        self.bsk = np.zeros(P, np.float32)
        self.bsv = np.zeros(P, np.float32)
        self.bkf = np.zeros((P, dk), np.float32)
        self.bvf = np.zeros((P, dv), np.float32)
        self.ba = np.zeros(P, np.float32)
        self.bb = np.zeros(P, np.float32)

    def _c(self) -> _Unit:
        return _Unit(_p(self.code, C.c_int32), _p(self.scale, C.c_float), _p(self.zp, C.c_int32),
                     _p(self.S, C.c_double), self.m, _p(self.bk, C.c_int32), _p(self.bv, C.c_int32),
                     _p(self.bsk, C.c_float), _p(self.bsv, C.c_float), _p(self.bkf, C.c_float),
                     _p(self.bvf, C.c_float), _p(self.ba, C.c_float), _p(self.bb, C.c_float))

    def state(self) -> np.ndarray:
        """The resident state as fp64 values (dequantized in quantized mode)."""
        if self.cfg.state_mode == STATE_QUANT:
            return dequantize_state(self.cfg, self.code, self.scale, self.zp)
        return self.S.copy()

    def copy(self) -> "Unit":
        u = Unit(self.cfg)
        for name in ("code", "scale", "zp", "S", "bk", "bv", "bsk", "bsv", "bkf", "bvf", "ba", "bb"):
            getattr(u, name)[...] = getattr(self, name)
        u.m = self.m
        return u


# ------------------------------------------------------------------------------------------------
# Element-level primitives

def bf16_rn(x) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    lib().orc_bf16_rn_array(_p(x, C.c_float), _p(y, C.c_float), C.c_long(x.size))
    return y


def quant_group_sym(x, bits: int):
    """Symmetric b-bit quantization of one group. Returns (scale, codes)."""
    x = _f32(x).ravel()
    c = np.zeros(x.size, np.int32)
    s = C.c_float()
    lib().orc_quant_group_sym(_p(x, C.c_float), x.size, 1, bits, C.byref(s), _p(c, C.c_int32), 1)
    return np.float32(s.value), c


def quant_group_zp(x, bits: int):
    """Zero-point b-bit quantization of one group. Returns (scale, zero_point, codes)."""
    x = _f32(x).ravel()
    c = np.zeros(x.size, np.int32)
    s = C.c_float()
    z = C.c_int32()
    lib().orc_quant_group_zp(_p(x, C.c_float), x.size, 1, bits, C.byref(s), C.byref(z), _p(c, C.c_int32), 1)
    return np.float32(s.value), int(z.value), c


def quantize_state(cfg: Cfg, S32):
    """fp32 state [d_k, d_v] -> (codes [d_k, d_v], scales [d_k/g, d_v], zero points [d_k/g, d_v])."""
    S32 = _f32(S32)
    assert S32.shape == (cfg.d_k, cfg.d_v)
    code = np.zeros((cfg.d_k, cfg.d_v), np.int32)
    scale = np.zeros((cfg.n_groups, cfg.d_v), np.float32)
    zp = np.zeros((cfg.n_groups, cfg.d_v), np.int32)
    c = cfg.c()
    lib().orc_quantize_state(C.byref(c), _p(S32, C.c_float), _p(code, C.c_int32), _p(scale, C.c_float),
                             _p(zp, C.c_int32))
    return code, scale, zp


def dequantize_state(cfg: Cfg, code, scale, zp) -> np.ndarray:
    code = np.ascontiguousarray(code, np.int32)
    scale = _f32(scale)
    zp = np.ascontiguousarray(zp, np.int32)
    S = np.zeros((cfg.d_k, cfg.d_v), np.float64)
    c = cfg.c()
    lib().orc_dequantize_state(C.byref(c), _p(code, C.c_int32), _p(scale, C.c_float), _p(zp, C.c_int32),
                               _p(S, C.c_double))
    return S


def buffer_quant(x, qmax: int):
    """Per-token buffer quantization. Returns (codes, scale)."""
    x = _f32(x).ravel()
    c = np.zeros(x.size, np.int32)
    s = C.c_float()
    lib().orc_buffer_quant(_p(x, C.c_float), x.size, qmax, _p(c, C.c_int32), C.byref(s))
    return c, np.float32(s.value)


def token_update(S: np.ndarray, k, v, a: float, beta: float) -> np.ndarray:
    """In-place gated delta rule on an fp64 state; returns u."""
    assert S.dtype == np.float64 and S.flags["C_CONTIGUOUS"]
    dk, dv = S.shape
    k = np.ascontiguousarray(k, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    u = np.zeros(dv, np.float64)
    lib().orc_token_update(dk, dv, _p(S, C.c_double), _p(k, C.c_double), _p(v, C.c_double), C.c_double(a),
                           C.c_double(beta), _p(u, C.c_double))
    return u


def readout(S: np.ndarray, q) -> np.ndarray:
    dk, dv = S.shape
    S = np.ascontiguousarray(S, np.float64)
    q = np.ascontiguousarray(q, np.float64)
    o = np.zeros(dv, np.float64)
    lib().orc_readout(dk, dv, _p(S, C.c_double), _p(q, C.c_double), _p(o, C.c_double))
    return o


# ------------------------------------------------------------------------------------------------
# Unit-level steps

def decode_step(unit: Unit, q, k, v, a: float, beta: float) -> np.ndarray:
    cfg = unit.cfg
    q, k, v = _f32(q), _f32(k), _f32(v)
    o = np.zeros(cfg.d_v, np.float64)
    cu, cc = unit._c(), cfg.c()
    lib().orc_decode_step(C.byref(cc), C.byref(cu), _p(q, C.c_float), _p(k, C.c_float), _p(v, C.c_float),
                          C.c_float(a), C.c_float(beta), _p(o, C.c_double))
    unit.m = cu.m
    return o


def flush(unit: Unit) -> None:
    cu, cc = unit._c(), unit.cfg.c()
    lib().orc_flush(C.byref(cc), C.byref(cu))
    unit.m = cu.m


def prefill(unit: Unit, q, k, v, a, beta) -> np.ndarray:
    """One chunk of n tokens: q, k [n, d_k], v [n, d_v], a, beta [n]. Returns o [n, d_v]."""
    cfg = unit.cfg
    q, k, v, a, beta = _f32(q), _f32(k), _f32(v), _f32(a), _f32(beta)
    n = a.size
    o = np.zeros((n, cfg.d_v), np.float64)
    cu, cc = unit._c(), cfg.c()
    lib().orc_prefill(C.byref(cc), C.byref(cu), n, _p(q, C.c_float), _p(k, C.c_float), _p(v, C.c_float),
                      _p(a, C.c_float), _p(beta, C.c_float), _p(o, C.c_double))
    unit.m = cu.m
    return o


def error_energy(cfg: Cfg, S32) -> float:
    S32 = _f32(S32)
    c = cfg.c()
    return float(lib().orc_error_energy(C.byref(c), _p(S32, C.c_float)))


def error_energy_axis(cfg: Cfg, S32, axis: int) -> float:
    """||Q(S) - S||_F^2 with the groups along the key axis (axis 0, PACE) or the value axis (axis 1, baseline)."""
    S32 = _f32(S32)
    c = cfg.c()
    return float(lib().orc_error_energy_axis(C.byref(c), _p(S32, C.c_float), int(axis)))


def retained_error(e_h: float, a_h: float, dP: int) -> float:
    return float(lib().orc_retained_error(e_h, a_h, dP))


def assign_heads(e_h, a_h, dP: int, frac: float = 0.25) -> np.ndarray:
    e = np.ascontiguousarray(e_h, np.float64)
    a = np.ascontiguousarray(a_h, np.float64)
    mask = np.zeros(e.size, np.uint8)
    lib().orc_assign_heads(_p(e, C.c_double), _p(a, C.c_double), e.size, dP, frac, _p(mask, C.c_uint8))
    return mask


def payload_bits(bits: int, g: int, zero_point: int) -> float:
    return float(lib().orc_payload_bits(bits, g, zero_point))


def buffer_bits(d_k: int, d_v: int, b_k: int, b_v: int, gamma: float, scalar_bits: int, dP: int) -> float:
    return float(lib().orc_buffer_bits(d_k, d_v, b_k, b_v, gamma, scalar_bits, dP))


def decode_batch(units: list[Unit], q, k, v, a, beta, nthreads: int = 0) -> np.ndarray:
    """Decode one token for many units of one config (OpenMP over units). q, k [n, d_k]; v [n, d_v]."""
    cfg = units[0].cfg
    n = len(units)
    arr = (_Unit * n)(*[u._c() for u in units])
    q, k, v, a, beta = _f32(q), _f32(k), _f32(v), _f32(a), _f32(beta)
    o = np.zeros((n, cfg.d_v), np.float64)
    cc = cfg.c()
    lib().orc_decode_batch(C.byref(cc), arr, n, _p(q, C.c_float), _p(k, C.c_float), _p(v, C.c_float),
                           _p(a, C.c_float), _p(beta, C.c_float), _p(o, C.c_double), nthreads)
    for i, u in enumerate(units):
        u.m = arr[i].m
    return o


def max_threads() -> int:
    return int(lib().orc_max_threads())
