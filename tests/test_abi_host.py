"""The C-ABI library loads, exports what include/pace.h declares, and its host-only logic (validation,
layout, head ranking, accounting) agrees with the oracle. CPU only: no compute call reaches a GPU."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle as O
from pace_testlib import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def P():
    ensure_built()
    import bit_gated_delta_gb300 as P
    P.lib()
    return P


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pace.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pace_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(P):
    names = declared_functions()
    assert len(names) >= 15
    lib = C.CDLL(P._lib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pace.h but not exported"
    assert set(names) == set(P._lib.exported_symbols())


def test_version_and_error_string(P):
    assert P.pace_version() >= 100
    with pytest.raises(P.PaceError) as ei:
        P.pace_state_bytes(P.make_config(4, 96, 2))
    assert ei.value.status == 2 and "96" in str(ei.value)
    assert "96" in P.pace_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(n_heads=0), 1), (dict(n_heads=257), 1), (dict(dP=0), 1), (dict(dP=33), 1), (dict(group=16), 2),
    (dict(zero_point=2), 1), (dict(prefill_chunk=128), 2), (dict(io_dtype=5), 1), (dict(max_batch=0), 1),
    (dict(state_mode=1), 1),                      # fp32 state with an int8 buffer
    (dict(buf_mode=2), 2),                        # quantized state with an fp32 buffer
])
def test_invalid_configs_are_rejected_on_the_host(P, kw, status):
    base = dict(n_heads=4, d=128, max_batch=2)
    base.update({k: v for k, v in kw.items() if k in ("n_heads", "max_batch")})
    extra = {k: v for k, v in kw.items() if k not in ("n_heads", "max_batch")}
    cfg = P.make_config(base["n_heads"], base["d"], base["max_batch"], **extra)
    with pytest.raises(P.PaceError) as ei:
        P.pace_state_bytes(cfg)
    assert ei.value.status == status


def test_alloc_and_calls_validate_before_any_launch(P):
    cfg = P.make_config(4, 64, 2)
    n = P.pace_state_bytes(cfg)
    with pytest.raises(P.PaceError):
        P.pace_state_alloc(cfg, None, 0, n, 1, 0)                    # NULL device memory
    with pytest.raises(P.PaceError):
        P.pace_state_alloc(cfg, None, 256 * 1000 + 8, n, 1, 0)       # misaligned
    with pytest.raises(P.PaceError):
        P.pace_state_alloc(cfg, None, 256 * 1000, n - 1, 1, 0)       # too small
    with pytest.raises(P.PaceError):
        P.pace_state_alloc(cfg, None, 256 * 1000, n, 3, 0)           # batch > max_batch
    assert P.lib().pace_decode_step(None, None, None, None, None, None, None, None) == 1
    assert P.lib().pace_flush(None, None) == 1
    with pytest.raises(P.PaceError):
        P.pace_state_bytes(P.make_config(4, 64, 2, state_mode=P.PACE_STATE_FP32, buf_mode=P.PACE_BUF_FP32),
                           np.array([1, 0, 0, 0], np.uint8))            # 8-bit heads need the quantized mode


def test_state_bytes_match_layout_arithmetic(P):
    H, D, B, dP = 32, 128, 64, 8
    cfg = P.make_config(H, D, B, dP=dP)
    n = P.pace_state_bytes(cfg)
    # every array is 256-byte aligned and followed by a guard region (one per array, 9 arrays here, the status
    # array 256 bytes)
    slack = 256 * 9 + 9 * P.PACE_GUARD_BYTES + 256
    expect = B * H * (D * D // 2 + (D // 64) * D * 2 + dP * D * 2 + dP * 16 + 4)
    assert expect <= n <= expect + slack
    mask = np.zeros(H, np.uint8)
    mask[::4] = 1
    cfg2 = P.make_config(H, D, B, dP=dP, group=32, zero_point=1, buf_mode=P.PACE_BUF_MIXED)
    n2 = P.pace_state_bytes(cfg2, mask)
    e2 = B * (24 * D * D // 2 + 8 * D * D) + B * H * ((D // 32) * D * 3 + dP * (D // 2 + 2 * D + 16) + 4)
    assert e2 <= n2 <= e2 + slack


def test_assign_heads_matches_oracle(P):
    rng = np.random.default_rng(7)
    for H in (4, 8, 16, 32, 48):
        for dP in (1, 8, 32):
            e = rng.uniform(1e-3, 2.0, H).astype(np.float32)
            a = rng.uniform(0.85, 0.999, H).astype(np.float32)
            a[rng.integers(H)] = 1.0
            got = P.pace_assign_heads(e, a, dP, 0.25)
            ref = O.assign_heads(e.astype(np.float64), a.astype(np.float64), dP, 0.25)
            assert np.array_equal(got, ref)
    # ties keep the lower head index
    assert list(np.flatnonzero(P.pace_assign_heads(np.ones(8), np.full(8, 0.9), 8, 0.25))) == [0, 1]
    with pytest.raises(P.PaceError):
        P.pace_assign_heads(np.ones(4), np.full(4, 0.9), 8, 1.5)


@pytest.mark.parametrize("zp,g,buf,n8,kh", [(0, 64, 0, 0, 32), (1, 32, 1, 8, 32), (1, 32, 0, 8, 32), (0, 32, 0, 0, 32),
                                             (0, 64, 0, 0, 16), (1, 32, 1, 8, 8)])
def test_resident_bits_formula_matches_oracle_accounting(P, zp, g, buf, n8, kh):
    H, D, dP = 32, 128, 8
    mask = np.zeros(H, np.uint8)
    mask[:n8] = 1
    cfg = P.make_config(H, D, 16, dP=dP, group=g, zero_point=zp, buf_mode=buf, key_heads=kh)
    got = P.pace_resident_bits(cfg, mask, True)
    f8 = n8 / H
    payload = (1 - f8) * O.payload_bits(4, g, zp) + f8 * O.payload_bits(8, g, zp)
    bk, bv = (4, 16) if buf == 1 else (8, 8)
    ref = payload + O.buffer_bits(D, D, bk, bv, H / kh, 32, dP)
    assert got == pytest.approx(ref, rel=1e-12)
    exact = P.pace_resident_bits(cfg, mask, False)
    assert exact >= got - 1e-9     # the layout keeps beta and per-token scales too
    if kh < H:                     # shared key heads keep one buffered key row per key head
        full = P.pace_resident_bits(P.make_config(H, D, 16, dP=dP, group=g, zero_point=zp, buf_mode=buf), mask, False)
        kbytes = (0.5 if buf == 1 else 1.0) * D * dP * 16 * (H - kh)
        assert full - exact == pytest.approx(8.0 * kbytes / (16 * H * D * D), rel=1e-3, abs=1e-3)


def test_bench_algorithmic_bytes_follow_the_state_layout(P):
    """The roofline's numerator (bench.py) is the layout's bytes: per unit-step the packed int4 codes and bf16 group
    scales read (and written at the rounding step), the buffered int8 entries read (k and v rows plus a, beta and
    the two scales), the new entry written, q/k/v read and o written in bf16, a and beta, and the count. The state
    and entry sizes are the ones pace_state_bytes allots per unit."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    H, D, B, dP, g = 32, 128, 64, 8, 64
    state = D * D // 2 + (D // g) * D * 2                  # codes + scales of one unit
    entry = 2 * D + 16                                     # int8 k and v rows + (a, beta, s_k, s_v)
    n = P.pace_state_bytes(P.make_config(H, D, B, dP=dP, group=g))
    slack = 256 * 9 + 9 * P.PACE_GUARD_BYTES + 256     # alignment, guard regions, status array
    assert B * H * (state + dP * entry + 4) <= n <= B * H * (state + dP * entry + 4) + slack
    io = 3 * D * 2 + D * 2 + 8
    for m0 in range(dP):
        want = state + m0 * entry + entry + io + 8 + (state if m0 + 1 == dP else 0)
        assert bench.decode_bytes_per_unit(D, g, dP, m0) == want
    avg = bench.decode_bytes_period_avg(D, g, dP)
    assert avg == 12056 and B * H * avg == 24690688
    # per-token bf16: the bf16 state read and written every step, plus the token I/O
    assert bench.bf16_bytes_per_unit(D) == 2 * D * D * 2 + io
    # buffered bf16: the state read every step, written once per period, the same buffer traffic as PACE-4
    assert bench.bf16buf_bytes_per_period_avg(D, dP) == D * D * 2 * (1 + 1 / dP) + sum(range(dP)) * entry / dP + entry + io + 8
