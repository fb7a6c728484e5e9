"""Pins of the CPU oracle against facts it did not produce itself (CPU only).

Each test checks the oracle against a closed form, an invariant, brute force on tiny inputs, a
library routine, or a number the pages print, so that a dropped term, a wrong sign, a wrong index
or a transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction
from itertools import combinations

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def rand_unit_vec(n, rng=RNG):
    x = rng.standard_normal(n)
    return x / np.linalg.norm(x)


# ------------------------------------------------------------------------------------------------
# bf16 rounding: against torch's bf16 conversion (round to nearest, ties to even).

def test_bf16_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    x = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** RNG.integers(-30, 30, 20000),
        # exact ties: low 16 bits == 0x8000, with even and odd kept halves
        (np.arange(1000, dtype=np.uint32) << 16 | 0x3F800000 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -2.5, 3.4e38, -3.4e38, 1e-40, np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = O.bf16_rn(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------------------------------------
# Gated delta rule: closed forms and invariants.

def test_one_token_from_zero_state_closed_form():
    dk, dv = 7, 5
    k, v, q = RNG.standard_normal(dk), RNG.standard_normal(dv), RNG.standard_normal(dk)
    a, beta = 0.83, 0.61
    S = np.zeros((dk, dv))
    u = O.token_update(S, k, v, a, beta)
    np.testing.assert_allclose(u, beta * v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(S, beta * np.outer(k, v), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.readout(S, q), beta * (k @ q) * v, rtol=1e-13, atol=1e-14)


def test_identity_when_a_is_one_and_beta_zero():
    S = RNG.standard_normal((6, 9))
    S0 = S.copy()
    O.token_update(S, RNG.standard_normal(6), RNG.standard_normal(9), 1.0, 0.0)
    assert np.array_equal(S, S0)


@pytest.mark.parametrize("a", [0.3, 0.9, 0.999, 1.0])
def test_unit_key_full_beta_writes_v_exactly(a):
    # With |k| = 1 and beta = 1 the new state returns v for key k: S_t^T k_t = v_t,
    # whatever a and S_{t-1} are (non-symmetric S catches a transposed product).
    dk, dv = 8, 6
    S = RNG.standard_normal((dk, dv)) * 3
    k = rand_unit_vec(dk)
    v = RNG.standard_normal(dv)
    O.token_update(S, k, v, a, 1.0)
    np.testing.assert_allclose(S.T @ k, v, rtol=0, atol=1e-12)


def test_decay_enters_the_prediction():
    # u = beta (v - a S^T k): with v = a S^T k the update leaves S scaled by a only.
    dk, dv = 5, 4
    S = RNG.standard_normal((dk, dv))
    k = RNG.standard_normal(dk)
    a = 0.7
    v = a * (S.T @ k)
    S1 = S.copy()
    u = O.token_update(S1, k, v, a, 0.9)
    np.testing.assert_allclose(u, 0.0, atol=1e-14)
    np.testing.assert_allclose(S1, a * S, rtol=1e-14)


@pytest.mark.parametrize("beta", [0.05, 0.5, 1.0])
def test_contraction_with_unit_keys(beta):
    # With v = 0: S <- a (I - beta k k^T) S, a contraction for |k| = 1, beta in (0, 1].
    dk, dv = 16, 12
    S = RNG.standard_normal((dk, dv))
    for _ in range(50):
        n0 = np.linalg.norm(S)
        O.token_update(S, rand_unit_vec(dk), np.zeros(dv), 0.97, beta)
        assert np.linalg.norm(S) <= 0.97 * n0 * (1 + 1e-12)


def test_readout_small_hand_example():
    S = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])   # d_k = 2, d_v = 3
    q = np.array([10.0, -1.0])
    np.testing.assert_array_equal(O.readout(S, q), [6.0, 15.0, 24.0])  # o = S^T q


# ------------------------------------------------------------------------------------------------
# Quantizers: hand-checked groups, error bounds, brute-force nearest code, grid round trips.

def test_sym_hand_examples():
    # zero group: zero scale, zero codes
    s, c = O.quant_group_sym(np.zeros(4), 4)
    assert s == 0.0 and not c.any()
    # single outlier: A = 100, s = bf16(100/7 = 14.2857...) = 14.3125 (229/16); 100/14.3125 = 6.99 -> 7
    s, c = O.quant_group_sym(np.array([100.0, 1.0, -1.0, 7.2]), 4)
    assert s == np.float32(14.3125)
    assert list(c) == [7, 0, 0, 1]          # 7.2/14.3125 = 0.503 -> 1
    # constant group: every code is qmax
    s, c = O.quant_group_sym(np.full(8, -0.37), 4)
    assert list(c) == [-7] * 8
    # ties go to even: s = 1 exactly (A = 7), x = 0.5, 1.5, 2.5, -2.5 -> 0, 2, 2, -2
    s, c = O.quant_group_sym(np.array([7.0, 0.5, 1.5, 2.5, -2.5]), 4)
    assert s == 1.0 and list(c) == [7, 0, 2, 2, -2]
    # 8-bit symmetric uses +-127
    s, c = O.quant_group_sym(np.array([127.0, -127.0, 0.5, 1.5]), 8)
    assert s == 1.0 and list(c) == [127, -127, 0, 2]


def test_zp_hand_examples():
    # all positive: range [0, 15] -> s = 1, z = 0
    s, z, c = O.quant_group_zp(np.array([15.0, 3.0, 0.4]), 4)
    assert (s, z, list(c)) == (1.0, 0, [15, 3, 0])
    # all negative: range [-15, 0] -> z = 15
    s, z, c = O.quant_group_zp(np.array([-15.0, -3.0, -0.6]), 4)
    assert (s, z, list(c)) == (1.0, 15, [0, 12, 14])
    # mixed signs: [-5, 10]: s = 1, z = 5
    s, z, c = O.quant_group_zp(np.array([-5.0, 10.0, 0.0, 2.5]), 4)
    assert (s, z, list(c)) == (1.0, 5, [0, 15, 5, 7])      # 2.5 -> 2 (ties to even) + 5
    # 8-bit zero point: [0, 255]
    s, z, c = O.quant_group_zp(np.array([255.0, 1.0]), 8)
    assert (s, z, list(c)) == (1.0, 0, [255, 1])
    s, z, c = O.quant_group_zp(np.zeros(5), 4)
    assert s == 0.0 and z == 0 and not c.any()


@pytest.mark.parametrize("bits", [4, 8])
def test_sym_error_at_most_half_step(bits):
    for trial in range(300):
        x = (RNG.standard_normal(64) * 10.0 ** RNG.uniform(-6, 3)).astype(np.float32)
        if trial % 3 == 0:
            x[RNG.integers(64)] *= 40.0                 # column outlier
        s, c = O.quant_group_sym(x, bits)
        qmax = 2 ** (bits - 1) - 1
        assert np.abs(c).max() <= qmax
        err = np.abs(x.astype(np.float64) - float(s) * c)
        assert err.max() <= float(s) * (0.5 + 1e-6)


@pytest.mark.parametrize("bits", [4, 8])
def test_zp_error_bound(bits):
    qm = 2 ** bits - 1
    for trial in range(300):
        x = (RNG.standard_normal(32) * 10.0 ** RNG.uniform(-5, 3) + RNG.uniform(-2, 2)).astype(np.float32)
        s, z, c = O.quant_group_zp(x, bits)
        assert 0 <= z <= qm and c.min() >= 0 and c.max() <= qm
        lo, hi = min(0.0, float(x.min())), max(0.0, float(x.max()))
        # half a step, plus the part of the range the rounded-down bf16 scale cannot reach
        overshoot = max(0.0, (hi - lo) - qm * float(s))
        err = np.abs(x.astype(np.float64) - float(s) * (c - z))
        assert err.max() <= float(s) * (0.5 + 1e-6) + overshoot + 1e-6 * float(s)
        assert overshoot <= (hi - lo) * 2.0 ** -8


@pytest.mark.parametrize("bits,zp", [(4, 0), (8, 0), (4, 1)])
def test_chosen_code_is_a_nearest_code_brute_force(bits, zp):
    for _ in range(200):
        x = RNG.standard_normal(6).astype(np.float32) * np.float32(RNG.uniform(0.01, 50))
        if zp:
            s, z, c = O.quant_group_zp(x, bits)
            grid = float(s) * (np.arange(0, 2 ** bits) - z)
            got = float(s) * (c - z)
        else:
            s, c = O.quant_group_sym(x, bits)
            q = 2 ** (bits - 1) - 1
            grid = float(s) * np.arange(-q, q + 1)
            got = float(s) * c
        best = np.min(np.abs(x[:, None].astype(np.float64) - grid[None, :]), axis=1)
        # the chosen code is nearest up to fp32 rounding of x * (1/s); the top code may be clamped
        slack = 1e-6 * float(s) + (float(np.abs(x).max()) * 2.0 ** -8 if zp else 0.0)
        assert np.all(np.abs(x - got) <= best + slack)


@pytest.mark.parametrize("bits,zp", [(4, 0), (8, 0), (4, 1), (8, 1)])
def test_values_on_the_grid_round_trip(bits, zp):
    cfg = O.Cfg(d_k=64, d_v=8, g=32, bits=bits, zero_point=zp)
    qm = 2 ** (bits - 1) - 1 if not zp else 2 ** bits - 1
    for _ in range(20):
        code = np.zeros((64, 8), np.int32)
        scale = O.bf16_rn(RNG.uniform(0.01, 3.0, (2, 8)).astype(np.float32))
        zpt = np.zeros((2, 8), np.int32)
        for gi in range(2):
            for j in range(8):
                if zp:
                    z = int(RNG.integers(0, qm + 1))
                    cc = RNG.integers(0, qm + 1, 32)
                    cc[0], cc[1] = 0, qm                     # range [-z, qm - z] contains 0
                    zpt[gi, j] = z
                else:
                    cc = RNG.integers(-qm, qm + 1, 32)
                    cc[0] = qm * (1 if RNG.random() < 0.5 else -1)
                code[gi * 32:(gi + 1) * 32, j] = cc
        S = O.dequantize_state(cfg, code, scale, zpt).astype(np.float32)
        c2, s2, z2 = O.quantize_state(cfg, S)
        assert np.array_equal(s2, scale)
        assert np.array_equal(c2, code)
        if zp:
            assert np.array_equal(z2, zpt)


def test_groups_run_along_the_key_axis_of_one_column():
    # An outlier in one column must not change any other column's codes, and one group of 32 rows
    # must not change the other group of the same column.
    cfg = O.Cfg(d_k=64, d_v=4, g=32, bits=4)
    S = RNG.standard_normal((64, 4)).astype(np.float32)
    c0, s0, _ = O.quantize_state(cfg, S)
    S2 = S.copy()
    S2[5, 2] = 1000.0
    c1, s1, _ = O.quantize_state(cfg, S2)
    changed = np.argwhere(c0 != c1)
    assert len(changed) > 0 and np.all(changed[:, 1] == 2) and np.all(changed[:, 0] < 32)
    assert np.array_equal(s0[1], s1[1]) and np.array_equal(s0[:, [0, 1, 3]], s1[:, [0, 1, 3]])


def test_buffer_quant_hand_examples():
    c, s = O.buffer_quant(np.array([1.0, -0.5, 0.25, 0.0]), 127)
    assert s == np.float32(1.0) / np.float32(127.0)
    assert list(c) == [127, -64, 32, 0]           # -63.5 -> -64 (ties to even), 31.75 -> 32
    c, s = O.buffer_quant(np.zeros(3), 127)
    assert s == 0.0 and not c.any()
    c, s = O.buffer_quant(np.array([-7.0, 3.5, 1.0]), 7)
    assert list(c) == [-7, 4, 1]                  # 3.5 -> 4 (ties to even)


def test_buffer_quant_error_bound():
    for _ in range(300):
        x = (RNG.standard_normal(128) * 10.0 ** RNG.uniform(-4, 2)).astype(np.float32)
        for qmax in (127, 7):
            c, s = O.buffer_quant(x, qmax)
            assert np.abs(c).max() <= qmax
            assert np.abs(x - float(s) * c).max() <= float(s) * (0.5 + 1e-6)


# ------------------------------------------------------------------------------------------------
# Decode step: buffer bookkeeping, flush timing, periodic rounding.

def _tokens(n, dk, dv, rng=RNG, f32=True):
    out = []
    for _ in range(n):
        q, k = rand_unit_vec(dk, rng), rand_unit_vec(dk, rng)
        v = rng.standard_normal(dv)
        v[1] *= 8.0
        out.append(dict(q=q.astype(np.float32), k=k.astype(np.float32), v=v.astype(np.float32),
                        a=np.float32(rng.uniform(0.9, 0.999)), beta=np.float32(1 / (1 + np.exp(-rng.standard_normal())))))
    return out


@pytest.mark.parametrize("dP", [1, 2, 3, 8, 32])
def test_unquantized_decode_equals_plain_recurrence_for_any_period(dP):
    dk, dv = 12, 10
    cfg = O.Cfg(d_k=dk, d_v=dv, g=4, dP=dP, buf_mode=O.BUF_FP32, state_mode=O.STATE_FP32)
    unit = O.Unit(cfg)
    S0 = RNG.standard_normal((dk, dv))
    unit.S[...] = S0
    S = S0.copy()
    for t, tk in enumerate(_tokens(40, dk, dv)):
        o = O.decode_step(unit, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
        O.token_update(S, tk["k"].astype(np.float64), tk["v"].astype(np.float64), float(tk["a"]), float(tk["beta"]))
        np.testing.assert_allclose(o, S.T @ tk["q"].astype(np.float64), rtol=1e-12, atol=1e-12)
        assert unit.m == (t + 1) % dP
    O.flush(unit)
    np.testing.assert_allclose(unit.S, S, rtol=1e-12, atol=1e-12)


def test_quantized_period_one_is_per_token_requantization():
    dk, dv = 16, 8
    cfg = O.Cfg(d_k=dk, d_v=dv, g=8, bits=4, dP=1)
    unit = O.Unit(cfg)
    code, scale, zp = O.quantize_state(cfg, RNG.standard_normal((dk, dv)).astype(np.float32))
    unit.code[...], unit.scale[...] = code, scale
    for tk in _tokens(12, dk, dv):
        S = O.dequantize_state(cfg, unit.code, unit.scale, unit.zp)
        kc, sk = O.buffer_quant(tk["k"], 127)
        vc, sv = O.buffer_quant(tk["v"], 127)
        O.token_update(S, float(sk) * kc.astype(np.float64), float(sv) * vc.astype(np.float64),
                       float(tk["a"]), float(tk["beta"]))
        expect_o = S.T @ tk["q"].astype(np.float64)
        expect_code, expect_scale, _ = O.quantize_state(cfg, S.astype(np.float32))
        o = O.decode_step(unit, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
        np.testing.assert_allclose(o, expect_o, rtol=1e-13, atol=1e-13)
        assert np.array_equal(unit.code, expect_code) and np.array_equal(unit.scale, expect_scale)
        assert unit.m == 0


@pytest.mark.parametrize("zp,bits,g,buf", [(0, 4, 64, O.BUF_INT8), (1, 4, 32, O.BUF_MIXED),
                                           (1, 8, 32, O.BUF_MIXED), (0, 8, 32, O.BUF_INT8)])
def test_state_rounded_once_per_period_from_buffered_tokens(zp, bits, g, buf):
    dk, dv, dP = 64, 16, 8
    cfg = O.Cfg(d_k=dk, d_v=dv, g=g, bits=bits, zero_point=zp, dP=dP, buf_mode=buf)
    unit = O.Unit(cfg)
    unit.code[...], unit.scale[...], unit.zp[...] = O.quantize_state(cfg, RNG.standard_normal((dk, dv)).astype(np.float32))
    toks = _tokens(2 * dP + 3, dk, dv)
    S = O.dequantize_state(cfg, unit.code, unit.scale, unit.zp)
    for t, tk in enumerate(toks):
        code_before = unit.code.copy()
        o = O.decode_step(unit, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
        # the buffered (quantized) token, applied to the running fp64 state
        if buf == O.BUF_MIXED:
            kc, sk = O.buffer_quant(tk["k"], 7)
            vd = O.bf16_rn(tk["v"]).astype(np.float64)
        else:
            kc, sk = O.buffer_quant(tk["k"], 127)
            vc, sv = O.buffer_quant(tk["v"], 127)
            vd = float(sv) * vc.astype(np.float64)
        O.token_update(S, float(sk) * kc.astype(np.float64), vd, float(tk["a"]), float(tk["beta"]))
        np.testing.assert_allclose(o, S.T @ tk["q"].astype(np.float64), rtol=1e-12, atol=1e-12)
        if (t + 1) % dP == 0:
            c, s, z = O.quantize_state(cfg, S.astype(np.float32))
            assert np.array_equal(unit.code, c) and np.array_equal(unit.scale, s)
            if zp:
                assert np.array_equal(unit.zp, z)
            S = O.dequantize_state(cfg, unit.code, unit.scale, unit.zp)
            assert unit.m == 0
        else:
            assert np.array_equal(unit.code, code_before) and unit.m == (t + 1) % dP
    # a pending buffer is applied and rounded by an explicit flush
    assert unit.m == 3
    O.flush(unit)
    c, s, z = O.quantize_state(cfg, S.astype(np.float32))
    assert unit.m == 0 and np.array_equal(unit.code, c) and np.array_equal(unit.scale, s)


def test_current_token_enters_its_output_through_buffered_values():
    # From a zero state the first output is beta (k_hat . q) v_hat with the int8-buffered k_hat, v_hat.
    dk, dv = 32, 16
    cfg = O.Cfg(d_k=dk, d_v=dv, g=32, dP=8)
    unit = O.Unit(cfg)
    tk = _tokens(1, dk, dv)[0]
    o = O.decode_step(unit, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
    kc, sk = O.buffer_quant(tk["k"], 127)
    vc, sv = O.buffer_quant(tk["v"], 127)
    kh, vh = float(sk) * kc, float(sv) * vc
    np.testing.assert_allclose(o, float(tk["beta"]) * (kh @ tk["q"].astype(np.float64)) * vh, rtol=1e-12)
    assert not np.allclose(o, float(tk["beta"]) * (tk["k"] @ tk["q"]) * tk["v"], rtol=1e-6)


@pytest.mark.parametrize("buf", [O.BUF_INT8, O.BUF_MIXED])
def test_buffered_bf16_state_rounds_once_per_period(buf):
    """Buffered bf16 mode: between roundings the outputs are the plain fp64 recurrence of the buffered
    (quantized) tokens from the last rounded state; every dP-th step the state becomes torch's bf16 rounding
    of that recurrence, and nothing else changes it."""
    import torch
    dk, dv, dP = 32, 16, 4
    cfg = O.Cfg(d_k=dk, d_v=dv, g=32, dP=dP, buf_mode=buf, state_mode=O.STATE_BF16_BUF)
    unit = O.Unit(cfg)
    S0 = torch.from_numpy(RNG.standard_normal((dk, dv)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    unit.S[...] = S0
    S = S0.copy()
    for t, tk in enumerate(_tokens(3 * dP + 2, dk, dv)):
        before = unit.S.copy()
        o = O.decode_step(unit, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
        if buf == O.BUF_MIXED:
            kc, sk = O.buffer_quant(tk["k"], 7)
            vd = O.bf16_rn(tk["v"]).astype(np.float64)
        else:
            kc, sk = O.buffer_quant(tk["k"], 127)
            vc, sv = O.buffer_quant(tk["v"], 127)
            vd = float(sv) * vc.astype(np.float64)
        O.token_update(S, float(sk) * kc.astype(np.float64), vd, float(tk["a"]), float(tk["beta"]))
        np.testing.assert_allclose(o, S.T @ tk["q"].astype(np.float64), rtol=1e-12, atol=1e-12)
        if (t + 1) % dP == 0:
            S = torch.from_numpy(S.astype(np.float32)).to(torch.bfloat16).double().numpy()
            assert np.array_equal(unit.S, S) and unit.m == 0
        else:
            assert np.array_equal(unit.S, before) and unit.m == (t + 1) % dP
    O.flush(unit)
    S = torch.from_numpy(S.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert unit.m == 0 and np.array_equal(unit.S, S)


def test_buffered_bf16_with_period_one_and_exact_buffer_is_the_per_token_mode():
    """dP = 1 with an unquantized buffer rounds after every token: the same trajectory as the per-token
    bf16 comparison mode, bit for bit."""
    dk, dv = 16, 8
    a = O.Unit(O.Cfg(d_k=dk, d_v=dv, g=16, dP=1, buf_mode=O.BUF_FP32, state_mode=O.STATE_BF16_BUF))
    b = O.Unit(O.Cfg(d_k=dk, d_v=dv, g=16, dP=1, buf_mode=O.BUF_FP32, state_mode=O.STATE_BF16))
    S0 = O.bf16_rn(RNG.standard_normal((dk, dv))).astype(np.float64)
    a.S[...] = S0
    b.S[...] = S0
    for tk in _tokens(12, dk, dv):
        oa = O.decode_step(a, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
        ob = O.decode_step(b, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
        assert np.array_equal(oa, ob) and np.array_equal(a.S, b.S)


def test_bf16_state_rounds_every_token():
    dk, dv = 16, 8
    cfg = O.Cfg(d_k=dk, d_v=dv, g=16, state_mode=O.STATE_BF16, buf_mode=O.BUF_FP32)
    unit = O.Unit(cfg)
    for tk in _tokens(10, dk, dv):
        S = unit.S.copy()
        O.token_update(S, tk["k"].astype(np.float64), tk["v"].astype(np.float64), float(tk["a"]), float(tk["beta"]))
        o = O.decode_step(unit, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
        np.testing.assert_allclose(o, S.T @ tk["q"].astype(np.float64), rtol=1e-13, atol=1e-13)
        torch = pytest.importorskip("torch")
        ref = torch.from_numpy(S.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(unit.S, ref)
        assert unit.m == 0


# ------------------------------------------------------------------------------------------------
# Prefill: the sequential oracle equals the chunked (WY / UT) closed form of the same recurrence.

def chunk_closed_form(S0, Q, K, V, a, beta):
    """Chunk form derived from the gated delta rule, independent of the oracle's token loop:
    (I + L) U = diag(beta) (V - diag(G) K S0),  L[t, s] = beta_t (G_t / G_s) k_t.k_s  (s < t),
    O = diag(G) Q S0 + (M o Q K^T) U,  M[t, s] = G_t / G_s (s <= t),
    S_C = G_C S0 + K^T diag(G_C / G) U,   G_t = a_1 ... a_t."""
    C = len(a)
    ratio = np.zeros((C, C))               # ratio[t, s] = a_{s+1} ... a_t for s <= t
    for t in range(C):
        for s in range(t + 1):
            ratio[t, s] = np.prod(a[s + 1:t + 1])
    G = np.array([np.prod(a[:t + 1]) for t in range(C)])
    L = np.tril(beta[:, None] * ratio * (K @ K.T), -1)
    U = np.linalg.solve(np.eye(C) + L, beta[:, None] * (V - G[:, None] * (K @ S0)))
    Oc = G[:, None] * (Q @ S0) + (ratio * (Q @ K.T)) @ U
    SC = G[-1] * S0 + K.T @ (ratio[-1][:, None] * U)
    return Oc, SC


@pytest.mark.parametrize("d", [4, 8, 16])
@pytest.mark.parametrize("C", [4, 8, 16])
@pytest.mark.parametrize("decay", ["random", "adversarial"])
def test_prefill_equals_chunk_closed_form(d, C, decay):
    rng = np.random.default_rng(d * 100 + C)
    cfg = O.Cfg(d_k=d, d_v=d + 2, g=d, buf_mode=O.BUF_FP32, state_mode=O.STATE_FP32)
    unit = O.Unit(cfg)
    S0 = rng.standard_normal((d, d + 2))
    unit.S[...] = S0
    Q = np.stack([rand_unit_vec(d, rng) for _ in range(C)]).astype(np.float32)
    K = np.stack([rand_unit_vec(d, rng) for _ in range(C)]).astype(np.float32)
    V = rng.standard_normal((C, d + 2)).astype(np.float32)
    if decay == "random":
        a = rng.uniform(0.8, 1.0, C).astype(np.float32)
    else:
        a = np.where(np.arange(C) % 3 == 0, 0.05, 0.9999).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, C).astype(np.float32)
    beta[0] = 1.0
    o = O.prefill(unit, Q, K, V, a, beta)
    Oc, SC = chunk_closed_form(S0, Q.astype(np.float64), K.astype(np.float64), V.astype(np.float64),
                               a.astype(np.float64), beta.astype(np.float64))
    np.testing.assert_allclose(o, Oc, rtol=0, atol=1e-12 * max(1.0, np.abs(Oc).max()))
    np.testing.assert_allclose(unit.S, SC, rtol=0, atol=1e-12 * max(1.0, np.abs(SC).max()))


@pytest.mark.parametrize("n", [256, 100, 1])
def test_quantized_prefill_rounds_once_at_chunk_end(n):
    dk, dv = 64, 16
    toks = _tokens(n, dk, dv)
    Q, K, V = (np.stack([t[x] for t in toks]) for x in ("q", "k", "v"))
    a = np.array([t["a"] for t in toks])
    beta = np.array([t["beta"] for t in toks])
    q_cfg = O.Cfg(d_k=dk, d_v=dv, g=64, bits=4)
    f_cfg = O.Cfg(d_k=dk, d_v=dv, g=64, buf_mode=O.BUF_FP32, state_mode=O.STATE_FP32)
    uq, uf = O.Unit(q_cfg), O.Unit(f_cfg)
    oq = O.prefill(uq, Q, K, V, a, beta)
    of = O.prefill(uf, Q, K, V, a, beta)
    assert np.array_equal(oq, of)          # no rounding inside the chunk
    c, s, _ = O.quantize_state(q_cfg, uf.S.astype(np.float32))
    assert np.array_equal(uq.code, c) and np.array_equal(uq.scale, s) and uq.m == 0


def test_prefill_after_pending_decode_flushes_first():
    dk, dv = 32, 8
    cfg = O.Cfg(d_k=dk, d_v=dv, g=32, dP=8)
    u1 = O.Unit(cfg)
    for tk in _tokens(3, dk, dv):
        O.decode_step(u1, tk["q"], tk["k"], tk["v"], tk["a"], tk["beta"])
    u2 = u1.copy()
    toks = _tokens(5, dk, dv)
    args = [np.stack([t[x] for t in toks]) for x in ("q", "k", "v")] + \
           [np.array([t["a"] for t in toks]), np.array([t["beta"] for t in toks])]
    o1 = O.prefill(u1, *args)
    O.flush(u2)
    o2 = O.prefill(u2, *args)
    assert np.array_equal(o1, o2) and np.array_equal(u1.code, u2.code) and u1.m == 0


# ------------------------------------------------------------------------------------------------
# Head precision allocation.

@pytest.mark.parametrize("a,dP", [(0.9, 8), (0.99, 1), (0.5, 32), (0.999, 8)])
def test_retained_error_equals_iterated_rounding(a, dP):
    # each period: the old error decays by a^dP in amplitude (a^(2dP) in energy), one new rounding adds e
    e, E = 0.37, 0.0
    for _ in range(200000):
        E_next = a ** (2 * dP) * E + e
        if abs(E_next - E) <= 1e-15 * E_next:
            break
        E = E_next
    assert O.retained_error(e, a, dP) == pytest.approx(E_next, rel=1e-12)
    assert math.isinf(O.retained_error(e, 1.0, dP))


@pytest.mark.parametrize("H", [4, 8, 12])
def test_assign_heads_matches_exhaustive_search(H):
    rng = np.random.default_rng(H)
    for _ in range(25):
        e = rng.uniform(0.1, 2.0, H)
        a = rng.uniform(0.85, 0.999, H)
        dP = int(rng.choice([1, 8, 32]))
        k = H // 4
        E = e / (1 - a ** (2 * dP))
        # best set: the k heads kept at 8 bit that leave the least retained error at 4 bit
        best = min(combinations(range(H), k), key=lambda s: sum(E[h] for h in range(H) if h not in s))
        mask = O.assign_heads(e, a, dP, 0.25)
        assert sorted(np.flatnonzero(mask)) == sorted(best)


def test_assign_heads_ties_infinite_and_fraction():
    e = np.array([1.0, 2.0, 2.0, 0.5, 2.0, 0.1, 0.1, 0.1])
    a = np.array([0.9, 0.9, 0.9, 0.9, 0.9, 1.0, 0.9, 0.9])
    mask = O.assign_heads(e, a, 8, 0.25)            # floor(8 / 4) = 2 heads
    assert list(np.flatnonzero(mask)) == [1, 5]     # a = 1 never forgets; tie 1/2/4 -> lowest index
    assert O.assign_heads(e, a, 8, 0.0).sum() == 0
    assert O.assign_heads(e[:6], a[:6], 8, 0.25).sum() == 1   # floor(6/4)


def test_error_energy_bounds():
    cfg = O.Cfg(d_k=64, d_v=16, g=32, bits=4, zero_point=1)
    S = RNG.standard_normal((64, 16)).astype(np.float32)
    code, scale, zp = O.quantize_state(cfg, S)
    on_grid = O.dequantize_state(cfg, code, scale, zp).astype(np.float32)
    assert O.error_energy(cfg, on_grid) == 0.0
    e = O.error_energy(cfg, S)
    direct = float(((O.dequantize_state(cfg, code, scale, zp) - S.astype(np.float64)) ** 2).sum())
    assert e == pytest.approx(direct, rel=1e-12)
    assert 0 < e <= float((np.repeat(scale, 32, axis=0).astype(np.float64) ** 2).sum()) * (0.53 ** 2)


# ------------------------------------------------------------------------------------------------
# Accounting: the numbers the pages print.

def _golden():
    with open(os.path.join(GOLDEN, "pages_numbers.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("bits,zp,g", [(4, 0, 8), (4, 1, 8), (8, 0, 4), (4, 0, 16)])
def test_value_axis_error_is_the_row_segment_quantizer(bits, zp, g):
    """Value-axis groups: brute force over every key row's g-element segments with the group quantizer."""
    dk, dv = 16, 32
    cfg = O.Cfg(d_k=dk, d_v=dv, g=g, bits=bits, zero_point=zp)
    S = (RNG.standard_normal((dk, dv)) * np.where(np.arange(dv) % 7 == 3, 8.0, 1.0)).astype(np.float32)
    e = 0.0
    for i in range(dk):
        for c0 in range(0, dv, g):
            x = S[i, c0:c0 + g]
            if zp:
                s_, z, c = O.quant_group_zp(x, bits)
                deq = np.float64(s_) * (c.astype(np.float64) - z)
            else:
                s_, c = O.quant_group_sym(x, bits)
                deq = np.float64(s_) * c.astype(np.float64)
            e += float(np.sum((deq - x.astype(np.float64)) ** 2))
    assert O.error_energy_axis(cfg, S, 1) == pytest.approx(e, rel=1e-12, abs=1e-30)
    assert O.error_energy_axis(cfg, S, 0) == O.error_energy(cfg, S)


def test_key_axis_groups_isolate_outlier_columns():
    """A state whose columns have very different magnitudes (outlier value channels): key-axis groups (one
    column each) leave the small columns at their own scale, value-axis groups mix them with the outliers."""
    dk, dv = 64, 64
    cfg = O.Cfg(d_k=dk, d_v=dv, g=32, bits=4)
    mag = np.ones(dv)
    mag[[3, 17, 40, 61]] = 8.0
    S = (RNG.standard_normal((dk, dv)) * mag[None, :]).astype(np.float32)
    ek, ev = O.error_energy_axis(cfg, S, 0), O.error_energy_axis(cfg, S, 1)
    assert ev > 2.0 * ek


def test_payload_bits_pace48_is_printed_value():
    gd = _golden()["payload_bits_pace48"]
    s = gd["setup"]
    p4 = O.payload_bits(**s["int4_heads"])
    p8 = O.payload_bits(**s["int8_heads"])
    mix = (1 - s["frac_int8"]) * p4 + s["frac_int8"] * p8
    assert Fraction(mix) == Fraction(181, 32)                  # 5.65625 exactly
    assert round(mix, gd["printed_digits"]) == gd["value"]


def test_buffer_cost_formula_reproduces_table1_pace4():
    gd = _golden()["resident_bits_table1_qwen35_27b"]
    total = O.payload_bits(4, 64, 0) + O.buffer_bits(128, 128, 8, 8, 2.0, 64, 8)
    assert Fraction(total) == Fraction(161, 32)                # 5.03125
    assert round(total, 2) == gd["PACE-4"]
    # the other two rows come out within one printed digit under the same reading (not a pin)
    mixed_buf = O.buffer_bits(128, 128, 4, 16, 2.0, 64, 8)
    assert abs(5.65625 + mixed_buf - gd["PACE-4/8"]) <= 0.0101
    assert abs(O.payload_bits(8, 32, 1) + mixed_buf - gd["DAMP INT8"]) <= 0.0101


def test_buffer_cost_scales_linearly_with_period():
    c1 = O.buffer_bits(128, 128, 8, 8, 1.0, 32, 1)
    assert Fraction(c1) == Fraction(8 * 128 + 8 * 128 + 32, 128 * 128)
    for dP in (1, 8, 32):
        assert O.buffer_bits(128, 128, 8, 8, 1.0, 32, dP) == pytest.approx(dP * c1, rel=1e-15)
