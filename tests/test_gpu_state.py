"""Bit-exact checks of the packed state and decode-buffer formats against the oracle (GPU).

Fed the same fp32 values, code assignment, packing and unpacking must agree bit for bit."""
import numpy as np
import pytest

import oracle as O
from pace_testlib import bf16_bits_to_f32, ensure_built, read_blob, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    ensure_built()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bit_gated_delta_gb300 as P
    return P


def column_outlier_states(rng, B, H, D, scale=1.0):
    S = rng.standard_normal((B, H, D, D)).astype(np.float32) * np.float32(scale)
    for b in range(B):
        for h in range(H):
            cols = rng.choice(D, 4, replace=False)
            S[b, h][:, cols] *= 8.0
    S[0, 0, :, 3] = 0.0                                 # an all-zero column: zero scales
    S[0, 0, 5, 7] = 1e3                                 # a single large outlier
    S[-1, -1, :, 1] = 0.25                              # a constant column
    return S


@pytest.mark.parametrize("D,g,zp,n8", [(128, 64, 0, 0), (128, 32, 0, 0), (128, 32, 1, 8), (64, 64, 0, 0),
                                       (64, 32, 1, 2), (128, 64, 0, 4), (128, 32, 1, 32)])
def test_quantize_state_is_bit_exact(P, D, g, zp, n8):
    import torch
    rng = np.random.default_rng(D + g + zp + n8)
    B, H = 3, max(8, n8)
    mask = np.zeros(H, np.uint8)
    mask[rng.choice(H, n8, replace=False)] = 1
    cfg = P.make_config(H, D, B, group=g, zero_point=zp)
    st = P.PaceState(cfg, B, mask)
    S = column_outlier_states(rng, B, H, D)
    Sd = torch.from_numpy(S).cuda()
    P.pace_quantize_state(st.handle, Sd)
    blob = read_blob(st)
    out = torch.empty_like(Sd)
    P.pace_dequantize_state(st.handle, out)
    deq = out.cpu().numpy()
    for b in range(B):
        for h in range(H):
            bits = 8 if mask[h] else 4
            ocfg = O.Cfg(d_k=D, d_v=D, g=g, bits=bits, zero_point=zp)
            code, scale, zpt = O.quantize_state(ocfg, S[b, h])
            assert np.array_equal(blob.codes(b, h), code), (b, h)
            assert np.array_equal(blob.scales()[b, h].view(np.uint32), scale.view(np.uint32)), (b, h)
            if zp:
                assert np.array_equal(blob.zps()[b, h], zpt), (b, h)
            ref = O.dequantize_state(ocfg, code, scale, zpt)
            assert np.array_equal(deq[b, h].astype(np.float64), ref), (b, h)
    assert (blob.m() == 0).all()


@pytest.mark.parametrize("mixed", [False, True])
def test_buffer_codes_are_bit_exact(P, mixed):
    import torch
    rng = np.random.default_rng(11 + mixed)
    B, H, D, dP = 2, 4, 128, 8
    cfg = P.make_config(H, D, B, dP=dP, group=32 if mixed else 64, zero_point=int(mixed),
                        buf_mode=P.PACE_BUF_MIXED if mixed else P.PACE_BUF_INT8)
    st = P.PaceState(cfg, B)
    ks, vs, av, bv = [], [], [], []
    for t in range(3):
        k = rng.standard_normal((B, H, D)).astype(np.float32)
        v = rng.standard_normal((B, H, D)).astype(np.float32) * 3
        if t == 1:
            k[0, 0] = 0.0                               # zero vector: zero codes, zero scale
        q = rng.standard_normal((B, H, D)).astype(np.float32)
        k, v, q = (torch.from_numpy(x).to(torch.bfloat16) for x in (k, v, q))
        a = torch.from_numpy(rng.uniform(0.9, 1.0, (B, H)).astype(np.float32))
        be = torch.from_numpy(rng.uniform(0, 1, (B, H)).astype(np.float32))
        o = torch.empty(B, H, D, dtype=torch.bfloat16, device="cuda")
        st.decode_step(q.cuda(), k.cuda(), v.cuda(), a.cuda(), be.cuda(), o)
        ks.append(k.float().numpy()), vs.append(v.float().numpy()), av.append(a.numpy()), bv.append(be.numpy())
    blob = read_blob(st)
    assert (blob.m() == 3).all()
    for b in range(B):
        for h in range(H):
            kc, vc, sc = blob.buffer(b, h)
            for t in range(3):
                rk, rsk = O.buffer_quant(ks[t][b, h], 7 if mixed else 127)
                assert np.array_equal(kc[t], rk) and sc[t, 2] == rsk
                assert sc[t, 0] == av[t][b, h] and sc[t, 1] == bv[t][b, h]
                if mixed:
                    assert np.array_equal(vc[t], O.bf16_rn(vs[t][b, h]))
                else:
                    rv, rsv = O.buffer_quant(vs[t][b, h], 127)
                    assert np.array_equal(vc[t], rv) and sc[t, 3] == rsv


@pytest.mark.parametrize("bits,g,zp", [(4, 64, 0), (4, 32, 1), (8, 32, 1)])
def test_calibration_error_energy(P, bits, g, zp):
    import torch
    rng = np.random.default_rng(bits * 100 + g)
    B, H, D = 2, 6, 128
    cfg = P.make_config(H, D, B, group=64, state_mode=P.PACE_STATE_FP32, buf_mode=P.PACE_BUF_FP32)
    st = P.PaceState(cfg, B)
    S = column_outlier_states(rng, B, H, D, 0.1)
    P.pace_quantize_state(st.handle, torch.from_numpy(S).cuda())
    e = torch.zeros(B * H, device="cuda")
    P.pace_calib_error_energy(st.handle, bits, g, zp, e)
    got = e.cpu().numpy()
    ocfg = O.Cfg(d_k=D, d_v=D, g=g, bits=bits, zero_point=zp)
    ref = np.array([O.error_energy(ocfg, S[b, h]) for b in range(B) for h in range(H)])
    np.testing.assert_allclose(got, ref, rtol=1e-4)


@pytest.mark.parametrize("bits,g,zp", [(4, 64, 0), (4, 32, 1), (8, 32, 0)])
def test_value_axis_error_energy(P, bits, g, zp):
    """The baseline grouping (g consecutive elements along the value axis of a key row) against the oracle, and
    on column-outlier states its error is above PACE's key-axis grouping (in total and for most units)."""
    import torch
    rng = np.random.default_rng(bits * 1000 + g + zp)
    B, H, D = 2, 6, 128
    cfg = P.make_config(H, D, B, group=64, state_mode=P.PACE_STATE_FP32, buf_mode=P.PACE_BUF_FP32)
    st = P.PaceState(cfg, B)
    S = column_outlier_states(rng, B, H, D, 0.1)
    P.pace_quantize_state(st.handle, torch.from_numpy(S).cuda())
    ev = torch.zeros(B * H, device="cuda")
    ek = torch.zeros(B * H, device="cuda")
    P.pace_calib_error_energy_axis(st.handle, bits, g, zp, 1, ev)
    P.pace_calib_error_energy_axis(st.handle, bits, g, zp, 0, ek)
    ocfg = O.Cfg(d_k=D, d_v=D, g=g, bits=bits, zero_point=zp)
    ref = np.array([O.error_energy_axis(ocfg, S[b, h], 1) for b in range(B) for h in range(H)])
    np.testing.assert_allclose(ev.cpu().numpy(), ref, rtol=1e-4)
    ev, ek = ev.cpu().numpy(), ek.cpu().numpy()
    assert ev.sum() > 1.2 * ek.sum() and np.mean(ev > ek) >= 0.75


def test_fresh_state_is_zero(P):
    import torch
    for zp in (0, 1):
        mask = np.array([0, 1, 0, 1], np.uint8)
        cfg = P.make_config(4, 64, 2, group=32, zero_point=zp)
        st = P.PaceState(cfg, 2, mask)
        out = torch.full((2, 4, 64, 64), 7.0, device="cuda")
        P.pace_dequantize_state(st.handle, out)
        assert float(out.abs().max()) == 0.0
        blob = read_blob(st)
        assert all((blob.codes(b, h) == 0).all() for b in range(2) for h in range(4))
