"""Helpers shared by the tests: building the library, decoding a state region, running the GPU path
and the oracle side by side on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle as O
import synth


def ensure_built():
    from bit_gated_delta_gb300 import build as B
    B.build()
    O.build()


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)


class Blob:
    """Decoded view of a state region (bytes copied to the host), following the layout in pace.h."""

    def __init__(self, raw: np.ndarray, layout, cfg, batch: int):
        self.raw = raw
        self.L = layout
        self.cfg = cfg
        self.B = batch
        self.H = cfg.n_heads
        self.D = cfg.d_k
        self.NG = self.D // cfg.group

    def _arr(self, off, dtype, shape):
        n = int(np.prod(shape))
        return np.frombuffer(self.raw, dtype=dtype, count=n, offset=off).reshape(shape)

    def m(self):
        return self._arr(self.L.m, np.int32, (self.B, self.H))

    def scales(self):
        return bf16_bits_to_f32(self._arr(self.L.scale, np.uint16, (self.B, self.H, self.NG, self.D)))

    def zps(self):
        return self._arr(self.L.zp, np.uint8, (self.B, self.H, self.NG, self.D)).astype(np.int32)

    def word_index(self, j: np.ndarray, i: np.ndarray) -> np.ndarray:
        """Index of the word holding key i of column j in a unit's code plane (fragment order, pace.h)."""
        mt, r8, hi = j >> 4, j & 7, (j >> 3) & 1
        t, p = (i >> 1) & 3, i >> 5
        return ((mt * (self.D // 64) + (p >> 1)) * 32 + r8 * 4 + t) * 4 + hi * 2 + (p & 1)

    def codes(self, b: int, h: int) -> np.ndarray:
        """Canonical codes [d_k][d_v] of unit (b, h), as the oracle writes them."""
        D = self.D
        is8 = bool(self.L.head_is_int8[h])
        slot = self.L.head_slot[h]
        npl = D * D // 8
        if not is8:
            planes = [self._arr(self.L.codes4, np.uint32, (self.B, self.L.H4, npl))[b, slot]]
        else:
            p2 = self._arr(self.L.codes8, np.uint32, (self.B, self.L.H8, 2, npl))[b, slot]
            planes = [p2[0], p2[1]]
        i = np.arange(D)[:, None]
        j = np.arange(D)[None, :]
        wi = self.word_index(j, i)
        shift = (((i >> 3) & 3) << 2) | ((i & 1) << 4)
        out = ((planes[0][wi] >> shift) & 0xF).astype(np.int32)
        if is8:
            out |= (((planes[1][wi] >> shift) & 0xF).astype(np.int32) << 4)
        off = 128 if is8 else 8
        return out if self.cfg.zero_point else out - off

    def buffer(self, b: int, h: int):
        """(key codes [dP, D], value codes or values [dP, D], scalars [dP, 4]) of unit (b, h)."""
        D, P = self.D, self.cfg.dP
        s = self._arr(self.L.buf_s, np.float32, (self.B, self.H, P, 4))[b, h]
        if self.cfg.buf_mode == 1:
            kb = self._arr(self.L.buf_k, np.uint8, (self.B, self.H, P, D // 2))[b, h]
            k = np.zeros((P, D), np.int32)
            k[:, 0::2] = (kb & 0xF).astype(np.int32) - 8
            k[:, 1::2] = (kb >> 4).astype(np.int32) - 8
            v = bf16_bits_to_f32(self._arr(self.L.buf_v, np.uint16, (self.B, self.H, P, D))[b, h])
        elif self.cfg.buf_mode == 2:
            k = self._arr(self.L.buf_k, np.float32, (self.B, self.H, P, D))[b, h]
            v = self._arr(self.L.buf_v, np.float32, (self.B, self.H, P, D))[b, h]
        else:
            k = self._arr(self.L.buf_k, np.int8, (self.B, self.H, P, D))[b, h].astype(np.int32)
            v = self._arr(self.L.buf_v, np.int8, (self.B, self.H, P, D))[b, h].astype(np.int32)
        return k, v, s


def read_blob(state) -> Blob:
    import torch
    torch.cuda.synchronize()
    raw = state.region().cpu().numpy().tobytes()
    return Blob(np.frombuffer(raw, np.uint8), state.layout, state.cfg, state.batch)


def oracle_cfg(wl: synth.Workload, bits: int = 4, state_mode: int = O.STATE_QUANT) -> O.Cfg:
    if state_mode == O.STATE_QUANT:
        buf = O.BUF_MIXED if wl.mixed_buffer else O.BUF_INT8
    elif state_mode == O.STATE_BF16_BUF:
        buf = O.BUF_INT8                             # the library keeps this mode's buffer in int8
    else:
        buf = O.BUF_FP32
    return O.Cfg(d_k=wl.d_k, d_v=wl.d_v, g=wl.g, bits=bits, zero_point=wl.zero_point, dP=wl.dP, buf_mode=buf,
                 state_mode=state_mode)


def rel_l2(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def bf16_within_ulp(got, ref):
    """Each element is within one bf16 ulp of the exact value, plus an fp32-arithmetic floor of 1e-5 of the
    largest magnitude in its output vector (an element that cancels to near zero carries the fp32 rounding
    of its terms, which exceeds the ulp of its own tiny value)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    mag = np.maximum(np.abs(ref), 1e-30)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    floor = 1e-5 * np.abs(ref).max(axis=-1, keepdims=True)
    bad = np.abs(got - ref) > ulp * (1 + 1e-6) + floor
    return (not bad.any()), f"{int(bad.sum())} elements more than one bf16 ulp away (max rel {np.max(np.abs(got - ref) / mag):.2e})"


def bf16_rn(x) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), from the float32 image of x."""
    b = np.ascontiguousarray(np.asarray(x, np.float32)).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32)


def bf16_outputs_ok(got, ref, min_exact: float = 0.99):
    """bf16 outputs: every element within one bf16 ulp of the exact value (bf16_within_ulp), and at least
    `min_exact` of them equal to the bf16 rounding of the oracle's value: the kernel rounds an fp32 value
    that differs from the oracle's fp64 one by the path's arithmetic error, so only elements that close to a
    bf16 rounding tie may take the other neighbour."""
    ok, msg = bf16_within_ulp(got, ref)
    same = float(np.mean(np.asarray(got, np.float32) == bf16_rn(ref)))
    return ok and same >= min_exact, f"{msg}; {same:.5f} equal to bf16(oracle)"


def check_bf16_state_and_sync(run, where):
    """bf16 states (per-token and buffered modes): every element within one bf16 ulp of the oracle's bf16
    rounding of the same values, with an fp32-arithmetic floor of 2^-16 of the unit's largest element (near-zero
    elements), and >= 99% identical; then the oracle continues from the GPU's state."""
    S = run.gpu_state()
    keys = list(run.units)                         # the sampled units (default: all)
    got = np.stack([S[b, h] for (b, h) in keys])
    ref = np.stack([run.units[k].S for k in keys])
    same = np.mean(got == ref.astype(np.float32))
    floor = 2.0 ** -16 * np.abs(ref).max(axis=(1, 2), keepdims=True)
    ulp = np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + floor
    assert same >= 0.99 and ulp.all(), f"{where}: {same:.5f} identical, {np.mean(~ulp):.2e} beyond one ulp"
    run.sync_state_from_gpu()


def code_agreement(gpu_codes: np.ndarray, ref_codes: np.ndarray):
    """(fraction identical, max |difference|)."""
    d = np.abs(gpu_codes.astype(np.int64) - ref_codes.astype(np.int64))
    return float((d == 0).mean()), int(d.max())


class RoundCheck:
    """Agreement of one rounding with the oracle's. The bar: >= 99.9% of levels identical and the rest one step
    apart (R17: fp32 and fp64 arithmetic may round a near-tie differently); >= 99.9% of the bf16 scales
    bit-identical and the rest one bf16 ulp apart (the group maximum sits near a bf16 rounding tie); every
    group the oracle rounds to zero is zero on the GPU too; zero points >= 99.9% identical, the rest one
    apart."""

    FRAC = 0.999

    def __init__(self, code_frac, code_dmax, scale_frac, scale_ulp, zero_exact, zp_frac, zp_dmax):
        self.code_frac, self.code_dmax = code_frac, code_dmax
        self.scale_frac, self.scale_ulp = scale_frac, scale_ulp
        self.zero_exact = zero_exact
        self.zp_frac, self.zp_dmax = zp_frac, zp_dmax

    def ok(self) -> bool:
        return (self.code_frac >= self.FRAC and self.code_dmax <= 1 and self.scale_frac >= self.FRAC
                and self.scale_ulp <= 1 and self.zero_exact and self.zp_frac >= self.FRAC and self.zp_dmax <= 1)

    def __iter__(self):
        return iter((self.code_frac, self.code_dmax))

    def __repr__(self):
        return (f"levels {self.code_frac:.5f} identical (max diff {self.code_dmax}); scales {self.scale_frac:.5f} "
                f"identical (max {self.scale_ulp} ulp); zero groups exact: {self.zero_exact}; zero points "
                f"{self.zp_frac:.5f} identical (max diff {self.zp_dmax})")


class PairRun:
    """Runs the CUDA path (through the C ABI) and the oracle on the same seeded workload inputs.

    The GPU processes every unit; the oracle the units listed in `sample` ((b, h) pairs, default all).
    Outputs are compared in the I/O precision: with bf16 I/O the oracle's output is rounded to bf16
    (the same rounding decision the kernel takes), so the comparison measures the path, not the format.
    """

    def __init__(self, wl: synth.Workload, state_mode: int = 0, mask=None, sample=None, dP=None, layer=0,
                 out_f32: bool = False, key_heads: int = 0):
        import torch
        import bit_gated_delta_gb300 as P
        self.P, self.torch = P, torch
        if dP is not None:
            wl = wl.with_(dP=dP)
        self.wl = wl
        self.layer = layer
        self.mask = np.zeros(wl.H, np.uint8) if mask is None else np.asarray(mask, np.uint8)
        if state_mode == P.PACE_STATE_QUANT:
            buf = P.PACE_BUF_MIXED if wl.mixed_buffer else P.PACE_BUF_INT8
        elif state_mode == P.PACE_STATE_FP32:
            buf = P.PACE_BUF_FP32
        else:
            buf = P.PACE_BUF_INT8
        # out_f32: run the (bf16-valued) workload through the library with fp32 I/O, so the outputs show the
        # path's arithmetic without the final bf16 rounding
        self.io_bf16 = wl.io == "bf16" and not out_f32
        self.cfg = P.make_config(wl.H, wl.d_k, wl.B, dP=wl.dP, group=wl.g, zero_point=wl.zero_point, buf_mode=buf,
                                 state_mode=state_mode,
                                 io_dtype=P.PACE_IO_BF16 if self.io_bf16 else P.PACE_IO_F32, key_heads=key_heads)
        # shared key heads: value head h reads the q and k of key head h // gamma (here: of value head
        # gamma * (h // gamma)); the library gets the [B, H_k, ...] tensors, the oracle each head's copy
        self.gamma = wl.H // key_heads if key_heads else 1
        self.state = P.PaceState(self.cfg, wl.B, self.mask if state_mode == 0 else None)
        self.sample = sample if sample is not None else [(b, h) for b in range(wl.B) for h in range(wl.H)]
        om = {0: O.STATE_QUANT, 1: O.STATE_FP32, 2: O.STATE_BF16, 3: O.STATE_BF16_BUF}[state_mode]
        self.units = {}
        for (b, h) in self.sample:
            c = oracle_cfg(wl, bits=8 if self.mask[h] else 4, state_mode=om)
            if om == O.STATE_BF16:
                c.buf_mode = O.BUF_FP32
            self.units[(b, h)] = O.Unit(c)
        self.t = 0

    def _dev(self, x: np.ndarray, io: bool):
        t = self.torch.from_numpy(np.ascontiguousarray(x)).cuda()
        return t.to(self.torch.bfloat16) if (io and self.io_bf16) else t

    def _ref_out(self, ref: np.ndarray) -> np.ndarray:
        return ref

    def out_ok(self, got, ref, tol: float = 1e-3):
        """fp32 outputs: relative L2 <= tol. bf16 outputs: each element is one of the two bf16 neighbours of
        the oracle's value (within one bf16 ulp), since near-ties may round either way, and >= 99% of them
        equal the bf16 rounding of the oracle's value (bf16_outputs_ok)."""
        if not self.io_bf16:
            e = rel_l2(got, ref)
            return e <= tol, f"rel_l2 {e:.3e}"
        return bf16_outputs_ok(got, ref)

    def _share_keys(self, x):
        if self.gamma == 1:
            return x, x["q"], x["k"]
        x = dict(x)
        for key in ("q", "k"):
            x[key] = np.repeat(x[key][:, ::self.gamma], self.gamma, axis=1)
        return x, np.ascontiguousarray(x["q"][:, ::self.gamma]), np.ascontiguousarray(x["k"][:, ::self.gamma])

    def prefill(self, n: int, inputs=None):
        wl = self.wl
        x = inputs if inputs is not None else synth.chunk_inputs(wl, self.t, n, self.layer)
        x, qg, kg = self._share_keys(x)
        o = self.torch.empty(wl.B, wl.H, n, wl.d_v, device="cuda",
                             dtype=self.torch.bfloat16 if self.io_bf16 else self.torch.float32)
        self.state.prefill_chunk(self._dev(qg, True), self._dev(kg, True), self._dev(x["v"], True),
                                 self._dev(x["a"], False), self._dev(x["beta"], False), o)
        got = o.float().cpu().numpy()
        refs, gots = [], []
        for (b, h), u in self.units.items():
            r = O.prefill(u, x["q"][b, h], x["k"][b, h], x["v"][b, h], x["a"][b, h], x["beta"][b, h])
            refs.append(self._ref_out(r))
            gots.append(got[b, h])
        self.t += n
        self.last = got
        return (np.stack(gots), np.stack(refs)) if refs else (got, None)

    def decode(self, inputs=None, gpu_call=None):
        """One decode step on both sides. gpu_call(q, k, v, a, beta, o), if given, runs the GPU step in place of
        a direct pace_decode_step call (e.g. the replay of a captured CUDA graph)."""
        wl = self.wl
        x = inputs if inputs is not None else synth.token_inputs(wl, self.t, self.layer)
        x, qg, kg = self._share_keys(x)
        o = self.torch.empty(wl.B, wl.H, wl.d_v, device="cuda",
                             dtype=self.torch.bfloat16 if self.io_bf16 else self.torch.float32)
        args = (self._dev(qg, True), self._dev(kg, True), self._dev(x["v"], True), self._dev(x["a"], False),
                self._dev(x["beta"], False), o)
        if gpu_call is None:
            self.state.decode_step(*args)
        else:
            gpu_call(*args)
        got = o.float().cpu().numpy()
        refs, gots = [], []
        for (b, h), u in self.units.items():
            r = O.decode_step(u, x["q"][b, h], x["k"][b, h], x["v"][b, h], x["a"][b, h], x["beta"][b, h])
            refs.append(self._ref_out(r))
            gots.append(got[b, h])
        self.t += 1
        self.last = got
        return (np.stack(gots), np.stack(refs)) if refs else (got, None)

    def flush(self):
        self.state.flush()
        for u in self.units.values():
            O.flush(u)

    def blob(self) -> Blob:
        return read_blob(self.state)

    def codes_vs_oracle(self):
        """(fraction of identical quantization levels, max |difference|) over the sampled units. The level is
        the code itself for symmetric groups and code - zero point for zero-point groups: a near-tie that
        flips a zero-point scale may move the stored code and the zero point together, while the represented
        level moves by at most one step."""
        r = self.round_vs_oracle()
        return r.code_frac, r.code_dmax

    def round_vs_oracle(self) -> "RoundCheck":
        """Everything a rounding writes, against the oracle's rounding of the same period: the levels (as in
        codes_vs_oracle), the bf16 group scales (bit patterns) and the zero points ([P1] 무엇과 다른가: the
        scale and, for PACE-4/8, the integer zero point are part of the code assignment)."""
        blob = self.blob()
        sc = blob.scales()
        zps = blob.zps() if self.wl.zero_point else None
        gl, rl, gs, rs, gz, rz = [], [], [], [], [], []
        for (b, h), u in self.units.items():
            gc, rc = blob.codes(b, h), u.code
            if zps is not None:
                gc = gc - np.repeat(zps[b, h], self.wl.g, axis=0)
                rc = rc - np.repeat(u.zp, self.wl.g, axis=0)
                gz.append(zps[b, h])
                rz.append(u.zp)
            gl.append(gc)
            rl.append(rc)
            gs.append(sc[b, h])
            rs.append(u.scale)
        if not gl:
            return RoundCheck(1.0, 0, 1.0, 0, True, 1.0, 0)
        code_frac, code_dmax = code_agreement(np.stack(gl), np.stack(rl))
        g_s = np.ascontiguousarray(np.stack(gs), np.float32)
        r_s = np.ascontiguousarray(np.stack(rs), np.float32)
        gb = (g_s.view(np.uint32) >> 16).astype(np.int64)
        rb = (r_s.view(np.uint32) >> 16).astype(np.int64)
        zero_exact = bool(np.all(g_s[r_s == 0] == 0))
        scale_frac = float((gb == rb).mean())
        scale_ulp = int(np.abs(gb - rb).max())
        zp_frac, zp_dmax = (1.0, 0) if not gz else code_agreement(np.stack(gz), np.stack(rz))
        return RoundCheck(code_frac, code_dmax, scale_frac, scale_ulp, zero_exact, zp_frac, zp_dmax)

    def gpu_state(self) -> np.ndarray:
        """The resident state of every unit as fp32 [B, H, d_k, d_v] (fp32 and bf16 modes)."""
        out = self.torch.empty(self.wl.B, self.wl.H, self.wl.d_k, self.wl.d_v, device="cuda")
        self.P.pace_dequantize_state(self.state.handle, out)
        return out.cpu().numpy()

    def sync_state_from_gpu(self):
        """Teacher forcing for the fp32 / bf16 modes: the oracle continues from the GPU's resident state."""
        S = self.gpu_state().astype(np.float64)
        for (b, h), u in self.units.items():
            u.S[...] = S[b, h]

    def state_vs_oracle(self) -> float:
        """Relative L2 distance of the resident states (fp32 / bf16 modes)."""
        out = self.torch.empty(self.wl.B, self.wl.H, self.wl.d_k, self.wl.d_v, device="cuda")
        self.P.pace_dequantize_state(self.state.handle, out)
        S = out.cpu().numpy()
        return rel_l2(np.stack([S[b, h] for (b, h) in self.units]), np.stack([u.S for u in self.units.values()]))

    def check_round_and_sync(self, where: str = "") -> "RoundCheck":
        """At a rounding: compare the GPU's levels, scales and zero points with the oracle's (both rounded from
        the same starting state of this period) and assert the bar, then hand the GPU's rounded state to the
        oracle for the next period. Returns the comparison."""
        res = self.round_vs_oracle()
        assert res.ok(), f"{where}: {res}"
        self.sync_oracle_from_gpu()
        return res

    def sync_oracle_from_gpu(self):
        """Teacher forcing: copy the GPU's resident quantized state into the oracle units."""
        blob = self.blob()
        sc = blob.scales()
        zps = blob.zps() if self.wl.zero_point else None
        for (b, h), u in self.units.items():
            u.code[...] = blob.codes(b, h)
            u.scale[...] = sc[b, h]
            if zps is not None:
                u.zp[...] = zps[b, h]
