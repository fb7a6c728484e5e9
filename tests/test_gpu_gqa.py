"""Shared key heads (gamma value heads per key head): value head h reads the q and k of key head h // gamma and
one buffered copy of its key codes ([P1] 어떻게 동작하나: the buffer term b_k d_k / gamma). The arithmetic of each
value head is unchanged, so every head is checked against the oracle fed its key head's q and k, at the usual
bars: bf16 outputs within one ulp, >= 99.9% of the rounded codes identical and the rest one level apart."""
import numpy as np
import pytest

import synth
from pace_testlib import PairRun, ensure_built, read_blob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    ensure_built()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bit_gated_delta_gb300 as P
    return P


def run_periods(run, periods, where):
    wl = run.wl
    for step in range(periods * wl.dP):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"{where} step {step}: {msg}"
        if (step + 1) % wl.dP == 0:
            frac, dmax = run.check_round_and_sync()
            assert frac >= 0.999 and dmax <= 1, f"{where} step {step}: {frac:.5f} identical"


@pytest.mark.parametrize("wname,H,kh", [("pace4", 8, 4), ("pace4", 8, 2), ("pace48", 8, 4)])
def test_shared_key_heads_small_batch(P, wname, H, kh):
    """CTA-per-unit decode (few units), the tensor-core prefill, symmetric and zero-point states, int8 and mixed
    buffers."""
    wl = synth.workload(wname, B=2, H=H)
    mask = np.zeros(H, np.uint8)
    if wname == "pace48":
        mask[1] = 1
    run = PairRun(wl, key_heads=kh, mask=mask)
    g, r = run.prefill(256)
    ok, msg = run.out_ok(g, r)
    assert ok, f"prefill: {msg}"
    run.check_round_and_sync()
    run_periods(run, 2, f"{wname} H={H} Hk={kh}")


def test_shared_key_heads_warp_per_unit(P):
    """The warp-per-unit decode (B*H large), a sample of units against the oracle."""
    wl = synth.workload("pace4", B=80, H=8)
    sample = [(0, 0), (0, 3), (41, 5), (79, 7)]
    run = PairRun(wl, key_heads=4, sample=sample)
    run.prefill(256)
    run.check_round_and_sync()
    run_periods(run, 2, "B=80 H=8 Hk=4")


def test_shared_key_buffer_is_written_once_per_key_head(P):
    """The buffered key codes live in one row per key head: the layout's key array is H_k / H of the
    unshared one, and the codes equal the oracle's buffer of every value head of that key head."""
    wl = synth.workload("pace4", B=2, H=8)
    run = PairRun(wl, key_heads=2)
    run.prefill(64)
    run.check_round_and_sync()
    for _ in range(3):
        run.decode()
    L = run.state.layout
    full = PairRun(wl, sample=[]).state.layout
    assert (L.buf_v - L.buf_k) * 4 <= (full.buf_v - full.buf_k) + 1024
    raw = read_blob(run.state).raw
    bk = np.frombuffer(raw, np.int8, count=wl.B * 2 * wl.dP * wl.d_k, offset=L.buf_k).reshape(wl.B, 2, wl.dP, wl.d_k)
    for (b, h), u in run.units.items():
        assert np.array_equal(bk[b, h // 4, :u.m], u.bk[:u.m]), (b, h)
