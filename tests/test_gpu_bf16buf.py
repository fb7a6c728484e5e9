"""Parity of the buffered bf16-state mode (bf16 state rounded once every dP tokens, int8 decode buffer) with
the oracle (GPU). This is the decode buffer without the 4-bit state, the decomposition the pages use for the
TPOT gain of periodic rounding ([P1] 전제와 한계).

Bars: bf16 outputs within one bf16 ulp of the oracle's value. At each rounding every bf16 state element is
within one bf16 ulp of the oracle's bf16 rounding of the same replay, with an fp32-arithmetic floor of 2^-16 of
the unit's largest element (near-zero elements), and >= 99% are identical: the rounding decision is taken on
fp32 values that differ from the oracle's fp64 ones by the path's arithmetic error (about 1e-6 relative for the
tensor-core prefill), and a bf16 ulp is 2^-8 relative, so values that close to a tie may round to the other
neighbour. Then the oracle continues from the GPU's state, as at every rounding of the quantized state."""
import numpy as np
import pytest

import synth
from pace_testlib import PairRun, check_bf16_state_and_sync, ensure_built, read_blob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    ensure_built()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bit_gated_delta_gb300 as P
    return P


def check_state_and_sync(run, where):
    check_bf16_state_and_sync(run, where)


@pytest.mark.parametrize("dP", [8, 1, 3, 32])
def test_decode_rounds_to_bf16_once_per_period(P, dP):
    wl = synth.workload("pace4", B=2, H=4)
    run = PairRun(wl, state_mode=P.PACE_STATE_BF16_BUF, dP=dP)
    g, r = run.prefill(256)
    ok, msg = run.out_ok(g, r)
    assert ok, f"prefill: {msg}"
    check_state_and_sync(run, "prefill")
    for step in range(2 * dP + 3):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"dP={dP} step {step}: {msg}"
        m = read_blob(run.state).m()
        assert (m == (step + 1) % dP).all()
        if (step + 1) % dP == 0:
            check_state_and_sync(run, f"dP={dP} step {step}")


def test_pending_buffer_flush_then_prefill(P):
    wl = synth.workload("pace4", B=2, H=2)
    run = PairRun(wl, state_mode=P.PACE_STATE_BF16_BUF)
    run.prefill(256)
    run.sync_state_from_gpu()
    for _ in range(5):
        g, r = run.decode()
        assert run.out_ok(g, r)[0]
    run.flush()
    assert (read_blob(run.state).m() == 0).all()
    check_state_and_sync(run, "explicit flush")
    for _ in range(3):
        run.decode()
    g, r = run.prefill(100)                      # the pending buffer is applied first
    ok, msg = run.out_ok(g, r)
    assert ok, f"prefill after decode: {msg}"


def test_small_head_dim_fp32_io(P):
    """d = 64 with fp32 I/O (per-token prefill kernel, fp32 outputs at the 1e-3 bar)."""
    wl = synth.workload("tiny", B=2, H=2, io="f32")
    run = PairRun(wl, state_mode=P.PACE_STATE_BF16_BUF)
    run.prefill(64)
    run.sync_state_from_gpu()
    for step in range(2 * wl.dP):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"step {step}: {msg}"
        if (step + 1) % wl.dP == 0:
            check_state_and_sync(run, f"step {step}")


@pytest.mark.parametrize("B", [24, 64])
def test_launch_shapes_at_32_heads(P, B):
    """d = 128, 32 heads: B = 24 runs two warps per unit, B = 64 (the bench configuration) one warp per unit and
    16 units per SM; 8 sampled units against the oracle over two periods."""
    wl = synth.workload("pace4", B=B)
    sample = [(b, h) for b, h in ((0, 0), (1, 31), (B // 2, 7), (B - 1, 16), (3, 3), (B - 2, 30), (5, 12), (B - 3, 1))]
    run = PairRun(wl, state_mode=P.PACE_STATE_BF16_BUF, sample=sample)
    run.prefill(256)
    check_state_and_sync(run, "prefill")
    for step in range(2 * wl.dP):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"B={B} step {step}: {msg}"
        if (step + 1) % wl.dP == 0:
            check_state_and_sync(run, f"B={B} step {step}")
