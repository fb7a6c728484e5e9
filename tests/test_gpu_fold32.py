"""Parity of the folded-readout decode kernel with 32-token tables (int4 symmetric state, g = 64, int8 decode
buffer, every head at 4 bits, rounding periods of 9 to 32 tokens) with the oracle (GPU).

The buffered tokens are replayed through one unit lower-triangular system per unit ([P1] 어떻게 동작하나: the
buffer is applied to the state together at the rounding); the tables hold up to 32 tokens, the rounding passes
over the state once per group of 8. Bars as for the 8-token kernel: outputs within 1e-3 per rounding period (one
bf16 ulp with bf16 I/O), and at every rounding the levels, bf16 scale bits and zero groups against the oracle's."""
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


@pytest.mark.parametrize("D,dP", [(128, 32), (128, 9), (128, 16), (64, 32), (64, 12)])
def test_periods_of_9_to_32_tokens(P, D, dP):
    # 32 units: at d = 64 that is 2,048 group scales per rounding, enough for the 99.9% bar to mean something
    wl = synth.workload("pace4", B=4, H=8, d_k=D, d_v=D)
    run = PairRun(wl, dP=dP)
    g, r = run.prefill(256)
    ok, msg = run.out_ok(g, r)
    assert ok, f"prefill: {msg}"
    run.check_round_and_sync("prefill")
    for step in range(2 * dP + 3):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"D={D} dP={dP} step {step}: {msg}"
        assert (read_blob(run.state).m() == (step + 1) % dP).all()
        if (step + 1) % dP == 0:
            run.check_round_and_sync(f"D={D} dP={dP} step {step}")


def test_explicit_flush_and_prefill_after_pending_tokens(P):
    """A flush with 13 pending tokens (two token groups, the second partial, no new token), then a prefill chunk
    after 5 pending tokens (applied first)."""
    wl = synth.workload("pace4", B=2, H=4)
    run = PairRun(wl, dP=32)
    run.prefill(256)
    run.check_round_and_sync("prefill")
    for step in range(13):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"step {step}: {msg}"
    run.flush()
    assert (read_blob(run.state).m() == 0).all()
    run.check_round_and_sync("explicit flush of 13 tokens")
    for _ in range(5):
        run.decode()
    g, r = run.prefill(100)
    ok, msg = run.out_ok(g, r)
    assert ok, f"prefill after 5 pending tokens: {msg}"
    run.check_round_and_sync("prefill after pending decode")


def test_shared_key_heads(P):
    """Two value heads per key head (one buffered key row per key head) with 32-token tables."""
    wl = synth.workload("pace4", B=4, H=8)
    run = PairRun(wl, dP=24, key_heads=4)
    g, r = run.prefill(256)
    ok, msg = run.out_ok(g, r)
    assert ok, f"prefill: {msg}"
    run.check_round_and_sync("prefill")
    for step in range(2 * 24 + 2):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"step {step}: {msg}"
        if (step + 1) % 24 == 0:
            run.check_round_and_sync(f"step {step}")
