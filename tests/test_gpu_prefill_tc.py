"""Parity of the tensor-core chunk prefill (d_k = d_v = 128, bf16 I/O) with the oracle's token-by-token prefill.

The kernel walks a chunk in 32-token sub-chunks with the state in tensor memory; these cases cover whole and
partial sub-chunks, one- and several-sub-chunk chunks, every state format and both decay ranges. The bars are the
ones of the decode path: unquantized fp32 state <= 1e-4 relative L2; bf16 outputs within one bf16 ulp of the
oracle's value; >= 99.9% of the rounded codes identical and the rest one level apart."""
import numpy as np
import pytest

import synth
from pace_testlib import PairRun, ensure_built, rel_l2

pytestmark = pytest.mark.gpu

S_TOL = 1e-4


@pytest.fixture(scope="module")
def P():
    ensure_built()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bit_gated_delta_gb300 as P
    return P


@pytest.mark.parametrize("n", [256, 100, 33, 32, 1])
@pytest.mark.parametrize("decay", ["fast", "slow"])
def test_fp32_state_prefill_matches_recurrence(P, n, decay):
    """Unquantized state, bf16 inputs: the chunk form equals the token loop to 1e-4 (state and outputs)."""
    kw = dict(a_lo=0.5, a_hi=0.9) if decay == "fast" else dict(a_lo=0.99, a_hi=0.9999)
    wl = synth.workload("pace4", B=2, H=3, **kw)
    run = PairRun(wl, state_mode=P.PACE_STATE_FP32)
    for c in range(3):                        # three chunks: each starts from the previous chunk's state
        g, r = run.prefill(n)
        ok, msg = run.out_ok(g, r)
        assert ok, f"chunk {c} n={n}: {msg}"
        e = run.state_vs_oracle()
        assert e <= S_TOL, f"chunk {c} n={n}: state rel_l2 {e:.3e}"


@pytest.mark.parametrize("g,zp,n8", [(64, 0, 0), (32, 1, 0), (32, 1, 2), (64, 0, 1)])
def test_quantized_prefill_rounds_once(P, g, zp, n8):
    """Quantized state (int4 heads, and int8 heads when n8 > 0): outputs within one bf16 ulp and the chunk-end
    codes agree with the oracle's rounding of the same chunk."""
    wl = synth.workload("pace4", B=2, H=4, g=g, zero_point=zp)
    mask = np.zeros(wl.H, np.uint8)
    mask[:n8] = 1
    run = PairRun(wl, mask=mask)
    for c, n in enumerate((256, 77, 256)):
        gg, r = run.prefill(n)
        ok, msg = run.out_ok(gg, r)
        assert ok, f"chunk {c}: {msg}"
        frac, dmax = run.check_round_and_sync()
        assert frac >= 0.999 and dmax <= 1, f"chunk {c}: {frac:.5f} identical, max diff {dmax}"
        assert (run.blob().m() == 0).all()


def test_bf16_state_prefill(P):
    """Per-token comparison mode: the chunk-end state is rounded to bf16 once; outputs within one ulp. Near a bf16
    tie the two sides may round one element differently (the fp32 chunk form and the fp64 loop differ by ~1e-6),
    so, as at every rounding of the quantized state, the oracle continues from the GPU's rounded state."""
    import torch
    wl = synth.workload("pace4", B=2, H=2)
    run = PairRun(wl, state_mode=P.PACE_STATE_BF16)
    for c in range(2):
        g, r = run.prefill(256)
        ok, msg = run.out_ok(g, r)
        assert ok, f"chunk {c}: {msg}"
        assert run.state_vs_oracle() <= 4e-3      # one bf16 rounding of the state
        out = torch.empty(wl.B, wl.H, wl.d_k, wl.d_v, device="cuda")
        P.pace_dequantize_state(run.state.handle, out)
        S = out.cpu().numpy().astype(np.float64)
        for (b, h), u in run.units.items():
            u.S[...] = S[b, h]


def test_prefill_then_decode_continues(P):
    """Decode after the tensor-core prefill: outputs within one bf16 ulp through two rounding periods."""
    wl = synth.workload("pace4", B=2, H=4)
    run = PairRun(wl)
    g, r = run.prefill(256)
    assert run.out_ok(g, r)[0]
    run.check_round_and_sync()
    for step in range(2 * wl.dP):
        g, r = run.decode()
        ok, msg = run.out_ok(g, r)
        assert ok, f"step {step}: {msg}"
        if (step + 1) % wl.dP == 0:
            frac, dmax = run.check_round_and_sync()
            assert frac >= 0.999 and dmax <= 1
    assert rel_l2(g, r) <= 1e-2
