"""Parity of the CUDA decode / flush / prefill path with the oracle (GPU).

Tolerances: unquantized fp32 state <= 1e-4 relative L2; quantized-path outputs <= 1e-3 relative L2 in
the I/O precision; >= 99.9% of requantized codes identical and the rest one step apart."""
import numpy as np
import pytest

import synth
from pace_testlib import PairRun, check_bf16_state_and_sync, ensure_built, read_blob, rel_l2

pytestmark = pytest.mark.gpu

O_TOL = 1e-3
S_TOL = 1e-4
CODE_FRAC = 0.999


@pytest.fixture(scope="module")
def P():
    ensure_built()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bit_gated_delta_gb300 as P
    return P


def check_out(run, g, r, where="", tol=O_TOL):
    ok, msg = run.out_ok(g, r, tol)
    assert ok, f"{where}: {msg}"


def check_codes(run, where):
    """Codes of one rounding against the oracle's from the same starting state, then re-synchronise."""
    frac, dmax = run.check_round_and_sync()
    assert frac >= CODE_FRAC and dmax <= 1, f"{where}: {frac:.5f} identical, max diff {dmax}"
    return frac


def test_tiny_workload_full(P):
    """The tiny PACE-4 workload end to end: one 256-token chunk, then 64 decode tokens (8 roundings)."""
    wl = synth.workload("tiny")
    run = PairRun(wl)
    g, r = run.prefill(wl.prefill)
    check_out(run, g, r, "prefill")
    check_codes(run, "after prefill")
    for step in range(wl.decode):
        g, r = run.decode()
        check_out(run, g, r, f"step {step}")
        if (step + 1) % wl.dP == 0:
            check_codes(run, f"flush after step {step}")
            assert (read_blob(run.state).m() == 0).all()
        else:
            assert (read_blob(run.state).m() == (step + 1) % wl.dP).all()


@pytest.mark.parametrize("D,g,dP", [(64, 64, 8), (128, 64, 8), (128, 32, 1), (128, 64, 32), (64, 32, 3)])
def test_unquantized_mode_matches_exact_recurrence(P, D, g, dP):
    wl = synth.workload("tiny", d_k=D, d_v=D, g=g, B=2, H=3, io="f32")
    run = PairRun(wl, state_mode=P.PACE_STATE_FP32, dP=dP)
    gp, rp = run.prefill(100)
    assert rel_l2(gp, rp) <= S_TOL
    assert run.state_vs_oracle() <= S_TOL
    for step in range(2 * dP + 5):
        go, ro = run.decode()
        assert rel_l2(go, ro) <= S_TOL, f"step {step}"
    run.flush()
    assert run.state_vs_oracle() <= S_TOL


def test_unquantized_outputs_do_not_depend_on_period(P):
    import torch
    wl = synth.workload("tiny", B=2, H=2, io="f32")
    outs = {}
    for dP in (1, 4, 8, 32):
        run = PairRun(wl, state_mode=P.PACE_STATE_FP32, dP=dP, sample=[])
        run.prefill(64)
        seq = []
        for _ in range(40):
            x = synth.token_inputs(wl, run.t)
            o = torch.empty(wl.B, wl.H, wl.d_v, device="cuda")
            run.state.decode_step(*(run._dev(x[k], True) for k in ("q", "k", "v")), run._dev(x["a"], False),
                                  run._dev(x["beta"], False), o)
            run.t += 1
            seq.append(o.cpu().numpy())
        outs[dP] = np.stack(seq)
    for dP in (4, 8, 32):
        assert rel_l2(outs[dP], outs[1]) <= 1e-5


@pytest.mark.parametrize("n", [256, 100, 17, 1])
@pytest.mark.parametrize("mode", ["quant", "fp32"])
def test_prefill_chunk_sizes(P, n, mode):
    wl = synth.workload("tiny", d_k=128, d_v=128, B=2, H=2, io="bf16" if mode == "quant" else "f32")
    run = PairRun(wl, state_mode=P.PACE_STATE_QUANT if mode == "quant" else P.PACE_STATE_FP32)
    for _ in range(2):                      # two chunks: the second starts from the rounded state
        g, r = run.prefill(n)
        check_out(run, g, r, f"prefill n={n}", O_TOL if mode == "quant" else S_TOL)
        if mode == "quant":
            check_codes(run, f"prefill n={n}")
        else:
            assert run.state_vs_oracle() <= S_TOL


def test_empty_prefill_and_idle_flush_are_no_ops(P):
    import torch
    wl = synth.workload("tiny")
    run = PairRun(wl)
    run.prefill(32)
    before = run.state.region().clone()
    P.pace_prefill_chunk(run.state.handle, 0, None, None, None, None, None, None)
    run.state.flush()
    torch.cuda.synchronize()
    assert torch.equal(before, run.state.region())


def test_misaligned_io_is_rejected_before_any_launch(P):
    """q, k, v, o are read and written as 8/16-byte vectors: an unaligned pointer is an argument error, raised on
    the host; the state is untouched."""
    import torch
    wl = synth.workload("tiny")
    run = PairRun(wl)
    run.prefill(32)
    torch.cuda.synchronize()
    before = run.state.region().clone()
    B, H, D = wl.B, wl.H, wl.d_k
    buf = torch.zeros(B * H * D + 16, dtype=torch.bfloat16, device="cuda")
    a = torch.full((B, H), 0.9, device="cuda")
    ok = buf.data_ptr()
    for bad in ("q", "o"):
        ptrs = dict(q=ok, k=ok, v=ok, o=ok)
        ptrs[bad] = ok + 2                              # bf16-aligned, not vector-aligned
        with pytest.raises(P.PaceError) as ei:
            P.pace_decode_step(run.state.handle, ptrs["q"], ptrs["k"], ptrs["v"], a, a, ptrs["o"], None)
        assert ei.value.status == 1 and "aligned" in str(ei.value)
        with pytest.raises(P.PaceError):
            P.pace_prefill_chunk(run.state.handle, 1, ptrs["q"], ptrs["k"], ptrs["v"], a, a, ptrs["o"], None)
    torch.cuda.synchronize()
    assert torch.equal(before, run.state.region())


def test_pending_buffer_flush_and_prefill_after_decode(P):
    wl = synth.workload("tiny")
    run = PairRun(wl)
    run.prefill(64)
    for _ in range(3):
        g, r = run.decode()
        check_out(run, g, r)
    assert (read_blob(run.state).m() == 3).all()
    run.flush()
    assert (read_blob(run.state).m() == 0).all()
    check_codes(run, "explicit flush")
    for _ in range(5):
        run.decode()
    g, r = run.prefill(40)                  # flushes the 5 pending tokens first
    check_out(run, g, r, "prefill after decode")
    check_codes(run, "prefill after pending decode")


@pytest.mark.parametrize("dP", [1, 2, 32])
def test_decode_periods(P, dP):
    wl = synth.workload("tiny", d_k=128, d_v=128, B=1, H=3, io="bf16")
    run = PairRun(wl, dP=dP)
    run.prefill(128)
    for step in range(dP * 2 + 2):
        g, r = run.decode()
        check_out(run, g, r, f"dP={dP} step {step}")
        if (step + 1) % dP == 0:
            check_codes(run, f"dP={dP} step {step}")


def test_mixed_precision_heads_zero_point_mixed_buffer(P):
    wl = synth.workload("pace48", B=2, H=8)
    mask = np.array([0, 1, 0, 0, 1, 0, 0, 0], np.uint8)
    run = PairRun(wl, mask=mask)
    g, r = run.prefill(256)
    check_out(run, g, r, "pace48 prefill")
    check_codes(run, "pace48 prefill")
    for step in range(3 * wl.dP):
        g, r = run.decode()
        check_out(run, g, r, f"step {step}")
        if (step + 1) % wl.dP == 0:
            check_codes(run, f"pace48 step {step}")


def test_bf16_per_token_comparison_kernel(P):
    wl = synth.workload("pace4", B=2, H=4)
    run = PairRun(wl, state_mode=P.PACE_STATE_BF16)
    g, r = run.prefill(256)
    check_out(run, g, r, "bf16-state prefill")
    for step in range(32):
        g, r = run.decode()
        # bf16 rounding of the state every token: the trajectories may take different roundings
        assert rel_l2(g, r) <= 1e-2, f"step {step}"


def test_bf16_per_token_state_every_step(P):
    """The per-token bf16 comparison kernel rounds the state after every token: at every step its state is
    within one bf16 ulp of the oracle's rounding of the same update (>= 99% identical), its outputs within one
    ulp; then the oracle continues from the GPU's state."""
    wl = synth.workload("pace4", B=2, H=4)
    run = PairRun(wl, state_mode=P.PACE_STATE_BF16)
    g, r = run.prefill(256)
    check_out(run, g, r, "bf16-state prefill")
    check_bf16_state_and_sync(run, "prefill")
    for step in range(24):
        g, r = run.decode()
        check_out(run, g, r, f"step {step}")
        check_bf16_state_and_sync(run, f"step {step}")


@pytest.mark.parametrize("out_f32", [True, False])
def test_pace4_small_batch_both_output_formats(P, out_f32):
    """bf16-valued inputs: fp32 outputs meet 1e-3 relative L2; bf16 outputs are within one ulp."""
    wl = synth.workload("pace4", B=4, H=8)
    run = PairRun(wl, out_f32=out_f32)
    for _ in range(2):
        g, r = run.prefill(256)
        check_out(run, g, r, "prefill")
        check_codes(run, "prefill")
    for step in range(4 * wl.dP):
        g, r = run.decode()
        check_out(run, g, r, f"step {step}")
        if (step + 1) % wl.dP == 0:
            check_codes(run, f"step {step}")


def test_export_import_resume_is_bit_identical(P):
    import torch
    wl = synth.workload("tiny", B=2, H=2)
    a = PairRun(wl, sample=[])
    a.prefill(64)
    for _ in range(5):
        a.decode()
    host = torch.empty(a.state.layout.total_bytes, dtype=torch.uint8).pin_memory()
    P.pace_state_export(a.state.handle, host, host.numel())
    torch.cuda.synchronize()
    b = PairRun(wl, sample=[])
    b.t = a.t
    P.pace_state_import(b.state.handle, host, host.numel())
    outs = []
    for run in (a, b):
        seq = []
        for _ in range(12):
            x = synth.token_inputs(wl, run.t)
            o = torch.empty(wl.B, wl.H, wl.d_v, device="cuda")
            run.state.decode_step(*(run._dev(x[k], True) for k in ("q", "k", "v")), run._dev(x["a"], False),
                                  run._dev(x["beta"], False), o)
            run.t += 1
            seq.append(o.cpu())
        outs.append(torch.stack(seq))
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(a.state.region(), b.state.region())
