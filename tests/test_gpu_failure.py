"""Failure detection without a GPU fault (GPU).

* A bounded device wait that runs out: the failure-detection probe of the tensor-core prefill waits on an
  mbarrier that nothing signals, gives up after a short limit, and the host reads PACE_ERR_TIMEOUT from the
  status word; the units and their outputs are unchanged, no MMA was issued, and the context stays usable (the
  same chunk then runs normally and matches the oracle).
* A unit whose buffer counter is out of range (a corrupted region, built on the host and imported) is left
  unchanged and its output is zero; every other unit decodes exactly as before."""
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


def _region_without_status(run):
    import torch
    torch.cuda.synchronize()
    raw = run.state.region().cpu().numpy().copy()
    L = run.state.layout
    raw[L.status:L.status + 4] = 0
    return raw


def test_bounded_wait_runs_out_and_is_reported(P):
    import torch
    wl = synth.workload("pace4", B=2, H=4)          # d = 128, bf16 I/O: the tensor-core prefill
    run = PairRun(wl)
    g, r = run.prefill(256)
    assert run.out_ok(g, r)[0]
    run.check_round_and_sync("first chunk")
    assert P.pace_get_status(run.state.handle) == 0
    before = _region_without_status(run)
    x = synth.chunk_inputs(wl, run.t, 256, run.layer)
    dev = {k: run._dev(x[k], k in ("q", "k", "v")) for k in ("q", "k", "v", "a", "beta")}
    o = torch.full((wl.B, wl.H, 256, wl.d_v), 7.0, device="cuda", dtype=torch.bfloat16)
    P.pace_test_wait_probe(run.state.handle, 2_000_000)          # 2 ms
    run.state.prefill_chunk(dev["q"], dev["k"], dev["v"], dev["a"], dev["beta"], o)
    with pytest.raises(P.PaceError) as ei:
        P.pace_get_status(run.state.handle, clear=True)
    assert ei.value.status == P.PACE_ERR_TIMEOUT
    assert np.array_equal(_region_without_status(run), before), "a unit changed although its wait gave up"
    assert bool((o == 7.0).all()), "outputs were written although the wait gave up"
    assert P.pace_get_status(run.state.handle) == 0               # cleared
    # the context is usable: the same chunk, probe off, matches the oracle
    P.pace_test_wait_probe(run.state.handle, 0)
    g, r = run.prefill(256, inputs=x)
    ok, msg = run.out_ok(g, r)
    assert ok, msg
    run.check_round_and_sync("second chunk")
    assert P.pace_get_status(run.state.handle) == 0


def test_out_of_range_counter_leaves_unit_unchanged(P):
    import torch
    wl = synth.workload("pace4", B=2, H=4)
    bad = (1, 2)
    run = PairRun(wl, sample=[(b, h) for b in range(wl.B) for h in range(wl.H) if (b, h) != bad])
    run.prefill(256)
    run.check_round_and_sync("prefill")
    for _ in range(3):
        run.decode()
    # corrupt the counter of one unit in a host copy of the region and import it
    L = run.state.layout
    host = torch.empty(L.total_bytes, dtype=torch.uint8).pin_memory()
    P.pace_state_export(run.state.handle, host, host.numel())
    torch.cuda.synchronize()
    m = host.numpy()[L.m:L.m + 4 * wl.B * wl.H].view(np.int32).reshape(wl.B, wl.H)
    m[bad] = wl.dP + 3
    P.pace_state_import(run.state.handle, host, host.numel())
    torch.cuda.synchronize()
    blob0 = read_blob(run.state)
    for step in range(wl.dP):                      # a whole period: the other units round once
        g, r = run.decode()
        assert run.out_ok(g, r)[0], step
        assert (run.last[bad] == 0).all(), f"step {step}: the corrupted unit emitted a non-zero output"
        if step == 4:
            run.check_round_and_sync("rounding of the other units")
    blob1 = read_blob(run.state)
    assert np.array_equal(blob1.codes(*bad), blob0.codes(*bad))
    assert np.array_equal(blob1.scales()[bad], blob0.scales()[bad])
    for a0, a1 in zip(blob0.buffer(*bad), blob1.buffer(*bad)):
        assert np.array_equal(a0, a1)
    assert blob1.m()[bad] == wl.dP + 3
