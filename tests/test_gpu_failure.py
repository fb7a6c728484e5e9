"""Failure detection without a GPU fault (GPU).

* A bounded device wait that runs out: the failure-detection probe of the tensor-core prefill waits on an
  mbarrier that nothing signals, gives up after a short limit, and the host reads PACE_ERR_TIMEOUT from the
  status word; the units and their outputs are unchanged, no MMA was issued, and the context stays usable (the
  same chunk then runs normally and matches the oracle).
* A unit whose buffer counter is out of range (a corrupted region, built on the host and imported) is left
  unchanged and its output is zero; every other unit decodes exactly as before.
* pace_validate_state counts exactly the corrupt values planted in a host copy of the region (counter, scale,
  zero point, unused code level, buffer entry, guard byte) and nothing in a clean state."""
import ctypes

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


def _export(P, state):
    import torch
    L = state.layout
    host = torch.empty(L.total_bytes, dtype=torch.uint8).pin_memory()
    P.pace_state_export(state.handle, host, host.numel())
    torch.cuda.synchronize()
    return host


def _import(P, state, host):
    import torch
    P.pace_state_import(state.handle, host, host.numel())
    torch.cuda.synchronize()


def test_validate_state_counts_planted_corruption(P):
    """pace_validate_state counts values that no step of the method writes. Each is planted in a host copy of
    the region and imported; a clean state counts zero everywhere, the corrupted one exactly what was planted."""
    wl = synth.workload("pace48", B=2, H=4)          # zero points, one int8 head, mixed buffer
    mask = np.array([0, 1, 0, 0], np.uint8)
    run = PairRun(wl, mask=mask)
    run.prefill(256)
    for _ in range(3):
        run.decode()
    clean = run.state.validate()
    assert not any(clean.values()), clean
    L, D, NG = run.state.layout, wl.d_k, wl.d_k // wl.g
    host = _export(P, run.state)
    raw = host.numpy()
    raw[L.m:L.m + 4 * wl.B * wl.H].view(np.int32)[1] = wl.dP + 2           # [0] unit (0, 1): counter
    raw[L.scale:L.scale + 2 * wl.B * wl.H * NG * D].view(np.uint16)[2 * NG * D] = 0x7FC0   # [1] unit 2: NaN scale
    raw[L.zp] = 20                                                          # [2] int4 head 0: zero point 20
    k3 = L.buf_k + (3 * wl.dP) * (D // 2)                                   # [4] unit 3, slot 0: key stored as 0
    assert raw[k3] & 0x0F
    raw[k3] &= 0xF0
    raw[L.codes8 - 1] = 0                                                   # [5] the guard before codes8
    _import(P, run.state, host)
    got = run.state.validate()
    want = dict(zip(P.VALIDATE_FIELDS, (1, 1, 1, 0, 1, 1)))
    assert got == want, got
    counts = (ctypes.c_int64 * P.PACE_VALIDATE_N)()
    assert P.lib().pace_validate_state(run.state.handle, counts, None) == P.PACE_ERR_STATE
    assert list(counts) == [1, 1, 1, 0, 1, 1]


def test_validate_state_counts_unused_symmetric_level(P):
    """Symmetric codes never take the level -2^(b-1) (stored 0): one planted int4 code at that level is counted."""
    wl = synth.workload("pace4", B=2, H=2)
    run = PairRun(wl)
    run.prefill(256)
    assert not any(run.state.validate().values())
    host = _export(P, run.state)
    raw = host.numpy()
    c4 = run.state.layout.codes4
    w = raw[c4:c4 + 4].view(np.uint32)
    assert w[0] & 0xF
    w[0] &= 0xFFFFFFF0
    _import(P, run.state, host)
    got = run.state.validate()
    assert got == dict(zip(P.VALIDATE_FIELDS, (0, 0, 0, 1, 0, 0))), got
