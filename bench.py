#!/usr/bin/env python
"""Benchmark of the PACE decode step (one layer, all sequences of the batch, one token per step).

Default workload: 32 heads, d_k = d_v = 128, batch 64, dP = 8, symmetric int4 state with key-axis groups
of 64, int8 decode buffer, bf16 q/k/v/o, after a 512-token prefill in two 256-token chunks.

Timing: CUDA events on the launching stream around exactly K decode steps (captured in CUDA graphs),
after W warm-up steps, with a device synchronize on both sides. Step s uses state set s mod R: R
independent state sets (one per "layer") rotate so that the working set is several times the 129 MB
L2, and the sets are staggered by buffer phase, so every window of R steps holds each of the dP phases
(append-only steps and the rounding step) equally often. `value` is sequences x steps / second.

Extra objects on the JSON line: `roofline` (algorithmic bytes of the decode kernel per launch over its
measured duration, against the measured HBM copy peak), `cpu_baseline` (the CPU oracle on a bounded
sample, host cores), `e2e` (the same metric with host buffers: pinned host->device inputs and the
device->host output copy inside the timed region), `bf16_pertoken` (the per-token bf16-state kernel,
the pages' comparison point), `prefill`, and `clocks`.

`--impl reference` times the CPU oracle (the reference arm) on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
ROTATE_TARGET = 4 * L2_BYTES


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=1000)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--batch", type=int, default=64)
    p.add_argument("--extra", type=int, default=1, help="also time batch 128, the bf16 kernel and prefill")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-oracle sample")
    p.add_argument("--pace48-only", type=int, default=0, metavar="K",
                   help="only time K steps of the PACE-4/8 leg (batch 128, 8 int8 heads by pace_assign_heads), print "
                        "one JSON line and exit (a short command for profiling its two pool kernels)")
    p.add_argument("--prefill-only", type=int, default=0, metavar="B",
                   help="only time two 256-token prefill chunks on one PACE-4 state of B sequences x 32 heads "
                        "(a small case for profiling the chunk kernel), print one JSON line and exit")
    return p.parse_args(argv)


NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e datasheet bandwidth (context beside the measured copy peak)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def read_tensor_peak():
    """Sustained dense bf16 TFLOP/s (a kernel timed inside a long run), measured, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def decode_bytes_per_unit(D: int, g: int, dP: int, m0: int, zp: int = 0, bits: int = 4, mixed: int = 0) -> int:
    """Algorithmic bytes one decode step of one unit moves when the buffer holds m0 tokens before it:
    packed codes and group scales (and zero points) read, the buffered entries read, the new entry
    written, q/k/v/a/beta read and o written, the counter, and on the rounding step the state written."""
    ng = D // g
    state = D * D * bits // 8 + ng * D * 2 + (ng * D if zp else 0)
    entry = (D // 2 + 2 * D + 16) if mixed else (2 * D + 16)
    io = 3 * D * 2 + D * 2 + 8
    b = state + m0 * entry + entry + io + 8
    if m0 + 1 == dP:
        b += state
    return b


def decode_bytes_period_avg(D, g, dP, **kw) -> float:
    return sum(decode_bytes_per_unit(D, g, dP, m0, **kw) for m0 in range(dP)) / dP


def bf16buf_bytes_per_period_avg(D: int, dP: int) -> float:
    """Buffered bf16 state, averaged over a period: the bf16 state read every step and written once per period,
    plus the same buffer and token traffic as PACE-4 (int8 buffer)."""
    entry = 2 * D + 16
    io = 3 * D * 2 + D * 2 + 8
    state = D * D * 2
    return state + state / dP + sum(m0 * entry for m0 in range(dP)) / dP + entry + io + 8


def bf16_bytes_per_unit(D: int) -> int:
    return 2 * D * D * 2 + 3 * D * 2 + D * 2 + 8


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


DECODE_SOURCES = ["bit_gated_delta_gb300/csrc/decode_fold.cuh", "bit_gated_delta_gb300/csrc/decode_fold_s8.cu",
                  "bit_gated_delta_gb300/csrc/decode_mma.cuh", "bit_gated_delta_gb300/csrc/pace_common.cuh",
                  "bit_gated_delta_gb300/csrc/pace_internal.h"]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d[kernel][workload]
        if rec.get("source_digest") == source_digest(DECODE_SOURCES):
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ------------------------------------------------------------------------------------------------------
# GPU arm

class DecodeSetup:
    """R state sets of one workload, prefilled and staggered by buffer phase, plus device-resident
    decode inputs (NI distinct tokens)."""

    NI = 8

    def __init__(self, P, torch, wl, state_mode, R, prefill_tokens=512, mask=None):
        import synth
        self.P, self.torch, self.wl = P, torch, wl
        bf16 = state_mode == P.PACE_STATE_BF16
        self.cfg = P.make_config(wl.H, wl.d_k, wl.B, dP=wl.dP, group=wl.g, zero_point=wl.zero_point,
                                 buf_mode=P.PACE_BUF_MIXED if wl.mixed_buffer else P.PACE_BUF_INT8,
                                 state_mode=state_mode)
        self.states = [P.PaceState(self.cfg, wl.B, mask) for _ in range(R)]
        self.uses = [0] * R              # decode steps launched on each set (its buffer phase, mod dP)
        self.R = R
        o = torch.empty(wl.B, wl.H, 256, wl.d_v, dtype=torch.bfloat16, device="cuda")
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # one untimed chunk on the last set first: the library's kernels are loaded on their first launch, a
        # one-time host cost that would otherwise land inside the first timed chunk (the set is overwritten below)
        x = synth.device_chunk_inputs(wl, 0, 256)
        self.states[-1].prefill_chunk(x["q"], x["k"], x["v"], x["a"], x["beta"], o)
        torch.cuda.synchronize()
        self.prefill_ms = 0.0
        for c, t0 in enumerate(range(0, prefill_tokens, 256)):
            x = synth.device_chunk_inputs(wl, t0, 256)
            ev0.record()
            self.states[0].prefill_chunk(x["q"], x["k"], x["v"], x["a"], x["beta"], o)
            ev1.record()
            torch.cuda.synchronize()
            self.prefill_ms += ev0.elapsed_time(ev1)
        self.prefill_tokens = prefill_tokens
        src = self.states[0].region()
        for st in self.states[1:]:
            st.region().copy_(src)
        x = synth.device_chunk_inputs(wl, prefill_tokens, self.NI)
        self.inputs = [{k: (v[:, :, i].contiguous()) for k, v in x.items()} for i in range(self.NI)]
        self.o = torch.empty(wl.B, wl.H, wl.d_v, dtype=torch.bfloat16, device="cuda")
        if not bf16:
            for r, st in enumerate(self.states):
                for i in range(r % wl.dP):
                    self.step_on(st, i)
        torch.cuda.synchronize()

    def step_on(self, st, i, stream=None):
        x = self.inputs[i % self.NI]
        st.decode_step(x["q"], x["k"], x["v"], x["a"], x["beta"], self.o, stream)
        self.uses[self.states.index(st)] += 1

    def replayed(self, n_steps):
        """Account the launches of one replay of a graph of n_steps steps."""
        for i in range(n_steps):
            self.uses[i % self.R] += 1

    def rounding_steps(self, n_steps):
        """How many of the next n_steps steps (sets in rotation) are rounding steps."""
        uses = list(self.uses)
        n = 0
        for i in range(n_steps):
            r = i % self.R
            if uses[r] % self.wl.dP == self.wl.dP - 1:
                n += 1
            uses[r] += 1
        return n

    def graph(self, n_steps):
        """A CUDA graph of n_steps consecutive decode steps over the rotating sets."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(2):                       # warm the launch path outside the capture
                self.step_on(self.states[i % self.R], i)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        uses = list(self.uses)
        with torch.cuda.graph(g):
            for i in range(n_steps):
                self.step_on(self.states[i % self.R], i)
        self.uses = uses                 # capture launches nothing
        return g

    def close(self):
        for st in self.states:
            st.close()


def time_steps(torch, setup, K, W, sampler=None):
    """Run W warm-up steps, then exactly K timed steps; returns ms per step (CUDA events)."""
    G = setup.R * setup.wl.dP if setup.cfg.state_mode != 2 else setup.R
    G = min(G, max(1, K))
    nvtx = torch.cuda.nvtx
    nvtx.range_push(f"decode warm-up B={setup.wl.B} H={setup.wl.H}")
    g = setup.graph(G)
    for _ in range((W + G - 1) // G):
        g.replay()
        setup.replayed(G)
    tail = K % G
    gt = setup.graph(tail) if tail else None
    torch.cuda.synchronize()
    nvtx.range_pop()
    setup.window_roundings = setup.rounding_steps(K)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        torch.cuda.synchronize()
        nvtx.range_push(f"decode timed {K} steps B={setup.wl.B} H={setup.wl.H}")
        ev0.record()
        for _ in range(K // G):
            g.replay()
        if gt is not None:
            gt.replay()
        ev1.record()
        torch.cuda.synchronize()
        nvtx.range_pop()
    return ev0.elapsed_time(ev1) / K


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def time_e2e(torch, P, setup, K, nbuf=2):
    """Same metric through the public API with host buffers: per step, one pinned host -> device copy of the
    step's packed inputs (q, k, v, a, beta back to back, each at a 16-byte aligned offset, as a model's fused
    projection would hand them over), the decode call on views of that buffer, and the device -> host copy of o,
    all inside the timed region. The steps are pipelined as a serving loop would run them: the input copy on a
    copy stream into one of two device buffers, the decode on the main stream, the output copy on a third stream
    from one of two output buffers, ordered by events (a buffer is refilled only after the step that used it is
    done), and the loop of G steps is captured once as a CUDA graph and replayed. The same steps issued one after
    the other on one stream, without a graph, are timed too (serial_ms_per_step)."""
    wl = setup.wl
    names = ("q", "k", "v", "a", "beta")
    x0 = setup.inputs[0]
    offs, off = {}, 0
    for k in names:
        offs[k] = off
        off += -(-x0[k].numel() * x0[k].element_size() // 256) * 256
    total = off
    host = []
    for i in range(DecodeSetup.NI):
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        for k in names:
            v = setup.inputs[i][k]
            n = v.numel() * v.element_size()
            hb[offs[k]:offs[k] + n].copy_(v.contiguous().view(-1).view(torch.uint8).cpu())
        host.append(hb)
    dbuf = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(nbuf)]
    dev = []
    for j in range(nbuf):
        d = {}
        for k in names:
            v = x0[k]
            n = v.numel() * v.element_size()
            d[k] = dbuf[j][offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
        dev.append(d)
    obuf = [torch.empty(wl.B, wl.H, wl.d_v, dtype=torch.bfloat16, device="cuda") for _ in range(nbuf)]
    o_host = [torch.empty(wl.B, wl.H, wl.d_v, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    h2d = sum(x0[k].numel() * x0[k].element_size() for k in names)
    d2h = o_host[0].numel() * o_host[0].element_size()
    n = min(K, 2000)

    # serial: each step's three operations back to back on one stream, issued from Python
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for i in range(n):
        dbuf[0].copy_(host[i % DecodeSetup.NI], non_blocking=True)
        d = dev[0]
        setup.states[i % setup.R].decode_step(d["q"], d["k"], d["v"], d["a"], d["beta"], obuf[0])
        o_host[0].copy_(obuf[0], non_blocking=True)
    ev1.record()
    torch.cuda.synchronize()
    ms_serial = ev0.elapsed_time(ev1) / n

    # pipelined and captured: G steps per graph (a multiple of the rotating sets and of the distinct inputs)
    G = setup.R * DecodeSetup.NI // math.gcd(setup.R, DecodeSetup.NI)
    while G < 16:
        G *= 2
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_dec = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        main = torch.cuda.current_stream()
        for e in ev_dec + ev_out:
            e.record(main)
        cin.wait_stream(main)
        cout.wait_stream(main)
        for i in range(G):
            b = i % nbuf
            cin.wait_event(ev_dec[b])              # the decode that read this input buffer is done
            with torch.cuda.stream(cin):
                dbuf[b].copy_(host[i % DecodeSetup.NI], non_blocking=True)
            ev_in[b].record(cin)
            main.wait_event(ev_in[b])
            main.wait_event(ev_out[b])             # the copy-out of this output buffer is done
            d = dev[b]
            setup.states[i % setup.R].decode_step(d["q"], d["k"], d["v"], d["a"], d["beta"], obuf[b], main)
            ev_dec[b].record(main)
            cout.wait_event(ev_dec[b])
            with torch.cuda.stream(cout):
                o_host[b].copy_(obuf[b], non_blocking=True)
            ev_out[b].record(cout)
        main.wait_stream(cin)
        main.wait_stream(cout)
    reps = max(1, n // G)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ev0.record()
    for _ in range(reps):
        graph.replay()
    ev1.record()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / (reps * G)
    # the host-to-device copy alone, the same packed pinned buffers back to back
    ev0.record()
    for i in range(n):
        dbuf[0].copy_(host[i % DecodeSetup.NI], non_blocking=True)
    ev1.record()
    torch.cuda.synchronize()
    ms_copy = ev0.elapsed_time(ev1) / n
    return {"value": wl.B / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": reps * G,
            "note": "per step: one packed pinned host-to-device copy (copy stream, two device buffers), the "
                    "pace_decode_step call, the device-to-host copy of o (third stream, two pinned buffers); "
                    f"{G} steps captured as one CUDA graph and replayed",
            "serial_ms_per_step": ms_serial, "serial_note": "the same three operations per step on one stream, "
                                                            "issued from Python without a graph",
            "h2d_copy_alone_ms": ms_copy, "h2d_copy_alone_gbs": total / (ms_copy * 1e-3) / 1e9}


# ------------------------------------------------------------------------------------------------------
# CPU oracle (the baseline, and the reference arm)

def oracle_decode_rate(wl, budget_s: float, n_units: int = 32):
    """Decode tokens/s of the CPU oracle on a bounded sample: n_units units of one sequence, prefilled
    with 512 tokens, then whole decode periods until the time budget is used (OpenMP over units)."""
    import oracle as O
    import synth
    wl1 = wl.with_(B=1, H=n_units)
    cfg = O.Cfg(d_k=wl.d_k, d_v=wl.d_v, g=wl.g, bits=4, zero_point=wl.zero_point, dP=wl.dP,
                buf_mode=O.BUF_MIXED if wl.mixed_buffer else O.BUF_INT8)
    units = [O.Unit(cfg) for _ in range(n_units)]
    for t0 in range(0, 512, 256):
        x = synth.chunk_inputs(wl1, t0, 256)
        for h, u in enumerate(units):
            O.prefill(u, x["q"][0, h], x["k"][0, h], x["v"][0, h], x["a"][0, h], x["beta"][0, h])
    toks = [synth.token_inputs(wl1, 512 + i) for i in range(wl.dP)]
    threads = O.max_threads()
    steps = 0
    t_start = time.perf_counter()
    while True:
        for i in range(wl.dP):
            x = toks[i]
            O.decode_batch(units, x["q"][0], x["k"][0], x["v"][0], x["a"][0], x["beta"][0], nthreads=threads)
        steps += wl.dP
        el = time.perf_counter() - t_start
        if el >= budget_s:
            break
    unit_steps_per_s = n_units * steps / el
    tokens_per_s = unit_steps_per_s / wl.H          # one sequence token = H unit steps
    return {"value": tokens_per_s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_units} heads of one sequence, 512-token prefill, {steps} decode steps "
                      f"({steps // wl.dP} periods), {el:.1f} s; tokens/s = unit-steps/s / {wl.H} heads"}


def oracle_rate(wl, n_units: int, budget_s: float, threads: int, prefill: int = 256, int8_heads=()):
    """Decode unit-steps/s of the CPU oracle: n_units heads of one sequence (heads listed in int8_heads kept at
    8 bits), `prefill` tokens of prefill, then whole decode periods until the budget is used."""
    import oracle as O
    import synth
    wl1 = wl.with_(B=1, H=n_units)
    buf = O.BUF_MIXED if wl.mixed_buffer else O.BUF_INT8
    units = [O.Unit(O.Cfg(d_k=wl.d_k, d_v=wl.d_v, g=wl.g, bits=8 if h in int8_heads else 4,
                          zero_point=wl.zero_point, dP=wl.dP, buf_mode=buf)) for h in range(n_units)]
    for t0 in range(0, prefill, 256):
        x = synth.chunk_inputs(wl1, t0, min(256, prefill - t0))
        for h, u in enumerate(units):
            O.prefill(u, x["q"][0, h], x["k"][0, h], x["v"][0, h], x["a"][0, h], x["beta"][0, h])
    toks = [synth.token_inputs(wl1, prefill + i) for i in range(wl.dP)]
    groups = [[h for h in range(n_units) if (h in int8_heads) == b] for b in (False, True)]
    steps, t_start = 0, time.perf_counter()
    while True:
        for i in range(wl.dP):
            x = toks[i]
            for hs in groups:
                if hs:
                    O.decode_batch([units[h] for h in hs], x["q"][0, hs], x["k"][0, hs], x["v"][0, hs], x["a"][0, hs],
                                   x["beta"][0, hs], nthreads=threads)
        steps += wl.dP
        el = time.perf_counter() - t_start
        if el >= budget_s:
            break
    return n_units * steps / el, steps, el


def oracle_rates(budget_s: float = 1.5):
    """The CPU oracle on configs 0-3, one thread and all cores (bounded samples; tokens/s of the whole
    configuration = unit-steps/s / units per token)."""
    import oracle as O
    import synth
    cores = O.max_threads()
    out = {"cores": cores}
    cases = [("tiny", synth.workload("tiny"), 4, 4, 256, ()),              # all 4 units (2 sequences x 2 heads)
             ("pace4", synth.workload("pace4"), 32, 32, 256, ()),
             ("pace48", synth.workload("pace48"), 32, 32, 256, tuple(range(0, 32, 4))),
             ("sweep_24x16", synth.workload("sweep"), 16, 24 * 16, 256, ())]
    for name, wl, n, per_token, pf, i8 in cases:
        row = {}
        for th in (1, cores):
            ups, steps, el = oracle_rate(wl, n, budget_s, th, pf, i8)
            row[f"tokens_per_s_{th}t"] = ups / per_token
        row["sample"] = (f"{n} units of one sequence ({len(i8)} at 8 bits), {pf}-token prefill, decode periods for "
                         f"{budget_s} s per thread count; one token of the configuration = {per_token} unit-steps")
        out[name] = row
    return out


def run_reference(args):
    import synth
    wl = synth.workload("pace4", B=args.batch)
    budget = max(2.0, min(args.cpu_seconds, 60.0))
    t0 = time.perf_counter()
    cb = oracle_decode_rate(wl, budget)
    wall = time.perf_counter() - t0
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wl.B / cb["value"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, None),
            "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


METRIC = "PACE decode tokens/s (B=64-128, dP=8) and achieved HBM GB/s vs GB300 peak"


def workload_config(wl, R):
    c = {"workload": f"PACE-4 decode, 1 layer, H={wl.H}, d_k=d_v={wl.d_k}, batch {wl.B}, dP={wl.dP}, "
                     f"key-axis g={wl.g} symmetric int4 state, int8 buffer, bf16 q/k/v/o, 512-token context",
         "B": wl.B, "H": wl.H, "d": wl.d_k, "dP": wl.dP, "g": wl.g}
    if R is not None:
        c["l2"] = (f"inputs larger than L2: {R} independent state sets rotate (one per step), staggered by "
                   f"buffer phase")
    return c


def rotation_count(nbytes: int, dP: int, align_dp: bool) -> int:
    R = max(2, -(-ROTATE_TARGET // nbytes))
    if align_dp:
        R = -(-R // dP) * dP
    return int(R)


def measure(P, torch, wl, state_mode, K, W, sampler=None, min_sets=2, mask=None):
    bytes1 = P.pace_state_bytes(P.make_config(wl.H, wl.d_k, wl.B, dP=wl.dP, group=wl.g, state_mode=state_mode,
                                              zero_point=wl.zero_point,
                                              buf_mode=P.PACE_BUF_MIXED if wl.mixed_buffer else P.PACE_BUF_INT8),
                                mask)
    periodic = state_mode in (P.PACE_STATE_QUANT, P.PACE_STATE_BF16_BUF)
    R = max(rotation_count(bytes1, wl.dP, periodic), min_sets)
    if periodic:
        R = -(-R // wl.dP) * wl.dP
    setup = DecodeSetup(P, torch, wl, state_mode, R, mask=mask)
    ms = time_steps(torch, setup, K, W, sampler)
    return setup, ms, R


def batch_sweep(P, torch, token_steps=100):
    """The pages' throughput study shape: 24 gated-delta layers x 16 heads, one token step = 24 sequential layer
    launches (each layer its own state set, in one CUDA graph); PACE-4 dP=8 against the per-token bf16 kernel at
    every batch size, with the buffered bf16 state (the decode buffer without the 4-bit state) beside them.
    Returns per-batch tokens/s and the smallest batch from which PACE-4 stays faster than per-token bf16."""
    import synth
    out, L = {}, 24
    for b in (1, 2, 4, 8, 16, 32, 64, 128):
        wl = synth.workload("sweep", B=b)
        row = {}
        for name, mode in (("pace4", P.PACE_STATE_QUANT), ("bf16", P.PACE_STATE_BF16),
                           ("bf16buf", P.PACE_STATE_BF16_BUF)):
            s, ms, R = measure(P, torch, wl, mode, token_steps * L, 3 * L, min_sets=L)
            row[f"{name}_tokens_per_s"] = b / (ms * L * 1e-3)
            row[f"{name}_ms_per_token_step"] = ms * L
            s.close()
            torch.cuda.empty_cache()
        row["speedup"] = row["pace4_tokens_per_s"] / row["bf16_tokens_per_s"]
        out[str(b)] = row
    faster = [int(b) for b, r in out.items() if r["speedup"] > 1.0]
    cross = None
    for b in sorted(int(x) for x in out):
        if all(out[str(c)]["speedup"] > 1.0 for c in out if int(c) >= b):
            cross = b
            break
    return {"layers": L, "heads": 16, "d": 128, "per_batch": out, "pace4_faster_from_batch": cross,
            "note": "one token step = 24 layer launches on distinct state sets; >= 24 sets rotate"}


def prefill_longctx(P, torch, n_tokens=32768, distinct=8):
    """Long-context prefill shaped like the pages' 32,768-token study: 48 heads, d=128, batch 16, PACE-4 g=64,
    slow decay, n_tokens in 256-token chunks (the state rounded once per chunk). `distinct` chunks of inputs are
    drawn on the device and reused cyclically (the state carries on); CUDA events time the chunk launches only.
    FLOPs per unit and chunk are those of the tensor-core form (the dense contractions of the chunk kernel)."""
    import synth
    wl = synth.workload("longctx")
    cfg = P.make_config(wl.H, wl.d_k, wl.B, dP=8, group=wl.g)
    st = P.PaceState(cfg, wl.B)
    chunks = [synth.device_chunk_inputs(wl, 256 * c, 256) for c in range(distinct)]
    o = torch.empty(wl.B, wl.H, 256, wl.d_v, dtype=torch.bfloat16, device="cuda")
    n_chunks = n_tokens // 256
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record()
    for c in range(n_chunks):
        x = chunks[c % distinct]
        st.prefill_chunk(x["q"], x["k"], x["v"], x["a"], x["beta"], o)
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1])
    st.close()
    units = wl.B * wl.H
    # per 32-token sub-chunk: S^T [k|q] (2 parts, 128x64x128), Gram (128x32x128), update (2 parts, 128x128x32)
    flop_sub = 2 * (2 * 128 * 64 * 128 + 128 * 32 * 128 + 2 * 128 * 128 * 32)
    tflops = units * n_chunks * 8 * flop_sub / (ms * 1e-3) / 1e12
    tpk, tpk_kind = read_tensor_peak()
    return {"B": wl.B, "H": wl.H, "d": wl.d_k, "tokens": n_tokens, "chunks": n_chunks, "ms": ms,
            "tokens_per_s": wl.B * n_tokens / (ms * 1e-3), "tensor_tflops": tflops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": tpk, "unit": "TFLOP/s", "frac": tflops / tpk,
                         "peak_kind": f"{tpk_kind} bf16 dense, sustained", "kernel": "pace::prefill_tc_kernel<64>"},
            "note": "tensor-core chunk prefill; inputs drawn on the device, 8 distinct chunks reused"}


def synthetic_error_study(P, torch, prefill_tokens=32768, decode_tokens=1024):
    """The pages' two claims on the synthetic column-outlier states (long-context shape: 48 heads, d=128,
    batch 16, slow decay): (1) the quantization error of the prefilled fp32 state with the scale shared along the
    key axis (PACE) and along the value axis (baseline), per head; (2) the drift of PACE-4 outputs against the
    unquantized state over `decode_tokens` decode steps for rounding periods dP = 1 (per-token rounding), 8, 32.
    All states start from the same prefill inputs (8 distinct device-drawn chunks reused cyclically) and decode
    the same device-drawn tokens."""
    import synth
    wl = synth.workload("longctx")
    B, H, D = wl.B, wl.H, wl.d_k
    chunks = [synth.device_chunk_inputs(wl, 256 * c, 256) for c in range(8)]
    dec = synth.device_chunk_inputs(wl, prefill_tokens, decode_tokens)
    modes = {"fp32": (P.PACE_STATE_FP32, P.PACE_BUF_FP32, 8)}
    for dP in (1, 8, 32):
        modes[f"pace4_dP{dP}"] = (P.PACE_STATE_QUANT, P.PACE_BUF_INT8, dP)
    states = {}
    o = torch.empty(B, H, 256, D, dtype=torch.bfloat16, device="cuda")
    for name, (sm, bm, dP) in modes.items():
        st = P.PaceState(P.make_config(H, D, B, dP=dP, group=wl.g, state_mode=sm, buf_mode=bm), B)
        for c in range(prefill_tokens // 256):
            x = chunks[c % 8]
            st.prefill_chunk(x["q"], x["k"], x["v"], x["a"], x["beta"], o)
        states[name] = st
    ek = torch.zeros(B * H, device="cuda")
    ev = torch.zeros(B * H, device="cuda")
    P.pace_calib_error_energy_axis(states["fp32"].handle, 4, wl.g, 0, 0, ek)
    P.pace_calib_error_energy_axis(states["fp32"].handle, 4, wl.g, 0, 1, ev)
    ratio = (ev / ek.clamp_min(1e-30)).cpu().numpy()
    outs = {}
    tail = {name: [] for name in modes if name != "fp32"}
    for t in range(decode_tokens):
        x = {k: v[:, :, t].contiguous() for k, v in dec.items()}
        for name, st in states.items():
            ob = torch.empty(B, H, D, dtype=torch.bfloat16, device="cuda")
            st.decode_step(x["q"], x["k"], x["v"], x["a"], x["beta"], ob)
            outs[name] = ob.float()
        if t >= decode_tokens - 256:
            r = outs["fp32"]
            rn = float(torch.linalg.vector_norm(r))
            for name in tail:
                tail[name].append(float(torch.linalg.vector_norm(outs[name] - r)) / rn)
    drift = {name: {"rel_l2_last_256_mean": float(np.mean(v)), "rel_l2_final": v[-1]} for name, v in tail.items()}
    for st in states.values():
        st.close()
    return {"B": B, "H": H, "d": D, "prefill_tokens": prefill_tokens, "decode_tokens": decode_tokens,
            "error_value_over_key_axis": {"mean": float(ratio.mean()), "median": float(np.median(ratio)),
                                          "min": float(ratio.min()), "heads_key_axis_lower": float(np.mean(ratio > 1))},
            "drift_vs_unquantized": drift,
            "note": "fp32 unquantized reference vs PACE-4 (g=64, int8 buffer) at dP 1/8/32; bf16 outputs"}


def pace48_leg(P, torch, peak, K, W):
    """PACE-4/8 (BASELINE config 2): batch 128, 32 heads, g = 32 with integer zero points, mixed decode buffer (int4
    keys, bf16 values); the quarter of heads with the largest E_h = e_h / (1 - a_h^(2 dP)) stay int8, chosen by
    pace_assign_heads from the GPU calibration of a 512-token fp32 prefill (e_h averaged over the sequences).
    Algorithmic bytes per unit-step as resident (u8 zero points), averaged over the 24 int4 and 8 int8 heads."""
    import synth
    wl = synth.workload("pace48")
    a_h = synth.head_decays(wl)
    cfg = P.make_config(wl.H, wl.d_k, wl.B, dP=wl.dP, group=wl.g, zero_point=1, state_mode=P.PACE_STATE_FP32,
                        buf_mode=P.PACE_BUF_FP32)
    st = P.PaceState(cfg, wl.B)
    o = torch.empty(wl.B, wl.H, 256, wl.d_v, dtype=torch.bfloat16, device="cuda")
    for c in range(2):
        x = synth.device_chunk_inputs(wl, 256 * c, 256)
        st.prefill_chunk(x["q"], x["k"], x["v"], x["a"], x["beta"], o)
    e = torch.zeros(wl.B * wl.H, device="cuda")
    P.pace_calib_error_energy(st.handle, 4, wl.g, 1, e)
    e_h = e.view(wl.B, wl.H).mean(0).cpu().numpy()
    st.close()
    mask = P.pace_assign_heads(e_h, a_h, wl.dP, 0.25)
    s, ms, R = measure(P, torch, wl, P.PACE_STATE_QUANT, K, W, mask=mask)
    rounding = s.window_roundings
    s.close()
    n8 = int(mask.sum())
    per = ((wl.H - n8) * decode_bytes_period_avg(wl.d_k, wl.g, wl.dP, zp=1, bits=4, mixed=1) +
           n8 * decode_bytes_period_avg(wl.d_k, wl.g, wl.dP, zp=1, bits=8, mixed=1)) / wl.H
    alg = wl.B * wl.H * per
    return {"B": wl.B, "H": wl.H, "int8_heads": [int(h) for h in np.flatnonzero(mask)], "tokens_per_s": wl.B / (ms * 1e-3),
            "ms_per_step": ms, "bytes_per_unit_step": per, "achieved_gbs": alg / (ms * 1e-3) / 1e9,
            "frac": alg / (ms * 1e-3) / 1e9 / peak, "rotating_sets": R, "rounding_steps_in_window": rounding,
            "steps": K, "note": "two launches per step: the int4 pool, and the int8 pool on the state's own stream "
                                "(forked and joined by events) so that both pools share the SMs"}


def longctx_decode(P, torch, peak, K, W):
    """Decode of the long-context shape (48 heads, d=128, batch 16, PACE-4 g=64) at rounding periods dP = 1, 8, 32,
    after a 512-token prefill (the decode cost does not depend on the context length: the state has a fixed size);
    rotating state sets as in the default line. Every period runs the folded-readout kernel (dP = 32 with its
    32-token tables)."""
    import synth
    out = {}
    for dP in (1, 8, 32):
        wl = synth.workload("longctx").with_(dP=dP)
        k = -(-K // dP) * dP
        s, ms, R = measure(P, torch, wl, P.PACE_STATE_QUANT, k, W)
        s.close()
        alg = wl.B * wl.H * decode_bytes_period_avg(wl.d_k, wl.g, dP)
        out[f"dP{dP}"] = {"tokens_per_s": wl.B / (ms * 1e-3), "ms_per_step": ms, "achieved_gbs": alg / (ms * 1e-3) / 1e9,
                          "frac": alg / (ms * 1e-3) / 1e9 / peak, "rotating_sets": R, "steps": k}
        torch.cuda.empty_cache()
    return out


def shared_key_heads(P, torch, peak, B=64, H=32, Hk=16, steps=2000):
    """PACE-4 decode with shared key heads (gamma = H / Hk value heads per key head, one buffered key copy per key
    head): the same workload shape as the default line with Hk key heads; rotating state sets as there."""
    import synth
    wl = synth.workload("pace4", B=B)
    cfg = P.make_config(H, 128, B, dP=8, group=64, key_heads=Hk)
    per = P.pace_state_bytes(cfg)
    R = max(2, -(-ROTATE_TARGET // per))
    R = -(-R // 8) * 8
    states = [P.PaceState(cfg, B) for _ in range(R)]
    o = torch.empty(B, H, 256, 128, dtype=torch.bfloat16, device="cuda")
    for c in range(2):
        x = synth.device_chunk_inputs(wl, 256 * c, 256)
        states[0].prefill_chunk(x["q"][:, ::H // Hk].contiguous(), x["k"][:, ::H // Hk].contiguous(), x["v"], x["a"],
                                x["beta"], o)
    for st in states[1:]:
        st.region().copy_(states[0].region())
    xs = synth.device_chunk_inputs(wl, 512, 8)
    toks = [{k: v[:, :, i].contiguous() for k, v in xs.items()} for i in range(8)]
    for t in toks:
        t["q"] = t["q"][:, ::H // Hk].contiguous()
        t["k"] = t["k"][:, ::H // Hk].contiguous()
    ob = torch.empty(B, H, 128, dtype=torch.bfloat16, device="cuda")
    for r, st in enumerate(states):
        for i in range(r % 8):
            x = toks[i]
            st.decode_step(x["q"], x["k"], x["v"], x["a"], x["beta"], ob)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(2):
            x = toks[i]
            states[i].decode_step(x["q"], x["k"], x["v"], x["a"], x["beta"], ob)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for i in range(R * 8):
            x = toks[i % 8]
            states[i % R].decode_step(x["q"], x["k"], x["v"], x["a"], x["beta"], ob)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(1, steps // (R * 8))
    ev0.record()
    for _ in range(n):
        g.replay()
    ev1.record()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / (n * R * 8)
    for st in states:
        st.close()
    # bytes per unit-step: as PACE-4 with the key rows of the buffer read and written once per key head
    D = 128
    full = decode_bytes_period_avg(D, 64, 8)
    key_rows = (sum(m0 for m0 in range(8)) / 8 + 1) * D     # buffered key bytes read + written per unit-step
    alg = B * H * (full - key_rows * (1 - Hk / H))
    return {"B": B, "H": H, "key_heads": Hk, "tokens_per_s": B / (ms * 1e-3), "ms_per_step": ms,
            "achieved_gbs": alg / (ms * 1e-3) / 1e9, "frac": alg / (ms * 1e-3) / 1e9 / peak, "rotating_sets": R}


def prefill_only(P, torch, B):
    """Two 256-token chunks of device-drawn inputs through pace_prefill_chunk on one PACE-4 state (B sequences,
    32 heads, d=128): the chunk kernel on a working set of a few hundred MB, for profiling."""
    import synth
    wl = synth.workload("pace4", B=B)
    st = P.PaceState(P.make_config(wl.H, 128, wl.B, dP=8, group=64), wl.B)
    o = torch.empty(wl.B, wl.H, 256, 128, dtype=torch.bfloat16, device="cuda")
    xs = [synth.device_chunk_inputs(wl, 256 * c, 256) for c in range(2)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    us = []
    for x in xs:
        ev[0].record()
        st.prefill_chunk(x["q"], x["k"], x["v"], x["a"], x["beta"], o)
        ev[1].record()
        torch.cuda.synchronize()
        us.append(ev[0].elapsed_time(ev[1]) * 1e3)
    st.close()
    print(json.dumps({"prefill_only": {"B": B, "H": wl.H, "chunk_us": us}}), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    import torch

    import bit_gated_delta_gb300 as P
    import synth
    from bit_gated_delta_gb300 import build as B
    if not B.up_to_date():
        B.build()
    torch.cuda.set_device(local)
    if args.prefill_only:
        prefill_only(P, torch, args.prefill_only)
        return
    if args.pace48_only:
        peak, _ = read_peaks()
        print(json.dumps({"pace48_only": pace48_leg(P, torch, peak, args.pace48_only, 3)}), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    peak, peak_kind = read_peaks()
    wl = synth.workload("pace4", B=args.batch)
    K, W = max(1, args.steps), max(3, args.warmup)

    sampler = ClockSampler(local)
    if dist:
        dist.barrier()
    setup, ms, R = measure(P, torch, wl, P.PACE_STATE_QUANT, K, W, sampler)
    from bit_gated_delta_gb300 import shard
    ms_max = shard.max_over_ranks(ms, dist)      # weak scaling: each rank owns its B sequences
    value = world * wl.B / (ms_max * 1e-3)
    units = wl.B * wl.H
    alg = units * decode_bytes_period_avg(wl.d_k, wl.g, wl.dP)
    achieved = alg / (ms * 1e-3) / 1e9
    traffic = recorded_traffic("decode_fold_kernel", f"pace4_b{wl.B}")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "frac_nominal": achieved / NOMINAL_HBM_GBS, "nominal_gbs": NOMINAL_HBM_GBS,
                "traffic": traffic, "peak_kind": peak_kind, "kernel": "pace::decode_fold_kernel<128,64,4,0,0,1,8>",
                "algorithmic_bytes_per_launch": alg,
                "note": "one decode_fold_kernel launch per step; duration = event time of K graph-replayed steps / K; "
                        "algorithmic bytes averaged over a rounding period"}
    rounding = setup.window_roundings
    e2e = time_e2e(torch, P, setup, K)
    e2e["value"] *= world
    prefill = {"tokens": setup.prefill_tokens, "ms": setup.prefill_ms,
               "tokens_per_s": wl.B * setup.prefill_tokens / (setup.prefill_ms * 1e-3)}
    setup.close()
    del setup
    torch.cuda.empty_cache()

    extra = {}
    if args.extra:
        k2 = max(1000, K // 4)
        for b in (64, 128):
            wlb = synth.workload("pace4", B=b)
            s2, ms2, R2 = measure(P, torch, wlb, P.PACE_STATE_BF16, k2, max(3, W // 4))
            extra[f"bf16_pertoken_b{b}"] = {"tokens_per_s": b / (ms2 * 1e-3), "ms_per_step": ms2, "rotating_sets": R2,
                                            "achieved_gbs": b * wlb.H * bf16_bytes_per_unit(128) / (ms2 * 1e-3) / 1e9}
            s2.close()
            s4, ms4, R4 = measure(P, torch, wlb, P.PACE_STATE_BF16_BUF, k2, max(3, W // 4))
            extra[f"bf16_buffered_b{b}"] = {
                "tokens_per_s": b / (ms4 * 1e-3), "ms_per_step": ms4, "rotating_sets": R4,
                "achieved_gbs": b * wlb.H * bf16buf_bytes_per_period_avg(128, 8) / (ms4 * 1e-3) / 1e9,
                "note": "bf16 state rounded once every dP=8 tokens, int8 decode buffer (no 4-bit state)"}
            s4.close()
            if b == 128:
                s3, ms3, R3 = measure(P, torch, wlb, P.PACE_STATE_QUANT, k2, max(3, W // 4))
                alg3 = b * wlb.H * decode_bytes_period_avg(128, 64, 8)
                extra["pace4_b128"] = {"tokens_per_s": b / (ms3 * 1e-3), "ms_per_step": ms3, "rotating_sets": R3,
                                       "achieved_gbs": alg3 / (ms3 * 1e-3) / 1e9,
                                       "frac": alg3 / (ms3 * 1e-3) / 1e9 / peak}
                s3.close()
            torch.cuda.empty_cache()
        extra["sweep_24x16"] = batch_sweep(P, torch)
        extra["prefill_longctx"] = prefill_longctx(P, torch)
        extra["synthetic_error"] = synthetic_error_study(P, torch)
        extra["pace4_shared_keys_b64"] = shared_key_heads(P, torch, peak)
        extra["pace48_b128"] = pace48_leg(P, torch, peak, k2, max(3, W // 4))
        extra["longctx_decode"] = longctx_decode(P, torch, peak, k2, max(3, W // 4))

    cb = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cb = oracle_decode_rate(wl, args.cpu_seconds)
        if args.extra:
            cb["configs"] = oracle_rates()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
                "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic", "config": {**workload_config(wl, R),
                                                              "rounding_steps_in_window": rounding},
                "roofline": roofline, "cpu_baseline": cb, "e2e": e2e, "gpu_launches": K,
                "clocks": sampler.summary(), "prefill": prefill, **extra}
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
