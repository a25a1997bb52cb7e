"""Benchmark of the KDA hot path on GB300.

Default (one GPU): the single-sequence prefill workload (B=1, H=32, T=8192,
dk=dv=128, bf16 inputs, fp32 state, chunk 64) timed through the C ABI, plus
the batched decode workload (256 sequences x 32 heads, fp32 128x128 states,
1000 consecutive steps).  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--impl reference times the CPU oracle (fp64, the machine's host cores) on a
bounded sample of the same workload and metric.
Under torchrun (N > 1) every rank runs its own copy of the workload (the
(sequence, head) units are independent: weak scaling, no collective on the
data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=32,d=128) and decode state GB/s vs roofline, 1 GB300"
PREFILL_WL = "prefill_8k"
DECODE_WL = "decode_256"
# Algorithmic work per unit (d = 128, chunk C = 64, bf16 inputs).
# Prefill bytes per token-head: q, k, v, g (4 x 128 x 2 B) and b (2 B) read,
# o (128 x 2 B) written; the fp32 states are per sequence, not per token.
PREFILL_BYTES_PER_TOKEN_HEAD = 4 * 128 * 2 + 2 + 128 * 2
# Intra-chunk kernel, per (chunk, head): four dense 64 x 64 x 128 products
# (A_kk, A_qk, W and U~ counted as dense tiles), 2 flop per multiply-add.
INTRA_FLOP_PER_CHUNK_HEAD = 4 * 2 * 64 * 64 * 128
# Inter-chunk kernel, per (chunk, head): [W; Qp] S (128 x 128 x 128), A_qk U
# (64 x 64 x 128) and Kr^T U (128 x 64 x 128).
INTER_FLOP_PER_CHUNK_HEAD = 2 * 64 * 128 * 128 * 2 + 2 * 64 * 64 * 128 + 2 * 128 * 64 * 128
# The intra-chunk kernel's algorithmic bytes are its inputs: 64 tokens of q, k,
# v, g and b per (chunk, head).  The 90,624-byte record it writes for the
# inter-chunk kernel (read back there) is an intermediate of this two-kernel
# design, reported as overhead, not as algorithmic traffic.
RECORD_BYTES = 90624
INTRA_BYTES_PER_CHUNK_HEAD = 64 * (4 * 128 * 2 + 2)
INTER_BYTES_PER_CHUNK_HEAD = 64 * 128 * 2                        # o rows (the record is overhead)
DECODE_STATE_BYTES_PER_HEAD = 2 * 128 * 128 * 4                # read + write fp32 state


# sources each kernel is built from: a profile summary counts only while
# these files hash to the value recorded in it
KERNEL_SOURCES = {
    "tc_intra": ["kda_tc_intra.cu", "kda_tc_intra.cuh", "kda_tc_handoff.cuh", "kda_tc_common.cuh",
                 "kda_tc.cuh", "kda_internal.cuh", "kda_common.cuh"],
    "tc_inter": ["kda_tc_inter.cu", "kda_tc_inter.cuh", "kda_tc_handoff.cuh", "kda_tc_common.cuh",
                 "kda_tc.cuh", "kda_internal.cuh", "kda_common.cuh"],
    "tc_intra_ovl": ["kda_tc_overlap.cu", "kda_tc_intra.cuh", "kda_tc_inter.cuh", "kda_tc_handoff.cuh",
                     "kda_tc_common.cuh", "kda_tc.cuh", "kda_internal.cuh", "kda_common.cuh"],
    "tc_inter_ovl": ["kda_tc_overlap.cu", "kda_tc_intra.cuh", "kda_tc_inter.cuh", "kda_tc_handoff.cuh",
                     "kda_tc_common.cuh", "kda_tc.cuh", "kda_internal.cuh", "kda_common.cuh"],
    "tc_fused": ["kda_tc_fused.cu", "kda_tc_intra.cuh", "kda_tc_inter.cuh", "kda_tc_handoff.cuh",
                 "kda_tc_common.cuh", "kda_tc.cuh", "kda_internal.cuh", "kda_common.cuh"],
    "decode_ring": ["kda_decode.cu", "kda_tc.cuh", "kda_internal.cuh", "kda_common.cuh"],
    "prep_vec": ["kda_prep.cu", "kda_internal.cuh", "kda_common.cuh"],
    "plan_kernel": ["kda_plan.cu", "kda_internal.cuh", "kda_common.cuh"],
}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary
    profiles/<kernel>_<workload>.md, or None if the kernel changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "linear_attention_serving_delta_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    rec = {}
    with open(path) as fh:
        for line in fh:
            if line.startswith("- ") and ":" in line:
                key, val = line[2:].split(":", 1)
                rec[key.strip()] = val.split()[0] if val.split() else ""
    if rec.get("source_sha256") != h.hexdigest()[:16]:
        return None
    try:
        return int(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm
def flush_l2(buf):
    buf.zero_()


def bench_prefill(torch, kda, W, steps, warmup, dev):
    """prefill_8k.  The step: the library's own choice of schedule (the
    overlapped kernels for this one sequence), timed with events around the
    call only, so that nothing sits between its launches.  Then the same
    call on the separate kernels with the phase events between them: the
    per-kernel times of the intra-chunk and inter-chunk kernels.  L2 flushed
    before every call."""
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    T = sum(inp["lens"])
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > L2 (129 MB)

    def make(schedule):
        return kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], inp["cu_seqlens"],
                           host_cu_seqlens=inp["cu_seqlens"].cpu(), schedule=schedule)

    p = make(kda.SCHEDULE_AUTO)
    path = kda.kda_prefill_schedule(p.args)
    for _ in range(warmup):
        flush_l2(flush)
        p.run()
    torch.cuda.synchronize()
    step_ms = []
    for _ in range(steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        p.run(stream)
        e1.record(stream)
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    assert p.device_status() == 0

    sep = make(kda.SCHEDULE_SEPARATE)
    nph = kda.PREFILL_PHASES
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)]
    for e in ev:  # torch creates the cudaEvent_t on first record
        e.record()
    torch.cuda.synchronize()
    assert all(e.cuda_event for e in ev)
    ev_handles = (kda.c_vp * (nph + 1))(*[e.cuda_event for e in ev])
    for _ in range(3):
        flush_l2(flush)
        sep.run()
    torch.cuda.synchronize()
    sep.args.phase_events = kda.ctypes.cast(ev_handles, kda.c_vp)
    sep_ms, phase_ms = [], [[] for _ in range(nph)]
    for _ in range(steps):
        flush_l2(flush)
        sep.run(stream)
        ev[-1].synchronize()
        sep_ms.append(ev[0].elapsed_time(ev[-1]))
        for i in range(nph):
            phase_ms[i].append(ev[i].elapsed_time(ev[i + 1]))
    sep.args.phase_events = None
    torch.cuda.synchronize()
    assert sep.device_status() == 0
    n_chunks = (T + 63) // 64
    return dict(T=T, H=w.H, step_ms=step_ms, phase_ms=phase_ms, n_chunks=n_chunks, path=path,
                separate_step_ms=sep_ms, launches_per_step=3, workload=w)


def bench_prep(torch, kda, W, dev, reps=10):
    """The preparation step alone (kda_prep: q^, k^, beta, chunk-restarted G)
    on the prefill_8k inputs, against HBM: it reads q, k, g (bf16) and b and
    writes q^, k^, G (fp32) and beta.  L2 flushed before every call."""
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    T, H, dk = inp["q"].shape
    f = dict(dtype=torch.float32, device=dev)
    qh, kh, G = (torch.empty(T, H, dk, **f) for _ in range(3))
    beta = torch.empty(T, H, **f)
    args = (inp["q"], inp["k"], inp["g"], inp["b"], inp["cu_seqlens"], qh, kh, G, beta)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        kda.kda_prep(*args)
    ms = []
    for _ in range(reps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        kda.kda_prep(*args)
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    t = sum(ms) / len(ms)
    nbytes = T * H * (3 * dk * 2 + 2) + T * H * (3 * dk * 4 + 4)
    return {"workload": "prefill_8k inputs (T=8192, H=32, dk=128, bf16 in, fp32 out)",
            "us": t * 1e3, "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (t * 1e-3) / 1e9}


def bench_gate_per_head(torch, kda, W, dev, steps=10):
    """prefill_8k with one decay per token and head (g [T, H], the gated
    delta rule) instead of one per key channel: the same prefill without
    the g rows (1282 - 254 = 1028 algorithmic bytes per token-head).  L2
    flushed before every call."""
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    gh = inp["g"][:, :, 0].contiguous()
    p = kda.Prefill(inp["q"], inp["k"], inp["v"], gh, inp["b"], inp["cu_seqlens"],
                    host_cu_seqlens=inp["cu_seqlens"].cpu())
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        p.run()
    ms = []
    for _ in range(steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        p.run()
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    assert p.device_status() == 0
    t = sum(ms) / len(ms)
    T = sum(inp["lens"])
    return {"workload": w.description + ", g [T, H] (one decay per token and head)",
            "ms_per_step": t, "tokens_per_s": T / (t * 1e-3), "steps": steps}


def bench_fused(torch, kda, W, dev, steps=10):
    """prefill_8k on the fused schedule (KDA_SCHEDULE_FUSED: the intra-chunk
    pipelines and the inter-chunk chains in one kernel, the records read
    back from L2), the same inputs and results as the default separate
    kernels.  L2 flushed before every call."""
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    p = kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], inp["cu_seqlens"],
                    host_cu_seqlens=inp["cu_seqlens"].cpu(), schedule=kda.SCHEDULE_FUSED)
    path = kda.kda_prefill_schedule(p.args)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        p.run()
    ms = []
    for _ in range(steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        p.run()
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    assert p.device_status() == 0
    t = sum(ms) / len(ms)
    T = sum(inp["lens"])
    return {"workload": w.description + ", fused schedule", "path": path,
            "ms_per_step": t, "tokens_per_s": T / (t * 1e-3), "steps": steps}


def bench_overlap(torch, kda, W, dev, steps=10):
    """One 8192-token sequence of 16 heads (dk = dv = 128), where the
    automatic choice overlaps the intra-chunk kernel's last items with the
    inter-chunk chains (64 chains of 32 state columns leave 88 SMs to it),
    against the separate kernels on the same inputs.  L2 flushed before every
    call."""
    w = W.PrefillWorkload("prefill_8k_h16", None, 1, 16, 128, 128, "bf16", 11, len_range=(1, 1))
    inp = W.prefill_inputs(w, lens=[8192], device=dev, gen_device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    out = {"workload": "one 8192-token sequence x 16 heads, dk = dv = 128, bf16"}
    for name, sch in (("separate", kda.SCHEDULE_SEPARATE), ("auto", kda.SCHEDULE_AUTO)):
        p = kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], inp["cu_seqlens"],
                        host_cu_seqlens=inp["cu_seqlens"].cpu(), schedule=sch)
        for _ in range(3):
            flush_l2(flush)
            p.run()
        ms = []
        for _ in range(steps):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            p.run()
            e1.record()
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        assert p.device_status() == 0
        out[name + "_ms"] = sum(ms) / len(ms)
        out[name + "_path"] = kda.kda_prefill_schedule(p.args)
    out["tokens_per_s"] = 8192 / (out["auto_ms"] * 1e-3)
    return out


def bench_layer_steps(torch, kda, W, dev, steps=10):
    """prefill_8k with the layer steps around the recurrence: the short
    convolution (4 taps, SiLU) on q, k, v inside the intra-chunk kernel, with
    windows in and out, and the per-channel output gate inside the
    inter-chunk kernel's store.  Algorithmic bytes per token-head: 1282 of
    the prefill + 256 of gate logits (the taps and windows are a few KB per
    call).  L2 flushed before every call."""
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    T = sum(inp["lens"])
    li = W.layer_inputs(w.seed + 7, 1, T, w.H, w.dk, w.dv, 4, w.dtype, device=dev)
    p = kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], inp["cu_seqlens"],
                    host_cu_seqlens=inp["cu_seqlens"].cpu(), conv_weights=li["taps"],
                    conv_silu=True, conv_window=li["windows"], conv_window_out=True,
                    out_gate=li["gate"])
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        p.run()
    nph = kda.PREFILL_PHASES
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)]
    for e in ev:  # torch creates the cudaEvent_t on first record
        e.record()
    torch.cuda.synchronize()
    handles = (kda.c_vp * (nph + 1))(*[e.cuda_event for e in ev])
    p.args.phase_events = kda.ctypes.cast(handles, kda.c_vp)
    ms, phase = [], [[] for _ in range(nph)]
    for _ in range(steps):
        flush_l2(flush)
        p.run()
        ev[-1].synchronize()
        ms.append(ev[0].elapsed_time(ev[-1]))
        for i in range(nph):
            phase[i].append(ev[i].elapsed_time(ev[i + 1]))
    p.args.phase_events = None
    torch.cuda.synchronize()
    assert p.device_status() == 0
    t = sum(ms) / len(ms)
    return {"workload": w.description + ", short convolution (4 taps, SiLU) on q, k, v and a "
                                        "per-channel output gate",
            "ms_per_step": t, "tokens_per_s": T / (t * 1e-3), "steps": steps,
            "algorithmic_bytes": T * w.H * (1282 + 256),
            "kernels_ms": {name: sum(x) / len(x) for name, x in
                           zip(("plan", "intra_chunk", "inter_chunk_and_windows"), phase)}}


def bench_wide_heads(torch, kda, W, dev, steps=5):
    """Head sizes other than 128 (bf16, fp32 state).  64 channels: a prefill
    of one 8192-token sequence with 32 heads, on the tensor-core kernels
    zero-padded to 128, and a decode step of 1024 rows x 32 heads.  256
    channels: a prefill of one 8192-token sequence with 16 heads (CUDA-core
    path) and a decode step of 64 rows x 16 heads (256 KB of state per head,
    read and written once: 2.15 GB a step).  L2 flushed before every call."""
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        ms = []
        for _ in range(steps):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        return sum(ms) / len(ms)

    def prefill_ms(H, d):
        w = W.PrefillWorkload("head_sizes", (8192,), 1, H, d, d, "bf16", 1005)
        inp = W.prefill_inputs(w, device=dev, gen_device=dev)
        p = kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], inp["cu_seqlens"],
                        host_cu_seqlens=inp["cu_seqlens"].cpu())
        t = timed(p.run)
        assert p.device_status() == 0
        return t

    t64 = prefill_ms(32, 64)
    t_pre = prefill_ms(16, 256)

    def decode_us(B, H, d):
        dw = W.DecodeWorkload("head_sizes_decode", B, H, d, d, 1, 1006)
        di = W.decode_inputs(dw, device=dev, gen_device=dev)
        x = [di[k][0] for k in "qkvgb"]
        o = torch.empty(B, H, d, dtype=x[0].dtype, device=dev)
        st = di["state"]
        return timed(lambda: kda.kda_decode_step(*x, st, o)) * 1e3

    t_d64 = decode_us(1024, 32, 64)
    dw = W.DecodeWorkload("wide_decode", 64, 16, 256, 256, 1, 1006)
    di = W.decode_inputs(dw, device=dev, gen_device=dev)
    state = di["state"]
    x = [di[k][0] for k in "qkvgb"]
    o = torch.empty(64, 16, 256, dtype=x[0].dtype, device=dev)
    t_dec = timed(lambda: kda.kda_decode_step(*x, state, o))
    state_bytes = 2 * 64 * 16 * 256 * 256 * 4
    return {"workload": "bf16; dk = dv = 64: prefill of one 8192-token sequence x 32 heads "
                        "(tensor cores, zero-padded), decode of 1024 rows x 32 heads (ring, 4 heads "
                        "an item); dk = dv = 256: prefill of one 8192-token sequence x 16 heads "
                        "(CUDA cores), decode of 64 rows x 16 heads (ring, 256 x 64 slices)",
            "d64_prefill_ms": t64, "d64_prefill_tokens_per_s": 8192 / (t64 * 1e-3),
            "d64_decode_workload": "1024 rows x 32 heads of 64 x 64 fp32 state (1.07 GB a step)",
            "d64_decode_us": t_d64, "d64_decode_state_gbs": 2 * 1024 * 32 * 64 * 64 * 4 / (t_d64 * 1e-6) / 1e9,
            "prefill_ms": t_pre, "prefill_tokens_per_s": 8192 / (t_pre * 1e-3),
            "decode_us": t_dec * 1e3, "decode_state_gbs": state_bytes / (t_dec * 1e-3) / 1e9,
            "steps": steps}


def bench_varlen(torch, kda, W, dev, steps=10):
    """The varlen configuration: 8 packed sequences of U[1024, 32768] tokens,
    H=32, d=128, bf16, seeded fp32 initial states, fp32 snapshots every 4096
    tokens and at the boundaries (one interior position and the end of each
    sequence).  Whole prefill per call, CUDA events, L2 flushed before each."""
    w = W.WORKLOADS["varlen_8"]
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    cu, bp, cb = inp["cu_seqlens"], inp["boundary_pos"], inp["cu_boundaries"]
    p = kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], cu, initial_state=inp["S0"],
                    snapshot_interval=w.snapshot_interval, boundary_pos=bp, cu_boundaries=cb,
                    host_cu_seqlens=cu.cpu(), host_boundary_pos=bp.cpu(), host_cu_boundaries=cb.cpu())
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        p.run()
    ms = []
    for _ in range(steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        p.run()
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    assert p.device_status() == 0
    t = sum(ms) / len(ms)
    T = sum(inp["lens"])
    return {"workload": w.description, "tokens": T, "ms_per_step": t, "tokens_per_s": T / (t * 1e-3),
            "snapshots": p.n_snap, "steps": steps}


def bench_1m(torch, kda, W, dev, steps=2):
    """The million-token configuration (one sequence of 2^20 tokens, H=32,
    d=128, bf16, fp32 snapshots every 65,536 tokens): whole prefill per call
    with CUDA events; inputs 34 GB, far larger than L2."""
    w = W.WORKLOADS["prefill_1m"]
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    cu = inp["cu_seqlens"]
    p = kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], cu,
                    snapshot_interval=w.snapshot_interval, host_cu_seqlens=cu.cpu())
    p.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        p.run()
    e1.record()
    e1.synchronize()
    assert p.device_status() == 0
    ms = e0.elapsed_time(e1) / steps
    T = sum(inp["lens"])
    out = {"workload": w.description, "tokens": T, "ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3),
           "snapshots": p.n_snap, "steps": steps}
    del p, inp
    torch.cuda.empty_cache()
    return out


def bench_scan(torch, kda, W, dev, T=131072, H=2, reps=5):
    """The segment scan against the plain chunk chain on a workload it is
    for: one sequence of T tokens with few heads (bf16, 128 x 128), so that
    the plain chain keeps 4 H of the SMs busy.  Whole prefill per call,
    CUDA events, inputs (268 MB) larger than L2."""
    w = W.PrefillWorkload("scan_probe", (T,), 1, H, 128, 128, "bf16", 77)
    inp = W.prefill_inputs(w, device=dev, gen_device=dev)
    args = [inp[x] for x in "qkvgb"] + [inp["cu_seqlens"]]
    hcu = inp["cu_seqlens"].cpu()
    out = {"workload": f"one sequence, T={T}, H={H}, dk=dv=128, bf16"}
    ws = {}
    for name, P in (("plain", 1), ("scan", 0)):
        p = kda.Prefill(*args, host_cu_seqlens=hcu, scan_segments=P)
        ws[name] = p.workspace.numel()
        for _ in range(2):
            p.run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            p.run()
        e1.record()
        e1.synchronize()
        assert p.device_status() == 0
        out[f"{name}_ms"] = e0.elapsed_time(e1) / reps
    # the automatic choice as include/kda.h states it (segment scan section)
    out["segments"] = int(min(152 // (8 * H), ((T + 63) // 64) // 16, 64))
    assert ws["scan"] > ws["plain"], "the automatic choice took the segment scan"
    out["speedup"] = out["plain_ms"] / out["scan_ms"]
    out["tokens_per_s"] = T / (out["scan_ms"] * 1e-3)
    return out


def bench_decode(torch, kda, W, steps, warmup, dev):
    dw = W.DECODE_WORKLOADS[DECODE_WL]
    n = steps + warmup
    inp = W.decode_inputs(dw, steps=n, device=dev, gen_device=dev)
    state = inp["state"]
    o = torch.empty(dw.batch, dw.H, dw.dv, dtype=torch.bfloat16, device=dev)
    args = [[inp[x][s] for x in "qkvgb"] for s in range(n)]
    for s in range(warmup):
        kda.kda_decode_step(*args[s], state, o)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(warmup, n):
        kda.kda_decode_step(*args[s], state, o)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    heads = dw.batch * dw.H
    return dict(ms_per_step=ms, heads=heads, batch=dw.batch, steps=steps, workload=dw)


def bench_e2e(torch, kda, W, steps, warmup, dev):
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w)  # host tensors
    host = {x: inp[x].pin_memory() for x in "qkvgb"}
    cu = inp["cu_seqlens"]
    T = sum(inp["lens"])
    h2d = sum(host[x].numel() * host[x].element_size() for x in "qkvgb") + cu.numel() * 8
    d2h = T * w.H * w.dv * 2 + w.n_seqs * w.H * w.dk * w.dv * 4
    # the planned host-buffer call: every run copies this step's inputs in
    # from pinned host memory and o and the final state back out
    plan = kda.PrefillHost(host["q"], host["k"], host["v"], host["g"], host["b"], cu, device=dev)
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        plan.run(s)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        plan.run(s)
        s.synchronize()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    return dict(value=T / dt, unit="tokens/s", h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                ms_per_step=dt * 1e3)


def cpu_baseline(seconds_budget=20.0):
    """The oracle, as it stands, on a bounded sample of the prefill workload:
    all T=8192 tokens of the first heads that fit the time budget."""
    import oracle
    from linear_attention_serving_delta_gb300 import workloads as W
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w)
    f = lambda t: t.float().numpy()
    q, k, v, g, b = (f(inp[x]) for x in "qkvgb")
    cu = inp["cu_seqlens"].numpy()
    cores = oracle.max_threads()
    heads = min(w.H, max(cores, 1))
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, g, b, cu, heads=(0, heads))
    dt = time.perf_counter() - t0
    if dt < seconds_budget / 4 and heads < w.H:
        heads = w.H
        t0 = time.perf_counter()
        oracle.prefill(q, k, v, g, b, cu, heads=(0, heads))
        dt = time.perf_counter() - t0
    T = sum(inp["lens"])
    # tokens/s at H=32: token-heads per second / 32
    value = T * heads / w.H / dt
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"prefill_8k, all {T} tokens of {heads}/{w.H} heads, fp64, {dt:.2f} s"}


def max_over_ranks(dist, world, values, device):
    """Each rank's per-step times reduced to their maximum over the ranks (the
    slowest replica sets the whole job's step time)."""
    if world <= 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tokens_per_s(world, tokens_per_replica, step_ms):
    """Throughput of N independent replicas (weak scaling): the tokens all
    ranks processed per step over the slowest rank's step time."""
    return world * tokens_per_replica / (step_ms * 1e-3)


def gpu_arm(a):
    import torch
    import torch.distributed as dist
    from linear_attention_serving_delta_gb300 import kda
    from linear_attention_serving_delta_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(dev))
    kda.lib()
    pk = peaks()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    if a.layer_only:
        print(json.dumps(bench_layer_steps(torch, kda, W, dev, steps=a.steps)))
        return
    if a.fused_only:
        print(json.dumps(bench_fused(torch, kda, W, dev, steps=a.steps)))
        return
    if a.overlap_only:
        print(json.dumps(bench_overlap(torch, kda, W, dev, steps=a.steps)))
        return
    if a.wide_only:
        print(json.dumps(bench_wide_heads(torch, kda, W, dev, steps=a.steps)))
        return
    if a.decode_only:
        dec = bench_decode(torch, kda, W, a.decode_steps, a.warmup, dev)
        gbs = DECODE_STATE_BYTES_PER_HEAD * dec["heads"] / (dec["ms_per_step"] * 1e-3) / 1e9
        print(json.dumps({"decode_us_per_step": dec["ms_per_step"] * 1e3, "state_gbs": gbs}))
        return
    if a.prep_only:
        print(json.dumps(bench_prep(torch, kda, W, dev, reps=a.steps)))
        return
    with ClockSampler(local) as clk:
        pre = bench_prefill(torch, kda, W, a.steps, a.warmup, dev)
        barrier()
        if a.prefill_only:
            print(json.dumps({"prefill_ms_per_step": sum(pre["step_ms"]) / len(pre["step_ms"]),
                              "path": pre["path"],
                              "separate_ms_per_step": sum(pre["separate_step_ms"]) / len(pre["separate_step_ms"]),
                              "separate_phase_ms": [sum(x) / len(x) for x in pre["phase_ms"]]}))
            return
        dec = bench_decode(torch, kda, W, a.decode_steps, max(3, a.warmup), dev)
        barrier()
    step_ms = sum(pre["step_ms"]) / len(pre["step_ms"])
    dec_ms = dec["ms_per_step"]
    step_ms, dec_ms = max_over_ranks(dist, world, [step_ms, dec_ms], dev)
    e2e = bench_e2e(torch, kda, W, max(1, min(a.steps, 5)), 1, dev) if rank == 0 else None
    scan = bench_scan(torch, kda, W, dev) if rank == 0 else None
    prep = bench_prep(torch, kda, W, dev) if rank == 0 else None
    m1 = bench_1m(torch, kda, W, dev) if rank == 0 and not a.no_1m else None
    vl = bench_varlen(torch, kda, W, dev) if rank == 0 else None
    gph = bench_gate_per_head(torch, kda, W, dev) if rank == 0 else None
    fus = bench_fused(torch, kda, W, dev) if rank == 0 else None
    ovl = bench_overlap(torch, kda, W, dev) if rank == 0 else None
    lay = bench_layer_steps(torch, kda, W, dev) if rank == 0 else None
    wide = bench_wide_heads(torch, kda, W, dev) if rank == 0 else None
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    T, H = pre["T"], pre["H"]
    value = whole_job_tokens_per_s(world, T, step_ms)
    ph = [sum(x) / len(x) for x in pre["phase_ms"]]
    sep_ms = sum(pre["separate_step_ms"]) / len(pre["separate_step_ms"])
    names = ["plan", "intra_chunk", "inter_chunk"]
    chunk_heads = pre["n_chunks"] * H
    r3 = lambda x: float(f"{x:.4g}")
    intra_tflops = INTRA_FLOP_PER_CHUNK_HEAD * chunk_heads / (ph[1] * 1e-3) / 1e12
    inter_tflops = INTER_FLOP_PER_CHUNK_HEAD * chunk_heads / (ph[2] * 1e-3) / 1e12
    intra_gbs = INTRA_BYTES_PER_CHUNK_HEAD * chunk_heads / (ph[1] * 1e-3) / 1e9
    prefill_gbs = PREFILL_BYTES_PER_TOKEN_HEAD * T * H / (step_ms * 1e-3) / 1e9
    # per-kernel times: the separate kernels, one after the other
    kernels = {
        "plan": {"ms": r3(ph[0])},
        "intra_chunk": {"ms": r3(ph[1]), "tflops": r3(intra_tflops),
                        "tensor_frac": r3(intra_tflops / pk["bf16_tflops"]),
                        "input_gbs": r3(intra_gbs), "input_hbm_frac": r3(intra_gbs / pk["hbm_gbs"])},
        "inter_chunk": {"ms": r3(ph[2]), "tflops": r3(inter_tflops),
                        "tensor_frac": r3(inter_tflops / pk["bf16_tflops"]),
                        "us_per_chunk_step": r3(ph[2] * 1e3 / pre["n_chunks"])},
    }
    for n, m in zip(names, ph):
        kernels[n]["share"] = r3(m / max(sum(ph), 1e-12))
    record_bytes = RECORD_BYTES * chunk_heads
    # The dominant kernel against its roofline as the scope table gives it:
    # the intra-chunk kernel is a dense contraction (tensor pipe, burst peak:
    # it is timed alone inside a sub-millisecond step); the inter-chunk kernel
    # is a latency-bound chain, reported against the tensor pipe too, with its
    # microseconds per chunk step beside it.
    dom = 1 if ph[1] >= ph[2] else 2
    flops = (INTRA_FLOP_PER_CHUNK_HEAD if dom == 1 else INTER_FLOP_PER_CHUNK_HEAD) * chunk_heads
    tfl = flops / (ph[dom] * 1e-3) / 1e12
    roof = {"kernel": names[dom], "bound": "tensor", "achieved": r3(tfl), "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": r3(tfl / pk["bf16_tflops"]),
            "traffic": ncu_traffic("tc_intra" if dom == 1 else "tc_inter", PREFILL_WL),
            "flop_per_chunk_head": (INTRA_FLOP_PER_CHUNK_HEAD if dom == 1 else INTER_FLOP_PER_CHUNK_HEAD),
            "chunk_heads_per_launch": chunk_heads,
            "algorithmic_bytes_per_launch": (INTRA_BYTES_PER_CHUNK_HEAD if dom == 1
                                             else INTER_BYTES_PER_CHUNK_HEAD) * chunk_heads,
            "traffic_overhead": record_bytes,
            "peak_source": pk["source"] + " (bf16 burst)"}
    dec_gbs = DECODE_STATE_BYTES_PER_HEAD * dec["heads"] / (dec_ms * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill_8k: B=1 H=32 T=8192 dk=dv=128 bf16 in, fp32 state, C=64",
                   "global_batch": world, "seq_len": T, "heads": H, "dk": 128, "dv": 128,
                   "chunk": 64, "parallelism": f"replicas{world}",
                   "l2": "512 MB buffer written between timed steps (inputs 268 MB > L2)",
                   "decode_workload": "decode_256: 256 seqs x H=32, fp32 128x128 states "
                                      "(537 MB), 1000 steps"},
        "roofline": roof,
        "e2e": {"value": e2e["value"], "unit": e2e["unit"],
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "ms_per_step": r3(e2e["ms_per_step"])},
        "gpu_launches": pre["launches_per_step"] * a.steps + dec["steps"],
        "clocks": clk.summary(),
        # the default call against the separate kernels timed with phase
        # events between them (the per-kernel split below)
        "prefill_schedule": {"path": {kda.PATH_OVERLAP: "overlapped", kda.PATH_SEPARATE: "separate",
                                      kda.PATH_FUSED: "fused"}.get(pre["path"], str(pre["path"])),
                             "separate_with_phase_events_ms": r3(sep_ms),
                             "vs_separate_with_phase_events": r3(sep_ms / step_ms)},
        "kernels": kernels,
        "decode": {"us_per_step": r3(dec_ms * 1e3), "state_gbs": r3(dec_gbs),
                   "tokens_per_s": r3(world * dec["batch"] / (dec_ms * 1e-3)),
                   "roofline": {"bound": "hbm", "achieved": r3(dec_gbs), "peak": pk["hbm_gbs"],
                                "unit": "GB/s", "frac": r3(dec_gbs / pk["hbm_gbs"]),
                                "traffic": ncu_traffic("decode_ring", DECODE_WL),
                                "algorithmic_bytes_per_launch": DECODE_STATE_BYTES_PER_HEAD * dec["heads"]},
                   "steps": dec["steps"]},
        "prefill_varlen": {"tokens": vl["tokens"], "ms": r3(vl["ms_per_step"]),
                           "tokens_per_s": r3(vl["tokens_per_s"]), "snapshots": vl["snapshots"]},
        "prefill_gate_per_head": {"ms": r3(gph["ms_per_step"]), "tokens_per_s": r3(gph["tokens_per_s"])},
        "prefill_fused": {"ms": r3(fus["ms_per_step"]), "tokens_per_s": r3(fus["tokens_per_s"]),
                          "fused_path": fus["path"] == kda.PATH_FUSED,
                          "vs_separate": r3(sep_ms / fus["ms_per_step"])},
        "prefill_overlap_h16": {"separate_ms": r3(ovl["separate_ms"]), "ms": r3(ovl["auto_ms"]),
                                "overlapped": ovl["auto_path"] == kda.PATH_OVERLAP,
                                "tokens_per_s": r3(ovl["tokens_per_s"]),
                                "vs_separate": r3(ovl["separate_ms"] / ovl["auto_ms"])},
        "prefill_layer_steps": {"ms": r3(lay["ms_per_step"]), "tokens_per_s": r3(lay["tokens_per_s"]),
                                "kernels_ms": {k: r3(v) for k, v in lay["kernels_ms"].items()}},
        "wide_heads": {k: (r3(v) if isinstance(v, float) else v) for k, v in wide.items()
                       if k not in ("workload", "d64_decode_workload")},
        "segment_scan": {k: (r3(v) if isinstance(v, float) else v) for k, v in scan.items()
                         if k != "workload"},
        "prep": {"us": r3(prep["us"]), "gbs": r3(prep["achieved_gbs"]),
                 "hbm_frac": r3(prep["achieved_gbs"] / pk["hbm_gbs"]),
                 "traffic": ncu_traffic("prep_vec", PREFILL_WL)},
    }
    if m1:
        out["prefill_1m"] = {"tokens": m1["tokens"], "ms": r3(m1["ms_per_step"]),
                             "tokens_per_s": r3(m1["tokens_per_s"]), "snapshots": m1["snapshots"],
                             "steps": m1["steps"]}
    if not a.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline()
    # the headline figures once more as short top-level keys at the end of the
    # line (a reader that keeps only the tail of the output still has them)
    out["headline"] = {
        "prefill_8k_tokens_per_s": r3(value), "prefill_hbm_frac": r3(prefill_gbs / pk["hbm_gbs"]),
        "intra_tensor_frac": kernels["intra_chunk"]["tensor_frac"],
        "inter_us_per_chunk_step": kernels["inter_chunk"]["us_per_chunk_step"],
        "decode_state_gbs": r3(dec_gbs), "decode_hbm_frac": r3(dec_gbs / pk["hbm_gbs"]),
        "prefill_1m_tokens_per_s": out["prefill_1m"]["tokens_per_s"] if m1 else None,
        "prefill_varlen_tokens_per_s": r3(vl["tokens_per_s"]),
        "e2e_tokens_per_s": r3(e2e["value"]),
    }
    print(json.dumps(out, separators=(",", ":")), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm
def reference_arm(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from linear_attention_serving_delta_gb300 import workloads as W
    oracle.build()
    w = W.WORKLOADS[PREFILL_WL]
    inp = W.prefill_inputs(w)
    f = lambda t: t.float().numpy()
    q, k, v, g, b = (f(inp[x]) for x in "qkvgb")
    cu = inp["cu_seqlens"].numpy()
    T = sum(inp["lens"])
    cores = oracle.max_threads()
    heads = min(w.H, max(1, cores))       # one head per core: a bounded sample per step
    for _ in range(a.warmup):
        oracle.prefill(q, k, v, g, b, cu, heads=(0, heads))
    t0 = time.perf_counter()
    for _ in range(a.steps):
        oracle.prefill(q, k, v, g, b, cu, heads=(0, heads))
    dt = (time.perf_counter() - t0) / a.steps
    value = T * heads / w.H / dt
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": a.steps,
           "warmup": a.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.description, "global_batch": 1, "seq_len": T,
                      "heads_per_step": heads, "parallelism": "cpu-oracle"},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": f"all {T} tokens of {heads}/{w.H} heads per step"},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--overlap-only", action="store_true",
                    help="only the 16-head prefill, separate and overlapped kernels (profiling)")
    ap.add_argument("--no-1m", action="store_true",
                    help="skip the million-token configuration (~100 GB of device memory)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time the prefill workload alone (for profiler captures)")
    ap.add_argument("--layer-only", action="store_true",
                    help="time the prefill with the layer steps alone (for profiler captures)")
    ap.add_argument("--fused-only", action="store_true",
                    help="time the prefill on the fused schedule alone (for profiler captures)")
    ap.add_argument("--wide-only", action="store_true",
                    help="time the 256-channel heads alone")
    ap.add_argument("--decode-only", action="store_true",
                    help="time the decode workload alone (for profiler captures)")
    ap.add_argument("--prep-only", action="store_true",
                    help="time the preparation step alone (for profiler captures)")
    a = ap.parse_args()
    if a.warmup < 3:
        a.warmup = 3
    if a.impl == "reference":
        reference_arm(a)
    else:
        gpu_arm(a)


if __name__ == "__main__":
    main()
