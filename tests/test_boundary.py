"""Host-side checks of the C-ABI library (no GPU needed).

* libkda.so builds for sm_103a and loads;
* it exports every function include/kda.h declares;
* the ctypes structures of the binding have the C layout (sizes and offsets
  from a C program compiled against kda.h);
* argument validation rejects bad arguments before any launch;
* the host snapshot plan agrees with the oracle's definition of the
  snapshot positions.
"""
import ctypes
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def kda():
    from linear_attention_serving_delta_gb300 import build, kda as binding
    build.build()
    binding.lib()
    return binding


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_function(kda):
    names = declared_functions()
    assert len(names) >= 8
    L = kda.lib()
    for n in names:
        assert hasattr(L, n), f"{n} declared in kda.h but not exported"
    assert set(names) == set(kda.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", kda.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), f"{n} not a defined text symbol"


def test_struct_layouts_match_c(kda, tmp_path):
    prog = r'''
#include <stdio.h>
#include <stddef.h>
#include "kda.h"
#define F(T, m) printf(#T "." #m " %zu\n", offsetof(T, m));
int main(void) {
  printf("kda_prefill_args %zu\n", sizeof(kda_prefill_args));
  printf("kda_decode_args %zu\n", sizeof(kda_decode_args));
  printf("kda_prep_args %zu\n", sizeof(kda_prep_args));
  printf("kda_prefill_host_args %zu\n", sizeof(kda_prefill_host_args));
  printf("kda_layer_args %zu\n", sizeof(kda_layer_args));
  printf("const.KDA_CONV_MAX %d\n", KDA_CONV_MAX);
  printf("const.KDA_CHUNK %d\n", KDA_CHUNK);
  printf("const.KDA_PREFILL_PHASES %d\n", KDA_PREFILL_PHASES);
  printf("const.KDA_SCHEDULE_AUTO %d\n", KDA_SCHEDULE_AUTO);
  printf("const.KDA_SCHEDULE_SEPARATE %d\n", KDA_SCHEDULE_SEPARATE);
  printf("const.KDA_SCHEDULE_FUSED %d\n", KDA_SCHEDULE_FUSED);
  printf("const.KDA_SCHEDULE_OVERLAP %d\n", KDA_SCHEDULE_OVERLAP);
  printf("const.KDA_PATH_OVERLAP %d\n", KDA_PATH_OVERLAP);
  printf("const.KDA_PATH_CUDA_CORES %d\n", KDA_PATH_CUDA_CORES);
  printf("const.KDA_PATH_SEPARATE %d\n", KDA_PATH_SEPARATE);
  printf("const.KDA_PATH_FUSED %d\n", KDA_PATH_FUSED);
  printf("const.KDA_PATH_SEGMENT_SCAN %d\n", KDA_PATH_SEGMENT_SCAN);
  F(kda_layer_args, conv_silu) F(kda_layer_args, conv_w) F(kda_layer_args, conv_in)
  F(kda_layer_args, conv_out) F(kda_layer_args, out_gate) F(kda_layer_args, out_gate_per_head)
  F(kda_prefill_args, layer) F(kda_decode_args, layer) F(kda_prep_args, layer)
  F(kda_prefill_host_args, cu_seqlens) F(kda_prefill_host_args, in_dtype)
  F(kda_prefill_host_args, scale) F(kda_prefill_host_args, final_state)
  F(kda_prefill_host_args, segments) F(kda_prefill_host_args, copy_in_stream)
  F(kda_prefill_host_args, copy_out_stream)
  F(kda_prefill_args, cu_seqlens) F(kda_prefill_args, in_dtype) F(kda_prefill_args, q)
  F(kda_prefill_args, scale) F(kda_prefill_args, initial_state)
  F(kda_prefill_args, snapshot_interval) F(kda_prefill_args, num_boundaries)
  F(kda_prefill_args, snapshots) F(kda_prefill_args, num_snapshots)
  F(kda_prefill_args, phase_events) F(kda_prefill_args, scan_segments)
  F(kda_prefill_args, snapshot_slot_map) F(kda_prefill_args, wait_limit_ns)
  F(kda_prefill_args, gate_per_head) F(kda_prefill_args, schedule) F(kda_decode_args, gate_per_head)
  F(kda_prep_args, gate_per_head) F(kda_prefill_host_args, gate_per_head)
  F(kda_decode_args, scale) F(kda_decode_args, q) F(kda_decode_args, state_slots)
  F(kda_decode_args, o) F(kda_decode_args, wait_limit_ns) F(kda_decode_args, status)
  F(kda_prep_args, total_tokens) F(kda_prep_args, in_dtype) F(kda_prep_args, beta)
  return 0;
}
'''
    c = tmp_path / "layout.c"
    c.write_text(prog)
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(c), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(l.rsplit(" ", 1) for l in lines if l)
    structs = {"kda_prefill_args": kda.PrefillArgs, "kda_decode_args": kda.DecodeArgs,
               "kda_prep_args": kda.PrepArgs, "kda_prefill_host_args": kda.PrefillHostArgs,
               "kda_layer_args": kda.LayerArgs}
    consts = {"KDA_CONV_MAX": kda.CONV_MAX, "KDA_CHUNK": kda.CHUNK,
              "KDA_PREFILL_PHASES": kda.PREFILL_PHASES,
              "KDA_SCHEDULE_AUTO": kda.SCHEDULE_AUTO, "KDA_SCHEDULE_SEPARATE": kda.SCHEDULE_SEPARATE,
              "KDA_SCHEDULE_FUSED": kda.SCHEDULE_FUSED, "KDA_SCHEDULE_OVERLAP": kda.SCHEDULE_OVERLAP,
              "KDA_PATH_OVERLAP": kda.PATH_OVERLAP,
              "KDA_PATH_CUDA_CORES": kda.PATH_CUDA_CORES, "KDA_PATH_SEPARATE": kda.PATH_SEPARATE,
              "KDA_PATH_FUSED": kda.PATH_FUSED, "KDA_PATH_SEGMENT_SCAN": kda.PATH_SEGMENT_SCAN}
    for key, val in got.items():
        if key.startswith("const."):
            assert consts[key[6:]] == int(val), key
        elif "." in key:
            s, m = key.split(".")
            assert getattr(structs[s], m).offset == int(val), key
        else:
            assert ctypes.sizeof(structs[key]) == int(val), key


def _args(kda, **over):
    a = kda.PrefillArgs()
    a.num_seqs, a.num_heads, a.dk, a.dv, a.total_tokens = 1, 2, 16, 16, 64
    a.cu_seqlens = 0x1000
    a.in_dtype = kda.KDA_F32
    a.q = a.k = a.v = a.g = a.b = a.o = 0x2000
    a.scale = 1.0
    for k_, v_ in over.items():
        setattr(a, k_, v_)
    return a


def test_workspace_size_and_validation(kda):
    L = kda.lib()
    good = _args(kda)
    ws = L.kda_prefill_workspace_size(ctypes.byref(good))
    assert ws > 0 and ws % 256 == 0
    # invalid arguments: size query returns 0 and the call returns a status, no launch
    for bad, code in [(dict(dk=24), 2), (dict(dv=512), 2), (dict(num_seqs=0), 1),
                      (dict(cu_seqlens=None), 1), (dict(q=None), 1),
                      (dict(snapshot_interval=100), 1), (dict(snapshot_interval=-64), 1),
                      (dict(boundary_pos=0x3000), 1), (dict(snapshots=0x3000), 1),
                      (dict(in_dtype=7), 1), (dict(total_tokens=-1), 1)]:
        a = _args(kda, **bad)
        assert L.kda_prefill_workspace_size(ctypes.byref(a)) == 0, bad
        assert L.kda_prefill(ctypes.byref(a), 0x4000, 1 << 30, None) == code, bad
    # workspace too small / missing / misaligned
    assert L.kda_prefill(ctypes.byref(good), None, ws, None) == 3
    assert L.kda_prefill(ctypes.byref(good), 0x4000, ws - 256, None) == 3
    assert L.kda_prefill(ctypes.byref(good), 0x4010, ws, None) == 3
    # bf16 heads of 64 channels take the tensor-core path (zero-padded to 128:
    # its 90,624-byte record per chunk-head), fp32 ones the CUDA-core path
    # (82,176 bytes): 2 chunk-table entries (64 tokens + one per sequence) x 2 heads
    tcp = _args(kda, in_dtype=kda.KDA_BF16, dk=64, dv=64, schedule=kda.SCHEDULE_SEPARATE)
    cup = _args(kda, dk=64, dv=64)
    assert (L.kda_prefill_workspace_size(ctypes.byref(tcp)) -
            L.kda_prefill_workspace_size(ctypes.byref(cup))) == 2 * 2 * (90624 - 82176)
    # the fused kernel reads the same record array; only its flags are added
    # (2 chunk-table entries x 2 heads, one 256-byte block); the overlapped
    # kernels (the automatic choice for one sequence) add the flags and their
    # counters (8 + 8 + 2 x 512 x 4 bytes, in 256-byte blocks); with several
    # sequences nothing is added; an unknown schedule is rejected
    fused = _args(kda, in_dtype=kda.KDA_BF16, dk=64, dv=64, schedule=kda.SCHEDULE_FUSED)
    auto = _args(kda, in_dtype=kda.KDA_BF16, dk=64, dv=64)
    ovl = _args(kda, in_dtype=kda.KDA_BF16, dk=64, dv=64, schedule=kda.SCHEDULE_OVERLAP)
    assert (L.kda_prefill_workspace_size(ctypes.byref(fused)) -
            L.kda_prefill_workspace_size(ctypes.byref(tcp))) == 256
    counters = -(-(16 + 2 * 512 * 4) // 256) * 256
    for a in (auto, ovl):
        assert (L.kda_prefill_workspace_size(ctypes.byref(a)) -
                L.kda_prefill_workspace_size(ctypes.byref(tcp))) == 256 + counters
    two = dict(in_dtype=kda.KDA_BF16, dk=64, dv=64, num_seqs=2)
    assert (L.kda_prefill_workspace_size(ctypes.byref(_args(kda, **two))) ==
            L.kda_prefill_workspace_size(ctypes.byref(_args(kda, schedule=kda.SCHEDULE_SEPARATE, **two))))
    a = _args(kda, schedule=4)
    assert L.kda_prefill_workspace_size(ctypes.byref(a)) == 0
    assert L.kda_prefill(ctypes.byref(a), 0x4000, 1 << 30, None) == 1
    # heads of 256 channels are taken (the CUDA-core path's blocked kernel)
    wide = _args(kda, dk=256, dv=256)
    assert L.kda_prefill_workspace_size(ctypes.byref(wide)) > ws
    # the workspace grows with tokens, sequences and boundaries
    big = _args(kda, total_tokens=8192)
    assert L.kda_prefill_workspace_size(ctypes.byref(big)) > ws
    # segment scan: out-of-range counts are rejected; on the tensor-core path
    # (bf16, 128 x 128) with few heads and one long sequence it adds its
    # per-segment state buffers (4 x P x H x 64 KB)
    a = _args(kda, gate_per_head=2)
    assert L.kda_prefill_workspace_size(ctypes.byref(a)) == 0
    a = _args(kda, wait_limit_ns=-1)
    assert L.kda_prefill_workspace_size(ctypes.byref(a)) == 0
    assert L.kda_prefill(ctypes.byref(a), 0x4000, 1 << 30, None) == 1
    for bad in (-1, 65):
        a = _args(kda, scan_segments=bad)
        assert L.kda_prefill_workspace_size(ctypes.byref(a)) == 0
        assert L.kda_prefill(ctypes.byref(a), 0x4000, 1 << 30, None) == 1
    tc = dict(in_dtype=kda.KDA_BF16, dk=128, dv=128, num_heads=2, total_tokens=65536)
    off = L.kda_prefill_workspace_size(ctypes.byref(_args(kda, scan_segments=1, **tc)))
    auto = L.kda_prefill_workspace_size(ctypes.byref(_args(kda, **tc)))
    four = L.kda_prefill_workspace_size(ctypes.byref(_args(kda, scan_segments=4, **tc)))
    mat = 2 * 128 * 128 * 4
    assert four - off >= 4 * 4 * mat and auto - off >= 4 * 9 * mat  # auto: 152 // 16 = 9
    # never with several sequences, snapshots, or on the fp32 path
    assert L.kda_prefill_workspace_size(ctypes.byref(_args(kda, scan_segments=4))) == ws
    assert L.kda_prefill(None, 0x4000, ws, None) == 1
    assert kda.kda_status_string(3).startswith("workspace")


def test_prefill_schedule(kda):
    """The path a prefill takes (kda_prefill_schedule, host logic only, for a
    given SM count): by default the overlapped tensor-core kernels for one
    sequence whose chains (heads x dv / 32) number 40 to half the SMs (with
    schedule = OVERLAP any number up to half the SMs), else the separate
    kernels; with schedule = FUSED the fused kernel where its chains
    (sequences x heads x dv / 32) are at most as many as the SMs; the segment
    scan and the fp32 CUDA-core path where they apply."""
    L = kda.lib()
    bf = dict(in_dtype=kda.KDA_BF16, dk=128, dv=128)
    fu = dict(schedule=kda.SCHEDULE_FUSED)
    ov = dict(schedule=kda.SCHEDULE_OVERLAP)

    def path(sms=152, **over):
        return L.kda_prefill_schedule(ctypes.byref(_args(kda, **over)), sms)

    assert path(num_heads=32, total_tokens=8192, **bf) == kda.PATH_SEPARATE       # 128 chains
    assert path(num_heads=32, total_tokens=8192, **ov, **bf) == kda.PATH_SEPARATE
    assert path(num_heads=16, total_tokens=8192, **bf) == kda.PATH_OVERLAP        # 64 chains
    assert path(num_heads=19, total_tokens=8192, **bf) == kda.PATH_OVERLAP        # 76 chains
    assert path(num_heads=20, total_tokens=8192, **bf) == kda.PATH_SEPARATE       # 80 chains
    assert path(num_heads=10, total_tokens=8192, **bf) == kda.PATH_OVERLAP        # 40 chains
    assert path(num_heads=8, total_tokens=8192, **bf) == kda.PATH_SEPARATE        # 32 chains
    assert path(num_heads=8, total_tokens=8192, **ov, **bf) == kda.PATH_OVERLAP
    assert path(sms=128, num_heads=16, total_tokens=8192, **bf) == kda.PATH_OVERLAP
    assert path(sms=127, num_heads=16, total_tokens=8192, **bf) == kda.PATH_SEPARATE
    assert path(num_seqs=2, num_heads=8, total_tokens=8192, **bf) == kda.PATH_SEPARATE
    assert path(num_heads=16, total_tokens=8192, wait_limit_ns=1000, **bf) == kda.PATH_SEPARATE
    assert path(num_heads=16, total_tokens=8192, wait_limit_ns=100000, **bf) == kda.PATH_OVERLAP
    assert path(num_heads=16, total_tokens=0, **bf) == kda.PATH_SEPARATE          # nothing to overlap
    assert path(num_heads=32, total_tokens=8192, in_dtype=kda.KDA_BF16, dk=64, dv=64) == kda.PATH_OVERLAP
    assert path(num_heads=2, total_tokens=65536, **bf) == kda.PATH_SEGMENT_SCAN
    assert path(num_heads=2, total_tokens=65536, scan_segments=1, **ov, **bf) == kda.PATH_OVERLAP
    assert path(num_heads=32, total_tokens=8192, schedule=kda.SCHEDULE_SEPARATE, **bf) == kda.PATH_SEPARATE
    assert path(num_heads=32, total_tokens=8192, **fu, **bf) == kda.PATH_FUSED    # 128 chains
    assert path(num_heads=38, total_tokens=8192, **fu, **bf) == kda.PATH_FUSED    # 152 chains
    assert path(num_heads=39, total_tokens=8192, **fu, **bf) == kda.PATH_SEPARATE  # 156 chains
    assert path(sms=100, num_heads=32, total_tokens=8192, **fu, **bf) == kda.PATH_SEPARATE
    assert path(num_seqs=8, num_heads=32, total_tokens=8192, **fu, **bf) == kda.PATH_SEPARATE
    assert path(num_heads=32, total_tokens=8192, in_dtype=kda.KDA_BF16, dk=64, dv=64, **fu) == kda.PATH_FUSED
    assert path(num_heads=32, total_tokens=8192, in_dtype=kda.KDA_BF16, dk=128, dv=32, **fu) == kda.PATH_FUSED
    assert path(num_heads=32, total_tokens=0, **fu, **bf) == kda.PATH_SEPARATE    # nothing to fuse
    assert path(num_heads=32, total_tokens=8192, **fu) == kda.PATH_CUDA_CORES     # fp32
    assert path(num_heads=2, total_tokens=65536, **fu, **bf) == kda.PATH_SEGMENT_SCAN
    assert path(num_heads=2, total_tokens=65536, scan_segments=1, **fu, **bf) == kda.PATH_FUSED
    assert path(num_seqs=0) == -1 and path(sms=-1) == -1


def test_layer_args_validation(kda):
    """The short convolution and output gate arguments are checked on the
    host: width outside 0..KDA_CONV_MAX, missing taps, a flag outside {0, 1},
    and input/output windows that partly overlap are rejected before any
    launch (a window updated in place, out == in, is allowed)."""
    L = kda.lib()
    W = 4
    rows_bytes = 1 * (W - 1) * 2 * 16 * 4  # N x (W-1) x H x d x fp32, per tensor

    def layer(**over):
        la = kda.LayerArgs()
        la.conv_width = W
        for t in range(3):
            la.conv_w[t] = 0x5000 + 0x100 * t
        for k_, v_ in over.items():
            setattr(la, k_, v_)
        return la

    def prefill_status(la):
        a = _args(kda)
        a.layer = ctypes.pointer(la)
        return L.kda_prefill_workspace_size(ctypes.byref(a)), a

    ok_ws, _ = prefill_status(layer())
    assert ok_ws == L.kda_prefill_workspace_size(ctypes.byref(_args(kda)))  # no extra workspace
    for bad in (dict(conv_width=5), dict(conv_width=-1), dict(out_gate_per_head=2)):
        ws, a = prefill_status(layer(**bad))
        assert ws == 0, bad
        assert L.kda_prefill(ctypes.byref(a), 0x4000, 1 << 30, None) == 1, bad
    la = layer()
    la.conv_w[1] = None                                            # a missing tap tensor
    assert prefill_status(la)[0] == 0
    la = layer()                                                   # windows partly overlapping
    la.conv_in[0], la.conv_out[0] = 0x10000, 0x10000 + rows_bytes // 2
    assert prefill_status(la)[0] == 0
    la.conv_out[0] = 0x10000                                       # in place: allowed
    assert prefill_status(la)[0] > 0
    la.conv_out[0] = 0x10000 + rows_bytes                          # adjacent: allowed
    assert prefill_status(la)[0] > 0
    la = layer(conv_width=0)                                       # off: taps not needed
    for t in range(3):
        la.conv_w[t] = None
    assert prefill_status(la)[0] > 0
    # decode: the same checks against the slot pool
    d = kda.DecodeArgs()
    d.batch, d.num_heads, d.dk, d.dv, d.num_slots = 4, 1, 16, 16, 4
    d.q = d.k = d.v = d.g = d.b = d.o = 0x2000
    d.state = 0x3000
    d.layer = ctypes.pointer(layer(conv_width=7))
    assert L.kda_decode_step(ctypes.byref(d), None) == 1
    # the convolution in decode needs dk * dv <= 128 * 128 (wider heads run as
    # several CTAs per row and head, which would race on an in-place window)
    d.dk = d.dv = 256
    d.layer = ctypes.pointer(layer())
    assert L.kda_decode_step(ctypes.byref(d), None) == 2


def test_decode_and_prep_validation(kda):
    L = kda.lib()
    d = kda.DecodeArgs()
    d.batch, d.num_heads, d.dk, d.dv, d.num_slots = 0, 1, 128, 128, 0
    assert L.kda_decode_step(ctypes.byref(d), None) == 0          # empty batch: nothing to do
    d.batch, d.num_slots = 4, 4
    assert L.kda_decode_step(ctypes.byref(d), None) == 1          # null pointers
    d.q = d.k = d.v = d.g = d.b = d.o = 0x2000
    d.state = 0x3008                                               # misaligned state
    assert L.kda_decode_step(ctypes.byref(d), None) == 1
    d.state = 0x3000
    d.num_slots = 2                                                # pool smaller than batch
    assert L.kda_decode_step(ctypes.byref(d), None) == 1
    d.num_slots = 4
    d.wait_limit_ns = -1                                           # negative wait limit
    assert L.kda_decode_step(ctypes.byref(d), None) == 1
    d.wait_limit_ns = 0
    d.dk = 96
    assert L.kda_decode_step(ctypes.byref(d), None) == 2
    p = kda.PrepArgs()
    p.num_seqs, p.num_heads, p.dk, p.total_tokens = 1, 1, 20, 4
    assert L.kda_prep(ctypes.byref(p), None) == 2
    assert L.kda_decode_step(None, None) == 1
    assert L.kda_prep(None, None) == 1


def test_snapshot_plan_matches_oracle_definition(kda, oracle_mod):
    rng = np.random.default_rng(5)
    for trial in range(20):
        n = int(rng.integers(1, 6))
        lens = rng.integers(0, 300, size=n)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        interval = int(rng.choice([0, 64, 128]))
        bpos, cub = [], [0]
        for L in lens:
            k = int(rng.integers(0, 4)) if L > 0 else 0
            pts = sorted(set(int(x) for x in rng.integers(1, L + 1, size=k))) if L > 0 else []
            bpos += pts
            cub.append(len(bpos))
        use_b = bool(rng.integers(0, 2))
        bp = np.array(bpos, np.int64) if use_b else None
        cb = np.array(cub, np.int64) if use_b else None
        cs, n_snap = kda.kda_snapshot_plan(cu, interval, bp, cb)
        pos, cs_ref = oracle_mod.snapshot_positions(lens, interval, bp, cb)
        assert list(cs) == list(cs_ref)
        assert n_snap == len(pos)
    with pytest.raises(ValueError):
        kda.kda_snapshot_plan([0, 10], 0, [5, 5], [0, 2])      # not strictly increasing
    with pytest.raises(ValueError):
        kda.kda_snapshot_plan([0, 10], 0, [11], [0, 1])        # beyond the sequence


def _host_args(kda, cu, **over):
    a = kda.PrefillHostArgs()
    a.num_seqs, a.num_heads, a.dk, a.dv = len(cu) - 1, 2, 128, 128
    a.total_tokens = int(cu[-1])
    a.cu_seqlens = cu.ctypes.data
    a.in_dtype = kda.KDA_BF16
    a.q = a.k = a.v = a.g = a.b = a.o = 0x2000
    a.scale = 1.0
    a.copy_in_stream, a.copy_out_stream = 0x10, 0x20
    for k_, v_ in over.items():
        setattr(a, k_, v_)
    return a


def test_host_entry_workspace_and_validation(kda):
    """kda_prefill_host: its workspace holds the device copies of every
    tensor, and host-side validation (cu_seqlens read on the host, streams,
    segment count) rejects bad arguments before any CUDA call."""
    L = kda.lib()
    T, H = 8192, 2
    cu = np.array([0, T], dtype=np.int64)
    good = _host_args(kda, cu)
    ws = L.kda_prefill_host_workspace_size(ctypes.byref(good))
    tensors = T * H * 128 * 2 * 5 + T * H * 2 + 3 * H * 128 * 128 * 4
    assert ws % 256 == 0 and ws > tensors
    # more pieces of one sequence: the per-piece prefill workspace shrinks
    one = L.kda_prefill_host_workspace_size(ctypes.byref(_host_args(kda, cu, segments=1)))
    eight = L.kda_prefill_host_workspace_size(ctypes.byref(_host_args(kda, cu, segments=8)))
    assert one > eight > tensors
    multi = np.array([0, 100, 100, 3000, T], dtype=np.int64)
    assert L.kda_prefill_host_workspace_size(ctypes.byref(_host_args(kda, multi, segments=3))) > 0
    bad_cus = [np.array([1, T], dtype=np.int64), np.array([0, 10, 5, T], dtype=np.int64),
               np.array([0, T - 1], dtype=np.int64)]
    for bad_cu in bad_cus:
        a = _host_args(kda, bad_cu)
        a.total_tokens = T
        assert L.kda_prefill_host_workspace_size(ctypes.byref(a)) == 0
        assert L.kda_prefill_host(ctypes.byref(a), 0x4000, 1 << 40, None) == 1
    for bad, code in [(dict(dk=24), 2), (dict(segments=-1), 1), (dict(segments=65), 1),
                      (dict(q=None), 1), (dict(in_dtype=5), 1), (dict(cu_seqlens=None), 1)]:
        a = _host_args(kda, cu, **bad)
        assert L.kda_prefill_host_workspace_size(ctypes.byref(a)) == 0, bad
        assert L.kda_prefill_host(ctypes.byref(a), 0x4000, 1 << 40, None) == code, bad
    # the copy streams are required and distinct from each other and `stream`
    for streams in [(None, 0x20), (0x10, None), (0x10, 0x10), (0x30, 0x20)]:
        a = _host_args(kda, cu)
        a.copy_in_stream, a.copy_out_stream = streams
        assert L.kda_prefill_host(ctypes.byref(a), 0x4000, 1 << 40, 0x30) == 1, streams
    # workspace too small or misaligned
    assert L.kda_prefill_host(ctypes.byref(good), 0x4000, ws - 256, None) == 3
    assert L.kda_prefill_host(ctypes.byref(good), 0x4010, ws, None) == 3


def test_layer_args_shapes_checked_in_the_binding(kda):
    """The binding checks the layer steps' shapes before it touches device
    memory: taps [W, H, d] with 1 <= W <= 4, windows [rows, W-1, H, d], the
    gate [T, H, dv] or [T, H] (one gate per head)."""
    import torch
    H, dk, dv, W = 2, 16, 8, 3
    taps = (torch.zeros(W, H, dk), torch.zeros(W, H, dk), torch.zeros(W, H, dv))
    kw = dict(rows=4, H=H, dk=dk, dv=dv, dtype=torch.float32)
    assert kda.make_layer_args(**kw) is None                      # nothing asked for
    with pytest.raises(ValueError, match="conv width"):
        kda.make_layer_args(conv_weights=tuple(torch.zeros(5, H, d) for d in (dk, dk, dv)), **kw)
    with pytest.raises(ValueError, match="conv weights 2"):
        kda.make_layer_args(conv_weights=taps[:2] + (torch.zeros(W, H, dk),), **kw)
    with pytest.raises(ValueError, match="conv window 1"):
        kda.make_layer_args(conv_weights=taps, conv_window=(None, torch.zeros(4, W, H, dk), None),
                            **kw)
    with pytest.raises(ValueError, match="out_gate"):
        kda.make_layer_args(out_gate=torch.zeros(10, H, dk), gate_rows=10, **kw)
    with pytest.raises(ValueError, match="out_gate"):
        kda.make_layer_args(out_gate=torch.zeros(10, H + 1), gate_rows=10, **kw)
    # shapes right: the host tensors are then refused as not on the device
    with pytest.raises(ValueError, match="CUDA"):
        kda.make_layer_args(conv_weights=taps, **kw)


def test_state_and_snapshot_shapes_checked_in_the_binding(kda):
    """The C ABI takes bare pointers and cannot see how large a state buffer
    is, so the binding checks every shape before it takes a pointer: initial
    and final states [N, H, dk, dv], snapshots [rows, H, dk, dv], the
    snapshot and boundary offsets [N + 1] -- for the device call and the
    host-buffer call -- and the decode and prep tensors.  Host tensors with
    the right shapes get as far as the device check."""
    import torch
    T, H, dk, dv, N = 10, 2, 16, 8, 3
    x = dict(q=torch.zeros(T, H, dk), k=torch.zeros(T, H, dk), v=torch.zeros(T, H, dv),
             g=torch.zeros(T, H, dk), b=torch.zeros(T, H),
             cu_seqlens=torch.tensor([0, 3, 7, 10]), o=torch.zeros(T, H, dv))
    good = torch.zeros(N, H, dk, dv)
    args = [x[n] for n in ("q", "k", "v", "g", "b", "cu_seqlens", "o")]
    for make in (kda.make_prefill_args, kda.make_prefill_host_args):
        for kw in (dict(initial_state=torch.zeros(N - 1, H, dk, dv)),
                   dict(final_state=torch.zeros(N, H, dv, dk)),
                   dict(initial_state=torch.zeros(N, H, dk, dv + 1))):
            name = next(iter(kw))
            with pytest.raises(ValueError, match=name):
                make(*args, **kw)
        with pytest.raises(ValueError, match="o has shape"):
            make(*args[:6], torch.zeros(T, H, dk + 1), initial_state=good)
    with pytest.raises(ValueError, match="snapshots"):
        kda.make_prefill_args(*args, snapshots=torch.zeros(4, H, dk, dv - 1))
    with pytest.raises(ValueError, match="cu_snapshots"):
        kda.make_prefill_args(*args, snapshots=torch.zeros(4, H, dk, dv),
                              cu_snapshots=torch.zeros(N, dtype=torch.int64))
    with pytest.raises(ValueError, match="cu_boundaries"):
        kda.make_prefill_args(*args, boundary_pos=torch.zeros(2, dtype=torch.int64),
                              cu_boundaries=torch.zeros(N + 2, dtype=torch.int64))
    # right shapes: refused only because the tensors are not on the device
    with pytest.raises(ValueError, match="CUDA"):
        kda.make_prefill_args(*args, initial_state=good, final_state=good,
                              snapshots=torch.zeros(4, H, dk, dv),
                              cu_snapshots=torch.zeros(N + 1, dtype=torch.int64))
    ha = kda.make_prefill_host_args(*args, initial_state=good, final_state=good)
    assert ha.num_seqs == N and ha.total_tokens == T
    # decode: every tensor against q's [B, H, dk] and v's dv
    B = 4
    d = dict(q=torch.zeros(B, H, dk), k=torch.zeros(B, H, dk), v=torch.zeros(B, H, dv),
             g=torch.zeros(B, H, dk), b=torch.zeros(B, H))
    st, o = torch.zeros(6, H, dk, dv), torch.zeros(B, H, dv)
    dargs = [d[n] for n in "qkvgb"]
    with pytest.raises(ValueError, match="state"):
        kda.kda_decode_step(*dargs, torch.zeros(6, H, dv, dk), o)
    with pytest.raises(ValueError, match="o has shape"):
        kda.kda_decode_step(*dargs, st, torch.zeros(B + 1, H, dv))
    with pytest.raises(ValueError, match="b has shape"):
        kda.kda_decode_step(*dargs[:4], torch.zeros(B, H + 1), st, o)
    with pytest.raises(ValueError, match="state_slots"):
        kda.kda_decode_step(*dargs, st, o, state_slots=torch.zeros(B + 1, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        kda.kda_decode_step(*dargs, st, o)
    # prep: outputs [T, H, dk] and beta [T, H]
    f = torch.zeros(T, H, dk)
    with pytest.raises(ValueError, match="beta"):
        kda.kda_prep(x["q"], x["k"], x["g"], x["b"], x["cu_seqlens"], f, f, f, torch.zeros(T, H + 1))
    with pytest.raises(ValueError, match="G has shape"):
        kda.kda_prep(x["q"], x["k"], x["g"], x["b"], x["cu_seqlens"], f, f, torch.zeros(T, H, dk - 1),
                     torch.zeros(T, H))
