"""Seeded synthetic inputs for the KDA prefill and decode paths.

This module holds random draws, dtype casts and sequence-length recipes only:
none of the method's arithmetic.  The tests and the benchmark call it to feed
the same tensors to the CUDA library and to the CPU oracle.

Distributions (shared by every workload): q, k, v ~ N(0, 1); the decay logit
g ~ N(-3, 1) (so alpha = exp(-softplus(g)) has median ~0.95); the update
logit b ~ N(0, 1) (beta = sigmoid(b)); initial states, where a workload has
them, ~ N(0, 0.02^2).  Values are drawn in float32 and then cast to the
workload's input dtype, so the bf16 tensors hold exactly the values the
oracle is given (it reads them back as float32).

Draw order for one generator seeded with ``seed``: sequence lengths, interior
boundaries, then q, k, v, g, b, initial state.  Large workloads draw on the
GPU with a CUDA generator seeded the same way (``device='cuda'``); those
values differ from the CPU draws but are equally reproducible.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

CHUNK = 64


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    lens: tuple | None            # fixed lengths, or None to draw them
    n_seqs: int
    H: int
    dk: int
    dv: int
    dtype: str                    # 'f32' or 'bf16' (inputs and o)
    seed: int
    len_range: tuple = (0, 0)     # inclusive range for drawn lengths
    s0_std: float = 0.0           # 0: no initial state
    snapshot_interval: int = 0
    interior_boundary: bool = False  # one seeded boundary per sequence + its end
    description: str = ""


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    H: int
    dk: int
    dv: int
    steps: int
    seed: int
    s0_std: float = 0.02
    description: str = ""


WORKLOADS = {
    "tiny_f32": PrefillWorkload(
        "tiny_f32", (64,), 1, 2, 16, 16, "f32", 1000,
        description="B=1 H=2 T=64 dk=dv=16 fp32, zero initial state"),
    "prefill_8k": PrefillWorkload(
        "prefill_8k", (8192,), 1, 32, 128, 128, "bf16", 1001,
        description="single-sequence prefill B=1 H=32 T=8192 dk=dv=128 bf16 in, "
                    "fp32 state, C=64, zero initial state"),
    "varlen_8": PrefillWorkload(
        "varlen_8", None, 8, 32, 128, 128, "bf16", 1002, len_range=(1024, 32768),
        s0_std=0.02, snapshot_interval=4096, interior_boundary=True,
        description="8 packed sequences, lengths U[1024,32768], H=32 dk=dv=128 bf16, "
                    "seeded initial states, snapshots every 4096 tokens and at boundaries"),
    "prefill_1m": PrefillWorkload(
        "prefill_1m", (1 << 20,), 1, 32, 128, 128, "bf16", 1004,
        snapshot_interval=65536,
        description="million-token prefill B=1 H=32 T=2^20 dk=dv=128 bf16, "
                    "snapshots every 65536 tokens"),
}

DECODE_WORKLOADS = {
    "decode_256": DecodeWorkload(
        "decode_256", 256, 32, 128, 128, 1000, 1003,
        description="256 sequences x H=32, fp32 128x128 states (537 MB), one bf16 token "
                    "per step, state updated in place"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_lengths(w: PrefillWorkload) -> list[int]:
    if w.lens is not None:
        return list(w.lens)
    g = _gen(w.seed, "cpu")
    lo, hi = w.len_range
    return [int(x) for x in torch.randint(lo, hi + 1, (w.n_seqs,), generator=g)]


def prefill_inputs(w: PrefillWorkload, device: str = "cpu", lens: list[int] | None = None,
                   seed: int | None = None, gen_device: str | None = None) -> dict:
    """Inputs of one prefill call: q, k, g [T,H,dk]; v [T,H,dv]; b [T,H] in the
    workload dtype; cu_seqlens int64 [N+1]; S0 float32 [N,H,dk,dv] or None;
    boundary_pos / cu_boundaries int64 (seq-relative, sorted) or None.

    ``lens`` overrides the workload's lengths (for scaled-down test cases)."""
    seed = w.seed if seed is None else seed
    gdev = gen_device or ("cpu" if device == "cpu" else device)
    g_cpu = _gen(seed, "cpu")
    if lens is None:
        if w.lens is not None:
            lens = list(w.lens)
        else:
            lo, hi = w.len_range
            lens = [int(x) for x in torch.randint(lo, hi + 1, (w.n_seqs,), generator=g_cpu)]
    else:
        lens = list(lens)
        if w.lens is None:  # keep the draw order identical
            torch.randint(1, 2, (len(lens),), generator=g_cpu)
    N = len(lens)
    boundary_pos = cu_boundaries = None
    if w.interior_boundary:
        bpos, cub = [], [0]
        for L in lens:
            pts = []
            if L >= 2:
                pts.append(int(torch.randint(1, L, (1,), generator=g_cpu)))
            pts.append(L)
            pts = sorted(set(pts))
            bpos += pts
            cub.append(len(bpos))
        boundary_pos = torch.tensor(bpos, dtype=torch.int64)
        cu_boundaries = torch.tensor(cub, dtype=torch.int64)
    T = sum(lens)
    cu = torch.zeros(N + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)
    dt = torch_dtype(w.dtype)
    gg = g_cpu if gdev == "cpu" else _gen(seed, gdev)
    kw = dict(generator=gg, device=gdev, dtype=torch.float32)
    q = torch.randn(T, w.H, w.dk, **kw).to(dt)
    k = torch.randn(T, w.H, w.dk, **kw).to(dt)
    v = torch.randn(T, w.H, w.dv, **kw).to(dt)
    g = (torch.randn(T, w.H, w.dk, **kw) - 3.0).to(dt)
    b = torch.randn(T, w.H, **kw).to(dt)
    S0 = None
    if w.s0_std > 0:
        S0 = torch.randn(N, w.H, w.dk, w.dv, **kw) * w.s0_std
    out = dict(q=q, k=k, v=v, g=g, b=b, S0=S0, cu_seqlens=cu, lens=lens,
               boundary_pos=boundary_pos, cu_boundaries=cu_boundaries,
               snapshot_interval=w.snapshot_interval)
    for key in ("q", "k", "v", "g", "b", "S0", "cu_seqlens", "boundary_pos", "cu_boundaries"):
        if out[key] is not None:
            out[key] = out[key].to(device)
    return out


def decode_inputs(w: DecodeWorkload, steps: int | None = None, device: str = "cpu",
                  gen_device: str | None = None, dtype: str = "bf16") -> dict:
    """Per-step decode inputs q, k, g [steps,B,H,dk], v [steps,B,H,dv], b [steps,B,H]
    and the initial state pool float32 [B,H,dk,dv]."""
    steps = w.steps if steps is None else steps
    gdev = gen_device or device
    gg = _gen(w.seed, gdev)
    kw = dict(generator=gg, device=gdev, dtype=torch.float32)
    dt = torch_dtype(dtype)
    state = torch.randn(w.batch, w.H, w.dk, w.dv, **kw) * w.s0_std
    q = torch.randn(steps, w.batch, w.H, w.dk, **kw).to(dt)
    k = torch.randn(steps, w.batch, w.H, w.dk, **kw).to(dt)
    v = torch.randn(steps, w.batch, w.H, w.dv, **kw).to(dt)
    g = (torch.randn(steps, w.batch, w.H, w.dk, **kw) - 3.0).to(dt)
    b = torch.randn(steps, w.batch, w.H, **kw).to(dt)
    out = dict(q=q, k=k, v=v, g=g, b=b, state=state)
    return {key: t.to(device) for key, t in out.items()}


def layer_inputs(seed: int, rows: int, T: int, H: int, dk: int, dv: int, width: int,
                 dtype: str = "bf16", device: str = "cpu", gate_per_head: bool = False) -> dict:
    """Inputs of the layer steps around the recurrence, from their own
    generator (seed): the short convolution's taps (float32 [W, H, d] for q,
    k, v, ~ N(0, 1/W) so that a convolved input keeps about unit variance),
    the windows before the call (the workload dtype, [rows, W-1, H, d],
    ~ N(0, 1) like the inputs they stand for) and the output gate's logits
    r ~ N(0, 1) ([T, H, dv], or [T, H] with one gate per head)."""
    gg = _gen(seed, device)
    kw = dict(generator=gg, device=device, dtype=torch.float32)
    dt = torch_dtype(dtype)
    dims = (dk, dk, dv)
    taps = tuple(torch.randn(width, H, d, **kw) / width ** 0.5 for d in dims)
    windows = tuple(torch.randn(rows, width - 1, H, d, **kw).to(dt) for d in dims)
    gate = torch.randn(*((T, H) if gate_per_head else (T, H, dv)), **kw).to(dt)
    return dict(taps=taps, windows=windows, gate=gate)
