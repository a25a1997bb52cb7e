"""The layer steps on either side of the KDA recurrence, in plain numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring): the tests, the smoke
check and the CPU-baseline leg of the benchmark use it; the CUDA library
never does.

"Kimi K3: The Manos, The Mythos, The Legendos" (bullet on the stability
details) lists a short convolution on q, k and v and a per-head output
forget gate around the recurrence, without formulas.  The readings taken
here (the same ones the C header of the library states):

* short convolution -- per channel, causal along the tokens of one
  sequence:  y_t[c] = sum_{j < W} w[j, h, c] * x_{t-j}[c].  Inputs before the
  sequence start come from a window of the W - 1 inputs that preceded it
  (oldest first), zeros without one.  Optionally SiLU, y * sigmoid(y).  The
  result is stored in the input dtype (a separate layer would write it so);
  the recurrence takes it as its q, k, v, so q and k are L2-normalised after
  the convolution.
* output gate -- o_t <- o_t * sigmoid(r_t), r per value channel [T, H, dv]
  or per head [T, H].

``prefill_layer`` and ``decode_layer`` compose these with the token-by-token
oracle of ``kda_oracle.c``.  All functions here are pinned in
``tests/test_layer_pins.py``.
"""
from __future__ import annotations

import numpy as np

from . import decode as _decode
from . import prefill as _prefill

DTYPES = ("float64", "float32", "bfloat16")


def round_to(x, dtype: str):
    """Round float64 values to ``dtype`` (nearest, ties to even), returned as
    float64.  bfloat16 keeps the top 16 bits of the float32 pattern; it is
    reached from the float32 rounding (float32 -> bfloat16 is how a GPU
    stores an fp32 result)."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "float64":
        return x.copy()
    f = x.astype(np.float32)
    if dtype == "float32":
        return f.astype(np.float64)
    assert dtype == "bfloat16", dtype
    u = f.view(np.uint32).astype(np.uint64)
    # add half an ulp of bfloat16, minus one when the kept part is even
    # (ties to even); then drop the low 16 bits
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def silu(y):
    """y * sigmoid(y)."""
    y = np.asarray(y, dtype=np.float64)
    return y * sigmoid(y)


def short_conv(x, w, cu_seqlens, window=None, use_silu=False, dtype="float64"):
    """Causal depthwise convolution over packed sequences.

    x: [T, H, d]; w: [W, H, d] (tap j multiplies the input j tokens back);
    window: [N, W-1, H, d] or None (zeros), the raw inputs before each
    sequence, oldest first.  Returns (y [T, H, d] float64 holding values of
    ``dtype``, window_out [N, W-1, H, d]: the raw inputs of the last W-1
    positions of window ++ sequence)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, H, d = x.shape
    W = w.shape[0]
    N = cu.shape[0] - 1
    assert w.shape == (W, H, d) and W >= 1
    y = np.zeros((T, H, d))
    win_out = np.zeros((N, W - 1, H, d))
    for s in range(N):
        a, e = int(cu[s]), int(cu[s + 1])
        pre = np.zeros((W - 1, H, d)) if window is None else np.asarray(window[s], dtype=np.float64)
        ext = np.concatenate([pre, x[a:e]], axis=0)  # row W-1+t is token t
        acc = np.zeros((e - a, H, d))
        for j in range(W):
            acc += w[j][None] * ext[W - 1 - j: W - 1 - j + (e - a)]
        if use_silu:
            acc = silu(acc)
        y[a:e] = round_to(acc, dtype)
        win_out[s] = ext[ext.shape[0] - (W - 1):]
    return y, win_out


def output_gate(o, r):
    """o [T, H, dv] times sigmoid(r), r [T, H, dv] or [T, H] (one gate per head)."""
    o = np.asarray(o, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if r.ndim == o.ndim - 1:
        r = r[..., None]
    return o * sigmoid(r)


def prefill_layer(q, k, v, g, b, cu_seqlens, conv_w=None, windows=None, use_silu=False,
                  dtype="float64", out_gate=None, **kw):
    """The oracle prefill with the layer steps: q, k, v convolved (conv_w =
    (wq, wk, wv) or None), the recurrence of ``kda_oracle.c`` on the results,
    the output gate on o.  windows = (q, k, v) windows or None; extra keyword
    arguments go to ``oracle.prefill``.  Returns (o, S_final, snaps,
    windows_out) with windows_out None without a convolution.  The
    recurrence of ``kda_oracle.c`` takes float32 inputs, so with dtype
    "float64" the convolved values enter it rounded to float32; the GPU
    paths store them in their input dtype ("float32" or "bfloat16")."""
    win_out = None
    if conv_w is not None:
        ys, win_out = [], []
        for t, (x, w) in enumerate(zip((q, k, v), conv_w)):
            wi = None if windows is None else windows[t]
            y, wo = short_conv(x, w, cu_seqlens, wi, use_silu, dtype)
            ys.append(y)
            win_out.append(wo)
        q, k, v = ys
    o, S, snaps = _prefill(q, k, v, g, b, cu_seqlens, **kw)
    if out_gate is not None:
        o = output_gate(o, out_gate)
    return o, S, snaps, win_out


def decode_layer(q, k, v, g, b, state, conv_w=None, windows=None, use_silu=False,
                 dtype="float64", out_gate=None, slots=None, **kw):
    """One oracle decode step with the layer steps.  q, k, g [B, H, dk];
    v [B, H, dv]; b [B, H]; state [n_slots, H, dk, dv] float64 (in place);
    windows = (q, k, v) windows [n_slots, W-1, H, d] float64, updated in place
    for the rows' slots.  Rows with slot < 0 are skipped."""
    B = q.shape[0]
    sl = np.arange(B) if slots is None else np.asarray(slots)
    if conv_w is not None:
        ys = []
        for t, (x, w) in enumerate(zip((q, k, v), conv_w)):
            x = np.asarray(x, dtype=np.float64)
            y = np.zeros_like(x)
            for r in range(B):
                if sl[r] < 0:
                    continue
                win = windows[t][sl[r]][None]  # one sequence of one token
                yr, wo = short_conv(x[r:r + 1], w, [0, 1], win, use_silu, dtype)
                y[r] = yr[0]
                windows[t][sl[r]] = wo[0]
            ys.append(y)
        q, k, v = ys
    o = _decode(q, k, v, g, b, state, slots=slots, **kw)
    if out_gate is not None:
        o = output_gate(o, out_gate)
    return o
