"""Pins of the oracle's layer steps (short convolution, output gate).

Each compares ``oracle.layer`` with something other than itself: an exact
special case (identity, a one-token shift), a library routine
(``np.convolve``, ``scipy.special.expit``, torch's bfloat16 conversion), an
invariant the ordering of the steps implies (L2 normalisation after the
convolution makes q's and k's taps scale-free), or the equivalence of a
split run with the whole one.  CPU only.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

from oracle import layer


def rnd(seed):
    return np.random.default_rng(seed)


def packed(rng, lens, H, d):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return rng.standard_normal((int(cu[-1]), H, d)), cu


def test_bf16_rounding_matches_torch():
    rng = rnd(1)
    x = rng.standard_normal(4096) * np.exp(rng.uniform(-20, 20, 4096))
    # exact ties of bfloat16: the kept part odd and even, halfway bits set
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(2.0 + 2.0 ** -7), 3.0 + 2.0 ** -7])
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(layer.round_to(x, "bfloat16"), ref)
    np.testing.assert_array_equal(layer.round_to(x, "float32"), x.astype(np.float32).astype(np.float64))


def test_conv_width1_unit_tap_is_identity():
    rng = rnd(2)
    x, cu = packed(rng, [5, 1, 9], 2, 4)
    y, win = layer.short_conv(x, np.ones((1, 2, 4)), cu)
    np.testing.assert_array_equal(y, x)
    assert win.shape == (3, 0, 2, 4)


def test_conv_lag_one_tap_shifts_each_sequence():
    rng = rnd(3)
    lens = [4, 1, 6]
    x, cu = packed(rng, lens, 3, 2)
    w = np.zeros((2, 3, 2))
    w[1] = 1.0
    window = rng.standard_normal((3, 1, 3, 2))
    for wi in (None, window):
        y, win = layer.short_conv(x, w, cu, wi)
        for s in range(3):
            a, e = cu[s], cu[s + 1]
            first = np.zeros((3, 2)) if wi is None else wi[s, 0]
            np.testing.assert_array_equal(y[a], first)          # the input before the start
            np.testing.assert_array_equal(y[a + 1:e], x[a:e - 1])
            np.testing.assert_array_equal(win[s, 0], x[e - 1])  # the last raw input


@pytest.mark.parametrize("W", [2, 3, 4])
def test_conv_matches_numpy_convolve(W):
    rng = rnd(10 + W)
    lens = [7, 2, 13]
    H, d = 2, 3
    x, cu = packed(rng, lens, H, d)
    w = rng.standard_normal((W, H, d))
    window = rng.standard_normal((3, W - 1, H, d))
    y, _ = layer.short_conv(x, w, cu, window)
    for s, L in enumerate(lens):
        a = cu[s]
        for h in range(H):
            for c in range(d):
                ext = np.concatenate([window[s, :, h, c], x[a:a + L, h, c]])
                ref = np.convolve(ext, w[:, h, c])[W - 1: W - 1 + L]
                np.testing.assert_allclose(y[a:a + L, h, c], ref, rtol=1e-13, atol=1e-13)


def test_conv_split_equals_whole_and_short_sequences_keep_the_window():
    rng = rnd(20)
    W, H, d, L = 4, 2, 3, 11
    x, _ = packed(rng, [L], H, d)
    w = rng.standard_normal((W, H, d))
    win0 = rng.standard_normal((1, W - 1, H, d))
    y, wend = layer.short_conv(x, w, [0, L], win0)
    for p in (1, 2, 3, 5):  # pieces shorter than the window too
        y1, w1 = layer.short_conv(x[:p], w, [0, p], win0)
        y2, w2 = layer.short_conv(x[p:], w, [0, L - p], w1)
        np.testing.assert_array_equal(np.concatenate([y1, y2]), y)
        np.testing.assert_array_equal(w2, wend)
    # one token: the window shifts by one
    _, w1 = layer.short_conv(x[:1], w, [0, 1], win0)
    np.testing.assert_array_equal(w1[0, :W - 2], win0[0, 1:])
    np.testing.assert_array_equal(w1[0, W - 2], x[0])


def test_silu_and_gate_match_expit():
    rng = rnd(30)
    y = rng.standard_normal(1000) * 10
    np.testing.assert_allclose(layer.silu(y), y * expit(y), rtol=1e-15, atol=1e-300)
    o = rng.standard_normal((5, 3, 4))
    r = rng.standard_normal((5, 3, 4)) * 4
    np.testing.assert_allclose(layer.output_gate(o, r), o * expit(r), rtol=1e-15)
    np.testing.assert_array_equal(layer.output_gate(o, np.zeros((5, 3, 4))), o / 2)  # sigmoid(0)
    np.testing.assert_array_equal(layer.output_gate(o, np.full((5, 3, 4), 40.0)), o)  # 1 in fp64
    rh = rng.standard_normal((5, 3))
    np.testing.assert_array_equal(layer.output_gate(o, rh),
                                  layer.output_gate(o, np.repeat(rh[..., None], 4, axis=2)))


def _layer_inputs(rng, lens, H, dk, dv, W):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    q = rng.standard_normal((T, H, dk)).astype(np.float32)
    k = rng.standard_normal((T, H, dk)).astype(np.float32)
    v = rng.standard_normal((T, H, dv)).astype(np.float32)
    g = (rng.standard_normal((T, H, dk)) - 3).astype(np.float32)
    b = rng.standard_normal((T, H)).astype(np.float32)
    cw = tuple(rng.standard_normal((W, H, n)) for n in (dk, dk, dv))
    return cu, q, k, v, g, b, cw


def test_normalisation_follows_the_convolution():
    """q^ and k^ are normalised after the convolution: scaling q's or k's taps
    by a positive constant leaves o unchanged; scaling v's scales o (zero
    initial state: o is linear in v).  Fails if the norm came first."""
    rng = rnd(40)
    cu, q, k, v, g, b, (wq, wk, wv) = _layer_inputs(rng, [9, 5], 2, 4, 3, 3)
    o, S, _, _ = layer.prefill_layer(q, k, v, g, b, cu, conv_w=(wq, wk, wv))
    # (the recurrence takes its inputs as float32: equal to that rounding;
    # the norm taken before the convolution would change o at O(1))
    o2, S2, _, _ = layer.prefill_layer(q, k, v, g, b, cu, conv_w=(3.0 * wq, 0.25 * wk, wv))
    np.testing.assert_allclose(o2, o, rtol=1e-5, atol=1e-6)
    o3, S3, _, _ = layer.prefill_layer(q, k, v, g, b, cu, conv_w=(wq, wk, 2.0 * wv))
    np.testing.assert_allclose(o3, 2.0 * o, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(S3, 2.0 * S, rtol=1e-5, atol=1e-6)
    assert np.abs(o).max() > 1e-2
    # with no taps beyond lag 0 and a unit tap the layer is the bare recurrence
    one = tuple(np.ones((1, 2, n)) for n in (4, 4, 3))
    o4, _, _, _ = layer.prefill_layer(q, k, v, g, b, cu, conv_w=one)
    o5, _, _, _ = layer.prefill_layer(q, k, v, g, b, cu)
    np.testing.assert_array_equal(o4, o5)


@pytest.mark.parametrize("dtype", ["float64", "bfloat16"])
def test_prefill_then_decode_equals_prefill(dtype):
    """The windows carry the convolution across calls: a prefill of the first
    p tokens followed by decode steps of the rest, windows and state handed
    over, equals one prefill of the whole sequence (gate and SiLU on)."""
    rng = rnd(50)
    W, H, dk, dv, L, p = 4, 2, 4, 3, 9, 5
    cu, q, k, v, g, b, cw = _layer_inputs(rng, [L], H, dk, dv, W)
    r = rng.standard_normal((L, H, dv)).astype(np.float32)
    win0 = tuple(rng.standard_normal((1, W - 1, H, n)) for n in (dk, dk, dv))
    o, S, _, wend = layer.prefill_layer(q, k, v, g, b, cu, conv_w=cw, windows=win0,
                                        use_silu=True, dtype=dtype, out_gate=r)
    o1, S1, _, w1 = layer.prefill_layer(q[:p], k[:p], v[:p], g[:p], b[:p], [0, p], conv_w=cw,
                                        windows=win0, use_silu=True, dtype=dtype, out_gate=r[:p])
    np.testing.assert_array_equal(o1, o[:p])
    state = S1.copy()
    wins = [w.copy() for w in w1]
    for t in range(p, L):
        sl = slice(t, t + 1)
        ot = layer.decode_layer(q[sl], k[sl], v[sl], g[sl], b[sl], state, conv_w=cw, windows=wins,
                                use_silu=True, dtype=dtype, out_gate=r[sl])
        np.testing.assert_allclose(ot[0], o[t], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(state, S, rtol=1e-11, atol=1e-13)
    for a, e in zip(wins, wend):
        np.testing.assert_array_equal(a, e)
