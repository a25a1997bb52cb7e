"""CPU oracle of the Kimi Delta Attention (KDA) recurrence.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check of ``__graft_entry__``
and the CPU-baseline leg of ``bench.py`` use it.  The CUDA library never
imports, links or calls anything here, and nothing here imports the CUDA
package.

Two independent implementations live in this package:

* ``kda_oracle.c`` (loaded through ctypes below): the token-by-token fp64
  delta form, with OpenMP over (sequence, head).  It is the oracle.
* ``forms.py``: numpy fp64 restatements used to pin the oracle -- the
  literal product form with explicit transition matrices, the brute-force
  expansion of the state as a sum over tokens, and the chunked form.

What the recurrence is and where each piece comes from is stated in the
header of ``kda_oracle.c``.  Parity is pinned for every function here (see
``tests/test_oracle_pins.py``); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: same results on x86 and Arm)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _nullable(ptr_type):
    """ctypes argtype accepting either an ndarray or None (NULL)."""
    class _Nullable:
        @classmethod
        def from_param(cls, obj):
            if obj is None:
                return ctypes.c_void_p(0)
            return ptr_type.from_param(obj)
    return _Nullable


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.kda_oracle_prep.argtypes = [ctypes.c_int64, ctypes.c_int32, _f32p, _f32p, _f32p,
                                          _f32p, _f64p, _f64p, _f64p, _f64p]
            L.kda_oracle_prep.restype = None
            L.kda_oracle_prefill.argtypes = [
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _i64p,
                _f32p, _f32p, _f32p, _f32p, _f32p, ctypes.c_double, _nullable(_f64p),
                _f64p, _nullable(_f64p), _nullable(_i64p), _nullable(_i64p), _nullable(_f64p),
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
            L.kda_oracle_prefill.restype = ctypes.c_int
            L.kda_oracle_recurrence.argtypes = [
                ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _f64p, _f64p,
                _f64p, _f64p, _f64p, ctypes.c_double, _nullable(_f64p), _f64p, _f64p]
            L.kda_oracle_recurrence.restype = None
            L.kda_oracle_decode.argtypes = [
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _f32p, _f32p,
                _f32p, _f32p, _f32p, ctypes.c_double, _f64p, _nullable(_i32p), _f64p,
                ctypes.c_int32]
            L.kda_oracle_decode.restype = None
            L.kda_oracle_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def max_threads() -> int:
    return int(lib().kda_oracle_max_threads())


def prep(q, k, g, b):
    """Per-row preparation: (q^, k^, log alpha, beta) for rows of q,k,g [R, dk], b [R]."""
    q, k, g = _f32(q), _f32(k), _f32(g)
    b = _f32(b)
    dk = q.shape[-1]
    R = int(np.prod(q.shape[:-1]))
    assert b.shape == q.shape[:-1] and k.shape == q.shape and g.shape == q.shape
    qh = np.empty((R, dk)); kh = np.empty((R, dk)); la = np.empty((R, dk)); be = np.empty(R)
    lib().kda_oracle_prep(R, dk, q.reshape(R, dk), k.reshape(R, dk), g.reshape(R, dk),
                          b.reshape(R), qh, kh, la, be)
    shp = q.shape
    return qh.reshape(shp), kh.reshape(shp), la.reshape(shp), be.reshape(b.shape)


def prefill(q, k, v, g, b, cu_seqlens, scale=1.0, S0=None, snap_pos=None, cu_snap=None,
            heads=None, nthreads=0):
    """Token-by-token fp64 prefill over packed sequences.

    q, k, g: [T, H, dk]; v: [T, H, dv]; b: [T, H] (any float dtype; converted to float32,
    which holds bf16 values exactly).  cu_seqlens: [N+1] int64.  S0: [N, H, dk, dv] or None.
    snap_pos / cu_snap: sorted seq-relative positions per sequence and their [N+1] offsets.
    heads: (h_begin, h_end) to compute a subset of heads.
    Returns (o [T, H, dv], S_final [N, H, dk, dv], snaps [n_snap, H, dk, dv] or None).
    """
    q, k, v, g, b = _f32(q), _f32(k), _f32(v), _f32(g), _f32(b)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu.shape[0] - 1
    assert k.shape == (T, H, dk) and g.shape == (T, H, dk) and v.shape[:2] == (T, H)
    assert b.shape == (T, H) and cu[-1] == T
    o = np.zeros((T, H, dv))
    S_final = np.zeros((N, H, dk, dv))
    snaps = None
    sp = cs = None
    if snap_pos is not None:
        sp = np.ascontiguousarray(np.asarray(snap_pos, dtype=np.int64))
        cs = np.ascontiguousarray(np.asarray(cu_snap, dtype=np.int64))
        snaps = np.zeros((max(int(cs[-1]), 1), H, dk, dv))
    h0, h1 = (0, H) if heads is None else heads
    rc = lib().kda_oracle_prefill(N, H, dk, dv, cu, q, k, v, g, b, float(scale), _f64(S0), o,
                                  S_final, sp, cs, snaps, h0, h1, int(nthreads))
    if rc != 0:
        raise ValueError("kda_oracle_prefill: inconsistent arguments")
    if snaps is not None:
        snaps = snaps[: int(cs[-1])]
    return o, S_final, snaps


def recurrence(qhat, khat, v, alpha, beta, scale=1.0, S0=None):
    """Recurrence of one sequence with gates given directly.

    qhat, khat, alpha: [T, H, dk] float64; v: [T, H, dv]; beta: [T, H]; S0: [H, dk, dv].
    Returns (o [T, H, dv], S_final [H, dk, dv]).
    """
    qhat, khat, v, alpha, beta = (_f64(x) for x in (qhat, khat, v, alpha, beta))
    T, H, dk = qhat.shape
    dv = v.shape[2]
    o = np.zeros((T, H, dv))
    S = np.zeros((H, dk, dv))
    lib().kda_oracle_recurrence(T, H, dk, dv, qhat, khat, v, alpha, beta, float(scale),
                                _f64(S0), o, S)
    return o, S


def decode(q, k, v, g, b, state, slots=None, scale=1.0, nthreads=0):
    """One decode step; ``state`` [n_slots, H, dk, dv] float64 is updated in place.

    q, k, g: [B, H, dk]; v: [B, H, dv]; b: [B, H].  slots: [B] int32 or None.
    Returns o [B, H, dv] (rows with slot < 0 stay zero).
    """
    q, k, v, g, b = _f32(q), _f32(k), _f32(v), _f32(g), _f32(b)
    assert state.dtype == np.float64 and state.flags["C_CONTIGUOUS"]
    B, H, dk = q.shape
    dv = v.shape[2]
    o = np.zeros((B, H, dv))
    sl = None if slots is None else np.ascontiguousarray(np.asarray(slots, dtype=np.int32))
    lib().kda_oracle_decode(B, H, dk, dv, q, k, v, g, b, float(scale), state, sl, o,
                            int(nthreads))
    return o


def snapshot_positions(lens, interval: int, boundary_pos=None, cu_boundaries=None):
    """Snapshot positions per sequence, as the oracle defines them: every
    multiple of ``interval`` in (0, len] together with the sequence's boundary
    positions (seq-relative, in [1, len]), sorted and de-duplicated.  The state
    after p tokens is the one kept for position p ("Kimi K3: The Manos, The
    Mythos, The Legendos", section Context: snapshots at prompt boundaries).
    Returns (positions int64 [n_snap], cu_snap int64 [N+1])."""
    pos, cu = [], [0]
    for s, L in enumerate(lens):
        pts = set()
        if interval > 0:
            pts.update(range(interval, int(L) + 1, interval))
        if boundary_pos is not None:
            b0, b1 = int(cu_boundaries[s]), int(cu_boundaries[s + 1])
            pts.update(int(x) for x in np.asarray(boundary_pos)[b0:b1])
        pos += sorted(pts)
        cu.append(len(pos))
    return np.asarray(pos, dtype=np.int64), np.asarray(cu, dtype=np.int64)
