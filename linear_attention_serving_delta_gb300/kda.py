"""Python binding of libkda (include/kda.h): argument marshalling only.

Every step of the KDA path runs in the library's CUDA kernels; PyTorch only
provides device memory, streams and the host<->device copies of the
end-to-end helper.  There is no CPU fallback: if libkda.so has not been
built, or no CUDA device is present, the calls raise.

The names follow the C ABI: ``kda_prefill``, ``kda_prefill_workspace_size``,
``kda_prefill_device_status``, ``kda_snapshot_plan``, ``kda_decode_step``,
``kda_prep``, ``kda_status_string``, ``kda_prefill_host`` (host buffers).
``prefill`` and ``prefill_host`` are conveniences that allocate outputs and
workspace with torch and call ``kda_prefill`` / ``kda_prefill_host``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

KDA_OK = 0
KDA_F32, KDA_BF16 = 0, 1
CHUNK = 64
PREFILL_PHASES = 3  # chunk planning, intra-chunk, inter-chunk
SCHEDULE_AUTO, SCHEDULE_SEPARATE, SCHEDULE_FUSED, SCHEDULE_OVERLAP = 0, 1, 2, 3  # kda_prefill_args.schedule
# kda_prefill_schedule: the path a prefill takes
PATH_CUDA_CORES, PATH_SEPARATE, PATH_FUSED, PATH_SEGMENT_SCAN, PATH_OVERLAP = 0, 1, 2, 3, 4
_STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED",
                 3: "KDA_ERR_WORKSPACE", 4: "KDA_ERR_CUDA", 5: "KDA_ERR_TIMEOUT",
                 6: "KDA_ERR_DEVICE_DATA"}
EXPORTED = ("kda_prefill_workspace_size", "kda_prefill", "kda_prefill_noalloc",
            "kda_prefill_noalloc_device_status", "kda_prefix_cache_forget",
            "kda_prefill_host_workspace_size", "kda_prefill_host",
            "kda_prefix_cache_create", "kda_prefix_cache_destroy", "kda_prefix_cache_entries",
            "kda_prefix_cache_lookup", "kda_prefix_cache_reserve",
            "kda_prefill_device_status", "kda_snapshot_plan", "kda_decode_step", "kda_prep",
            "kda_status_string", "kda_version", "kda_prefill_schedule")
NOALLOC_SCRATCH_BYTES = 64 << 20  # fixed workspace behind kda_prefill_noalloc


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS_NAMES.get(status, status)} "
                         f"({kda_status_string(status)})")


c_i32, c_i64, c_f32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
CONV_MAX = 4  # KDA_CONV_MAX: taps of the short convolution


class LayerArgs(ctypes.Structure):
    """kda_layer_args: the short convolution on q, k, v and the output gate."""
    _fields_ = [("conv_width", c_i32), ("conv_silu", c_i32), ("conv_w", c_vp * 3),
                ("conv_in", c_vp * 3), ("conv_out", c_vp * 3), ("out_gate", c_vp),
                ("out_gate_per_head", c_i32)]


class PrefillArgs(ctypes.Structure):
    _fields_ = [("num_seqs", c_i32), ("num_heads", c_i32), ("dk", c_i32), ("dv", c_i32),
                ("total_tokens", c_i64), ("cu_seqlens", c_vp), ("in_dtype", ctypes.c_int),
                ("q", c_vp), ("k", c_vp), ("v", c_vp), ("g", c_vp), ("b", c_vp),
                ("scale", c_f32), ("initial_state", c_vp), ("o", c_vp), ("final_state", c_vp),
                ("snapshot_interval", c_i64), ("boundary_pos", c_vp), ("cu_boundaries", c_vp),
                ("num_boundaries", c_i64), ("cu_snapshots", c_vp), ("snapshots", c_vp),
                ("num_snapshots", c_i64), ("phase_events", c_vp), ("scan_segments", c_i32),
                ("snapshot_slot_map", c_vp), ("snapshot_map_len", c_i64),
                ("wait_limit_ns", c_i64), ("gate_per_head", c_i32),
                ("layer", ctypes.POINTER(LayerArgs)), ("schedule", c_i32)]


class PrefillHostArgs(ctypes.Structure):
    _fields_ = [("num_seqs", c_i32), ("num_heads", c_i32), ("dk", c_i32), ("dv", c_i32),
                ("total_tokens", c_i64), ("cu_seqlens", c_vp), ("in_dtype", ctypes.c_int),
                ("q", c_vp), ("k", c_vp), ("v", c_vp), ("g", c_vp), ("b", c_vp),
                ("scale", c_f32), ("initial_state", c_vp), ("o", c_vp), ("final_state", c_vp),
                ("segments", c_i32), ("copy_in_stream", c_vp), ("copy_out_stream", c_vp),
                ("gate_per_head", c_i32)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("batch", c_i32), ("num_heads", c_i32), ("dk", c_i32), ("dv", c_i32),
                ("num_slots", c_i32), ("in_dtype", ctypes.c_int), ("scale", c_f32),
                ("q", c_vp), ("k", c_vp), ("v", c_vp), ("g", c_vp), ("b", c_vp),
                ("state", c_vp), ("state_slots", c_vp), ("o", c_vp), ("wait_limit_ns", c_i64),
                ("status", c_vp), ("gate_per_head", c_i32), ("layer", ctypes.POINTER(LayerArgs))]


class PrepArgs(ctypes.Structure):
    _fields_ = [("num_seqs", c_i32), ("num_heads", c_i32), ("dk", c_i32),
                ("total_tokens", c_i64), ("cu_seqlens", c_vp), ("in_dtype", ctypes.c_int),
                ("q", c_vp), ("k", c_vp), ("g", c_vp), ("b", c_vp), ("qhat", c_vp),
                ("khat", c_vp), ("G", c_vp), ("beta", c_vp), ("gate_per_head", c_i32),
                ("layer", ctypes.POINTER(LayerArgs))]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Loads libkda.so; raises if it was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libkda.so not built ({LIB_PATH}); run "
                                   "`python -m linear_attention_serving_delta_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            L.kda_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
            L.kda_prefill_workspace_size.restype = ctypes.c_size_t
            L.kda_prefill_schedule.argtypes = [ctypes.POINTER(PrefillArgs), c_i32]
            L.kda_prefill_schedule.restype = c_i32
            L.kda_prefill.argtypes = [ctypes.POINTER(PrefillArgs), c_vp, ctypes.c_size_t, c_vp]
            L.kda_prefill.restype = ctypes.c_int
            L.kda_prefill_host_workspace_size.argtypes = [ctypes.POINTER(PrefillHostArgs)]
            L.kda_prefill_host_workspace_size.restype = ctypes.c_size_t
            L.kda_prefill_host.argtypes = [ctypes.POINTER(PrefillHostArgs), c_vp, ctypes.c_size_t,
                                           c_vp]
            L.kda_prefill_host.restype = ctypes.c_int
            L.kda_prefix_cache_create.argtypes = [c_i64]
            L.kda_prefix_cache_create.restype = c_vp
            L.kda_prefix_cache_destroy.argtypes = [c_vp]
            L.kda_prefix_cache_destroy.restype = None
            L.kda_prefix_cache_entries.argtypes = [c_vp]
            L.kda_prefix_cache_entries.restype = c_i64
            L.kda_prefix_cache_lookup.argtypes = [c_vp, c_vp, c_i64, ctypes.POINTER(c_i32)]
            L.kda_prefix_cache_lookup.restype = c_i64
            L.kda_prefix_cache_reserve.argtypes = [c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i32,
                                                   c_vp]
            L.kda_prefix_cache_reserve.restype = c_i64
            L.kda_prefill_noalloc.argtypes = [ctypes.POINTER(PrefillArgs), c_vp]
            L.kda_prefill_noalloc.restype = ctypes.c_int
            L.kda_prefill_noalloc_device_status.argtypes = [ctypes.POINTER(c_i32), c_vp]
            L.kda_prefill_noalloc_device_status.restype = ctypes.c_int
            L.kda_prefix_cache_forget.argtypes = [c_vp, c_vp, c_i64]
            L.kda_prefix_cache_forget.restype = c_i64
            L.kda_prefill_device_status.argtypes = [c_vp, ctypes.POINTER(c_i32), c_vp]
            L.kda_prefill_device_status.restype = ctypes.c_int
            L.kda_snapshot_plan.argtypes = [c_vp, c_i32, c_i64, c_vp, c_vp, c_vp]
            L.kda_snapshot_plan.restype = c_i64
            L.kda_decode_step.argtypes = [ctypes.POINTER(DecodeArgs), c_vp]
            L.kda_decode_step.restype = ctypes.c_int
            L.kda_prep.argtypes = [ctypes.POINTER(PrepArgs), c_vp]
            L.kda_prep.restype = ctypes.c_int
            L.kda_status_string.argtypes = [ctypes.c_int]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def kda_version() -> str:
    return lib().kda_version().decode()


# ----------------------------------------------------------------- marshalling helpers
def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return KDA_F32
    if t == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"unsupported input dtype {t} (float32 or bfloat16)")


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, what: str):
    if status != KDA_OK:
        raise KdaError(status, what)


def make_layer_args(*, rows, H, dk, dv, dtype, conv_weights=None, conv_silu=False,
                    conv_window=None, conv_window_out=None, out_gate=None,
                    gate_rows=None) -> LayerArgs | None:
    """kda_layer_args from tensors (None when neither step is asked for).

    conv_weights: (wq, wk, wv) float32 [W, H, d]; conv_window / conv_window_out:
    (q, k, v) windows [rows, W-1, H, d] in the input dtype (an entry may be
    None); out_gate: [gate_rows, H, dv] or [gate_rows, H] (one gate per head)."""
    if conv_weights is None and out_gate is None:
        return None
    # every shape first, then the pointers
    W = 0
    if conv_weights is not None:
        W = conv_weights[0].shape[0]
        if not 1 <= W <= CONV_MAX:
            raise ValueError(f"conv width {W} outside 1..{CONV_MAX}")
        for t, (w, d) in enumerate(zip(conv_weights, (dk, dk, dv))):
            if tuple(w.shape) != (W, H, d):
                raise ValueError(f"conv weights {t} have shape {tuple(w.shape)}, expected {(W, H, d)}")
            for src in (conv_window, conv_window_out):
                x = None if src is None else src[t]
                if x is not None and tuple(x.shape) != (rows, W - 1, H, d):
                    raise ValueError(f"conv window {t} has shape {tuple(x.shape)}, "
                                     f"expected {(rows, W - 1, H, d)}")
    per_head = out_gate is not None and out_gate.dim() == 2
    if out_gate is not None:
        want = (gate_rows, H) if per_head else (gate_rows, H, dv)
        if tuple(out_gate.shape) != want:
            raise ValueError(f"out_gate has shape {tuple(out_gate.shape)}, expected {want}")
    la = LayerArgs()
    if conv_weights is not None:
        la.conv_width, la.conv_silu = W, 1 if conv_silu else 0
        for t in range(3):
            la.conv_w[t] = _ptr(conv_weights[t], torch.float32, "conv_weights")
            for arr, src in ((la.conv_in, conv_window), (la.conv_out, conv_window_out)):
                arr[t] = _ptr(None if src is None else src[t], dtype, "conv window")
    if out_gate is not None:
        la.out_gate = _ptr(out_gate, dtype, "out_gate")
        la.out_gate_per_head = 1 if per_head else 0
    return la


def _check_shapes(q, k, v, g, b, cu_seqlens, o, initial_state, final_state):
    """Shapes of the per-token tensors and of the states, from q's [T, H, dk]
    and v's dv.  The C ABI receives bare pointers and cannot check them, so a
    wrong shape would make the kernels (or the host copies) run past a buffer:
    every shape is checked before any pointer is taken."""
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError(f"q and v must be [T, H, d], got {tuple(q.shape)} and {tuple(v.shape)}")
    T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError(f"cu_seqlens must be [N + 1] with N >= 1, got {tuple(cu_seqlens.shape)}")
    N = cu_seqlens.numel() - 1
    gshape = (T, H) if g.dim() == 2 else (T, H, dk)  # [T, H]: one decay per token and head
    checks = [("k", k, (T, H, dk)), ("g", g, gshape), ("v", v, (T, H, dv)), ("b", b, (T, H)),
              ("o", o, (T, H, dv))]
    checks += [(name, t, (N, H, dk, dv)) for name, t in (("initial_state", initial_state),
                                                          ("final_state", final_state))
               if t is not None]
    for name, t, shp in checks:
        if tuple(t.shape) != shp:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shp}")
    return T, H, dk, dv, N


def make_prefill_args(q, k, v, g, b, cu_seqlens, o, *, scale=1.0, initial_state=None,
                      final_state=None, snapshot_interval=0, boundary_pos=None,
                      cu_boundaries=None, cu_snapshots=None, snapshots=None,
                      scan_segments=0, snapshot_slot_map=None, wait_limit_ns=0,
                      layer: LayerArgs | None = None, schedule=SCHEDULE_AUTO) -> PrefillArgs:
    T, H, dk, dv, N = _check_shapes(q, k, v, g, b, cu_seqlens, o, initial_state, final_state)
    dt = q.dtype
    if snapshots is not None and (snapshots.dim() != 4 or tuple(snapshots.shape[1:]) != (H, dk, dv)):
        raise ValueError(f"snapshots has shape {tuple(snapshots.shape)}, expected [rows, {H}, {dk}, {dv}]")
    if cu_snapshots is not None and tuple(cu_snapshots.shape) != (N + 1,):
        raise ValueError(f"cu_snapshots has shape {tuple(cu_snapshots.shape)}, expected ({N + 1},)")
    if cu_boundaries is not None and tuple(cu_boundaries.shape) != (N + 1,):
        raise ValueError(f"cu_boundaries has shape {tuple(cu_boundaries.shape)}, expected ({N + 1},)")
    a = PrefillArgs()
    a.num_seqs = N
    a.num_heads, a.dk, a.dv, a.total_tokens = H, dk, dv, T
    a.cu_seqlens = _ptr(cu_seqlens, torch.int64, "cu_seqlens")
    a.in_dtype = _dtype_code(dt)
    a.q, a.k, a.v = _ptr(q, dt, "q"), _ptr(k, dt, "k"), _ptr(v, dt, "v")
    a.g, a.b, a.o = _ptr(g, dt, "g"), _ptr(b, dt, "b"), _ptr(o, dt, "o")
    a.scale = float(scale)
    a.initial_state = _ptr(initial_state, torch.float32, "initial_state")
    a.final_state = _ptr(final_state, torch.float32, "final_state")
    a.snapshot_interval = int(snapshot_interval)
    a.boundary_pos = _ptr(boundary_pos, torch.int64, "boundary_pos")
    a.cu_boundaries = _ptr(cu_boundaries, torch.int64, "cu_boundaries")
    a.num_boundaries = 0 if boundary_pos is None else boundary_pos.numel()
    a.cu_snapshots = _ptr(cu_snapshots, torch.int64, "cu_snapshots")
    a.snapshots = _ptr(snapshots, torch.float32, "snapshots")
    a.num_snapshots = 0 if snapshots is None else snapshots.shape[0]
    a.scan_segments = int(scan_segments)
    a.snapshot_slot_map = _ptr(snapshot_slot_map, torch.int32, "snapshot_slot_map")
    a.snapshot_map_len = 0 if snapshot_slot_map is None else snapshot_slot_map.numel()
    a.wait_limit_ns = int(wait_limit_ns)
    a.gate_per_head = 1 if g.dim() == 2 else 0
    if layer is not None:
        a.layer = ctypes.pointer(layer)  # the pointer object keeps `layer` alive
    a.schedule = int(schedule)
    return a


# ----------------------------------------------------------------- the C entry points
def kda_prefill_workspace_size(args: PrefillArgs) -> int:
    return int(lib().kda_prefill_workspace_size(ctypes.byref(args)))


def kda_prefill_schedule(args: PrefillArgs, sm_count: int = 0) -> int:
    """The path kda_prefill takes for ``args`` on a GPU with ``sm_count`` SMs
    (0: the current device); one of the PATH_* values, -1 if invalid."""
    return int(lib().kda_prefill_schedule(ctypes.byref(args), int(sm_count)))


def kda_prefill(args: PrefillArgs, workspace: torch.Tensor, stream=None) -> None:
    """Launches the prefill described by ``args`` (see make_prefill_args)."""
    ws = _ptr(workspace, torch.uint8, "workspace")
    _check(lib().kda_prefill(ctypes.byref(args), ws, workspace.numel(), _stream(stream)),
           "kda_prefill")


def _host_ptr(t: torch.Tensor | None, dtype=None, name: str = "") -> int | None:
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def make_prefill_host_args(q, k, v, g, b, cu_seqlens, o, *, scale=1.0, initial_state=None,
                           final_state=None, segments=0, copy_in_stream=None,
                           copy_out_stream=None) -> PrefillHostArgs:
    """kda_prefill_host_args over HOST tensors (pinned for overlapped copies)."""
    T, H, dk, dv, N = _check_shapes(q, k, v, g, b, cu_seqlens, o, initial_state, final_state)
    dt = q.dtype
    a = PrefillHostArgs()
    a.num_seqs = N
    a.num_heads, a.dk, a.dv, a.total_tokens = H, dk, dv, T
    a.cu_seqlens = _host_ptr(cu_seqlens, torch.int64, "cu_seqlens")
    a.in_dtype = _dtype_code(dt)
    a.q, a.k, a.v = _host_ptr(q, dt, "q"), _host_ptr(k, dt, "k"), _host_ptr(v, dt, "v")
    a.g, a.b, a.o = _host_ptr(g, dt, "g"), _host_ptr(b, dt, "b"), _host_ptr(o, dt, "o")
    a.scale = float(scale)
    a.initial_state = _host_ptr(initial_state, torch.float32, "initial_state")
    a.final_state = _host_ptr(final_state, torch.float32, "final_state")
    a.segments = int(segments)
    a.copy_in_stream = None if copy_in_stream is None else _stream(copy_in_stream)
    a.copy_out_stream = None if copy_out_stream is None else _stream(copy_out_stream)
    a.gate_per_head = 1 if g.dim() == 2 else 0
    return a


def kda_prefill_host_workspace_size(args: PrefillHostArgs) -> int:
    return int(lib().kda_prefill_host_workspace_size(ctypes.byref(args)))


def kda_prefill_host(args: PrefillHostArgs, workspace: torch.Tensor, stream=None) -> None:
    """Enqueues the host-buffer prefill described by ``args``; the host
    outputs are complete once ``stream`` has passed this point."""
    ws = _ptr(workspace, torch.uint8, "workspace")
    _check(lib().kda_prefill_host(ctypes.byref(args), ws, workspace.numel(), _stream(stream)),
           "kda_prefill_host")


def kda_prefill_noalloc(args: PrefillArgs, stream=None) -> None:
    """kda_prefill on the library's fixed workspace (for callers that cannot
    allocate device memory at the call); see include/kda.h for its limits."""
    _check(lib().kda_prefill_noalloc(ctypes.byref(args), _stream(stream)), "kda_prefill_noalloc")


def kda_prefill_noalloc_device_status(stream=None) -> int:
    """The status word of the last kda_prefill_noalloc on the current device."""
    out = c_i32(0)
    _check(lib().kda_prefill_noalloc_device_status(ctypes.byref(out), _stream(stream)),
           "kda_prefill_noalloc_device_status")
    return int(out.value)


def kda_prefill_device_status(workspace: torch.Tensor, stream=None) -> int:
    out = c_i32(0)
    _check(lib().kda_prefill_device_status(_ptr(workspace, name="workspace"), ctypes.byref(out),
                                           _stream(stream)), "kda_prefill_device_status")
    return int(out.value)


def kda_snapshot_plan(cu_seqlens, interval: int, boundary_pos=None, cu_boundaries=None):
    """Host helper: (cu_snapshots int64 [N+1] numpy, n_snap)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens.cpu() if torch.is_tensor(cu_seqlens)
                                         else cu_seqlens, dtype=np.int64))
    n = cu.shape[0] - 1
    out = np.zeros(n + 1, dtype=np.int64)
    bp = cb = None
    if boundary_pos is not None:
        bp = np.ascontiguousarray(np.asarray(boundary_pos.cpu() if torch.is_tensor(boundary_pos)
                                             else boundary_pos, dtype=np.int64))
        cb = np.ascontiguousarray(np.asarray(cu_boundaries.cpu() if torch.is_tensor(cu_boundaries)
                                             else cu_boundaries, dtype=np.int64))
    n_snap = lib().kda_snapshot_plan(cu.ctypes.data, n, int(interval),
                                     None if bp is None else bp.ctypes.data,
                                     None if cb is None else cb.ctypes.data, out.ctypes.data)
    if n_snap < 0:
        raise ValueError("kda_snapshot_plan: invalid sequence lengths or boundary positions")
    return out, int(n_snap)


def kda_decode_step(q, k, v, g, b, state, o, state_slots=None, scale=1.0, stream=None,
                    wait_limit_ns=0, status=None, conv_weights=None, conv_silu=False,
                    conv_window=None, out_gate=None) -> None:
    """One decode step.  With conv_weights (wq, wk, wv) [W, H, d] the short
    convolution runs on q, k, v; conv_window (q, k, v) [slots, W-1, H, d] holds
    each slot's window and is advanced in place.  out_gate [B, H, dv] or
    [B, H] gates o."""
    if q.dim() != 3 or v.dim() != 3 or state.dim() != 4:
        raise ValueError("q, v must be [B, H, d] and state [slots, H, dk, dv]")
    B, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if tuple(state.shape[1:]) != (H, dk, dv):
        raise ValueError(f"state has shape {tuple(state.shape)}, expected [slots, {H}, {dk}, {dv}]")
    gshape = (B, H) if g.dim() == 2 else (B, H, dk)  # [B, H]: one decay per row and head
    for name, t, shp in (("k", k, (B, H, dk)), ("g", g, gshape), ("v", v, (B, H, dv)),
                         ("b", b, (B, H)), ("o", o, (B, H, dv))):
        if tuple(t.shape) != shp:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shp}")
    if state_slots is not None and tuple(state_slots.shape) != (B,):
        raise ValueError(f"state_slots has shape {tuple(state_slots.shape)}, expected ({B},)")
    if status is not None and status.numel() < 1:
        raise ValueError("status needs one int32")
    a = DecodeArgs()
    a.batch, a.num_heads, a.dk, a.dv = B, H, dk, dv
    a.num_slots = state.shape[0]
    a.in_dtype = _dtype_code(dt)
    a.scale = float(scale)
    a.q, a.k, a.v = _ptr(q, dt, "q"), _ptr(k, dt, "k"), _ptr(v, dt, "v")
    a.g, a.b, a.o = _ptr(g, dt, "g"), _ptr(b, dt, "b"), _ptr(o, dt, "o")
    a.state = _ptr(state, torch.float32, "state")
    a.state_slots = _ptr(state_slots, torch.int32, "state_slots")
    a.wait_limit_ns = int(wait_limit_ns)
    a.status = _ptr(status, torch.int32, "status")
    a.gate_per_head = 1 if g.dim() == 2 else 0  # g [B, H]: one decay per row and head
    layer = make_layer_args(rows=a.num_slots, H=H, dk=dk, dv=dv, dtype=dt,
                            conv_weights=conv_weights, conv_silu=conv_silu,
                            conv_window=conv_window, conv_window_out=conv_window,
                            out_gate=out_gate, gate_rows=B)
    if layer is not None:
        a.layer = ctypes.pointer(layer)
    _check(lib().kda_decode_step(ctypes.byref(a), _stream(stream)), "kda_decode_step")


def kda_prep(q, k, g, b, cu_seqlens, qhat, khat, G, beta, stream=None, conv_weights=None,
             conv_silu=False, conv_window=None) -> None:
    """The preparation step.  With conv_weights (wq, wk, ...) [W, H, dk] q and k
    pass through the short convolution first (conv_window: (q, k) windows
    [N, W-1, H, dk] before each sequence, or None)."""
    if q.dim() != 3 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("q must be [T, H, dk] and cu_seqlens [N + 1]")
    T, H, dk = q.shape
    dt = q.dtype
    gshape = (T, H) if g.dim() == 2 else (T, H, dk)  # [T, H]: one decay per token and head
    for name, t, shp in (("k", k, (T, H, dk)), ("g", g, gshape), ("b", b, (T, H)),
                         ("qhat", qhat, (T, H, dk)), ("khat", khat, (T, H, dk)),
                         ("G", G, (T, H, dk)), ("beta", beta, (T, H))):
        if tuple(t.shape) != shp:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shp}")
    a = PrepArgs()
    a.num_seqs, a.num_heads, a.dk, a.total_tokens = cu_seqlens.numel() - 1, H, dk, T
    a.cu_seqlens = _ptr(cu_seqlens, torch.int64, "cu_seqlens")
    a.in_dtype = _dtype_code(dt)
    a.q, a.k, a.g, a.b = _ptr(q, dt, "q"), _ptr(k, dt, "k"), _ptr(g, dt, "g"), _ptr(b, dt, "b")
    a.qhat, a.khat = _ptr(qhat, torch.float32, "qhat"), _ptr(khat, torch.float32, "khat")
    a.G, a.beta = _ptr(G, torch.float32, "G"), _ptr(beta, torch.float32, "beta")
    a.gate_per_head = 1 if g.dim() == 2 else 0  # g [T, H]: one decay per token and head
    if conv_weights is not None:
        la = LayerArgs()
        W = conv_weights[0].shape[0]
        if not 1 <= W <= CONV_MAX:
            raise ValueError(f"conv width {W} outside 1..{CONV_MAX}")
        la.conv_width, la.conv_silu = W, 1 if conv_silu else 0
        N = cu_seqlens.numel() - 1
        for t in range(2):
            if tuple(conv_weights[t].shape) != (W, H, dk):
                raise ValueError(f"conv weights {t} have shape {tuple(conv_weights[t].shape)}")
            la.conv_w[t] = _ptr(conv_weights[t], torch.float32, "conv_weights")
            x = None if conv_window is None else conv_window[t]
            if x is not None and tuple(x.shape) != (N, W - 1, H, dk):
                raise ValueError(f"conv window {t} has shape {tuple(x.shape)}")
            la.conv_in[t] = _ptr(x, dt, "conv window")
        a.layer = ctypes.pointer(la)
    _check(lib().kda_prep(ctypes.byref(a), _stream(stream)), "kda_prep")


# ----------------------------------------------------------------- conveniences
class Prefill:
    """A planned prefill call: outputs, workspace and snapshot slots are
    allocated once (torch device memory); ``run()`` only launches kernels.

    Host copies of cu_seqlens (and boundaries) are needed to size the
    snapshot buffer; pass them as ``lens`` to avoid a device->host read."""

    def __init__(self, q, k, v, g, b, cu_seqlens, *, scale=1.0, initial_state=None,
                 snapshot_interval=0, boundary_pos=None, cu_boundaries=None,
                 want_final=True, host_cu_seqlens=None, host_boundary_pos=None,
                 host_cu_boundaries=None, o=None, scan_segments=0, snapshot_pool=None,
                 snapshot_slot_map=None, wait_limit_ns=0, conv_weights=None, conv_silu=False,
                 conv_window=None, conv_window_out=None, out_gate=None, schedule=SCHEDULE_AUTO):
        """The layer steps: conv_weights (wq, wk, wv) float32 [W, H, d] turn on
        the short convolution, with each sequence's window before the call in
        conv_window ((q, k, v) [N, W-1, H, d], None = zeros); conv_window_out
        receives the windows after it (True allocates them as
        ``self.conv_window_out``; it may be conv_window itself).  out_gate
        [T, H, dv] or [T, H] gates o."""
        dev = q.device
        T, H, dk = q.shape
        dv = v.shape[-1]
        N = cu_seqlens.numel() - 1
        self.o = torch.empty(T, H, dv, dtype=q.dtype, device=dev) if o is None else o
        self.final_state = (torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
                            if want_final else None)
        self.cu_snapshots = self.snapshots = None
        self.n_snap = 0
        if snapshot_interval > 0 or boundary_pos is not None:
            hcu = cu_seqlens.cpu() if host_cu_seqlens is None else host_cu_seqlens
            hbp = (None if boundary_pos is None else
                   (boundary_pos.cpu() if host_boundary_pos is None else host_boundary_pos))
            hcb = (None if cu_boundaries is None else
                   (cu_boundaries.cpu() if host_cu_boundaries is None else host_cu_boundaries))
            cs, n_snap = kda_snapshot_plan(hcu, snapshot_interval, hbp, hcb)
            self.n_snap = n_snap
            self.cu_snapshots = torch.from_numpy(cs).to(dev)
            if snapshot_pool is not None:
                # snapshots go to the pool rows the slot map names
                self.snapshots = snapshot_pool
            else:
                self.snapshots = torch.empty(max(n_snap, 1), H, dk, dv, dtype=torch.float32,
                                             device=dev)
        self.conv_window_out = None
        if conv_weights is not None and conv_window_out is not None:
            W = conv_weights[0].shape[0]
            if conv_window_out is True:
                conv_window_out = tuple(torch.empty(N, W - 1, H, d, dtype=q.dtype, device=dev)
                                        for d in (dk, dk, dv))
            self.conv_window_out = conv_window_out
        self.layer = make_layer_args(rows=N, H=H, dk=dk, dv=dv, dtype=q.dtype,
                                     conv_weights=conv_weights, conv_silu=conv_silu,
                                     conv_window=conv_window,
                                     conv_window_out=self.conv_window_out, out_gate=out_gate,
                                     gate_rows=T)
        self.args = make_prefill_args(
            q, k, v, g, b, cu_seqlens, self.o, scale=scale, initial_state=initial_state,
            final_state=self.final_state, snapshot_interval=snapshot_interval,
            boundary_pos=boundary_pos, cu_boundaries=cu_boundaries,
            cu_snapshots=self.cu_snapshots, snapshots=self.snapshots,
            scan_segments=scan_segments,
            snapshot_slot_map=snapshot_slot_map if self.snapshots is not None else None,
            wait_limit_ns=wait_limit_ns, layer=self.layer, schedule=schedule)
        nbytes = kda_prefill_workspace_size(self.args)
        if nbytes == 0:
            raise ValueError("kda_prefill_workspace_size rejected the arguments")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self._keep = (q, k, v, g, b, cu_seqlens, initial_state, boundary_pos, cu_boundaries,
                      snapshot_slot_map, conv_weights, conv_window, out_gate)

    def run(self, stream=None):
        kda_prefill(self.args, self.workspace, stream)
        return self

    def device_status(self, stream=None) -> int:
        return kda_prefill_device_status(self.workspace, stream)

    @property
    def snapshot_view(self):
        return None if self.snapshots is None else self.snapshots[: self.n_snap]


def prefill(q, k, v, g, b, cu_seqlens, **kw):
    """Allocates, runs and returns (o, final_state, snapshots) on the device."""
    p = Prefill(q, k, v, g, b, cu_seqlens, **kw).run()
    return p.o, p.final_state, p.snapshot_view


_side_streams = {}


def _streams(device):
    """Two side streams per device (host->device copies, device->host copies)."""
    key = torch.device(device).index or 0
    if key not in _side_streams:
        _side_streams[key] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    return _side_streams[key]


def prefill_host(q, k, v, g, b, cu_seqlens, *, device="cuda", stream=None, segments=None,
                 scale=1.0, initial_state=None, want_final=True, **kw):
    """End-to-end prefill from host tensors through ``kda_prefill_host``:
    inputs copied in, prefill, o and the final state copied back, pipelined
    over ``segments`` pieces of the batch (None = the library's choice).
    Returns host (o, final_state), complete when this returns.

    Snapshots and boundary positions need device buffers: with those
    arguments the inputs are copied to the device and ``kda_prefill`` runs
    as one call."""
    s = torch.cuda.current_stream(device) if stream is None else stream
    if kw.get("snapshot_interval", 0) or kw.get("boundary_pos") is not None:
        with torch.cuda.stream(s):
            dq, dk_, dv_, dg, db = (t.to(device, non_blocking=True) for t in (q, k, v, g, b))
            dcu = cu_seqlens.to(device, non_blocking=True)
            dinit = None if initial_state is None else initial_state.to(device, non_blocking=True)
            p = Prefill(dq, dk_, dv_, dg, db, dcu, scale=scale, initial_state=dinit,
                        want_final=want_final, host_cu_seqlens=cu_seqlens, **kw).run(s)
            o = torch.empty(p.o.shape, dtype=p.o.dtype, pin_memory=True)
            o.copy_(p.o, non_blocking=True)
            fs = None
            if p.final_state is not None:
                fs = torch.empty(p.final_state.shape, dtype=torch.float32, pin_memory=True)
                fs.copy_(p.final_state, non_blocking=True)
        s.synchronize()
        return o, fs
    if kw:
        raise TypeError(f"unexpected arguments {sorted(kw)}")
    p = PrefillHost(q, k, v, g, b, cu_seqlens, device=device, segments=segments, scale=scale,
                    initial_state=initial_state, want_final=want_final)
    p.run(s)
    s.synchronize()
    return p.o, p.final_state


class PrefillHost:
    """A planned host-buffer prefill (``kda_prefill_host``): the pinned host
    outputs, the device workspace and the argument block are made once;
    ``run()`` enqueues the copies in, the kernels and the copies out.  The
    inputs are the host tensors given here (refill them in place between
    runs); o and final_state are complete once ``stream`` passes the run."""

    def __init__(self, q, k, v, g, b, cu_seqlens, *, device="cuda", segments=None, scale=1.0,
                 initial_state=None, want_final=True):
        T, H, dk = q.shape
        dv = v.shape[-1]
        N = cu_seqlens.numel() - 1
        self.o = torch.empty(T, H, dv, dtype=q.dtype, pin_memory=True)
        self.final_state = (torch.empty(N, H, dk, dv, dtype=torch.float32, pin_memory=True)
                            if want_final else None)
        self.copy_in, self.copy_out = _streams(device)
        self.args = make_prefill_host_args(
            q, k, v, g, b, cu_seqlens, self.o, scale=scale, initial_state=initial_state,
            final_state=self.final_state, segments=segments or 0, copy_in_stream=self.copy_in,
            copy_out_stream=self.copy_out)
        nbytes = kda_prefill_host_workspace_size(self.args)
        if nbytes == 0:
            raise ValueError("kda_prefill_host_workspace_size rejected the arguments")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self._keep = (q, k, v, g, b, cu_seqlens, initial_state)

    def run(self, stream=None):
        kda_prefill_host(self.args, self.workspace, stream)
        return self


class PrefixCache:
    """The snapshot retention policy of kda.h (``kda_prefix_cache_*``): which
    row of a device state pool holds the state after which prefix of token
    ids.  Host-side only; the pool itself is a tensor the caller owns."""

    def __init__(self, num_rows: int):
        self._h = lib().kda_prefix_cache_create(int(num_rows))
        if not self._h:
            raise ValueError("kda_prefix_cache_create failed")
        self.num_rows = int(num_rows)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.kda_prefix_cache_destroy(h)

    @staticmethod
    def _tokens(tokens):
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return t, (t.ctypes.data if t.size else None)

    def entries(self) -> int:
        return int(lib().kda_prefix_cache_entries(self._h))

    def lookup(self, tokens):
        """(p, row): the longest cached prefix of ``tokens`` and its pool row
        (0, -1 if none)."""
        t, tp = self._tokens(tokens)
        row = c_i32(-1)
        p = lib().kda_prefix_cache_lookup(self._h, tp, t.size, ctypes.byref(row))
        if p < 0:
            raise ValueError("kda_prefix_cache_lookup rejected the arguments")
        return int(p), int(row.value)

    def reserve(self, tokens, positions, boundary=None, keep_row=-1):
        """Rows for the states at ``positions`` (increasing, 1..len(tokens));
        ``boundary``: per position, True for prompt-boundary checkpoints;
        ``keep_row``: a row not to evict (the one being resumed from).
        Returns an int32 array (-1: already cached or no row)."""
        t, tp = self._tokens(tokens)
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
        bnd = None if boundary is None else np.ascontiguousarray(np.asarray(boundary, dtype=np.uint8))
        if bnd is not None and bnd.size != pos.size:
            raise ValueError("boundary needs one flag per position")
        rows = np.full(pos.size, -1, dtype=np.int32)
        n = lib().kda_prefix_cache_reserve(self._h, tp, t.size, pos.ctypes.data if pos.size else None,
                                           None if bnd is None else bnd.ctypes.data, pos.size,
                                           int(keep_row), rows.ctypes.data if pos.size else None)
        if n < 0:
            raise ValueError("kda_prefix_cache_reserve rejected the arguments")
        return rows

    def forget(self, rows) -> int:
        """Drops the entries of ``rows`` (as returned by reserve; -1 entries
        are ignored) and frees their rows: for a prefill that failed before
        writing them.  Returns the number of rows freed."""
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n = lib().kda_prefix_cache_forget(self._h, r.ctypes.data if r.size else None, r.size)
        if n < 0:
            raise ValueError("kda_prefix_cache_forget rejected the arguments")
        return int(n)


def prefill_cached(cache: PrefixCache, pool, tokens, q, k, v, g, b, *, interval=4096,
                   scale=1.0, stream=None):
    """One prompt through the prefix cache (single sequence, device tensors
    [T, H, .] for all of its tokens): resume from the longest cached prefix
    p, prefill tokens p..T with ``kda_prefill`` from the pool row's state,
    and save the states at the multiples of ``interval`` past p and at the
    prompt end into the rows the cache assigns (``snapshot_slot_map``).
    Returns (p, o for tokens p..T, final state [1, H, dk, dv])."""
    T = q.shape[0]
    if len(tokens) != T:
        raise ValueError("one token id per row of q")
    if T == 0:
        raise ValueError("an empty prompt has nothing to prefill")
    p, row = cache.lookup(tokens)
    if p == T:
        # the whole prompt is cached: nothing to run, the state is the row's
        return p, q.new_empty((0,) + tuple(v.shape[1:])), pool[row:row + 1].clone()
    absolute = [x for x in range(interval * (p // interval + 1), T, interval)] if interval > 0 else []
    absolute.append(T)
    rows = cache.reserve(tokens, absolute, [False] * (len(absolute) - 1) + [True], keep_row=row)
    dev = q.device
    rel = torch.tensor([x - p for x in absolute], dtype=torch.int64)
    cu_b = torch.tensor([0, len(absolute)], dtype=torch.int64)
    hcu = torch.tensor([0, T - p], dtype=torch.int64)
    try:
        pr = Prefill(q[p:], k[p:], v[p:], g[p:], b[p:], hcu.to(dev),
                     scale=scale, initial_state=pool[row:row + 1] if p > 0 else None,
                     boundary_pos=rel.to(dev), cu_boundaries=cu_b.to(dev),
                     host_cu_seqlens=hcu, host_boundary_pos=rel, host_cu_boundaries=cu_b,
                     snapshot_pool=pool, snapshot_slot_map=torch.from_numpy(rows).to(dev))
        pr.run(stream)
    except Exception:
        cache.forget(rows)  # the rows were never written: no lookup may resume from them
        raise
    return p, pr.o, pr.final_state


def decode_step(q, k, v, g, b, state, state_slots=None, scale=1.0, o=None, stream=None, **layer):
    """Allocates o and runs kda_decode_step; ``layer`` takes conv_weights,
    conv_silu, conv_window and out_gate (see kda_decode_step)."""
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[-1], dtype=q.dtype, device=q.device)
    kda_decode_step(q, k, v, g, b, state, o, state_slots=state_slots, scale=scale, stream=stream,
                    **layer)
    return o


def prep(q, k, g, b, cu_seqlens, stream=None, **conv):
    """Allocates and runs kda_prep; ``conv`` takes conv_weights, conv_silu and
    conv_window (see kda_prep)."""
    T, H, dk = q.shape
    f = dict(dtype=torch.float32, device=q.device)
    qhat, khat, G = (torch.empty(T, H, dk, **f) for _ in range(3))
    beta = torch.empty(T, H, **f)
    kda_prep(q, k, g, b, cu_seqlens, qhat, khat, G, beta, stream=stream, **conv)
    return qhat, khat, G, beta
