"""Thin Python binding of libgsa (include/gsa.h): argument marshalling only.

Functions with the C names (``grouped_scaled_act_fwd``, ``grouped_scaled_act_bwd``,
``gsa_layout``, ``gsa_workspace_size``, ``gsa_workspace_status``) take raw
pointers/ints exactly like the C ABI.  ``fwd`` / ``bwd`` are conveniences that
allocate output tensors with PyTorch (device memory is PyTorch's job here) and
call the C functions; every step of the computation runs in the CUDA kernel.
There is no fallback: if libgsa.so is missing or cannot load, this module
raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgsa.so")

ACT = {"srelu": 0, "tanh_srelu": 1, "swiglu": 2, "clamped_swiglu": 3, "gelu": 4, "sigmoid": 5, "identity": 6}
GLU_ACTS = (2, 3)
MXFP8, NVFP4 = 0, 1
SCALES_COMPACT, SCALES_TILED = 0, 1
STATUS = {0: "GSA_OK", 1: "GSA_ERR_INVALID_ARG", 2: "GSA_ERR_UNSUPPORTED", 3: "GSA_ERR_ALIGNMENT",
          4: "GSA_ERR_WORKSPACE", 5: "GSA_ERR_CUDA", 6: "GSA_ERR_DEVICE_TIMEOUT"}

EXPORTED = ["gsa_layout", "gsa_workspace_size", "grouped_scaled_act_fwd", "grouped_scaled_act_bwd",
            "gsa_workspace_status", "gsa_last_launch_count", "gsa_status_string", "gsa_version",
            "gsa_fwd_noalloc", "gsa_fwd_noalloc_status", "gsa_layout_bound", "gsa_workspace_size_graph_safe",
            "grouped_scaled_act_fwd_graph_safe", "grouped_scaled_act_bwd_graph_safe", "gsa_selftest_wait_timeout",
            "gsa_layout_ex", "gsa_layout_bound_ex"]


class GsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class ActParams(ctypes.Structure):
    _fields_ = [("s", ctypes.c_float), ("limit", ctypes.c_float), ("alpha", ctypes.c_float),
                ("glu_linear_offset", ctypes.c_float)]


class Recipe(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("rht_colwise", ctypes.c_int32), ("rht_sign_mask", ctypes.c_uint32),
                ("scale_layout", ctypes.c_int32)]


class QOut(ctypes.Structure):
    _fields_ = [("row_data", ctypes.c_void_p), ("row_scale", ctypes.c_void_p), ("col_data", ctypes.c_void_p),
                ("col_scale", ctypes.c_void_p), ("amax_row", ctypes.c_void_p), ("amax_col", ctypes.c_void_p)]


class LayoutInfo(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("row_data_bytes", ctypes.c_int64), ("row_scale_bytes", ctypes.c_int64),
                ("col_data_bytes", ctypes.c_int64), ("col_scale_bytes", ctypes.c_int64),
                ("amax_floats", ctypes.c_int64)]


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def load():
    """Load libgsa.so (building it first if only the sources are present)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            from . import build
            build.build()
        L = ctypes.CDLL(LIB_PATH)
        L.gsa_layout.restype = ctypes.c_int
        L.gsa_layout.argtypes = [_I64, _P, _I64, ctypes.c_int32, ctypes.POINTER(LayoutInfo), _P, _P]
        L.gsa_workspace_size.restype = ctypes.c_size_t
        L.gsa_workspace_size.argtypes = [_I64, _P, _I64, ctypes.c_int32, ctypes.c_int32]
        L.grouped_scaled_act_fwd.restype = ctypes.c_int
        L.grouped_scaled_act_fwd.argtypes = [_P, _P, _P, _I64, _I64, ctypes.c_int32, ctypes.POINTER(ActParams),
                                             ctypes.POINTER(Recipe), ctypes.POINTER(QOut), _P, _P, ctypes.c_size_t, _P]
        L.grouped_scaled_act_bwd.restype = ctypes.c_int
        L.grouped_scaled_act_bwd.argtypes = [_P, _P, _P, _P, _I64, _I64, ctypes.c_int32, ctypes.POINTER(ActParams),
                                             ctypes.POINTER(Recipe), _P, ctypes.POINTER(QOut), _P,
                                             ctypes.POINTER(QOut), _P, ctypes.c_size_t, _P]
        L.gsa_fwd_noalloc.restype = ctypes.c_int
        L.gsa_fwd_noalloc.argtypes = [_P, _P, _P, _I64, _I64, ctypes.c_int32, ctypes.POINTER(ActParams),
                                      ctypes.POINTER(Recipe), ctypes.POINTER(QOut), _P, _P]
        L.gsa_fwd_noalloc_status.restype = ctypes.c_int
        L.gsa_fwd_noalloc_status.argtypes = [_P]
        L.gsa_layout_ex.restype = ctypes.c_int
        L.gsa_layout_ex.argtypes = [_I64, _P, _I64, ctypes.POINTER(Recipe), ctypes.POINTER(LayoutInfo), _P, _P, _P]
        L.gsa_layout_bound_ex.restype = ctypes.c_int
        L.gsa_layout_bound_ex.argtypes = [_I64, _I64, _I64, ctypes.POINTER(Recipe), ctypes.POINTER(LayoutInfo)]
        L.gsa_layout_bound.restype = ctypes.c_int
        L.gsa_layout_bound.argtypes = [_I64, _I64, _I64, ctypes.c_int32, ctypes.POINTER(LayoutInfo)]
        L.gsa_workspace_size_graph_safe.restype = ctypes.c_size_t
        L.gsa_workspace_size_graph_safe.argtypes = [_I64, _I64, _I64, ctypes.c_int32, ctypes.c_int32]
        L.grouped_scaled_act_fwd_graph_safe.restype = ctypes.c_int
        L.grouped_scaled_act_fwd_graph_safe.argtypes = [_P, _P, _P, _I64, _I64, _I64, ctypes.c_int32,
                                                        ctypes.POINTER(ActParams), ctypes.POINTER(Recipe),
                                                        ctypes.POINTER(QOut), _P, _P, _P, ctypes.c_size_t, _P]
        L.grouped_scaled_act_bwd_graph_safe.restype = ctypes.c_int
        L.grouped_scaled_act_bwd_graph_safe.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int32,
                                                        ctypes.POINTER(ActParams), ctypes.POINTER(Recipe), _P,
                                                        ctypes.POINTER(QOut), _P, ctypes.POINTER(QOut), _P, _P,
                                                        ctypes.c_size_t, _P]
        L.gsa_selftest_wait_timeout.restype = ctypes.c_int
        L.gsa_selftest_wait_timeout.argtypes = [_P, ctypes.c_int32, ctypes.c_uint32, _P]
        L.gsa_workspace_status.restype = ctypes.c_int
        L.gsa_workspace_status.argtypes = [_P, _P]
        L.gsa_last_launch_count.restype = ctypes.c_int32
        L.gsa_last_launch_count.argtypes = []
        L.gsa_status_string.restype = ctypes.c_char_p
        L.gsa_status_string.argtypes = [ctypes.c_int]
        L.gsa_version.restype = ctypes.c_int32
        L.gsa_version.argtypes = []
        _lib = L
    return _lib


# ------------------------------------------------------------ C-named calls

def _split_array(split_sizes):
    arr = (ctypes.c_int64 * len(split_sizes))(*[int(s) for s in split_sizes])
    return arr


def gsa_layout(split_sizes, width: int, recipe_kind: int):
    """-> (LayoutInfo, col_data_offsets[E+1], col_scale_offsets[E+1])."""
    E = len(split_sizes)
    info = LayoutInfo()
    d = (ctypes.c_int64 * (E + 1))()
    s = (ctypes.c_int64 * (E + 1))()
    st = load().gsa_layout(E, ctypes.cast(_split_array(split_sizes), _P), int(width), int(recipe_kind),
                           ctypes.byref(info), ctypes.cast(d, _P), ctypes.cast(s, _P))
    if st != 0:
        raise GsaError(st, "gsa_layout")
    return info, list(d), list(s)


def gsa_layout_ex(split_sizes, width: int, recipe: Recipe):
    """-> (LayoutInfo, col_data_offsets[E+1], col_scale_offsets[E+1], row_scale_offsets[E+1])."""
    E = len(split_sizes)
    info = LayoutInfo()
    d = (ctypes.c_int64 * (E + 1))()
    s = (ctypes.c_int64 * (E + 1))()
    r = (ctypes.c_int64 * (E + 1))()
    st = load().gsa_layout_ex(E, ctypes.cast(_split_array(split_sizes), _P), int(width), ctypes.byref(recipe),
                              ctypes.byref(info), ctypes.cast(d, _P), ctypes.cast(s, _P), ctypes.cast(r, _P))
    if st != 0:
        raise GsaError(st, "gsa_layout_ex")
    return info, list(d), list(s), list(r)


def gsa_layout_bound_ex(E: int, M: int, width: int, recipe: Recipe) -> LayoutInfo:
    info = LayoutInfo()
    st = load().gsa_layout_bound_ex(int(E), int(M), int(width), ctypes.byref(recipe), ctypes.byref(info))
    if st != 0:
        raise GsaError(st, "gsa_layout_bound_ex")
    return info


def gsa_workspace_size(split_sizes, w_in: int, act_kind: int, recipe_kind: int) -> int:
    return int(load().gsa_workspace_size(len(split_sizes), ctypes.cast(_split_array(split_sizes), _P), int(w_in),
                                         int(act_kind), int(recipe_kind)))


def grouped_scaled_act_fwd(x_ptr, probs_ptr, split_sizes, w_in, act_kind, act_params: ActParams, recipe: Recipe,
                           y_q: QOut, y_bf16_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    return load().grouped_scaled_act_fwd(x_ptr, probs_ptr, ctypes.cast(_split_array(split_sizes), _P),
                                         len(split_sizes), int(w_in), int(act_kind), ctypes.byref(act_params),
                                         ctypes.byref(recipe), ctypes.byref(y_q) if y_q is not None else None,
                                         y_bf16_ptr, ws_ptr, int(ws_bytes), stream_ptr)


def grouped_scaled_act_bwd(dy_ptr, x_ptr, probs_ptr, split_sizes, w_in, act_kind, act_params: ActParams,
                           recipe: Recipe, dx_bf16_ptr, dx_q: QOut | None, dprobs_ptr, y_regen: QOut | None,
                           ws_ptr, ws_bytes, stream_ptr) -> int:
    return load().grouped_scaled_act_bwd(dy_ptr, x_ptr, probs_ptr, ctypes.cast(_split_array(split_sizes), _P),
                                         len(split_sizes), int(w_in), int(act_kind), ctypes.byref(act_params),
                                         ctypes.byref(recipe), dx_bf16_ptr,
                                         ctypes.byref(dx_q) if dx_q is not None else None, dprobs_ptr,
                                         ctypes.byref(y_regen) if y_regen is not None else None,
                                         ws_ptr, int(ws_bytes), stream_ptr)


def gsa_fwd_noalloc(x_ptr, probs_ptr, split_sizes, w_in, act_kind, act_params: ActParams, recipe: Recipe,
                    y_q: QOut, y_bf16_ptr, stream_ptr) -> int:
    """Forward with the library's own fixed scratch instead of a workspace (no allocation)."""
    return load().gsa_fwd_noalloc(x_ptr, probs_ptr, ctypes.cast(_split_array(split_sizes), _P), len(split_sizes),
                                  int(w_in), int(act_kind), ctypes.byref(act_params), ctypes.byref(recipe),
                                  ctypes.byref(y_q) if y_q is not None else None, y_bf16_ptr, stream_ptr)


def gsa_fwd_noalloc_status(stream_ptr) -> int:
    """Error word of the last gsa_fwd_noalloc call on the current device (synchronizes the stream)."""
    return load().gsa_fwd_noalloc_status(stream_ptr)


def gsa_layout_bound(E: int, M: int, width: int, recipe_kind: int) -> LayoutInfo:
    """Sizes of the quantized copies for any split of M rows over E experts."""
    info = LayoutInfo()
    st = load().gsa_layout_bound(int(E), int(M), int(width), int(recipe_kind), ctypes.byref(info))
    if st != 0:
        raise GsaError(st, "gsa_layout_bound")
    return info


def gsa_workspace_size_graph_safe(E: int, M: int, w_in: int, act_kind: int, recipe_kind: int) -> int:
    return int(load().gsa_workspace_size_graph_safe(int(E), int(M), int(w_in), int(act_kind), int(recipe_kind)))


def grouped_scaled_act_fwd_graph_safe(x_ptr, probs_ptr, split_dev_ptr, E, M, w_in, act_kind, act_params: ActParams,
                                      recipe: Recipe, y_q: QOut, y_bf16_ptr, pad_ptr, ws_ptr, ws_bytes,
                                      stream_ptr) -> int:
    return load().grouped_scaled_act_fwd_graph_safe(x_ptr, probs_ptr, split_dev_ptr, int(E), int(M), int(w_in),
                                                    int(act_kind), ctypes.byref(act_params), ctypes.byref(recipe),
                                                    ctypes.byref(y_q) if y_q is not None else None, y_bf16_ptr,
                                                    pad_ptr, ws_ptr, int(ws_bytes), stream_ptr)


def grouped_scaled_act_bwd_graph_safe(dy_ptr, x_ptr, probs_ptr, split_dev_ptr, E, M, w_in, act_kind,
                                      act_params: ActParams, recipe: Recipe, dx_bf16_ptr, dx_q: QOut | None,
                                      dprobs_ptr, y_regen: QOut | None, pad_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    return load().grouped_scaled_act_bwd_graph_safe(dy_ptr, x_ptr, probs_ptr, split_dev_ptr, int(E), int(M),
                                                    int(w_in), int(act_kind), ctypes.byref(act_params),
                                                    ctypes.byref(recipe), dx_bf16_ptr,
                                                    ctypes.byref(dx_q) if dx_q is not None else None, dprobs_ptr,
                                                    ctypes.byref(y_regen) if y_regen is not None else None,
                                                    pad_ptr, ws_ptr, int(ws_bytes), stream_ptr)


def gsa_selftest_wait_timeout(ws_ptr, which: int, limit_ms: int, stream_ptr) -> int:
    """Run a bounded wait that nothing signals (0: counter, 1: mbarrier) with a short limit."""
    return load().gsa_selftest_wait_timeout(ws_ptr, int(which), int(limit_ms), stream_ptr)


def gsa_workspace_status(ws_ptr, stream_ptr) -> int:
    return load().gsa_workspace_status(ws_ptr, stream_ptr)


def gsa_last_launch_count() -> int:
    return int(load().gsa_last_launch_count())


# ------------------------------------------------------- torch conveniences

def act_params(act: str | int, s: float = 4.0, limit: float = 7.0, alpha: float = 1.702,
               glu_linear_offset: float = 1.0) -> ActParams:
    return ActParams(s, limit, alpha, glu_linear_offset)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def alloc_qtensor(split_sizes, width: int, recipe_kind: int, rowwise: bool, columnwise: bool, device,
                  amax_experts: int | None = None, scale_layout: int = SCALES_COMPACT) -> dict:
    """Allocate the quantized copies of a [M, width] grouped tensor (uint8).
    Tiled scales are zero-filled (the library does not write their padding)."""
    import torch
    info = gsa_layout_ex(split_sizes, width, Recipe(recipe_kind, 0, 0, scale_layout))[0]
    E = len(split_sizes)
    sbuf = torch.zeros if scale_layout == SCALES_TILED else torch.empty
    out = {}
    if rowwise:
        out["row_data"] = torch.empty(max(1, info.row_data_bytes), dtype=torch.uint8, device=device)
        out["row_scale"] = sbuf(max(1, info.row_scale_bytes), dtype=torch.uint8, device=device)
    if columnwise:
        out["col_data"] = torch.empty(max(1, info.col_data_bytes), dtype=torch.uint8, device=device)
        out["col_scale"] = sbuf(max(1, info.col_scale_bytes), dtype=torch.uint8, device=device)
    if recipe_kind == NVFP4:
        if rowwise:
            out["amax_row"] = torch.empty(E, dtype=torch.float32, device=device)
        if columnwise:
            out["amax_col"] = torch.empty(E, dtype=torch.float32, device=device)
    out["_info"] = info
    return out


def qout_of(q: dict | None) -> QOut | None:
    if q is None:
        return None
    return QOut(*[(q[k].data_ptr() if k in q else None) for k in
                  ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col")])


class Workspace:
    """A device workspace sized by gsa_workspace_size (256-byte aligned)."""

    def __init__(self, split_sizes, w_in, act_kind, recipe_kind, device):
        import torch
        self.nbytes = gsa_workspace_size(split_sizes, w_in, act_kind, recipe_kind)
        if self.nbytes == 0:
            raise GsaError(1, "gsa_workspace_size")
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        self.ptr = (base + 255) // 256 * 256

    def status(self, stream=None) -> int:
        return gsa_workspace_status(ctypes.c_void_p(self.ptr), _stream_ptr(stream))


def _check(st, what):
    if st != 0:
        raise GsaError(st, what)


def fwd(x, probs, split_sizes, act: str, recipe_kind: int, rht: bool = False, rht_mask: int = 0,
        rowwise: bool = True, columnwise: bool = True, want_y: bool = False, params: ActParams | None = None,
        ws: Workspace | None = None, out: dict | None = None, stream=None, scale_layout: int = SCALES_COMPACT) -> dict:
    """Forward on device tensors x [M, W_in] bf16, probs [M] f32 (or None: p = 1).  Returns a dict
    with the quantized copies (row_data, row_scale, col_data, col_scale,
    amax_row, amax_col) and, with want_y, the BF16 Y."""
    import torch
    a = ACT[act] if isinstance(act, str) else int(act)
    w_in = x.shape[1]
    w = w_in // 2 if a in GLU_ACTS else w_in
    params = params or act_params(a)
    ws = ws or Workspace(split_sizes, w_in, a, recipe_kind, x.device)
    if out is None:
        out = alloc_qtensor(split_sizes, w, recipe_kind, rowwise, columnwise, x.device, scale_layout=scale_layout)
        if want_y:
            out["y"] = torch.empty((x.shape[0], w), dtype=torch.bfloat16, device=x.device)
    rec = Recipe(recipe_kind, int(bool(rht)), int(rht_mask) & 0xFFFF, scale_layout)
    st = grouped_scaled_act_fwd(_ptr(x), _ptr(probs), split_sizes, w_in, a, params, rec, qout_of(out),
                                _ptr(out.get("y")), ctypes.c_void_p(ws.ptr), ws.nbytes, _stream_ptr(stream))
    _check(st, "grouped_scaled_act_fwd")
    return out


def bwd(dy, x, probs, split_sizes, act: str, recipe_kind: int, rht: bool = False, rht_mask: int = 0,
        want_dx: bool = True, rowwise: bool = True, columnwise: bool = True, want_dprobs: bool = True,
        regen: bool = False, params: ActParams | None = None, ws: Workspace | None = None,
        out: dict | None = None, stream=None, scale_layout: int = SCALES_COMPACT) -> dict:
    """Backward on device tensors.  Returns dx (bf16 [M, W_in]), dprobs (f32 [M]),
    the quantized copies of dX and, with regen, the regenerated columnwise copy
    of Y under keys prefixed 'y_'."""
    import torch
    a = ACT[act] if isinstance(act, str) else int(act)
    w_in = x.shape[1]
    w = w_in // 2 if a in GLU_ACTS else w_in
    params = params or act_params(a)
    ws = ws or Workspace(split_sizes, w_in, a, recipe_kind, x.device)
    if out is None:
        out = {}
        if rowwise or columnwise:
            out.update(alloc_qtensor(split_sizes, w_in, recipe_kind, rowwise, columnwise, x.device,
                                     scale_layout=scale_layout))
        if want_dx:
            out["dx"] = torch.empty((x.shape[0], w_in), dtype=torch.bfloat16, device=x.device)
        if want_dprobs:
            out["dprobs"] = torch.empty(x.shape[0], dtype=torch.float32, device=x.device)
        if regen:
            yq = alloc_qtensor(split_sizes, w, recipe_kind, False, True, x.device, scale_layout=scale_layout)
            for k, v in yq.items():
                out["y_" + k] = v
    dxq = qout_of({k: v for k, v in out.items() if not k.startswith("y_") and k not in ("dx", "dprobs", "_info")}) \
        if (rowwise or columnwise) else None
    yq = qout_of({k[2:]: v for k, v in out.items() if k.startswith("y_") and k != "y__info"}) if regen else None
    rec = Recipe(recipe_kind, int(bool(rht)), int(rht_mask) & 0xFFFF, scale_layout)
    st = grouped_scaled_act_bwd(_ptr(dy), _ptr(x), _ptr(probs), split_sizes, w_in, a, params, rec,
                                _ptr(out.get("dx")), dxq, _ptr(out.get("dprobs")), yq,
                                ctypes.c_void_p(ws.ptr), ws.nbytes, _stream_ptr(stream))
    _check(st, "grouped_scaled_act_bwd")
    return out


# ------------------------------------------------- graph-safe conveniences

def alloc_qtensor_bound(E: int, M: int, width: int, recipe_kind: int, rowwise: bool, columnwise: bool,
                        device, scale_layout: int = SCALES_COMPACT) -> dict:
    """Quantized copies sized for any split of M rows over E experts."""
    import torch
    info = gsa_layout_bound_ex(E, M, width, Recipe(recipe_kind, 0, 0, scale_layout))
    sbuf = torch.zeros if scale_layout == SCALES_TILED else torch.empty
    out = {}
    if rowwise:
        out["row_data"] = torch.empty(max(1, info.row_data_bytes), dtype=torch.uint8, device=device)
        out["row_scale"] = sbuf(max(1, info.row_scale_bytes), dtype=torch.uint8, device=device)
    if columnwise:
        out["col_data"] = torch.empty(max(1, info.col_data_bytes), dtype=torch.uint8, device=device)
        out["col_scale"] = sbuf(max(1, info.col_scale_bytes), dtype=torch.uint8, device=device)
    if recipe_kind == NVFP4:
        if rowwise:
            out["amax_row"] = torch.empty(E, dtype=torch.float32, device=device)
        if columnwise:
            out["amax_col"] = torch.empty(E, dtype=torch.float32, device=device)
    out["_info"] = info
    return out


class GraphSafeWorkspace(Workspace):
    """Workspace of the graph-safe calls, sized by (E, M) alone."""

    def __init__(self, E, M, w_in, act_kind, recipe_kind, device):
        import torch
        self.nbytes = gsa_workspace_size_graph_safe(E, M, w_in, act_kind, recipe_kind)
        if self.nbytes == 0:
            raise GsaError(1, "gsa_workspace_size_graph_safe")
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        self.ptr = (self.buf.data_ptr() + 255) // 256 * 256


def fwd_graph_safe(x, probs, split_dev, act: str, recipe_kind: int, rht: bool = False, rht_mask: int = 0,
                   rowwise: bool = True, columnwise: bool = True, want_y: bool = False,
                   params: ActParams | None = None, ws: Workspace | None = None, out: dict | None = None,
                   stream=None, scale_layout: int = SCALES_COMPACT) -> dict:
    """Forward with split_dev ([E] int64 on the device).  Outputs sized by
    gsa_layout_bound; out["pad"] ([E+1] int64) receives the padded row
    offsets of the columnwise blocks.  Enqueues work only: capturable."""
    import torch
    a = ACT[act] if isinstance(act, str) else int(act)
    E, M, w_in = split_dev.numel(), x.shape[0], x.shape[1]
    w = w_in // 2 if a in GLU_ACTS else w_in
    params = params or act_params(a)
    ws = ws or GraphSafeWorkspace(E, M, w_in, a, recipe_kind, x.device)
    if out is None:
        out = alloc_qtensor_bound(E, M, w, recipe_kind, rowwise, columnwise, x.device, scale_layout)
        if want_y:
            out["y"] = torch.empty((M, w), dtype=torch.bfloat16, device=x.device)
        out["pad"] = torch.empty(E + 1, dtype=torch.int64, device=x.device)
    rec = Recipe(recipe_kind, int(bool(rht)), int(rht_mask) & 0xFFFF, scale_layout)
    st = grouped_scaled_act_fwd_graph_safe(_ptr(x), _ptr(probs), _ptr(split_dev), E, M, w_in, a, params, rec,
                                           qout_of(out), _ptr(out.get("y")), _ptr(out.get("pad")),
                                           ctypes.c_void_p(ws.ptr), ws.nbytes, _stream_ptr(stream))
    _check(st, "grouped_scaled_act_fwd_graph_safe")
    return out


def bwd_graph_safe(dy, x, probs, split_dev, act: str, recipe_kind: int, rht: bool = False, rht_mask: int = 0,
                   want_dx: bool = True, rowwise: bool = True, columnwise: bool = True, want_dprobs: bool = True,
                   regen: bool = False, params: ActParams | None = None, ws: Workspace | None = None,
                   out: dict | None = None, stream=None, scale_layout: int = SCALES_COMPACT) -> dict:
    """Backward with split_dev on the device; keys as for bwd, plus "pad"."""
    import torch
    a = ACT[act] if isinstance(act, str) else int(act)
    E, M, w_in = split_dev.numel(), x.shape[0], x.shape[1]
    w = w_in // 2 if a in GLU_ACTS else w_in
    params = params or act_params(a)
    ws = ws or GraphSafeWorkspace(E, M, w_in, a, recipe_kind, x.device)
    if out is None:
        out = {}
        if rowwise or columnwise:
            out.update(alloc_qtensor_bound(E, M, w_in, recipe_kind, rowwise, columnwise, x.device, scale_layout))
        if want_dx:
            out["dx"] = torch.empty((M, w_in), dtype=torch.bfloat16, device=x.device)
        if want_dprobs:
            out["dprobs"] = torch.empty(M, dtype=torch.float32, device=x.device)
        if regen:
            for k, v in alloc_qtensor_bound(E, M, w, recipe_kind, False, True, x.device, scale_layout).items():
                out["y_" + k] = v
        out["pad"] = torch.empty(E + 1, dtype=torch.int64, device=x.device)
    skip = ("dx", "dprobs", "_info", "pad")
    dxq = qout_of({k: v for k, v in out.items() if not k.startswith("y_") and k not in skip}) \
        if (rowwise or columnwise) else None
    yq = qout_of({k[2:]: v for k, v in out.items() if k.startswith("y_") and k != "y__info"}) if regen else None
    rec = Recipe(recipe_kind, int(bool(rht)), int(rht_mask) & 0xFFFF, scale_layout)
    st = grouped_scaled_act_bwd_graph_safe(_ptr(dy), _ptr(x), _ptr(probs), _ptr(split_dev), E, M, w_in, a, params,
                                           rec, _ptr(out.get("dx")), dxq, _ptr(out.get("dprobs")), yq,
                                           _ptr(out.get("pad")), ctypes.c_void_p(ws.ptr), ws.nbytes,
                                           _stream_ptr(stream))
    _check(st, "grouped_scaled_act_bwd_graph_safe")
    return out
