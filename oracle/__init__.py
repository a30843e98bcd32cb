"""CPU oracle for the grouped scaled activation + block-scaled quantization path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline / reference legs of ``bench.py``.  The product path
never imports it, and it never imports the product path; the two share only
the seeded input generator.

The arithmetic lives in ``gsa_oracle.c`` (scalar binary32, no FMA
contraction).  This module compiles and loads it and composes its steps in
the order the method takes them, expert by expert:

  forward  : Y = bf16(p * act(X)); rowwise quantization of Y; columnwise
             quantization of each expert's zero-padded transpose (NVFP4:
             through the 16-point random Hadamard transform).
  backward : dX = bf16(dY * p * act'(X)); dprobs = sum_j dY * act(X);
             dX quantized as above; optionally Y's columnwise copy again.

Sources: "Activation + GroupedLinear Fusion for MOE" (Greptile Summary and
sequence diagram: one pass of per-row scale x activation x grouped quantize,
backward returning quantized dX, dense dX and grad_scales); "Enable fused
activation recompute for ScaledTanhSReLU" (Description: recompute
regenerates FC2's input from the saved FC1 output; MXFP8 and NVFP4 recipes).

Parity unpinned (conventions): GLU half order, clamped-SwiGLU constants,
dprobs summation order, per-expert NVFP4 tensor scale, RHT signs/order.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gsa_oracle.c")
_LIB = os.path.join(_HERE, "_gsa_oracle.so")
_lock = threading.Lock()
_lib = None

ACT_SRELU, ACT_TANH_SRELU, ACT_SWIGLU, ACT_CLAMPED_SWIGLU = 0, 1, 2, 3
ACT_GELU, ACT_SIGMOID, ACT_IDENTITY = 4, 5, 6   # further unary activations (reading R16)
MXFP8, NVFP4 = 0, 1

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            sig = {
                "oracle_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "oracle_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
                "oracle_e4m3_decode": (ctypes.c_float, [ctypes.c_uint8]),
                "oracle_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
                "oracle_e2m1_decode": (ctypes.c_float, [ctypes.c_uint8]),
                "oracle_mx_scale_exp": (ctypes.c_int, [ctypes.c_float]),
                "oracle_mxfp8_block": (None, [_P, ctypes.c_int, _P, _P]),
                "oracle_nvfp4_tensor_scale": (ctypes.c_float, [ctypes.c_float]),
                "oracle_nvfp4_block": (None, [_P, ctypes.c_int, ctypes.c_float, _P, _P]),
                "oracle_rht16": (None, [_P, ctypes.c_uint16, _P]),
                "oracle_act_fwd_rows": (None, [_P, _P, _I64, _I64, ctypes.c_int, _P, _P]),
                "oracle_act_fwd_rows_f32": (None, [_P, _P, _I64, _I64, ctypes.c_int, _P, _P]),
                "oracle_act_bwd_rows": (None, [_P, _P, _P, _I64, _I64, ctypes.c_int, _P, _P, _P]),
                "oracle_dprobs_sum": (ctypes.c_float, [_P, _I64]),
                "oracle_mxfp8_rows": (None, [_P, _I64, _I64, _P, _P]),
                "oracle_nvfp4_rows": (None, [_P, _I64, _I64, ctypes.c_float, _P, _P]),
                "oracle_amax_bf16": (ctypes.c_float, [_P, _I64]),
                "oracle_mxfp8_cols": (None, [_P, _I64, _I64, _P, _P]),
                "oracle_amax_cols": (ctypes.c_float, [_P, _I64, _I64, ctypes.c_int, ctypes.c_uint16]),
                "oracle_nvfp4_cols": (None, [_P, _I64, _I64, ctypes.c_int, ctypes.c_uint16,
                                             ctypes.c_float, _P, _P]),
                "oracle_e4m3_encode_n": (None, [_P, _I64, _P]),
                "oracle_e2m1_encode_n": (None, [_P, _I64, _P]),
                "oracle_f32_to_bf16_n": (None, [_P, _I64, _P]),
                "oracle_act_grad_n": (None, [ctypes.c_int, _P, _P, _I64, _P, _P, _P, _P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _params(act_params) -> np.ndarray:
    return np.asarray(act_params, dtype=np.float32).reshape(4)


# ------------------------------------------------------------ primitives

def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_n(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_n(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_e2m1_encode_n(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e4m3_decode(int(c)) for c in np.asarray(codes).reshape(-1)],
                    dtype=np.float32).reshape(np.shape(codes))


def e2m1_decode(codes) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e2m1_decode(int(c)) for c in np.asarray(codes).reshape(-1)],
                    dtype=np.float32).reshape(np.shape(codes))


def mx_scale_exp(amax: float) -> int:
    return lib().oracle_mx_scale_exp(float(amax))


def mxfp8_block(v) -> tuple[np.ndarray, int]:
    v = np.ascontiguousarray(v, dtype=np.float32)
    codes = np.empty(v.size, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.uint8)
    lib().oracle_mxfp8_block(_ptr(v), v.size, _ptr(codes), _ptr(sc))
    return codes, int(sc[0])


def nvfp4_tensor_scale(amax: float) -> float:
    return float(np.float32(lib().oracle_nvfp4_tensor_scale(float(amax))))


def nvfp4_block(v, S_enc: float) -> tuple[np.ndarray, int]:
    v = np.ascontiguousarray(v, dtype=np.float32)
    codes = np.empty(v.size, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.uint8)
    lib().oracle_nvfp4_block(_ptr(v), v.size, float(S_enc), _ptr(codes), _ptr(sc))
    return codes, int(sc[0])


def rht16(v, mask: int) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32).reshape(16)
    w = np.empty(16, dtype=np.float32)
    lib().oracle_rht16(_ptr(v), int(mask) & 0xFFFF, _ptr(w))
    return w


def act_grad(act: int, a, b=None, act_params=(0, 0, 0, 0)):
    a = np.ascontiguousarray(a, dtype=np.float32)
    bb = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
    val = np.empty_like(a)
    da = np.empty_like(a)
    db = np.empty_like(a)
    prm = _params(act_params)
    lib().oracle_act_grad_n(act, _ptr(a), _ptr(bb), a.size, _ptr(prm), _ptr(val), _ptr(da), _ptr(db))
    return val, da, db


def dprobs_sum(terms) -> float:
    t = np.ascontiguousarray(terms, dtype=np.float32)
    return float(np.float32(lib().oracle_dprobs_sum(_ptr(t), t.size)))


# ------------------------------------------------------- composed steps

def is_glu(act: int) -> bool:
    return act in (ACT_SWIGLU, ACT_CLAMPED_SWIGLU)


def _probs(probs, n):
    """The per-row scale p; None means p = 1 for every row."""
    if probs is None:
        return np.ones(n, dtype=np.float32)
    return np.ascontiguousarray(probs, dtype=np.float32)


def act_fwd_rows(x, probs, act, act_params):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    p = _probs(probs, x.shape[0])
    n, w_in = x.shape
    w = w_in // 2 if is_glu(act) else w_in
    y = np.empty((n, w), dtype=np.uint16)
    prm = _params(act_params)
    lib().oracle_act_fwd_rows(_ptr(x), _ptr(p), n, w_in, act, _ptr(prm), _ptr(y))
    return y


def act_fwd_rows_f32(x32, probs, act, act_params):
    """Y = bf16(p * act(X)) from FP32 X (the FC1 accumulator, not rounded to BF16)."""
    x = np.ascontiguousarray(x32, dtype=np.float32)
    p = _probs(probs, x.shape[0])
    n, w_in = x.shape
    w = w_in // 2 if is_glu(act) else w_in
    y = np.empty((n, w), dtype=np.uint16)
    prm = _params(act_params)
    lib().oracle_act_fwd_rows_f32(_ptr(x), _ptr(p), n, w_in, act, _ptr(prm), _ptr(y))
    return y


def act_bwd_rows(dy, x, probs, act, act_params, want_dx=True, want_dprobs=True):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    dy = np.ascontiguousarray(dy, dtype=np.uint16)
    p = _probs(probs, x.shape[0])
    n, w_in = x.shape
    dx = np.empty((n, w_in), dtype=np.uint16) if want_dx else None
    dpr = np.empty(n, dtype=np.float32) if want_dprobs else None
    prm = _params(act_params)
    lib().oracle_act_bwd_rows(_ptr(dy), _ptr(x), _ptr(p), n, w_in, act, _ptr(prm), _ptr(dx), _ptr(dpr))
    return dx, dpr


def block_size(recipe: int) -> int:
    return 32 if recipe == MXFP8 else 16


def padded_rows(m: int, recipe: int) -> int:
    b = block_size(recipe)
    return (m + b - 1) // b * b


def quant_rows(v, recipe: int, S_enc: float = 1.0):
    v = np.ascontiguousarray(v, dtype=np.uint16)
    n, w = v.shape
    if recipe == MXFP8:
        data = np.empty((n, w), dtype=np.uint8)
        scale = np.empty((n, (w + 31) // 32), dtype=np.uint8)
        lib().oracle_mxfp8_rows(_ptr(v), n, w, _ptr(data), _ptr(scale))
    else:
        data = np.empty((n, w // 2), dtype=np.uint8)
        scale = np.empty((n, w // 16), dtype=np.uint8)
        lib().oracle_nvfp4_rows(_ptr(v), n, w, float(S_enc), _ptr(data), _ptr(scale))
    return data, scale


def amax_rows(v) -> float:
    v = np.ascontiguousarray(v, dtype=np.uint16)
    return float(np.float32(lib().oracle_amax_bf16(_ptr(v), v.size)))


def amax_cols(v, rht: bool, mask: int) -> float:
    v = np.ascontiguousarray(v, dtype=np.uint16)
    me, w = v.shape
    return float(np.float32(lib().oracle_amax_cols(_ptr(v), me, w, int(bool(rht)), int(mask) & 0xFFFF)))


def quant_cols(v, recipe: int, rht: bool = False, mask: int = 0, S_enc: float = 1.0):
    """Columnwise copy of one expert's values v [Me, W]: (data, scale) with
    data [W, Mp] (MXFP8) or [W, Mp/2] (NVFP4), scale [W, Mp/B]."""
    v = np.ascontiguousarray(v, dtype=np.uint16)
    me, w = v.shape
    mp = padded_rows(me, recipe)
    b = block_size(recipe)
    scale = np.empty((w, mp // b), dtype=np.uint8)
    if recipe == MXFP8:
        data = np.empty((w, mp), dtype=np.uint8)
        lib().oracle_mxfp8_cols(_ptr(v), me, w, _ptr(data), _ptr(scale))
    else:
        data = np.empty((w, mp // 2), dtype=np.uint8)
        lib().oracle_nvfp4_cols(_ptr(v), me, w, int(bool(rht)), int(mask) & 0xFFFF, float(S_enc),
                                _ptr(data), _ptr(scale))
    return data, scale


def dequant_cols(data, scale, recipe: int, S_enc: float = 1.0) -> np.ndarray:
    """Values of one expert's columnwise copy, [W, Mp] float64: MXFP8
    E4M3(code) * 2^(scale - 127); NVFP4 E2M1(code) * E4M3(scale) / S_enc, element
    2k in the low nibble (for the RHT copy these are the transformed values)."""
    b = block_size(recipe)
    sc = np.asarray(scale)
    w = sc.shape[0]
    if recipe == MXFP8:
        vals = e4m3_decode(np.asarray(data)).astype(np.float64)
        mult = np.ldexp(1.0, sc.astype(np.int64) - 127)
    else:
        d = np.asarray(data, dtype=np.uint8)
        codes = np.empty((w, d.shape[1] * 2), dtype=np.uint8)
        codes[:, 0::2] = d & 0xF
        codes[:, 1::2] = d >> 4
        vals = e2m1_decode(codes).astype(np.float64)
        mult = e4m3_decode(sc).astype(np.float64) / float(S_enc)
    return vals * np.repeat(mult, b, axis=1)


def rht_cols(v, mask: int) -> np.ndarray:
    """The columnwise copy's transform applied in float64 to the columns of v
    [Mp, N] (Mp a multiple of 16): each 16-row chunk c of a column becomes
    1/4 H16 D c, an orthogonal map, so the transformed copies of two tensors
    keep their inner products over rows."""
    v = np.asarray(v, dtype=np.float64)
    d = np.array([-1.0 if (int(mask) >> i) & 1 else 1.0 for i in range(16)])
    h = np.array([[(-1.0) ** bin(i & j).count("1") for j in range(16)] for i in range(16)])
    r = 0.25 * h * d[None, :]
    mp, n = v.shape
    return np.einsum("ij,cjn->cin", r, v.reshape(mp // 16, 16, n)).reshape(mp, n)


def tiled_scales(s) -> np.ndarray:
    """One [R, C] block-scale matrix in the tiled layout of block-scaled GEMM
    operands (cuBLASLt's 1D block-scaling factor layout, the consumer of the
    quantized tensor: "Activation + GroupedLinear Fusion for MOE", Greptile
    Summary; "Preserve FP8 recompute state for inner autocast", How much it
    costs): zero-padded to whole tiles of 128 rows x 4 columns (512 bytes) in
    row-major tile order; inside a tile, entry (r, c) at byte
    16 (r mod 32) + 4 floor(r / 32) + c (reading R18).  Returned flat."""
    s = np.asarray(s, dtype=np.uint8)
    R, C = s.shape
    R2, C2 = -(-R // 128) * 128, -(-C // 4) * 4
    p = np.zeros((R2, C2), dtype=np.uint8)
    p[:R, :C] = s
    # axes (row tile, r // 32 in the tile, r % 32, column tile, c % 4) -> tile order, then r % 32, r // 32, c % 4
    t = p.reshape(R2 // 128, 4, 32, C2 // 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(-1)


SCALES_COMPACT, SCALES_TILED = 0, 1


def quantize_grouped(v, split_sizes, recipe: int, rht: bool = False, mask: int = 0,
                     want_row: bool = True, want_col: bool = True, scale_layout: int = SCALES_COMPACT) -> dict:
    """Rowwise + columnwise quantized copies of a grouped [M, W] BF16 tensor.

    Returns a dict with row_data/row_scale ([M, ...]), col_data/col_scale
    (experts concatenated, flattened) and, for NVFP4, per-expert amax_row /
    amax_col.  With SCALES_TILED each expert's scale matrices (rowwise
    [M_e, W / B], columnwise [W, Mp_e / B]) are given in the tiled layout
    (tiled_scales), the experts' blocks concatenated, both flat."""
    v = np.ascontiguousarray(v, dtype=np.uint16)
    m, w = v.shape
    offs = np.concatenate([[0], np.cumsum(split_sizes)]).astype(np.int64)
    E = len(split_sizes)
    out: dict = {}
    amax_r = np.zeros(E, dtype=np.float32)
    amax_c = np.zeros(E, dtype=np.float32)
    if want_row:
        if recipe == MXFP8:
            out["row_data"], out["row_scale"] = quant_rows(v, recipe)
        else:
            rd = np.empty((m, w // 2), dtype=np.uint8)
            rs = np.empty((m, w // 16), dtype=np.uint8)
            for e in range(E):
                ve = v[offs[e]:offs[e + 1]]
                amax_r[e] = amax_rows(ve)
                if ve.shape[0]:
                    rd[offs[e]:offs[e + 1]], rs[offs[e]:offs[e + 1]] = quant_rows(
                        ve, recipe, nvfp4_tensor_scale(amax_r[e]))
            out["row_data"], out["row_scale"] = rd, rs
            out["amax_row"] = amax_r
    if want_col:
        cd, cs = [], []
        for e in range(E):
            ve = v[offs[e]:offs[e + 1]]
            if ve.shape[0] == 0:
                continue
            if recipe == MXFP8:
                d, s = quant_cols(ve, recipe)
            else:
                amax_c[e] = amax_cols(ve, rht, mask)
                d, s = quant_cols(ve, recipe, rht, mask, nvfp4_tensor_scale(amax_c[e]))
            cd.append(d.reshape(-1))
            cs.append(s.reshape(-1))
        out["col_data"] = np.concatenate(cd) if cd else np.zeros(0, np.uint8)
        out["col_scale"] = np.concatenate(cs) if cs else np.zeros(0, np.uint8)
        if recipe == NVFP4:
            out["amax_col"] = amax_c
    if scale_layout == SCALES_TILED:
        B = block_size(recipe)
        if want_row:
            rs = out["row_scale"]
            out["row_scale"] = np.concatenate([tiled_scales(rs[offs[e]:offs[e + 1]]) for e in range(E)] +
                                              [np.zeros(0, np.uint8)])
        if want_col:
            parts, pos = [], 0
            for e in range(E):
                me = int(split_sizes[e])
                if me == 0:
                    continue
                n = padded_rows(me, recipe) // B
                parts.append(tiled_scales(out["col_scale"][pos:pos + w * n].reshape(w, n)))
                pos += w * n
            out["col_scale"] = np.concatenate(parts + [np.zeros(0, np.uint8)])
    return out


def fwd(x, probs, split_sizes, act: int, act_params, recipe: int, rht: bool = False,
        mask: int = 0, want_row: bool = True, want_col: bool = True) -> dict:
    """Forward: Y and its quantized copies (see module docstring)."""
    y = act_fwd_rows(x, probs, act, act_params)
    out = quantize_grouped(y, split_sizes, recipe, rht, mask, want_row, want_col)
    out["y"] = y
    return out


def bwd(dy, x, probs, split_sizes, act: int, act_params, recipe: int, rht: bool = False,
        mask: int = 0, want_row: bool = True, want_col: bool = True,
        want_regen: bool = False) -> dict:
    """Backward: dX (BF16), dprobs, dX's quantized copies and, on request,
    the regenerated columnwise copy of Y (keys prefixed ``y_``)."""
    dx, dpr = act_bwd_rows(dy, x, probs, act, act_params)
    out = quantize_grouped(dx, split_sizes, recipe, rht, mask, want_row, want_col)
    out["dx"] = dx
    out["dprobs"] = dpr
    if want_regen:
        y = act_fwd_rows(x, probs, act, act_params)
        yq = quantize_grouped(y, split_sizes, recipe, rht, mask, False, True)
        for k, v in yq.items():
            out["y_" + k] = v
    return out


def expert_col_offsets(split_sizes, width: int, recipe: int):
    """Per-expert offsets (elements of the flattened col_data / col_scale)."""
    b = block_size(recipe)
    d, s = [0], [0]
    for m in split_sizes:
        mp = padded_rows(int(m), recipe)
        d.append(d[-1] + width * (mp if recipe == MXFP8 else mp // 2))
        s.append(s[-1] + width * (mp // b))
    return np.array(d, dtype=np.int64), np.array(s, dtype=np.int64)
