"""Block scales in the tiled layout of block-scaled GEMM operands.

The grouped-linear fusion page hands the quantized activation output to the
grouped GEMM as a pre-built grouped tensor ("Activation + GroupedLinear Fusion
for MOE", Greptile Summary), and the inner-autocast page's scales go to
cuBLASLt ("Preserve FP8 recompute state for inner autocast", How much it
costs).  With GSA_SCALES_TILED the library writes the block scales in
cuBLASLt's 1D block-scaling factor layout.  Checked here:
  * every call form (forward, backward with and without the regenerated copy,
    graph-safe, allocation-free) writes the same codes and amax as with compact
    scales, and tiled scales equal to the compact ones rearranged
    (oracle.tiled_scales);
  * SReLU against the oracle's own tiled quantization, bit for bit;
  * the layout itself, independently of the oracle: cuBLASLt's block-scaled
    GEMM (torch._scaled_mm) on the library's codes and tiled scales gives the
    product of the dequantized operands, for the rowwise copy (the FC2
    forward operand) and the columnwise copy (the FC2 wgrad operand), MXFP8
    and NVFP4 with the RHT.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import ACT_ID, GLU_NAMES, dev_bf16, dev_f32, params_tuple
from nvfp4_quantization_grouped_gb300 import gsa, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

T = gsa.SCALES_TILED
MASK = 0x4C2B


def _np(t):
    return t.view(torch.uint8).cpu().numpy() if t.dtype != torch.float32 else t.cpu().numpy()


def _tiled_from_compact(rs, cs, split, width, recipe):
    """The tiled scales a call must write, from its compact scales."""
    B = oracle.block_size(recipe)
    offs = np.concatenate([[0], np.cumsum(split)]).astype(np.int64)
    rows = None
    if rs is not None:
        r2 = rs[:offs[-1] * (width // B)].reshape(-1, width // B)
        rows = np.concatenate([oracle.tiled_scales(r2[offs[e]:offs[e + 1]]) for e in range(len(split))] +
                              [np.zeros(0, np.uint8)])
    cols = None
    if cs is not None:
        parts, pos = [], 0
        for m in split:
            if m == 0:
                continue
            n = oracle.padded_rows(int(m), recipe) // B
            parts.append(oracle.tiled_scales(cs[pos:pos + width * n].reshape(width, n)))
            pos += width * n
        cols = np.concatenate(parts + [np.zeros(0, np.uint8)])
    return rows, cols


def _same_as_compact(comp, tiled, split, width, recipe, prefix="", what=""):
    for k in ("row_data", "col_data", "amax_row", "amax_col"):
        if prefix + k in comp:
            a, b = _np(comp[prefix + k]), _np(tiled[prefix + k])
            assert np.array_equal(a, b[:a.size]), f"{what} {k}"
    rs = _np(comp[prefix + "row_scale"]) if prefix + "row_scale" in comp else None
    cs = _np(comp[prefix + "col_scale"]) if prefix + "col_scale" in comp else None
    want_r, want_c = _tiled_from_compact(rs, cs, split, width, recipe)
    if want_r is not None:
        got = _np(tiled[prefix + "row_scale"])
        assert np.array_equal(got[:want_r.size], want_r), f"{what} tiled row_scale"
    if want_c is not None:
        got = _np(tiled[prefix + "col_scale"])
        assert np.array_equal(got[:want_c.size], want_c), f"{what} tiled col_scale"


CASES = [([0, 1, 15, 17, 0, 31, 33, 128, 129, 255], 192), ([300, 77], 1024), ([0, 64], 64)]


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
@pytest.mark.parametrize("act", ["srelu", "tanh_srelu", "swiglu"])
def test_tiled_scales_every_call_form(recipe, act):
    rng = np.random.default_rng(500 + 10 * recipe + ACT_ID[act])
    glu = act in GLU_NAMES
    prm = gsa.ActParams(*params_tuple(act))
    for split, width in CASES:
        split, x, p, dy = inputs.random_problem(rng, split, width, glu, x_sigma=2.0)
        split = [int(v) for v in split]
        rht = recipe == oracle.NVFP4 and width != 192
        X, Pp, DY = dev_bf16(x), dev_f32(p), dev_bf16(dy)
        w_in = X.shape[1]
        # forward, host split
        fc = gsa.fwd(X, Pp, split, act, recipe, rht, MASK, True, True, True, prm)
        ft = gsa.fwd(X, Pp, split, act, recipe, rht, MASK, True, True, True, prm, scale_layout=T)
        torch.cuda.synchronize()
        _same_as_compact(fc, ft, split, width, recipe, what=f"{act} fwd w{width}")
        # backward, host split, with and without the regenerated copy (two kernel variants)
        for regen in (True, False):
            bc = gsa.bwd(DY, X, Pp, split, act, recipe, rht, MASK, True, True, True, True, regen, prm)
            bt = gsa.bwd(DY, X, Pp, split, act, recipe, rht, MASK, True, True, True, True, regen, prm,
                         scale_layout=T)
            torch.cuda.synchronize()
            _same_as_compact(bc, bt, split, w_in, recipe, what=f"{act} bwd dX regen={regen} w{width}")
            if regen:
                _same_as_compact(bc, bt, split, width, recipe, prefix="y_", what=f"{act} bwd regen Y w{width}")
        # graph-safe calls: outputs sized by the bound, the same bytes in front
        sd = torch.tensor(split, dtype=torch.int64, device="cuda")
        gf = gsa.fwd_graph_safe(X, Pp, sd, act, recipe, rht, MASK, True, True, True, prm, scale_layout=T)
        gb = gsa.bwd_graph_safe(DY, X, Pp, sd, act, recipe, rht, MASK, True, True, True, True, True, prm,
                                scale_layout=T)
        torch.cuda.synchronize()
        _same_as_compact(fc, gf, split, width, recipe, what=f"{act} graph-safe fwd w{width}")
        bc = gsa.bwd(DY, X, Pp, split, act, recipe, rht, MASK, True, True, True, True, True, prm)
        torch.cuda.synchronize()
        _same_as_compact(bc, gb, split, w_in, recipe, what=f"{act} graph-safe bwd w{width}")
        _same_as_compact(bc, gb, split, width, recipe, prefix="y_", what=f"{act} graph-safe regen w{width}")
        # allocation-free forward
        out = gsa.alloc_qtensor(split, width, recipe, True, True, X.device, scale_layout=T)
        st = gsa.gsa_fwd_noalloc(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(Pp.data_ptr()), split, w_in,
                                 gsa.ACT[act], prm, gsa.Recipe(recipe, int(rht), MASK, T), gsa.qout_of(out), None,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        assert gsa.gsa_fwd_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        _same_as_compact(fc, out, split, width, recipe, what=f"{act} allocation-free fwd w{width}")


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
def test_tiled_scales_srelu_against_oracle(recipe):
    rng = np.random.default_rng(77 + recipe)
    split, x, p, dy = inputs.random_problem(rng, [0, 200, 33, 129], 256, False)
    rht = recipe == oracle.NVFP4
    g = gsa.fwd(dev_bf16(x), dev_f32(p), list(split), "srelu", recipe, rht, MASK, True, True, False,
                gsa.ActParams(*params_tuple("srelu")), scale_layout=T)
    torch.cuda.synchronize()
    y = oracle.act_fwd_rows(x, p, ACT_ID["srelu"], params_tuple("srelu"))
    ref = oracle.quantize_grouped(y, split, recipe, rht, MASK, True, True, oracle.SCALES_TILED)
    for k in ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col"):
        if k in ref:
            a = np.asarray(ref[k]).reshape(-1).view(np.uint8)
            b = _np(g[k]).reshape(-1).view(np.uint8)
            assert np.array_equal(a, b[:a.size]), k


# ------------------------------------------ the layout consumed by cuBLASLt

def _decode(codes, scales, recipe, K):
    """[R, K] float64 values of rowwise-laid-out codes with compact [R, K / B] scales
    (no tensor scale: the GEMM multiplies codes by block scales only)."""
    B = oracle.block_size(recipe)
    R = scales.shape[0]
    if recipe == oracle.MXFP8:
        v = oracle.e4m3_decode(codes.reshape(R, K)).astype(np.float64)
        s = np.ldexp(1.0, scales.astype(np.int64) - 127)
    else:
        c = codes.reshape(R, K // 2)
        v = np.empty((R, K))
        v[:, 0::2] = oracle.e2m1_decode(c & 15)
        v[:, 1::2] = oracle.e2m1_decode(c >> 4)
        s = oracle.e4m3_decode(scales).astype(np.float64)
    return v * np.repeat(s, B, axis=1)


def _scaled_mm(a_codes, a_scales, b_codes, b_scales, recipe):
    """cuBLASLt block-scaled GEMM A B^T of two rowwise-laid-out operands with tiled scales."""
    if recipe == oracle.MXFP8:
        A, Bm = a_codes.view(torch.float8_e4m3fn), b_codes.view(torch.float8_e4m3fn)
        sa, sb = a_scales.view(torch.float8_e8m0fnu), b_scales.view(torch.float8_e8m0fnu)
    else:
        A, Bm = a_codes.view(torch.float4_e2m1fn_x2), b_codes.view(torch.float4_e2m1fn_x2)
        sa, sb = a_scales.view(torch.float8_e4m3fn), b_scales.view(torch.float8_e4m3fn)
    return torch._scaled_mm(A, Bm.t(), sa, sb, out_dtype=torch.float32).double().cpu().numpy()


def _close(got, a, b, what):
    """got = A B^T from the GEMM against float64, within FP32 accumulation of the
    absolute terms (a misplaced scale gives errors of the size of the result)."""
    ref = a @ b.T
    bound = 1e-5 * (np.abs(a) @ np.abs(b).T) + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outputs off, first {np.argwhere(bad)[:3].tolist()}"


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
def test_tiled_scales_feed_cublaslt_block_scaled_gemm(recipe):
    rng = np.random.default_rng(900 + recipe)
    split = [256, 128, 384]
    W, N = 256, 128
    rht = recipe == oracle.NVFP4
    B = oracle.block_size(recipe)
    _, x, p, _ = inputs.random_problem(rng, split, W, False, x_sigma=2.0)
    X, Pp = dev_bf16(x), dev_f32(p)
    prm = gsa.ActParams(*params_tuple("srelu"))
    yc = gsa.fwd(X, Pp, split, "srelu", recipe, rht, MASK, True, True, False, prm)
    yt = gsa.fwd(X, Pp, split, "srelu", recipe, rht, MASK, True, True, False, prm, scale_layout=T)
    # FC2 weight [N, W] (rowwise operand) and an output gradient per expert [M_e, N]
    # (columnwise operand of the wgrad), quantized by the library: identity, p = 1
    wt = dev_bf16(inputs.normal_bf16(rng, (N, W)))
    wc = gsa.fwd(wt, None, [N], "identity", recipe, False, 0, True, False, False)
    wtl = gsa.fwd(wt, None, [N], "identity", recipe, False, 0, True, False, False, scale_layout=T)
    torch.cuda.synchronize()
    rq = 1 if recipe == oracle.MXFP8 else 2      # elements per code byte
    _, _, _, roff = gsa.gsa_layout_ex(split, W, gsa.Recipe(recipe, 0, 0, T))
    _, cdoff, csoff_t, _ = gsa.gsa_layout_ex(split, W, gsa.Recipe(recipe, 0, 0, T))
    _, _, csoff_c = gsa.gsa_layout(split, W, recipe)
    offs = np.concatenate([[0], np.cumsum(split)])
    w_vals = _decode(_np(wc["row_data"]), _np(wc["row_scale"]).reshape(N, W // B), recipe, W)
    rows_c = _np(yc["row_data"]).reshape(-1, W // rq)
    rscale_c = _np(yc["row_scale"]).reshape(-1, W // B)
    for e, m in enumerate(split):
        lo, hi = int(offs[e]), int(offs[e + 1])
        # FC2 forward: Y_e W^T from the rowwise copy
        got = _scaled_mm(yt["row_data"].view(-1, W // rq)[lo:hi], yt["row_scale"][roff[e]:roff[e + 1]],
                         wtl["row_data"].view(N, W // rq), wtl["row_scale"], recipe)
        _close(got, _decode(rows_c[lo:hi], rscale_c[lo:hi], recipe, W), w_vals, f"rowwise operand, expert {e}")
        # FC2 wgrad: Y_e^T G_e from the two columnwise copies (both with the same RHT)
        g = dev_bf16(inputs.normal_bf16(rng, (m, N)))
        gc = gsa.fwd(g, None, [m], "identity", recipe, rht, MASK, False, True, False)
        gt = gsa.fwd(g, None, [m], "identity", recipe, rht, MASK, False, True, False, scale_layout=T)
        torch.cuda.synchronize()
        a_codes = yt["col_data"][cdoff[e]:cdoff[e + 1]].view(W, m // rq)
        got = _scaled_mm(a_codes, yt["col_scale"][csoff_t[e]:csoff_t[e + 1]],
                         gt["col_data"].view(N, m // rq), gt["col_scale"], recipe)
        a_vals = _decode(_np(yc["col_data"])[cdoff[e]:cdoff[e + 1]],
                         _np(yc["col_scale"])[csoff_c[e]:csoff_c[e + 1]].reshape(W, m // B), recipe, m)
        g_vals = _decode(_np(gc["col_data"]), _np(gc["col_scale"]).reshape(N, m // B), recipe, m)
        _close(got, a_vals, g_vals, f"columnwise operand, expert {e}")
