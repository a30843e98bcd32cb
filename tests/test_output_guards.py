"""Bounds checks with guard canaries: every output buffer and the workspace
are placed between 4 KiB guard regions filled with a pattern, the calls go
through the C ABI with the interior pointers, on ragged expert splits (empty
experts, 1, 15, 17, 31, 33, 129 rows) and narrow widths, and afterwards every
guard byte must still hold the pattern.  The interiors are compared with the
same call on plain buffers, so the guarded call did its work."""
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

GUARD = 4096
PATTERN = 0xA5
SPLIT = [0, 1, 15, 17, 0, 31, 33, 129]


class Guarded:
    """nbytes of device memory between two guard regions."""

    def __init__(self, nbytes):
        self.nbytes = int(nbytes)
        self.buf = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.ptr = self.buf.data_ptr() + GUARD

    def inner(self):
        return self.buf[GUARD:GUARD + self.nbytes]

    def guards_intact(self):
        return bool(torch.all(self.buf[:GUARD] == PATTERN)) and bool(torch.all(self.buf[GUARD + self.nbytes:] == PATTERN))


def _qout(info, E, recipe, row=True, col=True):
    g = {}
    if row:
        g["row_data"], g["row_scale"] = Guarded(info.row_data_bytes), Guarded(info.row_scale_bytes)
    if col:
        g["col_data"], g["col_scale"] = Guarded(info.col_data_bytes), Guarded(info.col_scale_bytes)
    if recipe == oracle.NVFP4:
        if row:
            g["amax_row"] = Guarded(4 * E)
        if col:
            g["amax_col"] = Guarded(4 * E)
    q = gsa.QOut(*[(g[k].ptr if k in g else None) for k in
                   ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col")])
    return g, q


def _check(guarded, ref, what):
    for k, g in guarded.items():
        assert g.guards_intact(), f"{what}: guard of {k} overwritten"
        if k in ref:
            r = ref[k].reshape(-1).view(torch.uint8)
            assert torch.equal(g.inner()[:r.numel()], r), f"{what}: {k} differs from the unguarded call"


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
@pytest.mark.parametrize("act", ["srelu", "tanh_srelu", "swiglu"])
@pytest.mark.parametrize("width", [64, 192])
def test_guards_fwd_bwd(act, recipe, width):
    rng = np.random.default_rng(400 + width + ACT_ID[act] + 9 * recipe)
    glu = act in GLU_NAMES
    split, x, p, dy = inputs.random_problem(rng, SPLIT, width, glu, x_sigma=2.0)
    split = [int(s) for s in split]
    E, M = len(split), int(sum(split))
    w_in = 2 * width if glu else width
    rht = recipe == oracle.NVFP4 and width % 64 == 0
    prm = gsa.ActParams(*params_tuple(act))
    rec = gsa.Recipe(recipe, int(rht), 0x2D4B)
    xd, pd, dyd = dev_bf16(x), dev_f32(p), dev_bf16(dy)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ws = Guarded(gsa.gsa_workspace_size(split, w_in, ACT_ID[act], recipe) + 256)
    ws_ptr = (ws.ptr + 255) // 256 * 256
    ws_bytes = ws.ptr + ws.nbytes - ws_ptr

    # forward: both copies and the dense Y
    info_y, _, _ = gsa.gsa_layout(split, width, recipe)
    gq, q = _qout(info_y, E, recipe)
    gy = Guarded(M * width * 2)
    st = gsa.grouped_scaled_act_fwd(xd.data_ptr(), pd.data_ptr(), split, w_in, ACT_ID[act], prm, rec, q, gy.ptr,
                                    ws_ptr, ws_bytes, stream)
    assert st == 0
    ref = gsa.fwd(xd, pd, split, act, recipe, rht, 0x2D4B, True, True, True, prm)
    torch.cuda.synchronize()
    _check(dict(gq, y=gy), ref, f"{act} fwd")

    # backward: dense dX, quantized dX, dprobs and the regenerated columnwise Y
    info_x, _, _ = gsa.gsa_layout(split, w_in, recipe)
    gx, qx = _qout(info_x, E, recipe)
    gr, qr = _qout(info_y, E, recipe, row=False, col=True)
    gdx, gdp = Guarded(M * w_in * 2), Guarded(4 * M)
    st = gsa.grouped_scaled_act_bwd(dyd.data_ptr(), xd.data_ptr(), pd.data_ptr(), split, w_in, ACT_ID[act], prm, rec,
                                    gdx.ptr, qx, gdp.ptr, qr, ws_ptr, ws_bytes, stream)
    assert st == 0
    refb = gsa.bwd(dyd, xd, pd, split, act, recipe, rht, 0x2D4B, True, True, True, True, True, prm)
    torch.cuda.synchronize()
    _check(dict(gx, dx=gdx, dprobs=gdp), refb, f"{act} bwd")
    _check({"y_" + k: v for k, v in gr.items()}, refb, f"{act} regen")
    assert ws.guards_intact(), "workspace guard overwritten"


def test_guards_graph_safe():
    """Graph-safe forward: outputs sized by gsa_layout_bound stay inside their
    bounds, and so does the padded-offset array."""
    rng = np.random.default_rng(401)
    split, x, p, _ = inputs.random_problem(rng, SPLIT, 128, False, x_sigma=2.0)
    split = [int(s) for s in split]
    E, M = len(split), int(sum(split))
    recipe = oracle.NVFP4
    prm = gsa.ActParams(*params_tuple("srelu"))
    rec = gsa.Recipe(recipe, 1, 0x2D4B)
    xd, pd = dev_bf16(x), dev_f32(p)
    sd = torch.tensor(split, dtype=torch.int64, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = Guarded(gsa.gsa_workspace_size_graph_safe(E, M, 128, 0, recipe) + 256)
    ws_ptr = (ws.ptr + 255) // 256 * 256
    info = gsa.gsa_layout_bound(E, M, 128, recipe)
    gq, q = _qout(info, E, recipe)
    gpad = Guarded(8 * (E + 1))
    st = gsa.grouped_scaled_act_fwd_graph_safe(xd.data_ptr(), pd.data_ptr(), sd.data_ptr(), E, M, 128, 0, prm, rec, q,
                                               None, gpad.ptr, ws_ptr, ws.ptr + ws.nbytes - ws_ptr, stream)
    assert st == 0
    ref = gsa.fwd(xd, pd, split, "srelu", recipe, True, 0x2D4B, True, True, False, prm)
    torch.cuda.synchronize()
    _check(gq, ref, "graph-safe fwd")
    assert gpad.guards_intact() and ws.guards_intact()
