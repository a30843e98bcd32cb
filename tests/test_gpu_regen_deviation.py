"""FC2-wgrad regeneration deviation with the CUDA path's regenerated copy.

The ScaledTanhSReLU recompute page (Description, regeneration-error table)
measures how FC2's wgrad moves when the columnwise quantized Y that FC2's
wgrad consumes is regenerated in the backward from the saved BF16 FC1 output
instead of being quantized in the forward from the FP32 accumulator.  Here the
regenerating side is the library itself: grouped_scaled_act_bwd with
y_regen_col_opt on bf16(X), through the C ABI.  The saving side is the oracle
(an FP32-input forward, which the kernel does not take).  Both quantized copies
are dequantized and multiplied with FC2's output gradient in float64 exactly
as in the oracle-only experiment (tests/test_regen_deviation.py).  On SReLU
the regenerated copy is bitwise the oracle's, so the figures are identical
bit for bit; on TanhSReLU they agree to the tolerance of its library tanh.
"""
import numpy as np
import pytest
import torch

import oracle
import test_regen_deviation as R
from gpu_util import dev_bf16, dev_f32
from nvfp4_quantization_grouped_gb300 import gsa

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _gpu_regen_wgrad(x32, p, dy2, split, act, recipe, rht):
    """FC2 wgrad from the CUDA path's regenerated columnwise copy of Y."""
    a, prm = R.ACTS[act]
    xb = oracle.f32_to_bf16(x32)
    dy = np.zeros((xb.shape[0], xb.shape[1]), np.uint16)      # the regenerated copy does not depend on dY
    out = gsa.bwd(dev_bf16(dy), dev_bf16(xb), dev_f32(p), list(split), act, recipe, rht, R.MASK,
                  False, False, False, True, True, gsa.ActParams(*prm))
    torch.cuda.synchronize()
    cd = out["y_col_data"].cpu().numpy()
    cs = out["y_col_scale"].cpu().numpy()
    am = out["y_amax_col"].cpu().numpy() if recipe == oracle.NVFP4 else None
    width = xb.shape[1]
    dof, sof = oracle.expert_col_offsets(split, width, recipe)
    b = oracle.block_size(recipe)
    offs = np.concatenate([[0], np.cumsum(split)]).astype(np.int64)
    res = []
    for e in range(len(split)):
        me = int(split[e])
        mp = oracle.padded_rows(me, recipe)
        d = cd[dof[e]:dof[e + 1]].reshape(width, mp if recipe == oracle.MXFP8 else mp // 2)
        s = cs[sof[e]:sof[e + 1]].reshape(width, mp // b)
        S = oracle.nvfp4_tensor_scale(float(am[e])) if recipe == oracle.NVFP4 else 1.0
        vals = oracle.dequant_cols(d, s, recipe, S)
        g = np.zeros((mp, dy2.shape[1]))
        g[:me] = dy2[offs[e]:offs[e + 1]]
        if recipe == oracle.NVFP4 and rht:
            g = oracle.rht_cols(g, R.MASK)
        res.append(g.T @ vals.T)
    return np.stack(res)


@pytest.mark.parametrize("act", ["srelu", "tanh_srelu"])
@pytest.mark.parametrize("recipe,rht", [(oracle.MXFP8, False), (oracle.NVFP4, True)])
def test_regeneration_deviation_through_the_cuda_path(act, recipe, rht):
    x32, p, dy2, split = R._inputs()
    a, prm = R.ACTS[act]
    y_saved = oracle.act_fwd_rows_f32(x32, p, a, prm)
    w_saved = R._wgrad(split, y_saved, dy2, recipe, rht)
    w_regen = _gpu_regen_wgrad(x32, p, dy2, split, act, recipe, rht)
    diff = w_regen - w_saved
    rms = np.sqrt(np.mean(w_saved ** 2))
    got = np.array([np.max(np.abs(diff)) / rms, np.sqrt(np.mean(diff ** 2)) / rms, np.mean(diff) / rms])
    ref = np.array(R._deviation(x32, p, dy2, split, act, recipe, rht))
    if act == "srelu":
        assert np.array_equal(got, ref), (got, ref)           # the regenerated copy is the oracle's, bit for bit
    else:
        assert np.allclose(got[:2], ref[:2], rtol=0.02), (got, ref)
        assert abs(got[2]) < 0.01
