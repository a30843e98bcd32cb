"""Activation-generic GPU tests: every activation through the same fused kernel.

Recompute (the ScaledTanhSReLU recompute page, Description; its review thread
asks for recompute tests that do not depend on the activation): for each
activation and recipe,
  - the forward's rowwise copy and Y do not depend on whether the columnwise
    copy is kept (recompute changes only what is stashed);
  - the backward's dX, dprobs and quantized dX are bitwise the same with and
    without the regeneration of Y's columnwise copy;
  - the regenerated copy equals the saving forward's columnwise copy bit for
    bit (NVFP4: its per-expert amax too).

Two-step path (the same page: under NVFP4 the activation returns BF16 and a
separate quantizer requantizes it): the activation alone (dense BF16 Y)
followed by the identity activation with p = 1 (a plain grouped quantizer)
gives the fused call's quantized copies bit for bit, forward and backward.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import ACT_ID, GLU_NAMES, dev_bf16, dev_f32, gpu_bwd, gpu_fwd, host, params_tuple
from nvfp4_quantization_grouped_gb300 import gsa, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

SPLIT = [0, 37, 128, 300, 5, 0, 211]
WIDTH = 256
MASK = 0x5A3C
RECIPES = [oracle.MXFP8, oracle.NVFP4]
QKEYS = ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col")


def _problem(act, recipe):
    rng = np.random.default_rng(700 + 10 * ACT_ID[act] + recipe)
    return inputs.random_problem(rng, SPLIT, WIDTH, act in GLU_NAMES, x_sigma=1.5)


def _same(a, b, what):
    assert a.shape == b.shape, what
    assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), what


@pytest.mark.parametrize("recipe", RECIPES)
@pytest.mark.parametrize("act", list(ACT_ID))
def test_recompute_is_bitwise_neutral(act, recipe):
    split, x, p, dy = _problem(act, recipe)
    rht = recipe == oracle.NVFP4
    saving = gpu_fwd(x, p, split, act, recipe, rht, MASK, rowwise=True, columnwise=True, want_y=True)
    recomp = gpu_fwd(x, p, split, act, recipe, rht, MASK, rowwise=True, columnwise=False, want_y=True)
    assert "col_data" not in recomp
    for k in ("y", "row_data", "row_scale", "amax_row"):
        if k in saving:
            _same(recomp[k], saving[k], f"{act} fwd {k}")
    plain = gpu_bwd(dy, x, p, split, act, recipe, rht, MASK, regen=False)
    regen = gpu_bwd(dy, x, p, split, act, recipe, rht, MASK, regen=True)
    for k, v in plain.items():
        _same(regen[k], v, f"{act} bwd {k}")
    _same(regen["y_col_data"], saving["col_data"], f"{act} regenerated col_data")
    _same(regen["y_col_scale"], saving["col_scale"], f"{act} regenerated col_scale")
    if recipe == oracle.NVFP4:
        _same(regen["y_amax_col"], saving["amax_col"], f"{act} regenerated amax_col")


def _quantize(t, split, recipe, rht):
    """Second step of the unfused path: identity activation, p = 1."""
    out = gsa.fwd(t, None, split, "identity", recipe, rht, MASK, True, True, False,
                  gsa.ActParams(*params_tuple("identity")))
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items() if k != "_info"}


@pytest.mark.parametrize("recipe", RECIPES)
@pytest.mark.parametrize("act", list(ACT_ID))
def test_two_step_path_equals_fused(act, recipe):
    split, x, p, dy = _problem(act, recipe)
    split = list(split)
    rht = recipe == oracle.NVFP4
    prm = gsa.ActParams(*params_tuple(act))
    xd, pd, dyd = dev_bf16(x), dev_f32(p), dev_bf16(dy)
    fused = gpu_fwd(x, p, split, act, recipe, rht, MASK, want_y=False)
    y = gsa.fwd(xd, pd, split, act, recipe, rht, MASK, False, False, True, prm)["y"]
    two = _quantize(y, split, recipe, rht)
    for k in QKEYS:
        if k in fused:
            _same(two[k], fused[k], f"{act} fwd two-step {k}")
    fb = gpu_bwd(dy, x, p, split, act, recipe, rht, MASK)
    b1 = gsa.bwd(dyd, xd, pd, split, act, recipe, rht, MASK, True, False, False, True, False, prm)
    torch.cuda.synchronize()
    _same(host(b1["dx"]), fb["dx"], f"{act} bwd dX")
    _same(host(b1["dprobs"]), fb["dprobs"], f"{act} bwd dprobs")
    two_b = _quantize(b1["dx"], split, recipe, rht)
    for k in QKEYS:
        if k in fb:
            _same(two_b[k], fb[k], f"{act} bwd two-step {k}")


def test_null_probs_means_unit_scale():
    split, x, p, dy = _problem("sigmoid", oracle.NVFP4)
    ones = np.ones_like(p)
    for recipe in RECIPES:
        a = gpu_fwd(x, None, split, "sigmoid", recipe, recipe == oracle.NVFP4, MASK)
        b = gpu_fwd(x, ones, split, "sigmoid", recipe, recipe == oracle.NVFP4, MASK)
        for k in a:
            _same(a[k], b[k], f"null probs fwd {k}")
        yo = oracle.act_fwd_rows(x, None, ACT_ID["identity"], params_tuple("identity"))
        c = gpu_fwd(x, None, split, "identity", recipe, recipe == oracle.NVFP4, MASK)
        _same(c["y"].reshape(yo.shape), x, "identity Y with p = 1 is X")
        _same(yo, x, "oracle identity")
