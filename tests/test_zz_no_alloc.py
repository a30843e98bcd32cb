"""The allocation-free forward, gsa_fwd_noalloc.

Some callers cannot allocate device memory where they run the forward: an
operator called from inside another runtime's allocator or memory-planning
hook, or a plugin whose execute callback has no workspace argument and must
not call cudaMalloc (it can synchronize the device and fragment a
pre-planned pool).  gsa_fwd_noalloc serves them from a fixed scratch array
inside the library.  These checks call it through the C ABI twice in a row,
on problems of different shapes, and compare every output with the
workspace-taking grouped_scaled_act_fwd (bit for bit: the SReLU path is
exact).  The file is named to run last.
"""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_quantization_grouped_gb300 import gsa, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _dev(pr):
    x = torch.from_numpy(pr[1].view(np.int16)).view(torch.bfloat16).cuda()
    p = torch.from_numpy(pr[2]).cuda()
    return x, p


def _run_noalloc(x, p, split, act, recipe, rht, mask, width):
    out = gsa.alloc_qtensor(split, width, recipe, True, True, x.device)
    out["y"] = torch.empty((x.shape[0], width), dtype=torch.bfloat16, device=x.device)
    st = gsa.gsa_fwd_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(p.data_ptr()), split, x.shape[1],
                             gsa.ACT[act], gsa.ActParams(4.0, 7.0, 1.702, 1.0),
                             gsa.Recipe(recipe, int(rht), mask), gsa.qout_of(out), ctypes.c_void_p(out["y"].data_ptr()),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, gsa.STATUS.get(st, st)
    return out


def _same(a, b):
    for k in ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col", "y"):
        if k in a:
            ta, tb = a[k], b[k]
            assert torch.equal(ta.view(torch.uint8), tb.view(torch.uint8)), k


def _status():
    return gsa.gsa_fwd_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_forward_matches_workspace_forward_on_consecutive_calls():
    rng = np.random.default_rng(42)
    cases = [
        ([300, 0, 17, 129, 5], 256, gsa.NVFP4, True, 0xC0DE),     # two-pass NVFP4: ticket, done and amax counters
        ([64, 64, 1, 0, 0, 200, 33], 128, gsa.NVFP4, True, 0x0F0F),
        ([96, 40], 192, gsa.MXFP8, False, 0),
    ]
    for split, width, recipe, rht, mask in cases:
        pr = inputs.random_problem(rng, split, width, False)
        x, p = _dev(pr)
        ref = gsa.fwd(x, p, list(split), "srelu", recipe, rht, mask, True, True, True,
                      gsa.ActParams(4.0, 7.0, 1.702, 1.0))
        first = _run_noalloc(x, p, list(split), "srelu", recipe, rht, mask, width)
        second = _run_noalloc(x, p, list(split), "srelu", recipe, rht, mask, width)
        torch.cuda.synchronize()
        assert _status() == 0
        _same(first, ref)
        _same(second, ref)


@pytest.mark.parametrize("act", ["tanh_srelu", "swiglu", "clamped_swiglu"])
def test_noalloc_forward_other_activations_nvfp4_rht(act):
    """Without a workspace the NVFP4 encode pass recomputes Y from X (no
    staging copy): the ranged TanhSReLU form and the GLU forms (two X loads
    per tile) go through it, bit for bit equal to the workspace forward."""
    rng = np.random.default_rng(7 + gsa.ACT[act])
    glu = act in ("swiglu", "clamped_swiglu")
    split = [200, 0, 33, 129, 1]
    pr = inputs.random_problem(rng, split, 256, glu, x_sigma=3.0)
    x, p = _dev(pr)
    ref = gsa.fwd(x, p, list(split), act, gsa.NVFP4, True, 0x3C5A, True, True, True,
                  gsa.ActParams(4.0, 7.0, 1.702, 1.0))
    first = _run_noalloc(x, p, list(split), act, gsa.NVFP4, True, 0x3C5A, 256)
    second = _run_noalloc(x, p, list(split), act, gsa.NVFP4, True, 0x3C5A, 256)
    torch.cuda.synchronize()
    assert _status() == 0
    _same(first, ref)
    _same(second, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 256 experts x 80 bands each needs more counter words than the 64 KiB array holds;
    # rejected on the host before anything touches the device
    split = [128 * 80] * 256
    q = gsa.QOut(0x100000, 0x200000, None, None, 0x300000, None)
    st = gsa.gsa_fwd_noalloc(0x400000, 0x500000, split, 256, 0, gsa.ActParams(4.0, 7.0, 1.702, 1.0),
                             gsa.Recipe(gsa.NVFP4, 1, 1), q, None, None)
    assert st == 4   # GSA_ERR_WORKSPACE
