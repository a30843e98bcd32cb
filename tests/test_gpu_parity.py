"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

SReLU and identity paths are compared bit for bit (Y, dX, dprobs, codes,
scales, amax).  TanhSReLU / SwiGLU / clamped SwiGLU / GeLU / sigmoid use
library transcendentals on both sides (CUDA's tanhf/expf/erfcf on the GPU, the
C library's on the CPU) and are held to:
  * BF16 Y and dX within 2 ULP;
  * quantized copies (codes, scales, amax) bit for bit equal to the oracle's
    quantization of the GPU's own BF16 values;
  * against the oracle's quantization of its own values: amax within the
    shift 2 ULP of BF16 can cause (experts whose amax moved are re-encoded by
    the oracle with the GPU's amax and counted), block scales equal except
    adjacent codes on at most 1e-3 of the blocks, codes one step apart on at
    most 1e-3 of the elements;
  * dprobs within the bound derived from the activation's error bound and
    the summation tree (``gpu_util.dprobs_bound``).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (assert_bf16, assert_dprobs, assert_quant, bf16_ulp_diff, gpu_bwd, gpu_fwd, host, params_tuple,
                      rht_amax_shift_bound, ACT_ID, EXACT_ACTS, GLU_NAMES, dev_bf16, dev_f32)
from nvfp4_quantization_grouped_gb300 import gsa, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _col_offsets(split, width, recipe):
    d, s = oracle.expert_col_offsets(split, width, recipe)
    return d, s


def _amax_within_bound(got, ref, v_e, col, rht):
    """Whether an expert's amax moved by no more than 2 BF16 ULP of its values
    allow: rowwise, and columnwise without the RHT, the amax is a BF16 value
    max |v| (2 ULP in the BF16 order); columnwise with the RHT, the shift
    bound of the transform."""
    if not (col and rht):
        return bf16_ulp_diff(np.float32(got).view(np.uint32) >> 16, np.float32(ref).view(np.uint32) >> 16) <= 2
    return abs(float(got) - float(ref)) <= rht_amax_shift_bound(v_e)


def _oracle_quant(v, split, recipe, rht, mask, want_row, want_col, amax_row=None, amax_col=None, what=""):
    """Oracle quantization of v.  For NVFP4, when the GPU's per-expert amax is
    given (approximate paths), an expert whose amax moved -- by no more than
    the 2-ULP shift bound, which is asserted -- is re-encoded with the GPU's
    amax, so that both sides take the integer decisions from the same scale.
    Returns (result, number of re-encoded experts)."""
    out = oracle.quantize_grouped(v, split, recipe, rht, mask, want_row, want_col)
    moved = 0
    if recipe != oracle.NVFP4 or (amax_row is None and amax_col is None):
        return out, moved
    offs = np.concatenate([[0], np.cumsum(split)]).astype(np.int64)
    if want_row and amax_row is not None:
        for e in range(len(split)):
            if split[e] and amax_row[e] != out["amax_row"][e]:
                ve = v[offs[e]:offs[e + 1]]
                assert _amax_within_bound(amax_row[e], out["amax_row"][e], ve, False, rht), \
                    f"{what} amax_row e{e}: {amax_row[e]} vs {out['amax_row'][e]}"
                d, s = oracle.quant_rows(ve, recipe, oracle.nvfp4_tensor_scale(amax_row[e]))
                out["row_data"][offs[e]:offs[e + 1]] = d
                out["row_scale"][offs[e]:offs[e + 1]] = s
                moved += 1
    if want_col and amax_col is not None:
        dof, sof = _col_offsets(split, v.shape[1], recipe)
        for e in range(len(split)):
            if split[e] and amax_col[e] != out["amax_col"][e]:
                ve = v[offs[e]:offs[e + 1]]
                assert _amax_within_bound(amax_col[e], out["amax_col"][e], ve, True, rht), \
                    f"{what} amax_col e{e}: {amax_col[e]} vs {out['amax_col'][e]}"
                d, s = oracle.quant_cols(ve, recipe, rht, mask, oracle.nvfp4_tensor_scale(amax_col[e]))
                out["col_data"][dof[e]:dof[e + 1]] = d.reshape(-1)
                out["col_scale"][sof[e]:sof[e + 1]] = s.reshape(-1)
                moved += 1
    return out, moved


def _check_amax(got, ref, what):
    assert np.array_equal(np.asarray(got).view(np.uint32), np.asarray(ref).view(np.uint32)), f"{what}: {got} vs {ref}"


def _quant_bitwise(g, vals, split, recipe, rht, mask, want_row, want_col, what, prefix=""):
    """The GPU's quantized copies equal the oracle's quantization of `vals`
    bit for bit (codes, scales and, for NVFP4, every expert's amax)."""
    B = 32 if recipe == oracle.MXFP8 else 16
    ref = oracle.quantize_grouped(vals, split, recipe, rht, mask, want_row, want_col)
    if want_row:
        if recipe == oracle.NVFP4:
            _check_amax(g[prefix + "amax_row"], ref["amax_row"], what + " amax_row")
        assert_quant(g[prefix + "row_data"], g[prefix + "row_scale"], ref["row_data"], ref["row_scale"], recipe,
                     True, what + " rowwise", B)
    if want_col:
        if recipe == oracle.NVFP4:
            _check_amax(g[prefix + "amax_col"], ref["amax_col"], what + " amax_col")
        n = ref["col_data"].size
        assert_quant(g[prefix + "col_data"][:n], g[prefix + "col_scale"][:ref["col_scale"].size],
                     ref["col_data"], ref["col_scale"], recipe, True, what + " columnwise", B)


def _compare_quant(g, o_vals, split, recipe, rht, mask, exact, want_row, want_col, what, prefix="", g_vals=None):
    """Quantized copies against the oracle: bit for bit on the exact paths;
    on the approximate paths bit for bit against the quantization of the
    GPU's own values (g_vals, when given) and within the tolerance against
    the quantization of the oracle's values.  Returns the re-encoded expert
    count."""
    B = 32 if recipe == oracle.MXFP8 else 16
    if exact:
        _quant_bitwise(g, o_vals, split, recipe, rht, mask, want_row, want_col, what, prefix)
        return 0
    if g_vals is not None:
        _quant_bitwise(g, g_vals, split, recipe, rht, mask, want_row, want_col, what + " (GPU values)", prefix)
    ar = g.get(prefix + "amax_row") if recipe == oracle.NVFP4 and want_row else None
    ac = g.get(prefix + "amax_col") if recipe == oracle.NVFP4 and want_col else None
    ref, moved = _oracle_quant(o_vals, split, recipe, rht, mask, want_row, want_col, ar, ac, what)
    if want_row:
        assert_quant(g[prefix + "row_data"], g[prefix + "row_scale"], ref["row_data"], ref["row_scale"], recipe,
                     False, f"{what} rowwise ({moved} expert amax re-encoded)", B)
    if want_col:
        n = ref["col_data"].size
        assert_quant(g[prefix + "col_data"][:n], g[prefix + "col_scale"][:ref["col_scale"].size],
                     ref["col_data"], ref["col_scale"], recipe, False,
                     f"{what} columnwise ({moved} expert amax re-encoded)", B)
    return moved


def run_fwd_case(split, x, p, act, recipe, rht=False, mask=0, rowwise=True, columnwise=True, prm=None):
    exact = act in EXACT_ACTS
    prm = prm or params_tuple(act)
    g = gpu_fwd(x, p, split, act, recipe, rht, mask, rowwise, columnwise, want_y=True, prm=prm)
    y = oracle.act_fwd_rows(x, p, ACT_ID[act], prm)
    gy = g["y"].reshape(y.shape)
    assert_bf16(gy, y, exact, f"{act} Y")
    _compare_quant(g, y, split, recipe, rht, mask, exact, rowwise, columnwise, f"{act} fwd", g_vals=gy)
    return g, y


def run_bwd_case(split, x, p, dy, act, recipe, rht=False, mask=0, rowwise=True, columnwise=True, regen=False,
                 prm=None):
    exact = act in EXACT_ACTS
    prm = prm or params_tuple(act)
    g = gpu_bwd(dy, x, p, split, act, recipe, rht, mask, rowwise, columnwise, regen, prm=prm)
    dx, dpr = oracle.act_bwd_rows(dy, x, p, ACT_ID[act], prm)
    gdx = g["dx"].reshape(dx.shape)
    assert_bf16(gdx, dx, exact, f"{act} dX")
    assert_dprobs(g["dprobs"], dpr, dy, x, p, act, exact, f"{act} dprobs", prm)
    if rowwise or columnwise:
        _compare_quant(g, dx, split, recipe, rht, mask, exact, rowwise, columnwise, f"{act} bwd dX", g_vals=gdx)
    if regen:
        y = oracle.act_fwd_rows(x, p, ACT_ID[act], prm)
        gy = None
        if not exact:   # the GPU's own Y, from a forward on the same inputs
            gy = gpu_fwd(x, p, split, act, recipe, rht, mask, False, False, want_y=True, prm=prm)["y"].reshape(y.shape)
        _compare_quant(g, y, split, recipe, rht, mask, exact, False, True, f"{act} regen Y", prefix="y_", g_vals=gy)
    return g


# ------------------------------------------------------------------ workloads

def test_tiny_srelu_mxfp8_fwd_bwd():
    pr = inputs.make_problem("tiny_srelu_mxfp8", 0)
    run_fwd_case(pr.split_sizes, pr.x, pr.probs, "srelu", oracle.MXFP8)
    run_bwd_case(pr.split_sizes, pr.x, pr.probs, pr.dy, "srelu", oracle.MXFP8)


@pytest.mark.parametrize("act", ["tanh_srelu", "srelu"])
def test_tanh_srelu_mxfp8_recompute(act):
    pr = inputs.make_problem("tanh_srelu_mxfp8_recompute", 0)
    # recompute mode: the forward writes the rowwise copy only
    g_row, _ = run_fwd_case(pr.split_sizes, pr.x, pr.probs, act, oracle.MXFP8, rowwise=True, columnwise=False)
    assert "col_data" not in g_row
    gb = run_bwd_case(pr.split_sizes, pr.x, pr.probs, pr.dy, act, oracle.MXFP8, regen=True)
    # the regenerated columnwise copy equals what a saving forward would have written, bit for bit
    g_full = gpu_fwd(pr.x, pr.probs, pr.split_sizes, act, oracle.MXFP8, rowwise=False, columnwise=True,
                     want_y=False)
    assert np.array_equal(gb["y_col_data"], g_full["col_data"])
    assert np.array_equal(gb["y_col_scale"], g_full["col_scale"])


@pytest.mark.parametrize("act", ["swiglu", "clamped_swiglu"])
def test_swiglu_mxfp8(act):
    pr = inputs.make_problem("swiglu_mxfp8", 0, rows=4096)
    assert (pr.split_sizes == 0).any()
    run_fwd_case(pr.split_sizes, pr.x, pr.probs, act, oracle.MXFP8)
    run_bwd_case(pr.split_sizes, pr.x, pr.probs, pr.dy, act, oracle.MXFP8)


@pytest.mark.parametrize("act", ["srelu", "tanh_srelu"])
def test_nvfp4_rht(act):
    pr = inputs.make_problem("nvfp4_rht", 0, rows=8192)
    run_fwd_case(pr.split_sizes, pr.x, pr.probs, act, oracle.NVFP4, True, pr.rht_mask)
    g = run_bwd_case(pr.split_sizes, pr.x, pr.probs, pr.dy, act, oracle.NVFP4, True, pr.rht_mask, regen=True)
    gf = gpu_fwd(pr.x, pr.probs, pr.split_sizes, act, oracle.NVFP4, True, pr.rht_mask, False, True, False)
    assert np.array_equal(g["y_col_data"], gf["col_data"]) and np.array_equal(g["y_col_scale"], gf["col_scale"])
    assert np.array_equal(g["y_amax_col"].view(np.uint32), gf["amax_col"].view(np.uint32))


@pytest.mark.parametrize("act", ["gelu", "sigmoid", "identity"])
def test_further_unary_acts_workloads(act):
    """GeLU, sigmoid and identity on the NVFP4 + RHT workload (8192 rows of it)
    and on the MXFP8 recompute workload, forward, backward and regeneration."""
    pr = inputs.make_problem("nvfp4_rht", 0, rows=8192)
    run_fwd_case(pr.split_sizes, pr.x, pr.probs, act, oracle.NVFP4, True, pr.rht_mask)
    run_bwd_case(pr.split_sizes, pr.x, pr.probs, pr.dy, act, oracle.NVFP4, True, pr.rht_mask, regen=True)
    pm = inputs.make_problem("tanh_srelu_mxfp8_recompute", 0)
    run_fwd_case(pm.split_sizes, pm.x, pm.probs, act, oracle.MXFP8, rowwise=True, columnwise=False)
    run_bwd_case(pm.split_sizes, pm.x, pm.probs, pm.dy, act, oracle.MXFP8, regen=True)


def test_moe_swiglu_mxfp8_recompute_reduced():
    pr = inputs.make_problem("moe_swiglu_mxfp8_recompute", 0, rows=6144)
    run_fwd_case(pr.split_sizes, pr.x, pr.probs, "swiglu", oracle.MXFP8, rowwise=True, columnwise=False)
    run_bwd_case(pr.split_sizes, pr.x, pr.probs, pr.dy, "swiglu", oracle.MXFP8, regen=True)


# ------------------------------------------------------------------ edge cases

EDGE_SPLITS = [[0, 1, 15, 17, 0, 31, 33, 128, 129, 255], [0], [0, 0, 5], [300]]


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
@pytest.mark.parametrize("act", list(ACT_ID))
@pytest.mark.parametrize("width", [64, 192, 1024])
def test_edge_shapes(recipe, act, width):
    rng = np.random.default_rng(100 + width + 7 * recipe + ACT_ID[act])
    glu = act in GLU_NAMES
    for split in EDGE_SPLITS:
        split, x, p, dy = inputs.random_problem(rng, split, width, glu, x_sigma=1.5)
        rht = recipe == oracle.NVFP4 and width != 192
        mask = 0xA5C3
        if sum(split) == 0:
            continue
        run_fwd_case(split, x, p, act, recipe, rht, mask)
        run_bwd_case(split, x, p, dy, act, recipe, rht, mask, regen=True)


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
@pytest.mark.parametrize("act,width", [("srelu", 16384), ("srelu", 65536), ("swiglu", 16384), ("tanh_srelu", 32768)])
def test_wide_rows(recipe, act, width):
    """Rows wide enough that the policy's item size would give a band more
    slabs than the dprobs slab merge holds take larger items: forward and
    backward (with regeneration) against the oracle on a ragged split."""
    rng = np.random.default_rng(400 + width // 1024 + 7 * recipe + ACT_ID[act])
    split, x, p, dy = inputs.random_problem(rng, [40, 0, 17, 1], width, act in GLU_NAMES, x_sigma=1.5)
    rht = recipe == oracle.NVFP4
    run_fwd_case(split, x, p, act, recipe, rht, 0x5A5A)
    run_bwd_case(split, x, p, dy, act, recipe, rht, 0x5A5A, regen=True)


@pytest.mark.parametrize("act", list(ACT_ID))
def test_nvfp4_bwd_without_regenerated_copy(act):
    """The NVFP4 backward that does not regenerate Y (the costly activations
    run their own kernel variant for it, with the columnwise codes from warps
    that own whole 16-row blocks): against the oracle on ragged splits and
    widths, and bit for bit equal to the same call with the regenerated copy."""
    rng = np.random.default_rng(300 + ACT_ID[act])
    glu = act in GLU_NAMES
    for split, width in (([0, 1, 15, 17, 0, 31, 33, 128, 129, 255], 192), ([300, 77], 1024), ([64], 64)):
        split, x, p, dy = inputs.random_problem(rng, split, width, glu, x_sigma=1.5)
        rht = width != 192
        a = run_bwd_case(split, x, p, dy, act, oracle.NVFP4, rht, 0xA5C3, regen=False)
        b = gpu_bwd(dy, x, p, split, act, oracle.NVFP4, rht, 0xA5C3, regen=True)
        for k, v in a.items():
            assert np.array_equal(np.asarray(v).view(np.uint8), np.asarray(b[k]).view(np.uint8)), (act, width, k)


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
@pytest.mark.parametrize("s", [3.0, 0.7, 8.0, 5.5])
def test_tanh_srelu_any_s(s, recipe):
    """TanhSReLU with s a power of two (x / s a product) and not (a true
    division, which also takes the exact derivative form): forward, backward
    and the regenerated copy against the oracle, and the regenerated copy
    bitwise equal to the forward's."""
    rng = np.random.default_rng(int(40 * s) + recipe)
    split, x, p, dy = inputs.random_problem(rng, [0, 200, 33, 129], 256, False, x_sigma=3.0)
    prm = (s, 7.0, 1.702, 1.0)
    rht = recipe == oracle.NVFP4
    gf, _ = run_fwd_case(split, x, p, "tanh_srelu", recipe, rht, 0x1F2E, prm=prm)
    gb = run_bwd_case(split, x, p, dy, "tanh_srelu", recipe, rht, 0x1F2E, regen=True, prm=prm)
    assert np.array_equal(gb["y_col_data"], gf["col_data"]) and np.array_equal(gb["y_col_scale"], gf["col_scale"])


def test_nvfp4_without_rht_and_partial_outputs():
    rng = np.random.default_rng(5)
    split, x, p, dy = inputs.random_problem(rng, [40, 0, 200], 128, False)
    run_fwd_case(split, x, p, "srelu", oracle.NVFP4, False, 0, rowwise=True, columnwise=False)
    run_fwd_case(split, x, p, "srelu", oracle.NVFP4, False, 0, rowwise=False, columnwise=True)
    g = gpu_bwd(dy, x, p, split, "srelu", oracle.NVFP4, False, 0, rowwise=False, columnwise=False,
                regen=False, want_dx=False, want_dprobs=True)   # frozen fc1: dprobs alone
    _, dpr = oracle.act_bwd_rows(dy, x, p, 0, params_tuple("srelu"))
    assert np.array_equal(g["dprobs"].view(np.uint32), dpr.view(np.uint32))


@pytest.mark.parametrize("act", ["srelu", "tanh_srelu", "swiglu"])
def test_nvfp4_regen_and_dprobs_without_dx(act):
    """A backward that asks only for dprobs and the regenerated columnwise Y
    (no dense and no quantized dX): its encode items load X alone."""
    rng = np.random.default_rng(11 + ACT_ID[act])
    glu = act in GLU_NAMES
    split, x, p, dy = inputs.random_problem(rng, [130, 0, 17, 300], 128, glu, x_sigma=1.5)
    prm = params_tuple(act)
    exact = act in EXACT_ACTS
    g = gpu_bwd(dy, x, p, split, act, oracle.NVFP4, True, 0x6B1D, rowwise=False, columnwise=False, regen=True,
                want_dx=False, want_dprobs=True)
    assert "dx" not in g and "row_data" not in g
    _, dpr = oracle.act_bwd_rows(dy, x, p, ACT_ID[act], prm)
    assert_dprobs(g["dprobs"], dpr, dy, x, p, act, exact, f"{act} dprobs", prm)
    y = oracle.act_fwd_rows(x, p, ACT_ID[act], prm)
    gy = None if exact else gpu_fwd(x, p, split, act, oracle.NVFP4, True, 0x6B1D, False, False, want_y=True,
                                    prm=prm)["y"].reshape(y.shape)
    _compare_quant(g, y, split, oracle.NVFP4, True, 0x6B1D, exact, False, True, f"{act} regen Y", prefix="y_",
                   g_vals=gy)


def test_all_experts_empty():
    split = [0, 0, 0]
    x = np.zeros((0, 64), np.uint16)
    g = gsa.fwd(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"),
                torch.zeros(0, dtype=torch.float32, device="cuda"), split, "srelu", oracle.NVFP4, True, 1)
    torch.cuda.synchronize()
    assert torch.all(g["amax_row"] == 0) and torch.all(g["amax_col"] == 0)


def test_repeatable_bitwise():
    pr = inputs.make_problem("nvfp4_rht", 1, rows=4096)
    a = gpu_bwd(pr.dy, pr.x, pr.probs, pr.split_sizes, "tanh_srelu", oracle.NVFP4, True, pr.rht_mask, regen=True)
    b = gpu_bwd(pr.dy, pr.x, pr.probs, pr.split_sizes, "tanh_srelu", oracle.NVFP4, True, pr.rht_mask, regen=True)
    for k in a:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


def test_recompute_drops_forward_memory():
    """Forward in recompute mode keeps no columnwise copy of Y; the backward
    regenerates it.  Memory held between forward and backward drops by exactly
    the columnwise copy's bytes."""
    pr = inputs.make_problem("tanh_srelu_mxfp8_recompute", 0)
    x, p = dev_bf16(pr.x), dev_f32(pr.probs)
    split = list(pr.split_sizes)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    saved = gsa.fwd(x, p, split, "tanh_srelu", oracle.MXFP8, rowwise=True, columnwise=True)
    torch.cuda.synchronize()
    held_save = torch.cuda.memory_allocated() - base
    del saved
    rec = gsa.fwd(x, p, split, "tanh_srelu", oracle.MXFP8, rowwise=True, columnwise=False)
    torch.cuda.synchronize()
    held_rec = torch.cuda.memory_allocated() - base
    info, _, _ = gsa.gsa_layout(split, 1024, oracle.MXFP8)
    assert held_save - held_rec >= info.col_data_bytes + info.col_scale_bytes
    del rec


def test_workspace_status_ok_after_calls():
    pr = inputs.make_problem("nvfp4_rht", 0, rows=2048)
    x, p, dy = dev_bf16(pr.x), dev_f32(pr.probs), dev_bf16(pr.dy)
    split = list(pr.split_sizes)
    ws = gsa.Workspace(split, 2048, 0, oracle.NVFP4, x.device)
    gsa.fwd(x, p, split, "srelu", oracle.NVFP4, True, pr.rht_mask, ws=ws)
    gsa.bwd(dy, x, p, split, "srelu", oracle.NVFP4, True, pr.rht_mask, ws=ws, regen=True)
    assert ws.status() == 0
    assert gsa.gsa_last_launch_count() == 1


def test_nvfp4_repeated_calls_match_oracle():
    """Back-to-back NVFP4 forwards with different output sets: every call's
    per-expert amax and codes must match the oracle (guards the cross-CTA
    amax publication and the Y staging copy against ordering races)."""
    pr = inputs.make_problem("nvfp4_rht", 2, rows=8192)
    split = [int(s) for s in pr.split_sizes]
    y = oracle.act_fwd_rows(pr.x, pr.probs, ACT_ID["srelu"], params_tuple("srelu"))
    ref = oracle.quantize_grouped(y, split, oracle.NVFP4, True, pr.rht_mask, True, True)
    x, p = dev_bf16(pr.x), dev_f32(pr.probs)
    prm = gsa.ActParams(*params_tuple("srelu"))
    for it in range(4):
        for rw, cw in [(True, True), (False, True), (True, False)]:
            out = gsa.fwd(x, p, split, "srelu", oracle.NVFP4, True, pr.rht_mask, rw, cw, False, prm)
            torch.cuda.synchronize()
            if rw:
                assert np.array_equal(out["amax_row"].cpu().numpy(), ref["amax_row"]), (it, rw, cw)
                assert np.array_equal(out["row_data"].cpu().numpy().reshape(ref["row_data"].shape), ref["row_data"])
            if cw:
                assert np.array_equal(out["amax_col"].cpu().numpy(), ref["amax_col"]), (it, rw, cw)
                assert np.array_equal(out["col_data"].cpu().numpy(), ref["col_data"])
                assert np.array_equal(out["col_scale"].cpu().numpy(), ref["col_scale"])


# ------------------------------------------------------- full-size workloads

def _expert_slice(split, e):
    offs = np.concatenate([[0], np.cumsum(split)]).astype(np.int64)
    return int(offs[e]), int(offs[e + 1])


def _check_full_size(name, act, recipe, rht, sample_experts):
    """Full-size workload in the benchmark's launch configuration.  The oracle
    recomputes a sample of whole experts element by element (rowwise,
    columnwise, dense dX, dprobs, regenerated copy) and, for NVFP4, the amax of
    every expert (forward Y, backward dX, regenerated Y): bit for bit on the
    exact paths; on the approximate ones bit for bit from the GPU's own BF16
    values and within the 2-ULP shift bound from the oracle's."""
    pr = inputs.make_problem(name, 0)
    split = [int(s) for s in pr.split_sizes]
    wl = pr.workload
    exact = act in EXACT_ACTS
    prm = params_tuple(act)
    g = gpu_fwd(pr.x, pr.probs, split, act, recipe, rht, pr.rht_mask, True, not wl.recompute, want_y=True)
    b = gpu_bwd(pr.dy, pr.x, pr.probs, split, act, recipe, rht, pr.rht_mask, True, True, regen=wl.recompute)
    g_y = g["y"].reshape(-1, wl.width)
    g_dx = b["dx"].reshape(-1, wl.w_in)
    offs = np.concatenate([[0], np.cumsum(split)]).astype(np.int64)
    if recipe == oracle.NVFP4:
        # every expert's amax, from the oracle's values and from the GPU's
        y_all = oracle.act_fwd_rows(pr.x, pr.probs, ACT_ID[act], prm)
        dx_all, _ = oracle.act_bwd_rows(pr.dy, pr.x, pr.probs, ACT_ID[act], prm, want_dprobs=False)
        checks = [("fwd amax_row", g["amax_row"], y_all, g_y, False),
                  ("bwd amax_row", b["amax_row"], dx_all, g_dx, False),
                  ("bwd amax_col", b["amax_col"], dx_all, g_dx, True)]
        if not wl.recompute:
            checks.append(("fwd amax_col", g["amax_col"], y_all, g_y, True))
        else:
            checks.append(("regen amax_col", b["y_amax_col"], y_all, g_y, True))
        for what, got, vals, gvals, col in checks:
            for e in range(len(split)):
                lo, hi = offs[e], offs[e + 1]
                if hi == lo:
                    assert got[e] == 0.0, f"{name} e{e} {what}: empty expert"
                    continue
                amax = (lambda v: oracle.amax_cols(v, rht, pr.rht_mask)) if col else oracle.amax_rows
                ref_own = np.float32(amax(gvals[lo:hi]))
                assert got[e].view(np.uint32) == ref_own.view(np.uint32), f"{name} e{e} {what} (GPU values)"
                ref = np.float32(amax(vals[lo:hi]))
                if exact:
                    assert got[e].view(np.uint32) == ref.view(np.uint32), f"{name} e{e} {what}"
                else:
                    assert _amax_within_bound(got[e], ref, vals[lo:hi], col, rht), f"{name} e{e} {what}"
    dof_y, sof_y = oracle.expert_col_offsets(split, wl.width, recipe)
    dof_x, sof_x = oracle.expert_col_offsets(split, wl.w_in, recipe)
    nb = 32 if recipe == oracle.MXFP8 else 16
    rw_y = wl.width if recipe == oracle.MXFP8 else wl.width // 2
    rw_x = wl.w_in if recipe == oracle.MXFP8 else wl.w_in // 2
    for e in sample_experts:
        lo, hi = _expert_slice(split, e)
        if hi == lo:
            continue
        se = [hi - lo]
        xs, ps, dys = pr.x[lo:hi], pr.probs[lo:hi], pr.dy[lo:hi]
        y = oracle.act_fwd_rows(xs, ps, ACT_ID[act], prm)
        dx, dpr = oracle.act_bwd_rows(dys, xs, ps, ACT_ID[act], prm)
        assert_bf16(g_y[lo:hi], y, exact, f"{name} e{e} Y")
        gy = {"row_data": g["row_data"].reshape(-1, rw_y)[lo:hi], "row_scale": g["row_scale"].reshape(-1, wl.width // nb)[lo:hi]}
        if not wl.recompute:
            gy.update(col_data=g["col_data"][dof_y[e]:dof_y[e + 1]], col_scale=g["col_scale"][sof_y[e]:sof_y[e + 1]])
        if recipe == oracle.NVFP4:
            gy.update(amax_row=g["amax_row"][e:e + 1], amax_col=g["amax_col"][e:e + 1] if "amax_col" in g else None)
        _compare_quant(gy, y, se, recipe, rht, pr.rht_mask, exact, True, not wl.recompute, f"{name} e{e} fwd",
                       g_vals=g_y[lo:hi])
        assert_bf16(g_dx[lo:hi], dx, exact, f"{name} e{e} dX")
        assert_dprobs(b["dprobs"][lo:hi], dpr, dys, xs, ps, act, exact, f"{name} e{e} dprobs")
        gx = {"row_data": b["row_data"].reshape(-1, rw_x)[lo:hi], "row_scale": b["row_scale"].reshape(-1, wl.w_in // nb)[lo:hi],
              "col_data": b["col_data"][dof_x[e]:dof_x[e + 1]], "col_scale": b["col_scale"][sof_x[e]:sof_x[e + 1]]}
        if recipe == oracle.NVFP4:
            gx.update(amax_row=b["amax_row"][e:e + 1], amax_col=b["amax_col"][e:e + 1])
        _compare_quant(gx, dx, se, recipe, rht, pr.rht_mask, exact, True, True, f"{name} e{e} bwd dX",
                       g_vals=g_dx[lo:hi])
        if wl.recompute:
            gr = {"col_data": b["y_col_data"][dof_y[e]:dof_y[e + 1]], "col_scale": b["y_col_scale"][sof_y[e]:sof_y[e + 1]]}
            if recipe == oracle.NVFP4:
                gr["amax_col"] = b["y_amax_col"][e:e + 1]
            _compare_quant(gr, y, se, recipe, rht, pr.rht_mask, exact, False, True, f"{name} e{e} regen Y",
                           g_vals=g_y[lo:hi])


def _sample_of(split):
    """Smallest non-empty, median and largest expert (plus any empty one)."""
    nz = [e for e in range(len(split)) if split[e] > 0]
    order = sorted(nz, key=lambda e: split[e])
    sample = [order[0], order[len(order) // 2], order[-1]]
    sample += [e for e in range(len(split)) if split[e] == 0][:1]
    return sample


@pytest.mark.parametrize("act", ["srelu", "tanh_srelu"])
def test_full_size_nvfp4_rht_sampled_experts(act):
    """NVFP4 + RHT workload at its full size (65536 x 2048, 32 experts)."""
    split, _ = inputs.make_split(inputs.WORKLOADS["nvfp4_rht"], np.random.default_rng(0))
    _check_full_size("nvfp4_rht", act, oracle.NVFP4, True, _sample_of(split))


def test_full_size_moe_swiglu_mxfp8_recompute_sampled_experts():
    """Routed MoE workload at its full size (262144 rows x 2 x 4096, 128 experts,
    four empty), forward in recompute mode (rowwise copy and Y) and backward with
    the regenerated copy, in the benchmark's launch configuration.  X and dY are
    drawn on the device (a host draw of the 4.3 GB input takes minutes); only the
    sampled experts' rows come back for the oracle: the smallest, median and
    largest expert (29629 rows) and an empty one."""
    wl, split, M, x, p, dy = inputs.device_problem("moe_swiglu_mxfp8_recompute", torch.device("cuda"))
    assert sum(1 for v in split if v == 0) == 4
    prm = params_tuple("swiglu")
    ap = gsa.ActParams(*prm)
    R = oracle.MXFP8
    g = gsa.fwd(x, p, split, "swiglu", R, False, 0, True, False, True, ap)
    b = gsa.bwd(dy, x, p, split, "swiglu", R, False, 0, True, True, True, True, True, ap)
    torch.cuda.synchronize()
    dof_y, sof_y = oracle.expert_col_offsets(split, wl.width, R)
    dof_x, sof_x = oracle.expert_col_offsets(split, wl.w_in, R)
    offs = np.concatenate([[0], np.cumsum(split)]).astype(np.int64)
    for e in _sample_of(split):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            assert dof_x[e + 1] == dof_x[e] and dof_y[e + 1] == dof_y[e]
            continue
        se = [hi - lo]
        xs, ps, dys = host(x[lo:hi]), host(p[lo:hi]), host(dy[lo:hi])
        y = oracle.act_fwd_rows(xs, ps, ACT_ID["swiglu"], prm)
        dx, dpr = oracle.act_bwd_rows(dys, xs, ps, ACT_ID["swiglu"], prm)
        gy = host(g["y"][lo:hi])
        assert_bf16(gy, y, False, f"moe e{e} Y")
        gq = {"row_data": host(g["row_data"].view(-1, wl.width)[lo:hi]),
              "row_scale": host(g["row_scale"].view(-1, wl.width // 32)[lo:hi])}
        _compare_quant(gq, y, se, R, False, 0, False, True, False, f"moe e{e} fwd", g_vals=gy)
        gdx = host(b["dx"][lo:hi])
        assert_bf16(gdx, dx, False, f"moe e{e} dX")
        assert_dprobs(host(b["dprobs"][lo:hi]), dpr, dys, xs, ps, "swiglu", False, f"moe e{e} dprobs")
        gx = {"row_data": host(b["row_data"].view(-1, wl.w_in)[lo:hi]),
              "row_scale": host(b["row_scale"].view(-1, wl.w_in // 32)[lo:hi]),
              "col_data": host(b["col_data"][dof_x[e]:dof_x[e + 1]]),
              "col_scale": host(b["col_scale"][sof_x[e]:sof_x[e + 1]])}
        _compare_quant(gx, dx, se, R, False, 0, False, True, True, f"moe e{e} bwd dX", g_vals=gdx)
        gr = {"col_data": host(b["y_col_data"][dof_y[e]:dof_y[e + 1]]),
              "col_scale": host(b["y_col_scale"][sof_y[e]:sof_y[e + 1]])}
        _compare_quant(gr, y, se, R, False, 0, False, False, True, f"moe e{e} regen Y", g_vals=gy)


@pytest.mark.parametrize("act", ["swiglu", "clamped_swiglu"])
def test_full_size_swiglu_mxfp8_sampled_experts(act):
    """SwiGLU / clamped SwiGLU MXFP8 workload at its full size (32768 rows x
    2 x 2048, 16 experts with one empty): one launch with several items per
    CTA, so the multi-item pipeline runs on both GLU forms."""
    split, _ = inputs.make_split(inputs.WORKLOADS["swiglu_mxfp8"], np.random.default_rng(0))
    assert (np.asarray(split) == 0).any()
    _check_full_size("swiglu_mxfp8", act, oracle.MXFP8, False, _sample_of(split))
