"""Host-side checks of the benchmark's byte accounting against the per-element
formulas (NVFP4: q = 1/2 + 1/16 bytes per quantized element, MXFP8: 1 + 1/32),
computed here independently of the library's layout query."""
import numpy as np

import bench
from nvfp4_quantization_grouped_gb300 import inputs


def _q_bytes(split, width, recipe):
    """Data + scale bytes of one quantized copy, rowwise and columnwise."""
    b = 16 if recipe == inputs.RECIPE_NVFP4 else 32
    per = (0.5 + 1 / 16) if recipe == inputs.RECIPE_NVFP4 else (1 + 1 / 32)
    M = int(np.sum(split))
    Mp = int(sum((int(m) + b - 1) // b * b for m in split))
    amax = 4 * len(split) if recipe == inputs.RECIPE_NVFP4 else 0
    return M * width * per + amax, Mp * width * per + amax


def test_algorithmic_bytes_match_the_per_element_formulas():
    for name in ("nvfp4_rht", "swiglu_mxfp8", "tanh_srelu_mxfp8_recompute", "tiny_srelu_mxfp8"):
        wl = inputs.WORKLOADS[name]
        rng = np.random.default_rng(0)
        split, _ = inputs.make_split(wl, rng)
        M = int(split.sum())
        fb, bb = bench.algorithmic_bytes(wl, list(split), M)
        y_row, y_col = _q_bytes(split, wl.width, wl.recipe)
        dx_row, dx_col = _q_bytes(split, wl.w_in, wl.recipe)
        fwd = M * wl.w_in * 2 + 4 * M + y_row + (0 if wl.recompute else y_col)
        bwd = (M * wl.w_in * 2 + M * wl.width * 2 + 4 * M) + (M * wl.w_in * 2 + 4 * M) + dx_row + dx_col \
            + (y_col if wl.recompute else 0)
        assert fb == fwd and bb == bwd, name


def test_two_step_path_moves_the_intermediate_twice():
    wl = inputs.WORKLOADS["nvfp4_rht"]
    split, _ = inputs.make_split(wl, np.random.default_rng(0))
    M = int(split.sum())
    fb, bb = bench.algorithmic_bytes(wl, list(split), M)
    (fa, fq), (ba, bq) = bench.two_step_bytes(wl, list(split), M)
    assert fa + fq - fb == 2 * M * wl.width * 2        # Y written, then read back
    assert ba + bq - bb == M * wl.w_in * 2             # dense dX read back (it is written either way)


def test_headline_workload_bytes():
    # the figures the benchmark reports per launch on the NVFP4 workload
    wl = inputs.WORKLOADS["nvfp4_rht"]
    split, _ = inputs.make_split(wl, np.random.default_rng(0))
    assert bench.algorithmic_bytes(wl, list(split), int(split.sum())) == (419932416, 957065472)


def test_reference_arm_counts_the_same_bytes_without_the_library():
    # the reference arm counts bytes with the oracle's layout; it must agree with the library's query
    for name in ("nvfp4_rht", "swiglu_mxfp8", "tanh_srelu_mxfp8_recompute", "moe_swiglu_mxfp8_recompute"):
        wl = inputs.WORKLOADS[name]
        split, _ = inputs.make_split(wl, np.random.default_rng(0))
        M = int(split.sum())
        assert bench.algorithmic_bytes(wl, list(split), M) == \
            bench.algorithmic_bytes(wl, list(split), M, bench.layout_bytes_oracle), name
