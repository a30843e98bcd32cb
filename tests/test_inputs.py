"""The seeded input generator: deterministic, shaped like each workload."""
import numpy as np
import pytest

from nvfp4_quantization_grouped_gb300 import inputs


def test_splitmix64_reference_values():
    # splitmix64 started from 0: first output of Vigna's reference generator
    assert inputs.splitmix64(0) == 0xE220A8397B1DCDAF
    assert inputs.rht_mask_from_seed(0) == 0xCDAF


@pytest.mark.parametrize("name", ["tiny_srelu_mxfp8", "tanh_srelu_mxfp8_recompute", "swiglu_mxfp8",
                                  "nvfp4_rht"])
def test_workload_shapes_and_determinism(name):
    wl = inputs.WORKLOADS[name]
    rows = None if wl.rows <= 8192 else 4096
    a = inputs.make_problem(name, 0, rows=rows)
    b = inputs.make_problem(name, 0, rows=rows)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.split_sizes, b.split_sizes)
    assert a.x.shape == (a.rows, wl.w_in) and a.dy.shape == (a.rows, wl.width)
    assert a.probs.shape == (a.rows,) and a.probs.dtype == np.float32
    assert len(a.split_sizes) == wl.experts and np.all(a.split_sizes >= 0)
    if rows is None:
        assert a.rows == wl.rows


def test_full_split_sizes():
    for name in ["swiglu_mxfp8", "nvfp4_rht"]:
        wl = inputs.WORKLOADS[name]
        rng = np.random.default_rng(0)
        split, _ = inputs.make_split(wl, rng)
        assert split.sum() == wl.rows and len(split) == wl.experts
    split, _ = inputs.make_split(inputs.WORKLOADS["swiglu_mxfp8"], np.random.default_rng(0))
    assert (split == 0).sum() >= 1


def test_topk_routing_small():
    rng = np.random.default_rng(0)
    split, probs = inputs.topk_routing(rng, 512, 128, 8, 1.1, n_empty=4)
    assert split.sum() == 512 * 8 and np.all(split[-4:] == 0)
    assert probs.shape == (4096,) and np.all((probs > 0) & (probs < 1))
