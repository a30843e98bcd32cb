"""GPU parity on seeded random configurations.

Each case draws, from its own seed, the activation, the recipe, whether the
NVFP4 columnwise copy takes the RHT (and its sign mask), the width, the expert
count and a ragged split (empty experts, single rows, sizes around the
128-row band and 16/32-row block boundaries), the spread of X, the sign of the
router scale p, which quantized copies are requested, whether the backward
regenerates Y's columnwise copy, and the activation's parameter (TanhSReLU's
bound s, clamped SwiGLU's limit).  Forward and backward go through the C ABI
and are held to the same rules as the workload tests (bit for bit on the
transcendental-free paths, the stated tolerance elsewhere).

The widths include 1024 and 2048 columns so that NVFP4 amax items of 8, 16 and
32 tiles, encode items of 8 tiles, and slab-split dprobs all occur.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import ACT_ID, GLU_NAMES
from nvfp4_quantization_grouped_gb300 import inputs

from test_gpu_parity import run_bwd_case, run_fwd_case

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

N_CASES = 160
MAX_ELEMS = 400_000   # rows x output width per case, so the oracle stays quick


def _split(rng, n_experts, width):
    cap = max(1, MAX_ELEMS // width)
    kinds = rng.integers(0, 5, n_experts)
    sizes = []
    for k in kinds:
        if k == 0:
            sizes.append(0)
        elif k == 1:
            sizes.append(int(rng.integers(1, 34)))
        elif k == 2:   # around a band or block boundary
            base = int(rng.choice([16, 32, 64, 128, 256]))
            sizes.append(max(0, base + int(rng.integers(-2, 3))))
        else:
            sizes.append(int(rng.integers(1, 700)))
    sizes = np.asarray(sizes, np.int64)
    while sizes.sum() > cap:
        i = int(np.argmax(sizes))
        sizes[i] //= 2
    if sizes.sum() == 0:
        sizes[int(rng.integers(0, n_experts))] = int(rng.integers(1, min(cap, 300) + 1))
    return [int(v) for v in sizes]


def _case(i):
    rng = np.random.default_rng(7_000 + i)
    acts = list(ACT_ID)
    act = acts[int(rng.integers(0, len(acts)))]
    recipe = oracle.NVFP4 if rng.random() < 0.6 else oracle.MXFP8
    width = int(rng.choice([64, 192, 320, 1024, 2048]))
    n_experts = int(rng.integers(1, 25))
    split = _split(rng, n_experts, width)
    rht = recipe == oracle.NVFP4 and rng.random() < 0.7
    mask = int(rng.integers(0, 1 << 16))
    x_sigma = float(rng.choice([0.3, 1.0, 3.0, 8.0]))
    signed_p = rng.random() < 0.25
    outs = [(True, True), (True, False), (False, True)][int(rng.choice([0, 0, 0, 1, 2]))]
    regen = bool(rng.random() < 0.5)
    s = float(rng.choice([4.0, 0.75, 2.5, 8.0]))
    limit = float(rng.choice([7.0, 0.5, 3.0]))
    return dict(act=act, recipe=recipe, width=width, split=split, rht=rht, mask=mask, x_sigma=x_sigma,
                signed_p=signed_p, outs=outs, regen=regen, prm=(s, limit, 1.702, 1.0), seed=7_000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(i):
    c = _case(i)
    rng = np.random.default_rng(c["seed"] + 1)
    glu = c["act"] in GLU_NAMES
    split, x, p, dy = inputs.random_problem(rng, c["split"], c["width"], glu, x_sigma=c["x_sigma"])
    if c["signed_p"]:
        p = (2.0 * p - 1.0).astype(np.float32)
        p[rng.random(p.size) < 0.05] = 0.0
    rowwise, columnwise = c["outs"]
    run_fwd_case(split, x, p, c["act"], c["recipe"], c["rht"], c["mask"], rowwise, columnwise, prm=c["prm"])
    run_bwd_case(split, x, p, dy, c["act"], c["recipe"], c["rht"], c["mask"], rowwise, columnwise, c["regen"],
                 prm=c["prm"])


def test_cases_cover_the_item_shapes():
    """The drawn cases include every activation, both recipes, the RHT, the
    widths whose NVFP4 items span several tiles, empty experts and signed p."""
    cs = [_case(i) for i in range(N_CASES)]
    assert {c["act"] for c in cs} == set(ACT_ID)
    assert {c["recipe"] for c in cs} == {oracle.MXFP8, oracle.NVFP4}
    assert any(c["rht"] for c in cs)
    assert any(c["recipe"] == oracle.NVFP4 and c["width"] == 2048 for c in cs)
    assert any(c["recipe"] == oracle.NVFP4 and c["width"] == 1024 for c in cs)
    assert any(0 in c["split"] for c in cs)
    assert any(c["signed_p"] for c in cs)
    assert any(c["regen"] for c in cs)


@pytest.mark.parametrize("i", range(0, N_CASES, 4))
def test_random_configuration_graph_safe(i):
    """The graph-safe calls (split on the device, schedule built by the plan
    kernel) give every output of the host-split calls bit for bit, on the
    same random configurations: widths whose NVFP4 amax and encode items
    differ in size included."""
    from nvfp4_quantization_grouped_gb300 import gsa
    from gpu_util import dev_bf16, dev_f32, host
    from test_graph_safe import _compare, _split_dev

    c = _case(i)
    rng = np.random.default_rng(c["seed"] + 1)
    glu = c["act"] in GLU_NAMES
    split, x, p, dy = inputs.random_problem(rng, c["split"], c["width"], glu, x_sigma=c["x_sigma"])
    split = [int(v) for v in split]
    rowwise, columnwise = c["outs"]
    prm = gsa.ActParams(*c["prm"])
    xd, pd, dyd, sd = dev_bf16(x), dev_f32(p), dev_bf16(dy), _split_dev(split)
    args = (c["act"], c["recipe"], c["rht"], c["mask"])
    hf = gsa.fwd(xd, pd, split, *args, rowwise, columnwise, True, prm)
    gf = gsa.fwd_graph_safe(xd, pd, sd, *args, rowwise, columnwise, True, prm)
    hb = gsa.bwd(dyd, xd, pd, split, *args, True, rowwise, columnwise, True, c["regen"], prm)
    gb = gsa.bwd_graph_safe(dyd, xd, pd, sd, *args, True, rowwise, columnwise, True, c["regen"], prm)
    torch.cuda.synchronize()
    _compare(gf, hf, f"case {i} fwd")
    _compare(gb, hb, f"case {i} bwd")
    b = 32 if c["recipe"] == oracle.MXFP8 else 16
    pad = np.concatenate([[0], np.cumsum([(m + b - 1) // b * b for m in split])]).astype(np.int64)
    assert np.array_equal(host(gf["pad"]), pad)
