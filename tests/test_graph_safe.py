"""Graph-safe calls (split_sizes on the device) against the host-split calls.

The grouped-linear fusion page names a graph-safe fuser path: the forward
runs under CUDA-graph capture, where the host cannot read the split.  The
graph-safe calls build the schedule on the device, so one captured graph
serves every split of the same row count.  Checked here: bitwise equality
with the host-split calls (all outputs, padded row offsets), capture once and
replay after changing the split in place, and the rejection of an invalid
device split.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import ACT_ID, GLU_NAMES, dev_bf16, dev_f32, host, params_tuple
from nvfp4_quantization_grouped_gb300 import gsa, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

MASK = 0x3C5A
RECIPES = [oracle.MXFP8, oracle.NVFP4]
QKEYS = ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col")


def _split_dev(split):
    return torch.tensor([int(s) for s in split], dtype=torch.int64, device="cuda")


def _host_pad(split, recipe):
    b = 32 if recipe == oracle.MXFP8 else 16
    return np.concatenate([[0], np.cumsum([(int(m) + b - 1) // b * b for m in split])]).astype(np.int64)


def _compare(dev_out, host_out, what):
    """Every output of the host-split call equals the graph-safe one (whose
    columnwise buffers are longer: they are sized for any split)."""
    for k, v in host_out.items():
        if k.endswith("_info") or k == "pad":
            continue
        a = host(v).view(np.uint8).reshape(-1)
        b = host(dev_out[k]).view(np.uint8).reshape(-1)
        assert b.size >= a.size, f"{what} {k} size"
        assert np.array_equal(b[:a.size], a), f"{what} {k}"


@pytest.mark.parametrize("recipe", RECIPES)
@pytest.mark.parametrize("act", ["srelu", "tanh_srelu", "swiglu", "gelu"])
def test_graph_safe_equals_host_split(act, recipe):
    rng = np.random.default_rng(900 + ACT_ID[act] + 10 * recipe)
    split, x, p, dy = inputs.random_problem(rng, [0, 300, 17, 0, 129, 513, 1], 256, act in GLU_NAMES)
    split = [int(s) for s in split]
    rht = recipe == oracle.NVFP4
    prm = gsa.ActParams(*params_tuple(act))
    xd, pd, dyd, sd = dev_bf16(x), dev_f32(p), dev_bf16(dy), _split_dev(split)
    hf = gsa.fwd(xd, pd, split, act, recipe, rht, MASK, True, True, True, prm)
    gf = gsa.fwd_graph_safe(xd, pd, sd, act, recipe, rht, MASK, True, True, True, prm)
    hb = gsa.bwd(dyd, xd, pd, split, act, recipe, rht, MASK, True, True, True, True, True, prm)
    gb = gsa.bwd_graph_safe(dyd, xd, pd, sd, act, recipe, rht, MASK, True, True, True, True, True, prm)
    torch.cuda.synchronize()
    _compare(gf, hf, f"{act} fwd")
    _compare(gb, hb, f"{act} bwd")
    assert np.array_equal(host(gf["pad"]), _host_pad(split, recipe))
    assert np.array_equal(host(gb["pad"]), _host_pad(split, recipe))


def test_captured_graph_replays_for_new_splits():
    """One CUDA graph of forward + backward, replayed for three splits of the
    same rows (one with empty experts): each replay equals the host-split calls."""
    recipe, act = oracle.NVFP4, "tanh_srelu"
    rng = np.random.default_rng(77)
    M, W = 2048, 512
    splits = [[512, 512, 512, 512], [0, 2000, 0, 48], [1, 1, 1, 2045]]
    _, x, p, dy = inputs.random_problem(rng, [M], W, False)
    prm = gsa.ActParams(*params_tuple(act))
    xd, pd, dyd = dev_bf16(x), dev_f32(p), dev_bf16(dy)
    sd = _split_dev(splits[0])
    E = len(splits[0])
    ws_f = gsa.GraphSafeWorkspace(E, M, W, ACT_ID[act], recipe, xd.device)
    ws_b = gsa.GraphSafeWorkspace(E, M, W, ACT_ID[act], recipe, xd.device)
    # first (eager) calls allocate the outputs and configure the kernels
    fo = gsa.fwd_graph_safe(xd, pd, sd, act, recipe, True, MASK, True, True, True, prm, ws_f)
    bo = gsa.bwd_graph_safe(dyd, xd, pd, sd, act, recipe, True, MASK, True, True, True, True, True, prm, ws_b)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gsa.fwd_graph_safe(xd, pd, sd, act, recipe, True, MASK, True, True, True, prm, ws_f, fo)
        gsa.bwd_graph_safe(dyd, xd, pd, sd, act, recipe, True, MASK, True, True, True, True, True, prm, ws_b, bo)
    for split in splits:
        sd.copy_(torch.tensor(split, dtype=torch.int64))
        for t in list(fo.values()) + list(bo.values()):
            if isinstance(t, torch.Tensor):
                t.fill_(0x5A) if t.dtype == torch.uint8 else t.zero_()
        g.replay()
        torch.cuda.synchronize()
        hf = gsa.fwd(xd, pd, split, act, recipe, True, MASK, True, True, True, prm)
        hb = gsa.bwd(dyd, xd, pd, split, act, recipe, True, MASK, True, True, True, True, True, prm)
        torch.cuda.synchronize()
        _compare(fo, hf, f"replay {split} fwd")
        _compare(bo, hb, f"replay {split} bwd")
        assert np.array_equal(host(fo["pad"]), _host_pad(split, recipe))
        assert ws_f.status() == 0 and ws_b.status() == 0


@pytest.mark.parametrize("bad", [[100, 100, 99], [300, -1, 1], [0, 0, 0], [301, 0, 0]])
def test_invalid_device_split_is_reported_and_not_processed(bad):
    rng = np.random.default_rng(5)
    _, x, p, _ = inputs.random_problem(rng, [300], 128, False)
    xd, pd = dev_bf16(x), dev_f32(p)
    sd = _split_dev(bad)
    ws = gsa.GraphSafeWorkspace(3, 300, 128, 0, oracle.NVFP4, xd.device)
    out = gsa.alloc_qtensor_bound(3, 300, 128, oracle.NVFP4, True, True, xd.device)
    for k, t in out.items():
        if isinstance(t, torch.Tensor):
            t.fill_(0x77) if t.dtype == torch.uint8 else t.fill_(5.0)
    out["pad"] = torch.full((4,), -9, dtype=torch.int64, device="cuda")
    gsa.fwd_graph_safe(xd, pd, sd, "srelu", oracle.NVFP4, True, MASK, True, True, False, None, ws, out)
    assert ws.status() == 1   # GSA_ERR_INVALID_ARG
    for k in ("row_data", "row_scale", "col_data", "col_scale"):
        assert torch.all(out[k] == 0x77), k
    assert torch.all(out["amax_row"] == 0) and torch.all(out["amax_col"] == 0)
    assert torch.all(out["pad"] == 0)


@pytest.mark.parametrize("name", ["nvfp4_rht", "swiglu_mxfp8"])
def test_full_size_graph_safe_equals_host_split(name):
    """At full size (the NVFP4 workload: 32 experts, 65536 x 2048, 530 bands,
    a lookahead of the whole persistent grid; the SwiGLU MXFP8 workload with an
    empty expert) the graph-safe calls, whose queues the plan kernel builds in
    parallel, give every output of the host-split calls bit for bit."""
    wl, split, M, x, p, dy = inputs.device_problem(name, torch.device("cuda"))
    sd = _split_dev(split)
    E = len(split)
    prm = gsa.ActParams(*params_tuple("tanh_srelu"))
    for act in wl.acts:
        ws = gsa.GraphSafeWorkspace(E, M, wl.w_in, ACT_ID[act], wl.recipe, x.device)
        hf = gsa.fwd(x, p, split, act, wl.recipe, wl.rht, MASK, True, not wl.recompute, False, prm)
        gf = gsa.fwd_graph_safe(x, p, sd, act, wl.recipe, wl.rht, MASK, True, not wl.recompute, False, prm, ws)
        torch.cuda.synchronize()
        _compare(gf, hf, f"{name} {act} fwd")
        del hf, gf
        hb = gsa.bwd(dy, x, p, split, act, wl.recipe, wl.rht, MASK, True, True, True, True, wl.recompute, prm)
        gb = gsa.bwd_graph_safe(dy, x, p, sd, act, wl.recipe, wl.rht, MASK, True, True, True, True, wl.recompute,
                                prm, ws)
        torch.cuda.synchronize()
        _compare(gb, hb, f"{name} {act} bwd")
        assert np.array_equal(host(gb["pad"]), _host_pad(split, wl.recipe))
        assert ws.status() == 0
        del hb, gb, ws
        torch.cuda.empty_cache()
