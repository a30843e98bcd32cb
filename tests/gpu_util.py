"""Helpers for the GPU parity tests: device copies, GPU runs through the C ABI,
and the comparison rules (bit-exact, or the tolerance of the tanh / SiLU
paths: BF16 within 2 ULP; quantized codes one step apart on at most 1e-3 of
the elements; block scales equal except where the block amax moved)."""
import numpy as np
import torch

import oracle
from nvfp4_quantization_grouped_gb300 import gsa, inputs

ACT_ID = {"srelu": 0, "tanh_srelu": 1, "swiglu": 2, "clamped_swiglu": 3, "gelu": 4, "sigmoid": 5, "identity": 6}
GLU_NAMES = ("swiglu", "clamped_swiglu")
EXACT_ACTS = ("srelu", "identity")


def params_tuple(act):
    return (4.0, 7.0, 1.702, 1.0)


def dev_bf16(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def gpu_fwd(x, p, split, act, recipe, rht=False, mask=0, rowwise=True, columnwise=True, want_y=True, prm=None):
    out = gsa.fwd(dev_bf16(x), None if p is None else dev_f32(p), list(split), act, recipe, rht, mask, rowwise,
                  columnwise, want_y, gsa.ActParams(*(prm or params_tuple(act))))
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items() if k != "_info"}


def gpu_bwd(dy, x, p, split, act, recipe, rht=False, mask=0, rowwise=True, columnwise=True, regen=False,
            want_dx=True, want_dprobs=True, prm=None):
    out = gsa.bwd(dev_bf16(dy), dev_bf16(x), dev_f32(p), list(split), act, recipe, rht, mask, want_dx, rowwise,
                  columnwise, want_dprobs, regen, gsa.ActParams(*(prm or params_tuple(act))))
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items() if not k.endswith("_info")}


def bf16_ulp_diff(a, b):
    """Distance in BF16 units in the last place (sign-aware ordering)."""
    ia = a.astype(np.int32)
    ib = b.astype(np.int32)
    oa = np.where(ia & 0x8000, 0x8000 - ia, ia)
    ob = np.where(ib & 0x8000, 0x8000 - ib, ib)
    return np.abs(oa - ob)


def code_index(codes, recipe):
    """Signed position of each code on the ordered value line."""
    c = codes.astype(np.int32)
    if recipe == oracle.MXFP8:
        mag, neg = c & 0x7F, (c & 0x80) != 0
    else:
        mag, neg = c & 0x7, (c & 0x8) != 0
    return np.where(neg, -mag, mag)


def unpack_fp4(data):
    d = data.astype(np.uint8)
    return np.stack([d & 0xF, d >> 4], axis=-1).reshape(*d.shape[:-1], d.shape[-1] * 2) if d.ndim > 1 else \
        np.stack([d & 0xF, d >> 4], axis=-1).reshape(-1)


def assert_bf16(got, ref, exact, what):
    assert got.shape == ref.shape, what
    if exact:
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, f"{what}: {bad.size} BF16 mismatches, first at {bad[:5]}"
    else:
        d = bf16_ulp_diff(got, ref)
        assert d.max() <= 2, f"{what}: max BF16 ULP distance {d.max()}"


def assert_quant(got_data, got_scale, ref_data, ref_scale, recipe, exact, what, block):
    """Quantized copy: bit-exact, or within the tolerance of the approximate paths."""
    gd, rd = got_data.reshape(-1), ref_data.reshape(-1)
    gs, rs = got_scale.reshape(-1), ref_scale.reshape(-1)
    assert gd.size == rd.size and gs.size == rs.size, what
    if exact:
        bs = np.flatnonzero(gs != rs)
        assert bs.size == 0, f"{what}: {bs.size} scale mismatches, first {bs[:5]}"
        bd = np.flatnonzero(gd != rd)
        assert bd.size == 0, f"{what}: {bd.size} data-byte mismatches, first {bd[:5]}"
        return
    if recipe == oracle.NVFP4:
        gc, rc = unpack_fp4(gd), unpack_fp4(rd)
    else:
        gc, rc = gd, rd
    sdiff = gs != rs
    assert sdiff.mean() <= 1e-3, f"{what}: {sdiff.mean():.2e} of block scales differ"
    if recipe == oracle.MXFP8:   # E8M0: a moved amax shifts the exponent by one
        assert np.all(np.abs(gs[sdiff].astype(int) - rs[sdiff].astype(int)) <= 1), what
    blk_ok = np.repeat(~sdiff, block)[: gc.size]
    di = np.abs(code_index(gc, recipe) - code_index(rc, recipe))
    assert di[blk_ok].max(initial=0) <= 1, f"{what}: code off by {di[blk_ok].max()} steps"
    assert (di[blk_ok] > 0).mean() <= 1e-3, f"{what}: {(di[blk_ok] > 0).mean():.2e} codes differ"


def assert_dprobs(got, ref, dy, x, p, act, exact, what, prm=None):
    if exact:
        bad = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
        assert bad.size == 0, f"{what}: {bad.size} dprobs mismatches, first {bad[:5]}"
        return
    # bound: 64 * 2^-24 * sum |dY * act|, from the binary32 activation error of
    # the library math routines (a few ULP) plus the common summation tree
    glu = act in GLU_NAMES
    w = dy.shape[1]
    xf = oracle.bf16_to_f32(x)
    val, _, _ = oracle.act_grad(ACT_ID[act], xf[:, :w], xf[:, w:] if glu else None, prm or params_tuple(act))
    mag = np.abs(oracle.bf16_to_f32(dy).astype(np.float64) * val.astype(np.float64)).sum(axis=1)
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert np.all(err <= 64 * 2.0 ** -24 * mag + 1e-30), f"{what}: dprobs off by {np.max(err / (mag + 1e-30)):.2e} rel"
