"""Helpers for the GPU parity tests: device copies, GPU runs through the C ABI,
and the comparison rules.

Exact paths (SReLU, identity) are compared bit for bit.  The paths with a
library transcendental (tanh / SiLU / erfc / sigmoid) are held to:
  * BF16 values (Y, dX) within 2 BF16 ULP of the oracle's;
  * quantized copies bit-exact against the oracle's quantization of the
    GPU's own BF16 values (the quantizer has no transcendental in it);
  * against the oracle's quantization of its own values: per-expert NVFP4
    amax within the shift that 2 ULP of BF16 can cause (rowwise: 2 ULP;
    columnwise with the RHT: the bound of ``rht_amax_shift_bound``), experts
    whose amax moved re-encoded with the GPU's amax and counted; block scale
    codes equal except adjacent codes on at most 1e-3 of the blocks; element
    codes one step apart on at most 1e-3 of the elements;
  * dprobs within the bound of ``dprobs_bound`` (derived from the
    activation's error bound and the summation tree).
"""
import numpy as np
import torch

import oracle
from nvfp4_quantization_grouped_gb300 import gsa, inputs

ACT_ID = {"srelu": 0, "tanh_srelu": 1, "swiglu": 2, "clamped_swiglu": 3, "gelu": 4, "sigmoid": 5, "identity": 6}
GLU_NAMES = ("swiglu", "clamped_swiglu")
EXACT_ACTS = ("srelu", "identity")

U = 2.0 ** -24   # unit roundoff of binary32

# Bound on |act_gpu - act_oracle| / |act_oracle| for the FP32 activation value
# (the dprobs factor).  From the library error bounds -- CUDA's tanhf within 2
# ulp, erfcf within 4 ulp; the C library's tanhf within 2, expf within 1, erfcf
# within 3; the GPU polynomial tanh within 1.6 -- and one rounding (at most u on
# each side) per FP32 operation after the library call.
ACT_REL_ERR = {
    "srelu": 0.0, "identity": 0.0,
    "tanh_srelu": 20 * U,       # t within 4 ulp (8u); t*t: 16u + 2u; s^2 * tt: + 2u
    "gelu": 16 * U,             # erfc within 7 ulp (14u); (x / 2) * c: 16u
}


def act_rel_err(act, a, prm=None):
    """ACT_REL_ERR, per element for the sigmoid-based activations, whose GPU
    sigmoid (sigmoid_fast) is within (12 + 2 |z|) u of the exact one at
    argument z (tests/test_gpu_fast_exp.py, every BF16 z) and whose FP32
    oracle 1 / (1 + expf(-z)) is within 4u (expf 2u, the sum and the divide u
    each): sigmoid (16 + 2 |z|) u; SwiGLU z = a, plus a * sg and * b (u on
    each side): (20 + 2 |z|) u; clamped SwiGLU the same with z = alpha min(a, L),
    formed alike on both sides.  a is the gate (FP32 array)."""
    if act in ACT_REL_ERR:
        return ACT_REL_ERR[act]
    z = np.abs(np.asarray(a, np.float64))
    if act == "clamped_swiglu":
        s, limit, alpha, off = prm or params_tuple(act)
        z = np.abs(np.float32(alpha) * np.minimum(np.asarray(a, np.float32), np.float32(limit)).astype(np.float32)
                   ).astype(np.float64)
    base = 16.0 if act == "sigmoid" else 20.0
    return (base + 2.0 * z) * U


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
    ia = np.asarray(a).astype(np.int32)
    ib = np.asarray(b).astype(np.int32)
    oa = np.where(ia & 0x8000, 0x8000 - ia, ia)
    ob = np.where(ib & 0x8000, 0x8000 - ib, ib)
    return np.abs(oa - ob)


def bf16_bits(v):
    """BF16 bit pattern of float32 values that are exactly BF16."""
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_shift_bound(h, k=2):
    """Largest |v' - v| over BF16 values v' within k ULP of each BF16 value
    v (bit patterns h): the step k places away from zero, the larger one."""
    mag = (np.asarray(h, np.uint16) & 0x7FFF).astype(np.int64)
    up = np.minimum(mag + k, 0x7F7F).astype(np.uint16)
    return oracle.bf16_to_f32(up).astype(np.float64) - oracle.bf16_to_f32(mag.astype(np.uint16)).astype(np.float64)


def rht_amax_shift_bound(h):
    """Bound on how far one expert's columnwise NVFP4 amax after the 16-point
    RHT can move when each BF16 value v (bit patterns h, [Me, W]) moves by up
    to 2 ULP: an output w = (1/4) sum_j d_j H_ij v_j moves by at most
    (1/4) sum_j |dv_j|, plus the two sides' FP32 rounding in the butterflies
    (four levels, at most 4u of (1/4) sum |v| each); the maximum over blocks
    moves by at most the largest such block bound."""
    h = np.asarray(h, np.uint16)
    me, w = h.shape
    mp = (me + 15) // 16 * 16
    dv = np.zeros((mp, w))
    av = np.zeros((mp, w))
    dv[:me] = bf16_shift_bound(h)
    av[:me] = np.abs(oracle.bf16_to_f32(h).astype(np.float64))
    sd = dv.reshape(mp // 16, 16, w).sum(axis=1)
    sa = av.reshape(mp // 16, 16, w).sum(axis=1)
    return float(np.max(0.25 * sd + 2 * 4 * U * 0.25 * sa, initial=0.0)) * (1 + 2.0 ** -10)


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
        assert d.max(initial=0) <= 2, f"{what}: max BF16 ULP distance {d.max()}"


def assert_quant(got_data, got_scale, ref_data, ref_scale, recipe, exact, what, block):
    """Quantized copy: bit-exact, or within the tolerance of the approximate
    paths (taken with both sides on the same per-expert tensor scale)."""
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
    # a block amax moved by the 2-ULP bound shifts an E8M0 exponent or a
    # (positive, monotone) E4M3 scale code by at most one place
    step = np.abs(gs[sdiff].astype(int) - rs[sdiff].astype(int))
    assert np.all(step <= 1), f"{what}: scale codes {step.max(initial=0)} places apart"
    blk_ok = np.repeat(~sdiff, block)[: gc.size]
    di = np.abs(code_index(gc, recipe) - code_index(rc, recipe))
    assert di[blk_ok].max(initial=0) <= 1, f"{what}: code off by {di[blk_ok].max()} steps"
    assert (di[blk_ok] > 0).mean() <= 1e-3, f"{what}: {(di[blk_ok] > 0).mean():.2e} codes differ"


def _r5_node_sum(t):
    """Sum over every addition of the R5 order (serial 32-blocks from 0, then
    the pairwise tree) of |its FP32 result|, per row; t [n, W] float32."""
    n, w = t.shape
    nb = (w + 31) // 32
    sums = np.zeros((n, nb), np.float32)
    acc_abs = np.zeros(n)
    for b in range(nb):
        s = np.zeros(n, np.float32)
        for k in range(b * 32, min(w, b * 32 + 32)):
            s = (s + t[:, k]).astype(np.float32)
            if k > b * 32:   # 0 + t is exact
                acc_abs += np.abs(s.astype(np.float64))
        sums[:, b] = s
    m = nb
    while m > 1:
        half = m // 2
        nxt = np.empty((n, half + (m & 1)), np.float32)
        nxt[:, :half] = (sums[:, 0:2 * half:2] + sums[:, 1:2 * half:2]).astype(np.float32)
        acc_abs += np.abs(nxt[:, :half].astype(np.float64)).sum(axis=1)
        if m & 1:
            nxt[:, half] = sums[:, m - 1]
        sums, m = nxt, half + (m & 1)
    return acc_abs


def dprobs_bound(dy, x, act, prm=None):
    """Per-row bound on |dprobs_gpu - dprobs_oracle| when both sum the same
    order and the activation values differ by at most ACT_REL_ERR:
    each term dY * act moves by at most (eps + 2u) |term|, and each addition
    of the tree by at most u (|result| on each side), so
      |D| <= (eps + 2u) sum_j |t_j| + 2u sum_nodes |s_node|  (+ 2^-10 slack
    for the second-order terms)."""
    glu = act in GLU_NAMES
    w = dy.shape[1]
    xf = oracle.bf16_to_f32(x)
    val, _, _ = oracle.act_grad(ACT_ID[act], xf[:, :w], xf[:, w:] if glu else None, prm or params_tuple(act))
    t = (oracle.bf16_to_f32(dy) * val).astype(np.float32)
    eps = act_rel_err(act, xf[:, :w], prm)
    at = np.abs(t.astype(np.float64))
    sum_t = at.sum(axis=1)
    return (((eps + 2 * U) * at).sum(axis=1) + 2 * U * _r5_node_sum(t)) * (1 + 2.0 ** -10), sum_t


def assert_dprobs(got, ref, dy, x, p, act, exact, what, prm=None):
    if exact:
        bad = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
        assert bad.size == 0, f"{what}: {bad.size} dprobs mismatches, first {bad[:5]}"
        return
    bound, sum_t = dprobs_bound(dy, x, act, prm)
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    worst = np.max(err / (U * sum_t + 1e-300), initial=0.0)
    assert np.all(err <= bound + 1e-38), f"{what}: dprobs outside the derived bound (worst {worst:.1f} u sum|t|)"
