"""Pins for the CPU oracle: each checks it against something other than itself.

- library routines (torch's BF16 and FP8-E4M3 conversions, scipy's Hadamard),
- values printed on the pages (the E4M3 cast-error table of the
  "Preserve FP8 recompute state for inner autocast" page),
- hand-worked encodings from the format definitions (tests/golden/),
- closed forms and finite differences of the activations,
- brute force on tiny inputs and invariants (half-bin bound, H^2 = 16 I,
  columnwise == rowwise of the padded transpose, exact-sum error bounds).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import parse_num, read_golden
from nvfp4_quantization_grouped_gb300 import inputs

# ---------------------------------------------------------------- BF16


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),   # subnormals
        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1.00390625, 1.01171875], np.float32),
    ])
    # exact ties: low 16 bits == 0x8000
    ties = (rng.integers(0, 2**31, 5000, dtype=np.uint32) & 0xFFFF0000) | 0x8000
    v = np.concatenate([v, ties.view(np.float32)])
    v = v[np.isfinite(v)]
    ours = oracle.f32_to_bf16(v)
    ref = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(oracle.bf16_to_f32(ours),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------- E4M3

def _torch_e4m3(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_e4m3_decode_matches_torch():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    ours = oracle.e4m3_decode(codes)
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    exps = rng.uniform(-14, 8.8, 400000)
    v = (np.sign(rng.standard_normal(exps.size)) * 2.0 ** exps).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    assert np.array_equal(oracle.e4m3_encode(v), _torch_e4m3(v))


def test_e4m3_every_midpoint_matches_torch():
    codes = np.arange(0, 126, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float64)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)  # exact in f32
    probe = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                            -mids, vals.astype(np.float32)])
    assert np.array_equal(oracle.e4m3_encode(probe), _torch_e4m3(probe))


def test_e4m3_saturates_and_keeps_sign_of_zero():
    enc = oracle.e4m3_encode(np.array([448.0, 460.0, 1e30, -1e30, 0.0, -0.0], np.float32))
    assert list(enc) == [0x7E, 0x7E, 0x7E, 0xFE, 0x00, 0x80]


def test_e4m3_cast_error_table_from_page():
    """Reproduce the page's simulated per-tensor E4M3 cast+descale error."""
    rng = np.random.default_rng(0)
    base = rng.standard_normal(1 << 21).astype(np.float32)
    for sigma, at_one, at_ideal in [tuple(map(float, r)) for r in read_golden("e4m3_cast_error.txt")]:
        x = (base * np.float32(sigma)).astype(np.float32)
        q = _decode_table()[oracle.e4m3_encode(x)]
        err1 = 100 * math.sqrt(np.mean((q.astype(np.float64) - x) ** 2) / np.mean(x.astype(np.float64) ** 2))
        scale = np.float32(448.0 / np.abs(x).max())
        qi = _decode_table()[oracle.e4m3_encode(x * scale)] / scale
        erri = 100 * math.sqrt(np.mean((qi.astype(np.float64) - x) ** 2) / np.mean(x.astype(np.float64) ** 2))
        digits = 2 if at_one < 10 else 1
        assert round(err1, digits) == pytest.approx(at_one, abs=0.011 if digits == 2 else 0.11), (sigma, err1)
        assert round(erri, 2) == pytest.approx(at_ideal, abs=0.011), (sigma, erri)


_TABLE = None


def _decode_table():
    global _TABLE
    if _TABLE is None:
        t = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
        _TABLE = np.nan_to_num(t, nan=0.0).astype(np.float32)
    return _TABLE


# ---------------------------------------------------------------- E2M1

E2M1_VALUES = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def _brute_e2m1(v):
    """Nearest of the eight magnitudes by exhaustive distance, ties to even code."""
    out = []
    for x in np.asarray(v, dtype=np.float64):
        a = abs(x)
        if a >= 6:
            c = 7
        else:
            d = np.abs(E2M1_VALUES - a)
            best = np.flatnonzero(d == d.min())
            c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
        out.append(c | (8 if math.copysign(1.0, x) < 0 else 0))
    return np.array(out, dtype=np.uint8)


def test_e2m1_ties_golden():
    rows = read_golden("e2m1_ties.txt")
    v = np.array([float(r[0]) for r in rows], np.float32)
    exp = np.array([parse_num(r[1]) for r in rows], np.uint8)
    assert np.array_equal(oracle.e2m1_encode(v), exp)


def test_e2m1_brute_force():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(-8, 8, 20000), rng.standard_normal(5000) * 0.3,
                        np.arange(-7, 7.01, 0.125)]).astype(np.float32)
    assert np.array_equal(oracle.e2m1_encode(v), _brute_e2m1(v))
    dec = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert list(np.abs(dec[:8])) == list(E2M1_VALUES) and np.all(dec[9:] < 0)


# ---------------------------------------------------------- MXFP8 block

def test_mxfp8_hand_worked_block():
    rows = read_golden("mxfp8_block.txt")
    elems = [(float(r[0]), parse_num(r[1])) for r in rows[:4]]
    amaxes = [(float(r[0]), int(r[1])) for r in rows[4:]]
    v = np.zeros(32, np.float32)
    v[:4] = [e[0] for e in elems]
    codes, sc = oracle.mxfp8_block(v)
    assert sc == 119
    assert list(codes[:4]) == [e[1] for e in elems]
    for amax, code in amaxes:
        assert oracle.mx_scale_exp(amax) + 127 == code


def test_mxfp8_scale_exponent_is_smallest_without_saturation():
    rng = np.random.default_rng(4)
    for amax in np.concatenate([2.0 ** rng.uniform(-120, 120, 2000), [448 * 2.0 ** k for k in range(-20, 20)]]):
        a = np.float32(amax)
        e = oracle.mx_scale_exp(a)
        assert float(a) <= 448 * 2.0 ** e
        assert e == -127 or float(a) > 448 * 2.0 ** (e - 1)


# ---------------------------------------------------------- NVFP4 block

def test_nvfp4_hand_worked_block():
    rows = read_golden("nvfp4_block.txt")
    def numeric(r):
        return (r[0][0].isdigit() or r[0][0] == "-") and "," not in r[0]
    kv = {r[0]: r[1] for r in rows if not numeric(r) and "," not in r[0]}
    S = oracle.nvfp4_tensor_scale(float(kv["tensor_amax"]))
    assert S == float(kv["S_enc"])
    elems = [(float(r[0]), parse_num(r[1])) for r in rows if numeric(r)]
    v = np.zeros(16, np.float32)
    v[:4] = [e[0] for e in elems]
    codes, sc = oracle.nvfp4_block(v, S)
    assert sc == parse_num(kv["block_scale_code"])
    assert list(codes[:4]) == [e[1] for e in elems]
    pair = [r for r in rows if "," in r[0]][0]
    a, b = map(float, pair[0].split(","))
    pv = np.zeros(16, np.float32)
    pv[:2] = [a, b]
    c2, _ = oracle.nvfp4_block(pv, S)
    assert (int(c2[0]) | (int(c2[1]) << 4)) == parse_num(pair[1])


def test_nvfp4_tensor_scale_edge_cases():
    assert oracle.nvfp4_tensor_scale(0.0) == 1.0
    assert oracle.nvfp4_tensor_scale(1e-44) == np.finfo(np.float32).max
    assert oracle.nvfp4_tensor_scale(2688.0) == 1.0


def test_nvfp4_overflowing_multiplier_is_capped_like_the_tensor_scale():
    """Reading R17, worked by hand.  Expert amax 1e-44 gives S = FLT_MAX (the
    cap of R8).  A block of amax 2^-126 gets (2^-126 / 6) * S ~ 0.667 ->
    E4M3 0.6875 (code 0x33), and S / 0.6875 overflows: the multiplier is held
    at FLT_MAX = (2 - 2^-23) 2^127.  Then 2^-126 * r = 3.99999976 -> 4 (0x6),
    2^-130 * r just below the 0.25 tie -> 0 (0x0), -2^-131 * r -> -0 (0x8),
    and the zeros keep their signs (no 0 * inf)."""
    S = oracle.nvfp4_tensor_scale(1e-44)
    assert S == np.finfo(np.float32).max
    v = np.zeros(16, np.float32)
    v[0], v[1], v[3], v[4] = 2.0 ** -126, 2.0 ** -130, -0.0, -(2.0 ** -131)
    codes, sc = oracle.nvfp4_block(v, S)
    assert sc == 0x33
    assert np.float64(S) / 0.6875 > np.finfo(np.float32).max   # the FP32 quotient would overflow
    assert list(codes[:5]) == [0x6, 0x0, 0x0, 0x8, 0x8]
    assert all(c == 0 for c in codes[5:])


def test_nvfp4_row_packing_order():
    """Element 2k goes to the low nibble, 2k+1 to the high nibble."""
    v = np.zeros((1, 16), np.float32)
    v[0, 0], v[0, 1] = 6.0, 0.5          # with tensor amax 6 -> S = 448, sb = 448
    y = oracle.f32_to_bf16(v)
    data, scale = oracle.quant_rows(y, oracle.NVFP4, oracle.nvfp4_tensor_scale(6.0))
    assert data[0, 0] == (0x7 | (0x1 << 4))
    assert scale[0, 0] == 0x7E


# --------------------------------------------------- half-bin invariant

def _mx_dequant(codes, scale_code):
    return _decode_table()[codes].astype(np.float64) * 2.0 ** (scale_code - 127)


def test_mxfp8_half_bin_invariant():
    rng = np.random.default_rng(5)
    for _ in range(300):
        v = (rng.standard_normal(32) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        codes, sc = oracle.mxfp8_block(v)
        dq = _mx_dequant(codes, sc)
        # local bin width of E4M3 at |v| * 2^-e, times 2^e
        e = sc - 127
        t = np.abs(v.astype(np.float64)) * 2.0 ** (-e)
        ulp = np.where(t < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(t, 1e-300))) - 3))
        assert np.all(np.abs(dq - v) <= 0.5 * ulp * 2.0 ** e + 1e-300)


def test_nvfp4_half_bin_invariant():
    rng = np.random.default_rng(6)
    for _ in range(300):
        v = (rng.standard_normal(16) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        amax_t = float(np.abs(v).max()) * float(rng.uniform(1, 50))
        S = oracle.nvfp4_tensor_scale(amax_t)
        codes, sc = oracle.nvfp4_block(v, S)
        sbf = float(oracle.e4m3_decode(np.array([sc]))[0])
        if sbf == 0:
            assert np.all(codes & 7 == 0)
            continue
        r = np.float32(np.float32(S) / np.float32(sbf))
        t = np.abs(v * r).astype(np.float64)
        step = np.where(t < 2, 0.5, np.where(t < 4, 1.0, 2.0))
        deq = oracle.e2m1_decode(codes).astype(np.float64)
        err = np.abs(deq - (v * r).astype(np.float64))
        within = err <= 0.5 * step + 1e-12
        assert np.all(within | (t > 6))   # top-bin saturation beyond 6 excluded


# ---------------------------------------------------------------- RHT

def test_rht_matches_scipy_hadamard_and_is_involutive():
    from scipy.linalg import hadamard
    H = hadamard(16).astype(np.float64)
    rng = np.random.default_rng(7)
    for mask in [0, 0xFFFF, 0x1234, inputs.rht_mask_from_seed(0)]:
        d = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
        v = rng.integers(-64, 64, 16).astype(np.float32)          # exact in every order
        w = oracle.rht16(v, mask)
        assert np.array_equal(w.astype(np.float64), 0.25 * H @ (d * v))
        # inverse: (1/4) D H undoes (1/4) H D, since H H = 16 I
        back = 0.25 * d * (H @ w.astype(np.float64))
        assert np.allclose(back, v, atol=0)
        vv = rng.standard_normal(16).astype(np.float32)
        ww = oracle.rht16(vv, mask).astype(np.float64)
        assert abs(np.linalg.norm(ww) - np.linalg.norm(vv.astype(np.float64))) < 1e-5
    e0 = np.zeros(16, np.float32)
    e0[0] = 1.0
    assert np.all(oracle.rht16(e0, 0) == 0.25)


# ------------------------------------------------------- activations

S4 = (4.0, 0.0, 0.0, 0.0)
CLAMP = (0.0, 7.0, 1.702, 1.0)


def test_srelu_closed_form():
    x = np.linspace(-3, 3, 601).astype(np.float32)
    val, da, _ = oracle.act_grad(oracle.ACT_SRELU, x)
    r = np.maximum(x, 0)
    assert np.array_equal(val, r * r) and np.array_equal(da, 2 * r)


def test_tanh_srelu_bound_and_limits():
    x = np.concatenate([np.linspace(-5, 60, 5000), [1e3, 1e6]]).astype(np.float32)
    val, da, _ = oracle.act_grad(oracle.ACT_TANH_SRELU, x, None, S4)
    assert np.all(val <= 16.0) and np.all(val >= 0)
    assert val[-1] == 16.0
    small = np.float32(0.01)
    v, _, _ = oracle.act_grad(oracle.ACT_TANH_SRELU, np.array([small]), None, S4)
    assert v[0] == pytest.approx(float(small) ** 2 * (1 - 2 * 0.01 ** 2 / (3 * 16)), rel=1e-5)
    ref = 16.0 * np.tanh(np.maximum(x.astype(np.float64), 0) / 4.0) ** 2
    assert np.allclose(val, ref, rtol=1e-5, atol=1e-6)
    assert np.all(da[x <= 0] == 0)


def _fd(f, x, h):
    return (f(x + h) - f(x - h)) / (2 * h)


@pytest.mark.parametrize("act,prm", [(oracle.ACT_SRELU, S4), (oracle.ACT_TANH_SRELU, S4)])
def test_unary_derivative_by_finite_differences(act, prm):
    x = np.concatenate([np.linspace(-4, -0.05, 50), np.linspace(0.05, 8, 200)])
    def f(z):
        return oracle.act_grad(act, z.astype(np.float32), None, prm)[0].astype(np.float64)
    num = _fd(f, x, 1e-2)
    _, da, _ = oracle.act_grad(act, x.astype(np.float32), None, prm)
    exact = 2 * np.maximum(x, 0) if act == oracle.ACT_SRELU else \
        8 * np.tanh(np.maximum(x, 0) / 4) * (1 - np.tanh(np.maximum(x, 0) / 4) ** 2)
    assert np.allclose(da, exact, rtol=1e-5, atol=1e-6)
    assert np.allclose(da, num, rtol=2e-3, atol=2e-3)


@pytest.mark.parametrize("act,prm", [(oracle.ACT_SWIGLU, S4), (oracle.ACT_CLAMPED_SWIGLU, CLAMP)])
def test_glu_derivatives_by_finite_differences(act, prm):
    rng = np.random.default_rng(8)
    a = rng.uniform(-9, 9, 400)
    b = rng.uniform(-9, 9, 400)
    if act == oracle.ACT_CLAMPED_SWIGLU:  # stay away from the kinks at a = L, |b| = L
        keep = (np.abs(a - 7) > 0.05) & (np.abs(np.abs(b) - 7) > 0.05)
        a, b = a[keep], b[keep]
    val, da, db = oracle.act_grad(act, a.astype(np.float32), b.astype(np.float32), prm)
    fa = _fd(lambda z: oracle.act_grad(act, z.astype(np.float32), b.astype(np.float32), prm)[0].astype(np.float64), a, 1e-2)
    fb = _fd(lambda z: oracle.act_grad(act, a.astype(np.float32), z.astype(np.float32), prm)[0].astype(np.float64), b, 1e-2)
    assert np.allclose(da, fa, rtol=5e-3, atol=5e-3)
    assert np.allclose(db, fb, rtol=5e-3, atol=5e-3)
    # closed forms in float64
    if act == oracle.ACT_SWIGLU:
        sg = 1 / (1 + np.exp(-a))
        ref = a * sg * b
        ref_da = b * (sg + a * sg * (1 - sg))
        ref_db = a * sg
    else:
        L, al, off = 7.0, 1.702, 1.0
        ac = np.minimum(a, L)
        bc = np.clip(b, -L, L)
        sg = 1 / (1 + np.exp(-al * ac))
        ref = ac * sg * (bc + off)
        ref_da = np.where(a <= L, (bc + off) * (sg + al * ac * sg * (1 - sg)), 0)
        ref_db = np.where(np.abs(b) <= L, ac * sg, 0)
    assert np.allclose(val, ref, rtol=1e-5, atol=1e-5)
    assert np.allclose(da, ref_da, rtol=1e-5, atol=1e-5)
    assert np.allclose(db, ref_db, rtol=1e-5, atol=1e-5)


def test_clamped_swiglu_passes_gradient_at_the_limit():
    val, da, db = oracle.act_grad(oracle.ACT_CLAMPED_SWIGLU, np.array([7.0, 7.5], np.float32),
                                  np.array([7.0, 7.5], np.float32), CLAMP)
    assert da[0] != 0 and db[0] != 0 and da[1] == 0 and db[1] == 0


# Further unary activations (GeLU, sigmoid, identity).  Pins: standard-normal
# table values of Phi, the identity gelu(x) - gelu(-x) = x, the Mills-ratio
# asymptotic series of the lower tail, sigmoid's symmetry and exact points,
# and finite differences for the derivatives.

PHI_TABLE = {1.0: 0.8413447460685429, 2.0: 0.9772498680518208, 3.0: 0.9986501019683699,
             0.5: 0.6914624612740131, -1.0: 0.15865525393145707}


def _phi_lower_tail(x):
    """Phi(-x) for large x from the asymptotic series phi(x)/x (1 - 1/x^2 + 3/x^4 - 15/x^6 + 105/x^8)."""
    dens = math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    z = 1.0 / (x * x)
    return dens / x * (1 - z + 3 * z ** 2 - 15 * z ** 3 + 105 * z ** 4)


def test_gelu_table_values_odd_identity_and_tail():
    xs = np.array(sorted(PHI_TABLE), np.float32)
    val, da, _ = oracle.act_grad(oracle.ACT_GELU, xs)
    for x, v in zip(xs, val):
        assert v == pytest.approx(float(x) * PHI_TABLE[float(x)], rel=3e-7)
    v0, d0, _ = oracle.act_grad(oracle.ACT_GELU, np.array([0.0], np.float32))
    assert v0[0] == 0.0 and d0[0] == 0.5                      # gelu'(0) = Phi(0) = 1/2
    x = np.linspace(-6, 6, 1201).astype(np.float32)
    vp, _, _ = oracle.act_grad(oracle.ACT_GELU, x)
    vm, _, _ = oracle.act_grad(oracle.ACT_GELU, -x)
    assert np.all(np.abs((vp.astype(np.float64) - vm) - x) <= 4 * 2.0 ** -24 * np.maximum(np.abs(x), 1e-30))
    # lower tail: relative accuracy where 1 + erf would cancel completely
    for t in (6.0, 8.0, 10.0):
        v, _, _ = oracle.act_grad(oracle.ACT_GELU, np.array([-t], np.float32))
        assert v[0] == pytest.approx(-t * _phi_lower_tail(t), rel=2e-5)
    big, dbig, _ = oracle.act_grad(oracle.ACT_GELU, np.array([10.0, 30.0], np.float32))
    assert np.array_equal(big, [10.0, 30.0]) and np.array_equal(dbig, [1.0, 1.0])


def test_sigmoid_symmetry_exact_points_and_tail():
    v, d, _ = oracle.act_grad(oracle.ACT_SIGMOID, np.array([0.0, math.log(3.0)], np.float32))
    assert v[0] == 0.5 and d[0] == 0.25
    assert v[1] == pytest.approx(0.75, rel=3e-7)             # 1 / (1 + 1/3)
    x = np.linspace(-12, 12, 2401).astype(np.float32)
    vp, _, _ = oracle.act_grad(oracle.ACT_SIGMOID, x)
    vm, _, _ = oracle.act_grad(oracle.ACT_SIGMOID, -x)
    assert np.all(np.abs(vp.astype(np.float64) + vm - 1.0) <= 2 * 2.0 ** -24)
    assert np.all(vp > 0) and np.all(vp <= 1)
    t, _, _ = oracle.act_grad(oracle.ACT_SIGMOID, np.array([-20.0], np.float32))
    assert t[0] == pytest.approx(math.exp(-20.0) / (1 + math.exp(-20.0)), rel=1e-6)


def test_identity_is_exact_and_rows_with_unit_probs_copy_x():
    rng = np.random.default_rng(14)
    _, x, _, _ = inputs.random_problem(rng, [5], 96, False)
    y = oracle.act_fwd_rows(x, None, oracle.ACT_IDENTITY, S4)
    assert np.array_equal(y, x)
    xf = oracle.bf16_to_f32(x[0]).astype(np.float32)
    v, d, _ = oracle.act_grad(oracle.ACT_IDENTITY, xf)
    assert np.array_equal(v, xf) and np.all(d == 1.0)


@pytest.mark.parametrize("act", [oracle.ACT_GELU, oracle.ACT_SIGMOID])
def test_further_unary_derivatives_by_finite_differences(act):
    x = np.linspace(-7, 7, 281)
    def f(z):
        return oracle.act_grad(act, z.astype(np.float32), None, S4)[0].astype(np.float64)
    num = _fd(f, x, 1e-2)
    _, da, _ = oracle.act_grad(act, x.astype(np.float32), None, S4)
    assert np.allclose(da, num, rtol=1e-3, atol=1e-4)


# ------------------------------------------------------------ dprobs

def test_dprobs_tree_order_hand_worked():
    # 4 blocks of 32, one nonzero term each: [1e8, 1, -1e8, 1]
    t = np.zeros(128, np.float32)
    t[0], t[32], t[64], t[96] = 1e8, 1.0, -1e8, 1.0
    # tree: (1e8 + 1) + (-1e8 + 1) = 1e8 + (-1e8) = 0 in binary32; serial order gives 1
    assert oracle.dprobs_sum(t) == 0.0
    # odd number of blocks: the unpaired last block moves up a level
    t3 = np.zeros(96, np.float32)
    t3[0], t3[32], t3[64] = 2.0 ** 24, 1.0, 1.0
    # (2^24 + 1) -> 2^24 (tie to even), then + 1 -> 2^24; pairing the last
    # two blocks first would give 2^24 + 2
    assert oracle.dprobs_sum(t3) == 2.0 ** 24


def test_dprobs_within_error_bound_of_exact_sum():
    rng = np.random.default_rng(9)
    for n in [32, 64, 96, 256, 1024, 2048, 4096]:
        t = rng.standard_normal(n).astype(np.float32)
        s = oracle.dprobs_sum(t)
        exact = math.fsum(t.astype(np.float64))
        bound = (32 + math.ceil(math.log2(max(1, n // 32))) + 1) * 2.0 ** -24 * float(np.abs(t).sum())
        assert abs(s - exact) <= bound


def test_bwd_rows_match_definition_sums():
    """dX and dprobs of the composed backward against float64 sums of the
    activation's value/derivative (pins the dY * p * act' wiring)."""
    rng = np.random.default_rng(10)
    for act, prm in [(oracle.ACT_SRELU, S4), (oracle.ACT_TANH_SRELU, S4), (oracle.ACT_SWIGLU, S4),
                     (oracle.ACT_CLAMPED_SWIGLU, CLAMP), (oracle.ACT_GELU, S4), (oracle.ACT_SIGMOID, S4),
                     (oracle.ACT_IDENTITY, S4)]:
        glu = oracle.is_glu(act)
        split, x, p, dy = inputs.random_problem(rng, [7], 64, glu)
        dx, dpr = oracle.act_bwd_rows(dy, x, p, act, prm)
        xf = oracle.bf16_to_f32(x).astype(np.float32)
        dyf = oracle.bf16_to_f32(dy).astype(np.float64)
        a = xf[:, :64]
        b = xf[:, 64:] if glu else None
        val, da, db = oracle.act_grad(act, a, b, prm)
        g = dyf * p[:, None].astype(np.float64)
        ref_da = g * da
        got = oracle.bf16_to_f32(dx).astype(np.float64)
        assert np.allclose(got[:, :64], ref_da, rtol=2 ** -7, atol=1e-30)
        if glu:
            assert np.allclose(got[:, 64:], g * db, rtol=2 ** -7, atol=1e-30)
        for r in range(7):
            terms = dyf[r] * val[r].astype(np.float64)
            bound = 40 * 2.0 ** -24 * float(np.abs(terms).sum()) + 1e-30
            assert abs(dpr[r] - math.fsum(terms)) <= bound
        # forward: Y = bf16(p * act)
        y = oracle.act_fwd_rows(x, p, act, prm)
        ref_y = p[:, None].astype(np.float64) * val.astype(np.float64)
        assert np.allclose(oracle.bf16_to_f32(y), ref_y, rtol=2 ** -8, atol=1e-30)


def test_dprobs_is_gradient_of_probs():
    """Finite difference of sum(dY * Y) w.r.t. p, with Y unrounded, equals dprobs."""
    rng = np.random.default_rng(11)
    split, x, p, dy = inputs.random_problem(rng, [3], 128, False)
    _, dpr = oracle.act_bwd_rows(dy, x, p, oracle.ACT_SRELU, S4)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    dyf = oracle.bf16_to_f32(dy).astype(np.float64)
    for r in range(3):
        f = lambda pp: float(np.sum(dyf[r] * pp * np.maximum(xf[r], 0) ** 2))
        fd = (f(p[r] + 1e-3) - f(p[r] - 1e-3)) / 2e-3
        assert dpr[r] == pytest.approx(fd, rel=1e-4, abs=1e-4)


# --------------------------------------------------------- columnwise

@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
@pytest.mark.parametrize("me", [1, 15, 17, 33, 64])
def test_columnwise_is_rowwise_of_padded_transpose(recipe, me):
    rng = np.random.default_rng(12 + me)
    y = oracle.f32_to_bf16(rng.standard_normal((me, 64)).astype(np.float32))
    mp = oracle.padded_rows(me, recipe)
    zt = np.zeros((64, mp), np.uint16)
    zt[:, :me] = y.T
    if recipe == oracle.MXFP8:
        d, s = oracle.quant_cols(y, recipe)
        rd, rs = oracle.quant_rows(zt, recipe)
    else:
        S = oracle.nvfp4_tensor_scale(oracle.amax_cols(y, False, 0))
        d, s = oracle.quant_cols(y, recipe, False, 0, S)
        rd, rs = oracle.quant_rows(zt, recipe, S)
        assert oracle.amax_cols(y, False, 0) == oracle.amax_rows(y)
    assert np.array_equal(d, rd) and np.array_equal(s, rs)


def test_rht_columnwise_equals_transform_then_quantize():
    rng = np.random.default_rng(13)
    mask = inputs.rht_mask_from_seed(0)
    y = oracle.f32_to_bf16(rng.standard_normal((37, 32)).astype(np.float32))
    amax = oracle.amax_cols(y, True, mask)
    S = oracle.nvfp4_tensor_scale(amax)
    d, s = oracle.quant_cols(y, oracle.NVFP4, True, mask, S)
    yf = oracle.bf16_to_f32(y)
    mp = 48
    zt = np.zeros((32, mp), np.float32)
    zt[:, :37] = yf.T
    m = 0.0
    for j in range(32):
        for i in range(3):
            w = oracle.rht16(zt[j, 16 * i:16 * i + 16], mask)
            m = max(m, float(np.abs(w).max()))
            codes, sc = oracle.nvfp4_block(w, S)
            assert sc == s[j, i]
            packed = codes[0::2] | (codes[1::2] << 4)
            assert np.array_equal(packed, d[j, 8 * i:8 * i + 8])
    assert m == amax


def test_quantize_grouped_layout_and_empty_experts():
    rng = np.random.default_rng(14)
    split = [5, 0, 40, 0, 1]
    v = oracle.f32_to_bf16(rng.standard_normal((46, 64)).astype(np.float32))
    for recipe in (oracle.MXFP8, oracle.NVFP4):
        out = oracle.quantize_grouped(v, split, recipe, rht=(recipe == oracle.NVFP4), mask=0x0F0F)
        doff, soff = oracle.expert_col_offsets(split, 64, recipe)
        assert out["col_data"].size == doff[-1] and out["col_scale"].size == soff[-1]
        if recipe == oracle.NVFP4:
            assert out["amax_row"][1] == 0 and out["amax_col"][3] == 0


# ------------------------------------------- the regeneration-deviation row

def test_fp32_accumulator_forward_equals_bf16_forward_on_bf16_values():
    rng = np.random.default_rng(11)
    x = inputs.normal_bf16(rng, (40, 64), 2.0)
    p = rng.random(40, dtype=np.float32)
    for act, prm in ((oracle.ACT_SRELU, (0.0, 0.0, 0.0, 0.0)), (oracle.ACT_TANH_SRELU, S4),
                     (oracle.ACT_CLAMPED_SWIGLU, CLAMP)):
        y16 = oracle.act_fwd_rows(x, p, act, prm)
        y32 = oracle.act_fwd_rows_f32(oracle.bf16_to_f32(x), p, act, prm)
        assert np.array_equal(y16, y32)


def test_dequant_cols_hand_worked_values():
    # MXFP8 (hand-worked block, amax 1.0, e = -8): 1.0 -> 0x78 -> 1.0, 0.3 -> 0x6A -> 0.3125
    v = np.zeros((32, 1), np.float32)
    v[0, 0], v[1, 0] = 1.0, 0.3
    d, s = oracle.quant_cols(oracle.f32_to_bf16(v), oracle.MXFP8)
    got = oracle.dequant_cols(d, s, oracle.MXFP8)
    assert got[0, 0] == 1.0 and got[0, 1] == 0.3125 and np.all(got[0, 2:] == 0)
    # NVFP4 (hand-worked block, tensor amax 12, block amax 3: S_enc 224, scale code 0x6E = 112,
    # multiplier 2): 3 -> 6 -> 3.0, 1.25 -> 2.5 -> tie to 2 -> 1.0, -0.6 -> -1.2 -> -1 -> -0.5
    v = np.zeros((32, 1), np.float32)
    v[0, 0], v[1, 0], v[2, 0], v[16, 0] = 3.0, 1.25, -0.625, 12.0
    vb = oracle.f32_to_bf16(v)
    S = oracle.nvfp4_tensor_scale(12.0)
    assert S == 224.0
    d, s = oracle.quant_cols(vb, oracle.NVFP4, False, 0, S)
    got = oracle.dequant_cols(d, s, oracle.NVFP4, S)
    assert s[0, 0] == 0x6E
    assert got[0, 0] == 3.0 and got[0, 1] == 1.0 and got[0, 2] == -0.5 and got[0, 16] == 12.0


def test_rht_cols_is_the_oracle_transform_and_keeps_inner_products():
    rng = np.random.default_rng(12)
    mask = 0x5A3C
    v = rng.integers(-64, 64, (32, 3)).astype(np.float32)     # exact in every order
    w = oracle.rht_cols(v, mask)
    for c in range(3):
        for k in range(2):
            assert np.array_equal(w[16 * k:16 * k + 16, c], oracle.rht16(v[16 * k:16 * k + 16, c], mask).astype(np.float64))
    a, b = rng.standard_normal((48, 5)), rng.standard_normal((48, 4))
    assert np.allclose(oracle.rht_cols(a, mask).T @ oracle.rht_cols(b, mask), a.T @ b, rtol=0, atol=1e-12)


# --------------------------------------------------------- tiled scale layout
# The tiled layout of block-scaled GEMM operands (cuBLASLt's 1D block-scaling
# factor layout: 128 x 4 tiles of 512 bytes, entry (r, c) of a tile at
# 16 (r mod 32) + 4 floor(r / 32) + c).  The GPU tests pin it independently by
# running cuBLASLt's block-scaled GEMM on the library's output.

def test_tiled_scales_hand_worked_positions():
    R, C = 130, 5                           # 2 x 2 tiles after padding to 256 x 8
    s = np.zeros((R, C), np.uint8)
    where = {(0, 0): 0, (1, 0): 16, (31, 0): 496, (32, 0): 4, (33, 0): 20, (127, 3): 511,
             (0, 4): 512, (31, 4): 512 + 496, (128, 0): 1024, (129, 4): 1024 + 512 + 16}
    for k, (r, c) in enumerate(where):
        s[r, c] = k + 1
    t = oracle.tiled_scales(s)
    assert t.size == 2048
    for k, ((r, c), off) in enumerate(where.items()):
        assert t[off] == k + 1, ((r, c), off)
    assert np.count_nonzero(t) == len(where)


def test_tiled_scales_is_a_bijection_with_zero_padding():
    rng = np.random.default_rng(7)
    for R, C in ((1, 1), (128, 4), (129, 3), (300, 17), (64, 8)):
        s = rng.integers(1, 256, size=(R, C)).astype(np.uint8)
        t = oracle.tiled_scales(s)
        assert t.size == -(-R // 128) * 128 * (-(-C // 4) * 4)
        assert np.count_nonzero(t) == R * C
        assert sorted(t[t != 0].tolist()) == sorted(s.reshape(-1).tolist())
        # each row's entries keep their column order inside a 4-column group
        if R >= 33 and C >= 4:
            assert t[16 * 1 + 4 * 1 + 0] == s[33, 0] and t[16 * 1 + 4 * 1 + 3] == s[33, 3]


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
def test_quantize_grouped_tiled_is_the_compact_scales_rearranged(recipe):
    rng = np.random.default_rng(11)
    split, x, p, dy = inputs.random_problem(rng, [0, 37, 130, 0, 5], 192, False)
    rht = recipe == oracle.NVFP4
    a = oracle.quantize_grouped(x, split, recipe, rht, 0x1357, True, True)
    b = oracle.quantize_grouped(x, split, recipe, rht, 0x1357, True, True, oracle.SCALES_TILED)
    for k in ("row_data", "col_data", "amax_row", "amax_col"):
        if k in a:
            assert np.array_equal(a[k], b[k]), k
    B = oracle.block_size(recipe)
    offs = np.concatenate([[0], np.cumsum(split)])
    rows = [oracle.tiled_scales(a["row_scale"][offs[e]:offs[e + 1]]) for e in range(len(split))]
    assert np.array_equal(b["row_scale"], np.concatenate(rows))
    assert b["row_scale"].size == sum(-(-m // 128) * 128 for m in split) * (-(-192 // B // 4) * 4)
    assert b["col_scale"].size == sum(-(-m // (4 * B)) for m in split) * 512 * 2

