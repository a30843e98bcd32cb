"""The kernel's conversions (E4M3 and E2M1 with round-to-nearest-even and
saturation, E8M0 shared exponents, E4M3 block scales, the NVFP4 tensor scale)
over their whole range, through the C ABI, bit for bit against the oracle's
encoders (which are pinned to the format tables on the CPU).

The inputs go through the identity activation with p = 1 (probs NULL), so the
quantized values are the BF16 inputs themselves, laid out so that:
  * MXFP8: every finite BF16 value is the amax of a 32-block (every E8M0 code
    a BF16 amax can produce), and every BF16 value of magnitude at most 448 is
    an element of a block whose scale is 2^0 (every E4M3 code and every E4M3
    rounding tie);
  * NVFP4 rowwise: a block of amax 6c for every positive E4M3 value c under a
    tensor scale of exactly 1 (every block-scale code), elements c * t for t
    on the E2M1 grid and, for power-of-two c, on every E2M1 tie; and every
    finite BF16 value as a block amax, in experts of 16 binades each, so the
    tensor scale takes values on both sides of 2^100 (both block-scale forms);
  * NVFP4 columnwise with the RHT: 16-row column chunks v = (1/4) D H w chosen
    so that the transformed chunk is exactly a designed w (the transform is
    exact on them), reaching every block-scale code and every E2M1 tie after
    the transform.
The test asserts that every code the format has was produced at least once.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_bf16, unpack_fp4
from nvfp4_quantization_grouped_gb300 import gsa

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

MASK = 0x5A3C


def _bits(v):
    """BF16 bit patterns of float32 values (truncated: exact for the designed ones)."""
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _finite_bf16():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return h[((h >> 7) & 0xFF) != 0xFF]                      # 65280 values, both zeros included


def _e4m3_values():
    """The 126 positive finite E4M3 values, by code."""
    return oracle.e4m3_decode(np.arange(1, 127, dtype=np.uint8)).astype(np.float64)


def _run_identity(x_bits, split, recipe, rht):
    x = dev_bf16(np.ascontiguousarray(x_bits))
    out = gsa.fwd(x, None, list(split), "identity", recipe, rht, MASK, True, True, False,
                  gsa.ActParams(4.0, 7.0, 1.702, 1.0))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items() if k != "_info"}


def _assert_same(g, ref, keys):
    for k in keys:
        a = np.asarray(g[k]).reshape(-1).view(np.uint8)
        b = np.asarray(ref[k]).reshape(-1).view(np.uint8)
        n = b.size
        bad = np.flatnonzero(a[:n] != b)
        assert bad.size == 0, f"{k}: {bad.size} bytes differ, first at {bad[:5]}"


def test_mxfp8_every_scale_and_element_code():
    fin = _finite_bf16()
    # every finite BF16 value v as a block amax: v, then v / 2^j (truncated to BF16)
    v = oracle.bf16_to_f32(fin).astype(np.float32)
    scaled = v[:, None] * np.ldexp(np.float32(1.0), -np.arange(32, dtype=np.int32))[None, :].astype(np.float32)
    part_a = _bits(scaled)                                    # [65280, 32]
    # every BF16 value of magnitude <= 448 as an element next to the anchor 448
    mag = oracle.bf16_to_f32(fin).astype(np.float64)
    small = fin[(np.abs(mag) <= 448.0)]
    nblk = -(-small.size // 31)
    elems = np.concatenate([small, np.zeros(nblk * 31 - small.size, np.uint16)]).reshape(nblk, 31)
    part_b = np.concatenate([np.full((nblk, 1), _bits(np.float32(448.0)), np.uint16), elems], axis=1)
    blocks = np.concatenate([part_a, part_b])                 # [n, 32]
    width = 256
    pad = (-blocks.shape[0]) % (width // 32)
    blocks = np.concatenate([blocks, np.zeros((pad, 32), np.uint16)])
    x = blocks.reshape(-1, width)
    split = [x.shape[0] // 3, x.shape[0] // 3, x.shape[0] - 2 * (x.shape[0] // 3)]
    g = _run_identity(x, split, oracle.MXFP8, False)
    ref = oracle.quantize_grouped(x, split, oracle.MXFP8, False, 0, True, True)
    _assert_same(g, ref, ("row_data", "row_scale", "col_data", "col_scale"))
    codes = set(np.unique(g["row_data"]).tolist())
    assert codes >= set(range(0, 127)) | set(range(128, 255)), "some E4M3 code never produced"
    scales = set(np.unique(g["row_scale"]).tolist())
    want = set(np.unique(ref["row_scale"]).tolist())
    assert scales == want and min(scales) == 0 and len(scales) >= 240, (min(scales), max(scales), len(scales))


def _nvfp4_row_design():
    """Expert 0 (tensor scale exactly 1): every block-scale code and E2M1 tie."""
    blocks = []
    for c in _e4m3_values():
        t = np.array([6, -6, 0.5, -0.5, 1, -1, 1.5, -1.5, 2, -2, 3, -3, 4, -4, 0, -0.0])
        blocks.append(c * t)
    for k in range(-9, 9):                                    # power-of-two values of E4M3
        c = 2.0 ** k
        t = np.array([6, 0.25, -0.25, 0.75, -0.75, 1.25, -1.25, 1.75, -1.75, 2.5, -2.5, 3.5, -3.5, 5, -5, -0.0])
        blocks.append(c * t)
    b = np.array(blocks, np.float32)
    assert np.max(np.abs(b)) == 2688.0                        # S = 2688 / 2688 = 1
    bits = _bits(b)
    assert np.array_equal(oracle.bf16_to_f32(bits), b)        # every designed value is exact in BF16
    return bits


def _nvfp4_binade_experts():
    """Every finite BF16 value as a block amax (v, v / 2, ..., v / 2^15), in
    experts of 16 binades each."""
    fin = _finite_bf16()
    e = (fin >> 7) & 0xFF
    experts = []
    for lo in range(0, 256, 16):
        sel = fin[(e >= lo) & (e < lo + 16)]
        if sel.size == 0:
            continue
        v = oracle.bf16_to_f32(sel).astype(np.float32)
        scaled = v[:, None] * np.ldexp(np.float32(1.0), -np.arange(16, dtype=np.int32))[None, :].astype(np.float32)
        experts.append(_bits(scaled))
    return experts


def test_nvfp4_rowwise_every_scale_code_tie_and_tensor_scale():
    width = 256
    groups = [_nvfp4_row_design()] + _nvfp4_binade_experts()
    rows, split = [], []
    for gb in groups:
        pad = (-gb.shape[0]) % (width // 16)
        gb = np.concatenate([gb, np.zeros((pad, 16), np.uint16)])
        r = gb.reshape(-1, width)
        rows.append(r)
        split.append(r.shape[0])
    x = np.concatenate(rows)
    g = _run_identity(x, split, oracle.NVFP4, False)
    ref = oracle.quantize_grouped(x, split, oracle.NVFP4, False, 0, True, True)
    _assert_same(g, ref, ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col"))
    assert g["amax_row"][0] == 2688.0
    # both block-scale forms: tensor scales below and above 2^100
    S = np.array([oracle.nvfp4_tensor_scale(float(a)) for a in g["amax_row"]])
    assert (S <= 2.0 ** 100).any() and (S > 2.0 ** 100).any()
    e0 = split[0]
    sc0 = set(np.unique(g["row_scale"].reshape(-1, width // 16)[:e0]).tolist())
    assert sc0 >= set(range(1, 127)), "some E4M3 block-scale code never produced"
    nib = set(np.unique(unpack_fp4(g["row_data"].reshape(-1, width // 2)[:e0])).tolist())
    assert nib == set(range(16)), f"E2M1 codes produced: {sorted(nib)}"


def _rht_inverse_block(w):
    """v with (1/4) H16 D v = w exactly: v = (1/4) D H16 w (H16 H16 = 16 I)."""
    d = np.array([-1.0 if (MASK >> i) & 1 else 1.0 for i in range(16)])
    h = np.array([[(-1.0) ** bin(i & j).count("1") for j in range(16)] for i in range(16)])
    return 0.25 * d * (h @ w)


def test_nvfp4_rht_columnwise_every_scale_code_and_tie():
    designs = []
    for c in _e4m3_values():                                  # every block-scale code
        w = np.zeros(16)
        w[0] = 6 * c
        designs.append(w)
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, 0.5, 1, 1.5, 2, 3, 4, 6]
    for k in range(-9, 9):                                    # E2M1 ties and values after the transform
        c = 2.0 ** k
        for sgn in (1, -1):
            for first in (0, 7):
                w = np.zeros(16)
                w[0] = 6 * c
                sel = ties[first:first + 7] + ties[:2]
                w[1:10] = sgn * c * np.array(sel[:9]) * np.array([1, -1, 1, -1, 1, -1, 1, -1, 1])
                designs.append(w)
    w = np.zeros(16)
    w[0], w[1] = 6.0, -0.125                                  # a negative value that rounds to -0
    designs.append(w)
    ncol = 64
    nblk = -(-len(designs) // ncol)
    x = np.zeros((16 * nblk, ncol), np.float32)
    for i, wd in enumerate(designs):
        b, j = divmod(i, ncol)
        v = _rht_inverse_block(wd)
        x[16 * b:16 * b + 16, j] = v
    bits = _bits(x)
    exact = oracle.bf16_to_f32(bits).astype(np.float64)
    assert np.array_equal(exact, x.astype(np.float64)), "a designed input is not exact in BF16"
    # the transform of every designed chunk is exactly its w (checked in float64)
    back = oracle.rht_cols(exact, MASK)
    for i, wd in enumerate(designs):
        b, j = divmod(i, ncol)
        if i != len(designs) - 1:
            assert np.array_equal(back[16 * b:16 * b + 16, j], wd)
    split = [bits.shape[0]]
    g = _run_identity(bits, split, oracle.NVFP4, True)
    ref = oracle.quantize_grouped(bits, split, oracle.NVFP4, True, MASK, True, True)
    _assert_same(g, ref, ("row_data", "row_scale", "col_data", "col_scale", "amax_row", "amax_col"))
    assert g["amax_col"][0] == 2688.0                         # columnwise tensor scale exactly 1
    sc = set(np.unique(g["col_scale"]).tolist())
    assert sc >= set(range(0, 127)), "some E4M3 block-scale code never produced after the transform"
    nib = set(np.unique(unpack_fp4(g["col_data"])).tolist())
    assert nib == set(range(16)), f"E2M1 codes produced: {sorted(nib)}"
