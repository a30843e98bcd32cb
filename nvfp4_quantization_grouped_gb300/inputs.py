"""Seeded synthetic inputs for the grouped scaled activation + quantization path.

This module holds only random draws and their bookkeeping -- none of the
method's arithmetic -- so that the CUDA path and the CPU oracle can both be
fed from it.  Every array is NumPy, host-resident:

* ``x``      -- FC1 output, BF16 bit patterns (uint16), ``[M, W_in]``
* ``probs``  -- per-row router scale, float32, ``[M]``
* ``dy``     -- gradient w.r.t. Y, BF16 bit patterns, ``[M, W]``
* ``split_sizes`` -- int64 ``[E]``, rows grouped by expert in expert order
* ``rht_mask``    -- the 16 random signs of the columnwise Hadamard, drawn
  as the low 16 bits of splitmix64(seed) (a published generator, written out
  below from its definition).

Normal draws are made in float32 and truncated toward zero to BF16 (the high
16 bits), so no rounding rule of the method is involved in making the data.

The five workloads follow the Activation + GroupedLinear Fusion for MOE page
(SReLU, SwiGLU, clamped SwiGLU grouped kernels) and the ScaledTanhSReLU
recompute page (hidden 256, 4 groups; MXFP8 and NVFP4 with RHT).
"""
from __future__ import annotations

import dataclasses

import numpy as np

ACT_SRELU, ACT_TANH_SRELU, ACT_SWIGLU, ACT_CLAMPED_SWIGLU = 0, 1, 2, 3
ACT_GELU, ACT_SIGMOID, ACT_IDENTITY = 4, 5, 6
ACT_NAMES = {"srelu": ACT_SRELU, "tanh_srelu": ACT_TANH_SRELU,
             "swiglu": ACT_SWIGLU, "clamped_swiglu": ACT_CLAMPED_SWIGLU,
             "gelu": ACT_GELU, "sigmoid": ACT_SIGMOID, "identity": ACT_IDENTITY}
RECIPE_MXFP8, RECIPE_NVFP4 = 0, 1

_MASK64 = (1 << 64) - 1


def splitmix64(seed: int) -> int:
    """One output of Vigna's splitmix64 generator started from ``seed``."""
    z = (seed + 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def rht_mask_from_seed(seed: int) -> int:
    return splitmix64(seed) & 0xFFFF


def default_act_params(act: int) -> tuple[float, float, float, float]:
    """(s, limit, alpha, glu_linear_offset) used by the workloads."""
    if act == ACT_TANH_SRELU:
        return (4.0, 0.0, 0.0, 0.0)
    if act == ACT_CLAMPED_SWIGLU:
        return (0.0, 7.0, 1.702, 1.0)
    return (0.0, 0.0, 0.0, 0.0)


def normal_bf16(rng: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    """N(0, sigma^2) draws as BF16 bit patterns (float32 truncated to BF16),
    drawn in chunks (the same stream as one draw) to bound host memory."""
    out = np.empty(int(np.prod(shape)), dtype=np.uint16)
    chunk = 1 << 24
    for i in range(0, out.size, chunk):
        f = rng.standard_normal(min(chunk, out.size - i), dtype=np.float32)
        if sigma != 1.0:
            f *= np.float32(sigma)
        out[i:i + f.size] = f.view(np.uint32) >> 16
    return out.reshape(shape)


def multinomial_split(rng, rows: int, weights: np.ndarray) -> np.ndarray:
    w = np.asarray(weights, dtype=np.float64)
    return rng.multinomial(rows, w / w.sum()).astype(np.int64)


def dirichlet_split(rng, rows: int, experts: int, alpha: float = 0.5) -> np.ndarray:
    return multinomial_split(rng, rows, rng.dirichlet(np.full(experts, alpha)))


def zipf_skew_split(rng, rows: int, experts: int, s: float = 1.1, n_empty: int = 1) -> np.ndarray:
    """Weights proportional to k^-s over a seeded permutation of the experts,
    with the last ``n_empty`` experts of that permutation forced empty."""
    w = np.arange(1, experts + 1, dtype=np.float64) ** (-s)
    w[experts - n_empty:] = 0.0
    perm = rng.permutation(experts)
    ww = np.empty(experts)
    ww[perm] = w
    return multinomial_split(rng, rows, ww)


def topk_routing(rng, tokens: int, experts: int, k: int, s: float = 1.1, n_empty: int = 4):
    """Route each token to k distinct experts drawn from Zipf(s) weights
    (Gumbel top-k), the last ``n_empty`` experts never chosen.  Returns
    (split_sizes, probs) with rows sorted by expert; probs is the softmax of
    N(0,1) logits over all experts, read at the routed expert."""
    w = np.arange(1, experts + 1, dtype=np.float64) ** (-s)
    w[experts - n_empty:] = 0.0
    with np.errstate(divide="ignore"):
        logw = np.log(w)
    split = np.zeros(experts, dtype=np.int64)
    chosen = np.empty((tokens, k), dtype=np.int64)
    probs_tok = np.empty((tokens, k), dtype=np.float32)
    chunk = 4096
    for t0 in range(0, tokens, chunk):
        t1 = min(tokens, t0 + chunk)
        g = rng.gumbel(size=(t1 - t0, experts)) + logw[None, :]
        top = np.argpartition(-g, k - 1, axis=1)[:, :k]
        logits = rng.standard_normal((t1 - t0, experts))
        ex = np.exp(logits - logits.max(axis=1, keepdims=True))
        sm = ex / ex.sum(axis=1, keepdims=True)
        chosen[t0:t1] = top
        probs_tok[t0:t1] = np.take_along_axis(sm, top, axis=1).astype(np.float32)
    flat_e = chosen.reshape(-1)
    order = np.argsort(flat_e, kind="stable")
    split = np.bincount(flat_e, minlength=experts).astype(np.int64)
    probs = probs_tok.reshape(-1)[order]
    return split, probs


@dataclasses.dataclass
class Workload:
    name: str
    acts: tuple[str, ...]
    recipe: int
    experts: int
    rows: int
    width: int             # Y width W
    glu: bool
    x_sigma: float
    recompute: bool
    rht: bool
    description: str

    @property
    def w_in(self) -> int:
        return 2 * self.width if self.glu else self.width


WORKLOADS = {
    "tiny_srelu_mxfp8": Workload(
        "tiny_srelu_mxfp8", ("srelu",), RECIPE_MXFP8, 4, 320, 256, False, 1.0, False, False,
        "SReLU MXFP8 fwd+bwd: 4 experts, split [64,128,32,96], width 256"),
    "tanh_srelu_mxfp8_recompute": Workload(
        "tanh_srelu_mxfp8_recompute", ("tanh_srelu", "srelu"), RECIPE_MXFP8, 8, 8192, 1024, False,
        2.0, True, False,
        "TanhSReLU(s=4)/SReLU MXFP8 recompute: 8 experts, 8192 rows (Dirichlet 0.5), width 1024"),
    "swiglu_mxfp8": Workload(
        "swiglu_mxfp8", ("swiglu", "clamped_swiglu"), RECIPE_MXFP8, 16, 32768, 2048, True, 1.0,
        False, False,
        "SwiGLU/clamped SwiGLU MXFP8: 16 experts, 32768 rows (Zipf skew, 1 empty), width 2x2048"),
    "nvfp4_rht": Workload(
        "nvfp4_rht", ("srelu", "tanh_srelu"), RECIPE_NVFP4, 32, 65536, 2048, False, 1.0, False, True,
        "SReLU/TanhSReLU(s=4) NVFP4 + 16-point RHT: 32 experts, 65536 rows (Dirichlet 0.5), width 2048"),
    "moe_swiglu_mxfp8_recompute": Workload(
        "moe_swiglu_mxfp8_recompute", ("swiglu",), RECIPE_MXFP8, 128, 262144, 4096, True, 1.0,
        True, False,
        "SwiGLU MXFP8 recompute: 128 experts, 32768 tokens x top-8 (Zipf 1.1, 4 empty), width 2x4096"),
}


@dataclasses.dataclass
class Problem:
    workload: Workload
    split_sizes: np.ndarray
    x: np.ndarray
    probs: np.ndarray
    dy: np.ndarray
    rht_mask: int
    seed: int

    @property
    def rows(self) -> int:
        return int(self.split_sizes.sum())


def make_split(wl: Workload, rng: np.random.Generator):
    """Split sizes (and, for the routed workload, the probs) -- drawn first."""
    if wl.name == "tiny_srelu_mxfp8":
        return np.array([64, 128, 32, 96], dtype=np.int64), None
    if wl.name in ("tanh_srelu_mxfp8_recompute", "nvfp4_rht"):
        return dirichlet_split(rng, wl.rows, wl.experts, 0.5), None
    if wl.name == "swiglu_mxfp8":
        return zipf_skew_split(rng, wl.rows, wl.experts, 1.1, n_empty=1), None
    if wl.name == "moe_swiglu_mxfp8_recompute":
        return topk_routing(rng, wl.rows // 8, wl.experts, 8, 1.1, n_empty=4)
    raise KeyError(wl.name)


def make_problem(name: str, seed: int = 0, rows: int | None = None) -> Problem:
    """Draw a workload's inputs in the fixed order: splits, X, probs, dY.

    ``rows`` (optional) rescales the split to a smaller total for quick runs;
    the expert count, width and distributions stay the workload's own."""
    wl = WORKLOADS[name]
    rng = np.random.default_rng(seed)
    split, probs = make_split(wl, rng)
    if rows is not None and rows != int(split.sum()):
        frac = split.astype(np.float64) / max(1, int(split.sum()))
        split = np.floor(frac * rows).astype(np.int64)
        split[np.argmax(split)] += rows - int(split.sum())
        probs = None
    M = int(split.sum())
    x = normal_bf16(rng, (M, wl.w_in), wl.x_sigma)
    if probs is None:
        probs = rng.random(M, dtype=np.float32)
    dy = normal_bf16(rng, (M, wl.width))
    return Problem(wl, split, x, probs.astype(np.float32), dy, rht_mask_from_seed(seed), seed)


def device_problem(name: str, dev, seed: int = 0):
    """A full-size workload with X and dY drawn on the device: the split (and
    the routed workload's probabilities) drawn as make_split does, X and dY by
    a seeded torch generator on `dev` with the workload's distributions
    (N(0, sigma^2) in FP32, truncated toward zero to BF16, as normal_bf16 does;
    p ~ U(0, 1) unless the workload routes).  The multi-GB host draws would
    take minutes.  Returns (workload, split list, M, x, p, dy)."""
    import torch
    wl = WORKLOADS[name]
    split, probs = make_split(wl, np.random.default_rng(seed))
    M = int(split.sum())
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def normal(shape, sigma):
        f = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if sigma != 1.0:
            f *= sigma
        return (f.view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)

    x = normal((M, wl.w_in), wl.x_sigma)
    p = (torch.rand(M, generator=g, device=dev, dtype=torch.float32) if probs is None
         else torch.from_numpy(np.asarray(probs, np.float32)).to(dev))
    dy = normal((M, wl.width), 1.0)
    return wl, [int(v) for v in split], M, x, p, dy


def random_problem(rng: np.random.Generator, split_sizes, width: int, glu: bool,
                   x_sigma: float = 1.0):
    """Ad-hoc problem for edge-case tests: (x, probs, dy) for a given split."""
    split = np.asarray(split_sizes, dtype=np.int64)
    M = int(split.sum())
    w_in = 2 * width if glu else width
    x = normal_bf16(rng, (M, w_in), x_sigma)
    probs = rng.random(M, dtype=np.float32)
    dy = normal_bf16(rng, (M, width))
    return split, x, probs, dy
