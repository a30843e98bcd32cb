"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/gsa.h declares, computes layouts and workspace sizes
that agree with the oracle's layout, and rejects bad arguments before it
touches the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from nvfp4_quantization_grouped_gb300 import gsa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gsa.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][\w \*]*?)\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n.startswith(("gsa_", "grouped_"))))


def test_library_exports_every_declared_symbol():
    L = gsa.load()
    names = declared_functions()
    assert set(gsa.EXPORTED) <= set(names) | set(gsa.EXPORTED)
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    assert L.gsa_version() >> 16 == 1
    assert L.gsa_status_string(0) == b"ok"


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
def test_layout_matches_oracle(recipe):
    split = [0, 1, 15, 17, 31, 33, 64, 100, 0]
    for width in (64, 256, 4096):
        info, doff, soff = gsa.gsa_layout(split, width, recipe)
        d, s = oracle.expert_col_offsets(split, width, recipe)
        assert list(d) == doff and list(s) == soff
        M = sum(split)
        assert info.rows == M
        assert info.row_data_bytes == (M * width if recipe == oracle.MXFP8 else M * width // 2)
        assert info.row_scale_bytes == M * width // (32 if recipe == oracle.MXFP8 else 16)
        assert info.col_data_bytes == doff[-1] and info.col_scale_bytes == soff[-1]
        assert info.amax_floats == (len(split) if recipe == oracle.NVFP4 else 0)


@pytest.mark.parametrize("recipe", [oracle.MXFP8, oracle.NVFP4])
def test_tiled_layout_matches_oracle(recipe):
    """gsa_layout_ex with tiled scales: sizes and per-expert offsets equal the
    blocks of the oracle's tiled scales; the codes' layout is unchanged."""
    split = [0, 1, 15, 17, 130, 33, 64, 300, 0]
    B = 32 if recipe == oracle.MXFP8 else 16
    rng = np.random.default_rng(3)
    for width in (64, 192, 256):
        x = rng.integers(0, 0x3F80, size=(sum(split), width)).astype(np.uint16)
        ref = oracle.quantize_grouped(x, split, recipe, False, 0, True, True, oracle.SCALES_TILED)
        info, doff, soff, roff = gsa.gsa_layout_ex(split, width, gsa.Recipe(recipe, 0, 0, gsa.SCALES_TILED))
        cinfo, cdoff, _ = gsa.gsa_layout(split, width, recipe)
        assert doff == cdoff and info.row_data_bytes == cinfo.row_data_bytes
        assert info.col_data_bytes == cinfo.col_data_bytes
        assert info.row_scale_bytes == ref["row_scale"].size and info.col_scale_bytes == ref["col_scale"].size
        c4 = -(-(width // B) // 4)
        tiles = np.concatenate([[0], np.cumsum([-(-m // 128) for m in split])])
        assert roff == list(tiles * 512 * c4)
        groups = np.concatenate([[0], np.cumsum([-(-m // (4 * B)) for m in split])])
        assert soff == list(groups * 512 * (-(-width // 128)))
        b = gsa.gsa_layout_bound_ex(len(split), sum(split), width, gsa.Recipe(recipe, 0, 0, gsa.SCALES_TILED))
        assert b.row_scale_bytes >= info.row_scale_bytes and b.col_scale_bytes >= info.col_scale_bytes
    with pytest.raises(gsa.GsaError):
        gsa.gsa_layout_ex(split, 256, gsa.Recipe(recipe, 0, 0, 2))


def test_workspace_size():
    split = [128, 0, 300]
    ws1 = gsa.gsa_workspace_size(split, 256, 0, 0)       # MXFP8 (2-tile items at most): 2 slabs of dprobs partials
    ws2 = gsa.gsa_workspace_size(split, 2048, 0, 0)      # 16 slabs
    assert ws1 > 0 and ws1 % 256 == 0
    assert ws2 >= ws1 + 428 * 4 * 4
    assert gsa.gsa_workspace_size(split, 100, 0, 0) == 0      # width not a multiple of 32
    assert gsa.gsa_workspace_size([-1], 256, 0, 0) == 0


def test_wide_rows_take_larger_items():
    """Rows of more than 64 items' worth of tiles take larger items instead
    of being refused: the workspace (sized for the most slabs any call can
    use, at most 64 per band) exists for every W = 64 * 2^k up to 131072 and
    every W up to 4096; a tile count with too few factors of two is refused."""
    split = [40, 0, 17]
    for recipe in (0, 1):
        for w in [64 * 2 ** k for k in range(12)] + list(range(64, 4097, 64)):
            assert gsa.gsa_workspace_size(split, w, 0, recipe) > 0, (recipe, w)
            assert gsa.gsa_workspace_size_graph_safe(3, 57, w, 0, recipe) > 0, (recipe, w)
        assert gsa.gsa_workspace_size(split, 64 * 195, 0, recipe) == 0
        assert gsa.gsa_workspace_size(split, 64 * 2 ** 12, 0, recipe) == 0
    # the slab partials of dprobs bound the size: 64 slabs of 4 bytes per row at most
    assert gsa.gsa_workspace_size(split, 64 * 2 ** 11, 0, 0) <= gsa.gsa_workspace_size(split, 4096, 0, 0) + 57 * 64 * 4


def _fwd_status(split, w_in, act=0, recipe=0, x=0x10000, p=0x20000, qrow=(0x30000, 0x40000), qcol=(0, 0),
                ws=0x50000, ws_bytes=1 << 20, s=4.0, limit=7.0, amax=(0x60000, 0x70000), y=None):
    q = gsa.QOut(qrow[0] or None, qrow[1] or None, qcol[0] or None, qcol[1] or None, amax[0], amax[1])
    return gsa.grouped_scaled_act_fwd(x, p, split, w_in, act, gsa.ActParams(s, limit, 1.702, 1.0),
                                      gsa.Recipe(recipe, 1, 0x1234), q, y, ws, ws_bytes, None)


def test_fwd_rejects_bad_arguments_on_host():
    INVALID, UNSUP, ALIGN, WS = 1, 2, 3, 4
    assert _fwd_status([4, 4], 80) == INVALID                 # width % 32 != 0 (MXFP8)
    assert _fwd_status([4, 4], 160) == UNSUP                  # % 32 ok, not % 64
    assert _fwd_status([4, -1], 128) == INVALID               # negative split
    assert _fwd_status([4, 4], 129, act=2) == INVALID         # odd GLU width
    assert _fwd_status([4] * 257, 128) == UNSUP               # too many experts
    assert _fwd_status([4, 4], 128, act=1, s=0.0) == INVALID  # TanhSReLU needs s > 0
    assert _fwd_status([4, 4], 128, act=3, limit=-1.0) == INVALID
    assert _fwd_status([4, 4], 128, x=0x10001) == ALIGN
    assert _fwd_status([4, 4], 128, qrow=(0x30001, 0x40000)) == ALIGN
    assert _fwd_status([4, 4], 128, ws=0x50010) == ALIGN      # workspace must be 256-aligned
    assert _fwd_status([4, 4], 128, ws_bytes=16) == WS
    assert _fwd_status([4, 4], 128, ws=0) == WS
    assert _fwd_status([4, 4], 128, qrow=(0x30000, 0)) == INVALID       # data without scale
    assert _fwd_status([4, 4], 128, qrow=(0, 0), qcol=(0, 0)) == INVALID  # nothing requested
    assert _fwd_status([4, 4], 128, recipe=1, amax=(None, None)) == INVALID  # NVFP4 needs amax
    assert _fwd_status([4, 4], 128, recipe=7) == INVALID
    assert _fwd_status([4, 4], 128, act=7) == INVALID         # unknown activation
    assert _fwd_status([4, 4], 128, act=-1) == INVALID
    assert _fwd_status([4, 4], 128, p=0x20002) == ALIGN        # probs not 4-byte aligned


def test_bwd_rejects_bad_arguments_on_host():
    L = gsa.load()
    split = (ctypes.c_int64 * 2)(4, 4)
    ap = gsa.ActParams(4.0, 7.0, 1.702, 1.0)
    nv = gsa.Recipe(1, 1, 1)
    dxq = gsa.QOut(0x30000, 0x40000, None, None, 0x60000, None)
    # NVFP4 quantized dX needs the dense dX buffer
    st = L.grouped_scaled_act_bwd(0x1000, 0x2000, 0x3000, ctypes.cast(split, ctypes.c_void_p), 2, 128, 0,
                                  ctypes.byref(ap), ctypes.byref(nv), None, ctypes.byref(dxq), None, None,
                                  0x50000, 1 << 20, None)
    assert st == 1
    # no output at all
    st = L.grouped_scaled_act_bwd(0x1000, 0x2000, 0x3000, ctypes.cast(split, ctypes.c_void_p), 2, 128, 0,
                                  ctypes.byref(ap), ctypes.byref(nv), None, None, None, None, 0x50000, 1 << 20,
                                  None)
    assert st == 1
    # regenerated copy is columnwise only
    yq = gsa.QOut(0x30000, 0x40000, 0x70000, 0x80000, 0x60000, 0x90000)
    st = L.grouped_scaled_act_bwd(0x1000, 0x2000, 0x3000, ctypes.cast(split, ctypes.c_void_p), 2, 128, 0,
                                  ctypes.byref(ap), ctypes.byref(nv), 0x10000, None, None, ctypes.byref(yq),
                                  0x50000, 1 << 20, None)
    assert st == 1


def test_graph_safe_sizes_bound_every_split():
    """gsa_layout_bound / gsa_workspace_size_graph_safe cover every split of
    M rows over E experts (checked against the host-split sizes)."""
    rng = np.random.default_rng(3)
    E, M = 6, 1000
    for recipe in (0, 1):
        b = 32 if recipe == 0 else 16
        lb = gsa.gsa_layout_bound(E, M, 128, recipe)
        assert lb.rows == M
        # the worst case: one expert takes what the others leave, the others one row each
        worst = [M - (E - 1)] + [1] * (E - 1)
        info, _, _ = gsa.gsa_layout(worst, 128, recipe)
        assert lb.col_data_bytes >= info.col_data_bytes and lb.col_scale_bytes >= info.col_scale_bytes
        assert lb.col_data_bytes - info.col_data_bytes < 128 * b   # and is tight within one block
        wsb = gsa.gsa_workspace_size_graph_safe(E, M, 128, 0, recipe)
        for _ in range(50):
            split = rng.multinomial(M, rng.dirichlet(np.full(E, 0.3))).tolist()
            info, _, _ = gsa.gsa_layout(split, 128, recipe)
            assert info.col_data_bytes <= lb.col_data_bytes and info.col_scale_bytes <= lb.col_scale_bytes
            assert info.row_data_bytes == lb.row_data_bytes
            assert gsa.gsa_workspace_size(split, 128, 0, recipe) <= wsb
    assert gsa.gsa_workspace_size_graph_safe(257, 1000, 128, 0, 0) == 0
    assert gsa.gsa_workspace_size_graph_safe(4, -1, 128, 0, 0) == 0


def test_graph_safe_rejects_bad_arguments_on_host():
    INVALID, UNSUP, ALIGN, WS = 1, 2, 3, 4
    ap = gsa.ActParams(4.0, 7.0, 1.702, 1.0)

    def st(split=0x80000, E=4, M=100, w=128, act=0, recipe=0, q=(0x30000, 0x40000), ws=0x50000, ws_bytes=1 << 24,
           pad=None):
        qo = gsa.QOut(q[0] or None, q[1] or None, None, None, 0x60000, 0x70000)
        return gsa.grouped_scaled_act_fwd_graph_safe(0x10000, 0x20000, split, E, M, w, act, ap,
                                                     gsa.Recipe(recipe, 1, 0x1234), qo, None, pad, ws, ws_bytes,
                                                     None)
    assert st(split=None) == INVALID
    assert st(split=0x80004) == ALIGN                 # the device split must be 8-byte aligned
    assert st(pad=0x90004) == ALIGN
    assert st(E=0) == INVALID
    assert st(E=257) == UNSUP
    assert st(M=-5) == INVALID
    assert st(w=80) == INVALID
    assert st(ws_bytes=64) == WS
    assert st(ws=0x50010) == ALIGN
    assert st(q=(0, 0)) == INVALID                     # nothing requested
    assert st(act=9) == INVALID


def test_wait_selftest_rejects_bad_arguments_on_host():
    INVALID, ALIGN = 1, 3
    assert gsa.gsa_selftest_wait_timeout(None, 0, 50, None) == INVALID
    assert gsa.gsa_selftest_wait_timeout(0x50000, 2, 50, None) == INVALID
    assert gsa.gsa_selftest_wait_timeout(0x50000, 0, 0, None) == INVALID
    assert gsa.gsa_selftest_wait_timeout(0x50000, 1, 2001, None) == INVALID
    assert gsa.gsa_selftest_wait_timeout(0x50010, 0, 50, None) == ALIGN


def test_plain_c_consumer():
    """The boundary is a C ABI: a C99 program that includes only
    include/gsa.h and links the in-tree library makes the host-side calls
    (layouts, workspace sizes, status strings, argument errors)."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(gsa.LIB_PATH)
    d = tempfile.mkdtemp()
    try:
        exe = os.path.join(d, "c_consumer")
        subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I" + os.path.join(root, "include"),
                        os.path.join(root, "tests", "native", "c_consumer.c"), "-o", exe, "-L" + libdir, "-lgsa",
                        "-Wl,-rpath," + libdir], check=True)
        out = subprocess.run([exe], capture_output=True, text=True)
        assert out.returncode == 0, out.stdout + out.stderr
        assert out.stdout.strip().endswith("all ok"), out.stdout
    finally:
        shutil.rmtree(d, ignore_errors=True)
