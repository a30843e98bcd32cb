"""The C ABI used from C with the program's own device buffers
(tests/native/c_gpu_consumer.c, CUDA runtime only, no Python on its path):
SReLU MXFP8 forward and backward on a ragged split with an empty expert,
every output bit for bit against the oracle on the inputs the program drew."""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from gpu_util import params_tuple
from nvfp4_quantization_grouped_gb300 import gsa

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
E, W, M = 3, 256, 115


def test_c_program_forward_backward_matches_oracle():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"))
    libdir = os.path.dirname(gsa.LIB_PATH)
    d = tempfile.mkdtemp()
    try:
        exe = os.path.join(d, "c_gpu_consumer")
        subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"),
                        "-I" + os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "native", "c_gpu_consumer.c"),
                        "-o", exe, "-L" + libdir, "-lgsa", "-L" + os.path.join(cuda, "lib64"), "-lcudart",
                        "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64")], check=True)
        run = subprocess.run([exe], capture_output=True)
        assert run.returncode == 0, run.stderr.decode()
        buf = run.stdout
    finally:
        shutil.rmtree(d, ignore_errors=True)

    info = gsa.gsa_layout([45, 0, 70], W, oracle.MXFP8)[0]
    pos = 0

    def take(n, dtype):
        nonlocal pos
        a = np.frombuffer(buf, dtype=dtype, count=n, offset=pos)
        pos += a.nbytes
        return a

    split = take(E, np.int64)
    assert split.tolist() == [45, 0, 70]
    x = take(M * W, np.uint16).reshape(M, W)
    dy = take(M * W, np.uint16).reshape(M, W)
    p = take(M, np.float32)
    sizes = (info.row_data_bytes, info.row_scale_bytes, info.col_data_bytes, info.col_scale_bytes)
    yq = [take(n, np.uint8) for n in sizes]
    dx = take(M * W, np.uint16).reshape(M, W)
    dpr = take(M, np.float32)
    dq = [take(n, np.uint8) for n in sizes]
    assert pos == len(buf)

    prm = params_tuple("srelu")
    y = oracle.act_fwd_rows(x, p, 0, prm)
    rdx, rdp = oracle.act_bwd_rows(dy, x, p, 0, prm)
    assert np.array_equal(dx, rdx)
    assert np.array_equal(dpr.view(np.uint32), rdp.view(np.uint32))
    for got, vals in ((yq, y), (dq, rdx)):
        ref = oracle.quantize_grouped(vals, split, oracle.MXFP8, False, 0, True, True)
        for g, k in zip(got, ("row_data", "row_scale", "col_data", "col_scale")):
            r = ref[k].reshape(-1).view(np.uint8)
            assert np.array_equal(g[: r.size], r), k
