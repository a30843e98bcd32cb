"""Failure detection on the GPU without a fault: the library's bounded waits
are made to run out (a counter and an mbarrier that nothing signals, limit
50 ms), the host reads GSA_ERR_DEVICE_TIMEOUT from the workspace, and the
context stays usable -- the next call on the same workspace runs clean and
matches the oracle bit for bit."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_bf16, dev_f32, host
from nvfp4_quantization_grouped_gb300 import gsa, inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

OK, TIMEOUT = 0, 6


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_runs_out_and_reports(which):
    rng = np.random.default_rng(31 + which)
    split, x, p, _ = inputs.random_problem(rng, [70, 0, 130], 128, False)
    split = [int(s) for s in split]
    ws = gsa.Workspace(split, 128, 0, oracle.NVFP4, "cuda")
    t0 = time.monotonic()
    assert gsa.gsa_selftest_wait_timeout(ctypes.c_void_p(ws.ptr), which, 50, None) == OK
    assert ws.status() == TIMEOUT
    assert time.monotonic() - t0 < 10.0
    # the context and the workspace are still usable
    out = gsa.fwd(dev_bf16(x), dev_f32(p), split, "srelu", oracle.NVFP4, True, 0x0F0F, ws=ws)
    assert ws.status() == OK
    ref = oracle.fwd(x, p, split, oracle.ACT_SRELU, (4.0, 7.0, 1.702, 1.0), oracle.NVFP4, True, 0x0F0F)
    for k in ("row_data", "row_scale", "col_data", "col_scale"):
        assert np.array_equal(host(out[k]).view(np.uint8).reshape(-1)[:ref[k].size], ref[k].reshape(-1)), k
