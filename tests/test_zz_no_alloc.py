"""mlstm_parallel_fwd_noalloc, the entry point for callers that cannot
allocate device memory (for example a plug-in whose host application owns all
GPU memory).  It keeps its scratch in an array built into the library instead
of a caller-provided workspace.

Called here through the C ABI with ctypes and compared, on two calls in a row
with different inputs, against mlstm_parallel_fwd with a normal workspace.
Both run the same kernels on the same inputs, so the outputs must be equal
bit for bit (a wrong scratch address or stale scratch would shift rows).  This file is collected last
so a failure here comes after every other test has run."""
import ctypes

import pytest
import torch

from gpu_util import to_dev
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import mlstm_matrix_memory_gb300 as M
    lib = M.library()
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.mlstm_parallel_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
    lib.mlstm_parallel_fwd_noalloc.restype = i
    return lib


def noalloc(lib, xd, dtype_code):
    B, H, T, dqk = xd["q"].shape
    dv = xd["v"].shape[-1]
    h = torch.empty((B, H, T, dv), dtype=xd["q"].dtype, device="cuda")
    m = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    n = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    rc = lib.mlstm_parallel_fwd_noalloc(xd["q"].data_ptr(), xd["k"].data_ptr(), xd["v"].data_ptr(),
                                        xd["igate_pre"].data_ptr(), xd["fgate_pre"].data_ptr(), h.data_ptr(),
                                        m.data_ptr(), n.data_ptr(), B, H, T, dqk, dv, dtype_code,
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    return h, m, n


@pytest.mark.parametrize("dtype,code,shape", [
    (torch.bfloat16, 1, (2, 2, 300, 64, 64)),
    (torch.float32, 0, (1, 3, 129, 16, 32)),
])
def test_noalloc_matches_workspace_path_twice(lib, dtype, code, shape):
    import mlstm_matrix_memory_gb300 as M
    B, H, T, dqk, dv = shape
    for seed in (11, 12):                 # two calls in a row, different inputs
        x = W.sequence_inputs(B, H, T, dqk, dv, dtype, seed=seed)
        xd = to_dev(x)
        h, m, n = noalloc(lib, xd, code)
        wh, wm, wn = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], return_mn=True)
        torch.cuda.synchronize()
        assert M.last_device_status() == 0
        # the same kernels run on the same inputs, only the scratch address
        # differs: the results must be identical, bit for bit
        assert torch.equal(h, wh)
        assert torch.equal(m, wm)
        assert torch.equal(n, wn)


def test_noalloc_rejects_jobs_beyond_its_scratch(lib):
    import mlstm_matrix_memory_gb300 as M
    limit = 4 << 20                      # MLSTM_NOALLOC_SCRATCH_BYTES
    T = 1
    while M.parallel_fwd_workspace_bytes(1, 1, T) <= limit:
        T *= 2
    lo, hi = T // 2, T                   # largest T that fits is in [lo, hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if M.parallel_fwd_workspace_bytes(1, 1, mid) <= limit:
            lo = mid
        else:
            hi = mid
    assert lo == 349504
    # buffers sized for the rejected length, so nothing could run out of bounds
    x = to_dev(W.sequence_inputs(1, 1, hi, 16, 16, torch.float32, seed=1))
    h = torch.empty((1, 1, hi, 16), device="cuda")
    p = [x[k].data_ptr() for k in ("q", "k", "v", "igate_pre", "fgate_pre")]
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.mlstm_parallel_fwd_noalloc(*p, h.data_ptr(), None, None, 1, 1, hi, 16, 16, 0, stream)
    assert rc == -7                      # MLSTM_EWORKSPACE, nothing launched
    rc = lib.mlstm_parallel_fwd_noalloc(*p, h.data_ptr(), None, None, 1, 1, 64, 16, 16, 0, stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
