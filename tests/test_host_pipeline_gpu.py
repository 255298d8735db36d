"""The parallel forward on host buffers (mlstm_parallel_fwd_host): chunked,
overlapped uploads / compute / downloads give exactly the device call's h."""
import pytest
import torch

from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


# (B, H, T, d_qk, d_v, dtype, pinned): fewer heads than chunks, a ragged last
# chunk (13 heads in chunks of 2), the 125M-scale layer, pageable memory, fp32
CASES = [
    (2, 3, 300, 64, 64, torch.bfloat16, True),
    (1, 13, 257, 128, 128, torch.bfloat16, True),
    (8, 4, 2048, 384, 384, torch.bfloat16, True),
    (1, 2, 200, 64, 64, torch.bfloat16, False),
    (2, 2, 100, 16, 16, torch.float32, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(v) for v in c[:5]) + f"-{c[5]}-{'pin' if c[6] else 'page'}")
def test_host_call_equals_device_call(M, case):
    B, H, T, dqk, dv, dtype, pinned = case
    x = W.sequence_inputs(B, H, T, dqk, dv, dtype, seed=T + H)
    xd = {k: v.cuda() for k, v in x.items()}
    want = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"]).cpu()
    xh = {k: (v.pin_memory() if pinned else v) for k, v in x.items()}
    h = M.parallel_fwd_host(xh["q"], xh["k"], xh["v"], xh["igate_pre"], xh["fgate_pre"])
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    assert torch.equal(h, want)
