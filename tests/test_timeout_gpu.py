"""The bounded waits of the tensor-core kernel: with a spin budget of one poll
the waits give up, the kernel reports MLSTM_ETIMEOUT through the device status
word and returns without faulting, and the next call (normal budget) on the
same context is correct.  The failure is injected from the host only."""
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, rel_err, to_dev
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_exhausted_wait_budget_reports_timeout_then_recovers():
    import mlstm_matrix_memory_gb300 as M
    x = W.sequence_inputs(2, 2, 1000, 128, 128, torch.bfloat16, seed=31)
    xd = to_dev(x)
    assert M.last_device_status() == 0
    M.set_spin_limit(1)
    try:
        M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], algo="tc")
        status = M.last_device_status()
    finally:
        M.set_spin_limit(0)
    assert status == -5                     # MLSTM_ETIMEOUT
    assert M.last_device_status() == 0      # reading clears it
    h = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], algo="tc")
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    want, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert rel_err(h, want) <= TOL_BF16
