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


def test_four_cta_forward_exhausted_wait_budget_reports_timeout_then_recovers(monkeypatch):
    """The same for the d_v = 512 form of the fused forward (clusters of four
    CTAs, P and row sums sent between the two pairs): a wait that gives up in
    one CTA leaves the others waiting on it to give up in turn, every warp
    group leaves through its agreement barriers, and the next call is correct."""
    import mlstm_matrix_memory_gb300 as M
    monkeypatch.setenv("MLSTM_TC_VARIANT", "pair")
    monkeypatch.setenv("MLSTM_TC_XCH", "1")
    x = W.sequence_inputs(1, 4, 700, 512, 512, torch.bfloat16, seed=33)
    xd = to_dev(x)
    assert M.last_device_status() == 0
    M.set_spin_limit(1)
    try:
        M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], algo="tc")
        status = M.last_device_status()
    finally:
        M.set_spin_limit(0)
    assert status == -5                     # MLSTM_ETIMEOUT
    h = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], algo="tc")
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    want, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert rel_err(h, want) <= TOL_BF16


@pytest.mark.parametrize("shape", [(10, 5, 150, 128, 128), (2, 2, 192, 512, 128)],
                         ids=["heads-cut-tmem-A", "dqk512-smem-A"])
def test_handoff_exhausted_wait_budget_reports_timeout_then_recovers(shape):
    """The same for the tensor-core hand-off: heads cut between CTAs with
    several pieces per CTA (weighted V^T in TMEM), and d_qk = 512 (weighted V
    in shared memory).  Every warp group leaves through its agreement
    barriers; the next call is correct."""
    import mlstm_matrix_memory_gb300 as M
    B, H, T, dqk, dv = shape
    x = W.sequence_inputs(B, H, T, dqk, dv, torch.bfloat16, seed=37)
    xd = to_dev(x)
    ws = torch.empty(M.parallel_fwd_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
    M.gate_prep(xd["igate_pre"], xd["fgate_pre"], ws)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    M.set_spin_limit(1)
    try:
        M.parallel_final_state(xd["k"], xd["v"], ws)
        torch.cuda.synchronize()
        status = M.last_device_status()
    finally:
        M.set_spin_limit(0)
    assert status == -5                     # MLSTM_ETIMEOUT
    C, n, m = M.parallel_final_state(xd["k"], xd["v"], ws)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    _, wC, wn, _ = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert rel_err(C, wC) <= TOL_BF16
    assert rel_err(n, wn) <= TOL_BF16
