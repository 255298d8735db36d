"""GPU parity of the options of part 28/30: the output gate in the parallel
forward (eq 78; fused in the CTA-pair kernel's epilogue, a separate pass
elsewhere) and the exponential forget-gate activation (eq 70: sigma or exp),
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, TOL_F32, rel_err, to_dev
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


def _tol(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


# (B, H, T, d, dtype, variant): the CTA-pair kernel (fused gate), the
# single-CTA kernel and the CUDA-core kernel (separate pass)
OG_CASES = [
    (1, 2, 600, 384, torch.bfloat16, "auto"),
    (2, 1, 300, 128, torch.bfloat16, "pair"),
    (1, 2, 200, 64, torch.bfloat16, "single"),
    (1, 2, 150, 32, torch.float32, "auto"),
]


@pytest.mark.parametrize("case", OG_CASES, ids=lambda c: "x".join(str(v) for v in c[:4]) + f"-{c[4]}-{c[5]}")
def test_output_gate(M, monkeypatch, case):
    B, H, T, d, dtype, variant = case
    if variant != "auto":
        monkeypatch.setenv("MLSTM_TC_VARIANT", variant)
    x = W.sequence_inputs(B, H, T, d, d, dtype, seed=T + d, with_ogate=True)
    xd = to_dev(x)
    h = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], ogate=xd["ogate_pre"])
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    want, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], x["ogate_pre"])
    assert rel_err(h, want) <= _tol(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_exp_forget_parallel(M, dtype):
    x = W.sequence_inputs(1, 2, 400, 64, 64, dtype, seed=31, fg=(0.0, 0.3))
    xd = to_dev(x)
    h = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], forget="exp")
    torch.cuda.synchronize()
    with oracle.forget_exp():
        want, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert rel_err(h, want) <= _tol(dtype)
    sig, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert rel_err(h, sig) > 10 * _tol(dtype)          # the variant is really in effect


def test_exp_forget_recurrent_and_hand_off(M):
    """Parallel prefill, hand-off and recurrent steps, all with the exp forget gate."""
    B, H, T1, L2, d = 1, 2, 160, 12, 64
    x = W.sequence_inputs(B, H, T1 + L2, d, d, torch.float32, seed=33, fg=(0.0, 0.3), with_ogate=True)
    xd = to_dev(x)
    pre = {k: v[:, :, :T1].contiguous() for k, v in xd.items()}
    gen = {k: v[:, :, T1:].contiguous() for k, v in xd.items()}
    ws = torch.empty(M.parallel_fwd_workspace_bytes(B, H, T1), dtype=torch.uint8, device="cuda")
    h1 = M.parallel_fwd(pre["q"], pre["k"], pre["v"], pre["igate_pre"], pre["fgate_pre"], workspace=ws, forget="exp")
    C, n, m = M.parallel_final_state(pre["k"], pre["v"], ws)
    h2 = M.step_seq(C, n, m, gen["q"], gen["k"], gen["v"], gen["igate_pre"], gen["fgate_pre"], gen["ogate_pre"],
                    forget="exp")
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    og = np.concatenate([np.full((B, H, T1, d), np.inf), oracle.f64(x["ogate_pre"][:, :, T1:])], axis=2)
    with oracle.forget_exp():
        wh, wC, wn, wm = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], og)
    assert rel_err(h1, wh[:, :, :T1]) <= TOL_F32
    assert rel_err(h2, wh[:, :, T1:]) <= TOL_F32
    assert rel_err(C, wC) <= TOL_F32
    assert rel_err(n, wn) <= TOL_F32
    assert np.max(np.abs(m.cpu().numpy() - wm)) <= 1e-4 * max(1.0, float(np.max(np.abs(wm))))
