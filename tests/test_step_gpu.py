"""GPU parity of the recurrent step (generation) against the fp64 oracle."""
import math

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


def run_step(M, xd, with_o=True):
    h = M.step(xd["C"], xd["n"], xd["m"], xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"],
               xd["o"] if with_o else None)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    return h


def check(M, x, with_o, tol_h, heads=None):
    xd = to_dev(x)
    h = run_step(M, xd, with_o)
    if heads is not None:       # oracle on a sample of heads only (flattened B*H index)
        pick = lambda t: t.reshape(-1, *t.shape[2:])[heads].unsqueeze(0)
        xs = {k: pick(v) for k, v in x.items()}
        got = {k: pick(v.cpu()) for k, v in xd.items()}
        h = pick(h.cpu())
    else:
        xs, got = x, {k: v.cpu() for k, v in xd.items()}
    wh, wC, wn, wm = oracle.step(xs["C"], xs["n"], xs["m"], xs["q"], xs["k"], xs["v"], xs["igate_pre"],
                                 xs["fgate_pre"], xs["o"] if with_o else None)
    assert rel_err(h, wh) <= tol_h
    assert rel_err(got["C"], wC) <= 1e-5
    assert rel_err(got["n"], wn) <= 1e-5
    assert np.max(np.abs(got["m"].numpy() - wm)) <= 1e-5


def test_step_full_size_sampled_heads(M):
    """B=256, H=4, d=512: the whole step runs; 24 heads are checked."""
    x = W.step_inputs(W.STEP, 0)
    heads = np.random.default_rng(0).choice(W.STEP.B * W.STEP.H, 24, replace=False)
    heads = torch.tensor(sorted(set(heads.tolist()) | {0, W.STEP.B * W.STEP.H - 1}))
    check(M, x, True, TOL_BF16, heads)


@pytest.mark.parametrize("dims", [(16, 24), (64, 64), (512, 8), (8, 12), (136, 200)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_step_shapes(M, dims, dtype):
    dqk, dv = dims
    w = W.StepWorkload("t", 3, 2, dqk, dv, dtype, state_std=0.3)
    x = W.step_inputs(w, dqk + dv)
    check(M, x, with_o=(dv % 2 == 0), tol_h=TOL_F32 if dtype == torch.float32 else TOL_BF16)


def test_step_fresh_state(M):
    w = W.StepWorkload("t", 2, 2, 64, 64, torch.float32)
    x = W.step_inputs(w, 7)
    x["C"].zero_()
    x["n"].zero_()
    x["m"].fill_(-math.inf)
    check(M, x, True, TOL_F32)


def test_step_twice_in_place(M):
    w = W.StepWorkload("t", 2, 3, 128, 128, torch.float32)
    x = W.step_inputs(w, 8)
    xd = to_dev(x)
    run_step(M, xd)
    h2 = run_step(M, xd)
    _, C, n, m = oracle.step(x["C"], x["n"], x["m"], x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], x["o"])
    wh, wC, _, _ = oracle.step(C, n, m, x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], x["o"])
    assert rel_err(h2, wh) <= TOL_F32
    assert rel_err(xd["C"], wC) <= 1e-5
