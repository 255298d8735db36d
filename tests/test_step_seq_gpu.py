"""GPU parity of the multi-token recurrent step (mlstm_step_seq) against the
fp64 oracle, against repeated single steps, and against the parallel form."""
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


def run(M, xd, with_o):
    h = M.step_seq(xd["C"], xd["n"], xd["m"], xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"],
                   xd["o"] if with_o else None)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    return h


def check(M, x, with_o, tol_h, heads=None):
    xd = to_dev(x)
    h = run(M, xd, with_o)
    got = {k: v.cpu() for k, v in xd.items()}
    h = h.cpu()
    if heads is not None:       # oracle on a sample of heads only (flattened B*H index)
        pick = lambda t: t.reshape(-1, *t.shape[2:])[heads].unsqueeze(0)
        x = {k: pick(v) for k, v in x.items()}
        got = {k: pick(v) for k, v in got.items()}
        h = pick(h)
    wh, wC, wn, wm = oracle.step_seq(x["C"], x["n"], x["m"], x["q"], x["k"], x["v"], x["igate_pre"],
                                     x["fgate_pre"], x["o"] if with_o else None)
    assert rel_err(h, wh) <= tol_h
    assert rel_err(got["C"], wC) <= 1e-5
    assert rel_err(got["n"], wn) <= 1e-5
    assert np.max(np.abs(got["m"].numpy() - wm)) <= 1e-4


# (B, H, L, d_qk, d_v, dtype, output gate): rows of C spanning one to eight
# CTAs, ragged row and column counts, L = 1 and longer runs
SHAPES = [
    (2, 2, 1, 64, 64, torch.float32, True),
    (1, 2, 17, 128, 96, torch.bfloat16, True),
    (2, 1, 40, 384, 384, torch.bfloat16, False),
    (1, 1, 33, 512, 512, torch.bfloat16, True),
    (3, 1, 9, 8, 40, torch.float32, True),
    (1, 2, 12, 136, 200, torch.float32, False),
    (2, 2, 25, 16, 24, torch.float32, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(str(v) for v in s[:5]) + f"-{s[5]}")
def test_step_seq_shapes(M, shape):
    B, H, L, dqk, dv, dtype, with_o = shape
    w = W.StepWorkload("t", B, H, dqk, dv, dtype, state_std=0.3)
    x = W.step_seq_inputs(w, L, seed=dqk + dv + L)
    check(M, x, with_o, TOL_F32 if dtype == torch.float32 else TOL_BF16)


def test_step_seq_fresh_state(M):
    w = W.StepWorkload("t", 2, 2, 64, 64, torch.float32)
    x = W.step_seq_inputs(w, 20, seed=7)
    x["C"].zero_()
    x["n"].zero_()
    x["m"].fill_(-math.inf)
    check(M, x, True, TOL_F32)


def test_step_seq_full_size_sampled_heads(M):
    """B=256, H=4, d=512 with 16 tokens: the whole call runs; 8 heads are checked."""
    x = W.step_seq_inputs(W.STEP, 16, seed=0)
    heads = torch.tensor([0, 1, 97, 400, 513, 800, 1022, 1023])
    check(M, x, True, TOL_BF16, heads)


def test_step_seq_equals_repeated_steps(M):
    w = W.StepWorkload("t", 2, 2, 128, 128, torch.float32, state_std=0.3)
    L = 6
    x = to_dev(W.step_seq_inputs(w, L, seed=11))
    ref = {k: x[k].clone() for k in ("C", "n", "m")}
    hs = []
    for t in range(L):
        hs.append(M.step(ref["C"], ref["n"], ref["m"], x["q"][:, :, t].contiguous(), x["k"][:, :, t].contiguous(),
                         x["v"][:, :, t].contiguous(), x["igate_pre"][:, :, t].contiguous(),
                         x["fgate_pre"][:, :, t].contiguous(), x["o"][:, :, t].contiguous()))
    h = run(M, x, True)
    want = torch.stack(hs, dim=2).double().cpu().numpy()
    assert rel_err(h, want) <= TOL_F32
    for k in ("C", "n"):
        assert rel_err(x[k], ref[k].double().cpu().numpy()) <= 1e-5
    assert torch.max(torch.abs(x["m"] - ref["m"])).item() <= 1e-5


def test_step_seq_from_fresh_state_equals_parallel_form(M):
    """Recurrent and parallel forms on the GPU (fp32, no output gate)."""
    B, H, T, d = 1, 2, 48, 32
    x = W.sequence_inputs(B, H, T, d, d, torch.float32, seed=9)
    xd = to_dev(x)
    hp = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"])
    C = torch.zeros((B, H, d, d), device="cuda")
    n = torch.zeros((B, H, d), device="cuda")
    m = torch.full((B, H), -math.inf, device="cuda")
    hr = M.step_seq(C, n, m, xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"])
    torch.cuda.synchronize()
    assert rel_err(hr, hp.double().cpu().numpy()) <= TOL_F32


def test_step_seq_empty_run_is_a_no_op(M):
    w = W.StepWorkload("t", 1, 1, 16, 16, torch.float32)
    x = to_dev(W.step_seq_inputs(w, 0, seed=1))
    before = {k: x[k].clone() for k in ("C", "n", "m")}
    h = run(M, x, True)
    assert h.shape == (1, 1, 0, 16)
    for k in before:
        assert torch.equal(before[k], x[k])
