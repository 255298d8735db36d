"""GPU parity of the stabilized parallel forward against the fp64 oracle.

Tolerances (max abs error relative to max|h|): 1e-4 for fp32 inputs, 2e-2 for
bf16 q, k, v with fp32 gates and accumulation."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, TOL_F32, rel_err, sample_rows, to_dev, tol_for
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


def run(M, x, algo="auto", return_mn=True):
    xd = to_dev(x)
    out = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], return_mn=return_mn,
                         algo=algo)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    return out


def args(x):
    return (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])


def check_full(M, x, algo, tol):
    h, m, n = run(M, x, algo)
    wh, wm, wn = oracle.parallel_stabilized(*args(x))
    e = rel_err(h, wh)
    assert e <= tol, f"h rel err {e:.3e}"
    assert np.max(np.abs(m.cpu().numpy() - wm) / np.maximum(1.0, np.abs(wm))) <= 1e-5
    assert np.max(np.abs(n.cpu().numpy() - wn) / np.abs(wn)) <= max(tol, 1e-4) * 10
    return e


def test_tiny_fp32_vs_oracle(M):
    x = W.parallel_inputs(W.TINY, 0)
    e = check_full(M, x, "auto", TOL_F32)
    # the tiny workload exercises the exp(-m) floor on a share of its rows
    _, wm, wn = oracle.parallel_stabilized(*args(x))
    assert np.any(np.isclose(wn, np.exp(-wm)))
    assert e <= TOL_F32


def test_tiny_gpu_recurrent_equals_gpu_parallel(M):
    """T recurrent steps on the GPU from (C, n, m) = (0, 0, -inf) give the
    parallel form's outputs (the two formulations of part 28/30)."""
    x = W.parallel_inputs(W.TINY, 0)
    hp = run(M, x, return_mn=False).cpu()
    B, H, T, d = x["q"].shape
    dev = "cuda"
    C = torch.zeros(B, H, d, d, device=dev)
    n = torch.zeros(B, H, d, device=dev)
    m = torch.full((B, H), -math.inf, device=dev)
    xd = to_dev(x)
    hs = []
    for t in range(T):
        hs.append(M.step(C, n, m, xd["q"][:, :, t].contiguous(), xd["k"][:, :, t].contiguous(),
                         xd["v"][:, :, t].contiguous(), xd["igate_pre"][:, :, t].contiguous(),
                         xd["fgate_pre"][:, :, t].contiguous()).cpu())
    torch.cuda.synchronize()
    hr = torch.stack(hs, dim=2)
    assert rel_err(hr, hp.double().numpy()) <= TOL_F32


@pytest.mark.parametrize("shape", [(2, 3, 77, 32, 48), (1, 2, 130, 8, 8), (1, 1, 1, 16, 16), (3, 1, 33, 512, 64)])
def test_simt_fp32_shapes(M, shape):
    B, H, T, dqk, dv = shape
    x = W.sequence_inputs(B, H, T, dqk, dv, torch.float32, seed=sum(shape))
    check_full(M, x, "simt", TOL_F32)


@pytest.mark.parametrize("shape", [(1, 2, 100, 16, 16), (2, 1, 70, 24, 40), (1, 1, 129, 128, 128)])
def test_simt_bf16_shapes(M, shape):
    B, H, T, dqk, dv = shape
    x = W.sequence_inputs(B, H, T, dqk, dv, torch.bfloat16, seed=sum(shape))
    check_full(M, x, "simt", TOL_BF16)


@pytest.mark.parametrize("gates", [((60.0, 1.0), (3.0, 1.0)), ((-60.0, 1.0), (3.0, 1.0)),
                                   ((0.0, 5.0), (-4.0, 3.0)), ((0.0, 1.0), (12.0, 1.0))])
def test_extreme_gates(M, gates):
    ig, fg = gates
    x = W.sequence_inputs(1, 2, 96, 16, 16, torch.float32, seed=3, ig=ig, fg=fg)
    check_full(M, x, "auto", TOL_F32)


def test_zero_query_rows_give_zero(M):
    x = W.sequence_inputs(1, 1, 40, 16, 16, torch.float32, seed=4)
    x["q"][0, 0, 7] = 0.0
    x["q"][0, 0, 0] = 0.0
    h, _, _ = run(M, x)
    assert torch.all(h[0, 0, 7] == 0) and torch.all(h[0, 0, 0] == 0)
    wh, _, _ = oracle.parallel_stabilized(*args(x))
    assert rel_err(h, wh) <= TOL_F32


def test_heads_are_independent_bit_exact(M):
    x = W.sequence_inputs(2, 3, 50, 32, 32, torch.float32, seed=5)
    h = run(M, x, return_mn=False).cpu()
    perm = torch.tensor([2, 0, 1])
    hp = run(M, {k: v[:, perm].contiguous() for k, v in x.items()}, return_mn=False).cpu()
    assert torch.equal(hp, h[:, perm])


def test_empty_sequence_is_noop(M):
    x = W.sequence_inputs(1, 1, 0, 16, 16, torch.float32)
    xd = to_dev(x)
    h = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"])
    assert h.shape == (1, 1, 0, 16)
