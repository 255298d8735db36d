"""GPU parity of the parallel backward (mlstm_parallel_bwd, _opt) against the
fp64 oracle's eqs (87)-(105), each gradient within the forward's tolerances
(relative to its own largest entry).  bf16 cases run the tensor-core tile
path; fp32 cases, and bf16 ones with MLSTM_BWD_PATH=blas in the environment,
run the CUDA-core path (the library's batched causal GEMM kernel).  The
output gate (eq 78) and the exponential forget activation (eq 70) are checked
against the oracle's backpropagation through time, which is pinned to the
oracle's parallel backward and to finite differences."""
import subprocess
import sys
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, TOL_F32, rel_err
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


# (B, H, T, d_qk, d_v, dtype, input-gate, forget-gate distributions)
CASES = [
    (1, 1, 64, 16, 16, torch.float32, (0.0, 1.0), (3.0, 1.0)),
    (2, 2, 130, 64, 48, torch.float32, (-2.0, 1.5), (0.5, 1.0)),     # floored rows and negative row sums
    (1, 2, 300, 64, 64, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),
    (1, 1, 777, 128, 96, torch.bfloat16, (0.0, 2.0), (5.0, 1.0)),     # long-memory gates
    (1, 1, 2048, 384, 384, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),   # one head of the 125M-scale layer
    (2, 3, 50, 40, 24, torch.bfloat16, (-2.0, 1.5), (0.5, 1.0)),      # one partial tile, d not a multiple of 64
    (1, 1, 129, 64, 64, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),      # a second tile row of one query
    (1, 2, 600, 128, 256, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),    # CTA-pair products, odd block count
    (2, 1, 129, 128, 128, torch.bfloat16, (-2.0, 1.5), (0.5, 1.0)),   # CTA-pair products, one-query block
    (1, 2, 576, 128, 128, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),    # CTA-pair products, A through the 4-D view, half a last key block
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(v) for v in c[:5]) + f"-{c[5]}")
def test_bwd_matches_oracle(M, case):
    B, H, T, dqk, dv, dtype, ig, fg = case
    x = W.sequence_inputs(B, H, T, dqk, dv, dtype, seed=T + dv, ig=ig, fg=fg)
    dh = torch.randn((B, H, T, dv), generator=torch.Generator().manual_seed(T)).to(dtype)
    xd = {k: v.cuda() for k, v in x.items()}
    got = M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh.cuda())
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    want = oracle.parallel_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for name, g, w in zip(("dq", "dk", "dv", "d_igate", "d_fgate"), got, want):
        assert rel_err(g, w) <= tol, name


@pytest.mark.parametrize("shape", [(1, 2, 300, 64, 64), (2, 2, 1024, 384, 384)])
def test_bwd_with_saved_forward(M, shape):
    """mlstm_parallel_bwd_saved with the forward's own H~, n and signed b gives
    bit for bit the gradients of the recomputing backward; |b| equals n where
    the normalizer floor exp(-m) is not engaged."""
    B, H, T, dqk, dv = shape
    x = W.sequence_inputs(B, H, T, dqk, dv, torch.bfloat16, seed=T + 3)
    dh = torch.randn((B, H, T, dv), generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    xd = {k: v.cuda() for k, v in x.items()}
    dhd = dh.cuda()
    h, m, n, b = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], return_stats=True)
    got = M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dhd, saved=(h, n, b))
    ref = M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dhd)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    for name, g, r in zip(("dq", "dk", "dv", "d_igate", "d_fgate"), got, ref):
        assert torch.equal(g, r), name
    above = n > torch.exp(-m) * 1.001
    assert torch.allclose(b.abs()[above], n[above], rtol=1e-6, atol=0)
    want = oracle.parallel_backward(x["q"][:1, :1], x["k"][:1, :1], x["v"][:1, :1], x["igate_pre"][:1, :1],
                                    x["fgate_pre"][:1, :1], dh[:1, :1])
    for name, g, w in zip(("dq", "dk", "dv", "d_igate", "d_fgate"), got, want):
        assert rel_err(g[:1, :1], w) <= TOL_BF16, name


def test_bwd_full_size_sampled_heads(M):
    """The 125M-scale layer (B=8, H=4, T=2048, d=384, bf16) in one launch, as
    the benchmark times it; the first and last heads against the oracle."""
    B, H, T, d = 8, 4, 2048, 384
    x = W.sequence_inputs(B, H, T, d, d, torch.bfloat16, seed=11)
    dh = torch.randn((B, H, T, d), generator=torch.Generator().manual_seed(11)).to(torch.bfloat16)
    xd = {k: v.cuda() for k, v in x.items()}
    got = M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh.cuda())
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    for b, h in ((0, 0), (B - 1, H - 1)):
        sl = lambda t: t[b:b + 1, h:h + 1]
        want = oracle.parallel_backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["igate_pre"]), sl(x["fgate_pre"]),
                                        sl(dh))
        for name, g, w in zip(("dq", "dk", "dv", "d_igate", "d_fgate"), got, want):
            assert rel_err(sl(g), w) <= TOL_BF16, f"head ({b},{h}) {name}"


# (B, H, T, d_qk, d_v, dtype): small enough for the oracle's recurrent backward
OPT_CASES = [
    (1, 2, 150, 64, 64, torch.bfloat16),     # tensor-core path
    (1, 1, 97, 32, 48, torch.float32),       # CUDA-core path, ragged tiles
    (2, 1, 130, 64, 64, torch.bfloat16),
]


@pytest.mark.parametrize("forget", ["sigmoid", "exp"])
@pytest.mark.parametrize("case", OPT_CASES, ids=lambda c: "x".join(str(v) for v in c[:5]) + f"-{c[5]}")
def test_bwd_output_gate_and_forget_activation(M, case, forget):
    B, H, T, dqk, dv, dtype = case
    fg = (0.0, 1.0) if forget == "exp" else (3.0, 1.0)
    x = W.sequence_inputs(B, H, T, dqk, dv, dtype, seed=T + 5, fg=fg, with_ogate=True)
    dh = torch.randn((B, H, T, dv), generator=torch.Generator().manual_seed(T + 5)).to(dtype)
    xd = {k: v.cuda() for k, v in x.items()}
    got = M.parallel_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh.cuda(),
                         ogate=xd["ogate_pre"], forget=forget)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    args = (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
    if forget == "exp":
        with oracle.forget_exp():
            want = oracle.recurrent_backward(*args, og=x["ogate_pre"])
    else:
        want = oracle.recurrent_backward(*args, og=x["ogate_pre"])
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for name, g, w in zip(("dq", "dk", "dv", "d_igate", "d_fgate", "d_ogate"), got, want):
        assert rel_err(g, w) <= tol, name


@pytest.mark.parametrize("forget", ["sigmoid", "exp"])
def test_bwd_opt_saved_forward(M, forget):
    """With an output gate and either forget activation, the backward given
    the forward's own H~ (no gate), n and b equals the recomputing one bit for
    bit on the tensor-core path."""
    B, H, T, d = 1, 2, 300, 128
    x = W.sequence_inputs(B, H, T, d, d, torch.bfloat16, seed=9, fg=(0.0, 1.0) if forget == "exp" else (3.0, 1.0),
                          with_ogate=True)
    dh = torch.randn((B, H, T, d), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    xd = {k: v.cuda() for k, v in x.items()}
    a = (xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"])
    h, m, n, b = M.parallel_fwd(*a, return_stats=True, forget=forget)
    got = M.parallel_bwd(*a, dh.cuda(), saved=(h, n, b), ogate=xd["ogate_pre"], forget=forget)
    ref = M.parallel_bwd(*a, dh.cuda(), ogate=xd["ogate_pre"], forget=forget)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    for name, g, r in zip(("dq", "dk", "dv", "d_igate", "d_fgate", "d_ogate"), got, ref):
        assert torch.equal(g, r), name


def test_bwd_cuda_core_path_bf16():
    """bf16 through the CUDA-core path (MLSTM_BWD_PATH=blas, read once per
    process, so in a child process) against the oracle."""
    code = (
        "import sys, torch; sys.path.insert(0, 'tests'); sys.path.insert(0, '.');"
        "import oracle, mlstm_matrix_memory_gb300 as M; from mlstm_matrix_memory_gb300 import workloads as W;"
        "from gpu_util import rel_err, TOL_BF16;"
        "x = W.sequence_inputs(1, 2, 200, 64, 64, torch.bfloat16, seed=4, with_ogate=True);"
        "dh = torch.randn((1, 2, 200, 64), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16);"
        "xd = {k: v.cuda() for k, v in x.items()};"
        "got = M.parallel_bwd(xd['q'], xd['k'], xd['v'], xd['igate_pre'], xd['fgate_pre'], dh.cuda(), ogate=xd['ogate_pre']);"
        "torch.cuda.synchronize(); assert M.last_device_status() == 0;"
        "want = oracle.recurrent_backward(x['q'], x['k'], x['v'], x['igate_pre'], x['fgate_pre'], dh, og=x['ogate_pre']);"
        "errs = [rel_err(g, w) for g, w in zip(got, want)]; print(errs); assert max(errs) <= TOL_BF16"
    )
    import os
    env = dict(os.environ, MLSTM_BWD_PATH="blas")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
