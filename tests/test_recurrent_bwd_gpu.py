"""GPU parity of the recurrent backward (mlstm_recurrent_bwd) against the fp64
oracle's backpropagation through time, eqs (59)-(70) of the recurrent form,
each gradient within the forward's tolerances (relative to its own largest
entry); at the full 125M-scale layer size, sampled heads against the oracle's
parallel backward (eqs 87-105), which the oracle pins equal to it."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, TOL_F32, rel_err
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "d_igate", "d_fgate", "d_ogate")


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


# (B, H, T, d_qk, d_v, dtype, input gate, forget gate, output gate, forget activation)
CASES = [
    (1, 1, 37, 16, 16, torch.float32, (0.0, 1.0), (3.0, 1.0), False, "sigmoid"),
    (2, 2, 130, 64, 48, torch.float32, (-2.0, 1.5), (0.5, 1.0), True, "sigmoid"),   # floored and negative n.q
    (1, 2, 100, 40, 72, torch.bfloat16, (0.0, 1.0), (0.0, 0.3), True, "exp"),       # ragged rows, exp forget
    (1, 1, 77, 24, 100, torch.float32, (0.0, 1.0), (3.0, 1.0), True, "sigmoid"),   # rows copied one by one
    (1, 1, 300, 64, 64, torch.bfloat16, (0.0, 1.0), (3.0, 1.0), False, "sigmoid"),
    (1, 1, 1, 64, 64, torch.float32, (0.0, 1.0), (3.0, 1.0), True, "sigmoid"),      # one token
    (1, 1, 17, 512, 512, torch.float32, (0.0, 1.0), (3.0, 1.0), True, "sigmoid"),  # largest head
    (1, 1, 512, 384, 384, torch.bfloat16, (0.0, 1.0), (3.0, 1.0), True, "sigmoid"),
    # enough heads that 96-row CTAs (12 warps) finish first: one full and one ragged CTA shape
    (8, 10, 40, 32, 96, torch.float32, (0.0, 1.0), (3.0, 1.0), True, "sigmoid"),
    (8, 10, 33, 64, 72, torch.bfloat16, (-1.0, 1.0), (0.0, 0.3), False, "exp"),
]


def _run(M, x, dh, og, forget):
    xd = {k: v.cuda() for k, v in x.items()}
    got = M.recurrent_bwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], dh.cuda(),
                          ogate=xd["ogate_pre"] if og else None, forget=forget)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    return got


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(v) for v in c[:5]) + f"-{c[5]}-{c[9]}"
                         + ("-og" if c[8] else ""))
def test_recurrent_bwd_matches_oracle(M, case):
    B, H, T, dqk, dv, dtype, ig, fg, og, forget = case
    x = W.sequence_inputs(B, H, T, dqk, dv, dtype, seed=T + dv + dqk, ig=ig, fg=fg, with_ogate=og)
    dh = torch.randn((B, H, T, dv), generator=torch.Generator().manual_seed(T + 1)).to(dtype)
    got = _run(M, x, dh, og, forget)
    if forget == "exp":
        with oracle.forget_exp():
            want = oracle.recurrent_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh,
                                             x["ogate_pre"] if og else None)
    else:
        want = oracle.recurrent_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh,
                                         x["ogate_pre"] if og else None)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for name, g, w in zip(NAMES, got, want):
        if w is None:
            assert g is None
            continue
        assert rel_err(g, w) <= tol, name


def test_recurrent_bwd_empty(M):
    x = W.sequence_inputs(1, 1, 0, 64, 64, torch.bfloat16, seed=1)
    dh = torch.zeros((1, 1, 0, 64), dtype=torch.bfloat16)
    got = _run(M, x, dh, False, "sigmoid")
    assert all(g is None or g.numel() == 0 for g in got)


def test_recurrent_bwd_full_size_sampled_heads(M):
    """The 125M-scale layer (B=8, H=4, T=2048, d=384, bf16) in one launch;
    two heads checked against the oracle's parallel backward."""
    B, H, T, d = 8, 4, 2048, 384
    x = W.sequence_inputs(B, H, T, d, d, torch.bfloat16, seed=5)
    dh = torch.randn((B, H, T, d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    got = _run(M, x, dh, False, "sigmoid")
    for b, h in ((0, 0), (B - 1, H - 1)):
        sl = lambda t: t[b:b + 1, h:h + 1]
        want = oracle.parallel_backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["igate_pre"]),
                                        sl(x["fgate_pre"]), sl(dh))
        for name, g, w in zip(NAMES, got, want):
            assert rel_err(sl(g), w) <= TOL_BF16, f"head ({b},{h}) {name}"
