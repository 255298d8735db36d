"""The closed form behind the parallel-to-recurrent hand-off, checked against
the oracle's stabilized recurrence ("xLSTM: Extended Long Short-Term Memory",
part 28/30, eqs 59-70 unrolled from C = 0, n = 0, m = -inf).

Unrolling gives, with log-forget terms lf_t (log sigmoid of the forget
pre-activation, or the pre-activation itself for the exponential forget gate):
  D~_Tj = sum_{k=j+1..T} lf_k + igate_j        (the last row of eq 79),
  m_T   = max_j D~_Tj                          (eq 80),
  C_T   = sum_j exp(D~_Tj - m_T) v_j (s k_j)^T,   n_T = sum_j exp(D~_Tj - m_T) s k_j,
with s = 1/sqrt(d_qk): the state the recurrence carries, stabilized by
exp(-m_T).  Here the closed form is evaluated in numpy (fp64) from the gate
definitions alone and compared with what the oracle's step-by-step
recurrence ends with.  A wrong sum range (k from j instead of j+1), a missing
input-gate term or a missing key scaling each fails it."""
import numpy as np
import pytest
import torch

import oracle
from mlstm_matrix_memory_gb300 import workloads as W


def _log_sigmoid(x):
    return np.minimum(x, 0.0) - np.log1p(np.exp(-np.abs(x)))


def _closed_form(x, exp_forget):
    q, k, v = (x[n].double().numpy() for n in ("q", "k", "v"))
    ig = x["igate_pre"].double().numpy()
    fg = x["fgate_pre"].double().numpy()
    B, H, T, dqk = k.shape
    s = 1.0 / np.sqrt(dqk)
    lf = fg if exp_forget else _log_sigmoid(fg)
    # suffix sums: sum_{k=j+1..T-1} lf_k (0-based tokens), then the input gate
    suffix = np.cumsum(lf[..., ::-1], axis=-1)[..., ::-1] - lf
    D = suffix + ig                                   # [B, H, T]
    m = D.max(axis=-1)                                # [B, H]
    w = np.exp(D - m[..., None])                      # [B, H, T]
    C = np.einsum("bht,bhtv,bhtk->bhvk", w, v, s * k)
    n = np.einsum("bht,bhtk->bhk", w, s * k)
    return C, n, m


@pytest.mark.parametrize("exp_forget", [False, True], ids=["sigmoid", "exp"])
@pytest.mark.parametrize("case", [
    (1, 1, 1, 4, 4, (0.0, 1.0), (3.0, 1.0)),       # one token: C = v (s k)^T, m = igate
    (2, 3, 37, 8, 6, (0.0, 1.0), (3.0, 1.0)),
    (1, 2, 64, 16, 8, (0.0, 2.0), (-1.0, 1.0)),    # forgetful gates: the max moves along the sequence
    (1, 1, 50, 8, 8, (-3.0, 0.5), (5.0, 1.0)),     # long memory
], ids=lambda c: "x".join(str(v) for v in c[:5]))
def test_final_state_closed_form_equals_recurrence(case, exp_forget):
    B, H, T, dqk, dv, ig, fg = case
    if exp_forget:
        fg = (-0.05, 0.05)                            # exp forget gates must stay near or below 1
    x = W.sequence_inputs(B, H, T, dqk, dv, torch.float32, seed=T + dqk, ig=ig, fg=fg)
    if exp_forget:
        with oracle.forget_exp():
            _, C, n, m = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    else:
        _, C, n, m = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    Cc, nc, mc = _closed_form(x, exp_forget)
    np.testing.assert_allclose(m, mc, rtol=0, atol=1e-12)
    np.testing.assert_allclose(C, Cc, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(n, nc, rtol=1e-11, atol=1e-12)
