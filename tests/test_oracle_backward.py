"""Pins of the oracle's parallel backward (part 28/30 eqs 87-105).

The backward is checked against central finite differences of the oracle's
own stabilized forward, in fp64, on small random inputs: for the scalar
L = sum(dH (.) H~(q, k, v, i~, f~)), every printed gradient must equal the
numerical derivative of L.  A dropped term, a wrong sign or index, or a
transposed operand anywhere in eqs (87)-(105) fails this.  The floor case
(|b| below exp(-m), where eq (90) zeroes db) is covered by the second case.
"""
import numpy as np
import pytest
import torch

import oracle
from mlstm_matrix_memory_gb300 import workloads as W


def loss(x, dh):
    h, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    return float(np.sum(h * dh))


def numeric_grad(x, dh, name, eps=1e-6):
    base = {k: oracle.f64(v) for k, v in x.items()}
    g = np.zeros_like(base[name])
    flat = g.reshape(-1)
    for idx in range(flat.size):
        for sgn in (1.0, -1.0):
            y = {k: v.copy() for k, v in base.items()}
            y[name].reshape(-1)[idx] += sgn * eps
            flat[idx] += sgn * loss(y, dh) / (2 * eps)
    return g


@pytest.mark.parametrize("case", [
    dict(T=7, d=4, ig=(0.0, 1.0), fg=(3.0, 1.0), seed=1),       # |b| above the floor almost everywhere
    dict(T=9, d=3, ig=(-4.0, 0.5), fg=(0.0, 1.0), seed=2),      # small input gates: the floor engages on some rows
])
def test_backward_equals_finite_differences(case):
    x = W.sequence_inputs(1, 1, case["T"], case["d"], case["d"] + 1, torch.float64, seed=case["seed"],
                          ig=case["ig"], fg=case["fg"])
    dh = np.random.default_rng(case["seed"]).standard_normal((1, 1, case["T"], case["d"] + 1))
    dq, dk, dv, dig, dfg = oracle.parallel_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
    got = {"q": dq, "k": dk, "v": dv, "igate_pre": dig, "fgate_pre": dfg}
    for name, g in got.items():
        num = numeric_grad(x, dh, name)
        scale = max(1e-12, float(np.max(np.abs(num))))
        assert np.max(np.abs(g - num)) <= 1e-6 * scale, name


def test_backward_floor_case_reaches_the_floor():
    """The second case above really has rows on the floor (|b| < exp(-m))."""
    x = W.sequence_inputs(1, 1, 9, 3, 4, torch.float64, seed=2, ig=(-4.0, 0.5), fg=(0.0, 1.0))
    h, m, n = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert np.any(np.isclose(n, np.exp(-m), rtol=0, atol=0))


def test_backward_heads_are_independent():
    x = W.sequence_inputs(2, 2, 6, 4, 5, torch.float64, seed=4)
    dh = np.random.default_rng(4).standard_normal((2, 2, 6, 5))
    full = oracle.parallel_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
    one = oracle.parallel_backward(*(t[1:2, 0:1] for t in (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])),
                                   dh[1:2, 0:1])
    for a, b in zip(full, one):
        assert np.array_equal(a[1:2, 0:1], b)


def test_backward_exp_forget_equals_finite_differences():
    """With the exponential forget activation, d f~ = d fbar (eq 103 without the sigma factor)."""
    x = W.sequence_inputs(1, 1, 7, 3, 4, torch.float64, seed=11, ig=(0.0, 1.0), fg=(0.0, 0.5))
    dh = np.random.default_rng(11).standard_normal((1, 1, 7, 4))
    with oracle.forget_exp():
        got = oracle.parallel_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
        for name, g in zip(("q", "k", "v", "igate_pre", "fgate_pre"), got):
            num = numeric_grad(x, dh, name)
            assert np.max(np.abs(g - num)) <= 1e-6 * max(1e-12, float(np.max(np.abs(num)))), name



def test_recurrent_backward_exp_forget_finite_differences():
    """Eqs (59)-(70) with the exponential forget activation (gamma = exp)
    against central differences of the unstabilized recurrence."""
    import pins
    x = W.sequence_inputs(1, 1, 6, 3, 4, torch.float64, seed=13, ig=(-0.5, 1.0), fg=(0.0, 0.3), with_ogate=True)
    dh = np.random.default_rng(13).standard_normal((1, 1, 6, 4))
    with oracle.forget_exp():
        got = oracle.recurrent_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh, x["ogate_pre"])
        pins._recurrent_fd(x, dh, got, 1e-6, "exp forget recurrent backward")


@pytest.mark.parametrize("exp_forget", [False, True], ids=["sigmoid", "exp"])
@pytest.mark.parametrize("case", [
    dict(B=2, H=2, T=40, dqk=8, dv=6, ig=(0.0, 1.0), fg=(3.0, 1.0), seed=3),
    dict(B=1, H=2, T=33, dqk=4, dv=8, ig=(-4.0, 0.5), fg=(0.0, 1.0), seed=4),   # the normaliser floor engages
])
def test_gate_gradients_from_the_products(case, exp_forget):
    """The gate gradients equal sums of the key and query products' own
    gradients: with S_ij = s q_i.k_j, the total gradient reaching D~_ij is
    dS_ij S_ij, so the column sums give d i~_j = k_j.dk_j and the row sums
    give q_i.dq_i, and d log f_t = sum_{u >= t} (q_u.dq_u - k_u.dk_u) (the
    rows from t on, minus the columns from t on).  The kernels of the
    recurrent backward rest on these; here they tie the oracle's gate
    gradients (eqs 101-105) to its dq, dk (eqs 98-99), two separate
    derivations."""
    c = case
    fg = (-0.05, 0.05) if exp_forget else c["fg"]
    x = W.sequence_inputs(c["B"], c["H"], c["T"], c["dqk"], c["dv"], torch.float32, seed=c["seed"], ig=c["ig"],
                          fg=fg)
    dh = np.random.default_rng(c["seed"]).standard_normal((c["B"], c["H"], c["T"], c["dv"]))
    if exp_forget:
        with oracle.forget_exp():
            dq, dk, _, dig, dfg = oracle.parallel_backward(x["q"], x["k"], x["v"], x["igate_pre"],
                                                           x["fgate_pre"], dh)
    else:
        dq, dk, _, dig, dfg = oracle.parallel_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
    q, k = oracle.f64(x["q"]), oracle.f64(x["k"])
    f = oracle.f64(x["fgate_pre"])
    col = np.einsum("bhtd,bhtd->bht", k, dk)
    row = np.einsum("bhtd,bhtd->bht", q, dq)
    dlogf = np.cumsum((row - col)[..., ::-1], axis=-1)[..., ::-1]
    dlogf_dpre = 1.0 if exp_forget else 1.0 / (1.0 + np.exp(f))          # d log sigmoid(x)/dx = sigmoid(-x)
    scale = max(1.0, float(np.max(np.abs(dig))), float(np.max(np.abs(dfg))))
    np.testing.assert_allclose(dig, col, rtol=0, atol=1e-10 * scale)
    np.testing.assert_allclose(dfg, dlogf_dpre * dlogf, rtol=0, atol=1e-10 * scale)
