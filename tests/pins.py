"""Pins of the fp64 oracle to facts other than itself.

Each ``pin_*`` function raises AssertionError when the oracle built with the
given planted ``mutation`` (0 = the real oracle) violates a fact fixed by the
pages or by mathematics:

* hand-derived worked examples (tests/golden/*.txt, closed forms);
* the parallel and recurrent formulations agree ("xLSTM", part 28/30,
  "Parallel mLSTM Forward Pass": the recurrence can be reformulated in
  parallel form and used recurrently after training);
* stabilized and unstabilized forms give identical H~ (below eq 77);
* forget gate 1 and input pre-activation 0 reduce the cell to causal linear
  attention with the max(|.|, 1) normalizer (textbook closed form);
* T = 1 closed form h = v (s q.k) / max(|s q.k|, exp(-i~));
* the row max of D~ equals cs_i + max_{j<=i}(i~_j - cs_j) (prefix-max identity);
* shifting all i~ by c leaves H~ unchanged wherever the floor is not engaged;
* heads are independent (part 17/30: multiple heads = multiple cells);
* the output gate is sigma(o~) applied elementwise (eq 78);
* the stored recurrent state is only defined up to (C e^c, n e^c, m - c).

tests/test_oracle_pins.py runs them on the real oracle and
tests/test_oracle_mutations.py checks each planted mistake trips one of them.
"""
import math

import numpy as np
import torch

import oracle
from golden_loader import load
from mlstm_matrix_memory_gb300 import workloads as W

TOL = 1e-11


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    return float(np.max(np.abs(a - b))) / scale if a.size else 0.0


def _close(a, b, tol=TOL, what=""):
    r = _rel(a, b)
    assert r <= tol, f"{what}: rel err {r:.3e} > {tol:.1e}"


def _seq(seed, B=1, H=2, T=48, dqk=16, dv=12, ig=(0.0, 1.0), fg=(3.0, 1.0), og=False):
    return W.sequence_inputs(B, H, T, dqk, dv, torch.float32, seed=seed, ig=ig, fg=fg,
                             with_ogate=og)


def _args(x):
    return (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])


def log_sigmoid_np(x):
    return -np.logaddexp(0.0, -np.asarray(x, dtype=np.float64))


# --------------------------------------------------------------------------
def pin_golden_parallel(mutation=0):
    for c in load("parallel_hand.txt"):
        T, dqk, dv = c["T"], c["dqk"], c["dv"]
        sh = lambda a, d: np.asarray(a, dtype=np.float64).reshape(1, 1, T, d)
        h, m, n = oracle.parallel_stabilized(sh(c["q"], dqk), sh(c["k"], dqk), sh(c["v"], dv),
                                             np.reshape(c["ig"], (1, 1, T)),
                                             np.reshape(c["fg"], (1, 1, T)), mutation=mutation)
        _close(h.reshape(-1), c["h"], 1e-13, c["name"] + " h")
        _close(m.reshape(-1), c["m"], 1e-13, c["name"] + " m")
        _close(n.reshape(-1), c["n"], 1e-13, c["name"] + " n")


def pin_golden_step(mutation=0):
    for c in load("step_hand.txt"):
        a = lambda key: np.asarray(c[key], dtype=np.float64)
        o = None if c["o"][0] is None else a("o").reshape(1, 1, 1)
        h, C, n, m = oracle.step(a("C").reshape(1, 1, 1, 1), a("n").reshape(1, 1, 1),
                                 a("m").reshape(1, 1), a("q").reshape(1, 1, 1), a("k").reshape(1, 1, 1),
                                 a("v").reshape(1, 1, 1), a("ig").reshape(1, 1), a("fg").reshape(1, 1),
                                 o, mutation=mutation)
        _close(h.reshape(-1), c["h"], 1e-13, c["name"] + " h")
        _close(C.reshape(-1), c["C_new"], 1e-13, c["name"] + " C")
        _close(n.reshape(-1), c["n_new"], 1e-13, c["name"] + " n")
        _close(m.reshape(-1), c["m_new"], 1e-13, c["name"] + " m")


def pin_parallel_equals_recurrent(mutation=0):
    for seed, kw in ((0, {}), (1, dict(dqk=8, dv=24, og=True)), (2, dict(T=64, ig=(0.0, 2.0), fg=(1.0, 2.0))),
                     (3, dict(T=33, ig=(-5.0, 1.0)))):
        x = _seq(seed, **kw)
        og = x.get("ogate_pre")
        hp, mp, _ = oracle.parallel_stabilized(*_args(x), og, mutation=mutation)
        hr, _, _, mr = oracle.recurrent_stabilized(*_args(x), og, mutation=mutation)
        _close(hp, hr, TOL, f"parallel vs recurrent seed {seed}")
        # the recurrent stabilizer after the last token is the last row's max (eq 80)
        _close(mp[..., -1], mr, TOL, f"final m seed {seed}")


def pin_stabilized_equals_unstabilized(mutation=0):
    x = _seq(4, T=40, ig=(0.0, 1.0), fg=(1.0, 1.5))
    hs, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    hu = oracle.parallel_unstabilized(*_args(x), mutation=mutation)
    hru = oracle.recurrent_unstabilized(*_args(x), mutation=mutation)
    _close(hs, hu, TOL, "parallel stabilized vs unstabilized")
    _close(hs, hru, TOL, "parallel stabilized vs recurrent unstabilized")


def pin_linear_attention_closed_form(mutation=0):
    """f~ = +inf (forget gate 1), i~ = 0: causal linear attention,
    H_i = sum_{j<=i} (s q_i.k_j) v_j / max(|sum_{j<=i} s q_i.k_j|, 1)."""
    for seed, (T, dqk, dv) in ((5, (30, 16, 16)), (6, (17, 4, 9))):
        x = _seq(seed, T=T, dqk=dqk, dv=dv)
        ig = torch.zeros_like(x["igate_pre"])
        fg = torch.full_like(x["fgate_pre"], math.inf)
        q, k, v = (oracle.f64(x[n]) for n in ("q", "k", "v"))
        S = np.einsum("bhid,bhjd->bhij", q, k) / math.sqrt(dqk)
        S = S * np.tril(np.ones((T, T)))
        want = (S @ v) / np.maximum(np.abs(S.sum(-1, keepdims=True)), 1.0)
        h, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], ig, fg, mutation=mutation)
        _close(h, want, TOL, "linear attention closed form")
        hr, _, _, _ = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], ig, fg, mutation=mutation)
        _close(hr, want, TOL, "linear attention closed form (recurrent)")


def pin_single_step_closed_form(mutation=0):
    """T = 1: h = v (s q.k) / max(|s q.k|, exp(-i~))."""
    x = _seq(7, B=2, H=3, T=1, dqk=16, dv=8, ig=(0.0, 3.0))
    q, k, v = (oracle.f64(x[n]) for n in ("q", "k", "v"))
    ig = oracle.f64(x["igate_pre"])
    sqk = np.einsum("bhtd,bhtd->bht", q, k) / 4.0
    want = v * (sqk / np.maximum(np.abs(sqk), np.exp(-ig)))[..., None]
    h, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    _close(h, want, TOL, "T=1 closed form")
    hr, _, _, _ = oracle.recurrent_stabilized(*_args(x), mutation=mutation)
    _close(hr, want, TOL, "T=1 closed form (recurrent)")


def pin_prefix_max_identity(mutation=0):
    x = _seq(8, H=3, T=50, ig=(0.0, 2.0), fg=(2.0, 2.0))
    ig, fg = oracle.f64(x["igate_pre"]), oracle.f64(x["fgate_pre"])
    cs = np.cumsum(log_sigmoid_np(fg), axis=-1)
    want = cs + np.maximum.accumulate(ig - cs, axis=-1)
    _, m, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    _close(m, want, TOL, "prefix-max identity")


def pin_input_shift_invariance(mutation=0):
    x = _seq(9, T=40)
    base, m0, n0 = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    outs = []
    for c in (20.0, 40.0):
        h, m, n = oracle.parallel_stabilized(x["q"], x["k"], x["v"], oracle.f64(x["igate_pre"]) + c,
                                             x["fgate_pre"], mutation=mutation)
        _close(m, m0 + c, TOL, "m shifts with i~")
        outs.append(h)
    _close(outs[0], outs[1], TOL, "floor-free invariance")
    free = n0 > np.exp(-m0) * (1 + 1e-9)          # rows where the floor was not engaged
    assert free.any() and (~free).any()
    _close(base[free], outs[0][free], TOL, "unchanged where the floor is not engaged")


def pin_head_independence(mutation=0):
    x = _seq(10, B=2, H=3, T=20)
    h, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    perm = torch.tensor([2, 0, 1])
    xp = {k: v[:, perm] for k, v in x.items()}
    hp, _, _ = oracle.parallel_stabilized(*_args(xp), mutation=mutation)
    assert np.array_equal(hp, h[:, perm.numpy()])
    one = {k: v[1:2, 2:3] for k, v in x.items()}
    h1, _, _ = oracle.parallel_stabilized(*_args(one), mutation=mutation)
    assert np.array_equal(h1, h[1:2, 2:3])


def pin_output_gate(mutation=0):
    x = _seq(11, T=24, og=True)
    og = oracle.f64(x["ogate_pre"])
    h0, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    hg, _, _ = oracle.parallel_stabilized(*_args(x), og, mutation=mutation)
    _close(hg, h0 / (1.0 + np.exp(-og)), TOL, "output gate")


def pin_rows_match_full(mutation=0):
    x = _seq(12, B=2, H=2, T=37)
    h, m, n = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    rows = np.array([0, 5, 36, 37, 74, 147, 100])
    hr, mr, nr = oracle.parallel_rows(*_args(x), rows, mutation=mutation)
    assert np.array_equal(hr, h.reshape(-1, h.shape[-1])[rows])
    assert np.array_equal(mr, m.reshape(-1)[rows]) and np.array_equal(nr, n.reshape(-1)[rows])


def pin_step_state_scale_invariance(mutation=0):
    """(C e^c, n e^c, m - c) is the same true state: the step's h must not change,
    and the new state must be the same true state."""
    w = W.StepWorkload("t", 3, 2, 16, 8, torch.float32, state_std=0.5)
    x = W.step_inputs(w, 13)
    args = (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], x["o"])
    h0, C0, n0, m0 = oracle.step(x["C"], x["n"], x["m"], *args, mutation=mutation)
    for c in (3.0, -2.0):
        C = oracle.f64(x["C"]) * math.exp(c)
        n = oracle.f64(x["n"]) * math.exp(c)
        m = oracle.f64(x["m"]) - c
        h1, C1, n1, m1 = oracle.step(C, n, m, *args, mutation=mutation)
        _close(h1, h0, TOL, f"step h invariant (c={c})")
        _close(C1 * np.exp(m1)[..., None, None], C0 * np.exp(m0)[..., None, None], TOL, "true C")
        _close(n1 * np.exp(m1)[..., None], n0 * np.exp(m0)[..., None], TOL, "true n")


def pin_step_continues_sequence(mutation=0):
    x = _seq(14, B=1, H=2, T=21, dqk=8, dv=8)
    h_all, _, _, _ = oracle.recurrent_stabilized(*_args(x), mutation=mutation)
    pre = {k: v[:, :, :20] for k, v in x.items()}
    _, C, n, m = oracle.recurrent_stabilized(*_args(pre), mutation=mutation)
    last = {k: v[:, :, 20] for k, v in x.items()}
    h, _, _, _ = oracle.step(C, n, m, last["q"], last["k"], last["v"], last["igate_pre"],
                             last["fgate_pre"], None, mutation=mutation)
    _close(h, h_all[:, :, 20], TOL, "step continues the sequence")
    hp, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    _close(h, hp[:, :, 20], TOL, "step continues the parallel form")


def pin_brute_force_dense(mutation=0):
    """Dense T x T matrices of eqs (71)-(73), (76) built with explicit products."""
    x = _seq(15, B=1, H=1, T=12, dqk=4, dv=3, fg=(1.0, 1.0))
    q, k, v = (oracle.f64(x[n])[0, 0] for n in ("q", "k", "v"))
    ig, fg = oracle.f64(x["igate_pre"])[0, 0], oracle.f64(x["fgate_pre"])[0, 0]
    T = q.shape[0]
    sig = 1.0 / (1.0 + np.exp(-fg))
    F = np.zeros((T, T))
    for i in range(T):
        for j in range(i + 1):
            F[i, j] = np.prod(sig[j + 1:i + 1])
    D = F * np.exp(ig)[None, :]
    Ct = (q @ k.T) / 2.0 * D
    want = (Ct / np.maximum(np.abs(Ct.sum(1, keepdims=True)), 1.0)) @ v
    h, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    _close(h[0, 0], want, TOL, "dense brute force")


def pin_backward_finite_differences(mutation=0):
    """Every gradient of eqs (87)-(105) equals the central finite difference of
    the (unmutated) forward, for L = sum(dH (.) H~), on a case with negative
    row sums and floored rows."""
    # seed 9: three rows with b < 0 above the floor and four rows on the floor
    x = W.sequence_inputs(1, 1, 8, 3, 4, torch.float64, seed=9, ig=(-2.0, 1.5), fg=(0.5, 1.0))
    dh = np.random.default_rng(9).standard_normal((1, 1, 8, 4))
    got = dict(zip(("q", "k", "v", "igate_pre", "fgate_pre"),
                   oracle.parallel_backward(*_args(x), dh, mutation=mutation)))
    base = {k: oracle.f64(v) for k, v in x.items()}
    eps = 1e-6
    for name, g in got.items():
        num = np.zeros_like(base[name])
        for idx in range(num.size):
            for sgn in (1.0, -1.0):
                y = {k: v.copy() for k, v in base.items()}
                y[name].reshape(-1)[idx] += sgn * eps
                hh, _, _ = oracle.parallel_stabilized(*_args(y))
                num.reshape(-1)[idx] += sgn * float(np.sum(hh * dh)) / (2 * eps)
        _close(g, num, 1e-6, f"backward d{name} vs finite differences")


def _recurrent_fd(x, dh, got, tol, what):
    base = {k: oracle.f64(v) for k, v in x.items()}
    eps = 1e-6
    for name, g in zip(("q", "k", "v", "igate_pre", "fgate_pre", "ogate_pre"), got):
        num = np.zeros_like(base[name])
        for idx in range(num.size):
            for sgn in (1.0, -1.0):
                y = {k: v.copy() for k, v in base.items()}
                y[name].reshape(-1)[idx] += sgn * eps
                hh = oracle.recurrent_unstabilized(y["q"], y["k"], y["v"], y["igate_pre"], y["fgate_pre"],
                                                   y["ogate_pre"])
                num.reshape(-1)[idx] += sgn * float(np.sum(hh * dh)) / (2 * eps)
        _close(g, num, tol, f"{what} d{name} vs finite differences")


def pin_recurrent_backward_finite_differences(mutation=0):
    """Every gradient of the recurrent backward, eqs (59)-(70), equals the
    central finite difference of the (unmutated) unstabilized recurrence for
    L = sum(dh (.) h), output gate included, on a case whose n^T q takes both
    signs above 1 in magnitude and stays below 1 on one step (all three
    branches of the normalizer max(|n^T q|, 1))."""
    x = W.sequence_inputs(1, 1, 7, 3, 4, torch.float64, seed=32, ig=(0.5, 1.0), fg=(1.0, 1.0), with_ogate=True)
    dh = np.random.default_rng(32).standard_normal((1, 1, 7, 4))
    got = oracle.recurrent_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh, x["ogate_pre"],
                                    mutation=mutation)
    _recurrent_fd(x, dh, got, 1e-6, "recurrent backward")


def pin_recurrent_backward_equals_parallel(mutation=0):
    """The recurrent (eqs 59-70) and parallel (eqs 87-105) backward passes
    give the same gradients where the two forwards are the same function: no
    output gate, sigma forget gate."""
    x = W.sequence_inputs(2, 1, 20, 8, 6, torch.float64, seed=17, ig=(0.0, 1.0), fg=(3.0, 1.0))
    dh = np.random.default_rng(17).standard_normal((2, 1, 20, 6))
    rec = oracle.recurrent_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh,
                                    mutation=mutation)[:5]
    par = oracle.parallel_backward(*_args(x), dh, mutation=mutation)
    for name, a, b in zip(("dq", "dk", "dv", "d_igate", "d_fgate"), rec, par):
        _close(a, b, 1e-9, f"recurrent vs parallel backward {name}")


def pin_forget_exp_variant(mutation=0):
    """The exponential forget activation: with f~ = 0 it gives f = 1 exactly,
    the same cell as the sigma activation with f~ = +inf; and its parallel and
    recurrent forms agree (part 28/30: gamma is sigma or exp)."""
    x = _seq(21, T=24, fg=(0.0, 1.0))
    x0 = dict(x, fgate_pre=torch.zeros_like(x["fgate_pre"]))
    xinf = dict(x, fgate_pre=torch.full_like(x["fgate_pre"], math.inf))
    with oracle.forget_exp(mutation):
        h_exp, _, _ = oracle.parallel_stabilized(*_args(x0), mutation=mutation)
        hp, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
        hr, _, _, _ = oracle.recurrent_stabilized(*_args(x), mutation=mutation)
        hu = oracle.parallel_unstabilized(*_args(x), mutation=mutation)
    h_sig, _, _ = oracle.parallel_stabilized(*_args(xinf), mutation=mutation)
    _close(h_exp, h_sig, TOL, "exp forget with f~=0 equals sigma forget with f~=+inf")
    _close(hp, hr, 1e-10, "exp forget: parallel equals recurrent")
    _close(hp, hu, 1e-10, "exp forget: stabilized equals unstabilized")
    # the exp variant really differs from sigma on generic f~
    h_sig_x, _, _ = oracle.parallel_stabilized(*_args(x), mutation=mutation)
    assert _rel(hp, h_sig_x) > 1e-3, "exp forget indistinguishable from sigma forget"


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
