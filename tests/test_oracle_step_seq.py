"""The oracle's multi-token step against its independent recurrent routine.

``oracle.step_seq`` applies the single-step routine token by token to a given
state.  From the fresh state (C = 0, n = 0, m = -inf) it must reproduce
``oracle.recurrent_stabilized``, which runs the same recurrence of
"xLSTM: Extended Long Short-Term Memory" (part 28/30, eqs 59-70) as a
separate C loop; and a run split in two must equal the run in one piece.
"""
import math

import numpy as np
import torch

import oracle
from mlstm_matrix_memory_gb300 import workloads as W


def _fresh(B, H, dqk, dv):
    return (np.zeros((B, H, dv, dqk)), np.zeros((B, H, dqk)), np.full((B, H), -math.inf))


def test_step_seq_from_fresh_state_is_the_recurrence():
    x = W.sequence_inputs(2, 2, 23, 16, 12, torch.float32, seed=3, with_ogate=True)
    C0, n0, m0 = _fresh(2, 2, 16, 12)
    h, C, n, m = oracle.step_seq(C0, n0, m0, x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], x["ogate_pre"])
    wh, wC, wn, wm = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"],
                                                 x["ogate_pre"])
    scale = np.max(np.abs(wh))
    assert np.max(np.abs(h - wh)) <= 1e-12 * scale
    assert np.max(np.abs(C - wC)) <= 1e-12 * np.max(np.abs(wC))
    assert np.max(np.abs(n - wn)) <= 1e-12 * np.max(np.abs(wn))
    assert np.max(np.abs(m - wm)) <= 1e-12 * np.max(np.abs(wm))


def test_step_seq_split_run_carries_the_state():
    w = W.StepWorkload("t", 1, 3, 24, 8, torch.float32, state_std=0.3)
    x = W.step_seq_inputs(w, 11, seed=5)
    a = (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], x["o"])
    h, C, n, m = oracle.step_seq(x["C"], x["n"], x["m"], *a)
    cut = 4
    first = [t[:, :, :cut] for t in a]
    rest = [t[:, :, cut:] for t in a]
    h1, C1, n1, m1 = oracle.step_seq(x["C"], x["n"], x["m"], *first)
    h2, C2, n2, m2 = oracle.step_seq(C1, n1, m1, *rest)
    assert np.array_equal(np.concatenate([h1, h2], axis=2), h)
    assert np.array_equal(C2, C) and np.array_equal(n2, n) and np.array_equal(m2, m)
    # the given state is not modified
    assert np.array_equal(oracle.f64(x["C"]), oracle.f64(W.step_seq_inputs(w, 11, seed=5)["C"]))
