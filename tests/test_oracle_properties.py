"""Randomised checks of the oracle's identities (hypothesis draws shapes,
seeds and gate regimes): the parallel and recurrent forms agree, the
stabilized and unstabilized forms agree, and the recurrent and parallel
backward passes agree, as the pins check on fixed cases."""
import numpy as np
import pytest
import torch

import oracle
from mlstm_matrix_memory_gb300 import workloads as W

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

shapes = st.tuples(st.integers(1, 2), st.integers(1, 2), st.integers(1, 24), st.sampled_from([2, 4, 8]),
                   st.sampled_from([1, 3, 8]))
gates = st.tuples(st.floats(-2.0, 2.0), st.floats(0.2, 2.0), st.floats(-1.0, 5.0), st.floats(0.2, 2.0))


def _inputs(shape, g, seed, ogate=False):
    B, H, T, dqk, dv = shape
    return W.sequence_inputs(B, H, T, dqk, dv, torch.float64, seed=seed, ig=(g[0], g[1]), fg=(g[2], g[3]),
                             with_ogate=ogate)


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b))) / max(float(np.max(np.abs(b))), 1e-300)


@settings(max_examples=40, deadline=None)
@given(shapes, gates, st.integers(0, 10_000))
def test_parallel_equals_recurrent(shape, g, seed):
    x = _inputs(shape, g, seed)
    hp, mp, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    hr, _, _, mr = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert _rel(hp, hr) <= 1e-10
    assert np.allclose(mp[..., -1], mr, rtol=1e-12, atol=1e-12)


@settings(max_examples=40, deadline=None)
@given(shapes, gates, st.integers(0, 10_000))
def test_stabilized_equals_unstabilized(shape, g, seed):
    x = _inputs(shape, g, seed)
    hs, _, _ = oracle.parallel_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    hu = oracle.parallel_unstabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    assert _rel(hs, hu) <= 1e-9


@settings(max_examples=25, deadline=None)
@given(shapes, st.integers(0, 10_000))
def test_recurrent_backward_equals_parallel_backward(shape, seed):
    x = _inputs(shape, (0.0, 1.0, 3.0, 1.0), seed)
    B, H, T, dqk, dv = shape
    dh = np.random.default_rng(seed).standard_normal((B, H, T, dv))
    rec = oracle.recurrent_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)[:5]
    par = oracle.parallel_backward(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], dh)
    for a, b in zip(rec, par):
        assert np.max(np.abs(a - b)) <= 1e-8 * max(1.0, float(np.max(np.abs(b))))
