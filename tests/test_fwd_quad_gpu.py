"""GPU parity of the four-CTA form of the fused forward (d_v = 512): two CTA
pairs over the same query rows, each owning half of d_v.  S is formed once per
key tile, by the pair whose turn it is; its P tile goes into that pair's TMEM
(the A operand of its own O product) and into the other pair's shared memory;
the row sums are exchanged before the epilogue.

Checked against the fp64 oracle and against the two-CTA form that forms S in
both d_v halves (MLSTM_TC_XCH=0).  The cases cover what the hand-offs depend
on: items of one key tile (one pair has no tile of its own), odd tile counts
(the pairs' turns shift from item to item), rows past T in the second CTA of
a pair, many items per cluster (several rounds of the schedule, so every
barrier runs through many phases and both S buffers are reused), the output
gate in the epilogue and the exponential forget activation.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, rel_err, to_dev
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


def args(x):
    return (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])


def run(M, xd, monkeypatch, xch, **kw):
    monkeypatch.setenv("MLSTM_TC_VARIANT", "pair")
    monkeypatch.setenv("MLSTM_TC_XCH", "1" if xch else "0")
    out = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], return_stats=True,
                         algo="tc", **kw)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    return out


SHAPES = [
    (1, 1, 1, 512, 512),        # one key tile: the second pair forms no S
    (1, 1, 100, 512, 512),
    (1, 2, 129, 512, 512),      # two tiles; the pair's second CTA holds one valid row
    (2, 1, 384, 128, 512),      # three tiles: the pairs' turns shift across items
    (1, 1, 777, 256, 512),      # five V granules: N=256 bursts alternate with N=128 pairs
    (1, 2, 500, 384, 512),      # d_qk 384: three K granules a tile
    (8, 8, 640, 512, 512),      # 192 items: several rounds of the schedule
    (1, 1, 2048, 512, 512),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_quad_vs_oracle_and_split(M, shape, monkeypatch):
    B, H, T, dqk, dv = shape
    x = W.sequence_inputs(B, H, T, dqk, dv, torch.bfloat16, seed=T + B * H)
    xd = to_dev(x)
    h, m, n, b = run(M, xd, monkeypatch, True)
    h2, m2, n2, b2 = run(M, xd, monkeypatch, False)
    if B * H * T <= 4096:
        wh, wm, wn = oracle.parallel_stabilized(*args(x))
        assert rel_err(h, wh) <= TOL_BF16
        assert np.max(np.abs(n.cpu().numpy() - wn) / np.abs(wn)) <= 2e-2
    # the same S and P tiles and products: only the order of the fp32 row sums
    # differs (each pair sums its own tiles, then the two partial sums are added)
    assert rel_err(h, h2.double().cpu().numpy()) <= 1e-2
    assert torch.equal(m, m2)
    assert np.max(np.abs(b.cpu().numpy() - b2.cpu().numpy()) / np.maximum(np.abs(n2.cpu().numpy()), 1e-30)) <= 1e-4


def test_quad_output_gate(M, monkeypatch):
    x = W.sequence_inputs(1, 2, 300, 512, 512, torch.bfloat16, seed=5, with_ogate=True)
    xd = to_dev(x)
    h, _, _, _ = run(M, xd, monkeypatch, True, ogate=xd["ogate_pre"])
    wh, _, _ = oracle.parallel_stabilized(*args(x), og=x["ogate_pre"])
    assert rel_err(h, wh) <= TOL_BF16


def test_quad_exp_forget(M, monkeypatch):
    x = W.sequence_inputs(1, 2, 520, 512, 512, torch.bfloat16, seed=6, fg=(0.0, 1.0))
    xd = to_dev(x)
    h, _, _, _ = run(M, xd, monkeypatch, True, forget="exp")
    with oracle.forget_exp():
        wh, _, _ = oracle.parallel_stabilized(*args(x))
    assert rel_err(h, wh) <= TOL_BF16


def test_quad_repeated_calls_bit_identical(M, monkeypatch):
    """Two launches over the same inputs give the same bits: no result depends
    on how the two pairs' hand-offs interleave."""
    x = W.sequence_inputs(4, 4, 1536, 512, 512, torch.bfloat16, seed=8)
    xd = to_dev(x)
    h1, m1, n1, b1 = run(M, xd, monkeypatch, True)
    h2, m2, n2, b2 = run(M, xd, monkeypatch, True)
    assert torch.equal(h1, h2) and torch.equal(n1, n2) and torch.equal(b1, b2)
