"""GPU parity of the tcgen05/TMEM tensor-core kernel (bf16 q, k, v) against the
fp64 oracle: several tile counts with ragged tails, every d_v tiling (one CTA
with 128-key tiles, one CTA with 64-key tiles, two CTAs splitting d_v), and
the full-size workloads on sampled rows in the launch configuration the
benchmark times."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, rel_err, sample_rows, to_dev
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


def run(M, x, algo="tc"):
    xd = to_dev(x)
    out = M.parallel_fwd(xd["q"], xd["k"], xd["v"], xd["igate_pre"], xd["fgate_pre"], return_mn=True, algo=algo)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    return out


def args(x):
    return (x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])


SHAPES = [
    (1, 1, 128, 64, 64),      # one tile
    (1, 2, 384, 128, 128),    # three query tiles: a CTA pair plus a pair whose second CTA is past T
    (2, 1, 600, 384, 384),
    (1, 2, 300, 64, 64),      # ragged tail, 128-key tiles
    (2, 1, 257, 128, 128),
    (1, 1, 520, 256, 256),
    (1, 2, 200, 384, 384),    # 64-key tiles
    (1, 1, 390, 128, 320),
    (1, 1, 333, 512, 512),    # d_v split over two CTAs
    (1, 1, 130, 192, 448),
    (1, 1, 64, 512, 512),     # shorter than one tile
]


@pytest.fixture(params=["auto", "single", "pair"])
def variant(request, monkeypatch):
    """auto: the library's choice; single: the one-CTA kernel; pair: the CTA-pair
    kernel (cta_group::2), skipped for shapes it does not tile."""
    if request.param == "auto":
        monkeypatch.delenv("MLSTM_TC_VARIANT", raising=False)
    else:
        monkeypatch.setenv("MLSTM_TC_VARIANT", request.param)
    return request.param


def pair_tiles(dqk, dv):
    return dqk % 128 == 0 and dqk <= 512 and ((dv <= 384 and dv % 128 == 0) or dv == 512)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tc_vs_oracle(M, shape, variant):
    B, H, T, dqk, dv = shape
    if variant == "pair" and not pair_tiles(dqk, dv):
        pytest.skip("the pair kernel tiles d_qk and each d_v slice in multiples of 128")
    x = W.sequence_inputs(B, H, T, dqk, dv, torch.bfloat16, seed=T + dqk)
    h, m, n = run(M, x)
    wh, wm, wn = oracle.parallel_stabilized(*args(x))
    assert rel_err(h, wh) <= TOL_BF16
    assert np.max(np.abs(m.cpu().numpy() - wm) / np.maximum(1.0, np.abs(wm))) <= 1e-5
    assert np.max(np.abs(n.cpu().numpy() - wn) / np.abs(wn)) <= 2e-2


def test_tc_matches_simt(M):
    x = W.sequence_inputs(2, 2, 700, 128, 128, torch.bfloat16, seed=21)
    h_tc, _, _ = run(M, x, "tc")
    h_simt, _, _ = run(M, x, "simt")
    assert rel_err(h_tc, h_simt.double().cpu().numpy()) <= TOL_BF16


def test_tc_heads_are_independent_bit_exact(M):
    x = W.sequence_inputs(1, 4, 260, 64, 64, torch.bfloat16, seed=22)
    h, _, _ = run(M, x)
    perm = torch.tensor([3, 1, 0, 2])
    hp, _, _ = run(M, {k: v[:, perm].contiguous() for k, v in x.items()})
    assert torch.equal(hp.cpu(), h.cpu()[:, perm])


@pytest.mark.parametrize("gates", [((20.0, 1.0), (3.0, 1.0)), ((-30.0, 3.0), (0.0, 3.0)), ((0.0, 2.0), (8.0, 1.0))])
def test_tc_gate_regimes(M, gates):
    x = W.sequence_inputs(1, 2, 400, 128, 128, torch.bfloat16, seed=23, ig=gates[0], fg=gates[1])
    h, _, _ = run(M, x)
    wh, _, _ = oracle.parallel_stabilized(*args(x))
    assert rel_err(h, wh) <= TOL_BF16


@pytest.mark.parametrize("w", [W.L125M, W.L350M, W.LONG], ids=lambda w: w.name)
def test_full_size_sampled_rows(M, w, variant):
    """Full B, H, T, d as benchmarked; the oracle evaluates sampled rows one by one."""
    x = W.parallel_inputs(w, 0)
    h, m, n = run(M, x)
    rows = sample_rows(w.B, w.H, w.T, n_random=8 if w.T > 4096 else 16)
    if w.T > 4096:                    # long sequences: keep the oracle within seconds
        rng = np.random.default_rng(1)
        rows = np.sort(rng.choice(rows, 160, replace=False))
    wh, wm, wn = oracle.parallel_rows(*args(x), rows)
    got = h.reshape(-1, w.d_v)[torch.from_numpy(rows).cuda()].cpu()
    assert rel_err(got, wh) <= TOL_BF16
    gm = m.reshape(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.max(np.abs(gm - wm) / np.maximum(1.0, np.abs(wm))) <= 1e-5
