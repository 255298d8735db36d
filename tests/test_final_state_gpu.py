"""GPU parity of the parallel-to-recurrent hand-off (mlstm_parallel_final_state)
against the fp64 oracle's recurrence, and the prefill -> generation join."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, TOL_F32, rel_err, to_dev
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


def final_state(M, xd):
    B, H, T, _ = xd["q"].shape
    ws = torch.empty(M.parallel_fwd_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
    M.gate_prep(xd["igate_pre"], xd["fgate_pre"], ws)
    C, n, m = M.parallel_final_state(xd["k"], xd["v"], ws)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    return C.cpu(), n.cpu(), m.cpu()


# (B, H, T, d_qk, d_v, dtype, input-gate and forget-gate distributions):
# short and ragged sequences, token ranges split over several CTAs, the
# long-memory gates of the long-sequence workload
SHAPES = [
    (1, 1, 64, 16, 16, torch.float32, (0.0, 1.0), (3.0, 1.0)),
    (2, 2, 300, 64, 48, torch.float32, (0.0, 1.0), (3.0, 1.0)),
    (1, 2, 1000, 128, 128, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),
    (1, 1, 5, 8, 8, torch.float32, (0.0, 1.0), (3.0, 1.0)),
    (1, 1, 777, 96, 200, torch.bfloat16, (0.0, 2.0), (5.0, 1.0)),
    (1, 2, 2048, 384, 384, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),
    (8, 4, 256, 384, 384, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),    # one token range per tile (96 tiles)
    (2, 2, 192, 512, 128, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),    # d_qk 512: 64 n chunks per tile
    # how the (tile, 64-token chunk) units fall on the CTAs of a 152-SM part:
    (76, 4, 128, 64, 128, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),    # 304 tiles: two whole tiles per CTA
    (25, 8, 128, 128, 128, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),   # ranges on tile bounds, two pieces per CTA
    (10, 5, 150, 128, 128, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),   # ranges cut tiles: pieces added in C
    (2, 3, 500, 128, 192, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),    # d_v 192: half of the last row tile unused
    (5, 1, 448, 384, 384, torch.bfloat16, (0.0, 1.0), (3.0, 1.0)),    # three row-tile groups, heads cut between CTAs
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(str(v) for v in s[:5]) + f"-{s[5]}")
def test_final_state_matches_recurrence(M, shape):
    B, H, T, dqk, dv, dtype, ig, fg = shape
    x = W.sequence_inputs(B, H, T, dqk, dv, dtype, seed=T + dqk, ig=ig, fg=fg)
    C, n, m = final_state(M, to_dev(x))
    _, wC, wn, wm = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"])
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert rel_err(C, wC) <= tol
    assert rel_err(n, wn) <= tol
    assert np.max(np.abs(m.numpy() - wm)) <= 1e-4 * max(1.0, float(np.max(np.abs(wm))))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_prefill_then_generation(M, dtype):
    """Parallel forward over a prompt, hand-off, then recurrent steps over the
    rest: the same outputs and final state as the recurrence over the whole
    sequence."""
    B, H, T1, L2, d = 2, 2, 200, 24, 64
    x = W.sequence_inputs(B, H, T1 + L2, d, d, dtype, seed=21, with_ogate=True)
    xd = to_dev(x)
    pre = {k: v[:, :, :T1].contiguous() for k, v in xd.items()}
    gen = {k: v[:, :, T1:].contiguous() for k, v in xd.items()}
    ws = torch.empty(M.parallel_fwd_workspace_bytes(B, H, T1), dtype=torch.uint8, device="cuda")
    h1 = M.parallel_fwd(pre["q"], pre["k"], pre["v"], pre["igate_pre"], pre["fgate_pre"], workspace=ws)
    C, n, m = M.parallel_final_state(pre["k"], pre["v"], ws)
    h2 = M.step_seq(C, n, m, gen["q"], gen["k"], gen["v"], gen["igate_pre"], gen["fgate_pre"], gen["ogate_pre"])
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    og = np.concatenate([np.ones((B, H, T1, d)) * np.inf, oracle.f64(x["ogate_pre"][:, :, T1:])], axis=2)
    wh, wC, wn, wm = oracle.recurrent_stabilized(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], og)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert rel_err(h1, wh[:, :, :T1]) <= tol          # sigma(+inf) = 1: no output gate on the prompt
    assert rel_err(h2, wh[:, :, T1:]) <= tol
    assert rel_err(C, wC) <= tol
    assert rel_err(n, wn) <= tol
    assert np.max(np.abs(m.cpu().numpy() - wm)) <= 1e-4 * max(1.0, float(np.max(np.abs(wm))))


@pytest.mark.parametrize("name", ["mlstm125m_B8_H4_T2048_d384_bf16", "mlstm350m_B4_H4_T2048_d512_bf16"])
def test_final_state_full_size_sampled_heads(M, name):
    """The benchmark's hand-off launch at full size (every head computed in one
    call, heads cut between CTAs and added in C), checked on sampled heads
    against the oracle's recurrence over those heads' inputs (heads are
    independent)."""
    w = W.PARALLEL_WORKLOADS[name]
    x = W.parallel_inputs(w, 0)
    C, n, m = final_state(M, to_dev(x))
    for b, h in ((0, 0), (w.B - 1, w.H - 1), (w.B // 2, 1)):
        xs = {k: v[b:b + 1, h:h + 1] for k, v in x.items()}
        _, wC, wn, wm = oracle.recurrent_stabilized(xs["q"], xs["k"], xs["v"], xs["igate_pre"], xs["fgate_pre"])
        assert rel_err(C[b:b + 1, h:h + 1], wC) <= TOL_BF16
        assert rel_err(n[b:b + 1, h:h + 1], wn) <= TOL_BF16
        assert np.max(np.abs(m[b:b + 1, h:h + 1].numpy() - wm)) <= 1e-4 * max(1.0, float(np.max(np.abs(wm))))
