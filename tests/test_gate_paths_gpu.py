"""The public forward call (gate pass, then the fused kernel started under
programmatic dependent launch) must equal, bit for bit, the two phases called
separately (``gate_prep`` then ``parallel_fwd_gated``): the outputs and the
gate terms it leaves in the workspace, which the hand-off and the backward
read.  Both forget activations; the CTA-pair kernel forced.
"""
import pytest
import torch

from gpu_util import to_dev
from mlstm_matrix_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import mlstm_matrix_memory_gb300 as M
    M.library()
    return M


SHAPES = [
    (2, 2, 600, 128, 128),
    (1, 3, 2048, 384, 384),     # the 125M-scale layer's head shape
    (1, 1, 333, 512, 512),      # two d_v splits: both scan the same rows
    (2, 1, 2047, 256, 256),
    (1, 2, 129, 128, 128),      # one pair, second CTA nearly empty
    (1, 1, 2100, 128, 128),
]


@pytest.mark.parametrize("forget", ["sigmoid", "exp"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_one_call_equals_separate_phases(M, shape, forget, monkeypatch):
    monkeypatch.setenv("MLSTM_TC_VARIANT", "pair")
    B, H, T, dqk, dv = shape
    fg = (0.0, 1.0) if forget == "exp" else (3.0, 1.0)    # exp forget: log f = f~, kept moderate
    x = to_dev(W.sequence_inputs(B, H, T, dqk, dv, torch.bfloat16, seed=T + dv, fg=fg))
    nbytes = M.parallel_fwd_workspace_bytes(B, H, T)
    ws1 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ws2 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    h1, m1, n1 = M.parallel_fwd(x["q"], x["k"], x["v"], x["igate_pre"], x["fgate_pre"], workspace=ws1,
                                return_mn=True, forget=forget)
    M.gate_prep(x["igate_pre"], x["fgate_pre"], ws2, forget=forget)
    h2 = torch.empty_like(h1)
    m2 = torch.empty_like(m1)
    n2 = torch.empty_like(n1)
    M.parallel_fwd_gated(x["q"], x["k"], x["v"], ws2, h2, m2, n2)
    torch.cuda.synchronize()
    assert M.last_device_status() == 0
    assert torch.equal(ws1, ws2)          # a2, p2, m for every token
    assert torch.equal(h1, h2)
    assert torch.equal(m1, m2)
    assert torch.equal(n1, n2)
