"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

TOL_F32 = 1e-4     # max abs error / max|h| for fp32 inputs
TOL_BF16 = 2e-2    # max abs error / max|h| for bf16 q, k, v with fp32 gates and accumulation


def tol_for(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def rel_err(got, want) -> float:
    got = got.float().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    want = np.asarray(want, dtype=np.float64)
    scale = float(np.max(np.abs(want))) if want.size else 1.0
    if scale == 0.0:
        scale = 1.0
    return float(np.max(np.abs(got.astype(np.float64) - want))) / scale


def to_dev(x, dev="cuda"):
    return {k: v.to(dev) for k, v in x.items()}


def sample_rows(B, H, T, n_random=24, seed=0):
    """Flat (bh, i) row indices: first/last rows, 128-row tile edges, random rows."""
    rng = np.random.default_rng(seed)
    base = {0, 1, 2, T - 1, T - 2, T - 3}
    for e in range(64, T, 64):
        base.update({e - 1, e, e + 1})
    base = sorted(i for i in base if 0 <= i < T)
    rows = []
    for bh in range(B * H):
        pick = list(base)
        if len(pick) > 40:
            pick = list(rng.choice(pick, 40, replace=False))
        pick += list(rng.integers(0, T, n_random))
        rows += [bh * T + int(i) for i in sorted(set(pick))]
    return np.array(rows, dtype=np.int64)
