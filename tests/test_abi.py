"""The C-ABI library loads, exports every symbol include/mlstm.h declares, and
rejects bad arguments on the host with the documented status codes (no GPU
work: every call here fails validation before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mlstm_matrix_memory_gb300 import build
    build.build()
    import mlstm_matrix_memory_gb300 as M
    return M.library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mlstm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mlstm_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.mlstm_status_str(code).decode() != "unknown status"
    assert lib.mlstm_status_str(42).decode() == "unknown status"
    assert lib.mlstm_version() >= 100


def test_workspace_size(lib):
    assert lib.mlstm_parallel_fwd_workspace(8, 4, 2048) == 3 * 8 * 4 * 2048 * 4
    assert lib.mlstm_parallel_fwd_workspace(1, 1, 3) == 3 * 256
    assert lib.mlstm_parallel_fwd_workspace(-1, 1, 3) == 0


A = 1 << 20        # fake, 16-byte aligned "device" addresses: never dereferenced


def fwd(lib, q=A, k=A, v=A, ig=A, fg=A, h=A, B=1, H=1, T=8, dqk=64, dv=64, dt=1, ws=A, wsb=1 << 20, algo=0):
    return lib.mlstm_parallel_fwd_ex(q, k, v, ig, fg, h, None, None, B, H, T, dqk, dv, dt, ws, wsb, algo, None)


def test_parallel_validation(lib):
    assert fwd(lib, dqk=0) == -1
    assert fwd(lib, dv=513) == -1
    assert fwd(lib, dqk=12) == -1            # bf16 rows must be 16 bytes
    assert fwd(lib, dt=7) == -3
    assert fwd(lib, B=-1) == -1
    assert fwd(lib, q=A + 2) == -2
    assert fwd(lib, h=A + 8) == -2
    assert fwd(lib, q=0) == -1
    assert fwd(lib, ws=0) == -7
    assert fwd(lib, wsb=16) == -7
    assert fwd(lib, algo=9) == -1
    assert fwd(lib, T=0, q=0, k=0, v=0, ig=0, fg=0, h=0) == 0      # empty input is a no-op
    assert fwd(lib, B=0) == 0


def test_step_validation(lib):
    def step(C=A, n=A, m=A, q=A, k=A, v=A, o=None, ig=A, fg=A, h=A, B=2, H=2, dqk=64, dv=64, dt=1):
        return lib.mlstm_step(C, n, m, q, k, v, o, ig, fg, h, B, H, dqk, dv, dt, None)
    assert step(dqk=0) == -1
    assert step(dqk=20) == -1
    assert step(dv=1024) == -1
    assert step(dt=3) == -3
    assert step(C=A + 4) == -2
    assert step(q=0) == -1
    assert step(B=0) == 0


def test_binding_rejects_cpu_tensors(lib):
    import torch
    import mlstm_matrix_memory_gb300 as M
    x = torch.zeros(1, 1, 4, 16)
    g = torch.zeros(1, 1, 4)
    with pytest.raises(ValueError):
        M.parallel_fwd(x, x, x, g, g)


def test_spin_limit_roundtrip(lib):
    old = lib.mlstm_set_spin_limit(5)
    assert lib.mlstm_set_spin_limit(0) == 5
    lib.mlstm_set_spin_limit(old)
