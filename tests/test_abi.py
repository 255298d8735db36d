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


def test_step_seq_validation(lib):
    def seq(C=A, n=A, m=A, q=A, k=A, v=A, o=None, ig=A, fg=A, h=A, B=2, H=2, L=4, dqk=64, dv=64, dt=1):
        return lib.mlstm_step_seq(C, n, m, q, k, v, o, ig, fg, h, B, H, L, dqk, dv, dt, None)
    assert seq(L=-1) == -1
    assert seq(dqk=20) == -1
    assert seq(dv=0) == -1
    assert seq(dt=5) == -3
    assert seq(n=A + 4) == -2
    assert seq(k=0) == -1
    assert seq(L=0) == 0                      # an empty run leaves the state as it is
    assert seq(B=0) == 0


def test_final_state_validation(lib):
    def fs(k=A, v=A, ws=A, wsb=1 << 20, C=A, n=A, m=A, B=1, H=2, T=16, dqk=64, dv=64, dt=1):
        return lib.mlstm_parallel_final_state(k, v, ws, wsb, C, n, m, B, H, T, dqk, dv, dt, None)
    assert fs(dqk=0) == -1
    assert fs(dt=2) == -3
    assert fs(T=0) == -1                      # a state after no tokens is not defined here
    assert fs(C=A + 4) == -2
    assert fs(ws=0) == -7
    assert fs(wsb=64) == -7
    assert fs(m=0) == -1
    assert fs(B=0) == 0


def test_host_call_validation(lib):
    assert lib.mlstm_parallel_fwd_host_workspace(0, 1, 8, 64, 64, 1) == 0
    assert lib.mlstm_parallel_fwd_host_workspace(1, 1, 8, 64, 64, 9) == 0
    need = lib.mlstm_parallel_fwd_host_workspace(2, 3, 100, 64, 64, 1)
    assert need >= 2 * 100 * (4 * 64 * 2)     # two slots of one head's q, k, v and h at least (6 chunks of 1 head)

    def host(ws=A, wsb=need, B=2, H=3, T=100, dqk=64, dv=64, dt=1, q=A):
        return lib.mlstm_parallel_fwd_host(q, A, A, A, A, A, B, H, T, dqk, dv, dt, ws, wsb, None)
    assert host(dqk=600) == -1
    assert host(dt=4) == -3
    assert host(wsb=need - 1) == -7
    assert host(ws=A + 16) == -2              # the workspace must be 256-byte aligned
    assert host(q=0) == -1
    assert host(T=0) == 0


def test_recurrent_bwd_validation(lib):
    need = lib.mlstm_recurrent_bwd_workspace(2, 3, 100, 64, 96)
    # per-CTA dq and dk shares (two 64-row CTAs), then three per-token scalars
    assert need >= 2 * 2 * 600 * 64 * 4 + 3 * 600 * 4
    assert lib.mlstm_recurrent_bwd_workspace(0, 3, 100, 64, 96) == 0
    assert lib.mlstm_recurrent_bwd_workspace(1, 1, 8, 64, 600) == 0

    from mlstm_matrix_memory_gb300.binding import _Options as Opt

    def rb(q=A, ws=A, wsb=need, B=2, H=3, T=100, dqk=64, dv=96, dt=1, dog=None, og=None):
        opt = Opt(0, 0, og)
        return lib.mlstm_recurrent_bwd(q, A, A, A, A, A, A, A, A, A, A, dog, B, H, T, dqk, dv, dt, ws, wsb,
                                       ctypes.byref(opt), None)
    assert rb(dqk=20) == -1                   # d_qk a multiple of 8
    assert rb(dv=513) == -1
    assert rb(dt=3) == -3
    assert rb(q=A + 4) == -2
    assert rb(q=0) == -1
    assert rb(og=A) == -1                     # an output gate needs its gradient's buffer
    assert rb(wsb=need - 1) == -7
    assert rb(ws=A + 16) == -2
    assert rb(T=0) == 0


def test_parallel_bwd_validation(lib):
    big = lib.mlstm_parallel_bwd_workspace(2, 3, 100, 1)
    ex = lib.mlstm_parallel_bwd_workspace_ex(2, 3, 100, 64, 64, 1)
    assert 0 < ex <= big                      # the exact size never exceeds the size for either path
    assert lib.mlstm_parallel_bwd_workspace_ex(2, 3, 100, 64, 600, 1) == 0
    assert lib.mlstm_parallel_bwd_workspace_ex(2, 3, 0, 64, 64, 1) == 0
    assert lib.mlstm_parallel_bwd_workspace_ex(2, 3, 100, 64, 64, 5) == 0

    def bwd(T=100, dqk=64, dv=64, dt=1, ws=A, wsb=big, q=A):
        return lib.mlstm_parallel_bwd(q, A, A, A, A, A, A, A, A, A, A, 2, 3, T, dqk, dv, dt, ws, wsb, None)

    def saved(h=A, n=A, b=A, T=100, dt=1, ws=A, wsb=big):
        return lib.mlstm_parallel_bwd_saved(A, A, A, A, A, A, h, n, b, A, A, A, A, A, 2, 3, T, 64, 64, dt, ws,
                                            wsb, None)
    assert bwd(dqk=0) == -1
    assert bwd(dv=513) == -1
    assert bwd(dt=4) == -3
    assert bwd(q=0) == -1
    assert bwd(ws=0) == -7
    assert bwd(ws=A + 16) == -2               # 256-byte aligned workspace
    assert bwd(T=0) == 0
    assert saved(h=0) == -1                   # the saved forward outputs are required
    assert saved(b=0) == -1
    assert saved(dt=7) == -3
    assert saved(T=0) == 0


def test_parallel_bwd_opt_validation(lib):
    from mlstm_matrix_memory_gb300.binding import _Options as Opt
    plain = Opt(0, 0, None, None)
    gated = Opt(0, 1, A, None)
    base = lib.mlstm_parallel_bwd_workspace_opt(2, 3, 100, 64, 64, 1, ctypes.byref(plain))
    assert base == lib.mlstm_parallel_bwd_workspace_ex(2, 3, 100, 64, 64, 1)
    with_og = lib.mlstm_parallel_bwd_workspace_opt(2, 3, 100, 64, 64, 1, ctypes.byref(gated))
    assert with_og >= base + 2 * 3 * 100 * 64 * 2        # at least one [B,H,T,d_v] bf16 buffer more
    assert lib.mlstm_parallel_bwd_workspace_opt(2, 3, 100, 64, 64, 1, None) == base
    assert lib.mlstm_parallel_bwd_workspace_opt(2, 3, 100, 64, 600, 1, ctypes.byref(plain)) == 0

    def bo(opt, dog=A, h=None, n=None, b=None, T=100, dt=1, wsb=with_og):
        return lib.mlstm_parallel_bwd_opt(A, A, A, A, A, A, h, n, b, A, A, A, A, A, dog, 2, 3, T, 64, 64, dt, A,
                                          wsb, ctypes.byref(opt), None)
    assert bo(gated, dog=None) == -1          # an output gate needs somewhere for its gradient
    assert bo(plain, h=A) == -1               # the saved forward outputs come all three or none
    assert bo(plain, h=A, n=A) == -1
    assert bo(gated, dt=9) == -3
    assert bo(gated, T=0) == 0
    assert bo(gated, wsb=base) == -7          # the path's workspace alone is too small with a gate


def test_plain_parallel_validation(lib):
    def pf(q=A, h=A, B=1, T=8, dqk=64, dv=64, dt=1, ws=A, wsb=1 << 20):
        return lib.mlstm_parallel_fwd(q, A, A, A, A, h, None, None, B, 1, T, dqk, dv, dt, ws, wsb, None)
    assert pf(dqk=0) == -1
    assert pf(dv=520) == -1
    assert pf(dt=7) == -3
    assert pf(q=A + 4) == -2
    assert pf(h=0) == -1
    assert pf(wsb=64) == -7
    assert pf(B=0) == 0


def test_gate_prep_validation(lib):
    from mlstm_matrix_memory_gb300.binding import _Options as Opt
    opt = Opt(0, 1, None, None)                # exponential forget gate: same argument rules

    def gp(ig=A, fg=A, B=2, T=100, ws=A, wsb=1 << 20, with_opt=False):
        if with_opt:
            return lib.mlstm_gate_prep_opt(ig, fg, B, 3, T, ws, wsb, ctypes.byref(opt), None)
        return lib.mlstm_gate_prep(ig, fg, B, 3, T, ws, wsb, None)
    need = lib.mlstm_parallel_fwd_workspace(2, 3, 100)
    for w in (False, True):
        assert gp(B=-1, with_opt=w) == -1
        assert gp(T=0, with_opt=w) == 0
        assert gp(ig=0, with_opt=w) == -1
        assert gp(fg=0, with_opt=w) == -1
        assert gp(ws=0, with_opt=w) == -7
        assert gp(wsb=need - 1, with_opt=w) == -7
        assert gp(ws=A + 8, with_opt=w) == -2


def test_gated_and_options_validation(lib):
    from mlstm_matrix_memory_gb300.binding import _Options as Opt

    def gated(q=A, h=A, T=8, dqk=64, dv=64, dt=1, ws=A, wsb=1 << 20, algo=0):
        return lib.mlstm_parallel_fwd_gated(q, A, A, h, None, None, 1, 1, T, dqk, dv, dt, ws, wsb, algo, None)
    assert gated(dqk=513) == -1
    assert gated(dqk=12) == -1                 # bf16 rows must be 16 bytes
    assert gated(dt=2) == -3
    assert gated(algo=9) == -1
    assert gated(h=A + 8) == -2
    assert gated(ws=0) == -7
    assert gated(T=0) == 0

    def opt_fwd(opt, dqk=64, dv=64, dt=1):
        return lib.mlstm_parallel_fwd_opt(A, A, A, A, A, A, None, None, 1, 1, 8, dqk, dv, dt, A, 1 << 20,
                                          ctypes.byref(opt), None)
    assert opt_fwd(Opt(9, 0, None, None)) == -1                    # unknown kernel choice
    assert opt_fwd(Opt(0, 0, A + 2, None)) == -2                   # output gate not 16-byte aligned
    assert opt_fwd(Opt(2, 0, None, None), dqk=40, dv=40) == -6     # tensor cores forced on d = 40
    assert opt_fwd(Opt(0, 0, None, None), dt=7) == -3


def test_noalloc_validation(lib):
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.mlstm_parallel_fwd_noalloc.argtypes = [vp] * 8 + [i] * 6 + [vp]
    lib.mlstm_parallel_fwd_noalloc.restype = i

    def na(B=1, T=8, dqk=64, dv=64, dt=1, H=1):
        return lib.mlstm_parallel_fwd_noalloc(A, A, A, A, A, A, None, None, B, H, T, dqk, dv, dt, None)
    assert na(B=-1) == -1
    big = (1 << 31) - 1
    assert na(B=big, H=big, T=big) == -1       # B*H beyond int: rejected before any product is formed
    assert na(B=1 << 16, H=1 << 16) == -1
    assert na(B=1 << 20, T=1 << 21) == -1      # B*H*T beyond 2^40, as mlstm_parallel_fwd
    assert na(dqk=0) == -1                      # shape checks come before the device scratch
    assert na(dt=5) == -3
    assert na(dv=12) == -1
    assert na(T=0) == 0
    assert na(T=1 << 20) == -7                 # beyond the fixed scratch


def test_step_seq_opt_validation(lib):
    from mlstm_matrix_memory_gb300.binding import _Options as Opt
    opt = Opt(0, 1, None, None)

    def ss(C=A, q=A, L=4, dqk=64, dv=64, dt=1):
        return lib.mlstm_step_seq_opt(C, A, A, q, A, A, None, A, A, A, 2, 2, L, dqk, dv, dt, ctypes.byref(opt),
                                      None)
    assert ss(L=-1) == -1
    assert ss(dqk=12) == -1
    assert ss(dv=600) == -1
    assert ss(dt=3) == -3
    assert ss(C=A + 4) == -2
    assert ss(q=0) == -1
    assert ss(L=0) == 0
