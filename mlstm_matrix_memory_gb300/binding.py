"""ctypes binding to ``libmlstm.so`` (argument marshalling only).

Every step of the mLSTM path runs in the library's CUDA kernels; this module
checks tensor shapes, dtypes, devices and contiguity, hands raw device
pointers plus the current CUDA stream to the C-ABI declared in
``include/mlstm.h``, and turns non-zero status codes into ``MlstmError``.
There is no fallback: if the library is missing or no GPU is present, the
calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libmlstm.so"
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

MLSTM_F32, MLSTM_BF16 = 0, 1
ALGOS = {"auto": 0, "simt": 1, "tc": 2}
_DTYPES = {torch.float32: MLSTM_F32, torch.bfloat16: MLSTM_BF16}


class MlstmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_str(code)} ({code})")


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def library() -> ctypes.CDLL:
    """Load ``libmlstm.so`` (built by ``__graft_entry__.build()`` or
    ``mlstm_matrix_memory_gb300.build``).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m mlstm_matrix_memory_gb300.build`")
        lib = ctypes.CDLL(path)
        vp, i, sz, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
        lib.mlstm_parallel_fwd_workspace.argtypes = [i, i, i]
        lib.mlstm_parallel_fwd_workspace.restype = sz
        lib.mlstm_parallel_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]
        lib.mlstm_parallel_fwd.restype = i
        lib.mlstm_parallel_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, i, vp]
        lib.mlstm_parallel_fwd_ex.restype = i
        lib.mlstm_gate_prep.argtypes = [vp, vp, i, i, i, vp, sz, vp]
        lib.mlstm_gate_prep.restype = i
        lib.mlstm_parallel_fwd_gated.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, i, vp]
        lib.mlstm_parallel_fwd_gated.restype = i
        lib.mlstm_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
        lib.mlstm_step.restype = i
        lib.mlstm_step_seq.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.mlstm_step_seq.restype = i
        lib.mlstm_parallel_final_state.argtypes = [vp, vp, vp, sz, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.mlstm_parallel_final_state.restype = i
        lib.mlstm_parallel_fwd_host_workspace.argtypes = [i, i, i, i, i, i]
        lib.mlstm_parallel_fwd_host_workspace.restype = sz
        lib.mlstm_parallel_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]
        lib.mlstm_parallel_fwd_host.restype = i
        lib.mlstm_parallel_bwd_workspace.argtypes = [i, i, i, i]
        lib.mlstm_parallel_bwd_workspace.restype = sz
        lib.mlstm_parallel_bwd_workspace_ex.argtypes = [i] * 6
        lib.mlstm_parallel_bwd_workspace_ex.restype = sz
        lib.mlstm_parallel_bwd.argtypes = [vp] * 11 + [i] * 6 + [vp, sz, vp]
        lib.mlstm_parallel_bwd.restype = i
        lib.mlstm_parallel_bwd_saved.argtypes = [vp] * 14 + [i] * 6 + [vp, sz, vp]
        lib.mlstm_parallel_bwd_saved.restype = i
        op = ctypes.POINTER(_Options)
        lib.mlstm_parallel_fwd_opt.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, op, vp]
        lib.mlstm_parallel_fwd_opt.restype = i
        lib.mlstm_gate_prep_opt.argtypes = [vp, vp, i, i, i, vp, sz, op, vp]
        lib.mlstm_gate_prep_opt.restype = i
        lib.mlstm_step_seq_opt.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, op, vp]
        lib.mlstm_step_seq_opt.restype = i
        lib.mlstm_parallel_bwd_workspace_opt.argtypes = [i] * 6 + [op]
        lib.mlstm_parallel_bwd_workspace_opt.restype = sz
        lib.mlstm_parallel_bwd_opt.argtypes = [vp] * 15 + [i] * 6 + [vp, sz, op, vp]
        lib.mlstm_parallel_bwd_opt.restype = i
        lib.mlstm_recurrent_bwd_workspace.argtypes = [i, i, i, i, i]
        lib.mlstm_recurrent_bwd_workspace.restype = sz
        lib.mlstm_recurrent_bwd.argtypes = [vp] * 12 + [i] * 6 + [vp, sz, op, vp]
        lib.mlstm_recurrent_bwd.restype = i
        lib.mlstm_last_device_status.argtypes = [vp]
        lib.mlstm_last_device_status.restype = i
        lib.mlstm_set_spin_limit.argtypes = [ll]
        lib.mlstm_set_spin_limit.restype = ll
        lib.mlstm_status_str.argtypes = [i]
        lib.mlstm_status_str.restype = ctypes.c_char_p
        lib.mlstm_version.argtypes = []
        lib.mlstm_version.restype = i
        _lib = lib
        return lib


def status_str(code: int) -> str:
    try:
        return library().mlstm_status_str(int(code)).decode()
    except Exception:
        return "unknown status"


class _Options(ctypes.Structure):
    """``mlstm_options`` of include/mlstm.h."""
    _fields_ = [("algo", ctypes.c_int), ("forget_exp", ctypes.c_int), ("ogate_pre", ctypes.c_void_p),
                ("b_out", ctypes.c_void_p)]


FORGET = {"sigmoid": 0, "exp": 1}


def _options(algo: str = "auto", forget: str = "sigmoid", ogate: Optional[torch.Tensor] = None,
             b_out: Optional[torch.Tensor] = None) -> _Options:
    if forget not in FORGET:
        raise ValueError(f"forget must be one of {sorted(FORGET)}")
    return _Options(ALGOS[algo], FORGET[forget], None if ogate is None else ogate.data_ptr(),
                    None if b_out is None else b_out.data_ptr())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, name: str, shape, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def parallel_fwd_workspace_bytes(B: int, H: int, T: int) -> int:
    return int(library().mlstm_parallel_fwd_workspace(B, H, T))


def parallel_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, igate_pre: torch.Tensor,
                 fgate_pre: torch.Tensor, *, h: Optional[torch.Tensor] = None,
                 return_mn: bool = False, return_stats: bool = False, workspace: Optional[torch.Tensor] = None,
                 algo: str = "auto", ogate: Optional[torch.Tensor] = None, forget: str = "sigmoid"):
    """Stabilized parallel mLSTM forward pass.

    q, k [B,H,T,d_qk], v [B,H,T,d_v] (fp32 or bf16, same dtype, contiguous,
    CUDA); igate_pre, fgate_pre [B,H,T] fp32.  Returns h [B,H,T,d_v] in the
    input dtype: H~, or sigmoid(ogate) * H~ when the output-gate
    pre-activations ``ogate`` [B,H,T,d_v] are given; ``forget`` selects the
    forget activation ("sigmoid" or "exp").  With ``return_mn`` also the row
    stabilizer m and the normalizer n, both [B,H,T] fp32; with
    ``return_stats`` (h, m, n, b), b the signed row sums [B,H,T] fp32 (what
    ``parallel_bwd(..., saved=(h, n, b))`` takes).  Runs on the
    current stream.
    """
    lib = library()
    if q.dim() != 4:
        raise ValueError("q must be [B,H,T,d_qk]")
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    _need(q, "q", (B, H, T, dqk), q.dtype, dev)
    _need(k, "k", (B, H, T, dqk), q.dtype, dev)
    _need(v, "v", (B, H, T, dv), q.dtype, dev)
    _need(igate_pre, "igate_pre", (B, H, T), torch.float32, dev)
    _need(fgate_pre, "fgate_pre", (B, H, T), torch.float32, dev)
    if h is None:
        h = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev)
    _need(h, "h", (B, H, T, dv), q.dtype, dev)
    m = n = None
    b = None
    if return_mn or return_stats:
        m = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        n = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    if return_stats:
        b = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    ws_bytes = int(lib.mlstm_parallel_fwd_workspace(B, H, T))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    if workspace.device != dev or workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError(f"workspace must hold {ws_bytes} bytes on {dev}")
    if ogate is not None:
        _need(ogate, "ogate", (B, H, T, dv), q.dtype, dev)
    opt = _options(algo, forget, ogate, b)
    rc = lib.mlstm_parallel_fwd_opt(_ptr(q), _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), _ptr(h),
                                    _ptr(m), _ptr(n), B, H, T, dqk, dv, _DTYPES[q.dtype],
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    ctypes.byref(opt), _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_parallel_fwd")
    if return_stats:
        return h, m, n, b
    return (h, m, n) if return_mn else h


def step(C: torch.Tensor, n: torch.Tensor, m: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
         v: torch.Tensor, igate_pre: torch.Tensor, fgate_pre: torch.Tensor,
         o: Optional[torch.Tensor] = None, *, h: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One stabilized recurrent mLSTM step; updates C [B,H,d_v,d_qk], n [B,H,d_qk],
    m [B,H] (fp32) in place and returns h = sigma(o) * h~ [B,H,d_v] (o=None: no
    output gate).  q, k [B,H,d_qk], v, o [B,H,d_v] share one dtype (fp32/bf16);
    igate_pre, fgate_pre [B,H] fp32."""
    lib = library()
    if C.dim() != 4:
        raise ValueError("C must be [B,H,d_v,d_qk]")
    B, H, dv, dqk = C.shape
    dev = C.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    _need(C, "C", (B, H, dv, dqk), torch.float32, dev)
    _need(n, "n", (B, H, dqk), torch.float32, dev)
    _need(m, "m", (B, H), torch.float32, dev)
    _need(q, "q", (B, H, dqk), q.dtype, dev)
    _need(k, "k", (B, H, dqk), q.dtype, dev)
    _need(v, "v", (B, H, dv), q.dtype, dev)
    if o is not None:
        _need(o, "o", (B, H, dv), q.dtype, dev)
    _need(igate_pre, "igate_pre", (B, H), torch.float32, dev)
    _need(fgate_pre, "fgate_pre", (B, H), torch.float32, dev)
    if h is None:
        h = torch.empty((B, H, dv), dtype=q.dtype, device=dev)
    _need(h, "h", (B, H, dv), q.dtype, dev)
    rc = lib.mlstm_step(_ptr(C), _ptr(n), _ptr(m), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(igate_pre),
                        _ptr(fgate_pre), _ptr(h), B, H, dqk, dv, _DTYPES[q.dtype], _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_step")
    return h


def parallel_fwd_host_workspace_bytes(B: int, H: int, T: int, d_qk: int, d_v: int, dtype: torch.dtype) -> int:
    return int(library().mlstm_parallel_fwd_host_workspace(B, H, T, d_qk, d_v, _DTYPES[dtype]))


def parallel_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, igate_pre: torch.Tensor,
                      fgate_pre: torch.Tensor, *, h: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, device=None) -> torch.Tensor:
    """``mlstm_parallel_fwd_host``: the parallel forward on CPU tensors (pin
    them for overlapped copies), computed on ``device`` (default: current CUDA
    device) in chunks of heads whose uploads, compute and downloads overlap.
    Returns h on the CPU; the current stream completes when h is written."""
    lib = library()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (igate_pre, "igate_pre"), (fgate_pre, "fgate_pre")):
        if t.device.type != "cpu":
            raise ValueError(f"{name} must be a CPU tensor")
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    cpu = torch.device("cpu")
    _need(q, "q", (B, H, T, dqk), q.dtype, cpu)
    _need(k, "k", (B, H, T, dqk), q.dtype, cpu)
    _need(v, "v", (B, H, T, dv), q.dtype, cpu)
    _need(igate_pre, "igate_pre", (B, H, T), torch.float32, cpu)
    _need(fgate_pre, "fgate_pre", (B, H, T), torch.float32, cpu)
    if h is None:
        h = torch.empty((B, H, T, dv), dtype=q.dtype, pin_memory=q.is_pinned())
    _need(h, "h", (B, H, T, dv), q.dtype, cpu)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    need = parallel_fwd_host_workspace_bytes(B, H, T, dqk, dv, q.dtype)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError("workspace too small")
    rc = lib.mlstm_parallel_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), _ptr(h),
                                     B, H, T, dqk, dv, _DTYPES[q.dtype], _ptr(workspace), need, _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_parallel_fwd_host")
    return h


def parallel_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, igate_pre: torch.Tensor,
                 fgate_pre: torch.Tensor, dh: torch.Tensor, *, workspace: Optional[torch.Tensor] = None,
                 saved=None, ogate: Optional[torch.Tensor] = None, forget: str = "sigmoid"):
    """``mlstm_parallel_bwd`` / ``mlstm_parallel_bwd_opt``: gradients (dq, dk,
    dv, d_igate, d_fgate) of the parallel forward for the output gradient dh
    (CUDA tensors); with ``ogate`` (the output-gate pre-activations
    [B,H,T,d_v], forward h = sigmoid(ogate) * H~) dh is dL/dh and d_ogate is
    returned sixth.  ``forget`` selects the forget activation ("sigmoid" or
    "exp").  ``saved`` = (h, n, b) from ``parallel_fwd(..., return_stats=True)``
    without an output gate, on the same inputs, lets the tensor-core path skip
    its forward pass."""
    lib = library()
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    _need(q, "q", (B, H, T, dqk), q.dtype, dev)
    _need(k, "k", (B, H, T, dqk), q.dtype, dev)
    _need(v, "v", (B, H, T, dv), q.dtype, dev)
    _need(igate_pre, "igate_pre", (B, H, T), torch.float32, dev)
    _need(fgate_pre, "fgate_pre", (B, H, T), torch.float32, dev)
    _need(dh, "dh", (B, H, T, dv), q.dtype, dev)
    if ogate is not None:
        _need(ogate, "ogate", (B, H, T, dv), q.dtype, dev)
    opt = _options(forget=forget, ogate=ogate)
    need = int(lib.mlstm_parallel_bwd_workspace_opt(B, H, T, dqk, dv, _DTYPES[q.dtype], ctypes.byref(opt)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dig, dfg = torch.empty_like(igate_pre), torch.empty_like(fgate_pre)
    dog = torch.empty_like(dh) if ogate is not None else None
    hs = ns = bs = None
    if saved is not None:
        hs, ns, bs = saved
        _need(hs, "saved h", (B, H, T, dv), q.dtype, dev)
        _need(ns, "saved n", (B, H, T), torch.float32, dev)
        _need(bs, "saved b", (B, H, T), torch.float32, dev)
    rc = lib.mlstm_parallel_bwd_opt(_ptr(q), _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), _ptr(dh),
                                    _ptr(hs), _ptr(ns), _ptr(bs), _ptr(dq), _ptr(dk), _ptr(dvv), _ptr(dig),
                                    _ptr(dfg), _ptr(dog), B, H, T, dqk, dv, _DTYPES[q.dtype], _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), ctypes.byref(opt), _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_parallel_bwd_opt")
    if ogate is not None:
        return dq, dk, dvv, dig, dfg, dog
    return dq, dk, dvv, dig, dfg


def recurrent_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, igate_pre: torch.Tensor,
                  fgate_pre: torch.Tensor, dh: torch.Tensor, *, ogate: Optional[torch.Tensor] = None,
                  forget: str = "sigmoid", workspace: Optional[torch.Tensor] = None):
    """``mlstm_recurrent_bwd``: gradients (dq, dk, dv, d_igate, d_fgate, d_ogate)
    of the recurrent form from a fresh state, for dh = dL/dh (CUDA tensors);
    d_ogate is None without an output gate."""
    lib = library()
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    _need(q, "q", (B, H, T, dqk), q.dtype, dev)
    _need(k, "k", (B, H, T, dqk), q.dtype, dev)
    _need(v, "v", (B, H, T, dv), q.dtype, dev)
    _need(igate_pre, "igate_pre", (B, H, T), torch.float32, dev)
    _need(fgate_pre, "fgate_pre", (B, H, T), torch.float32, dev)
    _need(dh, "dh", (B, H, T, dv), q.dtype, dev)
    if ogate is not None:
        _need(ogate, "ogate", (B, H, T, dv), q.dtype, dev)
    need = int(lib.mlstm_recurrent_bwd_workspace(B, H, T, dqk, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dig, dfg = torch.empty_like(igate_pre), torch.empty_like(fgate_pre)
    dog = torch.empty_like(ogate) if ogate is not None else None
    opt = _options("auto", forget, ogate)
    rc = lib.mlstm_recurrent_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), _ptr(dh), _ptr(dq),
                                 _ptr(dk), _ptr(dvv), _ptr(dig), _ptr(dfg), None if dog is None else _ptr(dog),
                                 B, H, T, dqk, dv, _DTYPES[q.dtype], _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), ctypes.byref(opt), _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_recurrent_bwd")
    return dq, dk, dvv, dig, dfg, dog


def parallel_final_state(k: torch.Tensor, v: torch.Tensor, workspace: torch.Tensor):
    """The recurrent state (C [B,H,d_v,d_qk], n [B,H,d_qk], m [B,H], fp32) after
    the last token of k [B,H,T,d_qk], v [B,H,T,d_v], from the gate terms that
    ``gate_prep`` or ``parallel_fwd(..., workspace=...)`` left in ``workspace``:
    the hand-off from a parallel prefill to ``step`` / ``step_seq``."""
    lib = library()
    if k.dim() != 4 or v.dim() != 4:
        raise ValueError("k and v must be [B,H,T,d]")
    B, H, T, dqk = k.shape
    dv = v.shape[-1]
    dev = k.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if k.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {k.dtype}")
    _need(k, "k", (B, H, T, dqk), k.dtype, dev)
    _need(v, "v", (B, H, T, dv), k.dtype, dev)
    C = torch.empty((B, H, dv, dqk), dtype=torch.float32, device=dev)
    n = torch.empty((B, H, dqk), dtype=torch.float32, device=dev)
    m = torch.empty((B, H), dtype=torch.float32, device=dev)
    rc = lib.mlstm_parallel_final_state(_ptr(k), _ptr(v), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _ptr(C), _ptr(n), _ptr(m), B, H, T, dqk, dv, _DTYPES[k.dtype], _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_parallel_final_state")
    return C, n, m


def step_seq(C: torch.Tensor, n: torch.Tensor, m: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
             v: torch.Tensor, igate_pre: torch.Tensor, fgate_pre: torch.Tensor,
             o: Optional[torch.Tensor] = None, *, h: Optional[torch.Tensor] = None,
             forget: str = "sigmoid") -> torch.Tensor:
    """L recurrent steps per head in one call (``mlstm_step_seq``).  The state
    C [B,H,d_v,d_qk], n [B,H,d_qk], m [B,H] (fp32) is updated in place; q, k
    [B,H,L,d_qk], v, o [B,H,L,d_v] share one dtype; igate_pre, fgate_pre
    [B,H,L] fp32.  Returns h [B,H,L,d_v]."""
    lib = library()
    if C.dim() != 4 or q.dim() != 4:
        raise ValueError("C must be [B,H,d_v,d_qk] and q [B,H,L,d_qk]")
    B, H, dv, dqk = C.shape
    L = q.shape[2]
    dev = C.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    _need(C, "C", (B, H, dv, dqk), torch.float32, dev)
    _need(n, "n", (B, H, dqk), torch.float32, dev)
    _need(m, "m", (B, H), torch.float32, dev)
    _need(q, "q", (B, H, L, dqk), q.dtype, dev)
    _need(k, "k", (B, H, L, dqk), q.dtype, dev)
    _need(v, "v", (B, H, L, dv), q.dtype, dev)
    if o is not None:
        _need(o, "o", (B, H, L, dv), q.dtype, dev)
    _need(igate_pre, "igate_pre", (B, H, L), torch.float32, dev)
    _need(fgate_pre, "fgate_pre", (B, H, L), torch.float32, dev)
    if h is None:
        h = torch.empty((B, H, L, dv), dtype=q.dtype, device=dev)
    _need(h, "h", (B, H, L, dv), q.dtype, dev)
    opt = _options(forget=forget)
    rc = lib.mlstm_step_seq_opt(_ptr(C), _ptr(n), _ptr(m), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(igate_pre),
                                _ptr(fgate_pre), _ptr(h), B, H, L, dqk, dv, _DTYPES[q.dtype], ctypes.byref(opt),
                                _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_step_seq")
    return h


def last_device_status(stream: Optional[int] = None) -> int:
    """Synchronize ``stream`` (default: current) and return, then clear, the
    status word the kernels set when a bounded wait gives up."""
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    return int(library().mlstm_last_device_status(stream))


def set_spin_limit(limit: int) -> int:
    """Set the per-wait spin budget of the kernels' bounded waits (0 = default);
    returns the previous value.  Small values make waits give up (fault injection)."""
    return int(library().mlstm_set_spin_limit(int(limit)))


def gate_prep(igate_pre: torch.Tensor, fgate_pre: torch.Tensor, workspace: torch.Tensor,
              forget: str = "sigmoid") -> None:
    """Gate phase of the parallel forward (log forget-gate prefix sums and the
    prefix-max stabilizer) into ``workspace``; [B,H,T] fp32 CUDA inputs."""
    lib = library()
    B, H, T = igate_pre.shape
    dev = igate_pre.device
    _need(igate_pre, "igate_pre", (B, H, T), torch.float32, dev)
    _need(fgate_pre, "fgate_pre", (B, H, T), torch.float32, dev)
    opt = _options(forget=forget)
    rc = lib.mlstm_gate_prep_opt(_ptr(igate_pre), _ptr(fgate_pre), B, H, T, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), ctypes.byref(opt), _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_gate_prep")


def parallel_fwd_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, workspace: torch.Tensor,
                       h: torch.Tensor, m: Optional[torch.Tensor] = None, n: Optional[torch.Tensor] = None,
                       algo: str = "auto") -> torch.Tensor:
    """Fused phase of the parallel forward, reading the gate terms that
    ``gate_prep`` left in ``workspace``.  Writes ``h`` (and m, n if given)."""
    lib = library()
    B, H, T, dqk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    _need(q, "q", (B, H, T, dqk), q.dtype, dev)
    _need(k, "k", (B, H, T, dqk), q.dtype, dev)
    _need(v, "v", (B, H, T, dv), q.dtype, dev)
    _need(h, "h", (B, H, T, dv), q.dtype, dev)
    rc = lib.mlstm_parallel_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(h), _ptr(m), _ptr(n), B, H, T, dqk, dv,
                                      _DTYPES[q.dtype], _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), ALGOS[algo], _stream(dev))
    if rc != 0:
        raise MlstmError(rc, "mlstm_parallel_fwd_gated")
    return h


def tc_supported(d_qk: int, d_v: int, dtype: torch.dtype) -> bool:
    """Whether the tensor-core kernel tiles this head size and dtype."""
    return dtype == torch.bfloat16 and d_qk % 64 == 0 and d_v % 64 == 0 and d_qk <= 512 and d_v <= 512
