"""GB300-native mLSTM matrix memory: stabilized parallel forward and recurrent step.

The compute runs in hand-written CUDA kernels for sm_103a behind the C-ABI
library ``libmlstm.so`` (declared in ``include/mlstm.h``).  This package is the
thin Python binding: it validates tensors, passes device pointers and the
current CUDA stream, and returns.  PyTorch supplies device memory and streams
only.  The library is loaded on first use; if it is missing the calls raise.
"""
from .binding import (  # noqa: F401
    MlstmError,
    parallel_fwd,
    parallel_fwd_workspace_bytes,
    step,
    step_seq,
    parallel_final_state,
    parallel_bwd,
    recurrent_bwd,
    parallel_fwd_host,
    parallel_fwd_host_workspace_bytes,
    last_device_status,
    set_spin_limit,
    gate_prep,
    parallel_fwd_gated,
    tc_supported,
    library,
    library_path,
)
