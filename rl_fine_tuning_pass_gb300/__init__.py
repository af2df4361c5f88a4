"""GRPO / entropy / selective-log-softmax row pass over LM-head logits, for GB300 (sm_103a).

The compute path is the C-ABI library ``libgrpo_rowpass.so`` (hand-written CUDA kernels,
declared in ``include/grpo_rowpass.h``); this package holds its build step, a thin ctypes
binding with the same function names, autograd wrappers, and the seeded workload
generators.  The library is loaded on first use; importing the package needs no GPU.
"""
from .binding import (  # noqa: F401
    GrpoError,
    entropy_from_logits,
    entropy_from_logits_bwd,
    grpo_loss_bwd,
    grpo_loss_fused,
    grpo_loss_fwd,
    grpo_seq_terms,
    load_library,
    selective_log_softmax_bwd,
    selective_log_softmax_fwd,
    status_string,
)
from .autograd import entropy, grpo_loss, selective_log_softmax  # noqa: F401,E402
