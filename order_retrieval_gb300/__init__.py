"""ZETA hot path on GB300: Z-order top-k attention with the Cauchy softmax.

The computation lives in ``libzeta.so`` (hand-written sm_103a CUDA behind the C
ABI in ``include/zeta.h``); ``binding`` is its thin ctypes binding with the same
function names, ``pipeline`` the user-facing plan / autograd wrapper, and
``workloads`` the seeded synthetic inputs.
"""
from . import binding, workloads  # noqa: F401
from .binding import (  # noqa: F401
    ZETA_BF16, ZETA_F32, ZetaError, problem, problem_of, zeta_attend_bwd, zeta_attend_fwd,
    zeta_bwd_workspace_bytes, zeta_code_bytes, zeta_encode, zeta_prefix_entries,
    zeta_select_topk, zeta_sort_chunks, zeta_sort_workspace_bytes, zeta_status_string)
from .pipeline import ZetaAttention, ZetaPlan, zeta_attention  # noqa: F401
