"""Exact tiled attention (forward + backward) for GB300 / sm_103a.

The compute path is the C-ABI library ``libfa.so`` built from ``csrc/``;
``fwd``/``bwd`` are thin argument-marshalling wrappers around it.  The shared
library is loaded on first use and the wrappers raise if it is missing: there
is no fallback implementation.  ``debug_checks()`` runs the calls inside its
block on ``libfa_debug.so``, whose kernels check every TMA coordinate,
shared-memory operand and tensor-memory column range before using it.
"""

from .binding import (  # noqa: F401
    FaError,
    bwd,
    bwd_stages,
    bwd_workspace_size,
    debug_checks,
    debug_lib,
    fwd,
    fwd_workspace_size,
    lib,
    library_path,
    merge,
    status_string,
    sync_status,
)
from .autograd import attention  # noqa: F401,E402
