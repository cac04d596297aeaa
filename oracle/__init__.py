"""fp64 CPU oracle for exact scaled-dot-product attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product path (the C-ABI library and
its Python binding) never imports, links or executes anything here, and this
package imports nothing from the product package.
"""

from .attention import (  # noqa: F401
    attention_backward,
    attention_backward_head,
    attention_backward_rows,
    attention_forward,
    attention_forward_head,
    attention_forward_rows,
    causal_mask,
    matmul_backward,
    merge_outputs,
    merge_partials,
    merge_stats,
    naive_softmax,
    online_softmax_steps,
    softmax_3pass,
    softmax_backward,
    tiled_forward_head,
)
