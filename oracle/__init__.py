"""fp64 CPU oracle (test infrastructure only; see ``oracle.attention``), and the bf16
standard-attention baseline of the error contract (``oracle.standard_bf16``).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` import
this package.  It shares no code with the CUDA library.
"""

from .attention import (  # noqa: F401
    attention_backward,
    attention_forward,
    key_gradients,
    masked_scores,
    probabilities,
    row_logsumexp,
    row_statistics,
    tiled_forward,
)
