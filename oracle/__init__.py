"""fp64 CPU oracle for the attention forward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA path never does.
"""
from .attention import (  # noqa: F401
    decode, decode_bf16, decode_f16,
    attention_reference, attention_reference_f64, attention_rows,
    softmax_probabilities, online_softmax_attention, attention_reference_varlen,
)
from .dropout import (  # noqa: F401
    philox4x32_10, dropout_keep, dropout_threshold, dropout_draws, attention_reference_dropout,
)
