"""fp64 CPU oracle for the exact attention forward (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA path never does, and this
package imports nothing from it.  See ``oracle/attention.py`` for the sources
each routine follows.
"""
from .attention import (  # noqa: F401
    attention_backward,
    attention_probabilities,
    blocked_normalised_attention,
    blocked_online_attention,
    brute_force_attention,
    naive_attention,
    naive_attention_bhnd,
    split_kv_attention,
)
