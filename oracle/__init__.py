"""CPU oracle for the exact attention forward pass — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or run anything in this
package.  The product path (``exact_attention_63_gb300``) never imports it and
never falls back to it.

The oracle is the plain two-pass definition of softmax attention in float64
(see ``attention.py``).  It shares no code with the CUDA path.  Every function
here is pinned by ``tests/test_oracle.py`` against brute force, closed forms,
library routines and invariants; no function is "parity unpinned".
"""

from .attention import (  # noqa: F401
    attention_backward,
    attention_backward_head,
    attention_backward_rows,
    attention_forward,
    attention_forward_fp8,
    attention_head,
    attention_rows,
    attention_varlen,
    head_probabilities,
    head_scores,
    kv_head,
    visible_mask,
    combine_partials,
    e4m3_to_f64,
    to_f64,
)
