"""CPU fp64 oracle for fused linear cross-entropy.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import or run anything in this
package.  The product path (``lm_head_linear_gb300``) never imports it, and this
package imports nothing from the product path: the two share no code.  The only
module both sides use is ``workloads`` (seeded random inputs, none of the
method's arithmetic).
"""

from .flce_oracle import (  # noqa: F401
    ForwardResult,
    argmax_rows,
    backward,
    dW_rows,
    forward,
    logits,
    naive_logits_bytes,
    sampled_rows,
    shard_partials,
    token_outputs_given_lse,
    upstream_grad,
    valid_mask,
)
