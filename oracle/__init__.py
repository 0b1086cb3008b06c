"""CPU oracle for the MTP draft-and-verify step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the bench's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  The product path (``mtp_self_speculative_gb300``) never imports it
and shares no code with it.

The oracle is plain numpy in float64: slow, per-request, obviously correct.
Each function cites the passage of the source pages it follows.
"""
from .mtp_oracle import (  # noqa: F401
    MTPWeights64,
    widen,
    round_to_bf16,
    bf16_bits_of,
    rmsnorm,
    rope,
    attention,
    silu,
    swiglu_mlp,
    eh_proj,
    lm_head,
    argmax_lowest,
    top2_gap,
    draft,
    verify,
    verify_sequential,
    kv_commit,
    kv_rollback,
    kv_truncate,
    kv_read_slots,
)
