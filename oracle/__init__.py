"""CPU oracle for the gated-DeltaNet decode step.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke check
and by the benchmark's CPU-baseline leg, never by the product path.  It is a
plain float64 numpy restatement of the step's definition and shares no code
with the CUDA library.
"""
from .dn_oracle import (  # noqa: F401
    OracleLayer,
    causal_conv_silu_step,
    gated_delta_rule_step,
    gate_transform,
    gated_rmsnorm,
    int8_rowscaled_gemv,
    l2_normalize,
    normalize_qk,
    prefill,
    rms_prenorm,
    sigmoid,
    silu,
    softplus,
    stack_step,
)
