"""GB300-native gated-DeltaNet decode step.

The layer runs in libdn.so (hand-written CUDA for sm_103a behind the C ABI
of include/dn.h).  This package holds the Python binding of that ABI
(``abi``), its build step (``build``) and the seeded workload generator
(``inputs``).
"""
from .abi import (  # noqa: F401
    ABI_SYMBOLS,
    DN_EFAILED,
    DN_ECUDA,
    DN_EINJECTED,
    DN_EINVAL,
    DN_ENOMEM,
    DN_OK,
    DN_PTR_DEVICE,
    DN_PTR_HOST,
    DNError,
    dn_create,
    dn_debug_fail_next,
    dn_destroy,
    dn_device_bytes,
    dn_get_state,
    dn_profile_next_step,
    dn_proj_i8_noalloc,
    dn_set_state,
    dn_step,
    load_library,
)
