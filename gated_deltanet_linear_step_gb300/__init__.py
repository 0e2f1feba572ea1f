"""GB300 (sm_103a) Gated DeltaNet decode step.

The package is a C-ABI CUDA library (``libgdn.so``, built from ``csrc/`` by
``_build.build()``; header ``include/gdn.h``) plus a thin torch binding with
the same function names. Importing the package loads nothing; the first call
loads the library and raises if it has not been built.
"""
from ._binding import (  # noqa: F401
    FLAG_GATES_READY,
    FLAG_NO_STATE_WRITE,
    FLAG_NO_Y,
    FLAG_SILU_GATE,
    FLAG_TEST_GIVE_UP,
    GdnError,
    gdn_ab_gates,
    gdn_decode_step,
    gdn_decode_step_ex,
    gdn_decode_step_varlen,
    gdn_dispatch_kernel,
    gdn_get_geometry,
    gdn_in_proj,
    gdn_in_proj_noalloc,
    gdn_in_proj_workspace_size,
    gdn_in_proj_packed,
    gdn_pack_proj_weights,
    gdn_proj_pack_bytes,
    gdn_last_error,
    gdn_read_device_error,
    gdn_step_inputs,
    gdn_step_inputs_packed,
    gdn_verify_commit,
    gdn_verify_window,
    load_library,
)
