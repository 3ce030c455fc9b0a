"""GB300-native channels-last GroupNorm(+SiLU).

The computation runs in ``libgnsilu.so`` (hand-written sm_103a CUDA behind
the C ABI of ``include/gnsilu.h``); ``gnsilu`` is its Python binding.
Build the library with ``python -m channels_last_groupnorm_gb300.build``.
"""
from .gnsilu import (  # noqa: F401
    ATTN_AUTO,
    ATTN_ONE_PASS,
    ATTN_STORED_WEIGHTS,
    GnError,
    attention_folded,
    attn_fold,
    VARIANT_AUTO,
    VARIANT_CLUSTER,
    VARIANT_FUSED,
    VARIANT_TWO_PASS,
    gn_abi_version,
    gn_device_status,
    gn_kernel_launch_count,
    gn_library_workspaces,
    gn_release_workspaces,
    gn_silu_ndhwc,
    gn_silu_nhwc,
    gn_silu_pick_variant,
    gn_silu_rows,
    gn_silu_rows_any,
    gn_silu_rows_ex,
    gn_silu_workspace_bytes,
    new_workspace,
    residual_gate_add,
    status_string,
    upconv_fold,
    upsample_conv_nhwc,
)
