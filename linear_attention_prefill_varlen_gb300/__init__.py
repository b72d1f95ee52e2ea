"""GB300 packed varlen causal depthwise conv1d (Kimi-K3 KDA Q|K|V short conv).

A thin ctypes binding over ``libkdaconv.so`` (C ABI declared in
``include/kda_conv.h``).  Every step of the conv runs in the library's CUDA
kernel; this module only turns torch tensors into pointers and sizes.  There
is no CPU fallback: if the library is missing, the calls raise.

Entry points mirror the C ABI (``kda_packed_conv1d``, ...), plus
``packed_causal_conv1d_fn`` / ``packed_causal_conv1d_supported`` with the
argument set of the vLLM page "vllm.models.kimi_k3.nvidia.ops.kda_conv"
(packed_causal_conv1d_fn, packed_causal_conv1d_supported).
"""

from __future__ import annotations

from ._binding import (  # noqa: F401
    KDA_ACT_NONE,
    KDA_ACT_SILU,
    KDA_DTYPE_BF16,
    KDA_DTYPE_F16,
    KDA_DTYPE_F32,
    KDA_ERR_CUDA,
    KDA_ERR_INVALID_ARG,
    KDA_ERR_METADATA,
    KDA_ERR_MISALIGNED,
    KDA_ERR_UNSUPPORTED,
    KDA_OK,
    KdaConvLayout,
    KdaError,
    KdaL2Norm,
    activation_code,
    causal_conv1d_update,
    epilogue_range,
    kda_conv1d_update,
    kda_conv1d_update_l2norm,
    kda_packed_conv1d,
    kda_packed_conv1d_ex,
    kda_packed_conv1d_l2norm,
    kda_packed_conv1d_preact_f32,
    l2norm_check,
    layout_of,
    make_l2norm,
    make_layout,
    launch_shape,
    lib,
    lib_path,
    packed_causal_conv1d_fn,
    packed_causal_conv1d_supported,
    validate_metadata,
    validate_metadata_device,
)
