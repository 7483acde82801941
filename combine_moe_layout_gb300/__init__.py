"""GB300-native MoE expert-parallel token dispatch and combine on one GPU.

The EP ranks are logical partitions of one device allocation. The work runs in
libmoe_layout.so (hand-written CUDA for sm_103a behind the C ABI of
include/moe_layout.h); this package holds its thin Python binding and the
seeded workload generators.
"""
from ._binding import (  # noqa: F401
    MOE_BF16,
    MOE_BF16_TO_FP8,
    MOE_ECUDA,
    MOE_EINVAL,
    MOE_ENOMEM,
    MOE_EOVERFLOW,
    MOE_ETIMEOUT,
    MOE_FP8_E4M3,
    MOE_OK,
    MoeBuffers,
    MoeDesc,
    MoeError,
    PackedBuffers,
    allocate_buffers,
    allocate_packed,
    library_path,
    load,
    moe_buffer_sizes,
    moe_combine,
    moe_combine_packed,
    moe_dispatch,
    moe_dispatch_recv,
    moe_expert_down,
    moe_expert_down_fp8,
    moe_expert_gate_up,
    moe_expert_gate_up_fp8,
    moe_expert_mlp_noalloc,
    moe_expert_mlp_noalloc_fp8,
    moe_expert_stub,
    moe_get_error,
    moe_layout,
    moe_layout_dispatch,
    moe_layout_dispatch_kernels,
    moe_reset,
    moe_route_stats,
    moe_status_string,
)
