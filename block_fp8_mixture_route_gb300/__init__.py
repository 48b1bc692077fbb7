"""Block-FP8 mixture-of-experts layer forward for NVIDIA GB300 (sm_103a).

The compute runs in the CUDA library libmoe_fp8_block.so (C ABI in
include/moe_fp8_block.h); this package is its thin Python binding plus the
seeded synthetic input generators.
"""
from .api import (  # noqa: F401
    forward_problem,
    moe_fp8_block_abi_version,
    moe_fp8_block_act_quant,
    moe_fp8_block_device_status,
    moe_fp8_block_default_path,
    moe_fp8_block_forward,
    moe_fp8_block_forward_act_codes,
    moe_fp8_block_forward_bias,
    moe_fp8_block_forward_decode_noalloc,
    moe_fp8_block_forward_host_experts,
    moe_fp8_block_forward_hostio,
    moe_fp8_block_last_launches,
    moe_fp8_block_last_path,
    moe_fp8_block_noalloc_status,
    moe_fp8_block_release,
    moe_fp8_block_reserve,
    moe_fp8_block_route,
    moe_fp8_block_widen_e4m3,
)
