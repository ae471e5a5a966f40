"""GB300-native paged KV-cache decode path (PagedAttention).

The work happens in libpkv.so (CUDA kernels for sm_103a behind the C ABI of
include/pkv.h); this package is the thin Python binding over it.
"""
from ._binding import (  # noqa: F401
    KERNEL_AUTO, KERNEL_CUDA_CORE, PKV_BF16, PKV_F16, PKV_F32, PREFILL_TCGEN05, PREFILL_WARP_MMA,
    WIDE_HEAD_SLICES, WIDE_TCGEN05,
    STATUS_BITS, BlockAllocator, NOALLOC_SCRATCH_BYTES, OutOfBlocks, PkvError, decode_step,
    decode_workspace_bytes, device_status, group_shared_tokens, prepare_group_shared_tokens,
    kv_copy_blocks, kv_swap_blocks, kv_write, lib, paged_decode_attention,
    paged_decode_attention_noalloc, paged_decode_grouped, paged_prefill_attention,
    selftest_bounded_wait, set_decode_kernel, set_prefill_kernel, set_wide_group_kernel,
)

__all__ = [
    "BlockAllocator", "OutOfBlocks", "PkvError", "decode_step", "decode_workspace_bytes",
    "device_status", "group_shared_tokens", "prepare_group_shared_tokens",
    "kv_copy_blocks", "kv_swap_blocks", "kv_write", "lib", "paged_decode_attention",
    "paged_decode_attention_noalloc", "paged_decode_grouped", "paged_prefill_attention",
    "selftest_bounded_wait",
    "set_decode_kernel", "set_prefill_kernel", "set_wide_group_kernel",
]
