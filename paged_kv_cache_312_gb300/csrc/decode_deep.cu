// Tensor-core paged decode attention with deep rings: launch entries for
// unsplit launches of few, long items.  The kernel (decode_tc.cuh) runs with
// three 8 KB stages per warp ring instead of two, two CTAs a SM instead of
// three: the same tile loads in flight per SM, but each warp keeps two stages
// in flight while it works on a third, so a CTA streams faster on its own.
// That is what bounds a launch whose last CTAs are its longest ones; many
// short items prefer more CTAs a SM.  One n8 column tile (up to 8 query heads
// a CTA) or two (up to 16), as in decode_tc.cu and decode_wide.cu.
#include "decode_tc.cuh"

cudaError_t launch_decode_tensor_core_deep(const DecodeParams& p, int kv_dtype, const void* k_map,
                                           const void* v_map, long long grid, bool wide,
                                           cudaStream_t stream)
{
    if (wide) {
        if (kv_dtype == PKV_BF16)
            return launch_tc_dtype<__nv_bfloat16, false, 2, 3>(p, k_map, v_map, grid, stream);
        return launch_tc_dtype<__half, false, 2, 3>(p, k_map, v_map, grid, stream);
    }
    if (kv_dtype == PKV_BF16)
        return launch_tc_dtype<__nv_bfloat16, false, 1, 3>(p, k_map, v_map, grid, stream);
    return launch_tc_dtype<__half, false, 1, 3>(p, k_map, v_map, grid, stream);
}
