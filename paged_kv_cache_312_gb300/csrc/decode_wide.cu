// Tensor-core paged decode attention for wide query-head groups: launch
// entry for CTAs that carry 9 to 16 query heads of one KV group as two n8
// column tiles of the mma (auturnal guide section 1: with GQA many query
// heads share one KV head; MQA is the limit of one KV head for all).  Every
// K/V tile then still leaves HBM once per 16 query heads.  Groups wider than
// 16 are cut into head slices by the caller.
#include "decode_tc.cuh"

cudaError_t launch_decode_tensor_core_wide(const DecodeParams& p, int kv_dtype, const void* k_map,
                                           const void* v_map, long long grid, cudaStream_t stream)
{
    if (kv_dtype == PKV_BF16)
        return launch_tc_dtype<__nv_bfloat16, false, 2>(p, k_map, v_map, grid, stream);
    return launch_tc_dtype<__half, false, 2>(p, k_map, v_map, grid, stream);
}
