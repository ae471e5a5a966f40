// Tensor-core paged decode attention: launch entry for one (sequence, KV
// head, partition) per CTA with up to 8 query heads of the KV group.  The
// kernel and its design notes are in decode_tc.cuh (shared with the wide-group
// launch in decode_wide.cu and the beam-group launch in decode_group.cu).
#include "decode_tc.cuh"

cudaError_t launch_decode_tensor_core(const DecodeParams& p, int kv_dtype, const void* k_map,
                                      const void* v_map, long long grid, cudaStream_t stream)
{
    if (kv_dtype == PKV_BF16)
        return launch_tc_dtype<__nv_bfloat16, false, 1>(p, k_map, v_map, grid, stream);
    return launch_tc_dtype<__half, false, 1>(p, k_map, v_map, grid, stream);
}
