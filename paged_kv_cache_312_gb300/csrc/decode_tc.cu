// Tensor-core paged decode attention: launch entry for one (sequence, KV
// head, partition) per CTA.  The kernel and its design notes are in
// decode_tc.cuh (shared with the beam-group launch in decode_group.cu).
#include "decode_tc.cuh"

cudaError_t launch_decode_tensor_core(const DecodeParams& p, int kv_dtype, const void* k_map,
                                      const void* v_map, long long grid, cudaStream_t stream)
{
    if (kv_dtype == PKV_BF16) return launch_tc_dtype<__nv_bfloat16, false>(p, k_map, v_map, grid, stream);
    return launch_tc_dtype<__half, false>(p, k_map, v_map, grid, stream);
}
