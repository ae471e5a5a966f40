// Tensor-core paged decode attention over beam groups: launch entry.  The
// kernel is the one in decode_tc.cuh, instantiated for groups of sequences
// that share a prefix of physical blocks (cayang0802 "Paged Attention" page,
// beam-search paragraph: the beams of a search keep one physical copy of the
// logical blocks they have in common).  Each shared K/V tile then leaves HBM
// once per group instead of once per member, the way a GQA group shares each
// tile across its query heads.
#include "decode_tc.cuh"

cudaError_t launch_decode_grouped(const DecodeParams& p, int kv_dtype, const void* k_map,
                                  const void* v_map, long long grid, bool wide,
                                  cudaStream_t stream)
{
    if (wide) {
        if (kv_dtype == PKV_BF16)
            return launch_tc_dtype<__nv_bfloat16, true, 2>(p, k_map, v_map, grid, stream);
        return launch_tc_dtype<__half, true, 2>(p, k_map, v_map, grid, stream);
    }
    if (kv_dtype == PKV_BF16)
        return launch_tc_dtype<__nv_bfloat16, true, 1>(p, k_map, v_map, grid, stream);
    return launch_tc_dtype<__half, true, 1>(p, k_map, v_map, grid, stream);
}
