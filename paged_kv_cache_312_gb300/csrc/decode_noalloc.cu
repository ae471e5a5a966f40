// Split-context decode attention that allocates nothing: its partition
// scratch lives in a fixed array in the library's own device memory.
//
// Who needs this: code that runs where it may not allocate device memory at
// all. Examples are a plugin called from a host framework's execute step,
// which forbids allocation there; a serving loop whose memory is carved up
// once at start-up by another allocator; and latency-critical code that
// cannot pay for cudaMalloc, which may synchronise the device. Such a caller
// has no way to obtain the workspace pkv_paged_decode_attention takes.
//
// The array below is a file-scope __device__ object, so every GPU that loads
// libpkv holds PKV_NOALLOC_SCRATCH_BYTES of it until the process exits. In
// host code its name is only a host-side stand-in, not a device address: the
// device address comes from cudaGetSymbolAddress, asked on every call with
// the caller's device current. The first call on a device is the set-up (it
// loads the library's device code there, if nothing has yet); later calls
// only look the address up, which allocates nothing. Asking each time, rather
// than keeping the first answer per device, means a call never uses an
// address from a context that has since been destroyed (cudaDeviceReset) or
// that is not the caller's current one.
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

const char* const kFn = "pkv_paged_decode_attention_noalloc";

// Device address of the scratch array in the current context.
int scratch_address(void** out)
{
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
        return pkv_fail(PKV_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", kFn,
                        cudaGetErrorString(e));
    *out = ptr;
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_decode_attention_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, float scale, int block_size,
    int num_kv_heads, int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq,
    int num_blocks, int kv_dtype, int out_dtype, int partition_size, void* stream)
{
    if (partition_size <= 0)
        return pkv_fail(PKV_ERR_SHAPE,
                        "%s: partition_size must be > 0 (this entry point is the split-context "
                        "decode)", kFn);
    // the same checks, in the same order, as the workspace entry point, so
    // that a malformed request gets the same code there and here
    const int chk = pkv_decode_check(kFn, kv_dtype, out_dtype, num_seqs, num_heads, num_kv_heads,
                                     head_dim, block_size, max_blocks_per_seq, num_blocks,
                                     partition_size, scale);
    if (chk != PKV_OK) return chk;
    if (num_seqs == 0) return PKV_OK;
    // the checks above bound the longest context by 2^30 tokens
    const int64_t max_ctx = (int64_t)max_blocks_per_seq * block_size;
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, (int)max_ctx,
                                                   partition_size);
    if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES)
        return pkv_fail(PKV_ERR_WORKSPACE,
                        "%s: these sizes need %zu bytes of scratch; the fixed array holds %zu "
                        "(use pkv_paged_decode_attention with a caller workspace, or a larger "
                        "partition_size)",
                        kFn, need, (size_t)PKV_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != PKV_OK) return rc;
    // The scratch needs no clearing here: the call below zeroes the
    // completion counters the tensor-core kernel uses, and every (max, sum,
    // output) slot a merge reads is written earlier in the same call.
    return pkv_paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                      block_size, num_kv_heads, num_seqs, num_heads, head_dim,
                                      max_blocks_per_seq, num_blocks, kv_dtype, out_dtype,
                                      partition_size, scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES,
                                      stream);
}
