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
// device address comes from cudaGetSymbolAddress, looked up once per device
// (with that device current) on the first call made on it.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
int scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return pkv_fail(PKV_ERR_CUDA, "pkv_paged_decode_attention_noalloc: cudaGetDevice: %s",
                        cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return pkv_fail(PKV_ERR_UNSUPPORTED,
                        "pkv_paged_decode_attention_noalloc: device %d beyond %d", dev,
                        kMaxDevices);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return pkv_fail(PKV_ERR_CUDA,
                            "pkv_paged_decode_attention_noalloc: cudaGetSymbolAddress: %s",
                            cudaGetErrorString(e));
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
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
                        "pkv_paged_decode_attention_noalloc: partition_size must be > 0 "
                        "(this entry point is the split-context decode)");
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
        block_size <= 0)
        return pkv_paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens,
                                          scale, block_size, num_kv_heads, num_seqs, num_heads,
                                          head_dim, max_blocks_per_seq, num_blocks, kv_dtype,
                                          out_dtype, partition_size, nullptr, 0, stream);
    const size_t need = pkv_decode_workspace_bytes(
        num_seqs, num_heads, head_dim, max_blocks_per_seq * block_size, partition_size);
    if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES)
        return pkv_fail(PKV_ERR_WORKSPACE,
                        "pkv_paged_decode_attention_noalloc: these sizes need %zu bytes of "
                        "scratch; the fixed array holds %zu (use pkv_paged_decode_attention "
                        "with a caller workspace, or a larger partition_size)",
                        need, (size_t)PKV_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
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
