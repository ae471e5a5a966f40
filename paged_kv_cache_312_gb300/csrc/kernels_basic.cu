// Cache write, copy-on-write block copy, CUDA-core paged decode and the
// log-sum-exp merge of split partitions, for sm_103a.
//
// Cache layout: [num_blocks][num_kv_heads][block_size][head_dim]; token i of a
// sequence sits in its logical block i / B at offset i % B (aiplusplus
// PagedAttention page, "core idea" 1-3).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pkv.h"
#include "pkv_kernels.h"

namespace {

// ---------------------------------------------------------------------------
// Device status word: kernels OR PKV_STATUS_* bits into it instead of touching
// memory an id points outside of.
// ---------------------------------------------------------------------------
__device__ unsigned int g_status_word;

__device__ __forceinline__ void flag(unsigned int* status, unsigned int bit)
{
    atomicOr(status, bit);
}

// ---------------------------------------------------------------------------
// kv_write: one thread moves one 16-byte vector of one token's K and V.
// (cayang0802 walkthrough, KV-cache paragraph: only the new token's K/V are
// produced each step and stored next to the earlier ones.)
// ---------------------------------------------------------------------------
__global__ void kv_write_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                const uint4* __restrict__ key, const uint4* __restrict__ value,
                                const int64_t* __restrict__ slot_mapping, int num_blocks,
                                int num_kv_heads, int vec_per_head, int block_size,
                                unsigned int* status)
{
    const int t = blockIdx.x;
    const int per_token = num_kv_heads * vec_per_head;
    const int i = blockIdx.y * blockDim.x + threadIdx.x;
    if (i >= per_token) return;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;  // padding token
    if (slot >= (int64_t)num_blocks * block_size) {
        if (i == 0) flag(status, PKV_STATUS_BAD_SLOT);
        return;
    }
    const int64_t blk = slot / block_size;
    const int off = (int)(slot - blk * block_size);
    const int h = i / vec_per_head, c = i - h * vec_per_head;
    const size_t dst = ((size_t)(blk * num_kv_heads + h) * block_size + off) * vec_per_head + c;
    const size_t src = (size_t)t * per_token + i;
    k_cache[dst] = key[src];
    v_cache[dst] = value[src];
}

// ---------------------------------------------------------------------------
// kv_append: the decode step's new token of sequence s (new_k/new_v
// [S][Hkv][D]) goes to position context_lens[s]-1, i.e. slot
// table[s][(L-1)/B] * B + (L-1) % B -- the slot mapping of the aiplusplus
// PagedAttention page (core idea 3-4) for the token just appended.  Used by
// the decode step when it runs on the CUDA-core kernel; the tensor-core
// kernel performs the same write itself.
// ---------------------------------------------------------------------------
__global__ void kv_append_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                 const uint4* __restrict__ new_k, const uint4* __restrict__ new_v,
                                 const int32_t* __restrict__ block_tables,
                                 const int32_t* __restrict__ context_lens, int max_blocks,
                                 int num_blocks, int num_kv_heads, int vec_per_head,
                                 int block_size, unsigned int* status)
{
    const int s = blockIdx.x;
    const int i = blockIdx.y * blockDim.x + threadIdx.x;  // (head, 16-byte chunk)
    if (i >= num_kv_heads * vec_per_head) return;
    const int L = context_lens[s];
    if (L <= 0) return;
    if ((int64_t)L > (int64_t)max_blocks * block_size) {
        if (i == 0) flag(status, PKV_STATUS_BAD_LEN);
        return;
    }
    const int id = block_tables[(size_t)s * max_blocks + (L - 1) / block_size];
    if (id < 0 || id >= num_blocks) {
        if (i == 0) flag(status, PKV_STATUS_BAD_BLOCK);
        return;
    }
    const int h = i / vec_per_head, c = i - h * vec_per_head;
    const size_t dst =
        (((size_t)id * num_kv_heads + h) * block_size + (L - 1) % block_size) * vec_per_head + c;
    const size_t src = (size_t)s * num_kv_heads * vec_per_head + i;
    k_cache[dst] = new_k[src];
    v_cache[dst] = new_v[src];
}

// ---------------------------------------------------------------------------
// kv_copy_blocks: physical block src -> dst for K and V; a block of all heads
// is one contiguous run of block_bytes in this layout.
// (auturnal guide, section 3: copy-on-write of a shared block that is not
// full keeps branches from overwriting each other.)
// ---------------------------------------------------------------------------
__global__ void copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                   const int64_t* __restrict__ pairs, int num_blocks,
                                   size_t vec_per_block, unsigned int* status)
{
    const int64_t src = pairs[2 * blockIdx.x], dst = pairs[2 * blockIdx.x + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) flag(status, PKV_STATUS_BAD_PAIR);
        return;
    }
    const uint4* ks = k_cache + (size_t)src * vec_per_block;
    const uint4* vs = v_cache + (size_t)src * vec_per_block;
    uint4* kd = k_cache + (size_t)dst * vec_per_block;
    uint4* vd = v_cache + (size_t)dst * vec_per_block;
    for (size_t i = (size_t)blockIdx.y * blockDim.x + threadIdx.x; i < vec_per_block;
         i += (size_t)gridDim.y * blockDim.x) {
        uint4 a = ks[i], b = vs[i];
        kd[i] = a;
        vd[i] = b;
    }
}

// ---------------------------------------------------------------------------
// kv_swap_blocks: whole blocks from one pool to another, e.g. the device cache
// and a pinned host swap pool that the GPU reaches directly over NVLink-C2C
// (aiplusplus page, section 4, and the cayang0802 walkthrough: a preempted
// sequence's KV blocks are swapped out to CPU memory and back).  Each thread
// keeps four 16-byte loads of K and four of V in flight before storing.
// ---------------------------------------------------------------------------
constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;

__global__ void __launch_bounds__(kSwapThreads)
swap_blocks_kernel(uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                   const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                   const int64_t* __restrict__ pairs, int num_src_blocks, int num_dst_blocks,
                   size_t vec_per_block, unsigned int* status)
{
    const int64_t src = pairs[2 * blockIdx.x], dst = pairs[2 * blockIdx.x + 1];
    if (src < 0 || src >= num_src_blocks || dst < 0 || dst >= num_dst_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) flag(status, PKV_STATUS_BAD_PAIR);
        return;
    }
    const uint4* ks = src_k + (size_t)src * vec_per_block;
    const uint4* vs = src_v + (size_t)src * vec_per_block;
    uint4* kd = dst_k + (size_t)dst * vec_per_block;
    uint4* vd = dst_v + (size_t)dst * vec_per_block;
    const size_t step = (size_t)gridDim.y * kSwapThreads * kSwapUnroll;
    for (size_t i0 = ((size_t)blockIdx.y * kSwapUnroll) * kSwapThreads + threadIdx.x;
         i0 < vec_per_block; i0 += step) {
        uint4 a[kSwapUnroll], b[kSwapUnroll];
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const size_t i = i0 + (size_t)u * kSwapThreads;
            if (i < vec_per_block) {
                a[u] = ks[i];
                b[u] = vs[i];
            }
        }
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const size_t i = i0 + (size_t)u * kSwapThreads;
            if (i < vec_per_block) {
                kd[i] = a[u];
                vd[i] = b[u];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// CUDA-core paged decode.  One CTA = one (partition, query head, sequence);
// its 4 warps take tokens round-robin, each lane holding D/32 elements of q,
// of the running output and of each K/V row it reads.  Scores are kept in
// base 2 (scale * log2 e folded into q), so exp2 replaces exp.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}

__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int out_dtype)
{
    if (out_dtype == PKV_F32)
        static_cast<float*>(out)[idx] = v;
    else if (out_dtype == PKV_F16)
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Context length of sequence s, or -1 (flagged) if it is out of range.
__device__ __forceinline__ int checked_len(const DecodeParams& p, int s)
{
    const int L = p.context_lens[s];
    if (L < 0 || (int64_t)L > (int64_t)p.max_blocks * p.block_size) {
        if (threadIdx.x == 0) flag(p.status, PKV_STATUS_BAD_LEN);
        return -1;
    }
    return L;
}

constexpr int kCoreWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kCoreWarps * 32)
decode_cuda_core_kernel(const DecodeParams p)
{
    constexpr int E = D / 32;  // elements per lane
    const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int L = checked_len(p, s);
    if (L < 0) L = 0;  // bad length: zero output, flagged above
    const int nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
    if (part >= (nparts > 0 ? nparts : 1)) return;
    const int begin = part * p.partition_tokens;
    const int end = min(L, begin + p.partition_tokens);
    const int G = p.num_heads / p.num_kv_heads;
    const int g = h / G;

    const T* qrow = static_cast<const T*>(p.q) + ((size_t)s * p.num_heads + h) * D + lane * E;
    float qv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) qv[e] = to_f32(qrow[e]) * p.scale_log2;

    const T* kc = static_cast<const T*>(p.k_cache);
    const T* vc = static_cast<const T*>(p.v_cache);
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
    float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;

    for (int t = begin + warp; t < end; t += kCoreWarps) {
        const int32_t blk = table[t / p.block_size];
        if (blk < 0 || blk >= p.num_blocks) {
            if (lane == 0) flag(p.status, PKV_STATUS_BAD_BLOCK);
            continue;
        }
        const size_t row = ((size_t)blk * p.num_kv_heads + g) * p.block_size + t % p.block_size;
        const T* kr = kc + row * D + lane * E;
        const T* vr = vc + row * D + lane * E;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot += qv[e] * to_f32(kr[e]);
        const float z = warp_sum(dot);
        const float m_new = fmaxf(m, z);
        const float alpha = exp2f(m - m_new);  // 0 when m is -inf
        const float pz = exp2f(z - m_new);
        l = l * alpha + pz;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = acc[e] * alpha + pz * to_f32(vr[e]);
        m = m_new;
    }

    // Merge the warps' running states.
    __shared__ float sm_m[kCoreWarps], sm_l[kCoreWarps];
    __shared__ float sm_o[kCoreWarps][D];
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sm_o[warp][lane * E + e] = acc[e];
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCoreWarps; ++w) M = fmaxf(M, sm_m[w]);
    float den = 0.f;
    float wgt[kCoreWarps];
#pragma unroll
    for (int w = 0; w < kCoreWarps; ++w) {
        wgt[w] = (M == -INFINITY) ? 0.f : exp2f(sm_m[w] - M);
        den += sm_l[w] * wgt[w];
    }
    const size_t orow = ((size_t)s * p.num_heads + h) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kCoreWarps; ++w) o += sm_o[w][d] * wgt[w];
        if (nparts <= 1) {
            store_out(p.out, orow + d, den > 0.f ? o / den : 0.f, p.out_dtype);
        } else {
            const size_t slot = ((size_t)s * p.num_heads + h) * p.max_partitions + part;
            p.ws_o[slot * D + d] = o;
            if (d == 0) p.ws_ml[slot] = make_float2(M, den);
        }
    }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge: with M = max_p m_p and w_p = 2^(m_p - M),
// out = sum_p w_p O_p / sum_p w_p l_p.  One CTA per (query head, sequence);
// sequences with a single partition were finished by the partition kernel.
// ---------------------------------------------------------------------------
__global__ void lse_reduce_kernel(const DecodeParams p)
{
    const int h = blockIdx.x, s = blockIdx.y;
    int L = p.context_lens[s];
    if (L < 0 || (int64_t)L > (int64_t)p.max_blocks * p.block_size) return;  // flagged
    const int nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
    if (nparts <= 1) return;
    const size_t base = ((size_t)s * p.num_heads + h) * p.max_partitions;
    const int D = p.head_dim;
    float M = -INFINITY;
    for (int i = 0; i < nparts; ++i) M = fmaxf(M, p.ws_ml[base + i].x);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float num = 0.f, den = 0.f;
        for (int i = 0; i < nparts; ++i) {
            const float2 ml = p.ws_ml[base + i];
            const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
            den += w * ml.y;
            num += w * p.ws_o[(base + i) * D + d];
        }
        store_out(p.out, ((size_t)s * p.num_heads + h) * D + d, den > 0.f ? num / den : 0.f,
                  p.out_dtype);
    }
}

}  // namespace

unsigned int* pkv_status_word_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    static unsigned int* cache[64] = {};
    if (dev < 0 || dev >= 64) return nullptr;
    if (!cache[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int*>(ptr);
    }
    return cache[dev];
}

cudaError_t launch_kv_write(void* k_cache, void* v_cache, const void* key, const void* value,
                            const int64_t* slot_mapping, int num_tokens, int num_blocks,
                            int num_kv_heads, int head_dim, int block_size, int elem_bytes,
                            unsigned int* status, cudaStream_t stream)
{
    const int vec_per_head = head_dim * elem_bytes / 16;
    const int per_token = num_kv_heads * vec_per_head;
    const int threads = per_token < 256 ? ((per_token + 31) / 32) * 32 : 256;
    dim3 grid(num_tokens, (per_token + threads - 1) / threads);
    kv_write_kernel<<<grid, threads, 0, stream>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
        static_cast<const uint4*>(key), static_cast<const uint4*>(value), slot_mapping,
        num_blocks, num_kv_heads, vec_per_head, block_size, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* new_k, const void* new_v,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int num_seqs, int max_blocks, int num_blocks, int num_kv_heads,
                             int head_dim, int block_size, int elem_bytes, unsigned int* status,
                             cudaStream_t stream)
{
    const int vec_per_head = head_dim * elem_bytes / 16;
    const int per_seq = num_kv_heads * vec_per_head;
    const int threads = per_seq < 256 ? ((per_seq + 31) / 32) * 32 : 256;
    dim3 grid(num_seqs, (per_seq + threads - 1) / threads);
    kv_append_kernel<<<grid, threads, 0, stream>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
        static_cast<const uint4*>(new_k), static_cast<const uint4*>(new_v), block_tables,
        context_lens, max_blocks, num_blocks, num_kv_heads, vec_per_head, block_size, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs,
                                  int num_pairs, int num_blocks, size_t block_bytes,
                                  unsigned int* status, cudaStream_t stream)
{
    const size_t vec = block_bytes / 16;
    const int threads = 256;
    size_t chunks = (vec + threads * 4 - 1) / (threads * 4);
    if (chunks < 1) chunks = 1;
    if (chunks > 65535) chunks = 65535;
    dim3 grid(num_pairs, (unsigned)chunks);
    copy_blocks_kernel<<<grid, threads, 0, stream>>>(static_cast<uint4*>(k_cache),
                                                     static_cast<uint4*>(v_cache), pairs,
                                                     num_blocks, vec, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_swap_blocks(void* dst_k, void* dst_v, const void* src_k, const void* src_v,
                                  const int64_t* pairs, int num_pairs, int num_src_blocks,
                                  int num_dst_blocks, size_t block_bytes, unsigned int* status,
                                  cudaStream_t stream)
{
    const size_t vec = block_bytes / 16;
    size_t chunks = (vec + kSwapThreads * kSwapUnroll - 1) / (kSwapThreads * kSwapUnroll);
    if (chunks < 1) chunks = 1;
    if (chunks > 65535) chunks = 65535;
    dim3 grid(num_pairs, (unsigned)chunks);
    swap_blocks_kernel<<<grid, kSwapThreads, 0, stream>>>(
        static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), static_cast<const uint4*>(src_k),
        static_cast<const uint4*>(src_v), pairs, num_src_blocks, num_dst_blocks, vec, status);
    return cudaGetLastError();
}

cudaError_t launch_decode_cuda_core(const DecodeParams& p, int kv_dtype, cudaStream_t stream)
{
    dim3 grid(p.max_partitions, p.num_heads, p.num_seqs);
    dim3 block(kCoreWarps * 32);
#define PKV_LAUNCH_CORE(T)                                                        \
    do {                                                                          \
        if (p.head_dim == 64)                                                     \
            decode_cuda_core_kernel<T, 64><<<grid, block, 0, stream>>>(p);        \
        else                                                                      \
            decode_cuda_core_kernel<T, 128><<<grid, block, 0, stream>>>(p);       \
    } while (0)
    if (kv_dtype == PKV_F32)
        PKV_LAUNCH_CORE(float);
    else if (kv_dtype == PKV_F16)
        PKV_LAUNCH_CORE(__half);
    else
        PKV_LAUNCH_CORE(__nv_bfloat16);
#undef PKV_LAUNCH_CORE
    return cudaGetLastError();
}

cudaError_t launch_lse_reduce(const DecodeParams& p, cudaStream_t stream)
{
    dim3 grid(p.num_heads, p.num_seqs);
    lse_reduce_kernel<<<grid, p.head_dim, 0, stream>>>(p);
    return cudaGetLastError();
}
