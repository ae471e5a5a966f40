// Cache write, copy-on-write block copy, CUDA-core paged decode and the
// log-sum-exp merge of split partitions, for sm_103a.
//
// Cache layout: [num_blocks][num_kv_heads][block_size][head_dim]; token i of a
// sequence sits in its logical block i / B at offset i % B (aiplusplus
// PagedAttention page, "core idea" 1-3).
#include <cuda_bf16.h>
#include <algorithm>
#include <climits>
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
// full keeps branches from overwriting each other.)  A step copies a few
// blocks at most, so the copy is one round trip if every load is in flight at
// once: CTA (pair, chunk) moves kCopyThreads * kCopyUnroll vectors of K and of
// V, each thread issuing its kCopyUnroll loads of both before it stores.
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int64_t* __restrict__ pairs, int num_blocks, size_t vec_per_block,
                   unsigned int* status)
{
    // a beam-group decode launched after this copy may start now: it waits
    // for this grid to complete before it touches the caches
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t src = pairs[2 * blockIdx.x], dst = pairs[2 * blockIdx.x + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) flag(status, PKV_STATUS_BAD_PAIR);
        return;
    }
    const uint4* ks = k_cache + (size_t)src * vec_per_block;
    const uint4* vs = v_cache + (size_t)src * vec_per_block;
    uint4* kd = k_cache + (size_t)dst * vec_per_block;
    uint4* vd = v_cache + (size_t)dst * vec_per_block;
    constexpr size_t per_cta = (size_t)kCopyThreads * kCopyUnroll;
    for (size_t i0 = (size_t)blockIdx.y * per_cta + threadIdx.x; i0 < vec_per_block;
         i0 += (size_t)gridDim.y * per_cta) {
        uint4 a[kCopyUnroll], b[kCopyUnroll];
#pragma unroll
        for (int k = 0; k < kCopyUnroll; ++k) {
            const size_t i = i0 + (size_t)k * kCopyThreads;
            if (i < vec_per_block) {
                a[k] = ks[i];
                b[k] = vs[i];
            }
        }
#pragma unroll
        for (int k = 0; k < kCopyUnroll; ++k) {
            const size_t i = i0 + (size_t)k * kCopyThreads;
            if (i < vec_per_block) {
                kd[i] = a[k];
                vd[i] = b[k];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// kv_swap_blocks: whole blocks from one pool to another, e.g. the device cache
// and a pinned host swap pool that the GPU reaches directly over NVLink-C2C
// (aiplusplus page, section 4, and the cayang0802 walkthrough: a preempted
// sequence's KV blocks are swapped out to CPU memory and back).  The work is
// cut into units of (pair, chunk of kSwapThreads * kSwapUnroll vectors); a
// grid of at most two CTAs per SM strides over them, so that a swap out and a
// swap in launched on two streams run side by side and use both directions
// of the link.  Each thread keeps four 16-byte loads of K and four of V in
// flight before storing.
// ---------------------------------------------------------------------------
constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;
constexpr int kSwapCtasPerSm = 2;

__global__ void __launch_bounds__(kSwapThreads)
swap_blocks_kernel(uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                   const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                   const int64_t* __restrict__ pairs, int num_pairs, int num_src_blocks,
                   int num_dst_blocks, size_t vec_per_block, int chunks, unsigned int* status)
{
    const long long units = (long long)num_pairs * chunks;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const int pi = (int)(u / chunks), chunk = (int)(u - (long long)pi * chunks);
        const int64_t src = pairs[2 * pi], dst = pairs[2 * pi + 1];
        if (src < 0 || src >= num_src_blocks || dst < 0 || dst >= num_dst_blocks) {
            if (chunk == 0 && threadIdx.x == 0) flag(status, PKV_STATUS_BAD_PAIR);
            continue;
        }
        const uint4* ks = src_k + (size_t)src * vec_per_block;
        const uint4* vs = src_v + (size_t)src * vec_per_block;
        uint4* kd = dst_k + (size_t)dst * vec_per_block;
        uint4* vd = dst_v + (size_t)dst * vec_per_block;
        const size_t i0 = (size_t)chunk * kSwapUnroll * kSwapThreads + threadIdx.x;
        uint4 a[kSwapUnroll], b[kSwapUnroll];
#pragma unroll
        for (int k = 0; k < kSwapUnroll; ++k) {
            const size_t i = i0 + (size_t)k * kSwapThreads;
            if (i < vec_per_block) {
                a[k] = ks[i];
                b[k] = vs[i];
            }
        }
#pragma unroll
        for (int k = 0; k < kSwapUnroll; ++k) {
            const size_t i = i0 + (size_t)k * kSwapThreads;
            if (i < vec_per_block) {
                kd[i] = a[k];
                vd[i] = b[k];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// CUDA-core paged decode (any KV dtype, any group size).  One CTA = one
// partition of one (sequence, KV head, head slice): the query heads of the
// KV group -- all of them, or a slice of at most kCoreCols -- attend
// together, so each K/V tile leaves memory once per group (auturnal guide
// section 1: GQA/MQA shrink the number of KV heads a token's K/V serve).
// Tiles of kCoreTile tokens of K and V are staged in shared memory by
// 16-byte cp.async copies, two tiles in flight.  Per tile:
//   scores   lane = token, warp w = heads w, w + 4, ...: s = q . k in fp32,
//            with scale * log2(e) folded into q (scores in base 2);
//   softmax  per head, against the running max (warp max over the tile);
//   P V      each thread owns a float4 of head_dim for a few heads.
// Masked tokens (past the partition's end or in a block whose id is out of
// range) are staged as zeros and get score -inf, so NaN or stale data in
// unused slots never reaches the output.
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

// The two elements of a 32-bit word of 16-bit T (low half first), widened.
template <typename T>
__device__ __forceinline__ float2 widen2(uint32_t w);
template <>
__device__ __forceinline__ float2 widen2<__nv_bfloat16>(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 widen2<__half>(uint32_t w)
{
    return make_float2(__half2float(__ushort_as_half((unsigned short)(w & 0xffffu))),
                       __half2float(__ushort_as_half((unsigned short)(w >> 16))));
}

// The elements of a 16-byte vector of T (4 fp32 or 8 16-bit), widened.
template <typename T>
__device__ __forceinline__ void widen_vec(const uint4 raw, float* f)
{
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(raw.x);
        f[1] = __uint_as_float(raw.y);
        f[2] = __uint_as_float(raw.z);
        f[3] = __uint_as_float(raw.w);
    } else {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = widen2<T>(w[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
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

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

constexpr int kCoreWarps = 4;
constexpr int kCoreThreads = kCoreWarps * 32;
constexpr int kCoreTile = 32;  // tokens per tile: one per lane in the score step
constexpr int kCoreCols = 16;  // query heads per CTA (wider groups: head slices)

// Shared-memory plan of the CUDA-core kernel for element type T, head_dim D.
template <typename T, int D>
struct CoreSmem {
    static constexpr int EPV = 16 / (int)sizeof(T);       // elements per 16-byte vector
    static constexpr int VPR = D / EPV;                    // vectors per K/V row
    static constexpr int ROW = D * (int)sizeof(T) + 16;    // padded row: conflict-free reads
    static constexpr int TILE = kCoreTile * ROW;           // K (or V) of one tile
    static constexpr int STAGE = 2 * TILE;                 // K then V
    static constexpr int Q_OFF = 2 * STAGE;                // float q [kCoreCols][D]
    static constexpr int P_OFF = Q_OFF + kCoreCols * D * 4;          // float p [cols][tile]
    static constexpr int A_OFF = P_OFF + kCoreCols * kCoreTile * 4;  // float alpha [cols]
    static constexpr int M_OFF = A_OFF + kCoreCols * 4;              // float m, l [cols]
    static constexpr int BYTES = M_OFF + 2 * kCoreCols * 4;
};

template <typename T, int D>
__global__ void __launch_bounds__(kCoreThreads)
decode_cuda_core_kernel(const DecodeParams p)
{
    using Sm = CoreSmem<T, D>;
    constexpr int ND4 = D / 4;                          // float4 columns of an output row
    constexpr int PAIRS = kCoreCols * ND4 / kCoreThreads;  // (head, float4) outputs a thread
    extern __shared__ __align__(16) uint8_t csm[];
    float* qs = reinterpret_cast<float*>(csm + Sm::Q_OFF);
    float* ps = reinterpret_cast<float*>(csm + Sm::P_OFF);
    float* al = reinterpret_cast<float*>(csm + Sm::A_OFF);
    float* ml = reinterpret_cast<float*>(csm + Sm::M_OFF);

    const int part = blockIdx.x, s = blockIdx.z;
    const int HS = p.head_slices;
    const int g = blockIdx.y / HS, hs = blockIdx.y - g * HS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L = checked_len(p, s);
    if (L < 0) L = 0;  // bad length: zero output, flagged above
    const int nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
    if (part >= (nparts > 0 ? nparts : 1)) return;
    const int begin = part * p.partition_tokens;
    const int end = min(L, begin + p.partition_tokens);
    const int G = p.num_heads / p.num_kv_heads;
    const int GC = (G + HS - 1) / HS;  // columns of a slice
    const int hb = hs * GC;
    const int ncol = min(GC, G - hb);
    const size_t hrow0 = (size_t)s * p.num_heads + (size_t)g * G + hb;  // first output row

    // q of this slice's heads, widened and scaled (scores in base 2)
    for (int i = threadIdx.x; i < kCoreCols * D; i += kCoreThreads) {
        const int c = i / D, d = i - c * D;
        qs[i] = c < ncol ? to_f32(static_cast<const T*>(p.q)[(hrow0 + c) * D + d]) * p.scale_log2
                         : 0.f;
    }

    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
    const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
    const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(csm);
    const int ntiles = (end - begin + kCoreTile - 1) / kCoreTile;

    // Stage tile i (tokens begin + i*tile ...) into buffer i & 1: a 16-byte
    // cp.async per vector of a valid token's K and V row, zeros otherwise.
    auto stage = [&](int i) {
        const int t0 = begin + i * kCoreTile;
        uint8_t* buf = csm + (i & 1) * Sm::STAGE;
        for (int v = threadIdx.x; v < kCoreTile * Sm::VPR; v += kCoreThreads) {
            const int r = v / Sm::VPR, c = v - r * Sm::VPR;
            const int t = t0 + r;
            const int off = r * Sm::ROW + c * 16;
            int32_t blk = -1;
            if (t < end) {
                blk = table[t / p.block_size];
                if (blk < 0 || blk >= p.num_blocks) {
                    if (c == 0) flag(p.status, PKV_STATUS_BAD_BLOCK);
                    blk = -1;
                }
            }
            if (blk >= 0) {
                const size_t row =
                    ((size_t)blk * p.num_kv_heads + g) * p.block_size + t % p.block_size;
                const size_t src = row * (D * sizeof(T)) + (size_t)c * 16;
                const uint32_t dst = sbase + (uint32_t)((i & 1) * Sm::STAGE + off);
                cp_async16(dst, kc + src);
                cp_async16(dst + Sm::TILE, vc + src);
            } else {
                *reinterpret_cast<uint4*>(buf + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(buf + Sm::TILE + off) = make_uint4(0, 0, 0, 0);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    // softmax state of the heads c = warp + 4k this warp scores (all lanes
    // hold the same copy), and this thread's output accumulators:
    // pair j = (head c_j, float4 column d4)
    constexpr int HPW = kCoreCols / kCoreWarps;
    float m_run[HPW], l_run[HPW];
#pragma unroll
    for (int k = 0; k < HPW; ++k) {
        m_run[k] = -INFINITY;
        l_run[k] = 0.f;
    }
    float4 acc[PAIRS];
#pragma unroll
    for (int j = 0; j < PAIRS; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int d4 = threadIdx.x % ND4;

    if (ntiles > 0) stage(0);
    for (int i = 0; i < ntiles; ++i) {
        if (i + 1 < ntiles) {
            stage(i + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const uint8_t* kt = csm + (i & 1) * Sm::STAGE;
        const uint8_t* vt = kt + Sm::TILE;
        // ---- scores: lane = token, this warp's heads
        const int t = begin + i * kCoreTile + lane;
        bool ok = t < end;
        if (ok) {
            const int32_t blk = table[t / p.block_size];
            ok = blk >= 0 && blk < p.num_blocks;
        }
        float sc[HPW];
#pragma unroll
        for (int k = 0; k < HPW; ++k) sc[k] = 0.f;
        const uint8_t* krow = kt + lane * Sm::ROW;
#pragma unroll 4
        for (int c = 0; c < Sm::VPR; ++c) {
            float kf[Sm::EPV];
            widen_vec<T>(*reinterpret_cast<const uint4*>(krow + c * 16), kf);
#pragma unroll
            for (int k = 0; k < HPW; ++k) {
                const float* qq = qs + (warp + kCoreWarps * k) * D + c * Sm::EPV;
#pragma unroll
                for (int u = 0; u < Sm::EPV; ++u) sc[k] += qq[u] * kf[u];
            }
        }
        // ---- online softmax per head (base 2)
#pragma unroll
        for (int k = 0; k < HPW; ++k) {
            const int col = warp + kCoreWarps * k;
            const float x = ok ? sc[k] : -INFINITY;
            const float m_new = fmaxf(m_run[k], warp_max(x));
            // nothing seen yet (m_new = -inf): alpha 1, p 0
            const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run[k] - m_new);
            const float pz = m_new == -INFINITY ? 0.f : exp2f(x - m_new);
            l_run[k] = l_run[k] * alpha + warp_sum(pz);
            m_run[k] = m_new;
            ps[col * kCoreTile + lane] = pz;
            if (lane == 0) al[col] = alpha;
        }
        __syncthreads();
        // ---- O += P V for this thread's (head, float4) outputs
#pragma unroll
        for (int j = 0; j < PAIRS; ++j) {
            const int col = (threadIdx.x + j * kCoreThreads) / ND4;
            const float a = al[col];
            acc[j].x *= a;
            acc[j].y *= a;
            acc[j].z *= a;
            acc[j].w *= a;
        }
#pragma unroll 4
        for (int r = 0; r < kCoreTile; ++r) {
            const T* vr = reinterpret_cast<const T*>(vt + r * Sm::ROW) + d4 * 4;
            float vf[4];
            if constexpr (sizeof(T) == 4) {
                const float4 v4 = *reinterpret_cast<const float4*>(vr);
                vf[0] = v4.x;
                vf[1] = v4.y;
                vf[2] = v4.z;
                vf[3] = v4.w;
            } else {
                const uint2 raw = *reinterpret_cast<const uint2*>(vr);
                const float2 lo = widen2<T>(raw.x), hi = widen2<T>(raw.y);
                vf[0] = lo.x;
                vf[1] = lo.y;
                vf[2] = hi.x;
                vf[3] = hi.y;
            }
#pragma unroll
            for (int j = 0; j < PAIRS; ++j) {
                const int col = (threadIdx.x + j * kCoreThreads) / ND4;
                const float pz = ps[col * kCoreTile + r];
                acc[j].x += pz * vf[0];
                acc[j].y += pz * vf[1];
                acc[j].z += pz * vf[2];
                acc[j].w += pz * vf[3];
            }
        }
        __syncthreads();  // buffer i & 1 and ps are reused by the next tile
    }

    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < HPW; ++k) {
            const int col = warp + kCoreWarps * k;
            ml[col] = m_run[k];
            ml[kCoreCols + col] = l_run[k];
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < PAIRS; ++j) {
        const int col = (threadIdx.x + j * kCoreThreads) / ND4;
        if (col >= ncol) continue;
        const size_t hrow = hrow0 + col;
        const float den = ml[kCoreCols + col];
        if (nparts <= 1) {
            const float inv = den > 0.f ? 1.f / den : 0.f;
            const size_t o = hrow * D + d4 * 4;
            store_out(p.out, o + 0, acc[j].x * inv, p.out_dtype);
            store_out(p.out, o + 1, acc[j].y * inv, p.out_dtype);
            store_out(p.out, o + 2, acc[j].z * inv, p.out_dtype);
            store_out(p.out, o + 3, acc[j].w * inv, p.out_dtype);
        } else {
            const size_t slot = hrow * p.max_partitions + part;
            *reinterpret_cast<float4*>(p.ws_o + slot * D + d4 * 4) = acc[j];
            if (d4 == 0) p.ws_ml[slot] = make_float2(ml[col], den);
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

// Looked up on every call, in the caller's current context: an address kept
// from an earlier call could belong to a context since destroyed (a device
// reset) or to another one.  The lookup allocates nothing.
unsigned int* pkv_status_word_ptr()
{
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned int*>(ptr);
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
    const size_t per_cta = (size_t)kCopyThreads * kCopyUnroll;
    size_t chunks = (vec + per_cta - 1) / per_cta;
    if (chunks < 1) chunks = 1;
    if (chunks > 65535) chunks = 65535;  // the CTAs then stride over the rest
    dim3 grid(num_pairs, (unsigned)chunks);
    copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(static_cast<uint4*>(k_cache),
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
    const size_t per_unit = (size_t)kSwapThreads * kSwapUnroll;
    const size_t chunks = (vec + per_unit - 1) / per_unit;
    if (chunks > (size_t)INT_MAX) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long units = (long long)num_pairs * (long long)chunks;
    const long long grid = std::min<long long>(units, (long long)kSwapCtasPerSm * sms);
    swap_blocks_kernel<<<(unsigned)grid, kSwapThreads, 0, stream>>>(
        static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), static_cast<const uint4*>(src_k),
        static_cast<const uint4*>(src_v), pairs, num_pairs, num_src_blocks, num_dst_blocks, vec,
        (int)chunks, status);
    return cudaGetLastError();
}

namespace {

template <typename T, int D>
cudaError_t launch_core(const DecodeParams& p, dim3 grid, cudaStream_t stream)
{
    constexpr int bytes = CoreSmem<T, D>::BYTES;
    auto kern = decode_cuda_core_kernel<T, D>;
    // set on every launch: the attribute belongs to the current device's copy
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kCoreThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_core_dim(const DecodeParams& p, dim3 grid, cudaStream_t stream)
{
    return p.head_dim == 64 ? launch_core<T, 64>(p, grid, stream)
                            : launch_core<T, 128>(p, grid, stream);
}

}  // namespace

cudaError_t launch_decode_cuda_core(const DecodeParams& p_in, int kv_dtype, cudaStream_t stream)
{
    // one CTA per (partition, KV head x head slice, sequence); a slice holds
    // at most kCoreCols query heads of the group
    DecodeParams p = p_in;
    const int G = p.num_heads / p.num_kv_heads;
    p.head_slices = (G + kCoreCols - 1) / kCoreCols;
    const long long gy = (long long)p.num_kv_heads * p.head_slices;
    if (gy > 65535 || p.num_seqs > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(p.max_partitions, (unsigned)gy, p.num_seqs);
    if (kv_dtype == PKV_F32) return launch_core_dim<float>(p, grid, stream);
    if (kv_dtype == PKV_F16) return launch_core_dim<__half>(p, grid, stream);
    return launch_core_dim<__nv_bfloat16>(p, grid, stream);
}

cudaError_t launch_lse_reduce(const DecodeParams& p, cudaStream_t stream)
{
    dim3 grid(p.num_heads, p.num_seqs);
    lse_reduce_kernel<<<grid, p.head_dim, 0, stream>>>(p);
    return cudaGetLastError();
}
