// Tensor-core paged decode attention for sm_103a (16-bit KV cache).
//
// What it computes (aiplusplus PagedAttention page, "key techniques" 1;
// lain42 journal, method: table lookup + block fetch + attention fused in one
// kernel): for each sequence s and query head h of KV group g,
//     out[s,h] = sum_i softmax_i(scale * q[s,h] . k_i) v_i,  i < context_len,
// with k_i, v_i found through the block table.
//
// How (GB300 design):
//  * One CTA = one (partition, KV head, sequence).  All G <= 8 query heads of
//    the group ride along, so every K/V tile is read from HBM once per group
//    (auturnal guide section 1: GQA/MQA shrink the KV head count).
//  * Each (physical block, KV head) tile is B*D contiguous elements.  A 2-D
//    TMA tensor map views a cache as [NB*Hkv*B rows][D cols]; one
//    cp.async.bulk.tensor per 64-column half lands a tile in shared memory
//    with the 128-byte swizzle, completing on an mbarrier.
//  * Each warp owns a ring of NS stages and streams every NW-th stage of the
//    partition; its lane 0 issues the loads NS stages ahead.
//  * Q K^T runs on mma.sync m16n8k16 with tokens on M (16 per tile), the
//    query heads of the group on N (8) and head_dim on K; the score fragment
//    is turned into the P^T operand of the P V product by movmatrix (an 8x8
//    transpose in registers), and P V accumulates O^T (head_dim x heads) in
//    fp32.  P is split into a 16-bit high part and a 16-bit remainder so the
//    product keeps ~16 significant bits.
//  * Online softmax in base 2 with fp32 running max / sum per head; warps
//    merge their states through shared memory at the end.
//  * Masked tokens (past context_len, or in a block whose id is out of range)
//    get score -inf and a zeroed V fragment, so NaN or stale data in unused
//    slots never reaches the output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "pkv.h"
#include "pkv_kernels.h"

namespace {

constexpr int kWarps = 4;

// ---- PTX wrappers -----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of the barrier, giving up after ~2^31 cycles
// (about a second), or at once when another CTA has already given up (the
// TIMEOUT bit of the status word); returns false on giving up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const unsigned int* status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    unsigned int it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > (1ll << 31)) return false;
        if ((++it & 255u) == 0 &&
            (*reinterpret_cast<const volatile unsigned int*>(status) & PKV_STATUS_TIMEOUT))
            return false;
    }
    return true;
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
struct Mma;

template <>
struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // Splits p into a rounded high part and the rounded remainder, packed as
    // (low half = first value) pairs.
    static __device__ __forceinline__ void split(float p0, float p1, uint32_t& hi, uint32_t& lo)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        float2 hf = __bfloat1622float2(h);
        __nv_bfloat162 l = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
        hi = *reinterpret_cast<uint32_t*>(&h);
        lo = *reinterpret_cast<uint32_t*>(&l);
    }
};

template <>
struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ void split(float p0, float p1, uint32_t& hi, uint32_t& lo)
    {
        __half2 h = __floats2half2_rn(p0, p1);
        float2 hf = __half22float2(h);
        __half2 l = __floats2half2_rn(p0 - hf.x, p1 - hf.y);
        hi = *reinterpret_cast<uint32_t*>(&h);
        lo = *reinterpret_cast<uint32_t*>(&l);
    }
};

__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int out_dtype)
{
    if (out_dtype == PKV_F32)
        static_cast<float*>(out)[idx] = v;
    else if (out_dtype == PKV_F16)
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

// Zeroes the 16-bit halves of a packed pair whose token is masked.
__device__ __forceinline__ uint32_t mask_pair(uint32_t x, bool keep_lo, bool keep_hi)
{
    return x & ((keep_lo ? 0x0000FFFFu : 0u) | (keep_hi ? 0xFFFF0000u : 0u));
}

// ---- compile-time geometry -----------------------------------------------------

template <int D, int B>
struct Geometry {
    static constexpr int SB = B >= 16 ? 1 : 16 / B;      // physical blocks per stage
    static constexpr int ST = SB * B;                    // tokens per stage
    static constexpr int TILES = ST / 16;                // 16-token mma tiles per stage
    static constexpr int NH = D / 64;                    // 128-byte column halves
    static constexpr int HALF_BYTES = B * 128;           // one block, one half
    static constexpr int BLOCK_BYTES = NH * HALF_BYTES;  // one block of K (or V)
    static constexpr int KV_BYTES = SB * BLOCK_BYTES;    // K (or V) part of a stage
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    // ring depth: ~24-32 KB of loads in flight per warp
    static constexpr int NS = STAGE_BYTES >= 16384 ? 2 : 3;
    static constexpr int RING_BYTES = NS * STAGE_BYTES;
    static constexpr int MERGE_BYTES = kWarps * 8 * (D + 2) * 4;
    static constexpr int DATA_BYTES =
        (kWarps * RING_BYTES > MERGE_BYTES ? kWarps * RING_BYTES : MERGE_BYTES);
    static constexpr int SMEM_BYTES =
        1024 /*align slack*/ + DATA_BYTES + kWarps * NS * 8 /*barriers*/ + kWarps * NS * SB * 4;
    static_assert(HALF_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");
};

// Shared-memory byte offset of (token row r of the 16-token tile, 16-byte
// chunk c of the head_dim row) inside a K or V stage buffer, honouring the
// 128-byte swizzle the TMA applied (chunk index XOR row % 8).
template <int D, int B>
__device__ __forceinline__ uint32_t tile_offset(int tile, int r, int c)
{
    using Gm = Geometry<D, B>;
    const int tok = tile * 16 + r;       // token within the stage
    const int u = tok / B;               // physical block within the stage
    const int row = tok % B;             // row within the block
    const int half = c >> 3, cc = c & 7;
    return u * Gm::BLOCK_BYTES + half * Gm::HALF_BYTES + row * 128 + ((cc ^ (row & 7)) << 4);
}

template <typename T, int D, int B>
__global__ void __launch_bounds__(kWarps * 32)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap)
{
    using Gm = Geometry<D, B>;
    constexpr int NS = Gm::NS;
    constexpr int KSTEPS = D / 16;  // QK^T k-steps
    constexpr int MTILES = D / 16;  // PV m-tiles (head_dim rows)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::DATA_BYTES);
    int* sid = reinterpret_cast<int*>(bars + kWarps * NS);  // block ids per [warp][slot][unit]

    const int part = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment row group / column pair

    // ---- extent of this CTA's work
    int L = p.context_lens[s];
    if (L < 0 || (int64_t)L > (int64_t)p.max_blocks * B) {
        if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
        L = 0;
    }
    const int nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
    if (part >= (nparts > 0 ? nparts : 1)) return;
    const int begin = part * p.partition_tokens;
    const int end = min(L, begin + p.partition_tokens);
    const int nblk = end > begin ? (end - begin + B - 1) / B : 0;
    const int nst = (nblk + Gm::SB - 1) / Gm::SB;
    const int first_blk = begin / B;
    const int G = p.num_heads / p.num_kv_heads;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;

    // ---- barriers
    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(smem_u32(&bars[warp * NS + i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    __syncwarp();

    // ---- this warp's stages: gs = warp + j * kWarps, j < cnt
    const int cnt = nst > warp ? (nst - warp + kWarps - 1) / kWarps : 0;
    uint8_t* ring = smem + warp * Gm::RING_BYTES;

    // Block ids of this warp's next 32 stages, one (or SB) per lane.
    int win_base = 0;
    int win_ids[Gm::SB];
    auto load_window = [&](int jbase) {
        win_base = jbase;
#pragma unroll
        for (int u = 0; u < Gm::SB; ++u) {
            const int j = jbase + lane;
            const int b = (warp + j * kWarps) * Gm::SB + u;  // block within partition
            int id = -1;
            if (j < cnt && b < nblk) {
                id = table[first_blk + b];
                if (id < 0 || id >= p.num_blocks) {
                    atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
                    id = -1;
                }
            }
            win_ids[u] = id;
        }
    };
    // Block id of stage j, unit u (all lanes call; win_base <= j < win_base + 32).
    auto stage_id = [&](int j, int u) { return __shfl_sync(0xffffffffu, win_ids[u], j - win_base); };

    // Starts the loads of stage j into slot j % NS and records its block ids
    // for the consumer.  Called by the whole warp.
    auto issue = [&](int j) {
        int ids[Gm::SB];
#pragma unroll
        for (int u = 0; u < Gm::SB; ++u) ids[u] = stage_id(j, u);
        if (lane == 0) {
            const int slot = j % NS;
#pragma unroll
            for (int u = 0; u < Gm::SB; ++u) sid[(warp * NS + slot) * Gm::SB + u] = ids[u];
            const uint32_t bar = smem_u32(&bars[warp * NS + slot]);
            const uint32_t kdst = smem_u32(ring + slot * Gm::STAGE_BYTES);
            const uint32_t vdst = kdst + Gm::KV_BYTES;
            uint32_t bytes = 0;
#pragma unroll
            for (int u = 0; u < Gm::SB; ++u)
                if (ids[u] >= 0) bytes += 2 * Gm::BLOCK_BYTES;
            fence_proxy_async();
            mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
            for (int u = 0; u < Gm::SB; ++u) {
                if (ids[u] < 0) continue;
                const int row = (ids[u] * p.num_kv_heads + g) * B;
#pragma unroll
                for (int hf = 0; hf < Gm::NH; ++hf) {
                    const uint32_t off = u * Gm::BLOCK_BYTES + hf * Gm::HALF_BYTES;
                    tma_load_2d(kdst + off, &kmap, hf * 64, row, bar);
                    tma_load_2d(vdst + off, &vmap, hf * 64, row, bar);
                }
            }
        }
    };

    if (cnt > 0) load_window(0);

    // ---- Q^T as the B operand of Q K^T: column n = query head g*G + n.
    uint32_t qb[KSTEPS][2];
    {
        const int n = gq;
        const T* qrow = static_cast<const T*>(p.q) + ((size_t)s * p.num_heads + g * G + n) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            if (n < G) {
                qb[kk][0] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * tq);
                qb[kk][1] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * tq);
            } else {
                qb[kk][0] = qb[kk][1] = 0u;
            }
        }
    }

    // prologue
    for (int j = 0; j < NS && j < cnt; ++j) issue(j);
    __syncwarp();

    // running state for heads 2*tq and 2*tq+1
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[MTILES][4];
#pragma unroll
    for (int i = 0; i < MTILES; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const float sl = p.scale_log2;

    // per-lane ldmatrix row/chunk assignments
    const int lj = lane >> 3, lr = lane & 7;
    const int k_row = (lj & 1) * 8 + lr, k_chunk_add = lj >> 1;  // K: non-transposed A
    const int v_row = (lj >> 1) * 8 + lr, v_chunk_add = lj & 1;  // V: transposed A

    for (int j = 0; j < cnt; ++j) {
        const int slot = j % NS;
        const uint32_t bar = smem_u32(&bars[warp * NS + slot]);
        if (!mbar_wait_bounded(bar, (j / NS) & 1, p.status)) {
            // The copies of this stage never landed: flag, stop issuing, and
            // give the ones still outstanding a bounded wait before leaving.
            if (lane == 0) atomicOr(p.status, PKV_STATUS_TIMEOUT);
            for (int jj = j + 1; jj < j + NS && jj < cnt; ++jj)
                mbar_wait_bounded(smem_u32(&bars[warp * NS + jj % NS]), (jj / NS) & 1, p.status);
            break;
        }
        const int gs = warp + j * kWarps;
        int ids[Gm::SB];
#pragma unroll
        for (int u = 0; u < Gm::SB; ++u) ids[u] = sid[(warp * NS + slot) * Gm::SB + u];
        const uint32_t kbase = smem_u32(ring + slot * Gm::STAGE_BYTES);
        const uint32_t vbase = kbase + Gm::KV_BYTES;
        const int stage_tok0 = begin + gs * Gm::ST;

#pragma unroll
        for (int tile = 0; tile < Gm::TILES; ++tile) {
            const int tok0 = stage_tok0 + tile * 16;
            // validity of this lane's score rows (tokens gq and gq + 8)
            auto valid = [&](int r) {
                const int u = (tile * 16 + r) / B;
                return tok0 + r < end && ids[u] >= 0;
            };
            const bool all_valid = tok0 + 16 <= end && (Gm::SB == 1 ? ids[0] >= 0 : (ids[0] >= 0 && ids[Gm::SB - 1] >= 0));

            // ---- S^T = K Q^T  (16 tokens x 8 heads)
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t a[4];
                ldsm_x4(kbase + tile_offset<D, B>(tile, k_row, 2 * kk + k_chunk_add), a);
                Mma<T>::run(sc, a, qb[kk][0], qb[kk][1]);
            }
            float x0 = sc[0] * sl, x1 = sc[1] * sl, x2 = sc[2] * sl, x3 = sc[3] * sl;
            if (!all_valid) {
                if (!valid(gq)) x0 = x1 = -INFINITY;
                if (!valid(gq + 8)) x2 = x3 = -INFINITY;
            }
            // ---- online softmax (per head: reduce over the 8 row groups)
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ex2(m0 - ms0), al1 = ex2(m1 - ms1);  // 0 while m is -inf
            m0 = mn0;
            m1 = mn1;
            const float p0 = ex2(x0 - ms0), p1 = ex2(x1 - ms1);
            const float p2 = ex2(x2 - ms0), p3 = ex2(x3 - ms1);
            l0 = l0 * al0 + p0 + p2;
            l1 = l1 * al1 + p1 + p3;
#pragma unroll
            for (int i = 0; i < MTILES; ++i) {
                acc[i][0] *= al0;
                acc[i][1] *= al1;
                acc[i][2] *= al0;
                acc[i][3] *= al1;
            }
            // ---- P^T operand: rows gq / gq+8 (tokens) x cols 2tq.. (heads),
            // transposed in registers to (tokens 2tq.. x head gq)
            uint32_t h01, l01, h23, l23;
            Mma<T>::split(p0, p1, h01, l01);
            Mma<T>::split(p2, p3, h23, l23);
            const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
            const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);

            // V fragment tokens held by this lane: 2tq, 2tq+1 (regs 0,1), +8 (regs 2,3)
            bool v0 = true, v1 = true, v8 = true, v9 = true;
            if (!all_valid) {
                v0 = valid(2 * tq);
                v1 = valid(2 * tq + 1);
                v8 = valid(2 * tq + 8);
                v9 = valid(2 * tq + 9);
            }
            // ---- O^T += V^T P^T
#pragma unroll
            for (int i = 0; i < MTILES; ++i) {
                uint32_t a[4];
                ldsm_x4_trans(vbase + tile_offset<D, B>(tile, v_row, 2 * i + v_chunk_add), a);
                if (!all_valid) {
                    a[0] = mask_pair(a[0], v0, v1);
                    a[1] = mask_pair(a[1], v0, v1);
                    a[2] = mask_pair(a[2], v8, v9);
                    a[3] = mask_pair(a[3], v8, v9);
                }
                Mma<T>::run(acc[i], a, bh0, bh1);
                Mma<T>::run(acc[i], a, bl0, bl1);
            }
        }
        __syncwarp();
        if (j + NS < cnt) {
            if (j + NS >= win_base + 32) load_window(j + NS);
            issue(j + NS);
        }
    }

    // ---- per-warp sums over the 8 row groups
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }

    // ---- merge the warps (shared memory reused once every ring is drained)
    __syncthreads();
    float* sm_m = reinterpret_cast<float*>(smem);            // [kWarps][8]
    float* sm_l = sm_m + kWarps * 8;                         // [kWarps][8]
    float* sm_o = sm_l + kWarps * 8;                         // [kWarps][8][D]
    if (gq == 0) {
        sm_m[warp * 8 + 2 * tq] = m0;
        sm_m[warp * 8 + 2 * tq + 1] = m1;
        sm_l[warp * 8 + 2 * tq] = l0;
        sm_l[warp * 8 + 2 * tq + 1] = l1;
    }
#pragma unroll
    for (int i = 0; i < MTILES; ++i) {
        float* o = sm_o + (size_t)warp * 8 * D;
        o[(2 * tq) * D + 16 * i + gq] = acc[i][0];
        o[(2 * tq + 1) * D + 16 * i + gq] = acc[i][1];
        o[(2 * tq) * D + 16 * i + gq + 8] = acc[i][2];
        o[(2 * tq + 1) * D + 16 * i + gq + 8] = acc[i][3];
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int n = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 8 + n]);
        float den = 0.f, num = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float wt = (sm_m[w * 8 + n] == -INFINITY) ? 0.f : ex2(sm_m[w * 8 + n] - M);
            den += wt * sm_l[w * 8 + n];
            num += wt * sm_o[((size_t)w * 8 + n) * D + d];
        }
        const int h = g * G + n;
        if (nparts <= 1) {
            store_out(p.out, ((size_t)s * p.num_heads + h) * D + d, den > 0.f ? num / den : 0.f,
                      p.out_dtype);
        } else {
            const size_t slot = ((size_t)s * p.num_heads + h) * p.max_partitions + part;
            p.ws_o[slot * D + d] = num;
            if (d == 0) p.ws_ml[slot] = make_float2(M, den);
        }
    }
}

template <typename T, int D, int B>
cudaError_t launch_tc(const DecodeParams& p, const void* kmap, const void* vmap,
                      cudaStream_t stream)
{
    using Gm = Geometry<D, B>;
    auto kern = decode_tc_kernel<T, D, B>;
    // set on every launch: the attribute belongs to the current device's copy
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(p.max_partitions, p.num_kv_heads, p.num_seqs);
    kern<<<grid, kWarps * 32, Gm::SMEM_BYTES, stream>>>(
        p, *static_cast<const CUtensorMap*>(kmap), *static_cast<const CUtensorMap*>(vmap));
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_tc_dtype(const DecodeParams& p, const void* kmap, const void* vmap,
                            cudaStream_t stream)
{
    if (p.head_dim == 128) {
        if (p.block_size == 16) return launch_tc<T, 128, 16>(p, kmap, vmap, stream);
        if (p.block_size == 32) return launch_tc<T, 128, 32>(p, kmap, vmap, stream);
        return launch_tc<T, 128, 8>(p, kmap, vmap, stream);
    }
    if (p.block_size == 16) return launch_tc<T, 64, 16>(p, kmap, vmap, stream);
    if (p.block_size == 32) return launch_tc<T, 64, 32>(p, kmap, vmap, stream);
    return launch_tc<T, 64, 8>(p, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_decode_tensor_core(const DecodeParams& p, int kv_dtype, const void* k_map,
                                      const void* v_map, cudaStream_t stream)
{
    if (kv_dtype == PKV_BF16) return launch_tc_dtype<__nv_bfloat16>(p, k_map, v_map, stream);
    return launch_tc_dtype<__half>(p, k_map, v_map, stream);
}
