// Tensor-core paged prefill attention for sm_103a (16-bit KV cache).
//
// What it computes: several new query tokens per sequence -- a prompt, or a
// chunk of one -- each attending causally to the sequence's cached tokens up
// to its own position (the parallel pass that recomputing a preempted
// sequence's KV relies on, cayang0802 walkthrough, recomputation).  Rows
// query_start[s] .. query_start[s+1]-1 are the last qn tokens of sequence s:
//     out[row t, h] = sum_{i <= L-qn+t} softmax_i(scale q[t,h] . k_i) v_i
// with k_i, v_i reached through the block table (aiplusplus PagedAttention
// page, "key techniques" 1).
//
// How (GB300 design):
//  * One CTA of 4 warps per (64-row query tile, query head, sequence); each
//    warp owns 16 query rows.  K/V arrive 64 keys at a time by TMA (16-token
//    boxes of the paged cache, 128-byte swizzle) through a 2-stage mbarrier
//    ring; thread 0 issues the next tile once every warp has left a stage.
//  * S = Q K^T on mma.sync m16n8k16 (query rows on M, keys on N, head_dim on
//    K), online softmax per row in base 2, then O += P V with the score
//    fragments reused directly as the A operand; P is split into a 16-bit
//    high part and remainder as in the decode kernel.
//  * Causal and validity masks by select; V rows of keys past the context or
//    in a bad block are zeroed so NaN in unused slots cannot leak.  Key tiles
//    entirely above a warp's last row are skipped by that warp.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "pkv.h"
#include "pkv_kernels.h"
#include "tc_common.cuh"

namespace {

using namespace pkv_tc;

constexpr int kQT = 64;     // query rows per CTA
constexpr int kKT = 64;     // keys per tile
constexpr int kStages = 2;  // K/V tiles in flight
constexpr int kThreads = 128;

template <int D, int B>
struct PGeom {
    static constexpr int ROWS = B < 16 ? B : 16;  // rows per TMA box
    static constexpr int IDS = 16 / ROWS;         // blocks per 16-token group
    static constexpr int NH = D / 64;             // 128-byte column halves
    static constexpr int SUB_BYTES = ROWS * 128;
    static constexpr int GROUP_BYTES = 16 * D * 2;        // 16 tokens of K (or V)
    static constexpr int KV_BYTES = (kKT / 16) * GROUP_BYTES;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int Q_BYTES = kQT * D * 2;
    static constexpr int Q_OFF = kStages * STAGE_BYTES;
    static constexpr int BAR_OFF = Q_OFF + Q_BYTES;
    static constexpr int KID_OFF = BAR_OFF + kStages * 8;          // [stage][4 groups][2] ids
    static constexpr int SMEM_BYTES = 1024 + KID_OFF + kStages * 8 * 4;
    static_assert(SUB_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "alignment");
};

// Offset of (key k of the tile, 16-byte chunk c) in a K or V tile buffer
// laid out [16-token group][block][half][row][128 B] with the 128-byte swizzle.
template <int D, int B>
__device__ __forceinline__ uint32_t key_offset(int k, int c)
{
    using Pg = PGeom<D, B>;
    const int grp = k >> 4, r = k & 15;
    const int u = r / Pg::ROWS, row = r % Pg::ROWS;
    const int half = c >> 3, cc = c & 7;
    return grp * Pg::GROUP_BYTES + (u * Pg::NH + half) * Pg::SUB_BYTES + row * 128 +
           ((cc ^ (row & 7)) << 4);
}

// Offset of (query row r of the tile, 16-byte chunk c) in the Q buffer laid
// out [half][row][128 B] with the same swizzle.
template <int D>
__device__ __forceinline__ uint32_t q_offset(int r, int c)
{
    const int half = c >> 3, cc = c & 7;
    return half * (kQT * 128) + r * 128 + ((cc ^ (r & 7)) << 4);
}

template <typename T, int D, int B>
__global__ void __launch_bounds__(kThreads, 2)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap)
{
    using Pg = PGeom<D, B>;
    constexpr int KSTEPS = D / 16;  // Q K^T k-steps
    constexpr int NT_D = D / 8;     // P V n-tiles (head_dim columns)
    constexpr int IDS = Pg::IDS;

    const int qtile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int r0 = p.query_start[s];
    const int qn = p.query_start[s + 1] - r0;
    int L = p.context_lens[s];
    const bool bad = L < 0 || (int64_t)L > (int64_t)p.max_blocks * B || qn < 0 || qn > L ||
                     qn > p.max_query_len;
    if (bad) {
        if (qtile == 0 && h == 0 && threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
        return;
    }
    const int q0 = qtile * kQT;
    if (q0 >= qn) return;
    const int G = p.num_heads / p.num_kv_heads;
    const int g = h / G;
    const int base_pos = L - qn;                      // position of query row 0
    const int last_pos = base_pos + min(qn, q0 + kQT) - 1;
    const int nkt = last_pos / kKT + 1;               // key tiles this CTA needs

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Pg::BAR_OFF);
    int* kid = reinterpret_cast<int*>(smem + Pg::KID_OFF);
    uint8_t* qs = smem + Pg::Q_OFF;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&bars[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    __syncthreads();

    // Thread 0: start the loads of key tile kt into stage kt % kStages.
    int issued = 0, landed = 0;  // thread 0: tiles whose copies it started / saw land
    auto issue = [&](int kt) {
        issued = kt + 1;
        const int st = kt % kStages;
        const uint32_t bar = smem_u32(&bars[st]);
        const uint32_t kdst = smem_u32(smem + st * Pg::STAGE_BYTES);
        const uint32_t vdst = kdst + Pg::KV_BYTES;
        int ids[kKT / 16][IDS];
        uint32_t bytes = 0;
        for (int grp = 0; grp < kKT / 16; ++grp) {
            for (int u = 0; u < IDS; ++u) {
                const int tok = kt * kKT + grp * 16 + u * Pg::ROWS;
                int id = -1;
                if (tok < L) {
                    id = table[tok / B];
                    if (id < 0 || id >= p.num_blocks) {
                        atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
                        id = -1;
                    }
                }
                ids[grp][u] = id;
                kid[(st * 4 + grp) * 2 + u] = id;
                if (IDS == 1) kid[(st * 4 + grp) * 2 + 1] = id;
                if (id >= 0) bytes += 2 * Pg::NH * Pg::SUB_BYTES;
            }
        }
        fence_proxy_async();
        mbar_arrive_expect_tx(bar, bytes);
        for (int grp = 0; grp < kKT / 16; ++grp) {
            for (int u = 0; u < IDS; ++u) {
                const int id = ids[grp][u];
                if (id < 0) continue;
                const int tok = kt * kKT + grp * 16 + u * Pg::ROWS;
                const int row = (id * p.num_kv_heads + g) * B + (IDS > 1 ? 0 : tok % B);
                for (int hf = 0; hf < Pg::NH; ++hf) {
                    const uint32_t off = grp * Pg::GROUP_BYTES + (u * Pg::NH + hf) * Pg::SUB_BYTES;
                    tma_load_2d(kdst + off, &kmap, hf * 64, row, bar);
                    tma_load_2d(vdst + off, &vmap, hf * 64, row, bar);
                }
            }
        }
    };
    if (threadIdx.x == 0)
        for (int kt = 0; kt < kStages && kt < nkt; ++kt) issue(kt);

    // ---- the query tile into shared memory (rows past qn are zero)
    {
        constexpr int CH = D / 8;  // 16-byte chunks per row
        for (int i = threadIdx.x; i < kQT * CH; i += kThreads) {
            const int r = i / CH, c = i - r * CH;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (q0 + r < qn)
                v = *reinterpret_cast<const uint4*>(
                    static_cast<const T*>(p.q) + ((size_t)(r0 + q0 + r) * p.num_heads + h) * D +
                    c * 8);
            *reinterpret_cast<uint4*>(qs + q_offset<D>(r, c)) = v;
        }
    }
    __syncthreads();
    uint32_t qa[KSTEPS][4];
    {
        const int lj = lane >> 3, lr = lane & 7;
        const int row = warp * 16 + (lj & 1) * 8 + lr;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk)
            ldsm_x4(smem_u32(qs) + q_offset<D>(row, 2 * kk + (lj >> 1)), qa[kk]);
    }

    // rows of this thread: warp*16 + gq and + 8; their positions
    const int tr0 = q0 + warp * 16 + gq, tr1 = tr0 + 8;
    const int pos0 = tr0 < qn ? base_pos + tr0 : -1;
    const int pos1 = tr1 < qn ? base_pos + tr1 : -1;
    const int warp_last = min(qn - 1, q0 + warp * 16 + 15);
    const int warp_last_pos = warp_last >= q0 + warp * 16 ? base_pos + warp_last : -1;

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[NT_D][4];
#pragma unroll
    for (int n = 0; n < NT_D; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    const float sl = p.scale_log2;
    const int lj = lane >> 3, lr = lane & 7;
    const int kb_key = (lj >> 1) * 8 + lr, kb_chunk = lj & 1;  // K as B: non-transposed
    const int vb_key = (lj & 1) * 8 + lr, vb_chunk = lj >> 1;  // V as B: transposed
    bool aborted = false;

    for (int kt = 0; kt < nkt; ++kt) {
        const int st = kt % kStages;
        if (!aborted && !mbar_wait_bounded(smem_u32(&bars[st]), (kt / kStages) & 1, p.status)) {
            if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_TIMEOUT);
            aborted = true;
        }
        if (!aborted) landed = kt + 1;
        const int key0 = kt * kKT;
        if (!aborted && key0 <= warp_last_pos) {
            const uint32_t kbase = smem_u32(smem + st * Pg::STAGE_BYTES);
            const uint32_t vbase = kbase + Pg::KV_BYTES;
            // key validity: inside the context and in a good block
            const bool tile_clean = key0 + kKT <= L && kid[(st * 4 + 0) * 2] >= 0 &&
                                    kid[(st * 4 + 1) * 2] >= 0 && kid[(st * 4 + 2) * 2] >= 0 &&
                                    kid[(st * 4 + 3) * 2] >= 0 && kid[(st * 4 + 0) * 2 + 1] >= 0 &&
                                    kid[(st * 4 + 1) * 2 + 1] >= 0 &&
                                    kid[(st * 4 + 2) * 2 + 1] >= 0 &&
                                    kid[(st * 4 + 3) * 2 + 1] >= 0;
            auto key_ok = [&](int k) {  // k within the tile
                const int grp = k >> 4, u = (k & 15) / PGeom<D, B>::ROWS;
                return key0 + k < L && kid[(st * 4 + grp) * 2 + u] >= 0;
            };
            // ---- S = Q K^T (16 rows x 64 keys per warp)
            float sc[kKT / 8][4];
#pragma unroll
            for (int n = 0; n < kKT / 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
                for (int jp = 0; jp < kKT / 16; ++jp) {
                    uint32_t b[4];
                    ldsm_x4(kbase + key_offset<D, B>(jp * 16 + kb_key, 2 * kk + kb_chunk), b);
                    Mma<T>::run(sc[2 * jp], qa[kk], b[0], b[1]);
                    Mma<T>::run(sc[2 * jp + 1], qa[kk], b[2], b[3]);
                }
            }
            // ---- masks (causal per row; validity per key) and online softmax
            const bool need_mask = !tile_clean || key0 + kKT - 1 > pos0 || key0 + kKT - 1 > pos1;
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < kKT / 8; ++n) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = n * 8 + 2 * tq + e;
                    float x0 = sc[n][e] * sl, x1 = sc[n][2 + e] * sl;
                    if (need_mask) {
                        const bool ok = key_ok(k);
                        if (!ok || key0 + k > pos0) x0 = -INFINITY;
                        if (!ok || key0 + k > pos1) x1 = -INFINITY;
                    }
                    sc[n][e] = x0;
                    sc[n][2 + e] = x1;
                    mx0 = fmaxf(mx0, x0);
                    mx1 = fmaxf(mx1, x1);
                }
            }
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ex2(m0 - ms0), al1 = ex2(m1 - ms1);
            m0 = mn0;
            m1 = mn1;
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int n = 0; n < kKT / 8; ++n) {
                sc[n][0] = ex2(sc[n][0] - ms0);
                sc[n][1] = ex2(sc[n][1] - ms0);
                sc[n][2] = ex2(sc[n][2] - ms1);
                sc[n][3] = ex2(sc[n][3] - ms1);
                rs0 += sc[n][0] + sc[n][1];
                rs1 += sc[n][2] + sc[n][3];
            }
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
#pragma unroll
            for (int n = 0; n < NT_D; ++n) {
                acc[n][0] *= al0;
                acc[n][1] *= al0;
                acc[n][2] *= al1;
                acc[n][3] *= al1;
            }
            // ---- O += P V: the score fragments of keys 16j..16j+15 are the A
            // operand of k-step j
#pragma unroll
            for (int j = 0; j < kKT / 16; ++j) {
                uint32_t ph[4], pl[4];
                Mma<T>::split(sc[2 * j][0], sc[2 * j][1], ph[0], pl[0]);
                Mma<T>::split(sc[2 * j][2], sc[2 * j][3], ph[1], pl[1]);
                Mma<T>::split(sc[2 * j + 1][0], sc[2 * j + 1][1], ph[2], pl[2]);
                Mma<T>::split(sc[2 * j + 1][2], sc[2 * j + 1][3], ph[3], pl[3]);
                // this lane's V keys: 16j + 2tq (+1) for b0, + 8 for b1
                bool k0 = true, k1 = true, k8 = true, k9 = true;
                if (!tile_clean) {
                    k0 = key_ok(16 * j + 2 * tq);
                    k1 = key_ok(16 * j + 2 * tq + 1);
                    k8 = key_ok(16 * j + 8 + 2 * tq);
                    k9 = key_ok(16 * j + 9 + 2 * tq);
                }
#pragma unroll
                for (int cp = 0; cp < NT_D / 2; ++cp) {
                    uint32_t b[4];
                    ldsm_x4_trans(vbase + key_offset<D, B>(16 * j + vb_key, 2 * cp + vb_chunk), b);
                    if (!tile_clean) {
                        b[0] = mask_pair(b[0], k0, k1);
                        b[1] = mask_pair(b[1], k8, k9);
                        b[2] = mask_pair(b[2], k0, k1);
                        b[3] = mask_pair(b[3], k8, k9);
                    }
                    Mma<T>::run(acc[2 * cp], ph, b[0], b[1]);
                    Mma<T>::run(acc[2 * cp], pl, b[0], b[1]);
                    Mma<T>::run(acc[2 * cp + 1], ph, b[2], b[3]);
                    Mma<T>::run(acc[2 * cp + 1], pl, b[2], b[3]);
                }
            }
        }
        __syncthreads();  // every warp is done with stage st
        if (threadIdx.x == 0 && !aborted && kt + kStages < nkt) issue(kt + kStages);
    }
    if (__syncthreads_or(aborted)) {
        // a wait gave up: the copies thread 0 started and did not see land get
        // a bounded wait before the CTA's shared memory goes away
        if (threadIdx.x == 0)
            for (int kt = landed; kt < issued; ++kt)
                mbar_drain_wait(smem_u32(&bars[kt % kStages]), (kt / kStages) & 1);
        return;
    }

    // ---- normalise and store this thread's two rows
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int n = 0; n < NT_D; ++n) {
        const int d = n * 8 + 2 * tq;
        if (pos0 >= 0) {
            const size_t o = ((size_t)(r0 + tr0) * p.num_heads + h) * D + d;
            store_out(p.out, o, acc[n][0] * inv0, p.out_dtype);
            store_out(p.out, o + 1, acc[n][1] * inv0, p.out_dtype);
        }
        if (pos1 >= 0) {
            const size_t o = ((size_t)(r0 + tr1) * p.num_heads + h) * D + d;
            store_out(p.out, o, acc[n][2] * inv1, p.out_dtype);
            store_out(p.out, o + 1, acc[n][3] * inv1, p.out_dtype);
        }
    }
}

template <typename T, int D, int B>
cudaError_t launch_prefill(const PrefillParams& p, const void* kmap, const void* vmap,
                           cudaStream_t stream)
{
    using Pg = PGeom<D, B>;
    auto kern = prefill_tc_kernel<T, D, B>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Pg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((p.max_query_len + kQT - 1) / kQT, p.num_heads, p.num_seqs);
    kern<<<grid, kThreads, Pg::SMEM_BYTES, stream>>>(p, *static_cast<const CUtensorMap*>(kmap),
                                                     *static_cast<const CUtensorMap*>(vmap));
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_dtype(const PrefillParams& p, const void* kmap, const void* vmap,
                                 cudaStream_t stream)
{
    if (p.head_dim == 128) {
        if (p.block_size == 16) return launch_prefill<T, 128, 16>(p, kmap, vmap, stream);
        if (p.block_size == 32) return launch_prefill<T, 128, 32>(p, kmap, vmap, stream);
        return launch_prefill<T, 128, 8>(p, kmap, vmap, stream);
    }
    if (p.block_size == 16) return launch_prefill<T, 64, 16>(p, kmap, vmap, stream);
    if (p.block_size == 32) return launch_prefill<T, 64, 32>(p, kmap, vmap, stream);
    return launch_prefill<T, 64, 8>(p, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_prefill_tensor_core(const PrefillParams& p, int kv_dtype, const void* k_map,
                                       const void* v_map, cudaStream_t stream)
{
    if (kv_dtype == PKV_BF16) return launch_prefill_dtype<__nv_bfloat16>(p, k_map, v_map, stream);
    return launch_prefill_dtype<__half>(p, k_map, v_map, stream);
}
