// Paged prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// for sm_103a, 16-bit KV cache.
//
// What it computes: the same as the warp-MMA prefill kernel -- rows
// query_start[s] .. query_start[s+1]-1 are the last qn tokens of sequence s
// and row t attends causally to the sequence's tokens 0 .. L-qn+t
// (cayang0802 walkthrough, recomputation; aiplusplus PagedAttention page,
// "key techniques" 1 for the block-table walk).
//
// How (GB300 design):
//  * One CTA of 4 warps per (128 query rows, query head, sequence), latest
//    (heaviest) query tiles first.  Thread r owns query row r: it reads that
//    row of S from tensor memory, so the row max and row sum need no shuffles.
//  * Key/value tiles of 64 tokens arrive by TMA (16-row boxes of the paged
//    cache, 128-byte swizzle, laid out [column half][key][128 B]) through a
//    3-stage mbarrier ring.
//  * S_j = Q K_j^T is one chain of tcgen05.mma (M=128, N=64, K=head_dim, both
//    operands K-major in shared memory) into one of two S buffers in tensor
//    memory, so S_{j+1} runs on the tensor cores while the threads do the
//    softmax of tile j.
//  * O += P_j V_j accumulates in tensor memory (M=128, N=head_dim, K=64; V is
//    the MN-major operand).  P goes to shared memory as a 16-bit high part and
//    remainder and both are multiplied, keeping ~16 bits of P.  A row whose
//    running max grew has its O row rescaled in place (tcgen05.ld / st).
//  * Thread 0 issues every TMA copy and MMA; tcgen05.commit arrives on the
//    mbarriers the threads wait on.  Every wait is bounded; a wait that gives
//    up sets the TIMEOUT status bit (which ends the waits of every other CTA
//    too), and the CTA drains its own copies and MMAs before it frees its
//    tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "pkv.h"
#include "pkv_kernels.h"
#include "tc_common.cuh"

namespace {

using namespace pkv_tc;

constexpr int kRows = 128;   // query rows per CTA (MMA M)
constexpr int kKeys = 64;    // keys per tile (N of S, K of P V)
constexpr int kStages = 3;
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 256;  // S0 [0,64), S1 [64,128), O [128, 128 + D)
constexpr int kBars = kStages + 4;   // kv_full[kStages], s_done[2], o_done, drain

template <int D, int B>
struct G5 {
    static constexpr int NH = D / 64;
    static constexpr int ROWS = B < 16 ? B : 16;  // rows per TMA box
    static constexpr int IDS = 16 / ROWS;         // blocks per 16-token group
    static constexpr int HALF_Q = kRows * 128;    // one 64-column half of Q
    static constexpr int HALF_KV = kKeys * 128;   // one 64-column half of a K or V tile
    static constexpr int Q_OFF = 0;
    static constexpr int STAGE_OFF = Q_OFF + NH * HALF_Q;
    static constexpr int STAGE_BYTES = 2 * NH * HALF_KV;  // K halves, then V halves
    static constexpr int P_OFF = STAGE_OFF + kStages * STAGE_BYTES;
    static constexpr int P_BYTES = kRows * 128;           // 64 keys x 2 bytes per row
    static constexpr int BAR_OFF = P_OFF + 2 * P_BYTES;   // P high part, remainder
    static constexpr int TSLOT_OFF = BAR_OFF + kBars * 8;
    static constexpr int KID_OFF = TSLOT_OFF + 16;        // [stage][4 groups][2] ids
    static constexpr int SMEM_BYTES = 1024 + KID_OFF + kStages * 8 * 4;
    static_assert(HALF_KV % 1024 == 0 && HALF_Q % 1024 == 0, "swizzle atoms");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    // shared-memory matrix descriptor of the sm_100 family: start address,
    // leading and stride byte offsets (all >> 4), version 1, 128-byte swizzle
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

template <typename T>
__device__ __forceinline__ uint32_t instr_desc(int M, int N, int b_mn_major)
{
    // kind::f16 instruction descriptor: fp32 accumulator, A and B of type T
    // (0 = f16, 1 = bf16), A K-major, B K- or MN-major
    const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     int accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// Byte offset of (row, 16-byte chunk) in a [rows][128 B] region with the
// 128-byte swizzle (the region starts on a 1024-byte boundary).
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Plain bounded wait (no early exit on the status bit): drains this CTA's
// own asynchronous work after one of its waits has given up.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > (1ll << 31)) return;
}

template <typename T, int D, int B>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc05_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap)
{
    using Gm = G5<D, B>;
    constexpr int IDS = Gm::IDS;
    const int qtile = gridDim.x - 1 - blockIdx.x;  // latest (heaviest) tiles first
    const int h = blockIdx.y, s = blockIdx.z;
    const int r0 = p.query_start[s];
    const int qn = p.query_start[s + 1] - r0;
    const int L = p.context_lens[s];
    if (L < 0 || (int64_t)L > (int64_t)p.max_blocks * B || qn < 0 || qn > L ||
        qn > p.max_query_len) {
        if (qtile == 0 && h == 0 && threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
        return;
    }
    const int q0 = qtile * kRows;
    if (q0 >= qn) return;
    const int g = h / (p.num_heads / p.num_kv_heads);
    const int base_pos = L - qn;
    const int last_pos = base_pos + min(qn, q0 + kRows) - 1;
    const int nkt = last_pos / kKeys + 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + Gm::BAR_OFF);
    uint64_t* s_done = kv_full + kStages;  // [2]
    uint64_t* o_done = s_done + 2;
    uint64_t* drain = o_done + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Gm::TSLOT_OFF);
    int* kid = reinterpret_cast<int*>(smem + Gm::KID_OFF);
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < kBars; ++i) mbar_init(smem_u32(&kv_full[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tslot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // ---- this thread's query row into shared memory (zero past qn)
    {
        const bool live = q0 + tid < qn;
        const T* src =
            static_cast<const T*>(p.q) + ((size_t)(r0 + q0 + tid) * p.num_heads + h) * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (live) v = *reinterpret_cast<const uint4*>(src + c * 8);
            *reinterpret_cast<uint4*>(smem + Gm::Q_OFF + (c >> 3) * Gm::HALF_Q + swz(tid, c & 7)) =
                v;
        }
    }
    fence_proxy_async();
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = *tslot;

    bool ok = true;
    // Waits for a phase unless this thread already gave up; a wait that gives
    // up flags TIMEOUT at once so that every other waiter stops too.
    auto wait = [&](uint64_t* bar, int parity) {
        if (!ok) return;
        if (!mbar_wait_bounded(smem_u32(bar), (uint32_t)parity, p.status)) {
            ok = false;
            atomicOr(p.status, PKV_STATUS_TIMEOUT);
        }
    };

    // thread 0: TMA loads of key tile kt into stage kt % kStages
    int issued = 0, landed = 0;
    auto issue_tile = [&](int kt) {
        const int st = kt % kStages;
        const uint32_t bar = smem_u32(&kv_full[st]);
        const uint32_t kdst = smem_u32(smem + Gm::STAGE_OFF + st * Gm::STAGE_BYTES);
        const uint32_t vdst = kdst + Gm::NH * Gm::HALF_KV;
        int ids[4][IDS];
        uint32_t bytes = 0;
#pragma unroll
        for (int grp = 0; grp < 4; ++grp)
#pragma unroll
            for (int u = 0; u < IDS; ++u) {
                const int tok = kt * kKeys + grp * 16 + u * Gm::ROWS;
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
                if (id >= 0) bytes += 2 * Gm::NH * Gm::ROWS * 128;
            }
        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int grp = 0; grp < 4; ++grp)
#pragma unroll
            for (int u = 0; u < IDS; ++u) {
                if (ids[grp][u] < 0) continue;
                const int tok = kt * kKeys + grp * 16 + u * Gm::ROWS;
                const int row = (ids[grp][u] * p.num_kv_heads + g) * B + (IDS > 1 ? 0 : tok % B);
                const uint32_t off = (grp * 16 + u * Gm::ROWS) * 128;
#pragma unroll
                for (int hf = 0; hf < Gm::NH; ++hf) {
                    tma_load_2d(kdst + hf * Gm::HALF_KV + off, &kmap, hf * 64, row, bar);
                    tma_load_2d(vdst + hf * Gm::HALF_KV + off, &vmap, hf * 64, row, bar);
                }
            }
        issued = kt + 1;
    };
    const uint32_t id_s = instr_desc<T>(kRows, kKeys, 0);
    const uint32_t id_o = instr_desc<T>(kRows, D, 1);
    // thread 0: S_kt = Q K_kt^T into S buffer kt % 2
    auto issue_s = [&](int kt) {
        const uint32_t q = smem_u32(smem + Gm::Q_OFF);
        const uint32_t kb = smem_u32(smem + Gm::STAGE_OFF + (kt % kStages) * Gm::STAGE_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;
            umma(tbase + (kt & 1) * kKeys, smem_desc(q + (kk >> 2) * Gm::HALF_Q + off, 16, 1024),
                 smem_desc(kb + (kk >> 2) * Gm::HALF_KV + off, 16, 1024), id_s, kk > 0);
        }
        umma_commit(smem_u32(&s_done[kt & 1]));
    };

    if (tid == 0) {
        for (int kt = 0; kt < kStages && kt < nkt; ++kt) issue_tile(kt);
        wait(&kv_full[0], 0);
        if (ok) {
            landed = 1;
            issue_s(0);
        }
    }
    __syncwarp();

    const int row_t = q0 + tid;                          // query row within the sequence
    const int pos = row_t < qn ? base_pos + row_t : -1;  // its position (-1: padding row)
    const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
    const uint32_t o_tmem = tbase + 2 * kKeys;           // O columns (lane 0)
    const float sl = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    uint8_t* phi = smem + Gm::P_OFF;
    uint8_t* plo = phi + Gm::P_BYTES;

    for (int j = 0; j < nkt; ++j) {
        const int st = j % kStages;
        // thread 0: S_{j+1} as soon as its K tile has landed, so the tensor
        // cores work while the threads run this tile's softmax
        if (tid == 0 && j + 1 < nkt) {
            wait(&kv_full[(j + 1) % kStages], ((j + 1) / kStages) & 1);
            if (ok) {
                landed = j + 2;
                issue_s(j + 1);
            }
        }
        __syncwarp();
        wait(&s_done[j & 1], (j >> 1) & 1);
        wait(&kv_full[st], (j / kStages) & 1);
        tmem_fence_after();
        const int key0 = j * kKeys;
        const int* kid_t = kid + st * 8;
        // ---- this row of S_j: scale, causal and validity mask, max
        float sv[kKeys];
        {
            float a[32];
            tmem_ld32(lane_base + (j & 1) * kKeys, a);
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[i] = a[i];
            tmem_ld32(lane_base + (j & 1) * kKeys + 32, a);
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[32 + i] = a[i];
        }
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kKeys; ++k) {
            const bool valid = key0 + k <= pos && kid_t[(k >> 4) * 2 + (k & 15) / Gm::ROWS] >= 0;
            sv[k] = valid ? sv[k] * sl : -INFINITY;
            mx = fmaxf(mx, sv[k]);
        }
        const float mn = fmaxf(m, mx);
        const float ms = mn == -INFINITY ? 0.f : mn;
        const float alpha = ex2(m - ms);  // 0 while m is -inf
        // O holds something to rescale only once m is finite
        const bool grew = m != -INFINITY && alpha != 1.f;
        m = mn;
        float rs = 0.f;
#pragma unroll
        for (int k = 0; k < kKeys; ++k) {
            sv[k] = ex2(sv[k] - ms);
            rs += sv[k];
        }
        l = l * alpha + rs;
        // ---- V rows of keys that were not loaded (past the context, bad
        // block) are zeroed: their P is 0, and 0 * NaN must not reach O
        {
            bool all_loaded = key0 + kKeys <= L;
#pragma unroll
            for (int i = 0; i < 8; ++i) all_loaded = all_loaded && kid_t[i] >= 0;
            if (!all_loaded) {
                uint8_t* vt = smem + Gm::STAGE_OFF + st * Gm::STAGE_BYTES + Gm::NH * Gm::HALF_KV;
                for (int i = tid; i < Gm::NH * kKeys * 8; i += kThreads) {
                    const int hf = i / (kKeys * 8), k = (i >> 3) % kKeys, c = i & 7;
                    if (key0 + k >= L || kid_t[(k >> 4) * 2 + (k & 15) / Gm::ROWS] < 0)
                        *reinterpret_cast<uint4*>(vt + hf * Gm::HALF_KV + k * 128 + c * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        // ---- P V_{j-1} must be done before O is rescaled and P rewritten
        if (j > 0) {
            wait(o_done, (j - 1) & 1);
            tmem_fence_after();
            if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(lane_base + 2 * kKeys + c * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(lane_base + 2 * kKeys + c * 32, o);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
        }
        // ---- P (high part and remainder), row-major by key, swizzled
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                Mma<T>::split(sv[c * 8 + 2 * e], sv[c * 8 + 2 * e + 1], hw[e], lw[e]);
            *reinterpret_cast<uint4*>(phi + swz(tid, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(plo + swz(tid, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async();
        tmem_fence_before();
        __syncthreads();
        tmem_fence_after();
        if (tid == 0 && ok) {
            // stage (j-1) % kStages is free (S_{j-1} and P V_{j-1} are done):
            // refill it with tile j + 2
            if (j > 0 && j + 2 < nkt) issue_tile(j + 2);
            const uint32_t vb =
                smem_u32(smem + Gm::STAGE_OFF + st * Gm::STAGE_BYTES + Gm::NH * Gm::HALF_KV);
            const uint32_t ph = smem_u32(phi), pl = smem_u32(plo);
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
                const uint64_t vd = smem_desc(vb + kk * 2048, Gm::HALF_KV, 1024);
                umma(o_tmem, smem_desc(ph + kk * 32, 16, 1024), vd, id_o, j > 0 || kk > 0);
                umma(o_tmem, smem_desc(pl + kk * 32, 16, 1024), vd, id_o, 1);
            }
            umma_commit(smem_u32(o_done));
        }
        __syncwarp();
    }
    // ---- epilogue: O / l for this thread's row
    wait(o_done, (nkt - 1) & 1);
    tmem_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(lane_base + 2 * kKeys + c * 32, o);
        if (pos >= 0 && ok) {
            const size_t at = ((size_t)(r0 + row_t) * p.num_heads + h) * D + c * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i) store_out(p.out, at + i, o[i] * inv, p.out_dtype);
        }
    }
    if (tid == 0 && !ok) {
        // a wait gave up: let this CTA's copies and MMAs finish before its
        // shared and tensor memory go away
        for (int t = landed; t < issued; ++t)
            drain_wait(smem_u32(&kv_full[t % kStages]), (t / kStages) & 1);
        umma_commit(smem_u32(drain));
        drain_wait(smem_u32(drain), 0);
    }
    __syncwarp();
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                     "r"(kTmemCols)
                     : "memory");
}

template <typename T, int D, int B>
cudaError_t launch5(const PrefillParams& p, const void* kmap, const void* vmap,
                    cudaStream_t stream)
{
    using Gm = G5<D, B>;
    auto kern = prefill_tc05_kernel<T, D, B>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((p.max_query_len + kRows - 1) / kRows, p.num_heads, p.num_seqs);
    kern<<<grid, kThreads, Gm::SMEM_BYTES, stream>>>(p, *static_cast<const CUtensorMap*>(kmap),
                                                     *static_cast<const CUtensorMap*>(vmap));
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch5_dtype(const PrefillParams& p, const void* kmap, const void* vmap,
                          cudaStream_t stream)
{
    if (p.head_dim == 128) {
        if (p.block_size == 16) return launch5<T, 128, 16>(p, kmap, vmap, stream);
        if (p.block_size == 32) return launch5<T, 128, 32>(p, kmap, vmap, stream);
        return launch5<T, 128, 8>(p, kmap, vmap, stream);
    }
    if (p.block_size == 16) return launch5<T, 64, 16>(p, kmap, vmap, stream);
    if (p.block_size == 32) return launch5<T, 64, 32>(p, kmap, vmap, stream);
    return launch5<T, 64, 8>(p, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_prefill_tcgen05(const PrefillParams& p, int kv_dtype, const void* k_map,
                                   const void* v_map, cudaStream_t stream)
{
    if (kv_dtype == PKV_BF16) return launch5_dtype<__nv_bfloat16>(p, k_map, v_map, stream);
    return launch5_dtype<__half>(p, k_map, v_map, stream);
}
