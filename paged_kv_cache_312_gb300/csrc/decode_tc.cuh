// Tensor-core paged decode attention for sm_103a (16-bit KV cache).
//
// What it computes (aiplusplus PagedAttention page, "key techniques" 1;
// lain42 journal, method: table lookup + block fetch + attention fused in one
// kernel): for each sequence s and query head h of KV group g,
//     out[s,h] = sum_i softmax_i(scale * q[s,h] . k_i) v_i,  i < context_len,
// with k_i, v_i found through the block table.
//
// How (GB300 design):
//  * One CTA per (sequence, KV head, partition of <= P tokens), or per four
//    consecutive partitions when they are short (<= 512 tokens, one per
//    warp, so that a CTA's start-up and end are spread over more bytes); the
//    slots of one (sequence, KV head) are adjacent in the grid and slots past
//    a sequence's end exit at once.  All G <= 8 query heads of the KV group
//    ride along, so every K/V tile is read from HBM once per group (auturnal
//    guide section 1: GQA/MQA shrink the KV head count).
//  * A stage is 16 tokens of K and V.  A 3-D TMA tensor map views a cache as
//    [D/64 column halves][NB*Hkv*B rows][64 cols] (the halves' stride, 128
//    bytes, is below the rows'); one cp.async.bulk.tensor per block of the
//    stage lands it in shared memory, half after half, with the 128-byte
//    swizzle, and completes on an mbarrier.  Each of the 4 warps
//    streams every 4th stage of its CTA's partition (or every stage of its
//    own partition) through its own ring of NS stages; its lane 0
//    issues loads NS stages ahead.  Block ids are fetched 32 stages at a time
//    (one per lane) and broadcast by shuffle.  Three CTAs share an SM, so one
//    CTA's start-up latency hides behind the others' streaming.
//  * Q K^T runs on mma.sync m16n8k16 with tokens on M, the group's query heads
//    on N (8) and head_dim on K (two independent accumulation chains);
//    movmatrix turns the score fragment into the P^T operand of P V, which
//    accumulates O^T in fp32.  P is split into a 16-bit high part and a
//    16-bit remainder (~16 significant bits).
//  * Online softmax in base 2 (fp32) against a per-head reference max that
//    moves only when a score passes it by more than 8, so most stages need
//    neither a cross-lane max nor a rescale of O; the warps of a partition merge through
//    shared memory (reusing the rings) at the end.  An unsplit item writes
//    the output; a partition writes (max, sum, unnormalised output) to the
//    workspace, the CTA bumps its (sequence, KV head) counter by its number
//    of partitions, and the CTA that completes the count merges all
//    partitions by log-sum-exp.
//  * Beam groups (GR): one CTA per (group, KV head) attends every member of a
//    group of sequences that share a prefix of physical blocks: the shared
//    prefix once with all members' query heads as the N columns, then each
//    member's own tail with the other columns masked (cayang0802 "Paged
//    Attention" page, beam-search paragraph: the beams keep one physical
//    copy of their common blocks).
//  * Masked tokens (past context_len, or in a block whose id is out of range)
//    get score -inf and a zeroed V fragment, so NaN or stale data in unused
//    slots never reaches the output.
//  * Every wait is bounded (~1 s); a wait that gives up sets the TIMEOUT
//    status bit, which makes every other wait give up at once.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <climits>
#include <cstdint>

#include "pkv.h"
#include "pkv_kernels.h"
#include "tc_common.cuh"

namespace {

using namespace pkv_tc;

// ---- compile-time geometry -----------------------------------------------------

template <int D, int B, int NW, int NS>
struct Geometry {
    static constexpr int ROWS = B < 16 ? B : 16;     // rows per TMA box
    static constexpr int IDS = 16 / ROWS;            // physical blocks per 16-token stage
    static constexpr int NH = D / 64;                // 128-byte column halves
    static constexpr int SUB_BYTES = ROWS * 128;     // one box
    static constexpr int KV_BYTES = 16 * D * 2;      // K (or V) of a 16-token stage
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int RING_BYTES = NS * STAGE_BYTES;
    static constexpr int MERGE_BYTES = NW * 8 * (D + 2) * 4;
    static constexpr int DATA_BYTES =
        NW * RING_BYTES > MERGE_BYTES ? NW * RING_BYTES : MERGE_BYTES;  // merge reuses rings
    static constexpr int BAR_OFF = DATA_BYTES;
    static constexpr int SID_OFF = BAR_OFF + NW * NS * 8;
    // per ring slot: block ids of the stage (2), and for beam groups its first
    // token, region end and member (3)
    static constexpr int SID_INTS = 8;
    static constexpr int SMEM_BYTES = 1024 /*align slack*/ + SID_OFF + NW * NS * SID_INTS * 4;
    // partition weights cached for the in-kernel merge (after the warp merge)
    static constexpr int WCACHE = ((DATA_BYTES - MERGE_BYTES) / 4 - 16 - NW * 32 * 4 - 4) & ~3;
    static_assert(WCACHE > 0, "room for merge weights");
    static_assert(SUB_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static_assert(STAGE_BYTES % 1024 == 0 && RING_BYTES % 1024 == 0, "stage alignment");
};

// Shared-memory offset of (token row r of the stage, 16-byte chunk c of the
// head_dim row) in a K or V stage buffer laid out [block][half][row][128 B],
// honouring the 128-byte swizzle (chunk XOR row % 8).
template <int D, int B, int NW, int NS>
__device__ __forceinline__ uint32_t stage_offset(int r, int c)
{
    using Gm = Geometry<D, B, NW, NS>;
    const int u = r / Gm::ROWS, row = r % Gm::ROWS;
    const int half = c >> 3, cc = c & 7;
    return (u * Gm::NH + half) * Gm::SUB_BYTES + row * 128 + ((cc ^ (row & 7)) << 4);
}

// One CTA = one work item: one partition of one (sequence, KV head), whose
// 16-token stages the NW warps stream in turn (warp w takes stages w, w + NW,
// ...) through rings of NS stages each, merging their softmax states at the
// end; or, for short split partitions, up to NW consecutive partitions, one
// per warp, each warp's state being its partition's result.
template <typename T, int D, int B, int NW, int NS, bool GR>
__global__ void __launch_bounds__(NW * 32)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap)
{
    using Gm = Geometry<D, B, NW, NS>;
    constexpr int KSTEPS = D / 16;  // Q K^T k-steps
    constexpr int MTILES = D / 16;  // P V m-tiles (head_dim rows)
    constexpr int IDS = Gm::IDS;    // physical blocks per stage (2 when B = 8)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.num_heads / p.num_kv_heads;
    int s, g, sg, L, nparts, p0, np_cta, wpp, wsub, part, begin, end, nst;
    bool solo;
    // Beam groups (GR): one CTA per (group, KV head).  The group's members
    // are sequences s0 .. s0 + nm - 1 whose first `shared` tokens sit in the
    // same physical blocks; the CTA streams that shared prefix once for all
    // members (their query heads are the mma's N columns, nm * G <= 8), then
    // each member's own tail with the other members' columns masked.
    int s0 = 0, nm = 1, shared = 0, nsh = 0;
    int Lm[8];
    if constexpr (GR) {
        const int gi = blockIdx.x / p.num_kv_heads;
        g = blockIdx.x - gi * p.num_kv_heads;
        s0 = p.group_start[gi];
        nm = p.group_start[gi + 1] - s0;
        if (nm < 1 || nm * G > 8 || s0 < 0 || s0 + nm > p.num_seqs) {
            if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
            return;
        }
        int min_len = INT_MAX;  // (the new token of a decode step stays private)
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            int l = 0;
            if (m < nm) {
                l = p.context_lens[s0 + m];
                if (l < 0 || (int64_t)l > (int64_t)p.max_blocks * B) {
                    if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
                    l = 0;
                }
                min_len = min(min_len, p.new_k != nullptr ? l - 1 : l);
            }
            Lm[m] = l;
        }
        shared = max(0, min(p.shared_tokens[gi], min_len)) & ~15;
        nsh = shared / 16;
        nst = nsh;
#pragma unroll
        for (int m = 0; m < 8; ++m)
            if (m < nm) nst += (Lm[m] - shared + 15) / 16;
        s = s0;
        sg = 0;
        L = Lm[0];
        nparts = 1;
        p0 = 0;
        np_cta = 1;
        solo = true;
        wpp = NW;
        wsub = warp;
        part = 0;
        begin = 0;
        end = 0;
    } else {
        // ---- which item: slot b = ((s * Hkv) + g) * max_groups + grp; group
        // grp holds partitions grp * cta_parts .. + cta_parts - 1 of (s, g)
        const int max_groups = (p.max_partitions + p.cta_parts - 1) / p.cta_parts;
        const int grp = blockIdx.x % max_groups;
        sg = blockIdx.x / max_groups;
        s = sg / p.num_kv_heads;
        g = sg - s * p.num_kv_heads;
        L = p.context_lens[s];
        if (L < 0 || (int64_t)L > (int64_t)p.max_blocks * B) {
            if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
            L = 0;
        }
        nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
        p0 = grp * p.cta_parts;
        if (p0 >= (nparts > 0 ? nparts : 1)) return;
        // np_cta partitions here: a single one is spread over all NW warps
        // (warp w streams its stages w, w + NW, ...); several get a warp each,
        // and warps past np_cta have nothing to stream.
        np_cta = min(p.cta_parts, (nparts > 0 ? nparts : 1) - p0);
        solo = np_cta == 1;
        wpp = solo ? NW : 1;       // warps per partition
        wsub = solo ? warp : 0;    // this warp's rank within it
        part = solo ? p0 : p0 + warp;
        begin = part * p.partition_tokens;
        end = min(L, begin + p.partition_tokens);
        nst = end > begin ? (end - begin + 15) / 16 : 0;
    }
    // GR: CTA stage q -> first token, end of its region, member (-1: shared)
    auto stage_at = [&](int q, int& tok0, int& endr, int& mem) {
        if (q < nsh) {
            tok0 = q * 16;
            endr = shared;
            mem = -1;
            return;
        }
        int r = q - nsh;
        mem = -1;
        tok0 = 0;
        endr = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int st = m < nm ? (Lm[m] - shared + 15) / 16 : 0;
            if (mem < 0) {
                if (r < st) {
                    mem = m;
                    tok0 = shared + r * 16;
                    endr = Lm[m];
                } else {
                    r -= st;
                }
            }
        }
    };
    auto table_of = [&](int mem) {
        return p.block_tables + (size_t)(GR ? s0 + max(mem, 0) : s) * p.max_blocks;
    };

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::BAR_OFF);
    int* sid = reinterpret_cast<int*>(smem + Gm::SID_OFF);  // [warp][slot][2] block ids

    const int gq = lane >> 2, tq = lane & 3;  // mma fragment row group / column pair
    uint8_t* ring = smem + warp * Gm::RING_BYTES;
    const int32_t* table = table_of(-1);

    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(smem_u32(&bars[warp * NS + i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    __syncwarp();

    // ---- this warp's stages of its partition: q = wsub + j * wpp, j < cnt
    const int cnt = nst > wsub ? (nst - wsub + wpp - 1) / wpp : 0;
    int win_base = 0;
    int win_ids[IDS];
    int win_tok = 0, win_end = 0, win_mem = -1;  // GR: the lane's stage
    // Block ids of this warp's stages jbase .. jbase+31, one per lane.
    auto load_window = [&](int jbase) {
        win_base = jbase;
        const int j = jbase + lane;
        int tk0 = begin + (wsub + j * wpp) * 16, endr = end, mem = -1;
        if constexpr (GR) {
            if (j < cnt) stage_at(warp + j * NW, tk0, endr, mem);
            win_tok = tk0;
            win_end = endr;
            win_mem = mem;
        }
        const int32_t* tab = GR ? table_of(mem) : table;
#pragma unroll
        for (int u = 0; u < IDS; ++u) {
            int id = -1;
            const int tok = tk0 + u * B;  // first token of the box
            if (j < cnt && tok < endr) {
                id = tab[tok / B];
                if (id < 0 || id >= p.num_blocks) {
                    atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
                    id = -1;
                }
            }
            win_ids[u] = id;
        }
    };
    // Starts the loads of stage j into slot j % NS (whole warp calls).
    auto issue = [&](int j) {
        int ids[IDS];
#pragma unroll
        for (int u = 0; u < IDS; ++u) ids[u] = __shfl_sync(0xffffffffu, win_ids[u], j - win_base);
        int tok0 = begin + (wsub + j * wpp) * 16;
        int endr = end, mem = -1;
        if constexpr (GR) {
            tok0 = __shfl_sync(0xffffffffu, win_tok, j - win_base);
            endr = __shfl_sync(0xffffffffu, win_end, j - win_base);
            mem = __shfl_sync(0xffffffffu, win_mem, j - win_base);
        }
        if (lane == 0) {
            const int slot = j % NS;
            int* sd = sid + (warp * NS + slot) * Gm::SID_INTS;
            sd[0] = ids[0];
            sd[1] = ids[IDS - 1];
            if constexpr (GR) {
                sd[2] = tok0;
                sd[3] = endr;
                sd[4] = mem;
            }
            const uint32_t bar = smem_u32(&bars[warp * NS + slot]);
            const uint32_t kdst = smem_u32(ring + slot * Gm::STAGE_BYTES);
            const uint32_t vdst = kdst + Gm::KV_BYTES;
            uint32_t bytes = 0;
#pragma unroll
            for (int u = 0; u < IDS; ++u)
                if (ids[u] >= 0) bytes += 2 * Gm::NH * Gm::SUB_BYTES;
            fence_proxy_async();
            mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
            for (int u = 0; u < IDS; ++u) {
                if (ids[u] < 0) continue;
                // B >= 16: one 16-row box at the stage's offset in its block;
                // B == 8: one 8-row box per block.
                const int row = (ids[u] * p.num_kv_heads + g) * B + (IDS > 1 ? 0 : tok0 % B);
                // one box brings both 64-column halves (the tensor map's
                // outer dimension steps over them)
                const uint32_t off = u * Gm::NH * Gm::SUB_BYTES;
                tma_load_3d(kdst + off, &kmap, 0, row, 0, bar);
                tma_load_3d(vdst + off, &vmap, 0, row, 0, bar);
            }
        }
        __syncwarp();
    };

    // ---- decode step with append: the warp that streams the stage holding
    // position len-1 of sequence seq first writes this KV head's slice of the
    // new token there (16 bytes per lane), then orders the write before its
    // own TMA reads
    auto append = [&](int seq, int len, const int32_t* tab) {
        const int id = tab[(len - 1) / B];
        if (id < 0 || id >= p.num_blocks) {
            if (lane == 0) atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
        } else {
            constexpr int CH = D * (int)sizeof(T) / 16;  // 16-byte chunks per row
            const int c = lane % CH;
            const bool is_v = lane >= CH;
            if (lane < 2 * CH) {
                const size_t src = ((size_t)seq * p.num_kv_heads + g) * D;
                const size_t dst = (((size_t)id * p.num_kv_heads + g) * B + (len - 1) % B) * D;
                const uint4 v = reinterpret_cast<const uint4*>(
                    static_cast<const T*>(is_v ? p.new_v : p.new_k) + src)[c];
                reinterpret_cast<uint4*>(
                    const_cast<T*>(static_cast<const T*>(is_v ? p.v_cache : p.k_cache)) + dst)[c] = v;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __syncwarp();
    };
    if (p.new_k != nullptr) {
        if constexpr (GR) {
            // member m's new token (always past the shared prefix) lies in
            // CTA stage nsh + (stages of members before m) + (L_m-1-shared)/16
            int qb0 = nsh;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                if (m < nm) {
                    if (Lm[m] > shared && (qb0 + (Lm[m] - 1 - shared) / 16) % NW == warp)
                        append(s0 + m, Lm[m], table_of(m));
                    qb0 += (Lm[m] - shared + 15) / 16;
                }
            }
        } else if (L > 0 && begin <= L - 1 && L - 1 < end && ((L - 1 - begin) / 16) % wpp == wsub) {
            append(s, L, table);
        }
    }

    if (cnt > 0) load_window(0);
    for (int j = 0; j < NS && j < cnt; ++j) issue(j);

    // ---- Q^T as the B operand of Q K^T: column n = query head g*G + n (GR:
    // member n / G, query head g*G + n % G).
    uint32_t qb[KSTEPS][2];
    {
        const int n = gq;
        const int mn = GR ? n / G : 0, hn = GR ? n - mn * G : n;
        const bool col = GR ? mn < nm : n < G;
        const T* qrow = static_cast<const T*>(p.q) +
                        ((size_t)(GR ? s0 + min(mn, nm - 1) : s) * p.num_heads + g * G + hn) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            if (col) {
                qb[kk][0] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * tq);
                qb[kk][1] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * tq);
            } else {
                qb[kk][0] = qb[kk][1] = 0u;
            }
        }
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2tq, 2tq+1
    float acc[MTILES][4];
#pragma unroll
    for (int i = 0; i < MTILES; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const float sl = p.scale_log2;
    const int lj = lane >> 3, lr = lane & 7;
    const int k_row = (lj & 1) * 8 + lr, k_chunk_add = lj >> 1;  // K: non-transposed A
    const int v_row = (lj >> 1) * 8 + lr, v_chunk_add = lj & 1;  // V: transposed A

    for (int j = 0; j < cnt; ++j) {
        const int slot = j % NS;
        const uint32_t bar = smem_u32(&bars[warp * NS + slot]);
        if (!mbar_wait_bounded(bar, (j / NS) & 1, p.status)) {
            // The copies of this stage never landed: flag, stop, and give this
            // stage and the ones still outstanding a bounded wait (one that
            // does not stop at the TIMEOUT bit just set) before leaving.
            if (lane == 0) atomicOr(p.status, PKV_STATUS_TIMEOUT);
            for (int jj = j; jj < j + NS && jj < cnt; ++jj)
                mbar_drain_wait(smem_u32(&bars[warp * NS + jj % NS]), (jj / NS) & 1);
            break;
        }
        const int* sinfo = sid + (warp * NS + slot) * Gm::SID_INTS;
        const int id0 = sinfo[0];
        const int id1 = sinfo[1];
        const uint32_t kbase = smem_u32(ring + slot * Gm::STAGE_BYTES);
        const uint32_t vbase = kbase + Gm::KV_BYTES;
        const int tok0 = GR ? sinfo[2] : begin + (wsub + j * wpp) * 16;
        const int endr = GR ? sinfo[3] : end;
        auto valid = [&](int r) {
            return tok0 + r < endr && ((IDS > 1 && r >= B) ? id1 : id0) >= 0;
        };
        const bool all_valid = tok0 + 16 <= endr && id0 >= 0 && id1 >= 0;

        // ---- S^T = K Q^T  (16 tokens x 8 heads), as two independent
        // accumulation chains (even and odd k-steps)
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            uint32_t a[4];
            ldsm_x4(kbase + stage_offset<D, B, NW, NS>(k_row, 2 * kk + k_chunk_add), a);
            if (kk & 1)
                Mma<T>::run(sd, a, qb[kk][0], qb[kk][1]);
            else
                Mma<T>::run(sc, a, qb[kk][0], qb[kk][1]);
        }
        float x0 = (sc[0] + sd[0]) * sl, x1 = (sc[1] + sd[1]) * sl;
        float x2 = (sc[2] + sd[2]) * sl, x3 = (sc[3] + sd[3]) * sl;
        if (!all_valid) {
            if (!valid(gq)) x0 = x1 = -INFINITY;
            if (!valid(gq + 8)) x2 = x3 = -INFINITY;
        }
        if constexpr (GR) {
            // a member's own tail: the other members' columns see nothing
            const int mem = sinfo[4];
            if (mem >= 0) {
                if ((2 * tq) / G != mem) x0 = x2 = -INFINITY;
                if ((2 * tq + 1) / G != mem) x1 = x3 = -INFINITY;
            }
        }
        // ---- online softmax in base 2 against a reference max per head that
        // moves only when a score passes it by more than 8 (so p <= 2^8): most
        // stages need neither the max over the 8 row groups nor a rescale of O
        const bool up = fmaxf(x0, x2) > m0 + 8.f || fmaxf(x1, x3) > m1 + 8.f;
        if (__any_sync(0xffffffffu, up)) {
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            // 0 while m is -inf (nothing accumulated yet), 1 if m stays
            const float al0 = mn0 == -INFINITY ? 1.f : ex2(m0 - mn0);
            const float al1 = mn1 == -INFINITY ? 1.f : ex2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int i = 0; i < MTILES; ++i) {
                acc[i][0] *= al0;
                acc[i][1] *= al1;
                acc[i][2] *= al0;
                acc[i][3] *= al1;
            }
        }
        const float ms0 = m0 == -INFINITY ? 0.f : m0;
        const float ms1 = m1 == -INFINITY ? 0.f : m1;
        const float p0 = ex2(x0 - ms0), p1 = ex2(x1 - ms1);
        const float p2 = ex2(x2 - ms0), p3 = ex2(x3 - ms1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // ---- P^T operand (tokens 2tq.. x head gq) via an in-register transpose
        uint32_t h01, l01, h23, l23;
        Mma<T>::split(p0, p1, h01, l01);
        Mma<T>::split(p2, p3, h23, l23);
        const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
        const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);

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
            ldsm_x4_trans(vbase + stage_offset<D, B, NW, NS>(v_row, 2 * i + v_chunk_add), a);
            if (!all_valid) {
                a[0] = mask_pair(a[0], v0, v1);
                a[1] = mask_pair(a[1], v0, v1);
                a[2] = mask_pair(a[2], v8, v9);
                a[3] = mask_pair(a[3], v8, v9);
            }
            Mma<T>::run(acc[i], a, bh0, bh1);
            Mma<T>::run(acc[i], a, bl0, bl1);
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

    const size_t hbase = (size_t)s * p.num_heads + (size_t)g * G;
    if (!solo) {
        // ---- a warp's own partition: its softmax state is the partition's
        // result, written straight to the workspace (heads 2tq and 2tq + 1)
        if (warp < np_cta) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = 2 * tq + h;
                if (n >= G) break;
                const size_t slot = (hbase + n) * p.max_partitions + part;
                if (gq == 0) p.ws_ml[slot] = make_float2(h ? m1 : m0, h ? l1 : l0);
                float* o = p.ws_o + slot * D;
#pragma unroll
                for (int i = 0; i < MTILES; ++i) {
                    o[16 * i + gq] = acc[i][h];
                    o[16 * i + gq + 8] = acc[i][2 + h];
                }
            }
        }
    } else {
        // ---- merge the warps (shared memory reused once every ring is drained)
        __syncthreads();
        float* wm = reinterpret_cast<float*>(smem) + warp * 8 * (D + 2);  // [8][D], m[8], l[8]
        if (gq == 0) {
            wm[8 * D + 2 * tq] = m0;
            wm[8 * D + 2 * tq + 1] = m1;
            wm[8 * D + 8 + 2 * tq] = l0;
            wm[8 * D + 8 + 2 * tq + 1] = l1;
        }
#pragma unroll
        for (int i = 0; i < MTILES; ++i) {
            wm[(2 * tq) * D + 16 * i + gq] = acc[i][0];
            wm[(2 * tq + 1) * D + 16 * i + gq] = acc[i][1];
            wm[(2 * tq) * D + 16 * i + gq + 8] = acc[i][2];
            wm[(2 * tq + 1) * D + 16 * i + gq + 8] = acc[i][3];
        }
        __syncthreads();
        const float* sm = reinterpret_cast<const float*>(smem);
        // four consecutive outputs of one head per thread
        const bool vec_out = (reinterpret_cast<uintptr_t>(p.out) & 15) == 0;
        const int ncol = GR ? nm * G : G;
        for (int idx = threadIdx.x; idx < ncol * D / 4; idx += blockDim.x) {
            const int n = idx / (D / 4), d = (idx - n * (D / 4)) * 4;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, sm[w * 8 * (D + 2) + 8 * D + n]);
            float den = 0.f;
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float* ww = sm + w * 8 * (D + 2);
                const float mw = ww[8 * D + n];
                const float wt = mw == -INFINITY ? 0.f : ex2(mw - M);
                den += wt * ww[8 * D + 8 + n];
                const float4 o = *reinterpret_cast<const float4*>(ww + n * D + d);
                num.x += wt * o.x;
                num.y += wt * o.y;
                num.z += wt * o.z;
                num.w += wt * o.w;
            }
            if (nparts <= 1) {
                const bool pos = den > 0.f;
                const size_t orow =
                    GR ? ((size_t)(s0 + n / G) * p.num_heads + g * G + n % G) : hbase + n;
                store_out4(p.out, orow * D + d,
                           make_float4(pos ? num.x / den : 0.f, pos ? num.y / den : 0.f,
                                       pos ? num.z / den : 0.f, pos ? num.w / den : 0.f),
                           p.out_dtype, vec_out);
            } else {
                const size_t slot = (hbase + n) * p.max_partitions + part;
                *reinterpret_cast<float4*>(p.ws_o + slot * D + d) = num;
                if (d == 0) p.ws_ml[slot] = make_float2(M, den);
            }
        }
        if (nparts <= 1) return;
    }

    // ---- split: the CTA that finishes the last partition of (s, g) merges
    // them by log-sum-exp: M = max_i m_i, w_i = 2^(m_i - M),
    // out = sum_i w_i O_i / sum_i w_i l_i.
    __shared__ int is_last;
    __syncthreads();  // this CTA's partition results are written ...
    if (threadIdx.x == 0) {
        // release: this CTA's partition results (ordered before this thread by
        // the barrier) are visible before the count goes up; acquire for the
        // CTA that completes the count: it sees every other partition's results
        unsigned prev;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                     : "=r"(prev)
                     : "l"(&p.done[sg]), "r"((unsigned)np_cta)
                     : "memory");
        is_last = prev == (unsigned)(nparts - np_cta);
    }
    __syncthreads();
    if (!is_last) return;
    constexpr int NT = NW * 32;
    float* wts = reinterpret_cast<float*>(smem) + NW * 8 * (D + 2);  // [G][nparts] weights
    float* hinv = wts + Gm::WCACHE;                                    // [8]
    float* hmax = hinv + 8;                                            // [8]
    float4* red = reinterpret_cast<float4*>(hmax + 8);                 // [NT] partial sums
    const bool cached = G * nparts <= Gm::WCACHE;
    for (int n = warp; n < G; n += NW) {
        const size_t base = (hbase + n) * p.max_partitions;
        // the (max, sum) pairs of the first 64 partitions are read once and
        // kept in registers for both passes; any further ones are re-read
        float2 ml[2];
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = lane + 32 * r;
            ml[r] = i < nparts ? __ldcg(&p.ws_ml[base + i]) : make_float2(-INFINITY, 0.f);
            M = fmaxf(M, ml[r].x);
        }
        for (int i = lane + 64; i < nparts; i += 32) M = fmaxf(M, __ldcg(&p.ws_ml[base + i]).x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float den = 0.f;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = lane + 32 * r;
            if (i < nparts) {
                const float w = ml[r].x == -INFINITY ? 0.f : ex2(ml[r].x - M);
                if (cached) wts[n * nparts + i] = w;
                den += w * ml[r].y;
            }
        }
        for (int i = lane + 64; i < nparts; i += 32) {
            const float2 mli = __ldcg(&p.ws_ml[base + i]);
            const float w = mli.x == -INFINITY ? 0.f : ex2(mli.x - M);
            if (cached) wts[n * nparts + i] = w;
            den += w * mli.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (lane == 0) {
            hmax[n] = M;
            hinv[n] = den > 0.f ? 1.f / den : 0.f;
        }
    }
    __syncthreads();
    // Outputs in float4 units; when the group has fewer of them than
    // threads, K threads share one output, each summing every K-th partition.
    const int O4 = G * D / 4;
    const int K = O4 >= NT ? 1 : NT / O4;
    for (int o0 = 0; o0 < O4; o0 += NT) {
        const int t = threadIdx.x;
        const int o = o0 + (K == 1 ? t : t % O4), k = K == 1 ? 0 : t / O4;
        float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
        const bool active = o < O4 && k < K;
        if (active) {
            const int n = o / (D / 4), d4 = o - n * (D / 4);
            const size_t base = (hbase + n) * p.max_partitions;
            const float4* src = reinterpret_cast<const float4*>(p.ws_o + base * D) + d4;
#pragma unroll 16
            for (int i = k; i < nparts; i += K) {
                float w;
                if (cached) {
                    w = wts[n * nparts + i];
                } else {
                    const float mi = __ldcg(&p.ws_ml[base + i]).x;
                    w = mi == -INFINITY ? 0.f : ex2(mi - hmax[n]);
                }
                const float4 v = __ldcg(src + (size_t)i * (D / 4));
                acc4.x += w * v.x;
                acc4.y += w * v.y;
                acc4.z += w * v.z;
                acc4.w += w * v.w;
            }
        }
        if (K > 1) {
            red[t] = acc4;
            __syncthreads();
            if (k == 0 && active) {
                for (int kk = 1; kk < K; ++kk) {
                    const float4 r = red[t + kk * O4];
                    acc4.x += r.x;
                    acc4.y += r.y;
                    acc4.z += r.z;
                    acc4.w += r.w;
                }
            }
        }
        if (k == 0 && active) {
            const int n = o / (D / 4), d = (o - n * (D / 4)) * 4;
            const float inv = hinv[n];
            const size_t at = (hbase + n) * D + d;
            store_out(p.out, at + 0, acc4.x * inv, p.out_dtype);
            store_out(p.out, at + 1, acc4.y * inv, p.out_dtype);
            store_out(p.out, at + 2, acc4.z * inv, p.out_dtype);
            store_out(p.out, at + 3, acc4.w * inv, p.out_dtype);
        }
    }
}

template <typename T, int D, int B, bool GR>
cudaError_t launch_tc(const DecodeParams& p, const void* kmap, const void* vmap, long long grid,
                      cudaStream_t stream)
{
    // 4 warps x 2-stage rings: 64 KB (D = 128) per CTA, three CTAs per SM,
    // up to 192 KB of tile loads in flight per SM
    constexpr int NW = kDecodeTcWarps, NS = 2;
    using Gm = Geometry<D, B, NW, NS>;
    auto kern = decode_tc_kernel<T, D, B, NW, NS, GR>;
    // set on every launch: the attribute belongs to the current device's copy
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, NW * 32, Gm::SMEM_BYTES, stream>>>(
        p, *static_cast<const CUtensorMap*>(kmap), *static_cast<const CUtensorMap*>(vmap));
    return cudaGetLastError();
}

template <typename T, bool GR>
cudaError_t launch_tc_dtype(const DecodeParams& p, const void* kmap, const void* vmap,
                            long long grid, cudaStream_t stream)
{
    if (p.head_dim == 128) {
        if (p.block_size == 16) return launch_tc<T, 128, 16, GR>(p, kmap, vmap, grid, stream);
        if (p.block_size == 32) return launch_tc<T, 128, 32, GR>(p, kmap, vmap, grid, stream);
        return launch_tc<T, 128, 8, GR>(p, kmap, vmap, grid, stream);
    }
    if (p.block_size == 16) return launch_tc<T, 64, 16, GR>(p, kmap, vmap, grid, stream);
    if (p.block_size == 32) return launch_tc<T, 64, 32, GR>(p, kmap, vmap, grid, stream);
    return launch_tc<T, 64, 8, GR>(p, kmap, vmap, grid, stream);
}

}  // namespace
