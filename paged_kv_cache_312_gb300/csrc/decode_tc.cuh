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
//    a sequence's end exit at once.  The query heads of the KV group ride
//    along as the mma's N columns, so every K/V tile is read from HBM once
//    per group (auturnal guide section 1: GQA/MQA shrink the KV head count):
//    one n8 tile for G <= 8, two for G <= 16 (NT = 2); a wider group is cut
//    into head slices of at most 16 columns, one CTA each, adjacent in the
//    grid so that the slices' repeated reads of a tile meet in L2.
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
//    on N (8 per tile) and head_dim on K (independent accumulation chains);
//    movmatrix turns the score fragment into the P^T operand of P V, which
//    accumulates O^T in fp32.  P is split into a 16-bit high part and a
//    16-bit remainder (~16 significant bits).
//  * Online softmax in base 2 (fp32) against a per-head reference max that
//    moves only when a score passes it by more than 8, so most stages need
//    neither a cross-lane max nor a rescale of O; the warps of a partition
//    merge through shared memory (reusing the rings) at the end.  An unsplit item writes
//    the output; a partition writes (max, sum, unnormalised output) to the
//    workspace, the CTA bumps its (sequence, KV head) counter by its number
//    of partitions, and the CTA that completes the count merges all
//    partitions by log-sum-exp.
//  * Beam groups (GR): one CTA per (group, KV head) attends every member of a
//    group of sequences that share a prefix of physical blocks: the shared
//    prefix once with all members' query heads as the N columns (up to 8 or
//    16), then each member's own tail with the other columns masked
//    (cayang0802 "Paged Attention" page, beam-search paragraph: the beams
//    keep one physical copy of their common blocks).  A group may be cut into
//    equal runs of its stage list, one CTA each, merged like partitions.
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

template <int D, int B, int NW, int NS, int NT = 1, int TPS = 1>
struct Geometry {
    static constexpr int NC = 8 * NT;                // query-head columns (n8 tiles x 8)
    static constexpr int ST = 16 * TPS;              // tokens per stage: TPS m16 token tiles
    static constexpr int ROWS = B < ST ? B : ST;     // rows per TMA box
    static constexpr int IDS = ST / ROWS;            // physical blocks per stage
    static constexpr int NH = D / 64;                // 128-byte column halves
    static constexpr int SUB_BYTES = ROWS * 128;     // one box
    static constexpr int KV_BYTES = ST * D * 2;      // K (or V) of a stage
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int RING_BYTES = NS * STAGE_BYTES;
    static constexpr int MERGE_BYTES = NW * NC * (D + 2) * 4;
    static constexpr int DATA_BYTES =
        NW * RING_BYTES > MERGE_BYTES ? NW * RING_BYTES : MERGE_BYTES;  // merge reuses rings
    static constexpr int BAR_OFF = DATA_BYTES;
    static constexpr int SID_OFF = BAR_OFF + NW * NS * 8;
    // per ring slot: block ids of the stage (IDS <= 4), and for beam groups its
    // first token, region end and member
    static constexpr int SID_INTS = 8;
    static constexpr int SID_TOK = 4, SID_END = 5, SID_MEM = 6;
    static_assert(IDS <= SID_TOK, "block ids of a stage fit the slot record");
    static constexpr int GM_OFF = SID_OFF + NW * NS * SID_INTS * 4;  // beam groups: [NC] lengths
    static constexpr int SMEM_BYTES = 1024 /*align slack*/ + GM_OFF + NC * 4;
    // partition weights cached for the in-kernel merge (after the warp merge)
    static constexpr int WCACHE = ((DATA_BYTES - MERGE_BYTES) / 4 - 2 * NC - NW * 32 * 4 - 4) & ~3;
    static_assert(WCACHE > 0, "room for merge weights");
    // CTAs per SM the register allocation is held to: as many as the shared
    // memory admits (8 KB stages -- D = 128, or D = 64 with 32-token stages --
    // 3 of ~66 KB, up to 168 registers a thread; 4 KB stages: 6 of ~34 KB, 80
    // registers), or 5 for two column tiles with 4 KB stages (96).  Left to
    // itself the compiler took 96 registers at D = 128, and the freedom to use
    // more is worth 1-4 % of HBM bandwidth there; with 4 KB stages it spilled.
    static constexpr int MIN_CTAS = KV_BYTES >= 4096 ? (NS >= 3 ? 2 : 3) : (NT == 1 ? 6 : 5);
    static_assert(SUB_BYTES % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static_assert(STAGE_BYTES % 1024 == 0 && RING_BYTES % 1024 == 0, "stage alignment");
};

// Shared-memory offset of (token row r of the stage, 16-byte chunk c of the
// head_dim row) in a K or V stage buffer laid out [block][half][row][128 B],
// honouring the 128-byte swizzle (chunk XOR row % 8).
template <class Gm>
__device__ __forceinline__ uint32_t stage_offset(int r, int c)
{
    const int u = r / Gm::ROWS, row = r % Gm::ROWS;
    const int half = c >> 3, cc = c & 7;
    return (u * Gm::NH + half) * Gm::SUB_BYTES + row * 128 + ((cc ^ (row & 7)) << 4);
}

// One CTA = one work item: one partition of one (sequence, KV head, head
// slice), or one run of a beam group's stage list, whose stages of 16 * TPS
// tokens the NW warps stream in turn (warp w takes stages w, w + NW, ...)
// through rings of NS stages each, merging their softmax states at the end;
// or, for short split partitions, up to NW consecutive partitions, one per
// warp, each warp's state being its partition's result.  NT n8 tiles carry up
// to 8 * NT query-head columns.  A stage of TPS = 2 (head_dim 64: 8 KB, as a
// 16-token stage at head_dim 128) is two m16 token tiles, taken one after the
// other against the same running softmax state.
template <typename T, int D, int B, int NW, int NS, bool GR, int NT, int TPS>
__global__ void __launch_bounds__(NW * 32, (Geometry<D, B, NW, NS, NT, TPS>::MIN_CTAS))
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap)
{
    using Gm = Geometry<D, B, NW, NS, NT, TPS>;
    static_assert(!GR || TPS == 1, "beam groups stream 16-token stages");
    constexpr int ST = Gm::ST;      // tokens per stage
    constexpr int NC = Gm::NC;      // query-head columns of the mma's N (8 per tile)
    constexpr int KSTEPS = D / 16;  // Q K^T k-steps
    constexpr int MTILES = D / 16;  // P V m-tiles (head_dim rows)
    constexpr int IDS = Gm::IDS;    // physical blocks per stage (2 when B = 8)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.num_heads / p.num_kv_heads;
    // a work plan for the next call (a programmatic dependent of this launch)
    // may start once every CTA has started: it reads only lengths until this
    // launch completes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int s, g, sg, L, nparts, p0, np_cta, wpp, wsub, part, begin, end, nst;
    // this CTA's partial: index pidx_v of ncp_v per (sequence, KV head, head
    // slice), or (GR) of (group, KV head); ncp_v <= 1: the output itself
    int ncp_v = 1, pidx_v = 0;
    // this CTA's query heads: g*G + hb .. + ncol - 1 (all of the KV group,
    // or one slice of at most NC of them when the group is wider)
    int hb = 0, ncol;
    bool solo;
    // Beam groups (GR): one CTA per (group, KV head, part).  The group's members
    // are sequences s0 .. s0 + nm - 1 whose first `shared` tokens sit in the
    // same physical blocks; the CTA streams that shared prefix once for all
    // members (their query heads are the mma's N columns, nm * G <= NC), then
    // each member's own tail with the other members' columns masked.
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* glen = reinterpret_cast<int*>(smem + Gm::GM_OFF);  // GR: members' context lengths
    int s0 = 0, nm = 1, shared = 0, nsh = 0, qbase = 0;
    // non-GR: block ids of this warp's first 32 stages, read before the
    // context length arrives (see below)
    int spec_ids[IDS];
    bool spec_solo = true;
    if constexpr (GR) {
        // slot b = (gi * Hkv + g) * parts + part: part `part` of the group's
        // stage list (shared prefix, then each member's tail) for KV head g
        const int gparts = p.max_partitions;
        sg = blockIdx.x / gparts;
        part = blockIdx.x - sg * gparts;
        const int gi = sg / p.num_kv_heads;
        g = sg - gi * p.num_kv_heads;
        s0 = p.group_start[gi];
        nm = p.group_start[gi + 1] - s0;
        if (nm < 1 || nm * G > NC || s0 < 0 || s0 + nm > p.num_seqs) {
            if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
            return;
        }
        if (threadIdx.x < nm) {
            int l = p.context_lens[s0 + threadIdx.x];
            if (l < 0 || (int64_t)l > (int64_t)p.max_blocks * B) {
                atomicOr(p.status, PKV_STATUS_BAD_LEN);
                l = 0;
            }
            glen[threadIdx.x] = l;
        }
        __syncthreads();
        int min_len = INT_MAX;  // (the new token of a decode step stays private)
        for (int m = 0; m < nm; ++m) min_len = min(min_len, p.new_k != nullptr ? glen[m] - 1 : glen[m]);
        shared = max(0, min(p.shared_tokens[gi], min_len)) & ~15;
        nsh = shared / 16;
        int total = nsh;
        for (int m = 0; m < nm; ++m) total += (glen[m] - shared + 15) / 16;
        // this CTA's run of the list: stages qbase .. qbase + nst - 1
        qbase = (int)((int64_t)part * total / gparts);
        nst = (int)((int64_t)(part + 1) * total / gparts) - qbase;
        s = s0;
        ncol = nm * G;
        L = glen[0];
        nparts = gparts;
        ncp_v = gparts;
        pidx_v = part;
        p0 = 0;
        np_cta = 1;
        solo = true;
        wpp = NW;
        wsub = warp;
        begin = 0;
        end = 0;
    } else {
        // ---- which item: with a work plan, record b = (s, L, g * HS + hs,
        // grp or piece); else slot b = (((s * Hkv) + g) * max_groups + grp) *
        // HS + hs.  Group grp holds partitions grp * cta_parts .. + cta_parts
        // - 1 of (s, g), for head slice hs of the KV group's query heads;
        // piece i of n holds stages [i * nst / n, (i + 1) * nst / n) of the
        // sequence's nst = ceil(L / ST).  The head slices of one group are
        // adjacent, so that their reads of the same K/V tiles meet in L2.
        const int HS = p.head_slices;
        int grp, plan_len = 0, piece = -1, npieces = 0;
        if (p.items != nullptr) {
            // launched as a dependent of the plan kernel: wait until it has
            // completed and its writes (records, zeroed counters) are visible
            asm volatile("griddepcontrol.wait;" ::: "memory");
            const int4 it = p.items[blockIdx.x];  // read with the count: past it, stale
            const int count = *p.item_count;
            if ((int)blockIdx.x >= count) return;
            if (it.x < 0 || it.x >= p.num_seqs || it.z < 0 || it.z >= p.num_kv_heads * HS) {
                if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
                return;
            }
            sg = it.x * (p.num_kv_heads * HS) + it.z;
            plan_len = it.y;
            grp = it.w;
            if (it.w & kPlanPieceFlag) {
                piece = it.w & kPlanPieceMask;
                npieces = (it.w >> kPlanPieceBits) & kPlanPieceMask;
                grp = 0;
                if (npieces < 1 || piece >= npieces || npieces > p.max_partitions) {
                    if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
                    return;
                }
            }
        } else {
            const int max_groups = (p.max_partitions + p.cta_parts - 1) / p.cta_parts;
            const int hs_b = blockIdx.x % HS, t = blockIdx.x / HS;
            grp = t % max_groups;
            sg = (t / max_groups) * HS + hs_b;
        }
        const int sgk = sg / HS, hs = sg - sgk * HS;
        s = sgk / p.num_kv_heads;
        g = sgk - s * p.num_kv_heads;
        const int GC = (G + HS - 1) / HS;
        hb = hs * GC;
        ncol = min(GC, G - hb);
        // a piece's stages [sb, se), from the length in its record
        int sb = 0, se = 0;
        if (piece >= 0) {
            const bool ok = plan_len >= 0 && (int64_t)plan_len <= (int64_t)p.max_blocks * B;
            const int nsq = ok ? (plan_len + ST - 1) / ST : 0;
            sb = (int)((int64_t)piece * nsq / npieces);
            se = (int)((int64_t)(piece + 1) * nsq / npieces);
        }
        // The first window of block ids depends on the context length only
        // through the partition-to-warp mapping, which is known in advance
        // unless a CTA of several partitions ends up with one: so it is read
        // now, overlapping the length's round trip, and used below when the
        // guess holds (entries past the context are then ignored).
        {
            spec_solo = piece >= 0 || p.cta_parts == 1;
            const int gpart = grp * p.cta_parts + (spec_solo ? 0 : warp);
            const int64_t gtok = (piece >= 0 ? (int64_t)sb * ST
                                             : (int64_t)gpart * p.partition_tokens) +
                                 (int64_t)(spec_solo ? warp + lane * NW : lane) * ST;
            const int32_t* row = p.block_tables + (size_t)s * p.max_blocks;
#pragma unroll
            for (int u = 0; u < IDS; ++u) {
                const int64_t tok = gtok + u * B;
                spec_ids[u] = tok < (int64_t)p.max_blocks * B ? row[tok / B] : -1;
            }
        }
        L = p.items != nullptr ? plan_len : p.context_lens[s];
        if (L < 0 || (int64_t)L > (int64_t)p.max_blocks * B) {
            if (threadIdx.x == 0) atomicOr(p.status, PKV_STATUS_BAD_LEN);
            L = 0;
        }
        if (piece >= 0) {
            // one run of stages, spread over all NW warps like one partition
            nparts = npieces;
            p0 = piece;
            np_cta = 1;
            solo = true;
            wpp = NW;
            wsub = warp;
            part = piece;
            begin = sb * ST;
            end = min(L, se * ST);
            nst = end > begin ? se - sb : 0;
            ncp_v = npieces;
            pidx_v = piece;
        } else {
            nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
            p0 = grp * p.cta_parts;
            if (p0 >= (nparts > 0 ? nparts : 1)) return;
            // np_cta partitions here: a single one is spread over all NW
            // warps (warp w streams its stages w, w + NW, ...); several get a
            // warp each, and warps past np_cta have nothing to stream.
            np_cta = min(p.cta_parts, (nparts > 0 ? nparts : 1) - p0);
            solo = np_cta == 1;
            wpp = solo ? NW : 1;       // warps per partition
            wsub = solo ? warp : 0;    // this warp's rank within it
            part = solo ? p0 : p0 + warp;
            begin = part * p.partition_tokens;
            end = min(L, begin + p.partition_tokens);
            nst = end > begin ? (end - begin + ST - 1) / ST : 0;
            ncp_v = (nparts + p.cta_parts - 1) / p.cta_parts;
            pidx_v = p0 / p.cta_parts;
        }
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
        for (int m = 0; m < nm; ++m) {
            const int lm = glen[m], st = (lm - shared + 15) / 16;
            if (r < st) {
                mem = m;
                tok0 = shared + r * 16;
                endr = lm;
                break;
            }
            r -= st;
        }
    };
    auto table_of = [&](int mem) {
        return p.block_tables + (size_t)(GR ? s0 + max(mem, 0) : s) * p.max_blocks;
    };

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::BAR_OFF);
    int* sid = reinterpret_cast<int*>(smem + Gm::SID_OFF);  // [warp][slot][SID_INTS] records

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
        int tk0 = begin + (wsub + j * wpp) * ST, endr = end, mem = -1;
        if constexpr (GR) {
            if (j < cnt) stage_at(qbase + warp + j * NW, tk0, endr, mem);
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
                id = !GR && jbase == 0 && solo == spec_solo ? spec_ids[u] : tab[tok / B];
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
        int tok0 = begin + (wsub + j * wpp) * ST;
        int endr = end, mem = -1;
        if constexpr (GR) {
            tok0 = __shfl_sync(0xffffffffu, win_tok, j - win_base);
            endr = __shfl_sync(0xffffffffu, win_end, j - win_base);
            mem = __shfl_sync(0xffffffffu, win_mem, j - win_base);
        }
        if (lane == 0) {
            const int slot = j % NS;
            int* sd = sid + (warp * NS + slot) * Gm::SID_INTS;
#pragma unroll
            for (int u = 0; u < IDS; ++u) sd[u] = ids[u];
            if constexpr (GR) {
                sd[Gm::SID_TOK] = tok0;
                sd[Gm::SID_END] = endr;
                sd[Gm::SID_MEM] = mem;
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
    // Every launch is a programmatic dependent of the kernel before it (the
    // previous decode call, the step's copy-on-write copies, or the work
    // plan, which this CTA has already waited for).  Lengths, group bounds
    // and the first block ids are read while that kernel runs; the new
    // tokens, K/V and q only once it has completed and its writes are
    // visible.  Kernels of this library never write lengths or tables.
    if constexpr (GR) {
        if (cnt > 0) load_window(0);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (p.new_k != nullptr) {
        if constexpr (GR) {
            // member m's new token (always past the shared prefix) lies in
            // list stage nsh + (stages of members before m) + (L_m-1-shared)/16;
            // the warp of the CTA whose run holds that stage writes it
            int qb0 = nsh;
            for (int m = 0; m < nm; ++m) {
                const int lm = glen[m], qm = qb0 + (lm - 1 - shared) / 16;
                if (lm > shared && qm >= qbase && qm < qbase + nst && (qm - qbase) % NW == warp)
                    append(s0 + m, lm, table_of(m));
                qb0 += (lm - shared + 15) / 16;
            }
        } else if (L > 0 && begin <= L - 1 && L - 1 < end && ((L - 1 - begin) / ST) % wpp == wsub) {
            append(s, L, table);
        }
    }

    if (!GR && cnt > 0) load_window(0);
    for (int j = 0; j < NS && j < cnt; ++j) issue(j);

    // ---- Q^T as the B operand of Q K^T: column n (tile n / 8) = query head
    // g*G + hb + n (GR: member n / G, query head g*G + n % G); columns past
    // ncol are zero.
    uint32_t qb[NT][KSTEPS][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int n = 8 * t + gq;
        const int mn = GR ? n / G : 0, hn = GR ? n - mn * G : hb + n;
        const bool col = n < ncol;
        const T* qrow = static_cast<const T*>(p.q) +
                        ((size_t)(GR ? s0 + min(mn, nm - 1) : s) * p.num_heads + g * G +
                         (col ? hn : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            if (col) {
                qb[t][kk][0] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * tq);
                qb[t][kk][1] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * tq);
            } else {
                qb[t][kk][0] = qb[t][kk][1] = 0u;
            }
        }
    }

    // softmax state of columns 8t + 2tq (index 0) and 8t + 2tq + 1 (index 1)
    float mr[NT][2], lr_[NT][2];
    float acc[NT][MTILES][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        mr[t][0] = mr[t][1] = -INFINITY;
        lr_[t][0] = lr_[t][1] = 0.f;
#pragma unroll
        for (int i = 0; i < MTILES; ++i) acc[t][i][0] = acc[t][i][1] = acc[t][i][2] = acc[t][i][3] = 0.f;
    }
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
        const uint32_t kbase = smem_u32(ring + slot * Gm::STAGE_BYTES);
        const uint32_t vbase = kbase + Gm::KV_BYTES;
        const int tok0 = GR ? sinfo[Gm::SID_TOK] : begin + (wsub + j * wpp) * ST;
        const int endr = GR ? sinfo[Gm::SID_END] : end;
        // row r of the stage: token tok0 + r of block sinfo[r / B] (one block
        // when a box holds the whole stage)
        auto valid = [&](int r) {
            return tok0 + r < endr && sinfo[IDS > 1 ? r / B : 0] >= 0;
        };
        bool all_valid = tok0 + ST <= endr;
#pragma unroll
        for (int u = 0; u < IDS; ++u) all_valid = all_valid && sinfo[u] >= 0;

        // the stage's m16 token tiles, one after the other
#pragma unroll
        for (int hf = 0; hf < TPS; ++hf) {
            const int r0 = 16 * hf;
            // ---- S^T = K Q^T  (16 tokens x 8 heads per tile); with one tile, as
            // two independent accumulation chains (even and odd k-steps)
            float sc[NT][4], sd[NT][4];
    #pragma unroll
            for (int t = 0; t < NT; ++t)
                sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = sd[t][0] = sd[t][1] = sd[t][2] =
                    sd[t][3] = 0.f;
    #pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t a[4];
                ldsm_x4(kbase + stage_offset<Gm>(r0 + k_row, 2 * kk + k_chunk_add), a);
    #pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (NT == 1 && (kk & 1))
                        Mma<T>::run(sd[t], a, qb[t][kk][0], qb[t][kk][1]);
                    else
                        Mma<T>::run(sc[t], a, qb[t][kk][0], qb[t][kk][1]);
                }
            }
            // x[t][0..3]: (token gq, column 8t+2tq), (gq, +1), (gq+8, 8t+2tq), (gq+8, +1)
            float x[NT][4];
            const bool vg = all_valid || valid(r0 + gq), vg8 = all_valid || valid(r0 + gq + 8);
    #pragma unroll
            for (int t = 0; t < NT; ++t) {
    #pragma unroll
                for (int e = 0; e < 4; ++e) x[t][e] = (sc[t][e] + sd[t][e]) * sl;
                if (!vg) x[t][0] = x[t][1] = -INFINITY;
                if (!vg8) x[t][2] = x[t][3] = -INFINITY;
                if constexpr (GR) {
                    // a member's own tail: the other members' columns see nothing
                    const int mem = sinfo[Gm::SID_MEM];
                    if (mem >= 0) {
                        if ((8 * t + 2 * tq) / G != mem) x[t][0] = x[t][2] = -INFINITY;
                        if ((8 * t + 2 * tq + 1) / G != mem) x[t][1] = x[t][3] = -INFINITY;
                    }
                }
            }
            // ---- online softmax in base 2 against a reference max per head that
            // moves only when a score passes it by more than 8 (so p <= 2^8): most
            // stages need neither the max over the 8 row groups nor a rescale of O
            bool up = false;
    #pragma unroll
            for (int t = 0; t < NT; ++t)
                up = up || fmaxf(x[t][0], x[t][2]) > mr[t][0] + 8.f ||
                     fmaxf(x[t][1], x[t][3]) > mr[t][1] + 8.f;
            if (__any_sync(0xffffffffu, up)) {
    #pragma unroll
                for (int t = 0; t < NT; ++t) {
                    float mx0 = fmaxf(x[t][0], x[t][2]), mx1 = fmaxf(x[t][1], x[t][3]);
    #pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                    }
                    const float mn0 = fmaxf(mr[t][0], mx0), mn1 = fmaxf(mr[t][1], mx1);
                    // 0 while m is -inf (nothing accumulated yet), 1 if m stays
                    const float al0 = mn0 == -INFINITY ? 1.f : ex2(mr[t][0] - mn0);
                    const float al1 = mn1 == -INFINITY ? 1.f : ex2(mr[t][1] - mn1);
                    mr[t][0] = mn0;
                    mr[t][1] = mn1;
                    lr_[t][0] *= al0;
                    lr_[t][1] *= al1;
    #pragma unroll
                    for (int i = 0; i < MTILES; ++i) {
                        acc[t][i][0] *= al0;
                        acc[t][i][1] *= al1;
                        acc[t][i][2] *= al0;
                        acc[t][i][3] *= al1;
                    }
                }
            }
            // ---- P^T operand (tokens 2tq.. x head gq) via an in-register transpose
            uint32_t bh0[NT], bh1[NT], bl0[NT], bl1[NT];
    #pragma unroll
            for (int t = 0; t < NT; ++t) {
                const float ms0 = mr[t][0] == -INFINITY ? 0.f : mr[t][0];
                const float ms1 = mr[t][1] == -INFINITY ? 0.f : mr[t][1];
                const float p0 = ex2(x[t][0] - ms0), p1 = ex2(x[t][1] - ms1);
                const float p2 = ex2(x[t][2] - ms0), p3 = ex2(x[t][3] - ms1);
                lr_[t][0] += p0 + p2;
                lr_[t][1] += p1 + p3;
                uint32_t h01, l01, h23, l23;
                Mma<T>::split(p0, p1, h01, l01);
                Mma<T>::split(p2, p3, h23, l23);
                bh0[t] = movmatrix_trans(h01);
                bh1[t] = movmatrix_trans(h23);
                bl0[t] = movmatrix_trans(l01);
                bl1[t] = movmatrix_trans(l23);
            }

            bool v0 = true, v1 = true, v8 = true, v9 = true;
            if (!all_valid) {
                v0 = valid(r0 + 2 * tq);
                v1 = valid(r0 + 2 * tq + 1);
                v8 = valid(r0 + 2 * tq + 8);
                v9 = valid(r0 + 2 * tq + 9);
            }
            // ---- O^T += V^T P^T
    #pragma unroll
            for (int i = 0; i < MTILES; ++i) {
                uint32_t a[4];
                ldsm_x4_trans(vbase + stage_offset<Gm>(r0 + v_row, 2 * i + v_chunk_add), a);
                if (!all_valid) {
                    a[0] = mask_pair(a[0], v0, v1);
                    a[1] = mask_pair(a[1], v0, v1);
                    a[2] = mask_pair(a[2], v8, v9);
                    a[3] = mask_pair(a[3], v8, v9);
                }
    #pragma unroll
                for (int t = 0; t < NT; ++t) {
                    Mma<T>::run(acc[t][i], a, bh0[t], bh1[t]);
                    Mma<T>::run(acc[t][i], a, bl0[t], bl1[t]);
                }
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
    for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            lr_[t][0] += __shfl_xor_sync(0xffffffffu, lr_[t][0], o);
            lr_[t][1] += __shfl_xor_sync(0xffffffffu, lr_[t][1], o);
        }
    }

    const size_t hbase = (size_t)s * p.num_heads + (size_t)g * G + hb;
    // output / workspace row of column n: query head g*G + hb + n of sequence
    // s, or (GR) query head g*G + n % G of member n / G
    auto row_of = [&](int n) -> size_t {
        return GR ? (size_t)(s0 + n / G) * p.num_heads + g * G + n % G : hbase + n;
    };
    // this CTA's partial: index pidx of ncp per (sequence, KV head, head
    // slice) -- one per CTA, its warps' partitions (or its share of one
    // partition or piece) merged first -- or (GR) of the group's runs
    const int ncp = ncp_v, pidx = pidx_v;
    // ---- merge the warps (shared memory reused once every ring is drained):
    // their states cover one partition (each a share of its stages) or, with
    // one partition per warp, consecutive partitions of the same sequence
    __syncthreads();
    float* wm = reinterpret_cast<float*>(smem) + warp * NC * (D + 2);  // [NC][D], m[NC], l[NC]
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int n = 8 * t + 2 * tq;
        if (gq == 0) {
            wm[NC * D + n] = mr[t][0];
            wm[NC * D + n + 1] = mr[t][1];
            wm[NC * D + NC + n] = lr_[t][0];
            wm[NC * D + NC + n + 1] = lr_[t][1];
        }
#pragma unroll
        for (int i = 0; i < MTILES; ++i) {
            wm[n * D + 16 * i + gq] = acc[t][i][0];
            wm[(n + 1) * D + 16 * i + gq] = acc[t][i][1];
            wm[n * D + 16 * i + gq + 8] = acc[t][i][2];
            wm[(n + 1) * D + 16 * i + gq + 8] = acc[t][i][3];
        }
    }
    __syncthreads();
    const float* sm = reinterpret_cast<const float*>(smem);
    // four consecutive outputs of one head per thread
    const bool vec_out = (reinterpret_cast<uintptr_t>(p.out) & 15) == 0;
    for (int idx = threadIdx.x; idx < ncol * D / 4; idx += blockDim.x) {
        const int n = idx / (D / 4), d = (idx - n * (D / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm[w * NC * (D + 2) + NC * D + n]);
        float den = 0.f;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* ww = sm + w * NC * (D + 2);
            const float mw = ww[NC * D + n];
            const float wt = mw == -INFINITY ? 0.f : ex2(mw - M);
            den += wt * ww[NC * D + NC + n];
            const float4 o = *reinterpret_cast<const float4*>(ww + n * D + d);
            num.x += wt * o.x;
            num.y += wt * o.y;
            num.z += wt * o.z;
            num.w += wt * o.w;
        }
        if (ncp <= 1) {
            const bool pos = den > 0.f;
            store_out4(p.out, row_of(n) * D + d,
                       make_float4(pos ? num.x / den : 0.f, pos ? num.y / den : 0.f,
                                   pos ? num.z / den : 0.f, pos ? num.w / den : 0.f),
                       p.out_dtype, vec_out);
        } else {
            const size_t slot = row_of(n) * p.max_partitions + pidx;
            *reinterpret_cast<float4*>(p.ws_o + slot * D + d) = num;
            if (d == 0) p.ws_ml[slot] = make_float2(M, den);
        }
    }
    if (ncp <= 1) return;

    // ---- split: the CTA that writes the last of the ncp partials of (s, g,
    // head slice), or (GR) of (group, g), merges them by log-sum-exp:
    // M = max_i m_i, w_i = 2^(m_i - M), out = sum_i w_i O_i / sum_i w_i l_i.
    __shared__ int is_last;
    __syncthreads();  // this CTA's partition results are written ...
    if (threadIdx.x == 0) {
        // release: this CTA's partition results (ordered before this thread by
        // the barrier) are visible before the count goes up; acquire for the
        // CTA that completes the count: it sees every other partition's results
        unsigned prev;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                     : "=r"(prev)
                     : "l"(&p.done[sg]), "r"(1u)
                     : "memory");
        is_last = prev == (unsigned)(ncp - 1);
    }
    __syncthreads();
    if (!is_last) return;
    constexpr int NTH = NW * 32;
    float* wts = reinterpret_cast<float*>(smem) + NW * NC * (D + 2);  // [ncol][ncp] weights
    float* hinv = wts + Gm::WCACHE;                                    // [NC]
    float* hmax = hinv + NC;                                           // [NC]
    float4* red = reinterpret_cast<float4*>(hmax + NC);                // [NTH] partial sums
    const bool cached = ncol * ncp <= Gm::WCACHE;
    for (int n = warp; n < ncol; n += NW) {
        const size_t base = row_of(n) * p.max_partitions;
        // the (max, sum) pairs of the first 64 partitions are read once and
        // kept in registers for both passes; any further ones are re-read
        float2 ml[2];
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = lane + 32 * r;
            ml[r] = i < ncp ? __ldcg(&p.ws_ml[base + i]) : make_float2(-INFINITY, 0.f);
            M = fmaxf(M, ml[r].x);
        }
        for (int i = lane + 64; i < ncp; i += 32) M = fmaxf(M, __ldcg(&p.ws_ml[base + i]).x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float den = 0.f;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = lane + 32 * r;
            if (i < ncp) {
                const float w = ml[r].x == -INFINITY ? 0.f : ex2(ml[r].x - M);
                if (cached) wts[n * ncp + i] = w;
                den += w * ml[r].y;
            }
        }
        for (int i = lane + 64; i < ncp; i += 32) {
            const float2 mli = __ldcg(&p.ws_ml[base + i]);
            const float w = mli.x == -INFINITY ? 0.f : ex2(mli.x - M);
            if (cached) wts[n * ncp + i] = w;
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
    // Outputs in float4 units; when the slice has fewer of them than
    // threads, K threads share one output, each summing every K-th partition.
    const int O4 = ncol * D / 4;
    const int K = O4 >= NTH ? 1 : NTH / O4;
    for (int o0 = 0; o0 < O4; o0 += NTH) {
        const int t = threadIdx.x;
        const int o = o0 + (K == 1 ? t : t % O4), k = K == 1 ? 0 : t / O4;
        float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
        const bool active = o < O4 && k < K;
        if (active) {
            const int n = o / (D / 4), d4 = o - n * (D / 4);
            const size_t base = row_of(n) * p.max_partitions;
            const float4* src = reinterpret_cast<const float4*>(p.ws_o + base * D) + d4;
#pragma unroll 16
            for (int i = k; i < ncp; i += K) {
                float w;
                if (cached) {
                    w = wts[n * ncp + i];
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
            const size_t at = row_of(n) * D + d;
            store_out(p.out, at + 0, acc4.x * inv, p.out_dtype);
            store_out(p.out, at + 1, acc4.y * inv, p.out_dtype);
            store_out(p.out, at + 2, acc4.z * inv, p.out_dtype);
            store_out(p.out, at + 3, acc4.w * inv, p.out_dtype);
        }
    }
}

template <typename T, int D, int B, bool GR, int NT, int NS = 2>
cudaError_t launch_tc(const DecodeParams& p, const void* kmap, const void* vmap, long long grid,
                      cudaStream_t stream)
{
    // 4 warps x 2-stage rings of 8 KB stages (16 tokens at D = 128, 32 at
    // D = 64; beam groups at D = 64 keep 16): 64 KB per CTA, three CTAs per
    // SM, up to 192 KB of tile loads in flight per SM; or (NS = 3) 3-stage
    // rings, 96 KB per CTA, two CTAs per SM: the same loads per SM, but each
    // warp keeps two stages in flight while it works on a third
    constexpr int NW = kDecodeTcWarps;
    constexpr int TPS = decode_stage_tokens(D, GR) / 16;
    using Gm = Geometry<D, B, NW, NS, NT, TPS>;
    static_assert(Gm::ROWS == decode_box_rows(D, B, GR), "tensor map box = stage box");
    auto kern = decode_tc_kernel<T, D, B, NW, NS, GR, NT, TPS>;
    // set on every launch: the attribute belongs to the current device's copy
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // a programmatic dependent launch (after a work plan, a copy-on-write
    // copy, the previous decode call or any kernel): the CTAs are resident
    // and have read what no kernel of this library writes while the kernel
    // before them runs, and go on the moment it completes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = Gm::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, *static_cast<const CUtensorMap*>(kmap),
                              *static_cast<const CUtensorMap*>(vmap));
}

// NT: n8 column tiles of query heads per CTA (1: up to 8 columns, 2: up to 16);
// NS: stages per warp ring
template <typename T, bool GR, int NT, int NS = 2>
cudaError_t launch_tc_dtype(const DecodeParams& p, const void* kmap, const void* vmap,
                            long long grid, cudaStream_t stream)
{
    if (p.head_dim == 128) {
        if (p.block_size == 16) return launch_tc<T, 128, 16, GR, NT, NS>(p, kmap, vmap, grid, stream);
        if (p.block_size == 32) return launch_tc<T, 128, 32, GR, NT, NS>(p, kmap, vmap, grid, stream);
        return launch_tc<T, 128, 8, GR, NT, NS>(p, kmap, vmap, grid, stream);
    }
    if (p.block_size == 16) return launch_tc<T, 64, 16, GR, NT, NS>(p, kmap, vmap, grid, stream);
    if (p.block_size == 32) return launch_tc<T, 64, 32, GR, NT, NS>(p, kmap, vmap, grid, stream);
    return launch_tc<T, 64, 8, GR, NT, NS>(p, kmap, vmap, grid, stream);
}

}  // namespace
