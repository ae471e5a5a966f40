// Paged decode attention for wide query-head groups on the 5th-generation
// tensor cores (tcgen05 + TMEM), for sm_103a: 16-bit KV cache, head_dim 128,
// a multiple of 32 query heads per KV head, in items of 64 heads when the
// group is a multiple of 64, else of 32.
//
// What it computes: the decode attention of every decode kernel here -- for
// sequence s and query head h, the softmax over the context's tokens of
// scale * q_h . k_t, applied to the v_t -- with the tokens reached through
// the block table (aiplusplus PagedAttention page, "key techniques" 1 and 3;
// auturnal guide section 1 for query heads that share a KV head).
//
// Why a second kernel: with G query heads on one KV head every K and V row
// feeds G dot products.  At G >= 32 the mma.sync kernel cuts the group into
// head slices, and each slice reads the K/V tiles again and repeats their
// fragment loads.  Here a tile's tokens are the MMA's M and the group's heads
// its N, so one K/V tile serves an item's NH = 32 or 64 heads and nothing is
// padded:
//   S^T(j) = K(j) Q^T         M = 128 tokens, N = NH heads,  K = head_dim
//   O^T   += V(j)^T P(j)^T    M = head_dim,   N = 2 NH,      K = 128 tokens
// both accumulated in fp32 in tensor memory.  P reaches the tensor cores as
// a 16-bit high part and its remainder (~16 bits of P, as in the prefill
// kernel), side by side in the N columns of one MMA: O^T is kept as a high
// and a low accumulator per half of 32 heads, added at the end.
//
// Work items are (sequence, KV head, slice of NH query heads).  One
// persistent CTA a SM takes them from the work plan's longest-first list
// through an atomic counter, or without a plan items b, b + grid, ...
// (With NH = 64 the counts below change: softmax warps 0-7, the MMA warp 8,
// load warps 9-11, one Q buffer and a ring of four slots.)
//  * warps 5-7 (loads): warp 5 takes an item's record and loads its 32 rows
//    of Q (plain loads, so q may be pinned host memory) into one of two Q
//    buffers; then all three load the item's K and V tiles of 128 tokens by
//    TMA (16-row boxes of the paged cache, 128-byte swizzle; K as [column
//    half][token][128 B], two copies a box; V as [16-token group][column
//    half][16 rows][128 B], one copy a box, the layout P V reads a 16-token
//    step from), each warp about a third of a tile's boxes, into a ring
//    of five 32 KB slots, in the order the MMAs use them: K(0) K(1) K(2) V(0)
//    K(3) V(1) ... V(n-2) V(n-1) (S^T runs two tiles ahead of P V).  A slot's
//    barrier takes one arrival (with its bytes) from each load warp: a single
//    warp issuing every copy of a tile holds the SM well below the HBM rate.
//    Lanes read their boxes' block-table entries two tiles ahead and record
//    bad ones.  While an item's tiles are issued, warp 5 already claims the
//    next record and reads the entries of its first two tiles, one stage a
//    step, so that the item boundary waits on no global round trip but the
//    Q rows'.  Eight warps, two a scheduler, leave the softmax its registers
//    (twelve, three a scheduler, with NH = 64: 168 registers a thread).
//  * warp 4 (MMA issue): S^T(j + 2) into S buffer j & 1 as soon as the
//    softmax has read S^T(j) out of it (early in its tile), then, once the
//    softmax has posted P(j) in shared memory, O^T += V(j)^T P(j)^T.
//  * warps 0-3 (softmax; with NH = 64 warps 4-7 take heads 32-63 of the same
//    tokens): thread t owns token t of each tile (row t of S^T) and row
//    d = t of O^T, for its 32 heads.  Every head's running max is shared by
//    the CTA (in shared memory) and moves only when a score passes it by
//    more than 8 (a factor 2^8): a barrier-reduction vote (per half of the
//    heads, a named barrier each) finds out, then the tile's scores, put through
//    a scratch in the tile's P buffer, give its maxima per head, and O^T and
//    the partial sums are rescaled.  Each thread sums P over its own tokens
//    per head; those sums are reduced across the 128 threads through the
//    same scratch once per item.  These rarely run paths are short loops:
//    fully unrolled, their cold code cost thousands of cycles an item.
// Tensor memory: S buffers at columns [0, NH) and [NH, 2 NH), O^T at
// [2 NH, 4 NH) (per half of 32 heads, high parts, then remainders).
// Every wait is bounded: one that gives up sets the TIMEOUT status bit (which
// ends the waits of every other CTA too), and before the CTA frees its
// tensor memory it waits (bounded) for its own copies and MMAs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <algorithm>

#include "pkv.h"
#include "pkv_kernels.h"
#include "tc_common.cuh"
#include "tc05_common.cuh"

namespace {

using namespace pkv_tc;
using namespace pkv_tc05;

constexpr int kD = 128;                // head_dim
constexpr int kTok = 128;              // tokens per K/V tile
constexpr int kRing = 16;              // bad-box masks kept per tile index
constexpr int kLoadWarps = 3;
constexpr unsigned kFull = 0xffffffffu;

// NH query heads an item (the S MMA's N; 32 or 64), in NH / 32 halves of 32
// heads, each owned by four softmax warps (one a TMEM lane quarter).
template <int B, int NH>
struct W5 {
    static constexpr int HALVES = NH / 32;
    static constexpr int SW = 4 * HALVES;            // softmax warps
    static constexpr int MMA_WARP = SW, LOAD_WARP0 = SW + 1;
    static constexpr int THREADS = 32 * (SW + 1 + kLoadWarps);
    static constexpr int QB = NH == 32 ? 2 : 1;      // Q buffers
    static constexpr int SLOTS = NH == 32 ? 5 : 4;   // K/V ring (one K or V tile each)
    static constexpr uint32_t TMEM_COLS = 4 * NH;    // S^T x 2, then O^T
    static constexpr uint32_t COL_O = 2 * NH;        // O^T: per half, high parts, remainders
    static constexpr int ROWS = B < 16 ? B : 16;     // rows per TMA box
    static constexpr int IDS = 16 / ROWS;            // boxes per 16-token group
    static constexpr int SUBS = (kTok / 16) * IDS;   // boxes per tile
    static constexpr int HALF_Q = NH * 128;          // Q: [half of D][head][128 B]
    static constexpr int Q_BYTES = 2 * HALF_Q;
    static constexpr int P_ATOM = kTok * 128;        // a head half's P^T: [token][high | low]
    static constexpr int P_BYTES = HALVES * P_ATOM;
    // K: [8-token group][half][token][128 B], a group's halves side by side
    // (2048 bytes a group); V: see V_GROUP
    static constexpr int HALF_KV = kTok * 128;
    static constexpr int SLOT_BYTES = 2 * HALF_KV;
    // V: per 16-token group (4 KB), both halves of each box from one copy:
    // [half][16 rows][128 B], or at block size 8 [8-row box][half][8 rows][128 B]
    static constexpr int V_GROUP = 4096;
    static constexpr int V_LBO = ROWS == 16 ? 2048 : 1024;  // between the halves
    static constexpr int V_SBO = ROWS == 16 ? 1024 : 2048;  // between 8-row groups
    static constexpr int P_OFF = QB * Q_BYTES;
    static constexpr int SLOT_OFF = P_OFF + 2 * P_BYTES;
    // full, empty per slot; q_full, q_empty per Q buffer; s_full, s_free,
    // p_full, o_done (two each); drain
    static constexpr int BARS = 2 * SLOTS + 2 * QB + 9;
    static constexpr int BAR_OFF = SLOT_OFF + SLOTS * SLOT_BYTES;
    static constexpr int REC_OFF = (BAR_OFF + BARS * 8 + 15) / 16 * 16;  // int4 [QB]
    static constexpr int RIDS_OFF = REC_OFF + QB * 16;    // int [QB][tiles 0, 1][32]
    static constexpr int RED_OFF = RIDS_OFF + QB * 2 * 32 * 4;  // float [half][4 warps][32]
    static constexpr int MROW_OFF = RED_OFF + HALVES * 4 * 32 * 4;  // float [half][32] max
    static constexpr int ALPHA_OFF = MROW_OFF + HALVES * 32 * 4;    // float [half][32] rescale
    static constexpr int INV_OFF = ALPHA_OFF + HALVES * 32 * 4;     // float [half][32] 1 / sum
    static constexpr int KBAD_OFF = INV_OFF + HALVES * 32 * 4;      // uint32 [kRing][load warp]
    static constexpr int TSLOT_OFF = KBAD_OFF + kRing * kLoadWarps * 4;
    static constexpr int SMEM_BYTES = 1024 + TSLOT_OFF + 16;
    static_assert(NH == 32 || NH == 64, "32 or 64 heads an item");
    static_assert(SUBS <= 32 && SUBS >= kLoadWarps, "boxes per load warp");
    static_assert(HALF_Q % 1024 == 0 && P_ATOM % 1024 == 0 && HALF_KV % 1024 == 0, "atoms");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(REC_OFF % 16 == 0 && MROW_OFF % 16 == 0 && ALPHA_OFF % 16 == 0 &&
                      INV_OFF % 16 == 0, "vector access");
};

// Row t (0..127) of a [128][32] fp32 scratch at `buf` (16 KB, 1024-byte
// aligned): v, in 16-byte chunks XOR-swizzled by t & 7 (conflict-free both
// ways below).
__device__ __forceinline__ void put_rows(uint8_t* buf, int t, const float (&v)[32])
{
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(buf + swz(t, c)) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// Thread t: the maximum (or the sum) of column t & 31 over rows 32 (t >> 5)
// .. + 31 of the scratch; a short loop, so that this code (run once per item,
// or when a max moves) stays small.
template <bool kMax>
__device__ __forceinline__ float column_op(const uint8_t* buf, int t)
{
    const int h = t & 31, r0 = (t >> 5) * 32;
    float acc = kMax ? -INFINITY : 0.f;
#pragma unroll 4
    for (int r = r0; r < r0 + 32; ++r) {
        const float v = *reinterpret_cast<const float*>(buf + swz(r, h >> 2) + (h & 3) * 4);
        acc = kMax ? fmaxf(acc, v) : acc + v;
    }
    return acc;
}

// out[at + h * head_dim] = o[h] for the 32 heads, in the output dtype.
__device__ __forceinline__ void store_column(void* out, size_t at, const float (&o)[32],
                                             int out_dtype)
{
    if (out_dtype == PKV_F32) {
        float* d = static_cast<float*>(out) + at;
#pragma unroll
        for (int h = 0; h < 32; ++h) d[(size_t)h * 128] = o[h];
    } else if (out_dtype == PKV_F16) {
        __half* d = static_cast<__half*>(out) + at;
#pragma unroll
        for (int h = 0; h < 32; ++h) d[(size_t)h * 128] = __float2half_rn(o[h]);
    } else {
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(out) + at;
#pragma unroll
        for (int h = 0; h < 32; ++h) d[(size_t)h * 128] = __float2bfloat16_rn(o[h]);
    }
}

// Named barrier 1 + hh over the four softmax warps of head half hh (128
// threads), plain and with an OR or AND vote.
__device__ __forceinline__ void softmax_sync(int id)
{
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}
__device__ __forceinline__ bool softmax_any(int id, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %2, 0;\n\t"
        "bar.red.or.pred q, %1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool softmax_all(int id, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %2, 0;\n\t"
        "bar.red.and.pred q, %1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// Step i (0 <= i < 2n) of an item of n tiles in ring order: K(0), K(1),
// then K(m + 2), V(m) for m = 0 .. n - 3, then V(n - 2), V(n - 1) (K(0),
// V(0) when n = 1).  kv: 0 for K, 1 for V; j: the tile.
__device__ __forceinline__ void ring_step(int i, int n, int& kv, int& j)
{
    if (n == 1) {
        kv = i;
        j = 0;
    } else if (i < 2) {
        kv = 0;
        j = i;
    } else if (i >= 2 * n - 2) {
        kv = 1;
        j = i - n;
    } else {
        const int m = (i - 2) >> 1;
        kv = (i - 2) & 1;
        j = kv ? m : m + 2;
    }
}

template <typename T, int B, int NH>
__global__ void __launch_bounds__(W5<B, NH>::THREADS, 1)
decode_tc05_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap)
{
    using W = W5<B, NH>;
    constexpr int IDS = W::IDS;
    constexpr int SW = W::SW, QB = W::QB, SLOTS = W::SLOTS;
    constexpr uint32_t COL_O = W::COL_O;
    const int HS = p.head_slices;
    const int G = p.num_heads / p.num_kv_heads;
    const int per_seq = p.num_kv_heads * HS;

    // dependents may launch now (they wait for this grid before touching
    // what it writes)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + W::BAR_OFF);
    uint64_t* empty = full + SLOTS;
    uint64_t* q_full = empty + SLOTS;   // [Q buffer], the lead load warp
    uint64_t* q_empty = q_full + QB;    // [Q buffer], MMA commit + the other warps
    uint64_t* s_full = q_empty + QB;    // [S buffer], MMA commit
    uint64_t* s_free = s_full + 2;      // [S buffer], one per softmax warp
    uint64_t* p_full = s_free + 2;      // [P buffer], one per softmax warp
    uint64_t* o_done = p_full + 2;      // [P buffer], MMA commit after P V
    uint64_t* drain = o_done + 2;
    int4* rec = reinterpret_cast<int4*>(smem + W::REC_OFF);
    int* rec_ids = reinterpret_cast<int*>(smem + W::RIDS_OFF);  // entries of tiles 0 and 1
    uint32_t* kbad = reinterpret_cast<uint32_t*>(smem + W::KBAD_OFF);
    // bad boxes of tile kt: one mask per load warp, each at its boxes' bits
    auto bad_boxes = [&](int kt) {
        const uint32_t* e = kbad + (kt % kRing) * kLoadWarps;
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < kLoadWarps; ++w) m |= e[w];
        return m;
    };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + W::TSLOT_OFF);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < W::BARS; ++i) {
            uint64_t* b = &full[i];
            uint32_t count = 1;
            if (b >= full && b < full + SLOTS) count = kLoadWarps;
            // the MMA warp's commit, the softmax warps, the other load warps
            if (b >= q_empty && b < q_empty + QB) count = 1 + SW + (kLoadWarps - 1);
            if (b == &p_full[0] || b == &p_full[1] || b == &s_free[0] || b == &s_free[1])
                count = SW;
            mbar_init(smem_u32(b), count);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tslot)),
                     "r"(W::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tbase = *tslot;
    // the plan, K/V, q and out are written (or read) by the kernels before
    asm volatile("griddepcontrol.wait;" ::: "memory");

    bool ok = true;
    auto wait = [&](uint64_t* bar, int parity) {
        if (!ok) return;
        if (!mbar_wait_bounded(smem_u32(bar), (uint32_t)parity, p.status)) {
            ok = false;
            atomicOr(p.status, PKV_STATUS_TIMEOUT);
        }
    };
    // lane 0 waits, the warp follows with its result
    auto warp_wait = [&](uint64_t* bar, int parity) {
        if (lane == 0) wait(bar, parity);
        ok = __shfl_sync(kFull, ok, 0);
        __syncwarp();
    };
    // ring position t: counted over all of this CTA's K and V tiles, in ring
    // order (ring_step)
    auto slot_of = [](int t) { return t % SLOTS; };
    auto phase_of = [](int t) { return (t / SLOTS) & 1; };

    if (warp >= W::LOAD_WARP0) {
        // ------------------------------------------------------------ loads
        const int lw = warp - W::LOAD_WARP0;
        const bool lead = lw == 0;  // takes the records and loads Q
        int t = 0, kt0 = 0, n = 0;
        int next_static = blockIdx.x;
        // this warp's boxes of a tile: [bx0, bx1), one a lane
        const int bx0 = lw * W::SUBS / kLoadWarps, bx1 = (lw + 1) * W::SUBS / kLoadWarps;
        const int bx = bx0 + lane;
        const bool mine = bx < bx1;
        // the lead warp: the next item, prefetched one stage a call of
        // advance(): 0 nothing yet, 1 index claimed, 2 record read, 3 the
        // entries of tiles 0 and 1 loaded (into registers)
        int stage = 0, nidx = 0;
        int4 nrec = make_int4(-1, 0, 0, 0);
        int nid[2] = {-1, -1};
        auto advance = [&]() {
            if (stage == 0) {
                if (lane == 0) {
                    if (p.items != nullptr) {
                        nidx = atomicAdd(p.item_next, 1);
                    } else {
                        nidx = next_static;
                        next_static += gridDim.x;
                    }
                }
                stage = 1;
            } else if (stage == 1) {
                // (sequence, length, KV head x slice, tiles), or sequence -1
                // when there is none; a bad record is flagged and skipped
                int4 r = make_int4(-1, 0, 0, 0);
                bool again = false;
                if (lane == 0) {
                    const bool have = p.items != nullptr
                                          ? nidx < *p.item_count
                                          : (long long)nidx < (long long)p.num_seqs * per_seq;
                    if (have) {
                        int s, z, L;
                        if (p.items != nullptr) {
                            const int4 it = p.items[nidx];
                            s = it.x;
                            L = it.y;
                            z = it.z;
                        } else {
                            s = nidx / per_seq;
                            z = nidx - s * per_seq;
                            L = p.context_lens[s];
                        }
                        if (s < 0 || s >= p.num_seqs || z < 0 || z >= per_seq) {
                            atomicOr(p.status, PKV_STATUS_BAD_LEN);
                            again = true;
                        } else {
                            if (L < 0 || (int64_t)L > (int64_t)p.max_blocks * B) {
                                atomicOr(p.status, PKV_STATUS_BAD_LEN);
                                L = 0;
                            }
                            r = make_int4(s, L, z, (L + kTok - 1) / kTok);
                        }
                    }
                }
                nrec.x = __shfl_sync(kFull, r.x, 0);
                nrec.y = __shfl_sync(kFull, r.y, 0);
                nrec.z = __shfl_sync(kFull, r.z, 0);
                nrec.w = __shfl_sync(kFull, r.w, 0);
                stage = __shfl_sync(kFull, again ? 0 : 2, 0);
            } else if (stage == 2) {
                if (nrec.x >= 0) {
                    // lane l < SUBS: box l of tiles 0 and 1
                    const int32_t* table = p.block_tables + (size_t)nrec.x * p.max_blocks;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int tok = j * kTok + lane * W::ROWS;
                        nid[j] = (lane < W::SUBS && j < nrec.w && tok < nrec.y) ? table[tok / B]
                                                                               : -1;
                    }
                }
                stage = 3;
            }
        };
        while (ok) {
            const int b = n % QB;
            int4 r;
            if (lead) {
                while (stage < 3) advance();
                r = nrec;
                // Q buffer b is free once the MMAs of item n - QB have read it
                // and every other warp has read its record
                if (n >= QB) warp_wait(&q_empty[b], ((n / QB) - 1) & 1);
                if (!ok) break;
                if (r.x >= 0) {
                    // lane l: query heads l, l + 32, ... of the item, 16-byte
                    // chunks into the K-major, 128-byte-swizzled [half of D]
                    // [head][128 B] layout
                    const int g = r.z / HS, hs = r.z - (r.z / HS) * HS;
                    uint8_t* qb = smem + b * W::Q_BYTES;
#pragma unroll
                    for (int hh = 0; hh < W::HALVES; ++hh) {
                        const int head = hh * 32 + lane;
                        const T* src = static_cast<const T*>(p.q) +
                                       ((size_t)r.x * p.num_heads + g * G + hs * NH + head) * kD;
                        uint4 v[kD / 8];
#pragma unroll
                        for (int c = 0; c < kD / 8; ++c)
                            v[c] = *reinterpret_cast<const uint4*>(src + c * 8);
#pragma unroll
                        for (int c = 0; c < kD / 8; ++c)
                            *reinterpret_cast<uint4*>(qb + (c >> 3) * W::HALF_Q +
                                                      swz(head, c & 7)) = v[c];
                    }
                    fence_proxy_async();
                }
                rec_ids[(b * 2 + 0) * 32 + lane] = nid[0];
                rec_ids[(b * 2 + 1) * 32 + lane] = nid[1];
                __syncwarp();
                if (lane == 0) {
                    rec[b] = r;
                    mbar_arrive(smem_u32(&q_full[b]));
                }
                stage = 0;
            } else {
                warp_wait(&q_full[b], (n / QB) & 1);
                if (!ok) break;
                r = rec[b];
            }
            // this warp's entries of tiles 0 and 1, then (others) the record is released
            int id_n1 = mine ? rec_ids[(b * 2 + 0) * 32 + bx] : -1;
            int id_n2 = mine ? rec_ids[(b * 2 + 1) * 32 + bx] : -1;
            __syncwarp();
            if (!lead && lane == 0) mbar_arrive(smem_u32(&q_empty[b]));
            ++n;
            const int s = r.x, L = r.y, nkt = r.w;
            if (s < 0) break;
            const int g = r.z / HS;
            const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
            // block-table entry of this lane's box in tile j (-1: past the
            // context or not this warp's), read two tiles ahead
            auto entry = [&](int j) {
                const int tok = j * kTok + bx * W::ROWS;
                return (mine && j < nkt && tok < L) ? table[tok / B] : -1;
            };
            // checked entries of tiles j mod 4: K(j + 1) and K(j + 2) come
            // between K(j) and V(j)
            int id_q0 = -1, id_q1 = -1, id_q2 = -1, id_q3 = -1;
            for (int i = 0; i < 2 * nkt; ++i, ++t) {
                int kv, j;
                ring_step(i, nkt, kv, j);
                const int tok = j * kTok + bx * W::ROWS;
                const int sl = slot_of(t);
                if (t >= SLOTS) warp_wait(&empty[sl], ((t / SLOTS) - 1) & 1);
                if (!ok) break;
                int id;
                if (kv == 0) {
                    // K(j) comes before V(j): check the entry and keep it for V
                    id = id_n1;
                    const bool bad = mine && tok < L && (id < 0 || id >= p.num_blocks);
                    if (bad) id = -1;
                    id_n1 = id_n2;
                    id_n2 = entry(j + 2);
                    const int q = j & 3;
                    id_q0 = q == 0 ? id : id_q0;
                    id_q1 = q == 1 ? id : id_q1;
                    id_q2 = q == 2 ? id : id_q2;
                    id_q3 = q == 3 ? id : id_q3;
                    const unsigned bads = __ballot_sync(kFull, bad) << bx0;
                    if (lane == 0) {
                        kbad[((kt0 + j) % kRing) * kLoadWarps + lw] = bads;
                        if (bads) atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
                    }
                } else {
                    const int q = j & 3;
                    id = q == 0 ? id_q0 : q == 1 ? id_q1 : q == 2 ? id_q2 : id_q3;
                }
                // a V box past the context or with a bad entry is loaded from
                // rows before the first (TMA fills them with zeros): P is 0
                // there, and 0 * NaN must not reach O
                const bool zero_box = kv == 1 && mine && id < 0;
                const unsigned have = __ballot_sync(kFull, id >= 0 || zero_box);
                const uint32_t bar = smem_u32(&full[sl]);
                if (lane == 0) mbar_arrive_expect_tx(bar, __popc(have) * 2 * W::ROWS * 128);
                __syncwarp();
                if (id >= 0 || zero_box) {
                    const int row = zero_box ? -W::ROWS
                                             : (id * p.num_kv_heads + g) * B + (IDS > 1 ? 0 : tok % B);
                    const uint32_t slot = smem_u32(smem + W::SLOT_OFF + sl * W::SLOT_BYTES);
                    if (kv == 0) {
                        // one copy brings the box's rows of both column halves
                        const uint32_t dst = slot + bx * W::ROWS * 256;
                        tma_load_4d(dst, &kmap, 0, 0, 0, row / 8, bar);
                    } else {
                        // box bx = 16-token group bx / IDS, 8-row box bx % IDS
                        const uint32_t dst = slot + (bx / IDS) * W::V_GROUP + (bx % IDS) * 2048;
                        tma_load_3d(dst, &vmap, 0, row, 0, bar);
                    }
                }
                if (lead && stage < 3) advance();
            }
            kt0 += nkt;
        }
        // the ring's last fills must have landed before the CTA exits
        if (lane == 0)
            for (int f = max(0, t - SLOTS); f < t; ++f)
                mbar_drain_wait(smem_u32(&full[slot_of(f)]), phase_of(f));
        __syncwarp();
    } else if (warp == W::MMA_WARP) {
        // ------------------------------------------------------- MMA issue
        const uint32_t id_s = instr_desc<T>(kTok, NH, 0, 0);      // K and Q K-major
        const uint32_t id_o = instr_desc<T>(kD, 2 * NH, 1, 1);    // V and P MN-major
        const uint32_t tm = __shfl_sync(kFull, tbase, 0);         // warp-uniform
        const uint32_t slot_base = smem_u32(smem + W::SLOT_OFF);
        // descriptors of Q buffer 0, P buffer 0 and ring slot 0; every
        // operand is one of these moved by a constant or per-buffer offset
        const uint64_t q_desc = smem_desc(smem_u32(smem), 16, 1024);
        const uint64_t k_desc = smem_desc(slot_base, 16, 2048);
        const uint64_t v_desc = smem_desc(slot_base, W::V_LBO, W::V_SBO);
        // P^T: MN-major, one 128-byte atom (64 columns) per head half
        const uint64_t p_desc = smem_desc(smem_u32(smem + W::P_OFF), W::P_ATOM, 1024);
        auto commit = [&](uint64_t* bar) {
            if (elect_one()) umma_commit(smem_u32(bar));
            __syncwarp();
        };
        // the next K or V in ring order has landed: its slot
        int tc = 0;
        auto take = [&]() {
            const int t = tc++;
            warp_wait(&full[slot_of(t)], phase_of(t));
            return slot_of(t);
        };
        // V(kt) in slot sl: the rows past the context inside its last loaded
        // box are cache memory past the sequence's end; zeroed (their P is 0,
        // and 0 * NaN must not reach O).  Later boxes and bad ones came in as
        // zeros.
        auto v_fix = [&](int sl, int tok0, int L) {
            const int k0 = L - tok0;
            if (ok && k0 < kTok && k0 % W::ROWS != 0) {
                const int k1 = (k0 / W::ROWS + 1) * W::ROWS;
                uint8_t* vt = smem + W::SLOT_OFF + sl * W::SLOT_BYTES;
                for (int i = lane; i < (k1 - k0) * 16; i += 32) {
                    const int k = k0 + (i >> 4), hf = (i >> 3) & 1, c = i & 7;
                    const int r = k & 15;
                    const int at = (k >> 4) * W::V_GROUP +
                                   (W::ROWS == 16 ? hf * 2048 + r * 128
                                                  : (r >> 3) * 2048 + hf * 1024 + (r & 7) * 128);
                    *reinterpret_cast<uint4*>(vt + at + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();
            }
            __syncwarp();
        };
        // S^T(kt) = K(kt) Q^T into S buffer kt & 1, from Q buffer b and slot sl
        auto issue_s = [&](int kt, int b, int sl) {
            const uint64_t qd = desc_add(q_desc, b * W::Q_BYTES);
            const uint64_t kd = desc_add(k_desc, sl * W::SLOT_BYTES);
            const uint32_t d = tm + (kt & 1) * NH;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma(d, desc_add(kd, (kk >> 2) * 1024 + (kk & 3) * 32),
                         desc_add(qd, (kk >> 2) * W::HALF_Q + (kk & 3) * 32), id_s, kk > 0);
                umma_commit(smem_u32(&s_full[kt & 1]));
            }
            __syncwarp();
        };
        // O^T (+)= V(kt)^T P(kt)^T for the high parts and the remainders of P
        // of every head at once (N = 2 NH), 16 tokens a step
        auto issue_pv = [&](int kt, int sl, bool first) {
            const uint64_t vd = desc_add(v_desc, sl * W::SLOT_BYTES);
            const uint64_t pd = desc_add(p_desc, (kt & 1) * W::P_BYTES);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTok / 16; ++kk)
                    umma(tm + COL_O, desc_add(vd, kk * W::V_GROUP), desc_add(pd, kk * 2048), id_o,
                         !first || kk > 0);
                umma_commit(smem_u32(&o_done[kt & 1]));
            }
            __syncwarp();
        };
        int kt0 = 0, n = 0;
        while (ok) {
            const int b = n % QB;
            warp_wait(&q_full[b], (n / QB) & 1);
            if (!ok) break;
            const int4 r = rec[b];
            ++n;
            if (r.x < 0) break;
            const int L = r.y, nkt = r.w;
            // S^T(kt) goes into S buffer kt & 1 once the softmax has read
            // S^T(kt - 2) out of it
            auto s_step = [&](int kt) {
                if (kt >= 2) warp_wait(&s_free[kt & 1], ((kt - 2) >> 1) & 1);
                const int sl = take();
                if (!ok) return;
                tmem_fence_after();
                issue_s(kt, b, sl);
                commit(&empty[sl]);
            };
            for (int j = 0; j < nkt && j < 2 && ok; ++j) s_step(kt0 + j);
            for (int j = 0; j < nkt && ok; ++j) {
                const int kt = kt0 + j;
                if (j + 2 < nkt) {
                    s_step(kt + 2);
                    if (!ok) break;
                }
                // P(kt) posted: the softmax has rescaled O^T too
                warp_wait(&p_full[kt & 1], (kt >> 1) & 1);
                if (!ok) break;
                const int sv = take();
                if (!ok) break;
                v_fix(sv, j * kTok, L);
                tmem_fence_after();
                issue_pv(kt, sv, j == 0);
                commit(&empty[sv]);
            }
            if (!ok) break;
            // every S MMA of the item has read Q buffer b when this arrives
            commit(&q_empty[b]);
            kt0 += nkt;
        }
        // every MMA this warp issued has finished before the CTA exits
        __syncwarp();
        commit(drain);
        if (lane == 0) mbar_drain_wait(smem_u32(drain), 0);
        __syncwarp();
    } else {
        // --------------------------------------------------------- softmax
        // Head half hh = warp / 4; within it thread t = token t of each tile
        // (row t of S^T) and row d = t of O^T.  Control flow is the same in a
        // half's four warps (trip counts and votes come from shared memory),
        // so its named barrier always meets; a wait that gave up only skips
        // the later waits of its warp.
        const int hh = warp >> 2, t = tid & 127, bar_id = 1 + hh;
        const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t col_s = hh * 32, col_o = COL_O + hh * 64;
        float* red = reinterpret_cast<float*>(smem + W::RED_OFF) + hh * 128;
        float* mrow = reinterpret_cast<float*>(smem + W::MROW_OFF) + hh * 32;
        float* alpha_s = reinterpret_cast<float*>(smem + W::ALPHA_OFF) + hh * 32;
        float* inv_s = reinterpret_cast<float*>(smem + W::INV_OFF) + hh * 32;
        const float sl = p.scale_log2;
        float l[32];
        int kt0 = 0, n = 0;
        for (;;) {
            const int b = n % QB;
            warp_wait(&q_full[b], (n / QB) & 1);
            if (!softmax_all(bar_id, ok)) break;
            const int4 r = rec[b];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&q_empty[b]));
            ++n;
            if (r.x < 0) break;
            const int s = r.x, L = r.y, z = r.z, nkt = r.w;
            const int g = z / HS, hs = z - (z / HS) * HS;
            const size_t out0 = ((size_t)s * p.num_heads + g * G + hs * NH + hh * 32) * kD + t;
            if (nkt == 0) {
#pragma unroll
                for (int h = 0; h < 32; ++h) store_out(p.out, out0 + (size_t)h * kD, 0.f, p.out_dtype);
                continue;
            }
            // the running max of each head lives in shared memory (mrow)
            if (warp % 4 == 0) mrow[lane] = -INFINITY;
#pragma unroll
            for (int h = 0; h < 32; ++h) l[h] = 0.f;
            softmax_sync(bar_id);
            for (int j = 0; j < nkt; ++j) {
                const int kt = kt0 + j, sb = kt & 1;
                uint8_t* pb = smem + W::P_OFF + sb * W::P_BYTES + hh * W::P_ATOM;
                warp_wait(&s_full[sb], (kt >> 1) & 1);
                tmem_fence_after();
                float x[32];
                tmem_ld32(tl + sb * NH + col_s, x);
                // S^T(kt) is in registers: its buffer may take S^T(kt + 2)
                tmem_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s_free[sb]));
                const uint32_t bm = bad_boxes(kt);
                const int box = (t >> 4) * IDS + (t & 15) / W::ROWS;
                const bool valid = j * kTok + t < L && !((bm >> box) & 1u);
                bool exceed = false;
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                    const float4 mv = *reinterpret_cast<const float4*>(mrow + h);
                    x[h] = valid ? x[h] * sl : -INFINITY;
                    x[h + 1] = valid ? x[h + 1] * sl : -INFINITY;
                    x[h + 2] = valid ? x[h + 2] * sl : -INFINITY;
                    x[h + 3] = valid ? x[h + 3] * sl : -INFINITY;
                    exceed |= x[h] > mv.x + 8.f || x[h + 1] > mv.y + 8.f ||
                              x[h + 2] > mv.z + 8.f || x[h + 3] > mv.w + 8.f;
                }
                // P buffer sb is free once P V(kt - 2) has read it; both the
                // vote's scratch and P go there
                if (kt >= 2) warp_wait(&o_done[sb], ((kt - 2) >> 1) & 1);
                if (softmax_any(bar_id, exceed)) {
                    // this tile's maximum per head, and the new running max
                    put_rows(pb, t, x);
                    softmax_sync(bar_id);
                    red[t] = column_op<true>(pb, t);
                    softmax_sync(bar_id);
                    if (warp % 4 == 0) {
                        const float mo = mrow[lane];
                        const float mn = fmaxf(fmaxf(fmaxf(red[lane], red[32 + lane]),
                                                     fmaxf(red[64 + lane], red[96 + lane])),
                                               mo);
                        alpha_s[lane] = mn == mo ? 1.f : ex2(mo - mn);  // mo = -inf: 0
                        mrow[lane] = mn;
                    }
                    softmax_sync(bar_id);
                    bool scaled = false;
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        const float a = alpha_s[h];
                        l[h] *= a;
                        scaled |= a != 1.f;
                    }
                    // O^T holds this item's earlier tiles: rescale its row once
                    // their P V has finished (scaled is the same in every thread)
                    if (j > 0 && scaled) {
                        warp_wait(&o_done[(kt - 1) & 1], ((kt - 1) >> 1) & 1);
                        tmem_fence_after();
#pragma unroll 1
                        for (int part = 0; part < 2; ++part) {
                            float o[32];
                            tmem_ld32(tl + col_o + part * 32, o);
#pragma unroll
                            for (int h = 0; h < 32; ++h) o[h] *= alpha_s[h];
                            tmem_st32(tl + col_o + part * 32, o);
                        }
                        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    }
                }
                // P = 2^(x - m) as 16-bit high parts and remainders, 8 heads
                // (one 16-byte chunk of each) at a time, heads in pairs (the
                // lower head in the low half); row t of P^T, MN-major with the
                // 128-byte swizzle: high parts in chunks 0-3, remainders 4-7
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int h = 8 * c + 2 * i;
                        const float2 mm = *reinterpret_cast<const float2*>(mrow + h);
                        const float m0 = mm.x == -INFINITY ? 0.f : mm.x;
                        const float m1 = mm.y == -INFINITY ? 0.f : mm.y;
                        float2 e = fsub2(make_float2(x[h], x[h + 1]), make_float2(m0, m1));
                        e.x = ex2(e.x);
                        e.y = ex2(e.y);
                        const float2 s2 = fadd2(make_float2(l[h], l[h + 1]), e);
                        l[h] = s2.x;
                        l[h + 1] = s2.y;
                        split_pair<T>(e.x, e.y, hw[i], lw[i]);
                    }
                    *reinterpret_cast<uint4*>(pb + swz(t, c)) =
                        make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(pb + swz(t, c + 4)) =
                        make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
                fence_proxy_async();
                tmem_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full[sb]));
            }
            // ---- epilogue: out[head][t] = O^T[t][head] / sum(head)
            const int kl = kt0 + nkt - 1;
            // the partial sums through a scratch in this half's atom of the P
            // buffer of tile kl - 1, free once its P V has finished, while the
            // last P V runs
            {
                uint8_t* scr = smem + W::P_OFF + ((kl - 1) & 1) * W::P_BYTES + hh * W::P_ATOM;
                if (kl >= 1) warp_wait(&o_done[(kl - 1) & 1], ((kl - 1) >> 1) & 1);
                put_rows(scr, t, l);
                softmax_sync(bar_id);
                red[t] = column_op<false>(scr, t);
                softmax_sync(bar_id);
                if (warp % 4 == 0) {
                    const float sum =
                        (red[lane] + red[32 + lane]) + (red[64 + lane] + red[96 + lane]);
                    inv_s[lane] = sum > 0.f ? 1.f / sum : 0.f;
                }
                softmax_sync(bar_id);
            }
            warp_wait(&o_done[kl & 1], (kl >> 1) & 1);
            tmem_fence_after();
            float o[32], o2[32];
            tmem_ld32(tl + col_o, o);
            tmem_ld32(tl + col_o + 32, o2);
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
                const float4 iv = *reinterpret_cast<const float4*>(inv_s + h);
                o[h] = (o[h] + o2[h]) * iv.x;
                o[h + 1] = (o[h + 1] + o2[h + 1]) * iv.y;
                o[h + 2] = (o[h + 2] + o2[h + 2]) * iv.z;
                o[h + 3] = (o[h + 3] + o2[h + 3]) * iv.w;
            }
            if (ok) store_column(p.out, out0, o, p.out_dtype);
            tmem_fence_before();
            kt0 += nkt;
        }
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                     "r"(W::TMEM_COLS)
                     : "memory");
}

template <typename T, int B, int NH>
cudaError_t launch_b(const DecodeParams& p, const void* kmap, const void* vmap, int items,
                     int sms, cudaStream_t stream)
{
    using W = W5<B, NH>;
    auto kern = decode_tc05_kernel<T, B, NH>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // persistent: one CTA a SM (its shared memory allows no second)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(items, sms));
    cfg.blockDim = dim3(W::THREADS);
    cfg.dynamicSmemBytes = W::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, *static_cast<const CUtensorMap*>(kmap),
                              *static_cast<const CUtensorMap*>(vmap));
}

template <typename T, int NH>
cudaError_t launch_t(const DecodeParams& p, const void* kmap, const void* vmap, int items, int sms,
                     cudaStream_t stream)
{
    if (p.block_size == 8) return launch_b<T, 8, NH>(p, kmap, vmap, items, sms, stream);
    if (p.block_size == 16) return launch_b<T, 16, NH>(p, kmap, vmap, items, sms, stream);
    if (p.block_size == 32) return launch_b<T, 32, NH>(p, kmap, vmap, items, sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

bool decode_wide_tcgen05_supported(int kv_dtype, int head_dim, int block_size, int group,
                                   const void* q)
{
    // q is read in 16-byte pieces
    return kv_dtype != PKV_F32 && head_dim == kD && group >= kDecodeWideHeads &&
           group % kDecodeWideHeads == 0 &&
           (block_size == 8 || block_size == 16 || block_size == 32) &&
           (reinterpret_cast<uintptr_t>(q) & 15) == 0;
}

int decode_wide_tcgen05_heads(int group) { return group % 64 == 0 ? 64 : 32; }

cudaError_t launch_decode_wide_tcgen05(const DecodeParams& p, int kv_dtype, const void* kmap,
                                       const void* vmap, int items, int sms, cudaStream_t stream)
{
    if (items <= 0) return cudaSuccess;
    if (sms <= 0) sms = 1;
    const int G = p.num_heads / p.num_kv_heads;
    if (G / p.head_slices == 64)
        return kv_dtype == PKV_BF16
                   ? launch_t<__nv_bfloat16, 64>(p, kmap, vmap, items, sms, stream)
                   : launch_t<__half, 64>(p, kmap, vmap, items, sms, stream);
    return kv_dtype == PKV_BF16 ? launch_t<__nv_bfloat16, 32>(p, kmap, vmap, items, sms, stream)
                                : launch_t<__half, 32>(p, kmap, vmap, items, sms, stream);
}
