// Paged prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// for sm_103a, 16-bit KV cache.
//
// What it computes: the same as the warp-MMA prefill kernel -- rows
// query_start[s] .. query_start[s+1]-1 are the last qn tokens of sequence s
// and row t attends causally to the sequence's tokens 0 .. L-qn+t
// (cayang0802 walkthrough, recomputation; aiplusplus PagedAttention page,
// "key techniques" 1 for the block-table walk).
//
// How (GB300 design): one CTA of 10 warps per (256 query rows, query head,
// sequence), latest (heaviest) rows first; the rows form two 128-row tiles
// A and B whose softmax work alternates with each other's tensor-core work.
//  * warp 9 (loads): K and V tiles of 128 tokens by TMA (one copy per
//    16-row box of the paged cache brings both column halves, 128-byte
//    swizzle, [8-key group][column half][key][128 B]) into a ring of slots,
//    K(0) V(0) K(1) V(1) ...; its lanes read the tile's block-table entries
//    in parallel (one tile ahead) and record bad entries.
//  * warp 8 (MMA issue): S_X(j) = Q_X K(j)^T into tensor memory (M=128,
//    N=128, K=head_dim; Q and K K-major in shared memory), then
//    O_X += P_X(j) V(j) with P read from tensor memory (M=128, N=head_dim,
//    K=128; V the MN-major operand).  The whole warp computes the operands
//    and one elected lane issues.
//  * warps 0-3 (tile A) and 4-7 (tile B): thread r owns row r of its tile.
//    It reads its row of S from tensor memory in four 32-key chunks, masks
//    (diagonal, tail and bad blocks only), keeps a running max and sum in
//    base 2 and writes P back over the chunk of S it came from, as a 16-bit
//    high part and remainder for each 16-key step (both are multiplied,
//    keeping ~16 bits of P).  The running max used for P moves only when the
//    row max exceeds it by more than 8 (a factor 2^8), and only then is the O
//    row rescaled; O and the sum always share the same max, so the result is
//    unchanged.
//  * Tensor memory (512 columns): tile A S/P [0,128) O [128,256), tile B the
//    same at +256.  S_X(j+1) is issued once P_X(j) V(j) has read P_X(j),
//    before the other tile's P V.
// Every wait is bounded; a wait that gives up sets the TIMEOUT status bit
// (which ends the waits of every other CTA too), and before the CTA frees
// its tensor memory it waits (bounded) for its own copies and MMAs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <algorithm>
#include <type_traits>

#include "pkv.h"
#include "pkv_kernels.h"
#include "tc_common.cuh"
#include "tc05_common.cuh"

namespace {

using namespace pkv_tc;
using namespace pkv_tc05;

constexpr int kTileRows = 128;  // query rows per tile (MMA M)
constexpr int kQTiles = 2;      // query tiles per CTA
constexpr int kKeys = 128;      // keys per K/V tile
constexpr int kRing = 16;       // bad-block masks kept per tile index
constexpr int kMmaWarp = 8, kLoadWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTileCols = 256;  // tensor-memory columns per query tile
constexpr uint32_t kColO = 128;      // S/P at columns [0,128), O at [128,256)

template <int D, int B>
struct G5 {
    static constexpr int NH = D / 64;
    static constexpr int ROWS = B < 16 ? B : 16;  // rows per TMA box
    static constexpr int IDS = 16 / ROWS;         // boxes per 16-token group
    static constexpr int SUBS = (kKeys / 16) * IDS;  // boxes (copies) per key tile
    static constexpr int HALF_Q = kTileRows * 128;
    static constexpr int HALF_KV = kKeys * 128;
    // K/V tiles hold 8-key groups of RG_BYTES, each group's column halves
    // side by side (1024-byte swizzle atoms): key k, half hf at
    // (k / 8) RG_BYTES + hf 1024 + (k % 8) 128
    static constexpr int RG_BYTES = NH * 1024;
    static constexpr int Q_BYTES = NH * HALF_Q;
    static constexpr int SLOT_BYTES = NH * HALF_KV;
    static constexpr int SLOTS = D == 128 ? 4 : 8;  // K/V ring (one K or V tile each)
    // full, empty per slot; s_full, o_full, q_full per tile; p_half per tile
    // and half; drain
    static constexpr int BARS = 2 * SLOTS + 11;
    static constexpr int SLOT_OFF = kQTiles * Q_BYTES;
    static constexpr int BAR_OFF = SLOT_OFF + SLOTS * SLOT_BYTES;
    static constexpr int TSLOT_OFF = BAR_OFF + BARS * 8;
    static constexpr int KBAD_OFF = TSLOT_OFF + 16;
    static constexpr int SMEM_BYTES = 1024 + KBAD_OFF + kRing * 4;
    static_assert(HALF_KV % 1024 == 0 && HALF_Q % 1024 == 0, "swizzle atoms");
    static_assert(SUBS <= 32, "one lane per box");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// One work item: 256 query rows (tiles A and B) of one query head of one
// sequence.  Items are numbered (item_coords) so that consecutive items,
// taken by neighbouring CTAs, have about equal cost and share K/V in L2.
struct Item {
    int h, s, r0, qn, L, q0, g, base_pos, nkt_a, nkt_b, nkt;
};

// Item v's row tile (counted from the first), sequence and head.  Items come
// in groups of kSeqGroup sequences (the last group may hold fewer); within a
// group, the latest (heaviest) row tiles first, then the sequence, the head
// fastest.  A group's K/V (a few tens of MB for long prompts) stays in L2
// while its row tiles pass over it; all sequences at once would not.
constexpr int kSeqGroup = 4;
__device__ __forceinline__ void item_coords(const PrefillParams& p, int items_x, int v, int& ct,
                                            int& s, int& h)
{
    const int per_group = items_x * kSeqGroup * p.num_heads;
    const int gi = v / per_group;
    const int s0 = gi * kSeqGroup;
    const int per_level = min(kSeqGroup, p.num_seqs - s0) * p.num_heads;
    const int rem = v - gi * per_group;
    ct = items_x - 1 - rem / per_level;
    const int r2 = rem - (rem / per_level) * per_level;
    s = s0 + r2 / p.num_heads;
    h = r2 - (r2 / p.num_heads) * p.num_heads;
}

template <int B>
__device__ __forceinline__ bool decode_item(const PrefillParams& p, int items_x, int v, Item& it)
{
    int ct;
    item_coords(p, items_x, v, ct, it.s, it.h);
    it.r0 = p.query_start[it.s];
    it.qn = p.query_start[it.s + 1] - it.r0;
    it.L = p.context_lens[it.s];
    if (it.L < 0 || (int64_t)it.L > (int64_t)p.max_blocks * B || it.qn < 0 || it.qn > it.L ||
        it.qn > p.max_query_len)
        return false;  // flagged once per sequence by the load warp
    it.q0 = ct * kQTiles * kTileRows;
    if (it.q0 >= it.qn) return false;
    it.g = it.h / (p.num_heads / p.num_kv_heads);
    it.base_pos = it.L - it.qn;
    auto tiles_for = [&](int x) {
        const int rows = min(it.qn - (it.q0 + x * kTileRows), kTileRows);
        return rows > 0 ? (it.base_pos + it.q0 + x * kTileRows + rows - 1) / kKeys + 1 : 0;
    };
    it.nkt_a = tiles_for(0);
    it.nkt_b = tiles_for(1);
    it.nkt = max(it.nkt_a, it.nkt_b);
    return true;
}

template <int B>
__device__ __forceinline__ bool item_bad_lengths(const PrefillParams& p, int items_x, int v)
{
    int ct, s, h;
    item_coords(p, items_x, v, ct, s, h);
    if (ct != items_x - 1 || h != 0) return false;  // once per sequence
    const int qn = p.query_start[s + 1] - p.query_start[s];
    const int L = p.context_lens[s];
    return L < 0 || (int64_t)L > (int64_t)p.max_blocks * B || qn < 0 || qn > L ||
           qn > p.max_query_len;
}

template <typename T, int D, int B>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc05_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, int items_x)
{
    using Gm = G5<D, B>;
    constexpr int IDS = Gm::IDS;
    constexpr int SLOTS = Gm::SLOTS;
    const int total_items = items_x * p.num_heads * p.num_seqs;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Gm::BAR_OFF);
    uint64_t* empty = full + SLOTS;
    uint64_t* s_full = empty + SLOTS;  // [tile]
    uint64_t* p_half = s_full + 2;     // [tile * 2 + half], one arrival per softmax warp
    uint64_t* o_full = p_half + 4;     // [tile]
    uint64_t* q_full = o_full + 2;     // [tile], one arrival per softmax warp
    uint64_t* drain = q_full + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Gm::TSLOT_OFF);
    uint32_t* kbad = reinterpret_cast<uint32_t*>(smem + Gm::KBAD_OFF);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < Gm::BARS; ++i) {
            uint64_t* b = &full[i];
            const bool per_warp = (b >= p_half && b < p_half + 4) || b == &q_full[0] ||
                                  b == &q_full[1];
            mbar_init(smem_u32(b), per_warp ? 4 : 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tslot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
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
    // ring position of K(kt) (t = 2 kt) and V(kt) (t = 2 kt + 1), kt counted
    // over all of this CTA's key tiles
    auto slot_of = [](int t) { return t % SLOTS; };
    auto phase_of = [](int t) { return (t / SLOTS) & 1; };

    if (warp == kLoadWarp) {
        // ------------------------------------------------------------ loads
        int t = 0, kt0 = 0;
        const int grp = lane / IDS, u = lane % IDS;
        for (int v = blockIdx.x; v < total_items && ok; v += gridDim.x) {
            if (lane == 0 && item_bad_lengths<B>(p, items_x, v))
                atomicOr(p.status, PKV_STATUS_BAD_LEN);
            Item it;
            if (!decode_item<B>(p, items_x, v, it)) continue;
            const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks;
            // block-table entry of this lane's box in key tile j (-1: past the
            // context); read one tile ahead so the load latency is hidden
            auto entry = [&](int j) {
                const int tok = j * kKeys + grp * 16 + u * Gm::ROWS;
                return (lane < Gm::SUBS && j < it.nkt && tok < it.L) ? table[tok / B] : -1;
            };
            int id_next = entry(0);
            for (int j = 0; j < it.nkt; ++j) {
                const int tok = j * kKeys + grp * 16 + u * Gm::ROWS;
                int id = id_next;
                const bool bad = lane < Gm::SUBS && tok < it.L && (id < 0 || id >= p.num_blocks);
                if (bad) id = -1;
                id_next = entry(j + 1);
                const unsigned have = __ballot_sync(0xffffffffu, id >= 0);
                const unsigned bads = __ballot_sync(0xffffffffu, bad);
                for (int kv = 0; kv < 2; ++kv, ++t) {
                    const int sl = slot_of(t);
                    if (t >= SLOTS && lane == 0) wait(&empty[sl], ((t / SLOTS) - 1) & 1);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    const uint32_t bar = smem_u32(&full[sl]);
                    if (lane == 0) {
                        if (kv == 0) {
                            kbad[(kt0 + j) % kRing] = bads;
                            if (bads) atomicOr(p.status, PKV_STATUS_BAD_BLOCK);
                        }
                        mbar_arrive_expect_tx(bar, __popc(have) * Gm::NH * Gm::ROWS * 128);
                    }
                    __syncwarp();
                    if (id >= 0) {
                        const int row =
                            (id * p.num_kv_heads + it.g) * B + (IDS > 1 ? 0 : tok % B);
                        const uint32_t dst =
                            smem_u32(smem + Gm::SLOT_OFF + sl * Gm::SLOT_BYTES) +
                            (grp * 16 + u * Gm::ROWS) / 8 * Gm::RG_BYTES;
                        // one copy brings the box's rows of every column half
                        tma_load_4d(dst, kv ? &vmap : &kmap, 0, 0, 0, row / 8, bar);
                    }
                }
                if (!ok) break;
            }
            kt0 += it.nkt;
        }
        // the ring's last fills must have landed before the CTA exits
        if (lane == 0)
            for (int f = max(0, t - SLOTS); f < t; ++f)
                mbar_drain_wait(smem_u32(&full[slot_of(f)]), phase_of(f));
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issue
        const uint32_t id_s = instr_desc<T>(kTileRows, kKeys, 0);
        const uint32_t id_o = instr_desc<T>(kTileRows, D, 1);
        const uint32_t tm = __shfl_sync(0xffffffffu, tbase, 0);  // warp-uniform
        const uint32_t q_base = smem_u32(smem);
        const uint32_t slot_base = smem_u32(smem + Gm::SLOT_OFF);
        // descriptors of Q and of ring slot 0; every operand is one of these
        // moved by a constant or per-slot offset
        const uint64_t q_desc = smem_desc(q_base, 16, 1024);
        const uint64_t k_desc = smem_desc(slot_base, 16, Gm::RG_BYTES);  // K-major
        const uint64_t v_desc = smem_desc(slot_base, 1024, Gm::RG_BYTES);  // MN-major
        // S_x = Q_x K(kt)^T into tile x's S/P columns
        auto issue_s = [&](int x, int kt) {
            const uint64_t qd = desc_add(q_desc, x * Gm::Q_BYTES);
            const uint64_t kd = desc_add(k_desc, slot_of(2 * kt) * Gm::SLOT_BYTES);
            const uint32_t d = tm + x * kTileCols;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma(d, desc_add(qd, (kk >> 2) * Gm::HALF_Q + (kk & 3) * 32),
                         desc_add(kd, (kk >> 2) * 1024 + (kk & 3) * 32), id_s, kk > 0);
                umma_commit(smem_u32(&s_full[x]));
            }
            __syncwarp();
        };
        // O_x (+)= P_x V(kt) for keys [64 hh, 64 hh + 64); P of 16-key step
        // kk at columns 16 kk (high parts) and 16 kk + 8 (remainders)
        auto issue_pv_half = [&](int x, int kt, int hh, bool first) {
            const uint64_t vd = desc_add(v_desc, slot_of(2 * kt + 1) * Gm::SLOT_BYTES);
            const uint32_t pc = tm + x * kTileCols;
            const uint32_t oc = tm + x * kTileCols + kColO;
            if (elect_one()) {
#pragma unroll
                for (int k4 = 0; k4 < kKeys / 32; ++k4) {
                    const int kk = hh * (kKeys / 32) + k4;
                    const uint64_t b = desc_add(vd, kk * 2 * Gm::RG_BYTES);
                    umma_ts(oc, pc + kk * 16, b, id_o, !first || kk > 0);
                    umma_ts(oc, pc + kk * 16 + 8, b, id_o, 1);
                }
                if (hh == 1) umma_commit(smem_u32(&o_full[x]));
            }
            __syncwarp();
        };
        // commit from the issuing lane (tracks every MMA it issued so far)
        auto commit = [&](uint64_t* bar) {
            if (elect_one()) umma_commit(smem_u32(bar));
            __syncwarp();
        };
        auto k_ready = [&](int kt) {
            if (lane == 0) wait(&full[slot_of(2 * kt)], phase_of(2 * kt));
            ok = __shfl_sync(0xffffffffu, ok, 0);
        };
        // V(kt) landed; rows of keys past the context or in a bad block are
        // zeroed (their P is 0, and 0 * NaN must not reach O)
        auto v_ready = [&](int kt, int key0, int L) {
            const int t = 2 * kt + 1;
            if (lane == 0) wait(&full[slot_of(t)], phase_of(t));
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();  // the other lanes read kbad after lane 0's acquire
            const uint32_t bm = kbad[kt % kRing];
            if (ok && (key0 + kKeys > L || bm)) {
                uint8_t* vt = smem + Gm::SLOT_OFF + slot_of(t) * Gm::SLOT_BYTES;
                for (int i = lane; i < Gm::NH * kKeys * 8; i += 32) {
                    const int hf = i / (kKeys * 8), k = (i >> 3) % kKeys, c = i & 7;
                    const int box = (k >> 4) * IDS + (k & 15) / Gm::ROWS;
                    if (key0 + k >= L || ((bm >> box) & 1u))
                        *reinterpret_cast<uint4*>(vt + (k >> 3) * Gm::RG_BYTES + hf * 1024 +
                                                  (k & 7) * 128 + c * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();
            }
            __syncwarp();
        };

        // per tile x: S/P/O phases count this CTA's key tiles of x so far
        // (n[x]); q_full phases count the items in which x has rows (nq[x])
        int n[kQTiles] = {0, 0}, nq[kQTiles] = {0, 0};
        int kt0 = 0;
        for (int v = blockIdx.x; v < total_items && ok; v += gridDim.x) {
            Item it;
            if (!decode_item<B>(p, items_x, v, it)) continue;
            auto nkt_of = [&](int x) { return x ? it.nkt_b : it.nkt_a; };
            // S_x of the first key tile: after the softmax of x has loaded the
            // new Q and read out the previous O, and the previous P V_x (which
            // read P in the S columns) has finished
            k_ready(kt0);
            for (int x = 0; x < kQTiles && ok; ++x) {
                if (nkt_of(x) == 0) continue;
                if (lane == 0) {
                    wait(&q_full[x], nq[x] & 1);
                    if (n[x] > 0) wait(&o_full[x], (n[x] - 1) & 1);
                }
                ++nq[x];
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                tmem_fence_after();
                issue_s(x, kt0);
            }
            if (!ok) break;
            commit(&empty[slot_of(2 * kt0)]);
            // per key tile j and query tile x: P_x(j) V(j), then S_x(j + 1) as
            // soon as that P V has read P_x(j) (it shares S_x's columns), ahead
            // of the other tile's P V
            for (int j = 0; j < it.nkt && ok; ++j) {
                const int kt = kt0 + j;
                v_ready(kt, j * kKeys, it.L);
                for (int x = 0; x < kQTiles && ok; ++x) {
                    if (j >= nkt_of(x)) continue;
                    // the first half of P_x(j) goes to the tensor cores while the
                    // softmax computes the second.  Usually the softmax has posted
                    // both halves before this warp gets here; a completed second
                    // half implies the first (each softmax warp arrives on the
                    // first half before the second), so one test covers both
                    bool both = false;
                    if (lane == 0) both = mbar_test_wait(smem_u32(&p_half[x * 2 + 1]), n[x] & 1);
                    both = __shfl_sync(0xffffffffu, both, 0);
                    for (int hh = 0; hh < 2 && ok; ++hh) {
                        if (!both) {
                            if (lane == 0) wait(&p_half[x * 2 + hh], n[x] & 1);
                            ok = __shfl_sync(0xffffffffu, ok, 0);
                            if (!ok) break;
                        }
                        tmem_fence_after();
                        issue_pv_half(x, kt, hh, j == 0);
                    }
                    if (!ok) break;
                    ++n[x];
                    if (j + 1 >= nkt_of(x)) continue;
                    k_ready(kt + 1);
                    if (lane == 0) wait(&o_full[x], (n[x] - 1) & 1);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok) issue_s(x, kt + 1);
                }
                if (!ok) break;
                commit(&empty[slot_of(2 * kt + 1)]);
                if (j + 1 < it.nkt) commit(&empty[slot_of(2 * kt + 2)]);
            }
            kt0 += it.nkt;
        }
        // every MMA this warp issued has finished before the CTA exits
        __syncwarp();
        commit(drain);
        if (lane == 0) mbar_drain_wait(smem_u32(drain), 0);
        __syncwarp();
    } else {
        // --------------------------------------------------------- softmax
        const int x = warp >> 2, r = tid & (kTileRows - 1);
        const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16) + x * kTileCols;
        const float sl = p.scale_log2;
        const bool vec = (reinterpret_cast<uintptr_t>(p.out) & 15) == 0;
        uint8_t* qx = smem + x * Gm::Q_BYTES;
        // This thread's row of item it2's Q into shared memory by asynchronous
        // 16-byte copies (zeros past qn), and the wait that makes them visible
        // to the tensor cores before the hand-over to the MMA warp.
        // The warp copies its 32 rows together, D / 8 16-byte pieces a row, so
        // that each instruction reads whole rows (rows are H D elements apart).
        auto issue_q = [&](const Item& it2) {
            constexpr int PIECES = D / 8;
            const int wrow0 = (warp & 3) * 32;
#pragma unroll
            for (int u = 0; u < PIECES; ++u) {
                const int idx = u * 32 + lane;
                const int t = wrow0 + idx / PIECES, c = idx % PIECES;
                const int row2 = it2.q0 + x * kTileRows + t;
                const bool have = row2 < it2.qn;
                const T* src = static_cast<const T*>(p.q) +
                               ((size_t)(it2.r0 + (have ? row2 : 0)) * p.num_heads + it2.h) * D +
                               c * 8;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                                 smem_u32(qx + (c >> 3) * Gm::HALF_Q + swz(t, c & 7))),
                             "l"(src), "r"(have ? 16u : 0u)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        auto hand_over_q = [&]() {
            asm volatile("cp.async.wait_all;" ::: "memory");
            fence_proxy_async();
            tmem_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&q_full[x]));
        };
        int n = 0, kt0 = 0;
        int preloaded = -1;  // the item whose Q the previous epilogue already brought in
        for (int v = blockIdx.x; v < total_items && ok; v += gridDim.x) {
            Item it;
            if (!decode_item<B>(p, items_x, v, it)) continue;
            const int my_nkt = x ? it.nkt_b : it.nkt_a;
            const int row = it.q0 + x * kTileRows + r;
            const int pos = row < it.qn ? it.base_pos + row : -1;  // -1: padding row
            if (my_nkt > 0) {
                // this row of Q into shared memory (zero past qn), unless this
                // tile's previous item's epilogue did it; the S MMAs of that item
                // finished before its last softmax
                if (preloaded != v) {
                    issue_q(it);
                    hand_over_q();
                }
                // the next item's Q row of this thread into L2 meanwhile
                {
                    Item nx;
                    const int vn = v + gridDim.x;
                    if (vn < total_items && decode_item<B>(p, items_x, vn, nx)) {
                        const int rn = nx.q0 + x * kTileRows + r;
                        if (rn < nx.qn) {
                            const T* qn_src = static_cast<const T*>(p.q) +
                                              ((size_t)(nx.r0 + rn) * p.num_heads + nx.h) * D;
#pragma unroll
                            for (int c = 0; c < D * (int)sizeof(T); c += 128)
                                asm volatile("prefetch.global.L2 [%0];" ::"l"(
                                    reinterpret_cast<const uint8_t*>(qn_src) + c));
                        }
                    }
                }
            }
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < my_nkt; ++j, ++n) {
                // S_x(j) done; K(j) had landed (and its kbad entry was written
                // before the load warp's release-arrive) before S_x(j) was
                // issued.  P V_x(j-1) finished before S_x(j) was issued; waiting
                // for it here keeps every o_full phase waited in turn (a parity
                // wait must not fall two phases behind)
                wait(&s_full[x], n & 1);
                if (j > 0) wait(&o_full[x], (n - 1) & 1);
                tmem_fence_after();
                const int key0 = j * kKeys;
                const uint32_t bm = kbad[(kt0 + j) % kRing];
                // unmasked tile for the whole warp (every key visible and loaded,
                // positive scale): scores stay raw and the scale is folded into
                // the exponent's FMA.  Otherwise pass 1 writes the scaled scores
                // back over S, -inf where a key is masked, for pass 2 to read
                const bool plain = key0 + kKeys - 1 <= pos && bm == 0 && sl > 0.f;
                const bool wplain = __all_sync(0xffffffffu, plain);
                const float mul = wplain ? sl : 1.f;
                // keys of chunk c this row may see: causally visible (k <= pos -
                // key0) and not in a bad block (one bit of bm per box of ROWS keys)
                auto chunk_valid = [&](int c) {
                    const int r = pos - key0 - c * 32;
                    uint32_t v = r >= 31 ? 0xffffffffu : r < 0 ? 0u : (2u << r) - 1u;
                    const uint32_t bb = bm >> (c * 2 * IDS);
#pragma unroll
                    for (int q = 0; q < 2 * IDS; ++q)
                        if ((bb >> q) & 1u) v &= ~(((1u << Gm::ROWS) - 1u) << (q * Gm::ROWS));
                    return v;
                };
                // pass 1: row max (eight independent partial maxima).  The
                // 32-key chunks of both passes are rolled loops: unrolled code
                // (with the masked variant of the diagonal tiles) did not stay in
                // the instruction cache
                float mp[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
                if (wplain) {
#pragma unroll 1
                    for (int c = 0; c < kKeys / 32; ++c) {
                        float vv[32];
                        tmem_ld32(tl + c * 32, vv);
#pragma unroll
                        for (int i = 0; i < 32; i += 16)
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                mp[e] = fmax3(mp[e], vv[i + e], vv[i + 8 + e]);
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < kKeys / 32; ++c) {
                        float vv[32];
                        tmem_ld32(tl + c * 32, vv);
                        const uint32_t valid = chunk_valid(c);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            vv[i] = (valid >> i) & 1u ? vv[i] * sl : -INFINITY;
                        tmem_st32(tl + c * 32, vv);
#pragma unroll
                        for (int i = 0; i < 32; i += 16)
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                mp[e] = fmax3(mp[e], vv[i + e], vv[i + 8 + e]);
                    }
                    // the masked scores are in place before pass 2 reads them
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
#pragma unroll
                for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                    for (int i = 0; i < w; ++i) mp[i] = fmaxf(mp[i], mp[i + w]);
                const float mx = mp[0] * mul;
                float alpha = 1.f;
                bool rescale = false;
                if (mx > m + 8.f) {  // also the first finite max (m = -inf)
                    rescale = m != -INFINITY;
                    alpha = ex2(m - mx);
                    m = mx;
                }
                const float ms = m == -INFINITY ? 0.f : m;
                // O is rescaled before P V_x(j) is issued (it waits for p_half).
                // A rolled loop: this path runs on an item's first tile and
                // rarely after, so its code is cold in the instruction cache
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tl + kColO + c * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(tl + kColO + c * 32, o);
                    }
                }
                // pass 2: P = 2^(s - m) per chunk, written over that chunk of S
                // as [16-key step][high parts 8 columns][remainders 8 columns]
                float2 sum2 = make_float2(0.f, 0.f);
                const float2 mul2 = make_float2(mul, mul), nms2 = make_float2(-ms, -ms);
#pragma unroll 1
                for (int c = 0; c < kKeys / 32; ++c) {
                    float vv[32];
                    tmem_ld32(tl + c * 32, vv);
                    float pw[32];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int k = half * 16 + 2 * i;
                            float2 e = ffma2(make_float2(vv[k], vv[k + 1]), mul2, nms2);
                            e.x = ex2(e.x);
                            e.y = ex2(e.y);
                            sum2 = fadd2(sum2, e);
                            uint32_t hw, lw;
                            split_pair<T>(e.x, e.y, hw, lw);
                            pw[half * 16 + i] = __uint_as_float(hw);
                            pw[half * 16 + 8 + i] = __uint_as_float(lw);
                        }
                    }
                    tmem_st32(tl + c * 32, pw);
                    if (c == kKeys / 64 - 1 || c == kKeys / 32 - 1) {
                        // a half of P_x(j) is in place: its P V may start
                        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                        tmem_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(smem_u32(&p_half[x * 2 + (c == kKeys / 32 - 1)]));
                    }
                }
                l = l * alpha + (sum2.x + sum2.y);
            }
            // ---- epilogue: O / l for this thread's row
            if (my_nkt > 0) {
                wait(&o_full[x], (n - 1) & 1);
                tmem_fence_after();
                // the next item in which this tile has rows: its Q comes in while
                // O is read out (this item's last S on this tile has completed)
                Item nx;
                int vn = v + gridDim.x;
                for (; vn < total_items; vn += gridDim.x)
                    if (decode_item<B>(p, items_x, vn, nx) && (x ? nx.nkt_b : nx.nkt_a) > 0) break;
                const bool early = ok && vn < total_items;
                if (early) issue_q(nx);
                const float inv = l > 0.f ? 1.f / l : 0.f;
                // rolled, like the rescale: once an item
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tl + kColO + c * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= inv;
                    if (pos >= 0 && ok)
                        store_row32(p.out,
                                    ((size_t)(it.r0 + row) * p.num_heads + it.h) * D + c * 32,
                                    o, p.out_dtype, vec);
                }
                tmem_fence_before();
                if (early) {
                    hand_over_q();
                    preloaded = vn;
                }
            }
            kt0 += it.nkt;
        }
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                     "r"(kTmemCols)
                     : "memory");
}

int sm_count()
{
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (count[dev] == 0) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
            c = 148;
        count[dev] = c;
    }
    return count[dev];
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
    const int rows = kQTiles * kTileRows;
    const int items_x = (p.max_query_len + rows - 1) / rows;
    const long long items = (long long)items_x * p.num_heads * p.num_seqs;
    if (items <= 0) return cudaSuccess;
    if (items > (1ll << 31) - 1) return cudaErrorInvalidValue;
    // persistent: one CTA per SM (shared memory and tensor memory allow one)
    const int grid = (int)std::min<long long>(items, sm_count());
    kern<<<grid, kThreads, Gm::SMEM_BYTES, stream>>>(p, *static_cast<const CUtensorMap*>(kmap),
                                                     *static_cast<const CUtensorMap*>(vmap),
                                                     items_x);
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
