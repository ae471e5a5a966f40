// Work plan of a split decode launch: the longest sequences first, no empty
// grid slots.
//
// A split launch's rectangular grid gives every (sequence, KV head, head
// slice) as many CTA slots as the longest context needs; with ragged
// lengths most of them are empty and exit at once, and the long items start
// wherever the caller put their sequence, so the launch often ends on a
// long item that started late.  This one-CTA kernel runs in place of the
// memset that zeroes the split's completion counters: it zeroes them, orders
// the sequences by context length, longest first (a counting sort on
// length buckets), and writes one record per CTA that has work -- (sequence,
// context length, KV head x head slice, partition group) -- consecutive in
// that order, plus their count.  The decode kernel's CTA b takes record b,
// or exits if b is past the count.  The order changes no result: every
// partition's softmax state and every merge are the same whichever CTA runs
// first.
//
// Both launches are programmatic dependent launches: the plan kernel starts
// while the previous decode launch's last CTAs still run (decode CTAs let
// dependents launch as they start), reads the lengths and builds the order
// in shared memory, then waits for that launch to complete before it writes
// counters and records; the decode CTAs are resident while the plan kernel
// finishes and wait for it to complete before they read a record.
#include <cuda_runtime.h>

#include <climits>

#include "pkv_kernels.h"

namespace {

constexpr int kPlanThreads = 1024;

struct PlanSmem {
    static constexpr int LENS = 0;                               // int [kPlanMaxSeqs]
    static constexpr int SORTED = LENS + kPlanMaxSeqs;           // int [kPlanMaxSeqs]
    static constexpr int OFF = SORTED + kPlanMaxSeqs;            // int [kPlanMaxSeqs]
    static constexpr int HIST = OFF + kPlanMaxSeqs;              // int [kPlanBuckets]
    static constexpr int WSUM = HIST + kPlanBuckets;             // int [32]
    static constexpr int INFO = WSUM + 32;                       // int [8], below
    static constexpr int INTS = INFO + 8;
    static constexpr int BYTES = INTS * 4;
    // INFO: over the non-empty sequences, the fewest and most stages, the
    // fewest partitions, their count; then the pieces per sequence (0: groups)
    static constexpr int MIN_NST = 0, MAX_NST = 1, MIN_PARTS = 2, NONEMPTY = 3, PIECES = 4;
};

// Pieces per sequence for near-equal contexts: the fewest c <= cmax whose
// items * c CTAs fill their last wave of `slots` to kPlanWaveFillPct; else
// the c with the fullest last wave (the fewest of equals).  One warp calls
// it, lane l trying c = l + 1, l + 33.  No c qualifies only when items is
// below ~20 waves of CTAs, so the products below stay far inside 64 bits.
__device__ int choose_pieces(long long items, int slots, int cmax)
{
    const int lane = threadIdx.x & 31;
    for (int c0 = 1; c0 <= cmax; c0 += 32) {
        const int c = c0 + lane;
        bool ok = false;
        if (c <= cmax) {
            const long long ctas = items * c;
            const long long room = (ctas + slots - 1) / slots * slots;
            ok = 100 * ctas >= (long long)kPlanWaveFillPct * room;
        }
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (m != 0u) return c0 + __ffs(m) - 1;
    }
    int best = 1;
    long long bc = 0, br = 1;  // fill of `best`: bc / br
    for (int c = 1 + lane; c <= cmax; c += 32) {
        const long long ctas = items * c;
        const long long room = (ctas + slots - 1) / slots * slots;
        if (ctas * br > bc * room) {
            best = c;
            bc = ctas;
            br = room;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const int b2 = __shfl_xor_sync(0xffffffffu, best, o);
        const long long c2 = __shfl_xor_sync(0xffffffffu, bc, o);
        const long long r2 = __shfl_xor_sync(0xffffffffu, br, o);
        const long long lhs = c2 * br, rhs = bc * r2;
        if (lhs > rhs || (lhs == rhs && b2 < best)) {
            best = b2;
            bc = c2;
            br = r2;
        }
    }
    return best;
}

// Exclusive prefix sum over the block of one value per thread; *total gets
// the sum.  Every thread of the block calls it.
__device__ int block_exclusive_scan(int v, int* wsum, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kPlanThreads / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = warp > 0 ? wsum[warp - 1] : 0;
    *total = wsum[kPlanThreads / 32 - 1];
    __syncthreads();  // wsum may be reused by the caller's next scan
    return before + x - v;
}

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const DecodePlanParams pp)
{
    extern __shared__ int psm[];
    int* lens = psm + PlanSmem::LENS;
    int* sorted = psm + PlanSmem::SORTED;
    int* off = psm + PlanSmem::OFF;
    int* hist = psm + PlanSmem::HIST;
    int* wsum = psm + PlanSmem::WSUM;
    const int tid = threadIdx.x;
    const int S = pp.num_seqs;
    // the decode launch that follows may start now: its CTAs wait for this
    // grid to complete (griddepcontrol.wait) before they read anything it
    // writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    int* info = psm + PlanSmem::INFO;
    for (int k = tid; k < kPlanBuckets; k += kPlanThreads) hist[k] = 0;
    if (tid == 0) {
        info[PlanSmem::MIN_NST] = INT_MAX;
        info[PlanSmem::MAX_NST] = 0;
        info[PlanSmem::MIN_PARTS] = INT_MAX;
        info[PlanSmem::NONEMPTY] = 0;
    }
    __syncthreads();
    // histogram of length buckets, longest bucket first (index 0); the
    // spread of the non-empty sequences' stage counts
    const int P = pp.partition_tokens;
    for (int s = tid; s < S; s += kPlanThreads) {
        const int L = pp.context_lens[s];
        lens[s] = L;
        const int Lc = (L < 0 || L > pp.max_len) ? 0 : L;  // the decode kernel flags it
        const int key = min(Lc >> pp.bucket_shift, kPlanBuckets - 1);
        atomicAdd(&hist[kPlanBuckets - 1 - key], 1);
        if (Lc > 0 && P > 0) {
            const int nst = (Lc + pp.stage_tokens - 1) / pp.stage_tokens;
            atomicMin(&info[PlanSmem::MIN_NST], nst);
            atomicMax(&info[PlanSmem::MAX_NST], nst);
            atomicMin(&info[PlanSmem::MIN_PARTS], (Lc + P - 1) / P);
            atomicAdd(&info[PlanSmem::NONEMPTY], 1);
        }
    }
    __syncthreads();
    // records per sequence: one per (KV head x head slice, partition group),
    // or, when the split contexts hold within 10 % the same number of stages,
    // one per (KV head x head slice, piece): `pieces` equal runs of stages
    // each, as many as fill the GPU's waves (at most the partitions, and the
    // groups, a sequence has room for)
    const int per_seq = pp.num_kv_heads * pp.head_slices;
    if (tid < 32) {  // warp 0; the condition is the same for all its lanes
        int pieces = 0;
        const int ne = info[PlanSmem::NONEMPTY];
        if (pp.slots > 0 && ne > 0 &&
            10LL * info[PlanSmem::MAX_NST] <= 11LL * info[PlanSmem::MIN_NST]) {
            const int cmax = min(min(info[PlanSmem::MIN_PARTS], pp.max_groups),
                                 min(kPlanMaxPieces, kPlanPieceMask));
            pieces = choose_pieces((long long)ne * per_seq, pp.slots, max(cmax, 1));
        }
        if (tid == 0) info[PlanSmem::PIECES] = pieces;
    }
    // bucket starts: exclusive scan, two buckets per thread
    {
        static_assert(kPlanBuckets == 2 * kPlanThreads, "two buckets a thread");
        const int a = hist[2 * tid], b = hist[2 * tid + 1];
        int total;
        const int ex = block_exclusive_scan(a + b, wsum, &total);
        __syncthreads();
        hist[2 * tid] = ex;
        hist[2 * tid + 1] = ex + a;
    }
    __syncthreads();
    // rank of each sequence (any order within a bucket)
    for (int s = tid; s < S; s += kPlanThreads) {
        const int L = lens[s];
        const int Lc = (L < 0 || L > pp.max_len) ? 0 : L;
        const int key = min(Lc >> pp.bucket_shift, kPlanBuckets - 1);
        sorted[atomicAdd(&hist[kPlanBuckets - 1 - key], 1)] = s;
    }
    __syncthreads();
    // a sequence with no tokens (or a bad length) keeps one record, whose
    // CTA writes its zero rows
    const int pieces = info[PlanSmem::PIECES];  // written before the barrier above
    auto groups_of = [&](int L) {
        const int Lc = (L < 0 || L > pp.max_len) ? 0 : L;
        if (pieces > 0) return Lc > 0 ? pieces : 1;
        const int np = max(1, (Lc + pp.partition_tokens - 1) / pp.partition_tokens);
        return (np + pp.cta_parts - 1) / pp.cta_parts;
    };
    int run = 0;
    for (int r0 = 0; r0 < S; r0 += kPlanThreads) {
        const int r = r0 + tid;
        const int c = r < S ? per_seq * groups_of(lens[sorted[r]]) : 0;
        int total;
        const int ex = block_exclusive_scan(c, wsum, &total);
        if (r < S) off[r] = run + ex;
        run += total;
    }
    __syncthreads();
    // Everything above read only the lengths.  When this kernel runs as a
    // programmatic dependent of the previous decode launch (which never
    // writes lengths), that much overlaps its last CTAs; the counters and
    // records it still reads are written only once it has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = tid; i < pp.num_counters; i += kPlanThreads) pp.done[i] = 0u;
    // a sequence's records: KV head, then partition group (or piece), then
    // head slice (the slices of one group adjacent: their reads of a K/V tile
    // meet in L2)
    const int HS = pp.head_slices;
    for (int r = tid; r < S; r += kPlanThreads) {
        const int s = sorted[r], L = lens[s];
        const int ng = groups_of(L);
        int4* out = pp.items + off[r];
        for (int g = 0; g < pp.num_kv_heads; ++g)
            for (int grp = 0; grp < ng; ++grp) {
                const int w = pieces > 0 ? kPlanPieceFlag | grp | (ng << kPlanPieceBits) : grp;
                for (int hs = 0; hs < HS; ++hs)
                    out[(g * ng + grp) * HS + hs] = make_int4(s, L, g * HS + hs, w);
            }
    }
    if (tid == 0) *pp.item_count = run;
}

}  // namespace

cudaError_t launch_decode_plan(const DecodePlanParams& pp, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(decode_plan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PlanSmem::BYTES);
    if (e != cudaSuccess) return e;
    // a programmatic dependent launch: it starts when the previous kernel on
    // the stream lets its dependents launch (the decode kernel does so as
    // its CTAs start; other kernels only at their end) and waits for that
    // kernel to complete before it writes anything
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = PlanSmem::BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_plan_kernel, pp);
}
