// Launch interfaces between the C-ABI layer (api.cu) and the kernel files.
// Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

// Everything one decode launch needs; passed by value as a kernel parameter.
struct DecodeParams {
    void* out;                   // [S][Hq][D], out_dtype
    const void* q;               // [S][Hq][D], kv dtype
    const void* k_cache;         // [NB][Hkv][B][D]
    const void* v_cache;
    const int32_t* block_tables; // [S][max_blocks]
    const int32_t* context_lens; // [S]
    float scale_log2;            // softmax scale * log2(e): scores live in base 2
    int block_size, num_kv_heads, num_heads, head_dim;
    int num_seqs, max_blocks, num_blocks;
    int partition_tokens;        // tokens per partition (>= max context if unsplit)
    int max_partitions;          // ceil(max_blocks * block_size / partition_tokens)
    int cta_parts;               // tensor-core kernel: consecutive partitions per CTA
                                 // (1, or kDecodeTcWarps: one partition per warp)
    int head_slices;             // tensor-core kernel: CTAs that split one KV group's
                                 // G query heads, ceil(G / HS) columns each (<= 16)
    int out_dtype;
    float2* ws_ml;               // [S][Hq][max_partitions] (max, sum) in base 2
    float* ws_o;                 // [S][Hq][max_partitions][D] unnormalised output
    unsigned int* done;          // [S][Hkv][HS] partitions finished (tensor-core split mode)
    unsigned int* status;        // device status word (PKV_STATUS_* bits)
    // Decode step with append (tensor-core kernel only; NULL otherwise): the
    // K/V of each sequence's new token, [S][Hkv][D] in the cache dtype, is
    // written at position context_lens[s]-1 before it is attended.
    const void* new_k;
    const void* new_v;
    // Beam groups (tensor-core kernel only; NULL otherwise): group i holds
    // sequences group_start[i] .. group_start[i+1]-1, whose first
    // shared_tokens[i] tokens use the same physical blocks.
    const int32_t* group_start;
    const int32_t* shared_tokens;
    int num_groups;
    // Split launches with a work plan (tensor-core kernel only; NULL
    // otherwise): CTA b takes record items[b] = (sequence, context length,
    // KV head * head_slices + head slice, w) if b < *item_count, and exits
    // otherwise.  w is a partition group, or (with kPlanPieceFlag set) piece
    // w & kPlanPieceMask of (w >> kPlanPieceBits) & kPlanPieceMask equal
    // runs of the sequence's stages.  Written by the plan kernel just before.
    const int4* items;
    const int* item_count;
    // Wide-group tcgen05 kernel with a work plan: CTAs take the records in
    // order through this counter (zeroed by the plan kernel); NULL otherwise.
    int* item_next;
};

// Work plan of a split tensor-core launch (decode_plan.cu): zeroes the
// completion counters, orders the sequences longest first and writes one
// record per CTA with work, in that order.  One CTA; num_seqs <= kPlanMaxSeqs.
// When every non-empty context of a split launch has about the same number
// of stages, the plan cuts each into the same number of equal runs (pieces)
// instead of partition groups, so that the CTAs fill whole waves.
constexpr int kPlanMaxSeqs = 4096;
constexpr int kPlanBuckets = 2048;  // length buckets of the counting sort
constexpr int kPlanPieceFlag = 1 << 30;
constexpr int kPlanPieceBits = 15;
constexpr int kPlanPieceMask = (1 << kPlanPieceBits) - 1;
constexpr int kPlanMaxPieces = 64;       // pieces per sequence the plan considers
constexpr int kPlanWaveFillPct = 95;     // the fewest pieces whose last wave is this full
struct DecodePlanParams {
    const int32_t* context_lens;  // [num_seqs]
    int num_seqs, num_kv_heads, head_slices;
    int partition_tokens, cta_parts;
    int stage_tokens;             // tokens per stage of the decode kernel
    int slots;                    // decode CTAs the GPU holds at once (0: no pieces)
    int max_groups;               // record slots a (sequence, KV head, slice) has in the grid
    int max_len;                  // max_blocks * block_size: longer lengths are bad
    int bucket_shift;             // bucket of a length L: min(L >> shift, kPlanBuckets - 1)
    int4* items;                  // capacity: the launch's grid
    int* item_count;
    unsigned int* done;           // completion counters to zero
    int num_counters;
};
cudaError_t launch_decode_plan(const DecodePlanParams& pp, cudaStream_t stream);

// Everything one prefill launch needs (passed by value).
struct PrefillParams {
    void* out;                   // [rows][Hq][D], out_dtype
    const void* q;               // [rows][Hq][D], kv dtype
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables; // [S][max_blocks]
    const int32_t* context_lens; // [S]
    const int32_t* query_start;  // [S + 1] first query row of each sequence
    float scale_log2;
    int block_size, num_kv_heads, num_heads, head_dim;
    int num_seqs, max_blocks, num_blocks, max_query_len;
    int out_dtype;
    unsigned int* status;
};

// Tensor-core paged prefill (16-bit KV): one CTA per (64 query rows, query
// head, sequence); tensor maps as for the decode kernel.
cudaError_t launch_prefill_tensor_core(const PrefillParams& p, int kv_dtype, const void* k_map,
                                       const void* v_map, cudaStream_t stream);

// The same on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory): one CTA per (128 query rows, query head, sequence).
cudaError_t launch_prefill_tcgen05(const PrefillParams& p, int kv_dtype, const void* k_map,
                                   const void* v_map, cudaStream_t stream);

// Device status word of the current device (address of a __device__ symbol).
unsigned int* pkv_status_word_ptr();

cudaError_t launch_kv_write(void* k_cache, void* v_cache, const void* key, const void* value,
                            const int64_t* slot_mapping, int num_tokens, int num_blocks,
                            int num_kv_heads, int head_dim, int block_size, int elem_bytes,
                            unsigned int* status, cudaStream_t stream);

// Appends one token per sequence: new_k/new_v [S][Hkv][D] go to position
// context_lens[s]-1 through the block table (one CTA per sequence and KV head).
cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* new_k, const void* new_v,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int num_seqs, int max_blocks, int num_blocks, int num_kv_heads,
                             int head_dim, int block_size, int elem_bytes, unsigned int* status,
                             cudaStream_t stream);

cudaError_t launch_kv_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs,
                                  int num_pairs, int num_blocks, size_t block_bytes,
                                  unsigned int* status, cudaStream_t stream);

// Whole blocks (all heads, K and V) from pool `src` to pool `dst`; either pool
// may be device memory or pinned host memory mapped into the address space.
cudaError_t launch_kv_swap_blocks(void* dst_k, void* dst_v, const void* src_k, const void* src_v,
                                  const int64_t* pairs, int num_pairs, int num_src_blocks,
                                  int num_dst_blocks, size_t block_bytes, unsigned int* status,
                                  cudaStream_t stream);

// CUDA-core decode (any dtype, any group size).  Grid: partitions x heads x seqs.
cudaError_t launch_decode_cuda_core(const DecodeParams& p, int kv_dtype, cudaStream_t stream);

// Tensor-core decode (16-bit KV), one CTA per (sequence, KV head, group of
// p.cta_parts consecutive partitions, head slice), in that order (the head
// slices of one partition group adjacent in the grid); the grid is
// S * Hkv * HS * ceil(max_partitions / cta_parts).  A CTA takes ceil(G / HS)
// query heads as the mma's N columns: launch_decode_tensor_core up to 8
// (one n8 tile), launch_decode_tensor_core_wide up to 16 (two tiles).  A CTA
// that holds one partition spreads it over all its warps; one that holds
// several gives each warp a partition of its own.  The tensor maps describe
// k_cache / v_cache as 3-D [D/64 halves][NB*Hkv*B rows][64 columns], loaded
// in boxes of both halves x min(B, 16) rows.  In split mode p.done must be
// zero; the CTA that finishes the last partition of a (sequence, KV head,
// head slice) merges its partitions.
constexpr int kDecodeTcWarps = 4;
// CTAs of the (ungrouped) tensor-core decode kernel one SM holds: its 8 KB
// stages (16 tokens at head_dim 128, 32 at 64) take ~67 KB of shared memory
constexpr int kDecodeTcCtasPerSm = 3;
// Split partitions of at most this many tokens get one warp each (four per
// CTA), so that a CTA's start-up and end are spread over more KV bytes, when
// the longest context spans at least kWarpPartitionMinCount of them.
constexpr int kWarpPartitionMaxTokens = 512;
constexpr int kWarpPartitionMinCount = 16;
constexpr int kDecodeTcMaxColumns = 16;
// Tokens per stage of the tensor-core decode kernel: 16 (one m16 token tile),
// or 32 at head_dim 64 outside beam groups, so that a stage is 8 KB of K and V
// at either head_dim.  The TMA boxes of its tensor maps hold
// min(block_size, stage tokens) rows.
constexpr int decode_stage_tokens(int head_dim, bool grouped)
{
    return head_dim == 64 && !grouped ? 32 : 16;
}
constexpr int decode_box_rows(int head_dim, int block_size, bool grouped)
{
    return block_size < decode_stage_tokens(head_dim, grouped)
               ? block_size
               : decode_stage_tokens(head_dim, grouped);
}
cudaError_t launch_decode_tensor_core(const DecodeParams& p, int kv_dtype, const void* k_map,
                                      const void* v_map, long long grid, cudaStream_t stream);
cudaError_t launch_decode_tensor_core_wide(const DecodeParams& p, int kv_dtype, const void* k_map,
                                           const void* v_map, long long grid, cudaStream_t stream);
// The same kernel with 3-stage rings, two CTAs a SM (wide: two column tiles),
// for unsplit launches of at most kDecodeTcDeepMaxWaves waves of
// kDecodeTcCtasPerSm CTAs a SM: few items, each streaming much.
constexpr int kDecodeTcDeepMaxWaves = 2;
cudaError_t launch_decode_tensor_core_deep(const DecodeParams& p, int kv_dtype, const void* k_map,
                                           const void* v_map, long long grid, bool wide,
                                           cudaStream_t stream);

// Unsplit decode for groups of G = 32 k query heads per KV head on the
// tcgen05 tensor cores (decode_tc05.cu): items (sequence, KV head, slice of
// decode_wide_tcgen05_heads(G) query heads: 64 when G is a multiple of 64,
// else 32), p.head_slices = G / that, taken by persistent CTAs (one a SM, at
// most `sms`) from p.items through p.item_next when p.items is set, else in
// grid-stride order.  16-bit KV, head_dim 128, block size 8, 16 or 32, q
// 16-byte aligned; a programmatic dependent launch.
constexpr int kDecodeWideHeads = 32;
bool decode_wide_tcgen05_supported(int kv_dtype, int head_dim, int block_size, int group,
                                   const void* q);
int decode_wide_tcgen05_heads(int group);
cudaError_t launch_decode_wide_tcgen05(const DecodeParams& p, int kv_dtype, const void* k_map,
                                       const void* v_map, int items, int sms,
                                       cudaStream_t stream);

// Tensor-core decode over beam groups: one CTA per (group, KV head, part),
// grid num_groups * num_kv_heads * p.max_partitions, the parts of one (group,
// KV head) adjacent.  Each shared-prefix K/V tile is read once for all members
// of the group; p.group_start / p.shared_tokens set.  With several parts, each
// takes an equal run of the group's 16-token stage list (shared prefix, then
// each member's tail) and the last to finish merges them (p.done zeroed).
constexpr int kMaxGroupParts = 64;
// wide: two n8 column tiles, members * G <= 16 (else one tile, <= 8).
cudaError_t launch_decode_grouped(const DecodeParams& p, int kv_dtype, const void* k_map,
                                  const void* v_map, long long grid, bool wide,
                                  cudaStream_t stream);

// Log-sum-exp merge of split partitions (only sequences with > 1 partition).
cudaError_t launch_lse_reduce(const DecodeParams& p, cudaStream_t stream);
