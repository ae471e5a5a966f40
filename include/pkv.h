/*
 * pkv.h -- C ABI of the GB300 paged KV-cache decode library (libpkv.so).
 *
 * The operations follow the method of "Efficient Memory Management for Large
 * Language Model Serving with PagedAttention" (Kwon et al., 2023) as the
 * following web pages describe it:
 *   [AIPP]  aiplusplus.yigather.com, "PagedAttention: bringing OS virtual
 *           memory to LLM inference"
 *   [AUT]   auturnal.com, "paged-attention serving guide" (v1)
 *   [CAY]   cayang0802.github.io, "Paged Attention" paper walkthrough
 *   [LAIN]  lain42.top reading journal on the paper
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every call returns an int status: PKV_OK (0) or a negative PKV_ERR_*.
 *   pkv_last_error_string() describes the most recent failure of the calling
 *   thread.  Argument errors are detected on the host before anything is
 *   launched; nothing is then written.
 * - Device calls take device pointers the CALLER owns (allocated by PyTorch or
 *   cudaMalloc).  The library never allocates or frees device memory.  Host
 *   allocator calls work on host memory only.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Device calls only enqueue work: they return once launched, and the output
 *   is ready when the stream reaches that point.
 * - Kernels check every block id, slot and context length they read against
 *   the sizes passed in.  A bad value is skipped (never dereferenced) and sets
 *   a bit in the device status word; pkv_device_status() reads it.
 * - dtype codes: PKV_F32, PKV_F16, PKV_BF16.  q, K and V share one dtype.
 * - The tensor-core decode kernels (pkv_paged_decode_attention, its
 *   allocation-free form, pkv_decode_step, pkv_paged_decode_grouped) are
 *   launched as programmatic dependents of the kernel before them on the
 *   stream.  When that kernel lets its dependents start early (this
 *   library's decode, work-plan and copy-on-write kernels do, as their CTAs
 *   start), the decode CTAs read context_lens, block_tables, group_start and
 *   shared_tokens while it still runs, and everything else only after it
 *   has completed.  No kernel of this library writes those four arrays; a
 *   kernel of the caller's that writes them must not let dependents start
 *   early (kernels that do not use programmatic launches never do).
 *
 * KV cache layout (the pages fix only that a block stores the K and V of B
 * consecutive tokens [AIPP core idea 1]; this layout is this library's
 * choice, made so one (block, head) tile is B*D contiguous elements):
 *     k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *     token i of a sequence lives in its logical block i / block_size, at
 *     offset i % block_size; block_tables[s][j] is the physical block of
 *     logical block j of sequence s [AIPP core idea 3].
 *     Both caches must start on a 16-byte boundary (tensor-memory-access
 *     tile loads); PKV_ERR_ALIGN otherwise.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define PKV_OK 0
#define PKV_ERR_NULL -1        /* a required pointer is NULL                  */
#define PKV_ERR_SHAPE -2       /* sizes out of range or inconsistent          */
#define PKV_ERR_DTYPE -3       /* unknown dtype code                          */
#define PKV_ERR_UNSUPPORTED -4 /* valid request the library does not implement */
#define PKV_ERR_CUDA -5        /* a CUDA runtime/driver call failed           */
#define PKV_ERR_BOUNDS -6      /* a kernel saw an out-of-range id (status)    */
#define PKV_ERR_OOM -7         /* allocator: not enough free blocks           */
#define PKV_ERR_WORKSPACE -8   /* workspace missing or too small              */
#define PKV_ERR_STATE -9       /* allocator: unknown / duplicate sequence     */
#define PKV_ERR_ALIGN -10      /* a pointer is not aligned as required        */

/* ---- dtypes -------------------------------------------------------------- */
#define PKV_F32 0
#define PKV_F16 1
#define PKV_BF16 2

/* ---- device status word bits (set by kernels, read by pkv_device_status) -- */
#define PKV_STATUS_BAD_BLOCK 1u  /* block-table entry outside [0, num_blocks)   */
#define PKV_STATUS_BAD_LEN 2u    /* context_len < 0 or > max_blocks*block_size  */
#define PKV_STATUS_BAD_SLOT 4u   /* slot >= num_blocks*block_size               */
#define PKV_STATUS_BAD_PAIR 8u   /* copy pair id outside [0, num_blocks)        */
#define PKV_STATUS_TIMEOUT 16u   /* a tile load did not arrive within ~1 s; the
                                    kernel stopped early (output invalid)       */

/* Text of the calling thread's most recent error ("" if none).  The pointer
 * stays valid until that thread's next failing call. */
const char* pkv_last_error_string(void);

/* Library ABI version (major * 100 + minor). */
int pkv_version(void);

/*
 * Reads (and, if reset != 0, clears) the device status word after waiting
 * for `stream`.  *bits receives the OR of PKV_STATUS_* seen since the last
 * reset on the current device.  Returns PKV_ERR_BOUNDS if any bit was set,
 * else PKV_OK.  This call synchronises the stream.
 */
int pkv_device_status(void* stream, uint32_t* bits, int reset);

/*
 * kv_write -- store each new token's K and V in its cache slot.
 * [CAY, KV-cache paragraph]: only the new token's key and value are computed
 * each step, the earlier ones are kept; [AIPP core idea 4 / LAIN on-demand
 * allocation]: the slot comes from a block allocated when the sequence grows.
 *
 * key, value   : [num_tokens][num_kv_heads][head_dim], dtype `dtype`.
 * slot_mapping : int64 [num_tokens]; slot = physical_block*block_size+offset.
 *                slot < 0 marks padding: that token is skipped.
 *                slot >= num_blocks*block_size is skipped and sets
 *                PKV_STATUS_BAD_SLOT.
 * k_cache, v_cache : cache arrays as laid out above; written in place.
 * Two tokens with the same slot race (either value may land).  Bit-exact copy.
 */
int pkv_kv_write(void* k_cache, void* v_cache, const void* key, const void* value,
                 const int64_t* slot_mapping, int num_tokens, int num_blocks,
                 int num_kv_heads, int head_dim, int block_size, int dtype, void* stream);

/*
 * paged_decode_attention -- one query token per sequence attends to that
 * sequence's cached tokens, which sit in fixed-size physical blocks reached
 * through the block table.  [AIPP key techniques 1]: the kernel follows the
 * block table to assemble scattered K/V blocks; [LAIN method]: table lookup,
 * block fetch and attention are fused in one kernel; [AUT section 1]: paging
 * changes storage, not what attention reads, so
 *     out[s,h,:] = sum_i softmax_i(scale * q[s,h,:] . K_s[i,g,:]) V_s[i,g,:]
 * over i < context_lens[s], with KV head g = h / (num_heads / num_kv_heads)
 * (grouped-query attention, [AUT section 1]: GQA/MQA change the KV head count).
 *
 * out          : [num_seqs][num_heads][head_dim], dtype out_dtype (written).
 *                Device memory, or pinned host memory that the GPU addresses
 *                directly (the same pointer): the launch then stores each
 *                output row over NVLink-C2C as its CTA finishes, and the
 *                stream's completion is the read-back, with no copy after it.
 *                The same holds for out and q of pkv_decode_step, of the
 *                allocation-free split form and of pkv_paged_decode_grouped.
 * q            : [num_seqs][num_heads][head_dim], dtype kv_dtype; device
 *                memory or pinned host memory, like out (each CTA loads its
 *                rows once, after it has started its first K/V loads).
 * block_tables : int32 [num_seqs][max_blocks_per_seq]; only the first
 *                ceil(context_lens[s]/block_size) entries of row s are read.
 * context_lens : int32 [num_seqs], tokens attended (the token written this
 *                step included).  0 gives an all-zero output row.
 * scale        : softmax scale (usually 1/sqrt(head_dim)).
 * partition_size : 0 = each (sequence, KV head) is handled in one pass.
 *                > 0 = split-context decode: each sequence's tokens are cut
 *                into partitions of this many tokens (a multiple of
 *                block_size), each attended with its own softmax state (max,
 *                sum, unnormalised output), and the partitions are merged by
 *                log-sum-exp through `workspace`: inside the same launch on
 *                the tensor-core kernel (which first merges the up to four
 *                partitions one CTA holds, one per warp, and writes one
 *                partial per CTA), by a second kernel otherwise.  (The pages
 *                are silent on splitting; the merge is exact in real
 *                arithmetic.)  On the tensor-core kernel, batches of up to
 *                4096 sequences first get a work plan (a one-CTA kernel in
 *                place of zeroing the merge counters): the CTAs with work are
 *                listed longest sequence first, so that long items do not
 *                start last and empty grid slots do not interleave with
 *                work.  When every non-empty context has within 10 % the
 *                same number of stages, the plan instead cuts each context
 *                into the same number of equal runs of stages (at most its
 *                partitions, at most 64), the fewest whose CTAs fill their
 *                last wave of the GPU to 95 %: partition_size then bounds
 *                the split and sizes the workspace.  Neither the order nor
 *                the cut changes the result in real arithmetic.
 * workspace    : device scratch of at least pkv_decode_workspace_bytes(...)
 *                bytes, 256-byte aligned, when partition_size > 0.  With
 *                partition_size == 0 it is optional: NULL attends the
 *                sequences in the caller's order; a workspace of
 *                pkv_decode_workspace_bytes(..., 0) bytes gets the unsplit
 *                launch a work plan too (longest sequence first), which
 *                keeps ragged batches from ending on a long sequence that
 *                started late.  Contents on entry are ignored; calls that
 *                share a workspace must not overlap on the GPU.
 * Supported: block_size in {8,16,32}; head_dim in {64,128}; num_heads a
 * multiple of num_kv_heads; out_dtype any of the three.  16-bit KV with
 * G = num_heads/num_kv_heads <= 256 runs on the tensor-core kernel (one CTA
 * carries up to 16 query heads of a KV group; a wider group is cut into
 * ceil(G/16) head slices, each reading the group's K/V), the rest (fp32 KV)
 * on a CUDA-core kernel; both accumulate in fp32.
 */
int pkv_paged_decode_attention(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, float scale, int block_size,
                               int num_kv_heads, int num_seqs, int num_heads, int head_dim,
                               int max_blocks_per_seq, int num_blocks, int kv_dtype,
                               int out_dtype, int partition_size, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * decode_step -- one decode step of every sequence in one call: each
 * sequence's new token is appended to the cache and then attended to along
 * with everything before it.  Equivalent to pkv_kv_write of the new tokens
 * followed by pkv_paged_decode_attention ([CAY] KV-cache paragraph: each
 * step's K/V is stored, then every step attends over all cached tokens;
 * [AIPP core idea 3-4]: the token at position p of sequence s sits at slot
 * table[s][p / block_size] * block_size + p % block_size).
 *
 * new_k, new_v : [num_seqs][num_kv_heads][head_dim], dtype kv_dtype, 16-byte
 *                aligned: the new token of sequence s, written at position
 *                context_lens[s] - 1 (context_lens counts the new token; its
 *                block must already be in the table, e.g. from
 *                pkv_step_append).
 * k_cache, v_cache : written at those positions, read as in
 *                pkv_paged_decode_attention.
 * All other arguments, the workspace and the error behaviour are those of
 * pkv_paged_decode_attention.  A sequence whose table entry for the new
 * position is out of range gets no write and sets PKV_STATUS_BAD_BLOCK.
 * On the tensor-core kernel the write happens inside the attention launch
 * (by the CTA that reads that position); on the CUDA-core kernel a separate
 * append launch precedes the attention.
 */
int pkv_decode_step(void* out, const void* q, const void* new_k, const void* new_v,
                    void* k_cache, void* v_cache, const int32_t* block_tables,
                    const int32_t* context_lens, float scale, int block_size, int num_kv_heads,
                    int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq,
                    int num_blocks, int kv_dtype, int out_dtype, int partition_size,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * paged_decode_grouped -- decode attention (optionally a decode step, with
 * new_k/new_v) for groups of sequences that share a prefix of physical
 * blocks, as the beams of a beam search or the samples of one prompt do
 * ([CAY beam search]: the common logical blocks of the beams map to one
 * physical copy).  The result is exactly that of pkv_decode_step /
 * pkv_paged_decode_attention for every sequence; the shared blocks are only
 * read once per group instead of once per member.
 *
 * group_start   : int32 [num_groups + 1], device memory, non-decreasing:
 *                 group i is sequences group_start[i] .. group_start[i+1]-1
 *                 (consecutive), with 1 <= members and members * G <= 16
 *                 (G = num_heads / num_kv_heads).  A group outside these
 *                 bounds (or above 8 columns when the one-tile kernel was
 *                 chosen, see max_members) is skipped and sets
 *                 PKV_STATUS_BAD_LEN.  Sequences in no group are not
 *                 attended: their output rows (and, in a decode step, their
 *                 caches) are left as they were.
 * max_members   : an upper bound on any group's members, or 0 for
 *                 num_seqs - num_groups + 1.  When max_members * G <= 8 the
 *                 kernel carries the group's query heads as one n8 column
 *                 tile, else as two (twice the mma work per K/V byte).
 * shared_tokens : int32 [num_groups], device memory: the first
 *                 shared_tokens[i] positions of every member of group i lie
 *                 in the same physical blocks (same table entries), e.g. from
 *                 pkv_group_shared_tokens.  The kernel uses it rounded down
 *                 to a multiple of 16, at most every member's context (and,
 *                 in a decode step, short of every member's new token).
 * new_k, new_v  : NULL for attention only; else as in pkv_decode_step, each
 *                 new token in a block private to its sequence.
 * parts         : 0 or 1: one CTA streams a whole group for one KV head.
 *                 2 .. 64: a group's list of 16-token stages (its shared
 *                 prefix, then each member's own tail) is cut into `parts`
 *                 runs of equal length, one CTA each; each run writes (max,
 *                 sum, unnormalised output) per member query head to the
 *                 workspace and the last run to finish merges them by
 *                 log-sum-exp inside the same launch (the pages are silent on
 *                 splitting; the merge is exact in real arithmetic).  More
 *                 parts even out the waves when num_groups * num_kv_heads is
 *                 not a large multiple of the CTAs the GPU holds at once.
 * workspace     : device scratch when parts > 1 (else may be NULL): at least
 *                 pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim,
 *                 parts, 1) bytes, 256-byte aligned; contents on entry are
 *                 ignored; calls that share it must not overlap on the GPU.
 * Other arguments as in pkv_decode_step (no partition_size).  Needs the
 * tensor-core kernel: 16-bit KV, G <= 16, kernel choice PKV_KERNEL_AUTO (else
 * PKV_ERR_UNSUPPORTED).  A group is read by at most `parts` CTAs a KV head,
 * so with few groups and long contexts the split, ungrouped pkv_decode_step
 * can keep more of the GPU busy.
 * Like the other decode calls it is a programmatic dependent launch (see the
 * conventions above): after pkv_kv_copy_blocks its CTAs read the group
 * bounds, lengths and tables while the copies run.
 */
int pkv_paged_decode_grouped(void* out, const void* q, const void* new_k, const void* new_v,
                             void* k_cache, void* v_cache, const int32_t* block_tables,
                             const int32_t* context_lens, const int32_t* group_start,
                             const int32_t* shared_tokens, int num_groups, int max_members,
                             float scale, int block_size, int num_kv_heads, int num_seqs,
                             int num_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                             int kv_dtype, int out_dtype, int parts, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * group_shared_tokens -- host helper for pkv_paged_decode_grouped: for each
 * group, the number of leading positions whose table entries every member
 * holds in common (whole blocks), capped at the shortest member's context.
 * All pointers are host memory; block_tables is [num_seqs][max_blocks_per_seq].
 * A group outside [0, num_seqs) or empty gives PKV_ERR_SHAPE.
 */
int pkv_group_shared_tokens(const int32_t* block_tables, const int32_t* context_lens,
                            const int32_t* group_start, int num_groups, int num_seqs,
                            int max_blocks_per_seq, int block_size, int32_t* shared_tokens);

/*
 * paged_prefill_attention -- several new query tokens per sequence (a prompt,
 * or a chunk of one), each attending causally over the sequence's cached
 * tokens up to its own position.  [CAY recomputation]: a whole sequence's KV
 * can be produced in one parallel pass, the prefill that recomputing a
 * preempted sequence relies on; the attention itself is the one above
 * ([AIPP key techniques 1], [AUT section 1]) with a causal limit:
 *     out[r,h,:] = sum_{i <= L_s - qn_s + t} softmax_i(scale q[r,h,:] . K_s[i,g,:]) V_s[i,g,:]
 * for row r = query_start[s] + t, t < qn_s = query_start[s+1] - query_start[s].
 * The new tokens' K/V must already be in the cache (pkv_kv_write).
 *
 * q, out      : [rows][num_heads][head_dim], rows = query_start[num_seqs];
 *               q 16-byte aligned.
 * query_start : int32 [num_seqs + 1], non-decreasing, device memory.
 * max_query_len : >= every qn_s (sizes the grid).  A sequence with qn_s >
 *               max_query_len or qn_s > context_lens[s] is skipped and sets
 *               PKV_STATUS_BAD_LEN.
 * 16-bit KV only (PKV_ERR_UNSUPPORTED for fp32); head_dim in {64,128};
 * block_size in {8,16,32}; no workspace.
 */
int pkv_paged_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* query_start, float scale, int block_size,
                                int num_kv_heads, int num_seqs, int num_heads, int head_dim,
                                int max_blocks_per_seq, int num_blocks, int max_query_len,
                                int kv_dtype, int out_dtype, void* stream);

/* Workspace bytes pkv_paged_decode_attention needs for these sizes, where
 * max_context_len = max_blocks_per_seq * block_size.  With H = num_heads and
 * P = ceil(max_context_len / partition_size), each part 256-byte aligned:
 * merge counters (S*H u32), per-partition (max, sum) (S*H*P float2) and
 * unnormalised outputs (S*H*P*head_dim float), the work plan's record count
 * (256 bytes) and records (S*H*P * 16 bytes).  partition_size == 0: the
 * optional workspace of an unsplit call, the work plan alone (256 + S*H*16
 * bytes).  0 for bad sizes. */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                  int max_context_len, int partition_size);

/*
 * paged_decode_attention_noalloc -- the split-context decode above
 * (partition_size > 0 required) without a caller workspace.  The pages have
 * no counterpart to this call; it exists for callers that cannot allocate
 * device memory at all -- e.g. a plugin invoked from a host framework's
 * execute step that forbids allocation there, a serving loop whose memory is
 * carved up once at start-up by another allocator, or latency-critical code
 * that cannot pay for cudaMalloc's possible device-wide synchronisation.
 *
 * The partition scratch lives in a fixed array inside libpkv's own device
 * memory, PKV_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU, held by every GPU that
 * loads the library until the process exits.  Sizes whose scratch need
 * (pkv_decode_workspace_bytes) exceeds it are rejected with
 * PKV_ERR_WORKSPACE and a message giving both figures; nothing is launched.
 * The call allocates nothing: no cudaMalloc / cudaFree, no allocating
 * library routine.  Every call looks up the array's device address
 * (cudaGetSymbolAddress, which allocates nothing) with the caller's device
 * current, so a reset or another context never sees a stale address; the
 * first call on a device is its set-up (it may load the library's device
 * code there), so make that first call before any stream capture.  The
 * request is checked like pkv_paged_decode_attention's (same codes) before
 * the scratch limit is.  All calls on a device share the one
 * array, and it keeps the last call's contents (no clearing is needed: each
 * call writes every scratch slot it reads before reading it), so calls that
 * overlap on the GPU -- on different streams, or different threads -- race
 * and give wrong results.  Arguments and results are otherwise those of
 * pkv_paged_decode_attention.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
int pkv_paged_decode_attention_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, float scale, int block_size,
                                       int num_kv_heads, int num_seqs, int num_heads,
                                       int head_dim, int max_blocks_per_seq, int num_blocks,
                                       int kv_dtype, int out_dtype, int partition_size,
                                       void* stream);

/*
 * kv_copy_blocks -- copy-on-write copy of whole physical blocks.
 * [AUT section 3]: when a branch must modify a shared block that is not yet
 * full, copy-on-write keeps branches from overwriting each other; [AIPP key
 * techniques 3]: several block tables point at one physical block and a copy
 * is made only on write.
 *
 * pairs : int64 [num_pairs][2] device array of (src, dst) physical block ids.
 *         For every KV head, all block_size slots of K and V are copied.
 *         Destinations must be distinct and must not appear as a source in
 *         the same call (the copies run in parallel); an id outside
 *         [0, num_blocks) skips that pair and sets PKV_STATUS_BAD_PAIR.
 * Bit-exact copy.  The kernel lets a programmatic dependent launch that
 * follows it start at once (pkv_paged_decode_grouped is launched that way and
 * waits for the copy to complete before it reads or writes the caches).
 */
int pkv_kv_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                       int num_blocks, int num_kv_heads, int head_dim, int block_size,
                       int dtype, void* stream);

/*
 * kv_swap_blocks -- move whole blocks between two KV pools, for preemption by
 * swapping.  [AIPP section 4] / [CAY preemption]: when GPU memory runs out, a
 * sequence's KV blocks can be moved to CPU memory and brought back later
 * (small blocks make that transfer less efficient).  On GB300 a pinned host
 * pool (cudaHostAlloc, or memory the CPU allocated on a coherent Grace
 * system) is reached by the kernel directly over NVLink-C2C, so one launch
 * gathers or scatters any set of scattered blocks.
 *
 * dst_* / src_* : pools laid out like the cache ([blocks][num_kv_heads]
 *                 [block_size][head_dim]); each pointer may be device memory or
 *                 host memory the GPU can address; 16-byte aligned.
 * pairs : int64 [num_pairs][2] (src block, dst block), in memory the GPU can
 *         read.  Destinations must be distinct; an id out of range skips the
 *         pair and sets PKV_STATUS_BAD_PAIR.  For every KV head, all
 *         block_size slots of K and V are copied, bit-exact.
 */
int pkv_kv_swap_blocks(void* dst_k_cache, void* dst_v_cache, const void* src_k_cache,
                       const void* src_v_cache, const int64_t* pairs, int num_pairs,
                       int num_src_blocks, int num_dst_blocks, int num_kv_heads, int head_dim,
                       int block_size, int dtype, void* stream);

/*
 * selftest_bounded_wait -- exercises the bounded waits the kernels use.
 * Launches num_ctas CTAs (1..65535); each waits on an mbarrier that nothing
 * arrives on.  The first wait to reach its bound (about 2^31 cycles, about a
 * second) sets PKV_STATUS_TIMEOUT; the other CTAs see the bit and give up at
 * once.  Each CTA then completes its barrier itself and increments *drained
 * (a device uint32 the caller zeroes) if the drain wait -- the one a kernel
 * uses for its own copies after a timeout -- returns in bound.  Expect the
 * TIMEOUT bit set (reset it with pkv_device_status) and *drained == num_ctas;
 * the context stays usable.  Nothing faults or stays in flight.
 */
int pkv_selftest_bounded_wait(int num_ctas, unsigned int* drained, void* stream);

/*
 * Kernel selection for pkv_paged_decode_attention (process-wide):
 * PKV_KERNEL_AUTO (default) picks the tensor-core kernel where supported;
 * PKV_KERNEL_CUDA_CORE forces the CUDA-core kernel for every shape (used to
 * test both).  Returns PKV_ERR_SHAPE for an unknown value.
 */
#define PKV_KERNEL_AUTO 0
#define PKV_KERNEL_CUDA_CORE 1
int pkv_set_decode_kernel(int which);

/*
 * Kernel for unsplit decode of wide query-head groups (process-wide): with
 * G = num_heads / num_kv_heads a multiple of 32, head_dim 128, 16-bit KV,
 * block size 8, 16 or 32, q 16-byte aligned and partition_size 0 (outside
 * beam groups),
 * PKV_WIDE_TCGEN05 (default) runs the 5th-generation tensor-core kernel: a
 * K/V tile's 128 tokens are the MMA's M and 64 query heads (when G is a
 * multiple of 64, else 32) its N, one persistent CTA a SM, the work plan's
 * longest-first order when a workspace is given (pkv_decode_workspace_bytes
 * with partition_size 0; its bytes 0-4 and 64-68 are the plan's count and
 * the kernel's record counter).  Split launches (partition_size > 0) of such
 * groups run head slices.
 * PKV_WIDE_HEAD_SLICES runs the mma.sync kernel on head slices of 16 query
 * heads (also used for every other shape).  Both compute the same result up
 * to fp32 accumulation order.  With new_k / new_v (pkv_decode_step) the
 * tcgen05 path writes the new tokens in a kernel of its own first.  Returns
 * PKV_ERR_SHAPE for an unknown value.
 */
#define PKV_WIDE_TCGEN05 0
#define PKV_WIDE_HEAD_SLICES 1
int pkv_set_wide_group_kernel(int which);

/*
 * Kernel selection for pkv_paged_prefill_attention (process-wide):
 * PKV_PREFILL_TCGEN05 (default) runs the 5th-generation tensor-core kernel
 * (tcgen05 MMAs with S, P and O in tensor memory, 256 query rows per CTA,
 * warp-specialised); PKV_PREFILL_WARP_MMA runs the warp-level mma.sync
 * kernel (64 rows per CTA).  Both compute the same result up to fp32
 * accumulation order.  Returns PKV_ERR_SHAPE for an unknown value.
 */
#define PKV_PREFILL_TCGEN05 0
#define PKV_PREFILL_WARP_MMA 1
int pkv_set_prefill_kernel(int which);

/* ==========================================================================
 * Host block allocator (host memory only; not thread-safe per handle).
 * [AIPP core idea 1-4, effects]: fixed-size blocks, a block table per
 * sequence, blocks allocated on demand and any free block serves;
 * [AIPP continuous batching]: a finished sequence frees its blocks at once;
 * [AUT section 3]: shared blocks carry a reference count that must match the
 * lifetime of the sequences using them, and a write into a shared block that
 * is not full copies it first; [AUT section 6]: OOM must be handled.
 *
 * Free list: a stack.  Blocks are first handed out in `free_order`
 * (identity if NULL); a block whose count drops to zero is pushed on top and
 * is handed out next.  A sequence releases its blocks last to first.
 * Any call that fails leaves the allocator unchanged.
 * ========================================================================== */
typedef struct pkv_allocator pkv_allocator;

/* free_order: NULL or a permutation of [0, num_blocks). */
int pkv_alloc_create(int num_blocks, int block_size, const int32_t* free_order,
                     pkv_allocator** out);
int pkv_alloc_destroy(pkv_allocator* a);

/* New sequence holding prompt_len tokens: takes ceil(prompt_len/B) blocks.
 * PKV_ERR_STATE if seq exists; PKV_ERR_OOM if too few free blocks. */
int pkv_seq_add(pkv_allocator* a, int64_t seq, int prompt_len);

/* Reserves the slot of the sequence's next token.  A fresh block is taken if
 * the token starts a block; if the last block is shared (count > 1) and not
 * full, a private copy target is taken instead: *cow_src/*cow_dst receive the
 * pair to pass to pkv_kv_copy_blocks before the write (else both are -1). */
int pkv_seq_append(pkv_allocator* a, int64_t seq, int64_t* slot, int64_t* cow_src,
                   int64_t* cow_dst);

/* One decode step: pkv_seq_append on each of seqs[0..n) in order, all or
 * nothing.  slots: [n]; cow_pairs: [n][2] capacity; *num_pairs = pairs made. */
int pkv_step_append(pkv_allocator* a, const int64_t* seqs, int n, int64_t* slots,
                    int64_t* cow_pairs, int* num_pairs);

/* The same step, keeping a dense batch table current in place: on entry
 * tables [n][max_blocks] and lens [n] hold sequence seqs[i]'s table and
 * length from before the step (from pkv_block_tables_dense, or from the
 * previous step's call with the same seqs); the call writes only what the
 * step changes -- the entry of each new token's block (a fresh block, or the
 * copy that replaced a shared one) and lens[i] + 1 -- so a serving loop can
 * keep the tables in the pinned buffer it copies to the device, with no
 * dense read-back each step.  Entries past a sequence's table are left as
 * they are.  All or nothing: PKV_ERR_SHAPE (nothing changed) if a table would
 * grow past max_blocks, PKV_ERR_STATE if a sequence is listed twice;
 * otherwise as pkv_step_append.  The step's plan lives in the allocator's
 * per-sequence and per-block scratch: a step call allocates host memory only
 * when it takes more sequences than any step before it, or when a sequence's
 * block list outgrows its capacity (amortised, once per doubling).  The time
 * is a hash lookup and a few comparisons per sequence. */
int pkv_step_append_tables(pkv_allocator* a, const int64_t* seqs, int n, int64_t* slots,
                           int64_t* cow_pairs, int* num_pairs, int32_t* tables, int max_blocks,
                           int32_t* lens);

/* child shares every block of parent (each count + 1).  PKV_ERR_STATE if the
 * parent is unknown or the child exists. */
int pkv_seq_fork(pkv_allocator* a, int64_t parent, int64_t child);

/* Drops the sequence; blocks whose count reaches zero return to the pool. */
int pkv_seq_free(pkv_allocator* a, int64_t seq);

/* Moves a sequence from allocator `from` to allocator `to` (same block size),
 * e.g. from the device pool to a host swap pool and back ([AIPP section 4],
 * [CAY preemption]): takes one fresh block of `to` per block of the sequence,
 * writes the (from block, to block) pairs in table order to pairs[0..2*n) for
 * pkv_kv_swap_blocks, then releases the sequence in `from` (blocks it shared
 * stay with their other users; the moved copy is private).  cap = pairs
 * capacity in pairs.  All or nothing: PKV_ERR_OOM if `to` lacks blocks,
 * PKV_ERR_SHAPE if cap is too small, PKV_ERR_STATE if seq is unknown in
 * `from` or already in `to`. */
int pkv_seq_swap(pkv_allocator* from, pkv_allocator* to, int64_t seq, int64_t* pairs, int cap,
                 int* num_pairs);

int pkv_seq_len(pkv_allocator* a, int64_t seq, int* len);

/* Copies the sequence's table into out[0..cap); *n = its length (may be > cap,
 * in which case only cap entries are written and PKV_ERR_SHAPE is returned). */
int pkv_block_table(pkv_allocator* a, int64_t seq, int32_t* out, int cap, int* n);

/* Dense tables for a batch: tables [n][max_blocks] (unused entries -1) and
 * lens [n].  PKV_ERR_SHAPE if a table is longer than max_blocks. */
int pkv_block_tables_dense(pkv_allocator* a, const int64_t* seqs, int n, int max_blocks,
                           int32_t* tables, int32_t* lens);

/* ---- automatic prefix caching ([CAY] prefix caching: each full block is
 * keyed by a hash of its own tokens and all preceding tokens; blocks with the
 * same key hold the same KV and are reused instead of recomputed).
 * Key of full block i: FNV-1a 64-bit over the key of block i-1 (0 for i = 0)
 * as 8 little-endian bytes, then the block's block_size token ids as 4
 * little-endian bytes each.  A hit is confirmed against the stored parent key
 * and token ids, so a hash collision cannot alias two different blocks.
 * A registered block whose count drops to zero stays findable in a
 * least-recently-freed list; it is handed out again (and unregistered) only
 * once the plain free list is empty.  Free-block counts include it. */

/* New sequence for the prompt tokens[0..n): reuses the cached blocks of the
 * longest prefix of full blocks found in the index, takes fresh blocks for
 * the rest.  *reused_tokens = tokens covered by reused blocks (a multiple of
 * block_size): their K/V is already in the cache; the caller writes the
 * remaining ones.  Errors as pkv_seq_add. */
int pkv_seq_add_cached(pkv_allocator* a, int64_t seq, const int32_t* tokens, int n,
                       int* reused_tokens);

/* Registers the full blocks covering tokens[0..n) of a sequence (n <= its
 * length; call once their K/V has been written).  Blocks already registered,
 * or whose key is already in the index, are skipped; *registered = blocks
 * added. */
int pkv_seq_register_blocks(pkv_allocator* a, int64_t seq, const int32_t* tokens, int n,
                            int* registered);

/* Blocks reused by pkv_seq_add_cached so far, blocks in the index, and
 * registered blocks currently unused (count 0). */
int pkv_prefix_cache_stats(pkv_allocator* a, int64_t* hit_blocks, int64_t* cached_blocks,
                           int64_t* cached_free_blocks);

int pkv_refcount(pkv_allocator* a, int block, int* count);
int pkv_num_free_blocks(pkv_allocator* a, int* n);

/* Eq. (2)-(3) of [AUT]: allocated positions = sum over sequences of
 * B * blocks held, valid positions = sum of lengths (position utilisation
 * U = valid / allocated); blocks_in_use counts physical blocks once. */
int pkv_stats(pkv_allocator* a, int64_t* allocated_positions, int64_t* valid_positions,
              int64_t* blocks_in_use);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
