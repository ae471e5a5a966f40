// C-ABI entry points of libpkv (declared in include/pkv.h): argument checks,
// workspace carving, TMA tensor maps and kernel selection.  All arithmetic of
// the path runs in the kernels (kernels_basic.cu, decode_tc.cu).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"
#include "pkv_kernels.h"

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
namespace {
thread_local char g_err[512] = "";
int g_decode_kernel = PKV_KERNEL_AUTO;
int g_prefill_kernel = PKV_PREFILL_TCGEN05;
int g_wide_kernel = PKV_WIDE_TCGEN05;
}  // namespace

int pkv_fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

static int cuda_fail(cudaError_t e, const char* where)
{
    return pkv_fail(PKV_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------------------
// TMA tensor maps: a cache viewed as [NB*Hkv*B rows][D columns] of 16-bit
// elements, loaded in boxes of 64 columns x min(B, 16) rows with the 128-byte
// swizzle.
// Encoded maps are cached by (address, rows, D, B, dtype).
// ---------------------------------------------------------------------------
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct MapEntry {
    const void* ptr = nullptr;
    uint64_t rows = 0;
    int D = 0, box_rows = 0, dtype = -1, halves = 0;
    CUtensorMap map;
};

std::mutex g_map_mu;
MapEntry g_maps[16];
int g_map_next = 0;
EncodeTiledFn g_encode = nullptr;

int get_encoder()
{
    if (g_encode) return PKV_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return pkv_fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return PKV_OK;
}

// A cache viewed as [rows][D] bf16/fp16, loaded in boxes of 64 columns x
// box_rows rows with the 128-byte swizzle.  halves = 0: a 2-D map, one box
// per 64-column half.  halves = 1: a 3-D map whose outermost dimension steps
// over the 64-column halves (stride 128 bytes), so that one box brings every
// half of box_rows rows, laid out half after half in shared memory.
// halves = 2: a 4-D map over [row group of 8][half][row in group][64 columns]
// (strides 8 rows, 128 bytes, one row), so that one box brings box_rows rows
// (a multiple of 8) of every half as 1024-byte swizzle atoms, row group by
// row group, each group's halves side by side.
int tensor_map(const void* cache, uint64_t rows, int D, int box_rows, int dtype, CUtensorMap* out,
               int halves = 0)
{
    if (halves == 2 && (rows % 8 != 0 || box_rows % 8 != 0))
        return pkv_fail(PKV_ERR_SHAPE, "row-group tensor map: rows %llu, box %d not multiples of 8",
                        (unsigned long long)rows, box_rows);
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (const MapEntry& m : g_maps) {
        if (m.ptr == cache && m.rows == rows && m.D == D && m.box_rows == box_rows &&
            m.dtype == dtype && m.halves == halves) {
            *out = m.map;
            return PKV_OK;
        }
    }
    int rc = get_encoder();
    if (rc != PKV_OK) return rc;
    MapEntry& m = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % 16;
    const cuuint64_t pitch = (cuuint64_t)D * 2;
    cuuint64_t dims[4] = {(cuuint64_t)(halves ? 64 : D), (cuuint64_t)rows, (cuuint64_t)(D / 64), 1};
    cuuint64_t strides[3] = {pitch, 128, 0};
    cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)(D / 64), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (halves == 2) {
        dims[1] = 8;
        dims[3] = rows / 8;
        strides[2] = 8 * pitch;
        box[1] = 8;
        box[3] = (cuuint32_t)(box_rows / 8);
    }
    const cuuint32_t rank = halves == 2 ? 4 : halves ? 3 : 2;
    CUresult r = g_encode(&m.map,
                          dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          rank, const_cast<void*>(cache), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        m.ptr = nullptr;
        return pkv_fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    m.ptr = cache;
    m.rows = rows;
    m.D = D;
    m.box_rows = box_rows;
    m.dtype = dtype;
    m.halves = halves;
    *out = m.map;
    return PKV_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split workspace, in order (each part 256-byte aligned):
//   done  : u32 [S][H]           partitions finished per (sequence, KV head)
//   ml    : float2 [S][H][P]     per-partition (max, sum), base 2
//   o     : float [S][H][P][D]   per-partition unnormalised output
//   count : int                  work records in the plan
//   items : int4 [S][H][P]       the plan's records, one per CTA with work
// with H the number of query heads (an upper bound for the KV heads times
// the head slices, so S*H*P bounds every split launch's grid).
struct WorkspaceLayout {
    size_t ml, o, count, items, total;
};

// Optional workspace of an unsplit launch: the work plan alone (record
// count, then one record per (sequence, KV head x head slice)).
// Optional workspace of an unsplit launch: the plan's record count at byte 0,
// the wide-group kernel's record counter at byte 64, records from byte 256.
size_t plan_bytes(size_t S, size_t H) { return 256 + S * H * 16; }
constexpr size_t kPlanNextOffset = 64;

WorkspaceLayout workspace_layout(size_t S, size_t H, size_t P, size_t D)
{
    WorkspaceLayout w;
    w.ml = align256(S * H * sizeof(unsigned));
    w.o = w.ml + align256(S * H * P * sizeof(float2));
    w.count = w.o + align256(S * H * P * D * sizeof(float));
    w.items = w.count + 256;
    w.total = w.items + S * H * P * 16;
    return w;
}

}  // namespace

extern "C" {

const char* pkv_last_error_string(void) { return g_err; }

int pkv_version(void) { return 100; }

int pkv_set_decode_kernel(int which)
{
    if (which != PKV_KERNEL_AUTO && which != PKV_KERNEL_CUDA_CORE)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_set_decode_kernel: unknown value %d", which);
    g_decode_kernel = which;
    return PKV_OK;
}

int pkv_set_wide_group_kernel(int which)
{
    if (which != PKV_WIDE_TCGEN05 && which != PKV_WIDE_HEAD_SLICES)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_set_wide_group_kernel: unknown value %d", which);
    g_wide_kernel = which;
    return PKV_OK;
}

int pkv_set_prefill_kernel(int which)
{
    if (which != PKV_PREFILL_TCGEN05 && which != PKV_PREFILL_WARP_MMA)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_set_prefill_kernel: unknown value %d", which);
    g_prefill_kernel = which;
    return PKV_OK;
}

int pkv_device_status(void* stream, uint32_t* bits, int reset)
{
    if (!bits) return pkv_fail(PKV_ERR_NULL, "pkv_device_status: bits is NULL");
    unsigned int* word = pkv_status_word_ptr();
    if (!word) return pkv_fail(PKV_ERR_CUDA, "pkv_device_status: no device status word");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && reset) e = cudaMemsetAsync(word, 0, sizeof(unsigned int), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_device_status");
    *bits = host;
    if (host) return pkv_fail(PKV_ERR_BOUNDS, "device status bits 0x%x", host);
    return PKV_OK;
}

int pkv_kv_write(void* k_cache, void* v_cache, const void* key, const void* value,
                 const int64_t* slot_mapping, int num_tokens, int num_blocks, int num_kv_heads,
                 int head_dim, int block_size, int dtype, void* stream)
{
    const int eb = pkv_dtype_bytes(dtype);
    if (!eb) return pkv_fail(PKV_ERR_DTYPE, "pkv_kv_write: dtype %d", dtype);
    if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_kv_write: bad sizes");
    if ((head_dim * eb) % 16 != 0)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_kv_write: head_dim*elem_bytes must be a multiple of 16");
    if (num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !key || !value || !slot_mapping)
        return pkv_fail(PKV_ERR_NULL, "pkv_kv_write: NULL pointer");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(key, 16) || !aligned(value, 16))
        return pkv_fail(PKV_ERR_ALIGN, "pkv_kv_write: caches, key and value need 16-byte alignment");
    unsigned int* status = pkv_status_word_ptr();
    if (!status) return pkv_fail(PKV_ERR_CUDA, "pkv_kv_write: no device status word");
    cudaError_t e = launch_kv_write(k_cache, v_cache, key, value, slot_mapping, num_tokens,
                                    num_blocks, num_kv_heads, head_dim, block_size, eb, status,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "pkv_kv_write launch");
}

int pkv_kv_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                       int num_blocks, int num_kv_heads, int head_dim, int block_size, int dtype,
                       void* stream)
{
    const int eb = pkv_dtype_bytes(dtype);
    if (!eb) return pkv_fail(PKV_ERR_DTYPE, "pkv_kv_copy_blocks: dtype %d", dtype);
    if (num_pairs < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_kv_copy_blocks: bad sizes");
    const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * eb;
    if (block_bytes % 16 != 0)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_kv_copy_blocks: block bytes must be a multiple of 16");
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !pairs) return pkv_fail(PKV_ERR_NULL, "pkv_kv_copy_blocks: NULL");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(pairs, 8))
        return pkv_fail(PKV_ERR_ALIGN, "pkv_kv_copy_blocks: misaligned pointer");
    unsigned int* status = pkv_status_word_ptr();
    if (!status) return pkv_fail(PKV_ERR_CUDA, "pkv_kv_copy_blocks: no device status word");
    cudaError_t e = launch_kv_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_blocks,
                                          block_bytes, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "pkv_kv_copy_blocks launch");
}

int pkv_kv_swap_blocks(void* dst_k_cache, void* dst_v_cache, const void* src_k_cache,
                       const void* src_v_cache, const int64_t* pairs, int num_pairs,
                       int num_src_blocks, int num_dst_blocks, int num_kv_heads, int head_dim,
                       int block_size, int dtype, void* stream)
{
    const int eb = pkv_dtype_bytes(dtype);
    if (!eb) return pkv_fail(PKV_ERR_DTYPE, "pkv_kv_swap_blocks: dtype %d", dtype);
    if (num_pairs < 0 || num_src_blocks < 0 || num_dst_blocks < 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_kv_swap_blocks: bad sizes");
    const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * eb;
    if (block_bytes % 16 != 0)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_kv_swap_blocks: block bytes must be a multiple of 16");
    if (num_pairs == 0) return PKV_OK;
    if (!dst_k_cache || !dst_v_cache || !src_k_cache || !src_v_cache || !pairs)
        return pkv_fail(PKV_ERR_NULL, "pkv_kv_swap_blocks: NULL pointer");
    if (!aligned(dst_k_cache, 16) || !aligned(dst_v_cache, 16) || !aligned(src_k_cache, 16) ||
        !aligned(src_v_cache, 16) || !aligned(pairs, 8))
        return pkv_fail(PKV_ERR_ALIGN, "pkv_kv_swap_blocks: misaligned pointer");
    unsigned int* status = pkv_status_word_ptr();
    if (!status) return pkv_fail(PKV_ERR_CUDA, "pkv_kv_swap_blocks: no device status word");
    cudaError_t e = launch_kv_swap_blocks(dst_k_cache, dst_v_cache, src_k_cache, src_v_cache,
                                          pairs, num_pairs, num_src_blocks, num_dst_blocks,
                                          block_bytes, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "pkv_kv_swap_blocks launch");
}

int pkv_paged_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* query_start, float scale, int block_size,
                                int num_kv_heads, int num_seqs, int num_heads, int head_dim,
                                int max_blocks_per_seq, int num_blocks, int max_query_len,
                                int kv_dtype, int out_dtype, void* stream)
{
    static const char* fn = "pkv_paged_prefill_attention";
    if (!pkv_dtype_bytes(kv_dtype) || !pkv_dtype_bytes(out_dtype))
        return pkv_fail(PKV_ERR_DTYPE, "%s: dtype kv=%d out=%d", fn, kv_dtype, out_dtype);
    if (kv_dtype == PKV_F32)
        return pkv_fail(PKV_ERR_UNSUPPORTED, "%s: fp32 KV is not supported (16-bit only)", fn);
    if (num_seqs < 0 || num_seqs > 65535)
        return pkv_fail(PKV_ERR_SHAPE, "%s: num_seqs %d outside [0, 65535]", fn, num_seqs);
    if (head_dim != 64 && head_dim != 128)
        return pkv_fail(PKV_ERR_SHAPE, "%s: head_dim %d not in {64,128}", fn, head_dim);
    if (block_size != 8 && block_size != 16 && block_size != 32)
        return pkv_fail(PKV_ERR_SHAPE, "%s: block_size %d not in {8,16,32}", fn, block_size);
    if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads != 0 ||
        num_heads > 65535)
        return pkv_fail(PKV_ERR_SHAPE, "%s: num_heads %d / num_kv_heads %d", fn, num_heads,
                        num_kv_heads);
    if (max_blocks_per_seq <= 0 || num_blocks <= 0 || max_query_len < 0)
        return pkv_fail(PKV_ERR_SHAPE, "%s: bad sizes", fn);
    if ((int64_t)max_blocks_per_seq * block_size > (1ll << 30))
        return pkv_fail(PKV_ERR_SHAPE, "%s: max context too long", fn);
    if ((int64_t)num_blocks * num_kv_heads * block_size >= (1ll << 31))
        return pkv_fail(PKV_ERR_SHAPE, "%s: cache has >= 2^31 rows", fn);
    if (!std::isfinite(scale)) return pkv_fail(PKV_ERR_SHAPE, "%s: scale is not finite", fn);
    if (num_seqs == 0 || max_query_len == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
        return pkv_fail(PKV_ERR_NULL, "%s: NULL pointer", fn);
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) ||
        !aligned(out, pkv_dtype_bytes(out_dtype)))
        return pkv_fail(PKV_ERR_ALIGN, "%s: caches and q need 16-byte alignment", fn);
    PrefillParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start = query_start;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.block_size = block_size;
    p.num_kv_heads = num_kv_heads;
    p.num_heads = num_heads;
    p.head_dim = head_dim;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.max_query_len = max_query_len;
    p.out_dtype = out_dtype;
    p.status = pkv_status_word_ptr();
    if (!p.status) return pkv_fail(PKV_ERR_CUDA, "%s: no device status word", fn);
    CUtensorMap kmap, vmap;
    const uint64_t rows = (uint64_t)num_blocks * num_kv_heads * block_size;
    // the tcgen05 kernel's boxes are 16-token groups (or one block of 8) of
    // both column halves in 8-row groups; the warp-MMA kernel's are per half
    const int box_rows = block_size < 16 ? block_size : 16;
    const int halves = g_prefill_kernel == PKV_PREFILL_WARP_MMA ? 0 : 2;
    int rc = tensor_map(k_cache, rows, head_dim, box_rows, kv_dtype, &kmap, halves);
    if (rc == PKV_OK) rc = tensor_map(v_cache, rows, head_dim, box_rows, kv_dtype, &vmap, halves);
    if (rc != PKV_OK) return rc;
    cudaError_t e =
        g_prefill_kernel == PKV_PREFILL_WARP_MMA
            ? launch_prefill_tensor_core(p, kv_dtype, &kmap, &vmap,
                                         static_cast<cudaStream_t>(stream))
            : launch_prefill_tcgen05(p, kv_dtype, &kmap, &vmap, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "pkv_paged_prefill_attention launch");
}

size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                  int partition_size)
{
    if (partition_size < 0 || num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 ||
        max_context_len <= 0)
        return 0;
    if (partition_size == 0) return plan_bytes(num_seqs, num_heads);
    const size_t P = ((size_t)max_context_len + partition_size - 1) / partition_size;
    return workspace_layout(num_seqs, num_heads, P, head_dim).total;
}

}  // extern "C"

// Checks of a decode request's dtypes and sizes that need no pointer (shared
// by every decode entry point, so that they report the same codes).
int pkv_decode_check(const char* fn, int kv_dtype, int out_dtype, int num_seqs, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                     int num_blocks, int partition_size, float scale)
{
    if (!pkv_dtype_bytes(kv_dtype) || !pkv_dtype_bytes(out_dtype))
        return pkv_fail(PKV_ERR_DTYPE, "%s: dtype kv=%d out=%d", fn, kv_dtype, out_dtype);
    if (num_seqs < 0 || num_seqs > 65535)
        return pkv_fail(PKV_ERR_SHAPE, "%s: num_seqs %d outside [0, 65535]", fn, num_seqs);
    if (head_dim != 64 && head_dim != 128)
        return pkv_fail(PKV_ERR_SHAPE, "%s: head_dim %d not in {64,128}", fn, head_dim);
    if (block_size != 8 && block_size != 16 && block_size != 32)
        return pkv_fail(PKV_ERR_SHAPE, "%s: block_size %d not in {8,16,32}", fn, block_size);
    if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads != 0 ||
        num_heads > 65535)
        return pkv_fail(PKV_ERR_SHAPE, "%s: num_heads %d / num_kv_heads %d", fn, num_heads,
                        num_kv_heads);
    if (max_blocks_per_seq <= 0 || num_blocks <= 0)
        return pkv_fail(PKV_ERR_SHAPE, "%s: max_blocks_per_seq %d, num_blocks %d", fn,
                        max_blocks_per_seq, num_blocks);
    if ((int64_t)max_blocks_per_seq * block_size > (1ll << 30))
        return pkv_fail(PKV_ERR_SHAPE, "%s: max context too long", fn);
    if ((int64_t)num_blocks * num_kv_heads * block_size >= (1ll << 31))
        return pkv_fail(PKV_ERR_SHAPE, "%s: cache has >= 2^31 rows", fn);
    if (partition_size < 0 || (partition_size > 0 && partition_size % block_size != 0))
        return pkv_fail(PKV_ERR_SHAPE, "%s: partition_size %d must be 0 or a multiple of %d", fn,
                        partition_size, block_size);
    if (!std::isfinite(scale)) return pkv_fail(PKV_ERR_SHAPE, "%s: scale is not finite", fn);
    return PKV_OK;
}

namespace {

int sm_count_of_device()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 0;
    return sms;
}

// Unsplit decode of groups of 32 k query heads on the tcgen05 kernel: the
// step's append first (its own kernel), then the plan when a workspace came
// with the call (records longest first, the kernel's counter zeroed), then
// the persistent kernel.
int decode_wide(const char* fn, DecodeParams& p, int kv_dtype, const void* k_cache,
                const void* v_cache, const void* new_k, const void* new_v, int* plan_count,
                int4* plan_items, cudaStream_t st)
{
    const int G = p.num_heads / p.num_kv_heads;
    p.head_slices = G / decode_wide_tcgen05_heads(G);
    CUtensorMap kmap, vmap;
    const uint64_t rows = (uint64_t)p.num_blocks * p.num_kv_heads * p.block_size;
    const int box_rows = p.block_size < 16 ? p.block_size : 16;
    // K in boxes of both halves by 8-row groups (its S MMA layout), V in boxes
    // of both halves (its P V layout)
    int rc = tensor_map(k_cache, rows, p.head_dim, box_rows, kv_dtype, &kmap, 2);
    if (rc == PKV_OK) rc = tensor_map(v_cache, rows, p.head_dim, box_rows, kv_dtype, &vmap, 1);
    if (rc != PKV_OK) return rc;
    const long long items = (long long)p.num_seqs * p.num_kv_heads * p.head_slices;
    if (items >= (1ll << 31)) return pkv_fail(PKV_ERR_SHAPE, "%s: more than 2^31 work items", fn);
    cudaError_t e;
    if (new_k != nullptr) {
        e = launch_kv_append(const_cast<void*>(k_cache), const_cast<void*>(v_cache), new_k, new_v,
                             p.block_tables, p.context_lens, p.num_seqs, p.max_blocks,
                             p.num_blocks, p.num_kv_heads, p.head_dim, p.block_size,
                             pkv_dtype_bytes(kv_dtype), p.status, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    const int sms = sm_count_of_device();
    if (plan_items != nullptr && p.num_seqs <= kPlanMaxSeqs) {
        int* next = reinterpret_cast<int*>(reinterpret_cast<char*>(plan_count) + kPlanNextOffset);
        DecodePlanParams pp;
        pp.context_lens = p.context_lens;
        pp.num_seqs = p.num_seqs;
        pp.num_kv_heads = p.num_kv_heads;
        pp.head_slices = p.head_slices;
        pp.partition_tokens = p.partition_tokens;
        pp.cta_parts = 1;
        pp.stage_tokens = 128;
        pp.slots = 0;
        pp.max_groups = 1;
        pp.max_len = p.max_blocks * p.block_size;
        int shift = 0;
        while ((pp.max_len >> shift) >= kPlanBuckets) ++shift;
        pp.bucket_shift = shift;
        pp.items = plan_items;
        pp.item_count = plan_count;
        pp.done = reinterpret_cast<unsigned*>(next);
        pp.num_counters = 1;
        e = launch_decode_plan(pp, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        p.items = plan_items;
        p.item_count = plan_count;
        p.item_next = next;
    }
    e = launch_decode_wide_tcgen05(p, kv_dtype, &kmap, &vmap, (int)items, sms > 0 ? sms : 148,
                                   st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return PKV_OK;
}

// Decode attention, optionally with the step's append fused in (new_k and
// new_v non-NULL: each sequence's new token goes to position
// context_lens[s]-1 first).
int decode_impl(const char* fn, void* out, const void* q, const void* k_cache,
                const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                float scale, int block_size, int num_kv_heads, int num_seqs, int num_heads,
                int head_dim, int max_blocks_per_seq, int num_blocks, int kv_dtype, int out_dtype,
                int partition_size, void* workspace, size_t workspace_bytes, void* stream,
                const void* new_k, const void* new_v, const int32_t* group_start = nullptr,
                const int32_t* shared_tokens = nullptr, int num_groups = 0, int group_parts = 1,
                int max_members = 0)
{
    const int chk = pkv_decode_check(fn, kv_dtype, out_dtype, num_seqs, num_heads, num_kv_heads,
                                     head_dim, block_size, max_blocks_per_seq, num_blocks,
                                     partition_size, scale);
    if (chk != PKV_OK) return chk;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return pkv_fail(PKV_ERR_NULL, "%s: NULL pointer", fn);
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) ||
        !aligned(out, pkv_dtype_bytes(out_dtype)))
        return pkv_fail(PKV_ERR_ALIGN, "%s: caches need 16-byte, q 4-byte alignment", fn);
    const bool append = new_k != nullptr;
    if (append && (!new_v || !aligned(new_k, 16) || !aligned(new_v, 16)))
        return pkv_fail(new_v ? PKV_ERR_ALIGN : PKV_ERR_NULL,
                        "%s: new_k and new_v need 16-byte alignment", fn);
    const bool grouped = group_start != nullptr;
    if (grouped) {
        if (!shared_tokens) return pkv_fail(PKV_ERR_NULL, "%s: NULL shared_tokens", fn);
        if (num_groups < 1 || num_groups > num_seqs)
            return pkv_fail(PKV_ERR_SHAPE, "%s: num_groups %d outside [1, %d]", fn, num_groups,
                            num_seqs);
        if (partition_size != 0)
            return pkv_fail(PKV_ERR_UNSUPPORTED, "%s: beam groups split by parts, not tokens", fn);
        if (group_parts < 1 || group_parts > kMaxGroupParts)
            return pkv_fail(PKV_ERR_SHAPE, "%s: parts %d outside [1, %d]", fn, group_parts,
                            kMaxGroupParts);
        if (kv_dtype == PKV_F32 || num_heads / num_kv_heads > kDecodeTcMaxColumns ||
            g_decode_kernel != PKV_KERNEL_AUTO)
            return pkv_fail(PKV_ERR_UNSUPPORTED,
                            "%s: beam groups need the tensor-core kernel (16-bit KV, G <= 16)",
                            fn);
        if (max_members < 0)
            return pkv_fail(PKV_ERR_SHAPE, "%s: max_members %d < 0", fn, max_members);
        if ((int64_t)num_groups * num_kv_heads * group_parts >= (1ll << 31))
            return pkv_fail(PKV_ERR_SHAPE, "%s: more than 2^31 work items", fn);
    }

    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    p.block_size = block_size;
    p.num_kv_heads = num_kv_heads;
    p.num_heads = num_heads;
    p.head_dim = head_dim;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.out_dtype = out_dtype;
    p.ws_ml = nullptr;
    p.ws_o = nullptr;
    p.done = nullptr;
    p.new_k = nullptr;
    p.new_v = nullptr;
    p.group_start = nullptr;
    p.shared_tokens = nullptr;
    p.num_groups = 0;
    p.items = nullptr;
    p.item_count = nullptr;
    p.item_next = nullptr;
    int* plan_count = nullptr;
    int4* plan_items = nullptr;
    const int max_ctx = max_blocks_per_seq * block_size;
    p.cta_parts = 1;
    p.head_slices = 1;
    if (partition_size == 0 && (!grouped || group_parts == 1)) {
        p.partition_tokens = max_ctx;
        p.max_partitions = 1;
        if (!grouped && workspace != nullptr) {
            // optional: a work plan orders the launch longest sequence first
            const size_t need = plan_bytes(num_seqs, num_heads);
            if (workspace_bytes < need)
                return pkv_fail(PKV_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given",
                                fn, need, workspace_bytes);
            if (!aligned(workspace, 256))
                return pkv_fail(PKV_ERR_ALIGN, "%s: workspace needs 256-byte alignment", fn);
            plan_count = static_cast<int*>(workspace);
            plan_items = reinterpret_cast<int4*>(static_cast<char*>(workspace) + 256);
        }
    } else {
        // token partitions, or (beam groups) parts of each group's stage list
        p.partition_tokens = grouped ? max_ctx : partition_size;
        p.max_partitions =
            grouped ? group_parts : (max_ctx + partition_size - 1) / partition_size;
        const size_t need =
            grouped ? pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, group_parts, 1)
                    : pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_ctx,
                                                 partition_size);
        if (!workspace || workspace_bytes < need)
            return pkv_fail(PKV_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn,
                            need, workspace ? workspace_bytes : (size_t)0);
        if (!aligned(workspace, 256))
            return pkv_fail(PKV_ERR_ALIGN, "%s: workspace needs 256-byte alignment", fn);
        if ((int64_t)p.max_partitions * num_heads >= (1ll << 31))
            return pkv_fail(PKV_ERR_SHAPE, "%s: too many partitions", fn);
        const WorkspaceLayout L = workspace_layout(num_seqs, num_heads, p.max_partitions, head_dim);
        char* base = static_cast<char*>(workspace);
        p.done = reinterpret_cast<unsigned*>(base);
        p.ws_ml = reinterpret_cast<float2*>(base + L.ml);
        p.ws_o = reinterpret_cast<float*>(base + L.o);
        plan_count = reinterpret_cast<int*>(base + L.count);
        plan_items = reinterpret_cast<int4*>(base + L.items);
    }
    p.status = pkv_status_word_ptr();
    if (!p.status) return pkv_fail(PKV_ERR_CUDA, "%s: no device status word", fn);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int G = num_heads / num_kv_heads;
    // wider KV groups are cut into head slices of <= 16 columns (each slice
    // reads the group's K/V; adjacent in the grid, the repeats meet in L2)
    const bool tensor_core =
        g_decode_kernel == PKV_KERNEL_AUTO && kv_dtype != PKV_F32 && G <= 256;
    cudaError_t e;
    if (tensor_core) {
        CUtensorMap kmap, vmap;
        const uint64_t rows = (uint64_t)num_blocks * num_kv_heads * block_size;
        const int box_rows = decode_box_rows(head_dim, block_size, grouped);
        int rc = tensor_map(k_cache, rows, head_dim, box_rows, kv_dtype, &kmap, 1);
        if (rc == PKV_OK) rc = tensor_map(v_cache, rows, head_dim, box_rows, kv_dtype, &vmap, 1);
        if (rc != PKV_OK) return rc;
        if (!grouped && p.max_partitions <= 1 && g_wide_kernel == PKV_WIDE_TCGEN05 &&
            decode_wide_tcgen05_supported(kv_dtype, head_dim, block_size, G, q))
            return decode_wide(fn, p, kv_dtype, k_cache, v_cache, new_k, new_v, plan_count,
                               plan_items, st);
        if (grouped) {
            // one CTA per (beam group, KV head, part); each writes the new
            // tokens of its run
            p.group_start = group_start;
            p.shared_tokens = shared_tokens;
            p.num_groups = num_groups;
            p.new_k = new_k;
            p.new_v = new_v;
            if (p.max_partitions > 1) {
                e = cudaMemsetAsync(p.done, 0, sizeof(unsigned) * (size_t)num_groups * num_kv_heads,
                                    st);
                if (e != cudaSuccess) return cuda_fail(e, fn);
            }
            // one n8 column tile when every group's members * G fits 8
            // (max_members 0: bounded by the sequences the other groups leave)
            const long long members =
                max_members > 0 ? max_members : (long long)num_seqs - num_groups + 1;
            const bool wide = members * G > 8;
            e = launch_decode_grouped(p, kv_dtype, &kmap, &vmap,
                                      (long long)num_groups * num_kv_heads * p.max_partitions, wide,
                                      st);
            if (e != cudaSuccess) return cuda_fail(e, fn);
            return PKV_OK;
        }
        // grid: every (sequence, KV head, partition group, head slice) slot, the
        // groups of one (sequence, KV head) adjacent and the slices of one
        // group next to each other; slots past a sequence's end exit at once
        // (with a work plan, the CTAs with work take its records instead).  Short partitions of long contexts go one per warp, four to a
        // CTA (with few partitions per sequence, a CTA would leave warps idle).
        if (p.partition_tokens <= kWarpPartitionMaxTokens &&
            p.max_partitions >= kWarpPartitionMinCount)
            p.cta_parts = kDecodeTcWarps;
        p.head_slices = (G + kDecodeTcMaxColumns - 1) / kDecodeTcMaxColumns;
        const int columns = (G + p.head_slices - 1) / p.head_slices;
        const long long groups = (p.max_partitions + p.cta_parts - 1) / p.cta_parts;
        const long long grid = (long long)num_seqs * num_kv_heads * p.head_slices * groups;
        if (grid >= (1ll << 31))
            return pkv_fail(PKV_ERR_SHAPE, "%s: more than 2^31 work items", fn);
        const int counters = p.max_partitions > 1 ? num_seqs * num_kv_heads * p.head_slices : 0;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = 0;
        // An unsplit launch of few items (at most two waves of three CTAs a
        // SM) runs deep rings: its last, longest CTAs then stream faster.
        const long long items = (long long)num_seqs * num_kv_heads * p.head_slices;
        const bool deep = p.max_partitions <= 1 && sms > 0 &&
                          items <= (long long)kDecodeTcDeepMaxWaves * kDecodeTcCtasPerSm * sms;
        if (plan_items != nullptr || counters > 0) {
            if (plan_items != nullptr && num_seqs <= kPlanMaxSeqs) {
                // the plan kernel zeroes the completion counters of the
                // in-kernel merge and lists the CTAs with work, longest
                // sequences first
                DecodePlanParams pp;
                pp.context_lens = context_lens;
                pp.num_seqs = num_seqs;
                pp.num_kv_heads = num_kv_heads;
                pp.head_slices = p.head_slices;
                pp.partition_tokens = p.partition_tokens;
                pp.cta_parts = p.cta_parts;
                pp.stage_tokens = decode_stage_tokens(head_dim, false);
                // pieces of near-equal contexts are sized to the CTAs the GPU
                // holds at once (split launches only: they merge partials)
                pp.slots = p.max_partitions > 1 ? kDecodeTcCtasPerSm * sms : 0;
                pp.max_groups = (int)groups;
                pp.max_len = max_ctx;
                int shift = 0;
                while ((max_ctx >> shift) >= kPlanBuckets) ++shift;
                pp.bucket_shift = shift;
                pp.items = plan_items;
                pp.item_count = plan_count;
                pp.done = p.done;
                pp.num_counters = counters;
                e = launch_decode_plan(pp, st);
                if (e != cudaSuccess) return cuda_fail(e, fn);
                p.items = plan_items;
                p.item_count = plan_count;
            } else if (counters > 0) {
                // completion counters for the in-kernel merge start at zero
                e = cudaMemsetAsync(p.done, 0, sizeof(unsigned) * (size_t)counters, st);
                if (e != cudaSuccess) return cuda_fail(e, fn);
            }
        }
        // the tensor-core kernel writes the new tokens itself
        p.new_k = new_k;
        p.new_v = new_v;
        if (deep)
            e = launch_decode_tensor_core_deep(p, kv_dtype, &kmap, &vmap, grid, columns > 8, st);
        else
            e = columns > 8 ? launch_decode_tensor_core_wide(p, kv_dtype, &kmap, &vmap, grid, st)
                            : launch_decode_tensor_core(p, kv_dtype, &kmap, &vmap, grid, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        return PKV_OK;
    }
    if (append) {
        e = launch_kv_append(const_cast<void*>(k_cache), const_cast<void*>(v_cache), new_k, new_v,
                             block_tables, context_lens, num_seqs, max_blocks_per_seq, num_blocks,
                             num_kv_heads, head_dim, block_size, pkv_dtype_bytes(kv_dtype),
                             p.status, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    e = launch_decode_cuda_core(p, kv_dtype, st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (p.max_partitions > 1) {
        e = launch_lse_reduce(p, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               float scale, int block_size, int num_kv_heads, int num_seqs,
                               int num_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                               int kv_dtype, int out_dtype, int partition_size, void* workspace,
                               size_t workspace_bytes, void* stream)
{
    return decode_impl("pkv_paged_decode_attention", out, q, k_cache, v_cache, block_tables,
                       context_lens, scale, block_size, num_kv_heads, num_seqs, num_heads, head_dim,
                       max_blocks_per_seq, num_blocks, kv_dtype, out_dtype, partition_size,
                       workspace, workspace_bytes, stream, nullptr, nullptr);
}

int pkv_paged_decode_grouped(void* out, const void* q, const void* new_k, const void* new_v,
                             void* k_cache, void* v_cache, const int32_t* block_tables,
                             const int32_t* context_lens, const int32_t* group_start,
                             const int32_t* shared_tokens, int num_groups, int max_members,
                             float scale, int block_size, int num_kv_heads, int num_seqs,
                             int num_heads, int head_dim, int max_blocks_per_seq, int num_blocks,
                             int kv_dtype, int out_dtype, int parts, void* workspace,
                             size_t workspace_bytes, void* stream)
{
    static const char* fn = "pkv_paged_decode_grouped";
    if (num_seqs > 0 && !group_start) return pkv_fail(PKV_ERR_NULL, "%s: NULL group_start", fn);
    if (num_seqs > 0 && (new_k == nullptr) != (new_v == nullptr))
        return pkv_fail(PKV_ERR_NULL, "%s: new_k and new_v must both be set or both NULL", fn);
    return decode_impl(fn, out, q, k_cache, v_cache, block_tables, context_lens, scale,
                       block_size, num_kv_heads, num_seqs, num_heads, head_dim, max_blocks_per_seq,
                       num_blocks, kv_dtype, out_dtype, 0, workspace, workspace_bytes, stream, new_k,
                       new_v, group_start, shared_tokens, num_groups, parts < 1 ? 1 : parts,
                       max_members);
}

int pkv_group_shared_tokens(const int32_t* block_tables, const int32_t* context_lens,
                            const int32_t* group_start, int num_groups, int num_seqs,
                            int max_blocks_per_seq, int block_size, int32_t* shared_tokens)
{
    static const char* fn = "pkv_group_shared_tokens";
    if (num_groups < 0 || num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0)
        return pkv_fail(PKV_ERR_SHAPE, "%s: bad sizes", fn);
    if (num_groups == 0) return PKV_OK;
    if (!block_tables || !context_lens || !group_start || !shared_tokens)
        return pkv_fail(PKV_ERR_NULL, "%s: NULL pointer", fn);
    for (int i = 0; i < num_groups; ++i) {
        const int a = group_start[i], b = group_start[i + 1];
        if (a < 0 || b <= a || b > num_seqs)
            return pkv_fail(PKV_ERR_SHAPE, "%s: group %d spans [%d, %d)", fn, i, a, b);
        // leading table entries that every member holds in common, within
        // every member's context
        int64_t shared = INT64_MAX;
        for (int s = a; s < b; ++s) shared = std::min<int64_t>(shared, context_lens[s]);
        const int32_t* t0 = block_tables + (size_t)a * max_blocks_per_seq;
        int blocks = 0;
        while (blocks < max_blocks_per_seq && (int64_t)blocks * block_size < shared) {
            bool same = t0[blocks] >= 0;
            for (int s = a + 1; s < b && same; ++s)
                same = block_tables[(size_t)s * max_blocks_per_seq + blocks] == t0[blocks];
            if (!same) break;
            ++blocks;
        }
        shared = std::min<int64_t>(shared, (int64_t)blocks * block_size);
        shared_tokens[i] = (int32_t)std::max<int64_t>(shared, 0);
    }
    return PKV_OK;
}

int pkv_decode_step(void* out, const void* q, const void* new_k, const void* new_v,
                    void* k_cache, void* v_cache, const int32_t* block_tables,
                    const int32_t* context_lens, float scale, int block_size, int num_kv_heads,
                    int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq,
                    int num_blocks, int kv_dtype, int out_dtype, int partition_size,
                    void* workspace, size_t workspace_bytes, void* stream)
{
    static const char* fn = "pkv_decode_step";
    if (num_seqs > 0 && (!new_k || !new_v)) return pkv_fail(PKV_ERR_NULL, "%s: NULL new_k/new_v", fn);
    return decode_impl(fn, out, q, k_cache, v_cache, block_tables, context_lens, scale,
                       block_size, num_kv_heads, num_seqs, num_heads, head_dim, max_blocks_per_seq,
                       num_blocks, kv_dtype, out_dtype, partition_size, workspace, workspace_bytes,
                       stream, new_k, new_v);
}

}  // extern "C"
