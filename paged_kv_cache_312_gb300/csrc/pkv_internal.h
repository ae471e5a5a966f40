// Internal host-side helpers of libpkv (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

// Records a formatted message as the calling thread's last error and returns
// `code`, so that call sites read `return pkv_fail(PKV_ERR_SHAPE, "...")`.
int pkv_fail(int code, const char* fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;

// Element size in bytes of a PKV_* dtype code, 0 if unknown.
inline int pkv_dtype_bytes(int dtype)
{
    return dtype == 0 ? 4 : (dtype == 1 || dtype == 2) ? 2 : 0;
}

// Checks of a decode request's dtypes and sizes that need no pointer:
// dtypes, num_seqs in [0, 65535], head_dim in {64, 128}, block_size in
// {8, 16, 32}, num_heads a multiple of num_kv_heads, positive table and pool
// sizes, a maximum context of at most 2^30 tokens, fewer than 2^31 cache
// rows, partition_size 0 or a multiple of block_size, a finite scale.
// Returns PKV_OK or the failing code (with the message recorded).
int pkv_decode_check(const char* fn, int kv_dtype, int out_dtype, int num_seqs, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                     int num_blocks, int partition_size, float scale);
