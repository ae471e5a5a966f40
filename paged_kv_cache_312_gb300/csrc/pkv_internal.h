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
