// Internal helpers shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstdarg>
#include <cstdio>

#include "pkv.h"

namespace pkv {

// Records a thread-local message for pkv_last_error() and returns `code`.
int fail(int code, const char* fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;

// Clears the thread-local message (called at the start of successful paths).
void clear_error();

// Per-translation-unit readers of the device check word; each .cu that
// launches kernels defines one.  They synchronise nothing themselves.
int read_device_error_attention(int reset, int* code);
int read_device_error_cache_ops(int reset, int* code);
int read_device_error_prefill(int reset, int* code);

}  // namespace pkv
