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

// Shared-prefix decode reads a group's prefix once only for groups of at least this many members;
// smaller groups (where the prefix mostly comes from L2 anyway and a 128-row tensor-core tile would
// be nearly empty) run their whole context through the split-K decode kernel.  Measured on a
// 1024-token prefix: 4 members break even, 8 are 1.4x faster, 64 are 1.9x.
constexpr int kMinSharedGroup = 8;

// Shared-prefix partials (prefill.cu, tensor cores): for every member s of every group g and every
// head h, the partial (max m and sum l in the base-2 log domain of scale * q.k, unnormalised
// output o) of q[s, h] over the keys [0, prefix_lens[g]) read through block_tables row
// group_start[g], written to slot 0 of the decode workspace: ws_ml[2 w], ws_ml[2 w + 1], ws_o[w D ..]
// with w = (s * num_heads + h) * max_parts.  Validates nothing the caller checked already.
int launch_prefix_partials(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                           const int32_t* block_tables, const int32_t* group_start, const int32_t* prefix_lens,
                           int num_groups, int max_group_size, int num_seqs, int num_heads, int head_dim,
                           int num_blocks, int max_blocks_per_seq, float scale, int block_size, float* ws_ml,
                           float* ws_o, int max_parts, void* stream);

}  // namespace pkv
