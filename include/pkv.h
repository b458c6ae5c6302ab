/*
 * pkv.h -- C ABI of the paged K/V-cache decode path (libpkv.so), sm_103a.
 *
 * Sources, cited by page title and section:
 *   [note]    "vLLM / PagedAttention -- 把 LLM 服务的瓶颈从显存碎片里救出来"
 *             (awesome.papernotes.org, 2023_vllm)
 *   [lecture] "vLLM" lecture notes (formulaic.cloudchewie.com, 5-vllm)
 *   [guide]   "vLLM / PagedAttention (SOSP 2023)" (upskillscore.com system-design guide)
 *
 * Conventions for every entry point:
 *   - fp16 tensors are passed as uint16_t bit patterns (IEEE binary16).
 *   - "device" pointers point into memory of the current CUDA device; "host"
 *     pointers into ordinary host memory.  The caller owns every buffer and the
 *     stream; the library never allocates device memory, never frees caller
 *     memory and keeps no pointer after a call returns.
 *   - The per-step inputs of the decode path may instead be page-locked host
 *     memory mapped into the device's address space (cudaHostAlloc; with unified
 *     addressing its host address is its device address).  These are q,
 *     block_tables, context_lens and out of pkv_paged_attention_decode; the same
 *     except q for pkv_paged_attention_decode_shared_prefix, plus group_start and
 *     prefix_lens; key, value and slot_mapping of pkv_reshape_and_cache; and
 *     block_mapping of pkv_copy_blocks.
 *     pkv_paged_attention_decode_append takes the same, plus key, value and
 *     slot_mapping.
 *     The kernels then read or write them across the host link (NVLink-C2C on a
 *     Grace-Blackwell node) with plain loads and stores, and no staging copy is
 *     needed.  K/V pools and workspaces must be device memory.  As with device
 *     buffers, the caller keeps such memory allocated and unchanged until the
 *     stream has finished the call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device work is
 *     asynchronous on it; arguments are validated on the host first.
 *   - Return value: PKV_OK or a negative pkv_status; pkv_last_error() gives a
 *     message (thread-local) for the last failing call.  No exception crosses
 *     the ABI.
 *   - Kernels check every block id, slot and context length they read against
 *     the sizes passed in; a bad value is skipped (never dereferenced) and its
 *     code is recorded in a per-device error word that pkv_device_error reads.
 *
 * K/V pool layout (the pages leave it open; [note] 关键设计 5 asks only for "a
 * layout suited to block reads"): each layer has a K pool and a V pool, each
 * [num_blocks, num_heads, block_size, head_dim] fp16, row-major.  Token slot
 * `slot` is row slot % block_size of physical block slot / block_size, so one
 * (block, head) tile of a pool is block_size*head_dim*2 contiguous bytes.
 *
 * Supported shapes: head_dim in {64, 128}, block_size in {4, 8, 16, 32}, one K/V
 * head per query head.  Other values return PKV_ERR_UNSUPPORTED.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = -1,   /* bad pointer, size, alignment or id */
  PKV_ERR_UNSUPPORTED = -2,   /* a shape outside the supported set */
  PKV_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
  PKV_ERR_WORKSPACE = -4,     /* workspace missing or too small */
  PKV_ERR_OOM = -5,           /* block manager: not enough free blocks (state unchanged) */
  PKV_ERR_DEVICE_CHECK = -6,  /* a kernel met an out-of-range id, slot or length */
  PKV_ERR_NOT_FOUND = -7      /* block manager: unknown sequence or prefix id */
} pkv_status;

/* Device-side check codes recorded by the kernels (first one wins). */
enum {
  PKV_DEV_OK = 0,
  PKV_DEV_BAD_BLOCK_ID = 1,     /* a block table entry outside [0, num_blocks) */
  PKV_DEV_BAD_CONTEXT_LEN = 2,  /* a context length < 0 or > max_blocks_per_seq*block_size */
  PKV_DEV_BAD_SLOT = 3,         /* a slot >= num_blocks*block_size */
  PKV_DEV_BAD_COPY_PAIR = 4,    /* a copy pair with an id outside [0, num_blocks) */
  PKV_DEV_WAIT_TIMEOUT = 5,     /* a shared-memory copy did not complete in time */
  PKV_DEV_BAD_QUERY_RANGE = 6,  /* prefill: new tokens outside [0, context_len] or outside q, or
                                   more new tokens than max_query_len covers */
  PKV_DEV_PREFIX_MISMATCH = 7   /* shared-prefix decode: a sequence's first prefix blocks differ
                                   from its group's first sequence's, a bad group layout, or a
                                   group larger than max_group_size */
};

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* pkv_last_error(void);

/* ABI version (major*100 + minor). */
int pkv_version(void);

/*
 * Synchronises `stream`, then returns PKV_OK if no kernel of this library on the
 * current device recorded a check failure, else PKV_ERR_DEVICE_CHECK with the
 * first recorded PKV_DEV_* code in *code (may be NULL).  reset != 0 clears the
 * recorded code.
 */
int pkv_device_error(void* stream, int reset, int* code);

/* ---------------------------------------------------------------------------
 * Paged decode attention ([note] 关键设计 1, both equations; 关键设计 5, "fusing
 * block read and attention").
 *
 * For every sequence s < num_seqs and head h < num_heads:
 *   out[s,h,:] = sum_{t < ctx_s} softmax_t(scale * q[s,h,:] . k_t) v_t
 * with k_t = k_cache[block_tables[s, t / B], h, t % B, :] (v_t likewise) and
 * ctx_s = context_lens[s].  The softmax normalises over all ctx_s tokens.
 * ctx_s = 0 gives a zero row.  Table entries at column >= ceil(ctx_s / B) are
 * never used and may hold anything: they can be read (within the table row),
 * but no K/V is fetched through them and they are not checked.  Accumulation is
 * fp32; out is rounded to nearest even.
 *
 *   q            device [num_seqs, num_heads, head_dim] fp16, 16-byte aligned
 *   k_cache,
 *   v_cache      device [num_blocks, num_heads, block_size, head_dim] fp16,
 *                16-byte aligned
 *   block_tables device [num_seqs, max_blocks_per_seq] int32 physical ids
 *   context_lens device [num_seqs] int32
 *   out          device [num_seqs, num_heads, head_dim] fp16, 16-byte aligned;
 *                must not overlap the inputs
 *   workspace    device scratch for the split over the context (partial
 *                max / sum / output per partition); at least
 *                pkv_paged_attention_workspace_size(...) bytes, 16-byte aligned.
 *                May be NULL when pkv_paged_attention_plan reports one kernel
 *                for these sizes (one partition per sequence, or partitions
 *                merged on chip).  Contents need no initialisation and are
 *                garbage afterwards.  Calls that share a workspace must be
 *                ordered on one stream.
 *
 * The context is split into partitions (one CTA each).  When a sequence has at
 * most 8 and the whole grid fits in one wave of resident CTAs, the partitions
 * of each (sequence, head) run as one thread-block cluster and the first
 * merges the others' partial results, which they store into its shared memory;
 * otherwise the partial results go to the workspace and a second kernel
 * merges them.
 *
 * Returns PKV_ERR_WORKSPACE if the workspace is needed and missing or small.
 * ------------------------------------------------------------------------- */
size_t pkv_paged_attention_workspace_size(int num_seqs, int num_heads, int head_dim,
                                          int max_blocks_per_seq, int block_size);

/* The launch plan pkv_paged_attention_decode uses on the current device for
 * these sizes: *part_tokens receives the context partition length (tokens per
 * CTA) and *num_kernels the kernels one call launches: 1 when a sequence spans
 * one partition or its partitions merge inside a thread-block cluster, 2 when
 * a merge kernel follows (only then is the workspace used).
 * Host only; queries the device's SM count once.  Context capacities above
 * 2^30 tokens are PKV_ERR_UNSUPPORTED. */
int pkv_paged_attention_plan(int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq,
                             int block_size, int* part_tokens, int* num_kernels);

int pkv_paged_attention_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int num_seqs, int num_heads, int head_dim, int num_blocks,
                               int max_blocks_per_seq, float scale, int block_size, uint16_t* out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Decode step with the new token's K/V write fused in: exactly
 * pkv_reshape_and_cache(key, value, slot_mapping) followed by
 * pkv_paged_attention_decode, in one launch (the write-then-attend order of
 * [note] 关键设计 1: the sum runs to t = i, so the new token attends to
 * itself).  Sequence s has one new token, rows key[s] and value[s]
 * ([num_seqs, num_heads, head_dim] fp16, 16-byte aligned), stored at
 * slot_mapping[s] (int64; < 0: none); context_lens[s] already counts it.
 *
 * The CTA that reads the context's last position stores the row and, where
 * the table maps that position to slot_mapping[s], uses the row it stored
 * instead of the copy in the pool.  The result and the pools then equal
 * those of the two separate calls, provided no other sequence of the batch
 * reads an appended slot.  Slots from pkv_bm_append_slot(s) meet that: a
 * shared block is copied before it is written.  A slot >= num_blocks *
 * block_size records PKV_DEV_BAD_SLOT and is not written.  Arguments, the
 * workspace and the error behaviour are otherwise those of
 * pkv_paged_attention_decode, including page-locked host memory for q,
 * key, value, slot_mapping, the tables, the lengths and out.  k_cache and
 * v_cache are written.
 * ------------------------------------------------------------------------- */
int pkv_paged_attention_decode_append(const uint16_t* q, const uint16_t* key, const uint16_t* value,
                                      const int64_t* slot_mapping, uint16_t* k_cache, uint16_t* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                      int num_heads, int head_dim, int num_blocks, int max_blocks_per_seq,
                                      float scale, int block_size, uint16_t* out, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Paged decode attention for batches whose sequences share prefix blocks
 * ([guide] 04: requests map their first logical blocks onto one cached
 * prefix; [lecture] Parallel Sampling 场景 and Beam Search 场景: siblings share
 * their prompt blocks).  Same result as pkv_paged_attention_decode (within its
 * tolerance); the shared prefix is read once per group instead of once per
 * sequence.
 *
 * Sequences [group_start[g], group_start[g+1]) form group g, whose members map
 * their first prefix_lens[g] / block_size logical blocks onto the same physical
 * blocks (the block manager's shared prefix or prompt).  For each group and
 * head, the prefix part of every member's attention runs as one tensor-core
 * product (queries of up to 256 members x the prefix keys, read through the
 * group's first sequence's table row), giving a partial (max, sum, output) per
 * sequence; the rest of each context [prefix_len, ctx) runs as in
 * pkv_paged_attention_decode; a log-sum-exp merge combines the parts.
 *
 *   group_start    device [num_groups + 1] int32: 0 = group_start[0] <= ... <=
 *                  group_start[num_groups] = num_seqs (the groups cover the batch)
 *   prefix_lens    device [num_groups] int32: multiples of block_size, each at
 *                  most the group's shortest context (0: no shared prefix)
 *   max_group_size host: the largest group_start[g+1] - group_start[g] (sizes the
 *                  grid).  A larger group records PKV_DEV_PREFIX_MISMATCH: its
 *                  members past the grid get no prefix part and their rows are
 *                  wrong.
 *   workspace      at least pkv_paged_attention_shared_prefix_workspace_size(...)
 *                  bytes, 16-byte aligned, required.
 *   other arguments as for pkv_paged_attention_decode.
 *
 * Groups of fewer than 8 members read their prefix per sequence, as plain
 * decode does (a shared block then mostly comes from L2, and the product's
 * 128-row tile would be nearly empty); if no group reaches 8 members the call
 * is pkv_paged_attention_decode.  A member of a larger group whose first prefix
 * blocks differ from the group's first sequence's, or a group layout that does
 * not cover the batch, records PKV_DEV_PREFIX_MISMATCH (the prefix is then the
 * first sequence's).
 * ------------------------------------------------------------------------- */
size_t pkv_paged_attention_shared_prefix_workspace_size(int num_seqs, int num_heads, int head_dim,
                                                        int max_blocks_per_seq, int block_size);

int pkv_paged_attention_decode_shared_prefix(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                             const int32_t* block_tables, const int32_t* context_lens,
                                             const int32_t* group_start, const int32_t* prefix_lens, int num_groups,
                                             int max_group_size, int num_seqs, int num_heads, int head_dim,
                                             int num_blocks, int max_blocks_per_seq, float scale, int block_size,
                                             uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Paged prefill attention: the new tokens of each sequence (the task input)
 * over its cached context plus, causally, themselves ([guide] 04: the prompt
 * phase runs only over the task input, the request's first logical blocks
 * mapped onto cached prefix blocks; [note] 关键设计 1, first equation).
 *
 * Sequence s has n_s = query_start[s+1] - query_start[s] new tokens, rows
 * query_start[s] .. query_start[s+1]-1 of q and out; their keys and values are
 * already in the pools (reshape_and_cache), and context_lens[s] counts the
 * cached tokens plus the new ones.  New token i (position p = ctx_s - n_s + i):
 *   out[query_start[s] + i, h, :] = sum_{t <= p} softmax_t(scale * q . k_t) v_t
 * with k_t read through block_tables as in pkv_paged_attention_decode.
 * Tensor cores: fp16 products, fp32 accumulation; the softmax weights are
 * rounded to fp16 before they multiply V.
 *
 *   q, out        device [total_q, num_heads, head_dim] fp16, 16-byte aligned;
 *                 out must not overlap the inputs
 *   query_start   device [num_seqs + 1] int32, non-decreasing, last = total_q
 *   max_query_len host: the largest n_s (sizes the grid).  A larger n_s records
 *                 PKV_DEV_BAD_QUERY_RANGE, and its rows past the grid are not
 *                 written.
 *   pools, tables, context_lens as for pkv_paged_attention_decode.
 * scale must be positive.  A sequence with n_s = 0 is skipped; n_s > ctx_s or
 * rows outside q record PKV_DEV_BAD_QUERY_RANGE; a table entry outside
 * [0, num_blocks) within the context records PKV_DEV_BAD_BLOCK_ID and the
 * sequence's rows (of the affected 256-token tile) are not written.  No
 * workspace.
 * ------------------------------------------------------------------------- */
int pkv_paged_attention_prefill(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* query_start, int num_seqs, int total_q, int max_query_len,
                                int num_heads, int head_dim, int num_blocks, int max_blocks_per_seq,
                                float scale, int block_size, uint16_t* out, void* stream);

/* ---------------------------------------------------------------------------
 * Paged decode attention with the library's own scratch (no counterpart in the
 * paper: an addition of this library for callers that cannot allocate).
 *
 * Callers without a device allocator of their own (a plain C host program, a
 * plugin inside an engine that has reserved all device memory for its block
 * pools) or on a path that must not pay for the device-wide synchronisation of
 * cudaMalloc/cudaFree use this instead of pkv_paged_attention_decode.  It takes
 * the same arguments minus the workspace, computes the same result, and keeps
 * the scratch in a fixed array of pkv_paged_attention_static_workspace_bytes()
 * bytes (16 MiB) inside the library; every device that loads the library holds
 * that array until the process exits.  It allocates nothing.
 *
 *   - A batch whose scratch would exceed the array is rejected with
 *     PKV_ERR_WORKSPACE (and a message) before anything is launched.
 *   - The first call on a device looks up the array's device address in the
 *     caller's current context (cudaGetSymbolAddress with the device current);
 *     make that first call before any stream capture.  The address is kept
 *     per context: after cudaDeviceReset, or from a thread whose current
 *     context is another one (a plugin's own cuCtxCreate), the next call looks
 *     it up again, and that call too should come before any capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  Nothing in it needs clearing: each call writes every partial
 *     result before reading it.  Calls whose kernels overlap on the GPU (on
 *     different streams, or from different host threads without ordering)
 *     race on the array: order them on one stream.
 * ------------------------------------------------------------------------- */
size_t pkv_paged_attention_static_workspace_bytes(void);

int pkv_paged_attention_decode_static_workspace(const uint16_t* q, const uint16_t* k_cache,
                                                const uint16_t* v_cache, const int32_t* block_tables,
                                                const int32_t* context_lens, int num_seqs, int num_heads,
                                                int head_dim, int num_blocks, int max_blocks_per_seq,
                                                float scale, int block_size, uint16_t* out, void* stream);

/* ---------------------------------------------------------------------------
 * For failure-detection tests only (not a computation of the paper): runs
 * pkv_paged_attention_decode on sizes whose partitions merge inside
 * thread-block clusters, but with every partition other than the first
 * skipping its stores into partition 0's shared memory and its arrivals on
 * partition 0's barrier, and partition 0's wait for them limited to wait_ms
 * (1..2000).  Nothing then completes that wait: partition 0 gives up after
 * wait_ms, records PKV_DEV_WAIT_TIMEOUT (read with pkv_device_error) and writes
 * an undefined output; no CTA touches another's memory and the context stays
 * usable.  PKV_ERR_UNSUPPORTED for sizes that would not merge on chip.  No
 * workspace.
 * ------------------------------------------------------------------------- */
int pkv_test_cluster_merge_timeout(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                   int num_heads, int head_dim, int num_blocks, int max_blocks_per_seq, float scale,
                                   int block_size, uint16_t* out, int wait_ms, void* stream);

/* ---------------------------------------------------------------------------
 * Reshape and cache ([note] 关键设计 5, "fused reshape and block write").
 *
 * For every token t < num_tokens with slot = slot_mapping[t] >= 0:
 *   k_cache[slot / B, h, slot % B, :] = key[t, h, :]   for all h  (value likewise)
 * A negative slot marks a padding token and is skipped.  Bit-exact copy.
 *
 *   key, value   device [num_tokens, num_heads, head_dim] fp16, contiguous,
 *                16-byte aligned
 *   k_cache,
 *   v_cache      device pools as above
 *   slot_mapping device [num_tokens] int64
 * Two tokens with the same slot race (one of them wins).
 * ------------------------------------------------------------------------- */
int pkv_reshape_and_cache(const uint16_t* key, const uint16_t* value, uint16_t* k_cache,
                          uint16_t* v_cache, const int64_t* slot_mapping, int num_tokens,
                          int num_heads, int head_dim, int block_size, int num_blocks, void* stream);

/* reshape_and_cache over num_layers layers in one launch (all layers' new
 * tokens share one slot mapping).  keys, values, k_caches, v_caches: HOST
 * arrays of num_layers device pointers, each laid out as above. */
int pkv_reshape_and_cache_layers(const uint16_t* const* keys, const uint16_t* const* values,
                                 uint16_t* const* k_caches, uint16_t* const* v_caches, int num_layers,
                                 const int64_t* slot_mapping, int num_tokens, int num_heads, int head_dim,
                                 int block_size, int num_blocks, void* stream);

/* ---------------------------------------------------------------------------
 * Batched block copy ([note] 关键设计 3 copy-on-write; 关键设计 5, "fused block
 * copy": many small block copies in one kernel instead of one memcpy each).
 *
 * For every pair p < num_pairs and every layer l < num_layers:
 *   k_caches[l][dst_p] = k_caches[l][src_p]; v_caches[l][dst_p] = v_caches[l][src_p]
 * with (src_p, dst_p) = (block_mapping[2p], block_mapping[2p+1]); whole blocks,
 * all heads and rows.  Bit-exact.  A destination must not be the source or
 * destination of another pair in the same call.
 *
 *   k_caches,
 *   v_caches      HOST arrays of num_layers device pool pointers (16-byte aligned)
 *   block_mapping device or page-locked host [num_pairs, 2] int64
 * ------------------------------------------------------------------------- */
int pkv_copy_blocks(uint16_t* const* k_caches, uint16_t* const* v_caches, int num_layers,
                    const int64_t* block_mapping, int num_pairs, int num_heads, int head_dim,
                    int block_size, int num_blocks, void* stream);

/* ---------------------------------------------------------------------------
 * Block swap between two pools ([lecture] 调度和抢占, Swapping: the blocks of a
 * preempted sequence move to CPU memory and back; [guide] 05).
 *
 * For every pair p < num_pairs and every layer l < num_layers:
 *   dst_k_caches[l][dst_p] = src_k_caches[l][src_p]   (V likewise)
 * with (src_p, dst_p) = (block_mapping[2p], block_mapping[2p+1]); whole blocks.
 * Bit-exact.  One launch moves every pair of every layer (no per-block memcpy).
 *
 *   src_*, dst_*  HOST arrays of num_layers pool pointers.  Each pool is
 *                 [num_blocks, num_heads, block_size, head_dim] fp16, 16-byte
 *                 aligned, in device memory OR in page-locked host memory
 *                 (cudaHostAlloc / cudaHostRegister), which the kernel reads or
 *                 writes directly over the host link.  Swap-out: device source,
 *                 host destination; swap-in: the reverse.  Pageable host memory
 *                 is refused (PKV_ERR_INVALID_ARG).
 *   block_mapping [num_pairs, 2] int64 in device or page-locked host memory;
 *                 src ids in [0, src_num_blocks), dst ids in [0, dst_num_blocks).
 *                 Destinations must be distinct and must not overlap sources.
 * ------------------------------------------------------------------------- */
int pkv_swap_blocks(const uint16_t* const* src_k_caches, const uint16_t* const* src_v_caches,
                    uint16_t* const* dst_k_caches, uint16_t* const* dst_v_caches, int num_layers,
                    const int64_t* block_mapping, int num_pairs, int num_heads, int head_dim,
                    int block_size, int src_num_blocks, int dst_num_blocks, void* stream);

/* ---------------------------------------------------------------------------
 * Host block manager ([note] 关键设计 2 and 3; [lecture] PagedAttention 原理 and
 * Parallel Sampling 场景; [guide] 03 and 04).  No device memory, no CUDA.
 *
 * Each sequence owns a list of logical blocks; each logical block records a
 * physical block id and how many of its B slots are filled.  Physical blocks
 * carry reference counts.  Rules:
 *   - prefill takes ceil(len / B) blocks; tokens fill blocks left to right;
 *   - append: if the last block is full, take a new block and write there;
 *     else if the last block's count is > 1, take a new block, report the
 *     copy (old -> new) the caller must run with pkv_copy_blocks before the
 *     write, decrement the old count and move the sequence onto the copy;
 *     else write in place;
 *   - fork: the child maps every logical block onto the parent's physical
 *     blocks (counts +1); free: counts -1, blocks reaching 0 return to the
 *     free list;
 *   - a registered prefix holds one reference on each of its blocks; a
 *     sequence added on a prefix maps its first logical blocks onto them.
 * The free list is FIFO over `free_order`: taking pops the front, a freed
 * block is pushed at the back.  slot = physical id * B + row.
 * Every call is all-or-nothing: PKV_ERR_OOM (and every other error) leaves
 * the state unchanged.  An instance is not thread-safe.
 * ------------------------------------------------------------------------- */
typedef struct pkv_bm pkv_bm;

/* free_order: host [num_blocks] permutation of 0..num_blocks-1, or NULL for
 * 0,1,2,...  Returns NULL on bad arguments (see pkv_last_error). */
pkv_bm* pkv_bm_create(int num_blocks, int block_size, const int32_t* free_order);
void pkv_bm_destroy(pkv_bm* bm);

/* Prefill a new sequence of prompt_len >= 1 tokens.  slots_out: host
 * [prompt_len] or NULL; receives the prompt tokens' slots. */
int pkv_bm_add_seq(pkv_bm* bm, int64_t seq_id, int prompt_len, int64_t* slots_out);

/* The child shares all of the parent's blocks. */
int pkv_bm_fork(pkv_bm* bm, int64_t parent, int64_t child);

/* Slot for the sequence's next token.  *cow_src / *cow_dst receive the block
 * copy to run first, or -1 / -1. */
int pkv_bm_append_slot(pkv_bm* bm, int64_t seq_id, int64_t* slot, int32_t* cow_src, int32_t* cow_dst);

/* One append for each of n distinct sequences, in order, all-or-nothing.
 * slots_out host [n]; cow_pairs_out host [n, 2] int64 receives the copies
 * (src, dst), *num_cow their number. */
int pkv_bm_append_slots(pkv_bm* bm, const int64_t* seq_ids, int n, int64_t* slots_out,
                        int64_t* cow_pairs_out, int* num_cow);

int pkv_bm_free(pkv_bm* bm, int64_t seq_id);

/* n >= 0 appends to one sequence in one all-or-nothing call: the slots of its
 * next n tokens, in order, to slots_out (host [n]).  Only the first append can
 * need a copy (of a shared partly filled last block; later appends find the
 * last block private): it goes to cow_pair_out (host [2] int64 (src, dst), may
 * be NULL) with *num_cow = 1, else *num_cow = 0 (num_cow may be NULL).  The
 * prompt phase of a request uses it to place all of its new tokens at once. */
int pkv_bm_extend(pkv_bm* bm, int64_t seq_id, int n, int64_t* slots_out, int64_t* cow_pair_out, int* num_cow);

/* A provider-stored prefix of len >= 1 tokens ([guide] 04); slots_out as in
 * pkv_bm_add_seq. */
int pkv_bm_register_prefix(pkv_bm* bm, int64_t prefix_id, int len, int64_t* slots_out);

/* A request on a registered prefix ([guide] 04, steps 2 and 4): its first
 * logical blocks map onto the prefix's physical blocks (reference counts +1),
 * then its suffix_len >= 0 own tokens (the task input its prompt phase runs
 * over) get slots as pkv_bm_extend gives them: slots_out host [suffix_len]
 * (may be NULL when suffix_len is 0).  A partly filled last prefix block is
 * shared with the prefix, so the first suffix token copies it (cow_pair_out,
 * *num_cow = 1; both may be NULL).  All-or-nothing: PKV_ERR_OOM if the suffix
 * needs more blocks than are free, and nothing changes. */
int pkv_bm_add_seq_with_prefix(pkv_bm* bm, int64_t seq_id, int64_t prefix_id, int suffix_len, int64_t* slots_out,
                               int64_t* cow_pair_out, int* num_cow);
int pkv_bm_drop_prefix(pkv_bm* bm, int64_t prefix_id);

/* One sequence's physical ids (host out[cap]), block count and token count. */
int pkv_bm_block_table(const pkv_bm* bm, int64_t seq_id, int32_t* out, int cap, int* n_blocks,
                       int* ctx_len);

/* Padded tables for a batch: tables_out host [n, max_blocks] int32 (-1 past
 * each sequence's blocks), ctx_lens_out host [n] int32. */
int pkv_bm_block_tables(const pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* tables_out,
                        int max_blocks, int32_t* ctx_lens_out);

/* One beam-search step ([lecture] Beam Search 场景; [guide] 04): child i
 * forks parent i (shares all its blocks); then every retired sequence (the
 * previous beam) is freed, returning the blocks no candidate still holds;
 * then each child appends one token, copying a shared partly filled last
 * block (reported in cow_pairs_out, host [k, 2] int64; *num_cow copies).
 * parents/children: host [k]; children are new distinct ids; retire: host
 * [n_retire] existing distinct ids (parents may be among them).
 * slots_out: host [k].  All-or-nothing. */
int pkv_bm_beam_step(pkv_bm* bm, const int64_t* parents, const int64_t* children, int k,
                     const int64_t* retire, int n_retire, int64_t* slots_out, int64_t* cow_pairs_out,
                     int* num_cow);

/* Swapping ([lecture] 调度和抢占, Swapping; [guide] 05): the sequences
 * seq_ids (host [n], distinct) -- a preempted group, such as a request's
 * samples or beams -- move whole from src to dst, typically the managers of
 * an HBM pool and of a page-locked host pool with the same block size.
 * Every distinct physical block the group maps gets one block taken from
 * dst's free list, in order of first appearance (sequences in the given
 * order, each in logical order), and keeps its reference count; the
 * sequences keep their logical layout and sharing; the old blocks return to
 * src's free list in the same order.  pairs_out (host [cap_pairs, 2] int64)
 * receives the moves (src block, dst block), *n_pairs their number: the
 * block_mapping for pkv_swap_blocks, which the caller runs before the
 * sequences are used on dst's pool.
 * The group must hold every reference to its blocks: a block also held by
 * another sequence or by a registered prefix is PKV_ERR_INVALID_ARG.
 * PKV_ERR_OOM if dst has too few free blocks, PKV_ERR_NOT_FOUND for an id not
 * on src, PKV_ERR_INVALID_ARG for an id already on dst, a repeated id,
 * different block sizes or cap_pairs too small.  All-or-nothing: on any error
 * neither manager changes. */
int pkv_bm_swap(pkv_bm* src, pkv_bm* dst, const int64_t* seq_ids, int n, int64_t* pairs_out,
                int cap_pairs, int* n_pairs);

/* Observability ([note] 局限与展望, 复杂系统带来新的调度和可观测性问题: a paged
 * cache should expose block occupancy, tail waste, the distribution of
 * reference counts, prefix-cache hits and preemptions).
 * pkv_bm_ref_histogram: hist (host [cap] int64) receives, for r < cap - 1,
 * the number of physical blocks whose reference count is r (hist[0] = free
 * blocks); hist[cap - 1] counts every block with a count >= cap - 1.
 * pkv_bm_counters: out (host [n] int64) receives the first n of, in order,
 * copy-on-write copies reported, sequences added on a registered prefix,
 * block references those sequences took from prefixes (prefix hits), groups
 * swapped away from this manager, blocks swapped away, groups swapped in,
 * blocks swapped in.  Returns how many were written (at most 7). */
int pkv_bm_ref_histogram(const pkv_bm* bm, int64_t* hist, int cap);
int pkv_bm_counters(const pkv_bm* bm, int64_t* out, int n);

/* Reference count of a physical block (negative status on a bad id). */
int pkv_bm_ref_count(const pkv_bm* bm, int32_t block);

/* Free blocks, unfilled slots summed over sequences, copies reported so far. */
int pkv_bm_stats(const pkv_bm* bm, int* free_blocks, int64_t* tail_waste_tokens, int64_t* cow_copies);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
