// Paged decode attention for sm_103a: one query per (sequence, head), K/V read
// block by block through the sequence's block table.
//
// What is computed ([note] "vLLM / PagedAttention -- 把 LLM 服务的瓶颈从显存碎片里救出来",
// section 关键设计 1, both equations): o = sum_t softmax_t(scale * q.k_t) v_t over
// the sequence's ctx tokens, where token t sits in physical block
// table[t / B] at row t % B.  Section 关键设计 5 ("fusing block read and
// attention") has the kernel read the blocks itself, a warp per block.
//
// GB300 design (decode attention is a batched GEMV: ~1 flop per byte, so HBM
// bandwidth is the roofline and no tensor cores are used):
//  * The context is split into partitions of `part_tokens` (128..1024) tokens, the longest
//    that still gives every SM a CTA; one CTA
//    handles one (partition, head, sequence).  The partitions of a (sequence, head)
//    merge with the log-sum-exp identity
//    m = max m_p, l = sum l_p 2^(m_p - m), o = sum o_p 2^(m_p - m) / l:
//    on a grid of at most one wave with at most 8 partitions, inside one
//    thread-block cluster (partition 0 gathers the others' partials from their
//    stores into its shared memory); otherwise in a second, tiny kernel over a
//    workspace.
//  * The unit of work is a chunk of R = min(B, 16) rows of one (block, head)
//    tile: R*D*2 contiguous bytes of K and as many of V.  Each warp owns a ring
//    of NST shared-memory stages; lane 0 fills a stage with two 1-D bulk async
//    copies (cp.async.bulk global->shared, completion counted in bytes on an
//    mbarrier), so a warp keeps NST chunks in flight while it computes.
//  * q.k: lane l holds 8 q values (16-byte column l % (D/8)) pre-multiplied by
//    scale*log2(e); partial dots of the rows it loaded are summed across the
//    D/8 lanes of a row with a transposing butterfly (R/2 + 1 .. shuffles per
//    chunk instead of one 4-step reduction per row).
//  * Online softmax in base 2 (exp2f), fp32 accumulators in registers; rows
//    past the context are excluded by select/branch, never multiplied by zero,
//    so stale NaN/Inf in unfilled slots cannot leak into the result.
//  * A partition's slice of the block table is read beside the context length
//    (without shared-prefix groups every range starts at token 0), one entry per chunk.
//  * pkv_paged_attention_decode_append runs the APPEND instantiation: the CTA
//    holding the context's last position also stores the new token's K/V row at
//    its slot and writes it over its staged copy of that chunk (section 关键设计 5's
//    fused reshape and block write, folded into the attention launch).
//  * Every wait is bounded by a global-timer deadline; on expiry the kernel
//    records PKV_DEV_WAIT_TIMEOUT, waits (bounded) for its own copies in
//    flight and returns.  In a cluster, partition 0 waits for the others with
//    a longer deadline than any of their own waits, and never exits before
//    their stores into its shared memory have landed.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "launch.cuh"
#include "pkv_internal.h"

namespace {

__device__ int g_dev_error_attention = 0;

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_dev_error_attention, 0, code); }

constexpr unsigned FULL = 0xffffffffu;
constexpr unsigned long long WAIT_NS = 2000000000ull;  // 2 s: a 16 KB copy takes microseconds

// ---- PTX wrappers --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for the phase of `parity` to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && global_ns() - t0 > WAIT_NS) return false;
  }
  return false;
}
// ---- thread-block cluster helpers (the partitions of one (sequence, head) as one cluster) -------
// Relaxed arrival: what the other CTAs need before they reach this one's shared memory is the
// receiving barrier's initialisation, which its own fence (fence.mbarrier_init.release.cluster)
// publishes.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// The shared::cluster address of this CTA's shared-memory location `addr` in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// One arrival on an mbarrier in another CTA of the cluster, releasing this thread's earlier
// shared::cluster stores to whoever acquires the barrier's phase.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (deadline `ns`) for a phase completed by other CTAs of the cluster.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, unsigned long long ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 255u) == 255u && global_ns() - t0 > ns) return false;
  }
  return false;
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted on `bar`.
// K/V tiles are streamed once per (sequence, head), so they are marked first to
// leave L2 (evict_first); a block shared by many sequences still hits in L2
// while it is being reused.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// ---- configuration ---------------------------------------------------------------------------
template <int D, int R>
struct Cfg {
  static constexpr int CPR = D / 8;                  // lanes per row (16-byte columns)
  static constexpr int RPI = 32 / CPR;               // rows covered by one warp-wide 16-byte load
  static constexpr int NJ = R / RPI;                 // rows each lane loads per chunk
  static constexpr int DUP = CPR / NJ;               // lanes holding the same reduced row
  static constexpr int CHUNK_BYTES = R * D * 2;      // K (or V) bytes of one chunk
  static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;
  static constexpr int NW = 4;                       // warps per CTA
  static constexpr int RING_BYTES = 64 * 1024;       // shared-memory ring per CTA
  static constexpr int NST = RING_BYTES / (NW * STAGE_BYTES) < 8 ? RING_BYTES / (NW * STAGE_BYTES) : 8;
  static constexpr int MAX_PART_TOKENS = 1024;       // longest partition the host plans
  static constexpr int SPEC = (MAX_PART_TOKENS / R + NW * 32 - 1) / (NW * 32);  // table reads per thread
  static constexpr int CLUSTER_MAX = 8;              // partitions merged inside one cluster, at most
  // mbarriers: one per ring stage, plus (cluster merge) the receiving barrier and one slot of
  // padding, so that the 16-byte row stage after them stays 16-byte aligned
  static constexpr int BARS = NW * NST;
  static constexpr int BARS_CLUSTER = NW * NST + 2;
  static_assert(NJ >= 1 && NJ <= CPR, "row split");
  static_assert(NST >= 1, "stages");
};

struct AttnParams {
  const __half* q;
  const __half* k;
  const __half* v;
  const int32_t* tables;
  const int32_t* lens;
  __half* out;
  float* ws_ml;  // [S, H, max_parts, 2] (m, l) in base-2 log domain
  float* ws_o;   // [S, H, max_parts, D] unnormalised partial outputs
  // shared-prefix groups (null for plain decode): sequences [group_start[g], group_start[g+1])
  // share their first prefix_lens[g] tokens; their partitions then cover tokens from
  // prefix_lens[g] on, written from slot part_base = 1 (slot 0 holds the prefix partial)
  const int32_t* group_start;
  const int32_t* prefix_lens;
  int num_groups;
  int part_base;
  int num_heads;
  int num_blocks;
  int max_blocks;
  int block_size;
  int part_tokens;
  int max_parts;
  float scale_log2;
  // append (null for plain decode): sequence s's new token, rows new_k / new_v [S, H, D], goes to
  // pool slot new_slot[s] (< 0: none) before the token attends, as reshape_and_cache would write it
  const __half* new_k;
  const __half* new_v;
  const int64_t* new_slot;
  // cluster merge: how long partition 0 waits for the others (RECV_WAIT_NS), and, for the
  // failure-detection test entry only, whether the other partitions skip their stores and arrivals
  // (so that the wait runs out on a phase nothing completes)
  unsigned long long recv_wait_ns;
  int test_skip_merge;
};

// First token of sequence s's own range: 0 for plain decode, else its group's shared-prefix
// length (binary search over the group starts; *first = the group's first sequence); -1 if s is
// in no group.
__device__ __forceinline__ int range_start(const AttnParams& p, int s, int* first = nullptr) {
  if (p.group_start == nullptr) return 0;
  int lo = 0, hi = p.num_groups;                       // find g with group_start[g] <= s < group_start[g+1]
  if (p.group_start[0] > s || p.group_start[hi] <= s) return -1;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.group_start[mid] <= s) lo = mid; else hi = mid;
  }
  if (first) *first = p.group_start[lo];
  if (p.group_start[lo + 1] - p.group_start[lo] < pkv::kMinSharedGroup) return 0;   // small group: no cascade
  return p.prefix_lens[lo];
}

// Sum of per-lane partial dots over the CPR lanes of a row, for NJ rows at once.
// On return every lane holds the full dot of reduced row jr = (lane % CPR) / DUP.
template <int NJ, int CPR>
__device__ __forceinline__ float butterfly_rows(float (&v)[NJ], int lane) {
#pragma unroll
  for (int n = NJ, mask = CPR / 2; n > 1; n /= 2, mask /= 2) {
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(FULL, send, mask);
    }
  }
  float r = v[0];
#pragma unroll
  for (int mask = CPR / NJ / 2; mask > 0; mask /= 2) r += __shfl_xor_sync(FULL, r, mask);
  return r;
}

__device__ __forceinline__ void dot8(const uint4& raw, const float (&qf)[8], float& acc) {
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(h2[e]);
    acc = fmaf(qf[2 * e], f.x, acc);
    acc = fmaf(qf[2 * e + 1], f.y, acc);
  }
}

__device__ __forceinline__ void axpy8(const uint4& raw, float p, float (&acc)[8]) {
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(h2[e]);
    acc[2 * e] = fmaf(p, f.x, acc[2 * e]);
    acc[2 * e + 1] = fmaf(p, f.y, acc[2 * e + 1]);
  }
}

// One chunk: update (m, l_lane, acc) with `valid` rows of K/V staged at ks/vs.
template <int D, int R, bool MASKED>
__device__ __forceinline__ void chunk_update(const unsigned char* ks, const unsigned char* vs, int valid,
                                             const float (&qf)[8], float& m, float& l_lane, float (&acc)[8],
                                             int lane) {
  using C = Cfg<D, R>;
  const int col = lane % C::CPR;
  const int grp = lane / C::CPR;
  float part[C::NJ];
#pragma unroll
  for (int j = 0; j < C::NJ; ++j) {
    const int row = j * C::RPI + grp;
    const uint4 raw = *reinterpret_cast<const uint4*>(ks + (row * D + col * 8) * 2);
    part[j] = 0.f;
    dot8(raw, qf, part[j]);
  }
  float x = butterfly_rows<C::NJ, C::CPR>(part, lane);
  const int rr = ((lane % C::CPR) / C::DUP) * C::RPI + grp;  // reduced row this lane holds
  if (MASKED && rr >= valid) x = -INFINITY;
  float cmax = x;
#pragma unroll
  for (int o = 16; o > 0; o /= 2) cmax = fmaxf(cmax, __shfl_xor_sync(FULL, cmax, o));
  const float m_new = fmaxf(m, cmax);
  const float alpha = exp2f(m - m_new);
  const float p = exp2f(x - m_new);
  l_lane = fmaf(l_lane, alpha, p);
  m = m_new;
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] *= alpha;
#pragma unroll
  for (int j = 0; j < C::NJ; ++j) {
    const int row = j * C::RPI + grp;
    const float pj = __shfl_sync(FULL, p, grp * C::CPR + j * C::DUP);
    if (!MASKED || row < valid) {
      const uint4 raw = *reinterpret_cast<const uint4*>(vs + (row * D + col * 8) * 2);
      axpy8(raw, pj, acc);
    }
  }
}

// APPEND: the fused new-token write of pkv_paged_attention_decode_append.  A compile-time switch:
// the plain decode kernel carries none of its registers or branches.
// CLUSTER: the partitions of one (sequence, head) form one thread-block cluster (the grid's x
// extent, max_parts <= CLUSTER_MAX, is the cluster's), and partition 0 merges the others' partial
// results, which they store into its shared memory: no workspace and no merge kernel.
constexpr unsigned long long RECV_WAIT_NS = 10000000000ull;  // 10 s: longer than any partition's bounded waits

template <int D, int R, bool APPEND, bool CLUSTER>
__global__ void __launch_bounds__(Cfg<D, R>::NW * 32, 3) paged_attention_partition_kernel(const AttnParams p) {
  using C = Cfg<D, R>;
  constexpr int NW = C::NW, NST = C::NST;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;                                                   // [NW][NST][K|V]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * NST * C::STAGE_BYTES);  // [NW][NST] (+ receive)
  float* comb = reinterpret_cast<float*>(bars + (CLUSTER ? C::BARS_CLUSTER : C::BARS));  // [NW][D + 2]
  // append only: the new K/V row of head h, handed from the warp that loads it to the one that
  // patches the staged chunk ([2 * D / 8] 16-byte vectors)
  uint4* row_stage = reinterpret_cast<uint4*>(comb + NW * (D + 2));
  // cluster only: partition 0 receives partition q's (o[D], m, l) in recv[q]
  float* recv = reinterpret_cast<float*>(row_stage + (APPEND ? 2 * C::CPR : 0));
  int64_t* chunk_off = reinterpret_cast<int64_t*>(recv + (CLUSTER ? C::CLUSTER_MAX * (D + 2) : 0));  // [chunks per part]
  const uint32_t recv_bar = smem_u32(&bars[NW * NST]);

  const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pkv::pdl_trigger();
  pkv::pdl_wait();  // inputs may come from the previous kernel on the stream
  const int B = p.block_size;
  const int H = p.num_heads;
  const size_t out_off = (static_cast<size_t>(s) * H + h) * D;
  // Append: the CTA of the last partition stores head h of the sequence's new K/V row at its slot,
  // as reshape_and_cache would before the call.  Which CTA that is depends on the context length,
  // so the slot and the row are read at once, beside the length, by every CTA: lanes 0..D/8-1 of
  // the last warp the K row, the next D/8 lanes the V row, one 16-byte vector each.  This CTA's
  // bulk copies may read the pool before or after the store, so where the table maps the
  // context's last position to the slot, the warp that owns that chunk writes the row over its
  // staged copy.  No other CTA reads the slot: other partitions end before the last position.
  const bool row_lane = lane < 2 * C::CPR;
  const bool row_is_v = lane >= C::CPR;
  const int row_col = row_is_v ? lane - C::CPR : lane;
  const bool row_loader = APPEND && warp == NW - 1 && row_lane;
  const int64_t slot = APPEND ? p.new_slot[s] : -1;
  uint4 new_row = make_uint4(0, 0, 0, 0);
  if (row_loader)
    new_row = *reinterpret_cast<const uint4*>((row_is_v ? p.new_v : p.new_k) + out_off + row_col * 8);
  // this lane's q slice, read now beside the length and the table; it is converted only after the
  // first bulk copies are issued, so its round trip overlaps theirs instead of delaying them
  const uint4 q_raw = *reinterpret_cast<const uint4*>(p.q + out_off + (lane % C::CPR) * 8);
  const int max_ctx = p.max_blocks * B;
  // Without groups every range starts at 0, so this partition's table entries are known before the
  // context length: they are read now, beside it, one per chunk (an index past the table row is not
  // read).  Entries past the context are dropped once the length is known.
  const bool spec = p.group_start == nullptr;
  int spec_phys[C::SPEC];
  if (spec) {
#pragma unroll
    for (int it = 0; it < C::SPEC; ++it) {
      const int i = tid + it * NW * 32;
      const int j = (part * (p.part_tokens / R) + i) / (B / R);
      spec_phys[it] = i < p.part_tokens / R && j < p.max_blocks
                          ? p.tables[static_cast<size_t>(s) * p.max_blocks + j] : -1;
    }
  }
  // this CTA's tokens: partition `part` of [start, ctx) (start = 0 unless a shared prefix precedes)
  const int ctx_full = p.lens[s];
  int first = s;
  const int start = range_start(p, s, &first);
  const bool bad_range = start < 0 || start % B != 0 || ctx_full <= start || ctx_full > max_ctx;
  const int ctx = ctx_full - start;                    // tokens of the range
  const int nparts = bad_range ? 1 : (ctx + p.part_tokens - 1) / p.part_tokens;
  if constexpr (CLUSTER) {
    // Partition 0 counts one arrival per thread of every other partition with tokens; its fence
    // publishes that initialisation and the cluster barrier orders it before any of them arrives.
    // Every thread of every CTA arrives here and waits once before it exits or reaches another
    // CTA's shared memory.
    if (part == 0 && tid == 0 && nparts > 1) {
      mbar_init(recv_bar, NW * 32 * (nparts - 1));
      fence_mbar_init();
    }
    cluster_arrive_relaxed();
    if (part >= nparts) {
      cluster_wait_acquire();
      return;
    }
  } else {
    if (part >= nparts) return;
  }
  const bool appends = APPEND && part == nparts - 1;
  const int64_t num_slots = static_cast<int64_t>(p.num_blocks) * B;
  const bool slot_ok = appends && slot >= 0 && slot < num_slots;
  auto store_row = [&]() {
    __half* pool = const_cast<__half*>(row_is_v ? p.v : p.k);
    *reinterpret_cast<uint4*>(pool + (((slot / B) * H + h) * B + slot % B) * D + row_col * 8) = new_row;
  };
  if (bad_range) {
    // an empty range (ctx = 0, or a context that is exactly its shared prefix) is no error; a
    // sequence in no group, a prefix that is not whole blocks or longer than the context is a
    // bad group layout
    if (tid == 0) {
      if (ctx_full > max_ctx || (p.group_start == nullptr && ctx_full < 0))
        record_error(PKV_DEV_BAD_CONTEXT_LEN);
      else if (start < 0 || start % B != 0 || ctx_full < start)
        record_error(PKV_DEV_PREFIX_MISMATCH);
    }
    if (appends && slot >= num_slots && tid == 0) record_error(PKV_DEV_BAD_SLOT);
    if (slot_ok && row_loader) store_row();
    if (p.part_base == 0) {
      for (int d = tid; d < D; d += NW * 32) p.out[out_off + d] = __float2half_rn(0.f);
    } else {
      const size_t w = (static_cast<size_t>(s) * H + h) * p.max_parts + p.part_base;
      for (int d = tid; d < D; d += NW * 32) p.ws_o[w * D + d] = 0.f;
      if (tid == 0) {
        p.ws_ml[2 * w] = -INFINITY;
        p.ws_ml[2 * w + 1] = 0.f;
      }
    }
    if constexpr (CLUSTER) cluster_wait_acquire();
    return;
  }

  const int chunks_per_block = B / R;
  const int chunks_per_part = p.part_tokens / R;
  const int total_chunks = (ctx + R - 1) / R;
  const int block0 = start / B;                        // first block of the range
  if (block0 > 0 && part == 0 && h == 0) {
    // the shared prefix is read once, through the group's first sequence: the others must map
    // their first blocks onto the same physical blocks
    int differs = 0;
    for (int j = tid; j < block0; j += NW * 32)
      differs |= p.tables[static_cast<size_t>(s) * p.max_blocks + j] != p.tables[static_cast<size_t>(first) * p.max_blocks + j];
    if (__syncthreads_or(differs) && tid == 0) record_error(PKV_DEV_PREFIX_MISMATCH);
  }
  const int c_begin = part * chunks_per_part;
  const int n_chunks = min(chunks_per_part, total_chunks - c_begin);

  // Table slice of this partition -> element offset of each chunk's K (and V) tile
  // (n_chunks <= MAX_PART_TOKENS / R: SPEC passes cover it).
  int bad = 0;
#pragma unroll
  for (int it = 0; it < C::SPEC; ++it) {
    const int i = tid + it * NW * 32;
    if (i < n_chunks) {
      const int c = c_begin + i;
      const int j = c / chunks_per_block;
      const int sub = c - j * chunks_per_block;
      const int phys = spec ? spec_phys[it] : p.tables[static_cast<size_t>(s) * p.max_blocks + block0 + j];
      if (phys < 0 || phys >= p.num_blocks) {
        bad = 1;
        chunk_off[i] = 0;
      } else {
        chunk_off[i] = ((static_cast<int64_t>(phys) * H + h) * B + sub * R) * D;
      }
    }
  }
  if (tid == 0) {
    for (int i = 0; i < NW * NST; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
  }
  if (appends && row_loader) {
    row_stage[lane] = new_row;
    if (slot_ok) store_row();
  }
  bad = __syncthreads_or(bad);
  // the appended row: which staged chunk and row it replaces, -1 = none
  int patch_chunk = -1, patch_row = 0;
  if (appends && slot >= num_slots && tid == 0) record_error(PKV_DEV_BAD_SLOT);
  if (slot_ok && !bad) {
    // element offset of the last position's row through the table (the last chunk's tile plus the
    // row within it) against the slot's: equal exactly when the table maps the position to it
    const int last_row = (ctx - 1) % R;
    if (chunk_off[n_chunks - 1] + static_cast<int64_t>(last_row) * D == (((slot / B) * H + h) * B + slot % B) * D) {
      patch_chunk = n_chunks - 1;
      patch_row = last_row;
    }
  }
  if (bad) {
    if (tid == 0) record_error(PKV_DEV_BAD_BLOCK_ID);
    if constexpr (!CLUSTER) {
      if (nparts == 1 && p.part_base == 0) {
        for (int d = tid; d < D; d += NW * 32) p.out[out_off + d] = __float2half_rn(0.f);
      } else {
        const size_t w = (static_cast<size_t>(s) * H + h) * p.max_parts + p.part_base + part;
        for (int d = tid; d < D; d += NW * 32) p.ws_o[w * D + d] = 0.f;
        if (tid == 0) {
          p.ws_ml[2 * w] = -INFINITY;
          p.ws_ml[2 * w + 1] = 0.f;
        }
      }
      return;
    }
    // in a cluster the partition still takes part in the merge, with an empty partial result
  }

  // Warp `warp` takes local chunks warp, warp + NW, ...
  const int my_n = (!bad && n_chunks > warp) ? (n_chunks - warp + NW - 1) / NW : 0;
  unsigned char* wring = ring + warp * NST * C::STAGE_BYTES;
  const uint32_t wbar = smem_u32(&bars[warp * NST]);
  const unsigned char* kbase = reinterpret_cast<const unsigned char*>(p.k);
  const unsigned char* vbase = reinterpret_cast<const unsigned char*>(p.v);

  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](int k) {
    const int stage = k % NST;
    const int i = warp + k * NW;
    const int64_t off = chunk_off[i] * 2;
    const uint32_t bar = wbar + stage * 8;
    const uint32_t dst = smem_u32(wring + stage * C::STAGE_BYTES);
    mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
    bulk_copy_g2s(dst, kbase + off, C::CHUNK_BYTES, bar, policy);
    bulk_copy_g2s(dst + C::CHUNK_BYTES, vbase + off, C::CHUNK_BYTES, bar, policy);
  };

  int issued = 0;
  if (lane == 0) {
    for (; issued < NST && issued < my_n; ++issued) issue(issued);
  }
  issued = __shfl_sync(FULL, issued, 0);

  // q slice of this lane, scaled into the base-2 log domain.
  float qf[8];
  {
    const __half2* h2 = reinterpret_cast<const __half2*>(&q_raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h2[e]);
      qf[2 * e] = f.x * p.scale_log2;
      qf[2 * e + 1] = f.y * p.scale_log2;
    }
  }

  float m = -INFINITY, l_lane = 0.f;
  float acc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] = 0.f;

  int k = 0;
  bool timed_out = false;
  for (; k < my_n; ++k) {
    const int stage = k % NST;
    const uint32_t parity = (k / NST) & 1;
    // every lane waits; the vote keeps the warp on one path even at the deadline
    if (!__all_sync(FULL, mbar_wait_bounded(wbar + stage * 8, parity))) {
      timed_out = true;
      break;
    }
    const unsigned char* ks = wring + stage * C::STAGE_BYTES;
    if (warp + k * NW == patch_chunk) {
      // the appended row replaces what the copy brought (this warp's stage, after it landed).  It is
      // the warp's last chunk, so no later bulk copy refills the stage and no proxy fence is needed.
      if (row_lane)
        *reinterpret_cast<uint4*>(const_cast<unsigned char*>(ks) + (row_is_v ? C::CHUNK_BYTES : 0) +
                                  (patch_row * D + row_col * 8) * 2) = row_stage[lane];
      __syncwarp();
    }
    const int c = c_begin + warp + k * NW;
    const int valid = min(R, ctx - c * R);
    if (valid == R)
      chunk_update<D, R, false>(ks, ks + C::CHUNK_BYTES, valid, qf, m, l_lane, acc, lane);
    else
      chunk_update<D, R, true>(ks, ks + C::CHUNK_BYTES, valid, qf, m, l_lane, acc, lane);
    __syncwarp();
    if (k + NST < my_n) {
      if (lane == 0) issue(k + NST);
      ++issued;
    }
  }
  if (timed_out) {
    if (lane == 0) record_error(PKV_DEV_WAIT_TIMEOUT);
    // let this warp's outstanding copies land before the CTA's shared memory is released
    for (int kk = k + 1; kk < issued; ++kk) mbar_wait_bounded(wbar + (kk % NST) * 8, (kk / NST) & 1);
  }

  // Per-warp results: sum acc over the row groups, l over distinct rows.
#pragma unroll
  for (int o = C::CPR; o < 32; o *= 2) {
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(FULL, acc[c], o);
  }
  float l = (lane % C::DUP) == 0 ? l_lane : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o /= 2) l += __shfl_xor_sync(FULL, l, o);

  float* wcomb = comb + warp * (D + 2);
  if (lane < C::CPR) {
#pragma unroll
    for (int c = 0; c < 8; ++c) wcomb[lane * 8 + c] = acc[c];
  }
  if (lane == 0) {
    wcomb[D] = m;
    wcomb[D + 1] = l;
  }
  __syncthreads();

  // this CTA's (M, L); a warp without tokens (m = -inf) weighs nothing
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, comb[w * (D + 2) + D]);
  float L = 0.f;
  float wgt[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const float mw = comb[w * (D + 2) + D];
    wgt[w] = mw == -INFINITY ? 0.f : exp2f(mw - M);
    L = fmaf(comb[w * (D + 2) + D + 1], wgt[w], L);
  }
  if (nparts == 1 && p.part_base == 0) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int d = tid; d < D; d += NW * 32) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) o = fmaf(comb[w * (D + 2) + d], wgt[w], o);
      p.out[out_off + d] = __float2half_rn(o * inv);
    }
    if constexpr (CLUSTER) cluster_wait_acquire();
  } else if constexpr (!CLUSTER) {
    const size_t w0 = (static_cast<size_t>(s) * H + h) * p.max_parts + p.part_base + part;
    for (int d = tid; d < D; d += NW * 32) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) o = fmaf(comb[w * (D + 2) + d], wgt[w], o);
      p.ws_o[w0 * D + d] = o;
    }
    if (tid == 0) {
      p.ws_ml[2 * w0] = M;
      p.ws_ml[2 * w0 + 1] = L;
    }
  } else {
    // the merge inside the cluster: m = max m_q, l = sum l_q 2^(m_q - m), o = sum o_q 2^(m_q - m) / l
    cluster_wait_acquire();                            // partition 0's receiving barrier is set up
    if (part != 0 && p.test_skip_merge) return;        // failure-detection test: nothing arrives
    if (part != 0) {
      const uint32_t dst = map_to_rank(smem_u32(recv + part * (D + 2)), 0);
      for (int d = tid; d < D; d += NW * 32) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) o = fmaf(comb[w * (D + 2) + d], wgt[w], o);
        st_cluster_f32(dst + 4u * d, o);
      }
      if (tid == 0) {
        st_cluster_f32(dst + 4u * D, M);
        st_cluster_f32(dst + 4u * (D + 1), L);
      }
      mbar_arrive_remote(map_to_rank(recv_bar, 0));    // every thread, after its own stores
      return;
    }
    // partition 0 stays until every other partition's threads have arrived: none of them may
    // store into its shared memory after it has exited
    if (!mbar_wait_cluster_bounded(recv_bar, 0, p.recv_wait_ns) && tid == 0) record_error(PKV_DEV_WAIT_TIMEOUT);
    float Mx = M;
    for (int q = 1; q < nparts; ++q) Mx = fmaxf(Mx, recv[q * (D + 2) + D]);
    const float w_own = M == -INFINITY ? 0.f : exp2f(M - Mx);
    float Lx = L * w_own;
    for (int q = 1; q < nparts; ++q) {
      const float mq = recv[q * (D + 2) + D];
      Lx = fmaf(recv[q * (D + 2) + D + 1], mq == -INFINITY ? 0.f : exp2f(mq - Mx), Lx);
    }
    const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
    for (int d = tid; d < D; d += NW * 32) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) o = fmaf(comb[w * (D + 2) + d], wgt[w], o);
      o *= w_own;
      for (int q = 1; q < nparts; ++q) {
        const float mq = recv[q * (D + 2) + D];
        o = fmaf(recv[q * (D + 2) + d], mq == -INFINITY ? 0.f : exp2f(mq - Mx), o);
      }
      p.out[out_off + d] = __float2half_rn(o * inv);
    }
  }
}

// Merge the partitions of every (sequence, head) that has more than one: one
// warp per (sequence, head); lanes read the partitions' (m, l) in parallel and
// each lane owns D/32 output columns, read as one vector per partition.
template <int D>
__global__ void __launch_bounds__(128) paged_attention_merge_kernel(const AttnParams p) {
  pkv::pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 4 + warp, s = blockIdx.y;
  if (h >= p.num_heads) return;
  const size_t w0 = (static_cast<size_t>(s) * p.num_heads + h) * p.max_parts;
  // The (m, l) of slots 0..31 are loaded together with the context length, before the slot count
  // is known (every slot below max_parts is inside the workspace; the ones past the count are
  // dropped below), so the chain of dependent memory round trips stays short.
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < p.max_parts) ml = *reinterpret_cast<const float2*>(p.ws_ml + 2 * (w0 + lane));
  const int ctx = p.lens[s];
  const int start = range_start(p, s);
  const int max_ctx = p.max_blocks * p.block_size;
  const bool bad_range = start < 0 || start % p.block_size != 0 || ctx <= start || ctx > max_ctx;
  // slots: the shared-prefix partial (if any) and the partitions of [start, ctx)
  const int nparts = p.part_base + (bad_range ? 1 : (ctx - start + p.part_tokens - 1) / p.part_tokens);
  if (nparts <= 1) return;
  constexpr int V = D / 32;
  float acc[V];
#pragma unroll
  for (int c = 0; c < V; ++c) acc[c] = 0.f;
  float M = -INFINITY, L = 0.f;
  // slots in batches of 32 (one per lane for m and l); more than one batch only past 32 slots
  for (int base = 0; base < nparts; base += 32) {
    const int i = base + lane;
    if (base > 0) ml = i < nparts ? *reinterpret_cast<const float2*>(p.ws_ml + 2 * (w0 + i)) : make_float2(-INFINITY, 0.f);
    if (i >= nparts) ml = make_float2(-INFINITY, 0.f);
    float Mb = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o /= 2) Mb = fmaxf(Mb, __shfl_xor_sync(FULL, Mb, o));
    // fold the batch into the running (M, L, acc): rescale what came before if the max moved
    const float Mn = fmaxf(M, Mb);
    const float carry = M == -INFINITY ? 0.f : exp2f(M - Mn);
    L *= carry;
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] *= carry;
    M = Mn;
    const float wi = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
    L = fmaf(ml.y, wi, L);
    const int n = min(32, nparts - base);
    // eight slots' partial outputs in flight at a time
    for (int j0 = 0; j0 < n; j0 += 8) {
      float4 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j0 + u < n) {
          const float* src = p.ws_o + (w0 + base + j0 + u) * D + lane * V;
          if constexpr (V == 4) {
            x[u] = *reinterpret_cast<const float4*>(src);
          } else {
            const float2 t = *reinterpret_cast<const float2*>(src);
            x[u] = make_float4(t.x, t.y, 0.f, 0.f);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float wj = __shfl_sync(FULL, wi, (j0 + u) & 31);
        if (j0 + u < n) {
          acc[0] = fmaf(wj, x[u].x, acc[0]);
          acc[1] = fmaf(wj, x[u].y, acc[1]);
          if constexpr (V == 4) {
            acc[2] = fmaf(wj, x[u].z, acc[2]);
            acc[3] = fmaf(wj, x[u].w, acc[3]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o /= 2) L += __shfl_xor_sync(FULL, L, o);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __half* dst = p.out + (static_cast<size_t>(s) * p.num_heads + h) * D + lane * V;
#pragma unroll
  for (int c = 0; c < V; c += 2) {
    *reinterpret_cast<__half2*>(dst + c) = __floats2half2_rn(acc[c] * inv, acc[c + 1] * inv);
  }
}

// Floats of the (m, l) block of the workspace, padded so the partial outputs start 16-byte aligned.
__host__ __device__ constexpr size_t ws_ml_floats(size_t pairs) { return (pairs * 2 + 3) / 4 * 4; }

// ---- host side ---------------------------------------------------------------------------------
constexpr int kMinPartTokens = 128;
constexpr int kMaxPartTokens = 1024;
static_assert(kMaxPartTokens == Cfg<128, 16>::MAX_PART_TOKENS, "the kernel's table pass covers the longest partition");

template <int D, int R>
constexpr size_t smem_bytes(int part_tokens, bool append, bool cluster) {
  using C = Cfg<D, R>;
  return static_cast<size_t>(C::NW) * C::NST * C::STAGE_BYTES +
         (cluster ? C::BARS_CLUSTER : C::BARS) * 8 +
         C::NW * (D + 2) * sizeof(float) + (append ? 2 * C::CPR * 16 : 0) +
         (cluster ? C::CLUSTER_MAX * (D + 2) * sizeof(float) : 0) +
         static_cast<size_t>(part_tokens / R) * sizeof(int64_t);
}

int device_sms(int dev) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> g(mu);
  if (dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

template <int D, int R, bool APPEND, bool CLUSTER>
cudaError_t set_smem(int part_tokens) {
  return cudaFuncSetAttribute(paged_attention_partition_kernel<D, R, APPEND, CLUSTER>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem_bytes<D, R>(part_tokens, APPEND, CLUSTER)));
}

template <int D, int R>
cudaError_t prepare_kernel(int dev) {
  static std::mutex mu;
  static bool done[64] = {false};
  std::lock_guard<std::mutex> g(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = set_smem<D, R, false, false>(kMaxPartTokens);
  if (e == cudaSuccess) e = set_smem<D, R, true, false>(kMaxPartTokens);
  if (e == cudaSuccess) e = set_smem<D, R, false, true>(kMaxPartTokens);
  if (e == cudaSuccess) e = set_smem<D, R, true, true>(kMaxPartTokens);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

int choose_part_tokens(int num_seqs, int num_heads, int max_ctx, int sms) {
  // The longest partition that still gives every SM a CTA: fewer, longer K/V streams per CTA
  // (fewer pipeline fills, less merge traffic) until the grid would leave SMs idle.  Measured with
  // L2 flushed between steps, ctx 2048, 40 heads: one sequence 26.4 us at 512 tokens (160 CTAs)
  // against 29.7 us at 128 and 30.1 us at 1024; four sequences 46.8 us at 1024 against 48.9 at 256.
  const long long target = sms;
  for (int pt : {1024, 512, 256}) {
    const long long ctas = static_cast<long long>(num_seqs) * num_heads * ((max_ctx + pt - 1) / pt);
    if (ctas >= target) return pt;
  }
  return kMinPartTokens;
}

// Whether a plain decode call merges its partitions inside thread-block clusters (one cluster per
// (sequence, head), partition 0 merging) rather than through the workspace and a merge kernel:
// when every (sequence, head) has at most CLUSTER_MAX partitions and the grid fits in one wave of
// resident CTAs (kResidentPerSm per SM).  There the merge kernel's launch and its dependency on the
// whole grid are a visible share of the call (one 2048-token sequence: 18.5 against 19.8 us);
// on grids of many waves the clusters' co-scheduling costs more than the merge kernel (the
// 64-sequence batch took 213 us against 194, 256 shared-prefix requests 818 against 535).
constexpr int kResidentPerSm = 3;                 // CTAs of the partition kernel per SM (launch bounds)
bool cluster_merge(int num_seqs, int num_heads, int max_parts, int sms) {
  const long long ctas = static_cast<long long>(num_seqs) * num_heads * max_parts;
  return max_parts > 1 && max_parts <= Cfg<128, 16>::CLUSTER_MAX && ctas <= static_cast<long long>(kResidentPerSm) * sms;
}

// join: if not null, the merge waits for this event (the shared-prefix product on a side stream).
template <int D, int R>
int launch(AttnParams p, int num_seqs, int part_tokens, size_t ws_bytes, void* ws, cudaStream_t st,
           cudaEvent_t join = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = prepare_kernel<D, R>(dev);
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged attention setup: %s", cudaGetErrorString(e));
  if (part_tokens > kMaxPartTokens || part_tokens % R != 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "paged attention: partition of %d tokens", part_tokens);
  const int max_ctx = p.max_blocks * p.block_size;
  p.part_tokens = part_tokens;
  p.max_parts = (max_ctx + part_tokens - 1) / part_tokens + p.part_base;
  const bool cluster = p.part_base == 0 && cluster_merge(num_seqs, p.num_heads, p.max_parts, device_sms(dev));
  if (p.max_parts > 1 && !cluster) {
    const size_t pairs = static_cast<size_t>(num_seqs) * p.num_heads * p.max_parts;
    const size_t need = (ws_ml_floats(pairs) + pairs * D) * sizeof(float);
    if (ws == nullptr || ws_bytes < need)
      return pkv::fail(PKV_ERR_WORKSPACE, "paged attention: workspace of %zu bytes needed, %zu given", need,
                       ws == nullptr ? static_cast<size_t>(0) : ws_bytes);
    p.ws_ml = static_cast<float*>(ws);
    p.ws_o = p.ws_ml + ws_ml_floats(pairs);
  }
  dim3 grid(p.max_parts, p.num_heads, num_seqs);
  const dim3 block(Cfg<D, R>::NW * 32);
  const bool append = p.new_slot != nullptr;
  const size_t smem = smem_bytes<D, R>(part_tokens, append, cluster);
  if (cluster)
    e = append ? pkv::launch_pdl_cluster(paged_attention_partition_kernel<D, R, true, true>, grid, block, smem, st,
                                         p.max_parts, p)
               : pkv::launch_pdl_cluster(paged_attention_partition_kernel<D, R, false, true>, grid, block, smem, st,
                                         p.max_parts, p);
  else
    e = append ? pkv::launch_pdl(paged_attention_partition_kernel<D, R, true, false>, grid, block, smem, st, p)
               : pkv::launch_pdl(paged_attention_partition_kernel<D, R, false, false>, grid, block, smem, st, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged attention launch: %s", cudaGetErrorString(e));
  if (p.max_parts > 1 && !cluster) {
    if (join != nullptr) {
      e = cudaStreamWaitEvent(st, join, 0);
      if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged attention join: %s", cudaGetErrorString(e));
    }
    e = pkv::launch_pdl(paged_attention_merge_kernel<D>, dim3((p.num_heads + 3) / 4, num_seqs), dim3(128), 0, st,
                        p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged attention merge launch: %s", cudaGetErrorString(e));
  }
  return PKV_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Per device: a non-blocking side stream and fork/join events for the shared-prefix product, which
// needs nothing from the split-K partitions and so runs beside them (a few dozen CTAs next to
// thousands).  Callers of the shared-prefix entry hold side_mutex() while they enqueue, so two host
// threads never interleave records and waits on the same events.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex& side_mutex() {
  static std::mutex mu;
  return mu;
}
// Under side_mutex(): the device's side stream, created on first use.
int side_stream(int dev, SideStream** out) {
  static SideStream side[64];
  if (dev < 0 || dev >= 64) return pkv::fail(PKV_ERR_UNSUPPORTED, "shared-prefix attention: device ordinal %d above 63", dev);
  SideStream& sd = side[dev];
  if (sd.stream == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      sd = SideStream{};
      return pkv::fail(PKV_ERR_CUDA, "shared-prefix attention: side stream: %s", cudaGetErrorString(e));
    }
  }
  *out = &sd;
  return PKV_OK;
}

// pkv_paged_attention_decode, and with new_slot set pkv_paged_attention_decode_append (fn names
// the entry in messages)
int decode_entry(const char* fn, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_heads,
                 int head_dim, int num_blocks, int max_blocks_per_seq, float scale, int block_size, uint16_t* out,
                 void* workspace, size_t workspace_bytes, void* stream, const uint16_t* new_k,
                 const uint16_t* new_v, const int64_t* new_slot, unsigned long long recv_wait_ns = RECV_WAIT_NS,
                 int test_skip_merge = 0) {
  if (num_seqs < 0 || num_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
    return pkv::fail(PKV_ERR_INVALID_ARG,
                     "%s: num_seqs=%d num_heads=%d num_blocks=%d max_blocks_per_seq=%d", fn,
                     num_seqs, num_heads, num_blocks, max_blocks_per_seq);
  if (head_dim != 64 && head_dim != 128)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "%s: head_dim %d not in {64, 128}", fn, head_dim);
  if (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "%s: block_size %d not in {4, 8, 16, 32}", fn,
                     block_size);
  if (num_seqs == 0) {
    pkv::clear_error();
    return PKV_OK;
  }
  if (num_seqs > 65535 || num_heads > 65535)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "%s: num_seqs/num_heads above 65535", fn);
  if (static_cast<long long>(max_blocks_per_seq) * block_size > (1LL << 30))
    return pkv::fail(PKV_ERR_UNSUPPORTED, "%s: context capacity above 2^30 tokens", fn);
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return pkv::fail(PKV_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return pkv::fail(PKV_ERR_INVALID_ARG, "%s: q, caches, out, workspace must be 16-byte aligned", fn);
  if (!std::isfinite(scale)) return pkv::fail(PKV_ERR_INVALID_ARG, "%s: scale not finite", fn);

  AttnParams p{};
  p.recv_wait_ns = recv_wait_ns;
  p.test_skip_merge = test_skip_merge;
  p.new_k = reinterpret_cast<const __half*>(new_k);
  p.new_v = reinterpret_cast<const __half*>(new_v);
  p.new_slot = new_slot;
  p.q = reinterpret_cast<const __half*>(q);
  p.k = reinterpret_cast<const __half*>(k_cache);
  p.v = reinterpret_cast<const __half*>(v_cache);
  p.tables = block_tables;
  p.lens = context_lens;
  p.out = reinterpret_cast<__half*>(out);
  p.num_heads = num_heads;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = block_size;
  p.scale_log2 = scale * 1.4426950408889634f;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const int pt = choose_part_tokens(num_seqs, num_heads, max_blocks_per_seq * block_size, device_sms(dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc;
  // chunk rows R = min(B, 16): a block of 32 rows is read as two chunks
  if (head_dim == 128) {
    rc = block_size == 4   ? launch<128, 4>(p, num_seqs, pt, workspace_bytes, workspace, st)
         : block_size == 8 ? launch<128, 8>(p, num_seqs, pt, workspace_bytes, workspace, st)
                           : launch<128, 16>(p, num_seqs, pt, workspace_bytes, workspace, st);
  } else {
    rc = block_size == 4   ? launch<64, 4>(p, num_seqs, pt, workspace_bytes, workspace, st)
         : block_size == 8 ? launch<64, 8>(p, num_seqs, pt, workspace_bytes, workspace, st)
                           : launch<64, 16>(p, num_seqs, pt, workspace_bytes, workspace, st);
  }
  if (rc == PKV_OK) pkv::clear_error();
  return rc;
}

}  // namespace

namespace pkv {
int read_device_error_attention(int reset, int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_error_attention, sizeof(int));
  if (e == cudaSuccess && reset && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error_attention, &zero, sizeof(int));
  }
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "reading the attention check word: %s", cudaGetErrorString(e));
  *code = v;
  return PKV_OK;
}
}  // namespace pkv

extern "C" {

size_t pkv_paged_attention_workspace_size(int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq,
                                          int block_size) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0) return 0;
  const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
  const long long parts = (max_ctx + kMinPartTokens - 1) / kMinPartTokens;
  if (parts <= 1) return 0;
  const size_t pairs = static_cast<size_t>(num_seqs) * num_heads * parts;
  return (ws_ml_floats(pairs) + pairs * head_dim) * sizeof(float);
}

int pkv_paged_attention_plan(int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq, int block_size,
                             int* part_tokens, int* num_kernels) {
  if (num_seqs < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || !part_tokens || !num_kernels)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_plan: bad argument");
  if ((head_dim != 64 && head_dim != 128) ||
      (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32))
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_plan: head_dim %d / block_size %d", head_dim,
                     block_size);
  if (static_cast<long long>(max_blocks_per_seq) * block_size > (1LL << 30))
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_plan: context capacity above 2^30 tokens");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const int max_ctx = max_blocks_per_seq * block_size;
  const int pt = choose_part_tokens(num_seqs, num_heads, max_ctx, device_sms(dev));
  const int max_parts = (max_ctx + pt - 1) / pt;
  *part_tokens = pt;
  *num_kernels = num_seqs == 0 ? 0 : (max_parts > 1 && !cluster_merge(num_seqs, num_heads, max_parts, device_sms(dev)) ? 2 : 1);
  pkv::clear_error();
  return PKV_OK;
}

int pkv_paged_attention_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                               int num_heads, int head_dim, int num_blocks, int max_blocks_per_seq, float scale,
                               int block_size, uint16_t* out, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return decode_entry("pkv_paged_attention_decode", q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                      num_heads, head_dim, num_blocks, max_blocks_per_seq, scale, block_size, out, workspace,
                      workspace_bytes, stream, nullptr, nullptr, nullptr);
}

int pkv_paged_attention_decode_append(const uint16_t* q, const uint16_t* key, const uint16_t* value,
                                      const int64_t* slot_mapping, uint16_t* k_cache, uint16_t* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                      int num_heads, int head_dim, int num_blocks, int max_blocks_per_seq,
                                      float scale, int block_size, uint16_t* out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (num_seqs > 0 && (!key || !value || !slot_mapping))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_decode_append: null key, value or slot_mapping");
  if (num_seqs > 0 && (!aligned16(key) || !aligned16(value)))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_decode_append: key and value must be 16-byte aligned");
  return decode_entry("pkv_paged_attention_decode_append", q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                      num_heads, head_dim, num_blocks, max_blocks_per_seq, scale, block_size, out, workspace,
                      workspace_bytes, stream, key, value, slot_mapping);
}

int pkv_test_cluster_merge_timeout(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                   int num_heads, int head_dim, int num_blocks, int max_blocks_per_seq, float scale,
                                   int block_size, uint16_t* out, int wait_ms, void* stream) {
  int part_tokens = 0, kernels = 0;
  int rc = pkv_paged_attention_plan(num_seqs, num_heads, head_dim, max_blocks_per_seq, block_size, &part_tokens,
                                    &kernels);
  if (rc != PKV_OK) return rc;
  if (num_seqs <= 0 || kernels != 1 || static_cast<long long>(max_blocks_per_seq) * block_size <= part_tokens)
    return pkv::fail(PKV_ERR_UNSUPPORTED,
                     "pkv_test_cluster_merge_timeout: these sizes do not merge partitions inside clusters");
  if (wait_ms < 1 || wait_ms > 2000)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_test_cluster_merge_timeout: wait_ms %d outside [1, 2000]", wait_ms);
  return decode_entry("pkv_test_cluster_merge_timeout", q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                      num_heads, head_dim, num_blocks, max_blocks_per_seq, scale, block_size, out, nullptr, 0,
                      stream, nullptr, nullptr, nullptr, 1000000ull * static_cast<unsigned long long>(wait_ms), 1);
}

size_t pkv_paged_attention_shared_prefix_workspace_size(int num_seqs, int num_heads, int head_dim,
                                                        int max_blocks_per_seq, int block_size) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0) return 0;
  const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
  const long long parts = (max_ctx + kMinPartTokens - 1) / kMinPartTokens + 1;   // + the prefix slot
  const size_t pairs = static_cast<size_t>(num_seqs) * num_heads * parts;
  return (ws_ml_floats(pairs) + pairs * head_dim) * sizeof(float);
}

int pkv_paged_attention_decode_shared_prefix(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                             const int32_t* block_tables, const int32_t* context_lens,
                                             const int32_t* group_start, const int32_t* prefix_lens, int num_groups,
                                             int max_group_size, int num_seqs, int num_heads, int head_dim,
                                             int num_blocks, int max_blocks_per_seq, float scale, int block_size,
                                             uint16_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (num_seqs < 0 || num_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || num_groups <= 0 ||
      max_group_size <= 0)
    return pkv::fail(PKV_ERR_INVALID_ARG,
                     "pkv_paged_attention_decode_shared_prefix: num_seqs=%d num_heads=%d num_blocks=%d "
                     "max_blocks_per_seq=%d num_groups=%d max_group_size=%d",
                     num_seqs, num_heads, num_blocks, max_blocks_per_seq, num_groups, max_group_size);
  if (head_dim != 64 && head_dim != 128)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_decode_shared_prefix: head_dim %d not in {64, 128}",
                     head_dim);
  if (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32)
    return pkv::fail(PKV_ERR_UNSUPPORTED,
                     "pkv_paged_attention_decode_shared_prefix: block_size %d not in {4, 8, 16, 32}", block_size);
  if (num_seqs == 0) {
    pkv::clear_error();
    return PKV_OK;
  }
  if (num_seqs > 65535 || num_heads > 65535 || num_groups > 65535)
    return pkv::fail(PKV_ERR_UNSUPPORTED,
                     "pkv_paged_attention_decode_shared_prefix: num_seqs/num_heads/num_groups above 65535");
  if (static_cast<long long>(max_blocks_per_seq) * block_size > (1LL << 30))
    return pkv::fail(PKV_ERR_UNSUPPORTED,
                     "pkv_paged_attention_decode_shared_prefix: context capacity above 2^30 tokens");
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !group_start || !prefix_lens || !out ||
      !workspace)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_decode_shared_prefix: null pointer");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
    return pkv::fail(PKV_ERR_INVALID_ARG,
                     "pkv_paged_attention_decode_shared_prefix: q, caches, out, workspace must be 16-byte aligned");
  if (!std::isfinite(scale) || !(scale > 0.f))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_decode_shared_prefix: scale must be finite and positive");

  AttnParams p{};
  p.recv_wait_ns = RECV_WAIT_NS;
  p.q = reinterpret_cast<const __half*>(q);
  p.k = reinterpret_cast<const __half*>(k_cache);
  p.v = reinterpret_cast<const __half*>(v_cache);
  p.tables = block_tables;
  p.lens = context_lens;
  p.out = reinterpret_cast<__half*>(out);
  p.num_heads = num_heads;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = block_size;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.group_start = group_start;
  p.prefix_lens = prefix_lens;
  p.num_groups = num_groups;
  p.part_base = 1;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const int max_ctx = max_blocks_per_seq * block_size;
  const int pt = choose_part_tokens(num_seqs, num_heads, max_ctx, device_sms(dev));
  const int max_parts = (max_ctx + pt - 1) / pt + 1;
  const size_t pairs = static_cast<size_t>(num_seqs) * num_heads * max_parts;
  const size_t need = (ws_ml_floats(pairs) + pairs * head_dim) * sizeof(float);
  if (workspace_bytes < need)
    return pkv::fail(PKV_ERR_WORKSPACE, "pkv_paged_attention_decode_shared_prefix: workspace of %zu bytes needed, %zu given",
                     need, workspace_bytes);
  if (max_group_size < pkv::kMinSharedGroup)        // every group is small: plain decode
    return pkv_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, head_dim,
                                      num_blocks, max_blocks_per_seq, scale, block_size, out, workspace,
                                      workspace_bytes, stream);
  float* ws_ml = static_cast<float*>(workspace);
  float* ws_o = ws_ml + ws_ml_floats(pairs);
  // the prefix partials (slot 0) on the side stream, forked from and joined back to the caller's
  // stream; the partitions of each [prefix_len, ctx) on the caller's stream; the merge after both
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> guard(side_mutex());
  SideStream* side = nullptr;
  int rc = side_stream(dev, &side);
  if (rc != PKV_OK) return rc;
  cudaError_t e = cudaEventRecord(side->fork, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "shared-prefix attention: fork: %s", cudaGetErrorString(e));
  rc = pkv::launch_prefix_partials(q, k_cache, v_cache, block_tables, group_start, prefix_lens, num_groups,
                                   max_group_size, num_seqs, num_heads, head_dim, num_blocks, max_blocks_per_seq,
                                   scale, block_size, ws_ml, ws_o, max_parts, side->stream);
  if (rc == PKV_OK) {
    e = cudaEventRecord(side->join, side->stream);
    if (e != cudaSuccess) rc = pkv::fail(PKV_ERR_CUDA, "shared-prefix attention: join: %s", cudaGetErrorString(e));
  }
  if (rc != PKV_OK) {
    cudaStreamWaitEvent(st, side->fork, 0);      // leave the caller's stream consistent
    return rc;
  }
  if (head_dim == 128) {
    rc = block_size == 4   ? launch<128, 4>(p, num_seqs, pt, workspace_bytes, workspace, st, side->join)
         : block_size == 8 ? launch<128, 8>(p, num_seqs, pt, workspace_bytes, workspace, st, side->join)
                           : launch<128, 16>(p, num_seqs, pt, workspace_bytes, workspace, st, side->join);
  } else {
    rc = block_size == 4   ? launch<64, 4>(p, num_seqs, pt, workspace_bytes, workspace, st, side->join)
         : block_size == 8 ? launch<64, 8>(p, num_seqs, pt, workspace_bytes, workspace, st, side->join)
                           : launch<64, 16>(p, num_seqs, pt, workspace_bytes, workspace, st, side->join);
  }
  if (rc != PKV_OK) cudaStreamWaitEvent(st, side->join, 0);   // join even when a launch failed
  if (rc == PKV_OK) pkv::clear_error();
  return rc;
}

}  // extern "C"

// ---- decode attention with library-owned scratch ------------------------------------------------
//
// Some callers cannot allocate device memory for the workspace: a plain C host
// program or a plugin that has no device allocator of its own, an engine that
// has already reserved all device memory for its block pools, or a path that
// must not pay for the device-wide synchronisation cudaMalloc/cudaFree imply.
// For them this entry point keeps the split-over-context scratch in a fixed
// array inside the library instead.
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;  // 16 MiB, held on every device that loads the library

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Driver calls that name the caller's current context, reached through the runtime's entry-point
// query so that the library does not link libcuda itself.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (never reused within the process, unlike the
// context handle, which a context created after cudaDeviceReset may share).  0 on failure.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_workspace in the caller's current context on `dev`.  The lookup
// (cudaGetSymbolAddress, with the device current) runs once per context: the first call on a
// device, and again after cudaDeviceReset or under another context (a plugin's own cuCtxCreate),
// since the array then lives at another address.  nullptr with the status in *rc on failure.
void* static_workspace_address(int dev, int* rc) {
  static std::mutex mu;
  static unsigned long long ctx_of[64] = {0};
  static void* addr[64] = {nullptr};
  std::lock_guard<std::mutex> g(mu);
  if (dev < 0 || dev >= 64) {
    *rc = pkv::fail(PKV_ERR_UNSUPPORTED, "static-workspace attention: device ordinal %d above 63", dev);
    return nullptr;
  }
  const unsigned long long ctx = current_context_id();
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess || ptr == nullptr) {
      addr[dev] = nullptr;
      *rc = pkv::fail(PKV_ERR_CUDA, "static-workspace attention: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      return nullptr;
    }
    addr[dev] = ptr;
    ctx_of[dev] = ctx;
  }
  *rc = PKV_OK;
  return addr[dev];
}

}  // namespace

extern "C" {

size_t pkv_paged_attention_static_workspace_bytes(void) { return kStaticWorkspaceBytes; }

int pkv_paged_attention_decode_static_workspace(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                int num_seqs, int num_heads, int head_dim, int num_blocks,
                                                int max_blocks_per_seq, float scale, int block_size, uint16_t* out,
                                                void* stream) {
  if (num_seqs <= 0 || num_heads <= 0 || max_blocks_per_seq <= 0)
    return pkv_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                                      head_dim, num_blocks, max_blocks_per_seq, scale, block_size, out, nullptr, 0,
                                      stream);
  if (static_cast<long long>(max_blocks_per_seq) * block_size > (1LL << 30))
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_decode_static_workspace: context capacity above 2^30 tokens");
  int part_tokens = 0, kernels = 0;
  int rc = pkv_paged_attention_plan(num_seqs, num_heads, head_dim, max_blocks_per_seq, block_size, &part_tokens,
                                    &kernels);
  if (rc != PKV_OK) return rc;
  const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
  const long long parts = (max_ctx + part_tokens - 1) / part_tokens;
  const size_t pairs = static_cast<size_t>(num_seqs) * num_heads * parts;
  // the plan's scratch: none for one partition, or when the partitions merge inside clusters
  const unsigned long long need = kernels == 2 ? (ws_ml_floats(pairs) + pairs * head_dim) * sizeof(float) : 0;
  if (need > kStaticWorkspaceBytes)
    return pkv::fail(PKV_ERR_WORKSPACE,
                     "pkv_paged_attention_decode_static_workspace: this batch needs %llu bytes of scratch, above "
                     "the library's fixed %zu; use pkv_paged_attention_decode with a caller workspace",
                     need, kStaticWorkspaceBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return pkv::fail(PKV_ERR_CUDA, "pkv_paged_attention_decode_static_workspace: cudaGetDevice: %s",
                     cudaGetErrorString(e));
  void* ws = static_workspace_address(dev, &rc);
  if (!ws) return rc;
  return pkv_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, head_dim,
                                    num_blocks, max_blocks_per_seq, scale, block_size, out, ws,
                                    kStaticWorkspaceBytes, stream);
}

}  // extern "C"
