// Paged prefill attention for sm_103a: the new tokens of each sequence (the task
// input) attend over the sequence's cached context plus, causally, themselves,
// with K/V read through the block table.
//
// What is computed ([guide] "vLLM / PagedAttention (SOSP 2023)", section 04: a
// request maps its first logical blocks onto cached prefix blocks and the prompt
// phase runs only over the task input; [note] "vLLM / PagedAttention -- 把 LLM 服务
// 的瓶颈从显存碎片里救出来", 关键设计 1, first equation, summed to t = i): new token i of
// sequence s, at position p = ctx_s - n_s + i, gets
// o = sum_{t <= p} softmax_t(scale * q.k_t) v_t.
//
// Design: a dense contraction, so it runs on the tensor cores (mma.sync
// m16n8k16, fp16 inputs, fp32 accumulation).  One CTA (4 warps) owns 64 new
// tokens of one (sequence, head); each warp owns 16 of them.  Key tiles of 64
// positions are gathered block by block through the table with 16-byte
// cp.async copies into XOR-swizzled shared memory (conflict-free ldmatrix),
// double-buffered.  S = Q K^T and O += P V per tile with an online softmax in
// base 2; P is rounded to fp16 for the second product, as flash attention does.
// Key rows past the context are zero-filled (never read), so stale NaN/Inf in
// unfilled slots cannot reach a product.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "launch.cuh"
#include "pkv_internal.h"

namespace {

__device__ int g_dev_error_prefill = 0;
__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_dev_error_prefill, 0, code); }

constexpr unsigned FULL = 0xffffffffu;
constexpr int BM = 64;   // new tokens per CTA
constexpr int BN = 64;   // key positions per tile
constexpr int NWARP = 4;

struct PrefillParams {
  const __half* q;
  const __half* k;
  const __half* v;
  const int32_t* tables;
  const int32_t* lens;
  const int32_t* qstart;
  __half* out;
  int num_heads;
  int num_blocks;
  int max_blocks;
  int log2_block;
  int total_q;
  float scale_log2;
};

// ---- PTX wrappers ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte async copy global -> shared; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a [rows][D] fp16 tile whose chunks are
// XOR-swizzled by the row's low three bits.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((row * (D / 8) + (chunk ^ (row & 7))) * 16);
}

template <int D>
__global__ void __launch_bounds__(NWARP * 32, 2) paged_prefill_kernel(const PrefillParams p) {
  constexpr int CPR = D / 8;                     // 16-byte chunks per row
  constexpr int KSTEPS = D / 16;                 // k16 steps over the head dimension
  constexpr int TILE = BN * D * 2;               // bytes of one K (or V) tile
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sq = smem;                      // [BM][D]
  unsigned char* sk = smem + BM * D * 2;         // [2][BN][D]
  unsigned char* sv = sk + 2 * TILE;             // [2][BN][D]

  pkv::pdl_trigger();
  pkv::pdl_wait();
  const int qt = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.num_heads;
  const int B = 1 << p.log2_block;
  const int ctx = p.lens[s];
  const int q0 = p.qstart[s];
  const int n = p.qstart[s + 1] - q0;
  const int i0 = qt * BM;
  if (n < 0 || n > ctx || ctx > p.max_blocks * B || q0 < 0 || q0 + n > p.total_q) {
    if (tid == 0 && qt == 0) record_error(ctx > p.max_blocks * B ? PKV_DEV_BAD_CONTEXT_LEN : PKV_DEV_BAD_QUERY_RANGE);
    return;
  }
  if (i0 >= n) return;
  const int first_pos = ctx - n + i0;                             // position of the tile's first token
  const int last_pos = ctx - n + min(i0 + BM, n) - 1;             // and of its last valid token
  const int n_tiles = last_pos / BN + 1;

  // Q tile -> shared memory (rows past the new tokens are zero)
  for (int e = tid; e < BM * CPR; e += NWARP * 32) {
    const int r = e / CPR, c = e % CPR;
    const int i = i0 + r;
    const __half* src = p.q + (static_cast<size_t>(q0 + min(i, n - 1)) * H + h) * D + c * 8;
    cp_async16(smem_u32(sq) + swz<D>(r, c), src, i < n ? 16 : 0);
  }
  const int32_t* table = p.tables + static_cast<size_t>(s) * p.max_blocks;
  int bad = 0;
  auto load_tile = [&](int j, int stage) {
    // two threads per key row, each half of the row's chunks
    const int r = tid >> 1;
    const int t = j * BN + r;
    const bool valid = t < ctx;
    int phys = 0;
    if (valid) {
      phys = table[t >> p.log2_block];
      if (phys < 0 || phys >= p.num_blocks) {
        bad = 1;
        phys = 0;
      }
    }
    const bool ok = valid && !bad;
    const size_t row = ((static_cast<size_t>(phys) * H + h) << p.log2_block) + (t & (B - 1));
    const __half* ksrc = p.k + row * D;
    const __half* vsrc = p.v + row * D;
    const uint32_t kdst = smem_u32(sk + stage * TILE), vdst = smem_u32(sv + stage * TILE);
#pragma unroll
    for (int c0 = 0; c0 < CPR / 2; ++c0) {
      const int c = (tid & 1) * (CPR / 2) + c0;
      cp_async16(kdst + swz<D>(r, c), ksrc + c * 8, ok ? 16 : 0);
      cp_async16(vdst + swz<D>(r, c), vsrc + c * 8, ok ? 16 : 0);
    }
  };
  load_tile(0, 0);
  cp_async_commit();

  // per-warp state: 16 rows (lane/4 and lane/4 + 8 of the warp's slice)
  float o[D / 8][4];
#pragma unroll
  for (int d = 0; d < D / 8; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  uint32_t qa[KSTEPS][4];
  const int g = lane >> 2, tq = lane & 3;
  const int row_lo = i0 + warp * 16 + g;                          // new-token index of this lane's rows
  const int pos_lo = ctx - n + row_lo, pos_hi = pos_lo + 8;

  for (int j = 0; j < n_tiles; ++j) {
    if (j + 1 < n_tiles) load_tile(j + 1, (j + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (j == 0) {
      // this warp's Q fragments, once
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int mi = lane >> 3, r = lane & 7;
        ldsm_x4(smem_u32(sq) + swz<D>(warp * 16 + r + (mi & 1) * 8, kk * 2 + (mi >> 1)), qa[kk]);
      }
    }
    const uint32_t kb = smem_u32(sk + (j & 1) * TILE), vb = smem_u32(sv + (j & 1) * TILE);

    // S = Q K^T for 16 rows x 64 keys
    float sc[BN / 8][4];
#pragma unroll
    for (int nt = 0; nt < BN / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
      for (int pr = 0; pr < BN / 16; ++pr) {
        uint32_t b[4];
        const int mi = lane >> 3, r = lane & 7;
        ldsm_x4(kb + swz<D>(pr * 16 + r + (mi >> 1) * 8, kk * 2 + (mi & 1)), b);
        mma16816(sc[2 * pr], qa[kk], b[0], b[1]);
        mma16816(sc[2 * pr + 1], qa[kk], b[2], b[3]);
      }
    }
    // scale, mask (causal and past the context), online softmax in base 2
    const bool need_mask = (j + 1) * BN - 1 > first_pos;
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = j * BN + nt * 8 + tq * 2 + e;
        float lo = sc[nt][e] * p.scale_log2, hi = sc[nt][2 + e] * p.scale_log2;
        if (need_mask) {
          if (t > pos_lo) lo = -INFINITY;
          if (t > pos_hi) hi = -INFINITY;
        }
        sc[nt][e] = lo;
        sc[nt][2 + e] = hi;
        mx_lo = fmaxf(mx_lo, lo);
        mx_hi = fmaxf(mx_hi, hi);
      }
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(FULL, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(FULL, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(FULL, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(FULL, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    // a row with every key masked so far keeps m = -inf; use 0 as its reference
    const float ref_lo = mn_lo == -INFINITY ? 0.f : mn_lo, ref_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float al_lo = exp2f(m_lo - ref_lo), al_hi = exp2f(m_hi - ref_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
    for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[nt][e] = exp2f(sc[nt][e] - ref_lo);
        sc[nt][2 + e] = exp2f(sc[nt][2 + e] - ref_hi);
        sum_lo += sc[nt][e];
        sum_hi += sc[nt][2 + e];
      }
    }
    l_lo = l_lo * al_lo + sum_lo;
    l_hi = l_hi * al_hi + sum_hi;
#pragma unroll
    for (int d = 0; d < D / 8; ++d) {
      o[d][0] *= al_lo;
      o[d][1] *= al_lo;
      o[d][2] *= al_hi;
      o[d][3] *= al_hi;
    }
    // O += P V: P's accumulators become the A fragments of 16-key steps
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_half2(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = pack_half2(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = pack_half2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = pack_half2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b[4];
        const int mi = lane >> 3, r = lane & 7;
        ldsm_x4_trans(vb + swz<D>(kk * 16 + r + (mi & 1) * 8, dp * 2 + (mi >> 1)), b);
        mma16816(o[2 * dp], pa, b[0], b[1]);
        mma16816(o[2 * dp + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();                               // the stage is refilled next iteration
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (tid == 0) record_error(PKV_DEV_BAD_BLOCK_ID);
    return;
  }

  // normalise and store the warp's rows that are real new tokens
  l_lo += __shfl_xor_sync(FULL, l_lo, 1);
  l_lo += __shfl_xor_sync(FULL, l_lo, 2);
  l_hi += __shfl_xor_sync(FULL, l_hi, 1);
  l_hi += __shfl_xor_sync(FULL, l_hi, 2);
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f, inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
  const int row_hi = row_lo + 8;
#pragma unroll
  for (int d = 0; d < D / 8; ++d) {
    const int col = d * 8 + tq * 2;
    if (row_lo < n) {
      __half2* dst = reinterpret_cast<__half2*>(p.out + (static_cast<size_t>(q0 + row_lo) * H + h) * D + col);
      *dst = __floats2half2_rn(o[d][0] * inv_lo, o[d][1] * inv_lo);
    }
    if (row_hi < n) {
      __half2* dst = reinterpret_cast<__half2*>(p.out + (static_cast<size_t>(q0 + row_hi) * H + h) * D + col);
      *dst = __floats2half2_rn(o[d][2] * inv_hi, o[d][3] * inv_hi);
    }
  }
}

template <int D>
constexpr size_t prefill_smem() {
  return static_cast<size_t>(BM) * D * 2 + 4 * static_cast<size_t>(BN) * D * 2;
}

template <int D>
int launch_prefill(const PrefillParams& p, int num_seqs, int max_query_len, cudaStream_t st) {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(paged_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(prefill_smem<D>()));
      if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged prefill setup: %s", cudaGetErrorString(e));
  dim3 grid((max_query_len + BM - 1) / BM, p.num_heads, num_seqs);
  e = pkv::launch_pdl(paged_prefill_kernel<D>, grid, dim3(NWARP * 32), prefill_smem<D>(), st, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged prefill launch: %s", cudaGetErrorString(e));
  return PKV_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

namespace pkv {
int read_device_error_prefill(int reset, int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_error_prefill, sizeof(int));
  if (e == cudaSuccess && reset && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error_prefill, &zero, sizeof(int));
  }
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "reading the prefill check word: %s", cudaGetErrorString(e));
  *code = v;
  return PKV_OK;
}
}  // namespace pkv

extern "C" {

int pkv_paged_attention_prefill(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens, const int32_t* query_start,
                                int num_seqs, int total_q, int max_query_len, int num_heads, int head_dim,
                                int num_blocks, int max_blocks_per_seq, float scale, int block_size, uint16_t* out,
                                void* stream) {
  if (num_seqs < 0 || total_q < 0 || max_query_len < 0 || num_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return pkv::fail(PKV_ERR_INVALID_ARG,
                     "pkv_paged_attention_prefill: num_seqs=%d total_q=%d max_query_len=%d num_heads=%d "
                     "num_blocks=%d max_blocks_per_seq=%d",
                     num_seqs, total_q, max_query_len, num_heads, num_blocks, max_blocks_per_seq);
  if (head_dim != 64 && head_dim != 128)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_prefill: head_dim %d not in {64, 128}", head_dim);
  if (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_prefill: block_size %d not in {4, 8, 16, 32}",
                     block_size);
  if (num_seqs == 0 || total_q == 0 || max_query_len == 0) {
    pkv::clear_error();
    return PKV_OK;
  }
  if (num_seqs > 65535 || num_heads > 65535)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_prefill: num_seqs/num_heads above 65535");
  if (static_cast<long long>(max_blocks_per_seq) * block_size > (1LL << 30))
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_paged_attention_prefill: context capacity above 2^30 tokens");
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: null pointer");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: q, caches and out must be 16-byte aligned");
  if (!std::isfinite(scale)) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: scale not finite");
  PrefillParams p{};
  p.q = reinterpret_cast<const __half*>(q);
  p.k = reinterpret_cast<const __half*>(k_cache);
  p.v = reinterpret_cast<const __half*>(v_cache);
  p.tables = block_tables;
  p.lens = context_lens;
  p.qstart = query_start;
  p.out = reinterpret_cast<__half*>(out);
  p.num_heads = num_heads;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  int lb = 0;
  while ((1 << lb) < block_size) ++lb;
  p.log2_block = lb;
  p.total_q = total_q;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rc = head_dim == 128 ? launch_prefill<128>(p, num_seqs, max_query_len, st)
                                 : launch_prefill<64>(p, num_seqs, max_query_len, st);
  if (rc == PKV_OK) pkv::clear_error();
  return rc;
}

}  // extern "C"
