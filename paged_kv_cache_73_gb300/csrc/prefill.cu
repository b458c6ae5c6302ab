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
// Design: a dense contraction, so it runs on the fifth-generation tensor cores
// (tcgen05.mma, fp16 inputs, fp32 accumulation in tensor memory); see the
// kernel's comment below.  Key tiles of 64 positions are gathered block by
// block through the table into the 128-byte swizzled layout the tensor cores
// read, through a four-slot ring: whole blocks by TMA (one tensor-map box per
// block), the block holding the context's end by 16-byte cp.async copies.  Q
// arrives by TMA as well.  P is rounded to fp16 for the second product, as flash
// attention does.  Key rows past the context are zero-filled (never read), so
// stale NaN/Inf in unfilled slots cannot reach a product.
//
// The same kernel, in its PARTIAL mode, gives the shared-prefix decode its
// prefix part: the decode queries of a group of sequences sharing prefix blocks
// form the query rows, every row sees every prefix key, and each row's
// unnormalised (max, sum, output) goes to the decode workspace for the
// log-sum-exp merge.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched through the runtime
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


struct PrefillParams {
  // K and V pools as 3-D tensors (D, H*B, num_blocks), boxes of 64 x B x 1 with 128-byte swizzle
  // (encoded only when use_tma is set)
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  // q as the 3-D tensor (D, H, total_q), boxes of 64 x 1 x 128 with 128-byte swizzle
  CUtensorMap tmap_q;
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
  int use_tma;
  // shared-prefix partials (PARTIAL kernels only): blockIdx.z is a group of sequences
  // [group_start[g], group_start[g+1]) (the query rows) sharing keys [0, prefix_lens[g]); each
  // row's (m, l, o) goes to slot 0 of the decode workspace
  const int32_t* group_start;
  const int32_t* prefix_lens;
  float* ws_ml;
  float* ws_o;
  int max_parts;
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
// Commits this thread's outstanding cp.async copies and waits until all of them have landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---- fifth-generation tensor cores (tcgen05): S, P and O live in tensor memory ---------------
//
// A softmax thread owns one new-token row, which is one TMEM lane of its query tile.  Per key
// tile of 64 positions one thread issues S = Q K^T (tcgen05.mma, M=128, N=64, fp16 in, fp32 in
// TMEM); every softmax thread reads its row of S (tcgen05.ld), masks it, updates its running
// max/sum and writes P = 2^(S - m) as fp16 back over the scores it read (tcgen05.st); one thread
// issues O += P V (A = P from TMEM, B = V from shared memory, MN-major) into the TMEM
// accumulator.  MMA groups complete on mbarriers.
// The running max m of a row is only moved (and O rescaled) when a tile raises it by more than
// 2^8, so P stays within fp16 range while most tiles skip the O read-modify-write.
// Q, K and V tiles sit in shared memory in the canonical K-major / MN-major layouts with 128-byte
// swizzle: rows of 64 elements (128 B), 16-byte chunks XOR-ed with the row's low three bits,
// 8-row groups 1024 B apart, head-dimension halves in separate regions.
constexpr int TC_BM = 128;  // new tokens per query tile (MMA M)
constexpr int TC_BN = 64;   // key positions per tile (S MMA N, PV MMA K)
constexpr float TC_RESCALE = 8.f;

__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // start >> 4 | LBO >> 4 | SBO >> 4 | fixed 0b001 at bit 46 | swizzle mode 2 (128-byte) at bit 61
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
// kind::f16 instruction descriptor: fp32 accumulate, fp16 A and B, dense.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// The same load without its wait: the values are valid only after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mbar_init_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Adds `bytes` to the transaction count the barrier's current phase waits for (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Arrives on the barrier and adds `bytes` to the transaction count of its current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// TMA tile load of the box at (x, y, z) of a 3-D tensor map into shared memory; completion is
// counted in bytes on `bar`.  Coordinates outside the tensor read as zero.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// Brings a tensor map (a kernel parameter) into the TMA unit's descriptor cache ahead of its first use.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_parity(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
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
// Bounded wait (2 s): false if the phase did not complete in time.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_parity(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait_parity(bar, parity)) return true;
    if ((it & 255u) == 255u && global_ns() - t0 > 2000000000ull) return false;
  }
  return false;
}
// The same wait, also false once another role has raised the CTA's abort flag.  The flag is read
// only on the slow path: a generic shared-memory read in an MMA-issuing thread stalls it until
// the MMAs it has queued are done, so no hot loop reads it.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
  if (mbar_try_wait_parity(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait_parity(bar, parity)) return true;
    if ((it & 255u) == 255u && (*abort_flag != 0 || global_ns() - t0 > 2000000000ull)) return false;
  }
  return false;
}

// Byte offset of (row, 16-byte chunk) in a K-major / MN-major tile with 128-byte swizzle whose
// head-dimension halves are regions of `rows` x 128 B.
__device__ __forceinline__ uint32_t sw128(int row, int chunk, int rows) {
  return static_cast<uint32_t>((chunk >> 3) * rows * 128 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D>
struct TcCfg {
  static constexpr int Q_BYTES = TC_BM * D * 2;          // one 128-token query tile
  static constexpr int KV_BYTES = TC_BN * D * 2;         // one 64-position key or value tile
  static constexpr int STAGES = 4;                       // ring slots each for K and for V
  // two query tiles + the K and V rings; sized as for D = 128 whatever D is so that one CTA
  // (holding all 512 tensor-memory columns) runs per SM
  static constexpr int SMEM = 1024 /*alignment slack*/ + 2 * TC_BM * 128 * 2 + 2 * STAGES * TC_BN * 128 * 2 + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  // tensor-memory columns of query tile g: O at 128 g (D used); two S buffers at 256 + 128 g and
  // 256 + 128 g + 64 (key tile j uses buffer j % 2), P(j) as fp16 pairs over the first 32 columns
  // of S(j)'s buffer
  static constexpr uint32_t O_COL = 0, S_COL = 256;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Paired fp32 arithmetic (one instruction for two lanes of work): the softmax threads share their
// SM quarter with the MMA-issuing threads, so every instruction they save is issue time for those.
// (y0, y1) = (x0, x1) * s + c, each rounded once as fmaf would.
__device__ __forceinline__ void fma2(float& y0, float& y1, float x0, float x1, float s, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(s), "f"(c));
}
// (a0, a1) += (x0, x1)
// a0 += the low fp16 of `packed`, a1 += the high one (mixed-precision adds: the sum is taken over
// exactly the rounded values that go to the tensor cores)
__device__ __forceinline__ void add_half2(float& a0, float& a1, uint32_t packed) {
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(packed));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One CTA owns 256 new tokens of one (sequence, head) as two 128-token query tiles that share
// every K/V tile it loads.  Key tiles are 64 positions.  Per query tile g tensor memory holds
// the O_g accumulator and two S buffers: S_g(j) lands in buffer j % 2 and P_g(j) is written back
// over its first 32 columns, so S_g(j+1) is computed while softmax g still works on tile j.
// Warp roles (12 warps):
//   warps 0-3 / 4-7  softmax of query tile 0 / 1: thread t of the group owns token row t = TMEM
//              lane t.  For key tile j it waits S_g(j) (and so releases K slot j%4 for the
//              loader), copies its row to registers, masks and takes the row maximum, moves its
//              running max only when the tile raises it by more than 2^8 (then, after PV_g(j-1)
//              is done, rescaling its O row), writes P = 2^(S - m) as fp16 over the scores and
//              arrives on p_full.
//   warp 8     one lane issues S_0(j) and S_1(j) once K(j) has landed and PV_g(j-2), the last
//              reader of buffer j % 2, is done.
//   warp 11    one lane issues O_g += P_g(j) V(j) once V(j) and P_g(j) are there, then releases
//              V slot j%4.  Each commit or barrier check costs an issuing thread on the order of
//              a hundred cycles and the issuing warps share their SM quarter with softmax warps,
//              so the two issuing threads do little besides issuing (descriptors precomputed).
//   warps 9, 10 loads: gather key tile j's K (warp 9) or V (warp 10) through the table into ring
//              slot j%4 once tile j-4 is done with it (k_free / v_free).  Whole blocks come by
//              TMA (one box per block and head-dimension half, landing in the 128-byte swizzle);
//              the rest by cp.async.  k_full / v_full complete when every lane has arrived and
//              the TMA bytes have landed.
// Per-slot and per-buffer barriers keep every waiter within one phase of the barrier it waits on.
// Every wait is bounded; a role that gives up records PKV_DEV_WAIT_TIMEOUT and leaves its loop,
// the others give up in turn, and the CTA still reaches its final barrier.
constexpr int TC_QTILES = 2;
constexpr int TC_THREADS = 384;

// PARTIAL = false: prefill (rows = a sequence's new tokens, causal, normalised fp16 output).
// PARTIAL = true: shared-prefix partials (rows = the members of a group, every row sees every
// prefix key, unnormalised fp32 (m, l, o) into the decode workspace).
template <int D, bool PARTIAL>
__global__ void __launch_bounds__(TC_THREADS, 1) paged_prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using C = TcCfg<D>;
  constexpr int CPR = D / 8;                                  // 16-byte chunks per row
  constexpr int NS = C::STAGES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  const uint32_t sq = base;                                   // [2][128 rows][D], per-tile regions
  const uint32_t sk = sq + TC_QTILES * C::Q_BYTES, sv = sk + NS * C::KV_BYTES;
  const uint32_t bars = sv + NS * C::KV_BYTES;
  // per query tile g and S buffer u (key tile j uses u = j % 2): s_full (S_g(j) landed), p_full
  // (P_g(j) written), pv_done (PV_g(j) done); per ring slot b: k_full / v_full (data landed),
  // k_free / v_free (the MMAs reading it are done).  A waiter on a per-buffer barrier can never
  // be two phases behind it, so the phase parity it waits on is unambiguous.
  auto s_full = [&](int g, int u) { return bars + 8u * (2 * g + u); };
  auto p_full = [&](int g, int u) { return bars + 32u + 8u * (2 * g + u); };
  auto pv_done = [&](int g, int u) { return bars + 64u + 8u * (2 * g + u); };
  auto k_full = [&](int b) { return bars + 96u + 8u * b; };
  auto v_full = [&](int b) { return bars + 96u + 8u * (NS + b); };
  auto k_free = [&](int b) { return bars + 96u + 8u * (2 * NS + b); };
  auto v_free = [&](int b) { return bars + 96u + 8u * (3 * NS + b); };
  const uint32_t q_full = bars + 96 + 32 * NS;                // the Q tiles landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bars + 104 + 32 * NS - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + (bars + 108 + 32 * NS - base));
  static_assert(112 + 32 * NS <= 256, "barrier area");

  pkv::pdl_trigger();
  pkv::pdl_wait();
  // the last query tiles of a sequence see the most keys: launch them first
  const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.num_heads;
  const int lb = p.log2_block;
  const int B = 1 << lb;
  const int i0 = qt * TC_QTILES * TC_BM;
  // keys [0, ctx) through table row `trow`; query rows q0 + i0 + r, r < n - i0
  int ctx, q0, n, trow;
  if constexpr (PARTIAL) {
    q0 = p.group_start[s];
    n = p.group_start[s + 1] - q0;
    ctx = p.prefix_lens[s];
    trow = q0;
    if (q0 < 0 || n < 0 || q0 + n > p.total_q || ctx < 0 || ctx > p.max_blocks * B || (ctx & (B - 1)) != 0) {
      if (tid == 0 && qt == 0 && h == 0) record_error(PKV_DEV_PREFIX_MISMATCH);
      return;
    }
    // a group larger than the grid covers (the caller's max_group_size understated it): its later
    // members would get no prefix partial, so the call is flagged
    if (tid == 0 && qt == 0 && h == 0 && n > static_cast<int>(gridDim.x) * TC_QTILES * TC_BM)
      record_error(PKV_DEV_PREFIX_MISMATCH);
    if (i0 >= n) return;
    if (ctx == 0 || n < pkv::kMinSharedGroup) {
      // no shared prefix, or a group too small to share it (its members read their whole context
      // in the split-K decode): an empty partial for every row
      if (tid < TC_QTILES * TC_BM && i0 + tid < n) {
        const size_t w = (static_cast<size_t>(q0 + i0 + tid) * H + h) * p.max_parts;
        p.ws_ml[2 * w] = -INFINITY;
        p.ws_ml[2 * w + 1] = 0.f;
        for (int d = 0; d < D; d += 4) *reinterpret_cast<float4*>(p.ws_o + w * D + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      return;
    }
  } else {
    ctx = p.lens[s];
    q0 = p.qstart[s];
    n = p.qstart[s + 1] - q0;
    trow = s;
    if (n < 0 || n > ctx || ctx > p.max_blocks * B || q0 < 0 || q0 + n > p.total_q) {
      if (tid == 0 && qt == 0) record_error(ctx > p.max_blocks * B ? PKV_DEV_BAD_CONTEXT_LEN : PKV_DEV_BAD_QUERY_RANGE);
      return;
    }
    // more new tokens than the grid covers (the caller's max_query_len understated them): the rows
    // past the grid are not written, so the call is flagged
    if (tid == 0 && qt == 0 && h == 0 && n > static_cast<int>(gridDim.x) * TC_QTILES * TC_BM)
      record_error(PKV_DEV_BAD_QUERY_RANGE);
    if (i0 >= n) return;
  }
  const int ntile_q = i0 + TC_BM < n ? 2 : 1;                 // query tiles with real tokens
  // positions of the first and last query rows (every partial row sits after the whole prefix)
  const int first_pos = PARTIAL ? ctx - 1 : ctx - n + i0;
  const int last_pos = PARTIAL ? ctx - 1 : ctx - n + min(i0 + TC_QTILES * TC_BM, n) - 1;
  const int n_tiles = last_pos / TC_BN + 1;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  if (tid == 0) {
    for (int g = 0; g < TC_QTILES; ++g)
      for (int u = 0; u < 2; ++u) {
        mbar_init_count(s_full(g, u), 1);
        mbar_init_count(p_full(g, u), 128);
        mbar_init_count(pv_done(g, u), 1);
      }
    for (int b = 0; b < NS; ++b) {
      mbar_init_count(k_full(b), 32);
      mbar_init_count(v_full(b), 32);
      // K: released by one lane of each softmax warp once it has seen S(j) complete; V: by the
      // PV-issuing thread's commit after the last PV of tile j
      mbar_init_count(k_free(b), 4 * ntile_q);
      mbar_init_count(v_free(b), 1);
    }
    *abort_flag = 0;
    // the Q tiles by TMA, right away, overlapping the first K/V loads: rows i0 + 128 g + r of
    // head h, landing in the 128-byte swizzle.  Rows past the sequence's new tokens read the next
    // sequence's (or, past total_q, zeros); their results are never stored.
    mbar_init_count(q_full, 1);
    mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(ntile_q) * C::Q_BYTES);
    for (int g = 0; g < ntile_q; ++g)
#pragma unroll
      for (int half = 0; half < D / 64; ++half)
        tma_load_3d(sq + g * C::Q_BYTES + half * (TC_BM * 128), &p.tmap_q, half * 64, h, q0 + i0 + g * TC_BM, q_full);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto t_s = [&](int g, int u) { return tmem + C::S_COL + 128u * g + 64u * u; };
  auto t_o = [&](int g) { return tmem + C::O_COL + 128u * g; };
  auto wait = [&](uint32_t bar, uint32_t parity) { return mbar_wait_or_abort(bar, parity, abort_flag); };
  auto give_up = [&]() {
    if (!*abort_flag) record_error(PKV_DEV_WAIT_TIMEOUT);
    *abort_flag = 1;
  };
  int bad = 0;
  bool failed = false;
  float l = 0.f, m_ref = -INFINITY;

  if (warp == 9 || warp == 10) {
    // ---------------- loads: warp 9 gathers K tiles, warp 10 V tiles ----------------
    // Lane b handles the tile's b-th block: it issues that block's TMA boxes itself (the lanes'
    // copies go out together), and its table entry for the next tile is read while this tile's
    // copies are issued.
    const bool is_k = warp == 9;
    const __half* pool = is_k ? p.k : p.v;
    const CUtensorMap* map = is_k ? &p.tmap_k : &p.tmap_v;
    if (lane == 0 && p.use_tma) prefetch_tensormap(map);
    const int32_t* table = p.tables + static_cast<size_t>(trow) * p.max_blocks;
    constexpr int ROWS = 32 / CPR;                            // rows per warp-wide cp.async
    const int c = lane % CPR, rsub = lane / CPR;              // this lane's chunk and row offset
    const int nb = TC_BN >> lb;                               // blocks per tile (2..16)
    const uint32_t all_blocks = (nb == 32 ? 0xffffffffu : (1u << nb) - 1u);
    auto entry = [&](int j) {                                 // this lane's table entry for tile j
      const int t0 = j * TC_BN + (lane << lb);
      return lane < nb && t0 < ctx ? __ldg(table + (t0 >> lb)) : -1;
    };
    int next_entry = entry(0);
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % NS;
      // lane b < nb maps the tile's b-th block: phys = -1 past the context or for a bad entry
      const int t0 = j * TC_BN + (lane << lb);
      const bool in_ctx = lane < nb && t0 < ctx;
      int phys = next_entry;
      if (j + 1 < n_tiles) next_entry = entry(j + 1);
      if (in_ctx && (phys < 0 || phys >= p.num_blocks)) bad = 1;
      if (!in_ctx || phys < 0 || phys >= p.num_blocks) phys = -1;
      // slot j%4 is free once the MMAs of tile j-4 that read it are done
      if (j >= NS && !wait(is_k ? k_free(st) : v_free(st), (j / NS - 1) & 1)) {
        failed = true;
        break;
      }
      const uint32_t full = is_k ? k_full(st) : v_full(st);
      const uint32_t dst = (is_k ? sk : sv) + st * C::KV_BYTES;
      // whole blocks inside the context arrive by TMA (B >= 8, so each lands on a 1024-byte
      // boundary of the swizzled tile); the block holding the context's end, blocks past it and
      // bad entries are copied (or zero-filled) by cp.async
      const bool by_tma = p.use_tma && phys >= 0 && t0 + B <= ctx;
      const uint32_t tma_mask = __ballot_sync(0xffffffffu, by_tma);
      if (lane == 0 && tma_mask) mbar_expect_tx(full, static_cast<uint32_t>(__popc(tma_mask)) * B * D * 2);
      __syncwarp();
      if (by_tma) {
#pragma unroll
        for (int half = 0; half < D / 64; ++half)
          tma_load_3d(dst + half * (TC_BN * 128) + lane * B * 128, map, half * 64, h * B, phys, full);
      }
      if (tma_mask != all_blocks) {
        for (int r0 = 0; r0 < TC_BN; r0 += ROWS) {
          const int b = r0 >> lb;                             // ROWS <= 4 <= B: one block per pass
          const int pb = __shfl_sync(0xffffffffu, phys, b);
          if ((tma_mask >> b) & 1u) continue;
          const int r = r0 + rsub;
          const int t = j * TC_BN + r;
          const bool ok = t < ctx && pb >= 0;
          const __half* src =
              pool + (((static_cast<size_t>(ok ? pb : 0) * H + h) << lb) + (t & (B - 1))) * D + c * 8;
          cp_async16(dst + sw128(r, c, TC_BN), src, ok ? 16 : 0);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();                             // cp.async writes -> tensor-core reads
      }
      mbar_arrive(full);
      ++issued;
    }
    if (failed) give_up();
    if (*abort_flag) {
      // let the copies this warp issued land (bounded) before the CTA's shared memory is released
      for (int t = max(0, issued - NS); t < issued; ++t)
        mbar_wait(is_k ? k_full(t % NS) : v_full(t % NS), (t / NS) & 1);
    }
  } else if (warp == 8) {
    // ---------------- S = Q K^T issue (one lane) ----------------
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = umma_idesc_f16(TC_BM, TC_BN, false);
      const uint64_t a_desc0 = umma_smem_desc(sq, 16, 1024), a_desc1 = umma_smem_desc(sq + C::Q_BYTES, 16, 1024);
      int issued[TC_QTILES] = {0, 0};
      failed = !wait(q_full, 0);
      for (int j = 0; j < n_tiles && !failed; ++j) {
        if (!wait(k_full(j % NS), (j / NS) & 1)) {
          failed = true;
          break;
        }
        const uint32_t kb = sk + (j % NS) * C::KV_BYTES;
        const int u = j & 1;
        // the descriptors of a K-step differ from the first by the start-address field alone
        // (shared-memory byte offset / 16, far from overflowing its 14 bits): one add per MMA
        const uint64_t b0 = umma_smem_desc(kb, 16, 1024);
        for (int g = 0; g < ntile_q; ++g) {
          // S buffer u of tile g is free once PV_g(j-2), which read P_g(j-2) from it, is done
          if (j >= 2 && !wait(pv_done(g, u), ((j - 2) >> 1) & 1)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t a0 = g == 0 ? a_desc0 : a_desc1;
          const uint32_t d = t_s(g, u);
          umma_ss(d, a0, b0, IDESC_QK, 0u);
#pragma unroll
          for (int kk = 1; kk < D / 16; ++kk)
            umma_ss(d, a0 + (((kk >> 2) * (TC_BM * 128) + (kk & 3) * 32) >> 4),
                    b0 + (((kk >> 2) * (TC_BN * 128) + (kk & 3) * 32) >> 4), IDESC_QK, 1u);
          umma_commit(s_full(g, u));
          ++issued[g];
        }
      }
      if (failed) {
        give_up();
        // let the tensor-core work this lane issued finish (bounded) before memory is released
        for (int g = 0; g < ntile_q; ++g)
          if (issued[g] > 0) mbar_wait(s_full(g, (issued[g] - 1) & 1), ((issued[g] - 1) >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 11) {
    // ---------------- O += P V issue (one lane) ----------------
    if (lane == 0) {
      constexpr uint32_t IDESC_PV = umma_idesc_f16(TC_BM, D, true);
      int issued[TC_QTILES] = {0, 0};
      for (int j = 0; j < n_tiles && !failed; ++j) {
        if (!wait(v_full(j % NS), (j / NS) & 1)) {
          failed = true;
          break;
        }
        const uint32_t vb = sv + (j % NS) * C::KV_BYTES;
        const int u = j & 1;
        for (int g = 0; g < ntile_q; ++g) {
          // softmax g has written P_g(j) (and finished any rescale of O_g)
          if (!wait(p_full(g, u), (j >> 1) & 1)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t v0 = umma_smem_desc(vb, TC_BN * 128, 1024);
          const uint32_t o = t_o(g), pa = t_s(g, u);
          umma_ts(o, pa, v0, IDESC_PV, j > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < TC_BN / 16; ++kk) umma_ts(o, pa + kk * 8, v0 + ((kk * 16 * 128) >> 4), IDESC_PV, 1u);
          umma_commit(pv_done(g, u));
          ++issued[g];
        }
        if (failed) break;
        umma_commit(v_free(j % NS));               // every PV of tile j issued
      }
      if (failed) {
        give_up();
        for (int g = 0; g < ntile_q; ++g)
          if (issued[g] > 0) mbar_wait(pv_done(g, (issued[g] - 1) & 1), ((issued[g] - 1) >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp < 4 * ntile_q) {
    // ---------------- softmax (warps 0-3: query tile 0, warps 4-7: query tile 1) ----------------
    const int g = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t to = t_o(g);
    const int row_i = i0 + tid;                        // tid = g * 128 + row within the tile
    const int pos = PARTIAL ? ctx - 1 : ctx - n + row_i;
    const int tile_first = PARTIAL ? ctx - 1 : first_pos + g * TC_BM;   // the tile's first token
    for (int j = 0; j < n_tiles; ++j) {
      // decisions stay warp-uniform: the tcgen05.ld/st below are warp-collective
      const int u = j & 1;
      const uint32_t ts = t_s(g, u);
      if (!__all_sync(0xffffffffu, wait(s_full(g, u), (j >> 1) & 1))) {
        failed = true;
        break;
      }
      tc_fence_after();
      if (lane == 0) mbar_arrive(k_free(j % NS));     // S_g(j) is done reading K(j)
      float sv[TC_BN];
      tmem_ld32_nowait(ts + lane_off, *reinterpret_cast<float(*)[32]>(sv));
      tmem_ld32_nowait(ts + lane_off + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
      tmem_ld_wait();
      const int key0 = j * TC_BN;
      if (key0 + TC_BN - 1 > tile_first) {             // the diagonal tiles: keys after the token
#pragma unroll
        for (int c = 0; c < TC_BN; ++c)
          if (key0 + c > pos) sv[c] = -INFINITY;
      }
      // row maximum: three-input maxima in eight independent chains; scale > 0, so the maximum of
      // the scaled scores is the scaled maximum
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
      for (int c = 16; c < TC_BN; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = max3(m8[i], sv[c + i], sv[c + 8 + i]);
      float mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      mx *= p.scale_log2;
      const bool rescale = mx > m_ref + TC_RESCALE;   // also true for the first finite max
      float alpha = 1.f;
      if (rescale) {
        alpha = exp2f(m_ref - mx);                     // 0 when m_ref = -inf
        m_ref = mx;
      }
      const float nref = m_ref == -INFINITY ? 0.f : -m_ref;
      // if any row of the warp moved its max after the first tile, the whole warp rescales its O
      // rows (alpha is 1 for the rows that did not move), once PV_g(j-1) has finished with O_g
      if (__any_sync(0xffffffffu, rescale && j > 0)) {
        if (!__all_sync(0xffffffffu, wait(pv_done(g, (j - 1) & 1), ((j - 1) >> 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(to + lane_off + c * 32, o);
          uint32_t ob[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) ob[e] = __float_as_uint(o[e] * alpha);
          tmem_st32(to + lane_off + c * 32, ob);
        }
      }
      // P = 2^(scale*S - m) as fp16: one paired FMA per two scores, one ex2 per score; the row
      // sum, in eight accumulators, adds the fp16-rounded weights that multiply V, so the
      // normalised weights sum to one (summing the unrounded values instead leaves the output off
      // by up to 2^-11 of |v| where one key dominates)
      float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[TC_BN / 2];
#pragma unroll
      for (int e = 0; e < TC_BN / 2; ++e) {
        float x0, x1;
        fma2(x0, x1, sv[2 * e], sv[2 * e + 1], p.scale_log2, nref);
        pk[e] = pack_half2(fast_exp2(x0), fast_exp2(x1));
        add_half2(sum8[2 * (e & 3)], sum8[2 * (e & 3) + 1], pk[e]);
      }
      float sum4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sum4[i] = sum8[2 * i] + sum8[2 * i + 1];
      tmem_st32(ts + lane_off, pk);                    // P_g(j) over the scores already read
      l = l * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full(g, u));
    }
    if (!failed) {
      failed = !__all_sync(0xffffffffu, wait(pv_done(g, (n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1));
      tc_fence_after();
    }
    if (failed) give_up();
  }

  // ---------------- epilogue (all warps) ----------------
  bad = __syncthreads_or(bad);
  const bool aborted = *abort_flag != 0;
  if (PARTIAL && warp < 4 * ntile_q) {
    // each member's partial straight from tensor memory (every lane loads: tcgen05.ld is
    // warp-collective): m and l in the base-2 log domain, o unnormalised; an empty partial if a
    // block id was bad or a role gave up
    const int g = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool ok = !aborted && !bad;
    const bool row_ok = i0 + tid < n;
    const size_t w = (static_cast<size_t>(q0 + i0 + min(tid, n - 1 - i0)) * H + h) * p.max_parts;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      tmem_ld32(t_o(g) + lane_off + c * 32, o);
      if (row_ok) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(p.ws_o + w * D + c * 32 + e) =
              ok ? make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (row_ok) {
      p.ws_ml[2 * w] = ok ? m_ref : -INFINITY;
      p.ws_ml[2 * w + 1] = ok ? l : 0.f;
    }
  } else if (!PARTIAL && warp < 4 * ntile_q && !aborted && !bad) {
    // Each thread normalises its O row (every lane loads: tcgen05.ld is warp-collective) and
    // stages it in the K/V ring, free now that every MMA is done, as 16-byte chunks XOR-ed with
    // the row's low bits (no bank conflicts either way).  The warp then writes its 32 rows back
    // whole: each row is D*2 contiguous bytes of out, stored by D/8 lanes at once.  Rows past the
    // sequence's new tokens are not stored.
    const int g = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    unsigned char* stage = smem + (sk - base);                // [256 rows][D * 2 bytes]
    constexpr int RB = D * 2;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      tmem_ld32(t_o(g) + lane_off + c * 32, o);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 w;
        w.x = pack_half2(o[8 * k] * inv, o[8 * k + 1] * inv);
        w.y = pack_half2(o[8 * k + 2] * inv, o[8 * k + 3] * inv);
        w.z = pack_half2(o[8 * k + 4] * inv, o[8 * k + 5] * inv);
        w.w = pack_half2(o[8 * k + 6] * inv, o[8 * k + 7] * inv);
        *reinterpret_cast<uint4*>(stage + tid * RB + (((c * 4 + k) ^ (tid & (CPR - 1))) << 4)) = w;
      }
    }
    __syncwarp();
    constexpr int RPI = 32 / CPR;                             // rows per warp-wide store
    const int c = lane % CPR;
#pragma unroll 4
    for (int r0 = 0; r0 < 32; r0 += RPI) {
      const int row = warp * 32 + r0 + lane / CPR;            // CTA row = token i0 + row
      if (i0 + row < n) {
        const uint4 w = *reinterpret_cast<const uint4*>(stage + row * RB + ((c ^ (row & (CPR - 1))) << 4));
        *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(q0 + i0 + row) * H + h) * D + c * 8) = w;
      }
    }
  }
  // the Q copies have landed (they have, unless the CTA gave up early): bounded
  if (tid == 0) mbar_wait(q_full, 0);
  if (bad && tid == 0) record_error(PKV_DEV_BAD_BLOCK_ID);
  cp_async_wait_all();
  // all tensor-memory reads are done (tcgen05.ld waits inline); release the columns
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
  }
}

template <int D, bool PARTIAL>
int launch_prefill(const PrefillParams& p, int num_seqs, int max_query_len, cudaStream_t st) {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(paged_prefill_tc_kernel<D, PARTIAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               TcCfg<D>::SMEM);
      if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged prefill setup: %s", cudaGetErrorString(e));
  dim3 grid((max_query_len + TC_QTILES * TC_BM - 1) / (TC_QTILES * TC_BM), p.num_heads, num_seqs);
  e = pkv::launch_pdl(paged_prefill_tc_kernel<D, PARTIAL>, grid, dim3(TC_THREADS), TcCfg<D>::SMEM, st, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "paged prefill launch: %s", cudaGetErrorString(e));
  return PKV_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched once through the runtime (no link against libcuda).
EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// A pool [num_blocks][H][B][D] fp16 as the 3-D tensor (D, H*B, num_blocks); a box is one head's
// B rows of one 64-element half of the head dimension, written with the 128-byte swizzle.
int encode_pool_map(CUtensorMap* map, const void* pool, int D, int H, int B, int num_blocks) {
  const EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return pkv::fail(PKV_ERR_CUDA, "paged prefill: cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H) * B,
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * B * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(B), 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(pool), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "paged prefill: tensor map encoding failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// q [T][H][D] fp16 as the 3-D tensor (D, H, T); a box is 128 tokens of one head and one 64-element
// half of the head dimension, written with the 128-byte swizzle.
int encode_q_map(CUtensorMap* map, const void* q, int D, int H, int T) {
  const EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return pkv::fail(PKV_ERR_CUDA, "paged prefill: cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(TC_BM)};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(q), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "paged prefill: q tensor map encoding failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

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
  if (!std::isfinite(scale) || !(scale > 0.f))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: scale must be finite and positive");
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
  {
    const int rc = encode_q_map(&p.tmap_q, q, head_dim, num_heads, total_q);
    if (rc != PKV_OK) return rc;
  }
  // whole blocks of 8 or more rows are fetched by TMA; smaller blocks by cp.async
  p.use_tma = block_size >= 8 ? 1 : 0;
  if (p.use_tma) {
    int rc = encode_pool_map(&p.tmap_k, k_cache, head_dim, num_heads, block_size, num_blocks);
    if (rc == PKV_OK) rc = encode_pool_map(&p.tmap_v, v_cache, head_dim, num_heads, block_size, num_blocks);
    if (rc != PKV_OK) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rc = head_dim == 128 ? launch_prefill<128, false>(p, num_seqs, max_query_len, st)
                                 : launch_prefill<64, false>(p, num_seqs, max_query_len, st);
  if (rc == PKV_OK) pkv::clear_error();
  return rc;
}

}  // extern "C"

namespace pkv {
int launch_prefix_partials(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                           const int32_t* block_tables, const int32_t* group_start, const int32_t* prefix_lens,
                           int num_groups, int max_group_size, int num_seqs, int num_heads, int head_dim,
                           int num_blocks, int max_blocks_per_seq, float scale, int block_size, float* ws_ml,
                           float* ws_o, int max_parts, void* stream) {
  PrefillParams p{};
  p.q = reinterpret_cast<const __half*>(q);
  p.k = reinterpret_cast<const __half*>(k_cache);
  p.v = reinterpret_cast<const __half*>(v_cache);
  p.tables = block_tables;
  p.group_start = group_start;
  p.prefix_lens = prefix_lens;
  p.ws_ml = ws_ml;
  p.ws_o = ws_o;
  p.max_parts = max_parts;
  p.num_heads = num_heads;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  int lb = 0;
  while ((1 << lb) < block_size) ++lb;
  p.log2_block = lb;
  p.total_q = num_seqs;                                // q [num_seqs][H][D]: one row per sequence
  p.scale_log2 = scale * 1.4426950408889634f;
  int rc = encode_q_map(&p.tmap_q, q, head_dim, num_heads, num_seqs);
  if (rc != PKV_OK) return rc;
  p.use_tma = block_size >= 8 ? 1 : 0;
  if (p.use_tma) {
    rc = encode_pool_map(&p.tmap_k, k_cache, head_dim, num_heads, block_size, num_blocks);
    if (rc == PKV_OK) rc = encode_pool_map(&p.tmap_v, v_cache, head_dim, num_heads, block_size, num_blocks);
    if (rc != PKV_OK) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // grid: (256-member query tiles, heads, groups)
  return head_dim == 128 ? launch_prefill<128, true>(p, num_groups, max_group_size, st)
                         : launch_prefill<64, true>(p, num_groups, max_group_size, st);
}
}  // namespace pkv
