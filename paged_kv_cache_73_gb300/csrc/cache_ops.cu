// The two byte-moving kernels around decode attention, for sm_103a.
//
// [note] "vLLM / PagedAttention -- 把 LLM 服务的瓶颈从显存碎片里救出来", section
// 关键设计 5, names them: "fused reshape and block write" (each new token's
// key/value rows go to their slot in the block layout, all heads in one
// launch) and "fused block copy" (the many small copies that copy-on-write
// triggers, section 关键设计 3, done by one kernel instead of one memcpy each).
//
// Both are HBM-bound copies: 16-byte vector loads and stores, 64-bit offsets
// (a pool can fill most of a 288 GB HBM), every slot and block id checked
// against the pool before it is used.
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.cuh"
#include "pkv_internal.h"

namespace {

__device__ int g_dev_error_cache_ops = 0;

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_dev_error_cache_ops, 0, code); }

// Token t's key and value rows (all heads) go to slot slot_mapping[t]: one CTA per token, its
// threads walking the H * D/8 16-byte columns.  head_dim/8 and block_size are powers of two, so
// every index is a shift or a mask.
__device__ __forceinline__ void store_tokens(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                             uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                             const int64_t* __restrict__ slot_mapping, int num_tokens,
                                             int num_heads, int log2_vec, int log2_block, int64_t num_slots) {
  const int per_token = num_heads << log2_vec;
  const int vec_mask = (1 << log2_vec) - 1;
  const int row_mask = (1 << log2_block) - 1;
  for (int t = blockIdx.x; t < num_tokens; t += gridDim.x) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;                        // padding token
    if (slot >= num_slots) {
      if (threadIdx.x == 0) record_error(PKV_DEV_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot >> log2_block;
    const int row = static_cast<int>(slot & row_mask);
    const uint4* __restrict__ ksrc = key + static_cast<int64_t>(t) * per_token;
    const uint4* __restrict__ vsrc = value + static_cast<int64_t>(t) * per_token;
    for (int e = threadIdx.x; e < per_token; e += blockDim.x) {
      const int h = e >> log2_vec;
      const int c = e & vec_mask;
      const int64_t dst = ((((blk * num_heads + h) << log2_block) + row) << log2_vec) + c;
      k_cache[dst] = ksrc[e];
      v_cache[dst] = vsrc[e];
    }
  }
}

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const uint4* __restrict__ key,
                                                                const uint4* __restrict__ value,
                                                                uint4* __restrict__ k_cache,
                                                                uint4* __restrict__ v_cache,
                                                                const int64_t* __restrict__ slot_mapping,
                                                                int num_tokens, int num_heads, int log2_vec,
                                                                int log2_block, int64_t num_slots) {
  pkv::pdl_trigger();
  pkv::pdl_wait();  // key/value/slots may come from the previous kernel on the stream
  store_tokens(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_heads, log2_vec, log2_block, num_slots);
}

constexpr int kMaxLayersPerLaunch = 64;

struct TokenLayerPtrs {
  const uint4* key[kMaxLayersPerLaunch];
  const uint4* value[kMaxLayersPerLaunch];
  uint4* k_cache[kMaxLayersPerLaunch];
  uint4* v_cache[kMaxLayersPerLaunch];
};

// reshape_and_cache for many layers at once: grid.y is the layer; the same slots for every layer.
__global__ void __launch_bounds__(256) reshape_and_cache_layers_kernel(const TokenLayerPtrs ptrs,
                                                                       const int64_t* __restrict__ slot_mapping,
                                                                       int num_tokens, int num_heads, int log2_vec,
                                                                       int log2_block, int64_t num_slots) {
  pkv::pdl_trigger();
  pkv::pdl_wait();
  const int layer = blockIdx.y;
  store_tokens(ptrs.key[layer], ptrs.value[layer], ptrs.k_cache[layer], ptrs.v_cache[layer], slot_mapping,
               num_tokens, num_heads, log2_vec, log2_block, num_slots);
}

struct LayerPtrs {
  uint4* k[kMaxLayersPerLaunch];
  uint4* v[kMaxLayersPerLaunch];
};

// grid (num_pairs, num_layers, splits): CTA (p, l, z) copies slice z of block pair p in layer l.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const LayerPtrs ptrs, const int64_t* __restrict__ mapping,
                                                          int64_t vec_per_block, int num_blocks) {
  pkv::pdl_trigger();
  pkv::pdl_wait();
  const int pair = blockIdx.x;
  const int layer = blockIdx.y;
  const int64_t src = mapping[2 * pair];
  const int64_t dst = mapping[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.z == 0) record_error(PKV_DEV_BAD_COPY_PAIR);
    return;
  }
  const uint4* __restrict__ ks = ptrs.k[layer] + src * vec_per_block;
  const uint4* __restrict__ vs = ptrs.v[layer] + src * vec_per_block;
  uint4* __restrict__ kd = ptrs.k[layer] + dst * vec_per_block;
  uint4* __restrict__ vd = ptrs.v[layer] + dst * vec_per_block;
  const int64_t stride = static_cast<int64_t>(gridDim.z) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.z) * blockDim.x + threadIdx.x;
  // four 16-byte loads of K and four of V in flight per thread before the stores
  for (; i + 3 * stride < vec_per_block; i += 4 * stride) {
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u] = ks[i + u * stride];
      b[u] = vs[i + u * stride];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      kd[i + u * stride] = a[u];
      vd[i + u * stride] = b[u];
    }
  }
  for (; i < vec_per_block; i += stride) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

struct PoolPairPtrs {
  const uint4* src_k[kMaxLayersPerLaunch];
  const uint4* src_v[kMaxLayersPerLaunch];
  uint4* dst_k[kMaxLayersPerLaunch];
  uint4* dst_v[kMaxLayersPerLaunch];
};

// grid (num_pairs, num_layers, splits): CTA (p, l, z) copies slice z of block src_p of layer l's
// source pools into block dst_p of its destination pools.  Either side may be page-locked host
// memory (reached over the C2C link) or device memory.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const PoolPairPtrs ptrs, const int64_t* __restrict__ mapping,
                                                          int64_t vec_per_block, int src_blocks, int dst_blocks) {
  pkv::pdl_trigger();
  pkv::pdl_wait();
  const int pair = blockIdx.x;
  const int layer = blockIdx.y;
  const int64_t src = mapping[2 * pair];
  const int64_t dst = mapping[2 * pair + 1];
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.z == 0) record_error(PKV_DEV_BAD_COPY_PAIR);
    return;
  }
  const uint4* __restrict__ ks = ptrs.src_k[layer] + src * vec_per_block;
  const uint4* __restrict__ vs = ptrs.src_v[layer] + src * vec_per_block;
  uint4* __restrict__ kd = ptrs.dst_k[layer] + dst * vec_per_block;
  uint4* __restrict__ vd = ptrs.dst_v[layer] + dst * vec_per_block;
  const int64_t stride = static_cast<int64_t>(gridDim.z) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.z) * blockDim.x + threadIdx.x;
  // eight 16-byte loads in flight per thread: reads over the host link have a long latency
  for (; i + 3 * stride < vec_per_block; i += 4 * stride) {
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u] = ks[i + u * stride];
      b[u] = vs[i + u * stride];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      kd[i + u * stride] = a[u];
      vd[i + u * stride] = b[u];
    }
  }
  for (; i < vec_per_block; i += stride) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// A pointer a kernel may dereference: device, managed or page-locked (registered) host memory.
bool device_accessible(const void* ptr) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
         (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr);
}

int ilog2(int x) {
  int r = 0;
  while ((1 << (r + 1)) <= x) ++r;
  return r;
}

// One CTA per token (grid-stride beyond 2^20 tokens); threads cover a token's H * D/8 columns.
void reshape_launch_shape(int num_tokens, int num_heads, int head_dim, int* threads, int* grid) {
  const int per_token = num_heads * (head_dim / 8);
  int t = per_token < 256 ? (per_token + 31) / 32 * 32 : 256;
  *threads = t;
  *grid = num_tokens < (1 << 20) ? num_tokens : (1 << 20);
}

int check_shape(const char* fn, int num_heads, int head_dim, int block_size, int num_blocks) {
  if (num_heads <= 0 || num_blocks <= 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "%s: num_heads=%d num_blocks=%d", fn, num_heads, num_blocks);
  if (head_dim != 64 && head_dim != 128)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "%s: head_dim %d not in {64, 128}", fn, head_dim);
  if (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "%s: block_size %d not in {4, 8, 16, 32}", fn, block_size);
  return PKV_OK;
}

}  // namespace

namespace pkv {
int read_device_error_cache_ops(int reset, int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_error_cache_ops, sizeof(int));
  if (e == cudaSuccess && reset && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error_cache_ops, &zero, sizeof(int));
  }
  if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "reading the cache-op check word: %s", cudaGetErrorString(e));
  *code = v;
  return PKV_OK;
}
}  // namespace pkv

extern "C" {

int pkv_reshape_and_cache(const uint16_t* key, const uint16_t* value, uint16_t* k_cache, uint16_t* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_heads, int head_dim, int block_size,
                          int num_blocks, void* stream) {
  int rc = check_shape("pkv_reshape_and_cache", num_heads, head_dim, block_size, num_blocks);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_reshape_and_cache: num_tokens=%d", num_tokens);
  if (num_tokens == 0) {
    pkv::clear_error();
    return PKV_OK;
  }
  if (!key || !value || !k_cache || !v_cache || !slot_mapping)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_reshape_and_cache: null pointer");
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_reshape_and_cache: key, value and caches must be 16-byte aligned");
  int threads = 0, grid = 0;
  reshape_launch_shape(num_tokens, num_heads, head_dim, &threads, &grid);
  cudaError_t e = pkv::launch_pdl(reshape_and_cache_kernel, dim3(grid), dim3(threads), 0,
                                  static_cast<cudaStream_t>(stream), reinterpret_cast<const uint4*>(key),
                                  reinterpret_cast<const uint4*>(value), reinterpret_cast<uint4*>(k_cache),
                                  reinterpret_cast<uint4*>(v_cache), slot_mapping, num_tokens, num_heads,
                                  ilog2(head_dim / 8), ilog2(block_size), static_cast<int64_t>(num_blocks) * block_size);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "pkv_reshape_and_cache launch: %s", cudaGetErrorString(e));
  pkv::clear_error();
  return PKV_OK;
}

int pkv_copy_blocks(uint16_t* const* k_caches, uint16_t* const* v_caches, int num_layers,
                    const int64_t* block_mapping, int num_pairs, int num_heads, int head_dim, int block_size,
                    int num_blocks, void* stream) {
  int rc = check_shape("pkv_copy_blocks", num_heads, head_dim, block_size, num_blocks);
  if (rc != PKV_OK) return rc;
  if (num_pairs < 0 || num_layers < 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_copy_blocks: num_pairs=%d num_layers=%d", num_pairs, num_layers);
  if (num_pairs == 0 || num_layers == 0) {
    pkv::clear_error();
    return PKV_OK;
  }
  if (!k_caches || !v_caches || !block_mapping)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_copy_blocks: null pointer");
  for (int l = 0; l < num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
      return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_copy_blocks: layer %d cache pointer null or not 16-byte aligned", l);
  }
  const int64_t vec_per_block = static_cast<int64_t>(num_heads) * block_size * head_dim / 8;
  // enough CTAs per pair to keep every SM streaming even when there are few pairs
  int splits = static_cast<int>((vec_per_block + 256 * 8 - 1) / (256 * 8));
  if (splits < 1) splits = 1;
  if (splits > 64) splits = 64;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
    const int nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0 : kMaxLayersPerLaunch;
    LayerPtrs ptrs{};
    for (int l = 0; l < nl; ++l) {
      ptrs.k[l] = reinterpret_cast<uint4*>(k_caches[l0 + l]);
      ptrs.v[l] = reinterpret_cast<uint4*>(v_caches[l0 + l]);
    }
    cudaError_t e = pkv::launch_pdl(copy_blocks_kernel, dim3(num_pairs, nl, splits), dim3(256), 0, st, ptrs,
                                    block_mapping, vec_per_block, num_blocks);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "pkv_copy_blocks launch: %s", cudaGetErrorString(e));
  }
  pkv::clear_error();
  return PKV_OK;
}

int pkv_swap_blocks(const uint16_t* const* src_k_caches, const uint16_t* const* src_v_caches,
                    uint16_t* const* dst_k_caches, uint16_t* const* dst_v_caches, int num_layers,
                    const int64_t* block_mapping, int num_pairs, int num_heads, int head_dim, int block_size,
                    int src_num_blocks, int dst_num_blocks, void* stream) {
  int rc = check_shape("pkv_swap_blocks", num_heads, head_dim, block_size, src_num_blocks);
  if (rc != PKV_OK) return rc;
  if (dst_num_blocks <= 0 || num_pairs < 0 || num_layers < 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_swap_blocks: dst_num_blocks=%d num_pairs=%d num_layers=%d",
                     dst_num_blocks, num_pairs, num_layers);
  if (num_pairs == 0 || num_layers == 0) {
    pkv::clear_error();
    return PKV_OK;
  }
  if (!src_k_caches || !src_v_caches || !dst_k_caches || !dst_v_caches || !block_mapping)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_swap_blocks: null pointer");
  if (!device_accessible(block_mapping))
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_swap_blocks: block_mapping is not device-accessible memory");
  for (int l = 0; l < num_layers; ++l) {
    const void* p4[4] = {src_k_caches[l], src_v_caches[l], dst_k_caches[l], dst_v_caches[l]};
    for (const void* ptr : p4) {
      if (!ptr || !aligned16(ptr))
        return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_swap_blocks: layer %d pool pointer null or not 16-byte aligned", l);
      if (!device_accessible(ptr))
        return pkv::fail(PKV_ERR_INVALID_ARG,
                         "pkv_swap_blocks: layer %d pool is neither device memory nor page-locked host memory", l);
    }
  }
  const int64_t vec_per_block = static_cast<int64_t>(num_heads) * block_size * head_dim / 8;
  int splits = static_cast<int>((vec_per_block + 256 * 8 - 1) / (256 * 8));
  if (splits < 1) splits = 1;
  if (splits > 64) splits = 64;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
    const int nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0 : kMaxLayersPerLaunch;
    PoolPairPtrs ptrs{};
    for (int l = 0; l < nl; ++l) {
      ptrs.src_k[l] = reinterpret_cast<const uint4*>(src_k_caches[l0 + l]);
      ptrs.src_v[l] = reinterpret_cast<const uint4*>(src_v_caches[l0 + l]);
      ptrs.dst_k[l] = reinterpret_cast<uint4*>(dst_k_caches[l0 + l]);
      ptrs.dst_v[l] = reinterpret_cast<uint4*>(dst_v_caches[l0 + l]);
    }
    cudaError_t e = pkv::launch_pdl(swap_blocks_kernel, dim3(num_pairs, nl, splits), dim3(256), 0, st, ptrs,
                                    block_mapping, vec_per_block, src_num_blocks, dst_num_blocks);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "pkv_swap_blocks launch: %s", cudaGetErrorString(e));
  }
  pkv::clear_error();
  return PKV_OK;
}

int pkv_reshape_and_cache_layers(const uint16_t* const* keys, const uint16_t* const* values, uint16_t* const* k_caches,
                                 uint16_t* const* v_caches, int num_layers, const int64_t* slot_mapping, int num_tokens,
                                 int num_heads, int head_dim, int block_size, int num_blocks, void* stream) {
  int rc = check_shape("pkv_reshape_and_cache_layers", num_heads, head_dim, block_size, num_blocks);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0 || num_layers < 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_reshape_and_cache_layers: num_tokens=%d num_layers=%d", num_tokens,
                     num_layers);
  if (num_tokens == 0 || num_layers == 0) {
    pkv::clear_error();
    return PKV_OK;
  }
  if (!keys || !values || !k_caches || !v_caches || !slot_mapping)
    return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_reshape_and_cache_layers: null pointer");
  for (int l = 0; l < num_layers; ++l) {
    const void* p4[4] = {keys[l], values[l], k_caches[l], v_caches[l]};
    for (const void* ptr : p4)
      if (!ptr || !aligned16(ptr))
        return pkv::fail(PKV_ERR_INVALID_ARG, "pkv_reshape_and_cache_layers: layer %d pointer null or not 16-byte aligned", l);
  }
  int threads = 0, grid = 0;
  reshape_launch_shape(num_tokens, num_heads, head_dim, &threads, &grid);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
    const int nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0 : kMaxLayersPerLaunch;
    TokenLayerPtrs ptrs{};
    for (int l = 0; l < nl; ++l) {
      ptrs.key[l] = reinterpret_cast<const uint4*>(keys[l0 + l]);
      ptrs.value[l] = reinterpret_cast<const uint4*>(values[l0 + l]);
      ptrs.k_cache[l] = reinterpret_cast<uint4*>(k_caches[l0 + l]);
      ptrs.v_cache[l] = reinterpret_cast<uint4*>(v_caches[l0 + l]);
    }
    cudaError_t e = pkv::launch_pdl(reshape_and_cache_layers_kernel, dim3(grid, nl), dim3(threads), 0, st, ptrs,
                                    slot_mapping, num_tokens, num_heads, ilog2(head_dim / 8), ilog2(block_size),
                                    static_cast<int64_t>(num_blocks) * block_size);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess)
      return pkv::fail(PKV_ERR_CUDA, "pkv_reshape_and_cache_layers launch: %s", cudaGetErrorString(e));
  }
  pkv::clear_error();
  return PKV_OK;
}

}  // extern "C"
