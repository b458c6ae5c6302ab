/*
 * A plain C caller of libpkv.so: one decode step of a small batch with nothing but the C ABI and
 * the CUDA runtime (no Python, no PyTorch).
 *
 *   decode_step <dir> <num_seqs> <num_heads> <head_dim> <block_size> <num_blocks>
 *
 * <dir> holds, written by the test that runs this program:
 *   prompts.i32   [num_seqs]                         prompt length of each sequence
 *   order.i32     [num_blocks]                       the block manager's free-list order
 *   k.f16, v.f16  [num_blocks, H, B, D]              K/V pools, prompts already in place
 *   q.f16         [num_seqs, H, D]                   this step's queries
 *   key.f16, value.f16 [num_seqs, H, D]              this step's new K/V rows
 * and receives:
 *   tables.i32 [num_seqs, max_blocks], lens.i32 [num_seqs]   the manager's tables after the step
 *   out.f16         the fused step's output (pkv_paged_attention_decode_append, caller workspace)
 *   out_static.f16  the same attention through pkv_paged_attention_decode_static_workspace
 *   k_after.f16, v_after.f16  the pools after the step
 *
 * The block manager assigns each sequence's new slot (pkv_bm_append_slots) and writes the tables
 * (pkv_bm_block_tables); copy-on-write pairs, if any, go through pkv_copy_blocks first.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pkv.h"

static int fail(const char* what, int rc) {
  fprintf(stderr, "%s: status %d: %s\n", what, rc, pkv_last_error());
  return 1;
}

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes);
  size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : 1;
}

#define CUDA_OK(call)                                                              \
  do {                                                                             \
    cudaError_t e_ = (call);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                  \
      return 1;                                                                    \
    }                                                                              \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 7) {
    fprintf(stderr, "usage: %s dir num_seqs num_heads head_dim block_size num_blocks\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  const int S = atoi(argv[2]), H = atoi(argv[3]), D = atoi(argv[4]), B = atoi(argv[5]), N = atoi(argv[6]);
  const size_t pool_elems = (size_t)N * H * B * D, row_elems = (size_t)S * H * D;

  int32_t* prompts = (int32_t*)read_file(dir, "prompts.i32", sizeof(int32_t) * S);
  int32_t* order = (int32_t*)read_file(dir, "order.i32", sizeof(int32_t) * N);
  uint16_t* k_h = (uint16_t*)read_file(dir, "k.f16", 2 * pool_elems);
  uint16_t* v_h = (uint16_t*)read_file(dir, "v.f16", 2 * pool_elems);
  uint16_t* q_h = (uint16_t*)read_file(dir, "q.f16", 2 * row_elems);
  uint16_t* key_h = (uint16_t*)read_file(dir, "key.f16", 2 * row_elems);
  uint16_t* value_h = (uint16_t*)read_file(dir, "value.f16", 2 * row_elems);
  if (!prompts || !order || !k_h || !v_h || !q_h || !key_h || !value_h) {
    fprintf(stderr, "missing or short input file in %s\n", dir);
    return 1;
  }

  /* host: the block manager places the prompts, then this step's token of every sequence */
  pkv_bm* bm = pkv_bm_create(N, B, order);
  if (!bm) return fail("pkv_bm_create", PKV_ERR_INVALID_ARG);
  int max_len = 0;
  for (int s = 0; s < S; ++s) {
    int rc = pkv_bm_add_seq(bm, s, prompts[s], NULL);
    if (rc != PKV_OK) return fail("pkv_bm_add_seq", rc);
    if (prompts[s] + 1 > max_len) max_len = prompts[s] + 1;
  }
  const int max_blocks = (max_len + B - 1) / B;
  int64_t* ids = (int64_t*)malloc(sizeof(int64_t) * S);
  int64_t* slots = (int64_t*)malloc(sizeof(int64_t) * S);
  int64_t* pairs = (int64_t*)malloc(sizeof(int64_t) * 2 * S);
  int32_t* tables = (int32_t*)malloc(sizeof(int32_t) * S * max_blocks);
  int32_t* lens = (int32_t*)malloc(sizeof(int32_t) * S);
  for (int s = 0; s < S; ++s) ids[s] = s;
  int num_cow = 0;
  int rc = pkv_bm_append_slots(bm, ids, S, slots, pairs, &num_cow);
  if (rc != PKV_OK) return fail("pkv_bm_append_slots", rc);
  rc = pkv_bm_block_tables(bm, ids, S, tables, max_blocks, lens);
  if (rc != PKV_OK) return fail("pkv_bm_block_tables", rc);

  /* device: buffers owned by this caller */
  uint16_t *k_d, *v_d, *q_d, *key_d, *value_d, *out_d, *out2_d;
  int32_t *tables_d, *lens_d;
  int64_t *slots_d, *pairs_d;
  CUDA_OK(cudaMalloc((void**)&k_d, 2 * pool_elems));
  CUDA_OK(cudaMalloc((void**)&v_d, 2 * pool_elems));
  CUDA_OK(cudaMalloc((void**)&q_d, 2 * row_elems));
  CUDA_OK(cudaMalloc((void**)&key_d, 2 * row_elems));
  CUDA_OK(cudaMalloc((void**)&value_d, 2 * row_elems));
  CUDA_OK(cudaMalloc((void**)&out_d, 2 * row_elems));
  CUDA_OK(cudaMalloc((void**)&out2_d, 2 * row_elems));
  CUDA_OK(cudaMalloc((void**)&tables_d, sizeof(int32_t) * S * max_blocks));
  CUDA_OK(cudaMalloc((void**)&lens_d, sizeof(int32_t) * S));
  CUDA_OK(cudaMalloc((void**)&slots_d, sizeof(int64_t) * S));
  CUDA_OK(cudaMalloc((void**)&pairs_d, sizeof(int64_t) * 2 * (num_cow > 0 ? num_cow : 1)));
  CUDA_OK(cudaMemcpy(k_d, k_h, 2 * pool_elems, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(v_d, v_h, 2 * pool_elems, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(q_d, q_h, 2 * row_elems, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(key_d, key_h, 2 * row_elems, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(value_d, value_h, 2 * row_elems, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(tables_d, tables, sizeof(int32_t) * S * max_blocks, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(lens_d, lens, sizeof(int32_t) * S, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(slots_d, slots, sizeof(int64_t) * S, cudaMemcpyHostToDevice));
  const size_t ws_bytes = pkv_paged_attention_workspace_size(S, H, D, max_blocks, B);
  void* ws_d = NULL;
  if (ws_bytes) CUDA_OK(cudaMalloc(&ws_d, ws_bytes));
  cudaStream_t st;
  CUDA_OK(cudaStreamCreate(&st));

  const float scale = 1.0f / sqrtf((float)D);
  if (num_cow > 0) {
    CUDA_OK(cudaMemcpy(pairs_d, pairs, sizeof(int64_t) * 2 * num_cow, cudaMemcpyHostToDevice));
    uint16_t* kl[1] = {k_d};
    uint16_t* vl[1] = {v_d};
    rc = pkv_copy_blocks(kl, vl, 1, pairs_d, num_cow, H, D, B, N, st);
    if (rc != PKV_OK) return fail("pkv_copy_blocks", rc);
  }
  rc = pkv_paged_attention_decode_append(q_d, key_d, value_d, slots_d, k_d, v_d, tables_d, lens_d, S, H, D, N,
                                         max_blocks, scale, B, out_d, ws_d, ws_bytes, st);
  if (rc != PKV_OK) return fail("pkv_paged_attention_decode_append", rc);
  rc = pkv_paged_attention_decode_static_workspace(q_d, k_d, v_d, tables_d, lens_d, S, H, D, N, max_blocks, scale,
                                                   B, out2_d, st);
  if (rc != PKV_OK) return fail("pkv_paged_attention_decode_static_workspace", rc);
  int code = 0;
  rc = pkv_device_error(st, 1, &code);
  if (rc != PKV_OK) return fail("pkv_device_error", rc);

  uint16_t* out_h = (uint16_t*)malloc(2 * row_elems);
  uint16_t* out2_h = (uint16_t*)malloc(2 * row_elems);
  CUDA_OK(cudaMemcpy(out_h, out_d, 2 * row_elems, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out2_h, out2_d, 2 * row_elems, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(k_h, k_d, 2 * pool_elems, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(v_h, v_d, 2 * pool_elems, cudaMemcpyDeviceToHost));
  int bad = write_file(dir, "tables.i32", tables, sizeof(int32_t) * S * max_blocks) |
            write_file(dir, "lens.i32", lens, sizeof(int32_t) * S) |
            write_file(dir, "slots.i64", slots, sizeof(int64_t) * S) |
            write_file(dir, "out.f16", out_h, 2 * row_elems) |
            write_file(dir, "out_static.f16", out2_h, 2 * row_elems) |
            write_file(dir, "k_after.f16", k_h, 2 * pool_elems) |
            write_file(dir, "v_after.f16", v_h, 2 * pool_elems);
  if (bad) {
    fprintf(stderr, "writing the results to %s failed\n", dir);
    return 1;
  }
  printf("ok max_blocks=%d num_cow=%d workspace=%zu\n", max_blocks, num_cow, ws_bytes);

  cudaStreamDestroy(st);
  cudaFree(k_d); cudaFree(v_d); cudaFree(q_d); cudaFree(key_d); cudaFree(value_d); cudaFree(out_d);
  cudaFree(out2_d); cudaFree(tables_d); cudaFree(lens_d); cudaFree(slots_d); cudaFree(pairs_d);
  if (ws_d) cudaFree(ws_d);
  pkv_bm_destroy(bm);
  free(prompts); free(order); free(k_h); free(v_h); free(q_h); free(key_h); free(value_h);
  free(ids); free(slots); free(pairs); free(tables); free(lens); free(out_h); free(out2_h);
  return 0;
}
