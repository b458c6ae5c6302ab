// Error reporting and version entry points of the C ABI.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "pkv_internal.h"

namespace pkv {

static thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

void clear_error() { g_last_error.clear(); }

}  // namespace pkv

extern "C" {

const char* pkv_last_error(void) { return pkv::g_last_error.c_str(); }

int pkv_version(void) { return 100; }

int pkv_device_error(void* stream, int reset, int* code) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return pkv::fail(PKV_ERR_CUDA, "pkv_device_error: cudaStreamSynchronize: %s", cudaGetErrorString(e));
  int a = 0, c = 0, f = 0;
  int st = pkv::read_device_error_attention(reset, &a);
  if (st != PKV_OK) return st;
  st = pkv::read_device_error_cache_ops(reset, &c);
  if (st != PKV_OK) return st;
  st = pkv::read_device_error_prefill(reset, &f);
  if (st != PKV_OK) return st;
  int first = a ? a : (c ? c : f);
  if (code) *code = first;
  if (first) return pkv::fail(PKV_ERR_DEVICE_CHECK, "a kernel recorded device check code %d", first);
  return PKV_OK;
}

}  // extern "C"
