// Host-side utilities of libfg.so: error strings, the device error word and
// device queries.
#include <stdarg.h>
#include <stdio.h>

#include "fg_internal.cuh"

namespace fg {

static thread_local char g_detail[512] = "";

fg_status fail(fg_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return s;
}

fg_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return FG_OK;
}

static constexpr int kMaxDevices = 64;

int num_sms() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

__device__ unsigned int g_device_error_word = 0;

unsigned int* device_error_word() {
  static unsigned int* cache[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned int*>(p);
  }
  return cache[dev];
}

}  // namespace fg

extern "C" {

const char* fg_status_str(fg_status s) {
  switch (s) {
    case FG_OK: return "FG_OK";
    case FG_ERR_ARG: return "FG_ERR_ARG";
    case FG_ERR_SHAPE: return "FG_ERR_SHAPE";
    case FG_ERR_ALIGN: return "FG_ERR_ALIGN";
    case FG_ERR_CAPACITY: return "FG_ERR_CAPACITY";
    case FG_ERR_WORKSPACE: return "FG_ERR_WORKSPACE";
    case FG_ERR_CUDA: return "FG_ERR_CUDA";
    case FG_ERR_DEVICE_TIMEOUT: return "FG_ERR_DEVICE_TIMEOUT";
    case FG_ERR_UNSUPPORTED: return "FG_ERR_UNSUPPORTED";
  }
  return "FG_ERR_UNKNOWN";
}

const char* fg_last_error(void) { return fg::g_detail; }

const char* fg_version(void) { return "fg 0.1 sm_103a"; }

fg_status fg_sync_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fg::fail(FG_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
  unsigned int* w = fg::device_error_word();
  if (w == nullptr) return fg::fail(FG_ERR_CUDA, "error word unavailable");
  unsigned int v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fg::fail(FG_ERR_CUDA, "error word read: %s", cudaGetErrorString(e));
  if (v != 0) {
    unsigned int zero = 0;
    cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    return fg::fail(FG_ERR_DEVICE_TIMEOUT, "device error word 0x%x", v);
  }
  return FG_OK;
}

}  // extern "C"
