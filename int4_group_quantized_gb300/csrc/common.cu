// Host-side utilities of libfg.so: error strings, the device error word and
// device queries.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <vector>

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

static std::atomic<uint32_t> g_wait_limit{FG_WAIT_LIMIT_DEFAULT};
uint32_t wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

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

// ---- launch tracing ----------------------------------------------------------
namespace {
const char* const kClassNames[KC_COUNT] = {
    "quantize_g64", "dequant_g64", "kv_store_q4", "gemm_simt", "gemm_tc",
    "gemm_splitk_reduce", "attn_decode", "attn_decode_combine", "attn_prefill", "gemm_q4_decode",
    "pack_weight", "attn_decode_topk"};

// Launches of the same class that follow one another on a stream form one
// timed run (one event pair): events between them would break the overlap
// that programmatic dependent launch gives consecutive products, and add each
// launch's gap to its time.  A run ends at the next launch of another class,
// at a phase change and at fg_profile_stop.
struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> ev;   // 2 per run
  std::vector<int> cls;          // class + KC_COUNT * phase, per run
  std::vector<int64_t> count;    // launches per run
  size_t used = 0;
  int64_t dropped = 0;
  int phase = 0;
  int open = -1;                 // run still accepting launches
  cudaStream_t open_st = nullptr;
  int64_t launches[kProfilePhases * KC_COUNT] = {0};
  double ms[kProfilePhases * KC_COUNT] = {0};
};
Profiler g_prof;
std::atomic<uint64_t> g_launches{0};

void close_run_locked() {
  if (g_prof.open >= 0) {
    cudaEventRecord(g_prof.ev[2 * g_prof.open + 1], g_prof.open_st);
    g_prof.open = -1;
  }
}
}  // namespace

void trace_begin(int c, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_prof.on) return;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.on) return;
  const int key = c + KC_COUNT * g_prof.phase;
  if (g_prof.open >= 0 && g_prof.cls[g_prof.open] == key && g_prof.open_st == st) {
    ++g_prof.count[g_prof.open];
    return;
  }
  close_run_locked();
  if (g_prof.used >= g_prof.cls.size()) {
    ++g_prof.dropped;
    return;
  }
  const size_t i = g_prof.used++;
  g_prof.cls[i] = key;
  g_prof.count[i] = 1;
  cudaEventRecord(g_prof.ev[2 * i], st);
  g_prof.open = static_cast<int>(i);
  g_prof.open_st = st;
}

void trace_extra_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
void count_launches_undo(uint64_t n) { g_launches.fetch_sub(n, std::memory_order_relaxed); }
bool profiling() { return g_prof.on; }

void trace_end(int c, cudaStream_t st) {
  (void)c;
  (void)st;   // runs are closed by the next launch of another class
}

}  // namespace fg

extern "C" {

fg_status fg_profile_start(int32_t max_launches) {
  using fg::g_prof;
  if (max_launches <= 0) return fg::fail(FG_ERR_ARG, "max_launches");
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.on) return fg::fail(FG_ERR_ARG, "profiling already active");
  const size_t need = 2 * static_cast<size_t>(max_launches);
  while (g_prof.ev.size() < need) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return fg::fail(FG_ERR_CUDA, "cudaEventCreate");
    g_prof.ev.push_back(e);
  }
  g_prof.cls.assign(max_launches, 0);
  g_prof.count.assign(max_launches, 0);
  g_prof.open = -1;
  g_prof.used = 0;
  g_prof.dropped = 0;
  for (int i = 0; i < fg::kProfilePhases * fg::KC_COUNT; ++i) {
    g_prof.launches[i] = 0;
    g_prof.ms[i] = 0;
  }
  g_prof.phase = 0;
  g_prof.on = true;
  return FG_OK;
}

fg_status fg_profile_stop(void) {
  using fg::g_prof;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.on) return fg::fail(FG_ERR_ARG, "profiling not active");
  fg::close_run_locked();
  g_prof.on = false;
  for (size_t i = 0; i < g_prof.used; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess)
      return fg::fail(FG_ERR_CUDA, "event timing");
    g_prof.launches[g_prof.cls[i]] += g_prof.count[i];
    g_prof.ms[g_prof.cls[i]] += ms;
  }
  return g_prof.dropped ? fg::fail(FG_ERR_WORKSPACE, "%lld launches not timed (pool full)",
                                   (long long)g_prof.dropped)
                        : FG_OK;
}

int32_t fg_profile_kernel_classes(void) { return fg::KC_COUNT; }

const char* fg_profile_kernel_name(int32_t i) {
  return (i >= 0 && i < fg::KC_COUNT) ? fg::kClassNames[i] : "";
}

fg_status fg_profile_phase(int32_t phase) {
  if (phase < 0 || phase >= fg::kProfilePhases) return fg::fail(FG_ERR_ARG, "phase");
  std::lock_guard<std::mutex> lk(fg::g_prof.mu);
  fg::close_run_locked();
  fg::g_prof.phase = phase;
  return FG_OK;
}

fg_status fg_profile_query(int32_t phase, int32_t i, int64_t* launches, double* total_ms) {
  if (phase < 0 || phase >= fg::kProfilePhases || i < 0 || i >= fg::KC_COUNT || !launches ||
      !total_ms)
    return fg::fail(FG_ERR_ARG, "phase/class");
  *launches = fg::g_prof.launches[phase * fg::KC_COUNT + i];
  *total_ms = fg::g_prof.ms[phase * fg::KC_COUNT + i];
  return FG_OK;
}

uint64_t fg_launch_count(void) { return fg::g_launches.load(); }

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

uint32_t fg_set_wait_limit(uint32_t polls) { return fg::g_wait_limit.exchange(polls); }

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
