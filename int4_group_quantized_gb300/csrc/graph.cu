// Decode steps replayed as CUDA graphs (FlexGen notes, "4. 卸载策略": the
// zig-zag block runs the same loop over the layers at every decode step).
//
// A decode step of a block is ~9 launches per layer.  For small layers the
// host's launch rate, not the GPU, sets the step time.  The first call of a
// step with given arguments runs it directly; it then records the same
// launches into a CUDA graph (stream capture: nothing runs) and keeps the
// instantiated graph.  Later calls with the same arguments launch the graph:
// one host call per step, the kernels (and their programmatic dependent
// launches) in the order the direct call issues them.
//
// The key is every argument of the step (pointers and sizes) and the bytes
// of the layer and cache structures it reads, so a change to any of them
// makes a new graph.  A graph reads and writes memory through the pointers
// it was recorded with: the buffers must stay allocated while the cache
// holds graphs for them.
#include <string.h>

#include <map>
#include <mutex>
#include <string>

#include "fg_internal.cuh"

struct fg_graph_cache {
  std::mutex mu;
  struct Entry {
    cudaGraphExec_t exec = nullptr;
    uint64_t launches = 0;   // kernels one replay launches
  };
  std::map<std::string, Entry> steps;
  // Steps are recorded on a stream of the cache's own: the legacy default
  // stream cannot be captured, and recording runs nothing, so the stream the
  // caller names needs no part in it.
  cudaStream_t capture = nullptr;
  int capture_dev = -1;
  std::mutex capture_mu;
};

namespace {

std::string step_key(const fg_layer* layers, int32_t l, const void* t, int64_t b, int64_t pos, const fg_kv* kvs,
                     const void* y, const void* ws, size_t ws_bytes) {
  std::string k;
  auto put = [&k](const void* p, size_t n) { k.append(static_cast<const char*>(p), n); };
  put(&l, sizeof(l));
  put(&t, sizeof(t));
  put(&b, sizeof(b));
  put(&pos, sizeof(pos));
  put(&y, sizeof(y));
  put(&ws, sizeof(ws));
  put(&ws_bytes, sizeof(ws_bytes));
  put(layers, sizeof(fg_layer) * static_cast<size_t>(l));
  put(kvs, sizeof(fg_kv) * static_cast<size_t>(l));
  return k;
}

}  // namespace

extern "C" {

fg_status fg_graph_cache_create(fg_graph_cache** out) {   // no CUDA call until the first recording
  if (!out) return fg::fail(FG_ERR_ARG, "null output");
  *out = new (std::nothrow) fg_graph_cache();
  return *out ? FG_OK : fg::fail(FG_ERR_ARG, "out of host memory");
}

void fg_graph_cache_destroy(fg_graph_cache* c) {
  if (!c) return;
  for (auto& kv : c->steps)
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
  if (c->capture) cudaStreamDestroy(c->capture);
  delete c;
}

int64_t fg_graph_cache_size(const fg_graph_cache* c) { return c ? static_cast<int64_t>(c->steps.size()) : 0; }

fg_status fg_decode_block_step_graphed(fg_graph_cache* c, const fg_layer* layers, int32_t l, const void* t,
                                       int64_t b, int64_t pos, const fg_kv* kvs, void* y, void* ws,
                                       size_t ws_bytes, cudaStream_t stream) {
  if (!c) return fg::fail(FG_ERR_ARG, "null graph cache");
  if (!layers || !kvs || l <= 0) return fg::fail(FG_ERR_ARG, "layers/kvs/l");
  const std::string key = step_key(layers, l, t, b, pos, kvs, y, ws, ws_bytes);
  {
    std::lock_guard<std::mutex> lk(c->mu);
    auto it = c->steps.find(key);
    if (it != c->steps.end()) {
      if (cudaGraphLaunch(it->second.exec, stream) != cudaSuccess) return fg::check_launch("cudaGraphLaunch");
      fg::count_launches(it->second.launches);
      return FG_OK;
    }
  }
  // first call with these arguments: run the step (it checks them), then
  // record it; a stream already being captured, or the profiler, get the
  // direct call only
  FG_TRY(fg_decode_block_step(layers, l, t, b, pos, kvs, y, ws, ws_bytes, stream));
  if (b == 0 || fg::profiling()) return FG_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return fg::check_launch("cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone) return FG_OK;
  std::lock_guard<std::mutex> cap(c->capture_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fg::check_launch("cudaGetDevice");
  if (c->capture && c->capture_dev != dev) {
    cudaStreamDestroy(c->capture);
    c->capture = nullptr;
  }
  if (!c->capture) {
    if (cudaStreamCreateWithFlags(&c->capture, cudaStreamNonBlocking) != cudaSuccess)
      return fg::check_launch("cudaStreamCreateWithFlags");
    c->capture_dev = dev;
  }
  const uint64_t n0 = fg_launch_count();
  if (cudaStreamBeginCapture(c->capture, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return fg::check_launch("cudaStreamBeginCapture");
  const fg_status s = fg_decode_block_step(layers, l, t, b, pos, kvs, y, ws, ws_bytes, c->capture);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(c->capture, &g);
  const uint64_t recorded = fg_launch_count() - n0;
  fg::count_launches_undo(recorded);   // recorded, not run
  if (s != FG_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return s != FG_OK ? s : fg::fail(FG_ERR_CUDA, "stream capture of a decode step: %s", cudaGetErrorString(e));
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&exec, g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess) {
    cudaGetLastError();
    return fg::fail(FG_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(ie));
  }
  std::lock_guard<std::mutex> lk(c->mu);
  auto& ent = c->steps[key];
  if (ent.exec) cudaGraphExecDestroy(ent.exec);   // another thread recorded the same step meanwhile
  ent.exec = exec;
  ent.launches = recorded;
  return FG_OK;
}

}  // extern "C"
