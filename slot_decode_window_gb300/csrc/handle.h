// Internal: the window handle, shared by the window and stack entry points.
#pragma once
#include "common.cuh"
#include "strata_window.h"

// One instantiated CUDA graph of a window launch, keyed by its arguments.
struct strata_graph_entry {
  int T = 0;
  const float* x = nullptr;
  float* y = nullptr;
  cudaGraphExec_t exec = nullptr;
  unsigned long long last_use = 0;
};
constexpr int kGraphCache = 16;  // graphs a handle keeps (least recently used evicted)

struct strata_window {
  strata_moe_desc desc;
  int device = 0;
  int nsm = 0;
  strata::LayerDev L{};
  strata::WindowBufs W{};
  strata::KernelCfg cfg{};
  float* partial = nullptr;
  void* wmem = nullptr;
  void* ws = nullptr;
  long long packed = 0, ws_bytes = 0;
  cudaEvent_t done = nullptr;
  bool profiling = false;
  bool profiled_once = false;
  cudaEvent_t prof[2] = {nullptr, nullptr};
  strata_graph_entry graphs[kGraphCache];
  unsigned long long graph_clock = 0;
  cudaStream_t capture_stream = nullptr;
};

namespace strata {
// The STRATA_FAULT test hook: true when the environment names `what`.
bool fault_is(const char* what);
// An integer from the environment, or dflt when unset, malformed or outside [lo, hi].
long long env_int(const char* name, long long dflt, long long lo, long long hi);
}  // namespace strata
