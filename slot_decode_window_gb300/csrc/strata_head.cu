// C ABI of the window's output head: the head matrix repacked into the kernel
// tile format, a workspace for the head kernel, and the per-window launch
// (RMSNorm, the head GEMV, each row's token and each slot's proposal check in
// one cooperative launch; head_kernel in window.cu).
#include <cstring>
#include <new>

#include "common.cuh"
#include "handle.h"
#include "kernels.h"
#include "strata_window.h"

using namespace strata;

struct strata_head {
  strata_head_desc desc;
  int device = 0, nsm = 0;
  LayerDev L{};
  WindowBufs W{};
  KernelCfg cfg{};
  HeadArgs H{};
  void* wmem = nullptr;
  void* ws = nullptr;
  float* logits = nullptr;  // workspace logits [max_rows][V]
  long long ws_bytes = 0;
  cudaEvent_t done = nullptr;
  bool profiling = false, profiled_once = false;
  cudaEvent_t prof[2] = {nullptr, nullptr};
};

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

void free_head(strata_head* h) {
  if (!h) return;
  if (h->done) cudaEventDestroy(h->done);
  for (cudaEvent_t& ev : h->prof)
    if (ev) cudaEventDestroy(ev);
  if (h->wmem) cudaFree(h->wmem);
  if (h->ws) cudaFree(h->ws);
  delete h;
}

strata_status check_head_desc(const strata_head_desc* d) {
  if (!d) return STRATA_EINVAL;
  if (d->hidden <= 0 || d->vocab <= 0 || d->max_rows < 1 || d->max_rows > kMaxRows) return STRATA_EINVAL;
  if (!((d->bits == 4 && d->block == 32) || (d->bits == 2 && d->block == 16))) return STRATA_EUNSUPPORTED;
  const int ks = d->bits == 4 ? 64 : 128;
  if (d->hidden % ks != 0 || d->hidden > 16384 || d->vocab % 16 != 0 || d->vocab > (1 << 22))
    return STRATA_EUNSUPPORTED;
  return STRATA_OK;
}

}  // namespace

extern "C" {

strata_status strata_head_create(const strata_head_desc* desc, const strata_qmat* weight, void* cuda_stream,
                                 strata_head** out) {
  if (!out) return STRATA_EINVAL;
  *out = nullptr;
  strata_status st = check_head_desc(desc);
  if (st != STRATA_OK) return st;
  if (!weight || !weight->codes || !weight->scale || !weight->min) return STRATA_EINVAL;
  if (fault_is("alloc")) return STRATA_ENOMEM;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  strata_head* h = new (std::nothrow) strata_head();
  if (!h) return STRATA_ENOMEM;
  h->desc = *desc;
  const int d = desc->hidden, V = desc->vocab, bits = desc->bits, block = desc->block;
  int optin = 0;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->nsm, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess) {
    cudaGetLastError();
    free_head(h);
    return STRATA_ECUDA;
  }
  const long long pbytes = packed_bytes(1, V, d, bits);
  if (cudaMalloc(&h->wmem, (size_t)pbytes) != cudaSuccess) {
    cudaGetLastError();
    free_head(h);
    return STRATA_ENOMEM;
  }
  // workspace: error word, barrier word, x fragments, logits, per-CTA partials
  const int nmk = (d / block + 15) / 16;
  size_t w = 0;
  const size_t o_err = w; w = align_up(w + 8, 256);
  const size_t o_gbar = w; w = align_up(w + 8, 256);
  const size_t o_xf = w; w = align_up(w + (size_t)kMaxRows * frag_halves(d, nmk) * 2, 256);
  const size_t o_lg = w; w = align_up(w + (size_t)kMaxRows * V * 4, 256);
  const size_t o_pm = w; w = align_up(w + (size_t)h->nsm * kMaxRows * 4, 256);
  const size_t o_pa = w; w = align_up(w + (size_t)h->nsm * kMaxRows * 4, 256);
  const size_t o_ps = w; w = align_up(w + (size_t)h->nsm * kMaxRows * 4, 256);
  h->ws_bytes = (long long)w;
  if (cudaMalloc(&h->ws, w) != cudaSuccess) {
    cudaGetLastError();
    free_head(h);
    return STRATA_ENOMEM;
  }
  uint8_t* wsb = static_cast<uint8_t*>(h->ws);
  cudaError_t e = cudaMemsetAsync(h->ws, 0, w, s);
  if (e == cudaSuccess)
    e = launch_repack(static_cast<const uint8_t*>(weight->codes), weight->scale, weight->min, 1, V, d, bits,
                      static_cast<uint8_t*>(h->wmem), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->done, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_head(h);
    return STRATA_ECUDA;
  }
  LayerDev& L = h->L;
  L.d = d;
  L.E = 1;
  L.k = 1;
  L.F = d;
  L.Fs = 0;
  L.bits = bits;
  L.qkv = packed_desc(static_cast<const uint8_t*>(h->wmem), V, d, bits);
  L.dq = V;
  L.dkv = 0;
  WindowBufs& W = h->W;
  W.err = reinterpret_cast<unsigned*>(wsb + o_err);
  W.gbar = reinterpret_cast<unsigned long long*>(wsb + o_gbar);
  W.xfrag = reinterpret_cast<__half*>(wsb + o_xf);
  W.wait_cycles = env_int("STRATA_WAIT_CYCLES", 1LL << 31, 1000, 1LL << 40);
  W.bar_extra = (int)env_int("STRATA_TEST_BARRIER_EXTRA", 0, 0, 1 << 20);
  h->logits = reinterpret_cast<float*>(wsb + o_lg);
  h->H.part_max = reinterpret_cast<float*>(wsb + o_pm);
  h->H.part_arg = reinterpret_cast<int*>(wsb + o_pa);
  h->H.part_sum = reinterpret_cast<float*>(wsb + o_ps);
  h->H.V = V;
  h->cfg = head_cfg(d, bits, desc->max_rows, optin - 12288);
  if (h->cfg.nstages < 2) {
    free_head(h);
    return STRATA_EUNSUPPORTED;
  }
  if (head_set_attrs(bits, h->cfg.total_bytes) != cudaSuccess) {
    cudaGetLastError();
    free_head(h);
    return STRATA_ECUDA;
  }
  if (head_blocks_per_sm(bits, h->cfg.total_bytes) < 1) {
    free_head(h);
    return STRATA_EUNSUPPORTED;
  }
  *out = h;
  return STRATA_OK;
}

strata_status strata_head_forward(strata_head* h, const float* x, int32_t T, const strata_draw_in* in,
                                  const strata_draw_out* out, void* cuda_stream) {
  if (!h || !x || !in || !out) return STRATA_EINVAL;
  if (T < 1 || T > h->desc.max_rows) return STRATA_EINVAL;
  if (!in->position || !in->seed || !in->temperature || !in->fed || !out->tokens || !out->n_emit)
    return STRATA_EINVAL;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return STRATA_EINVAL;
  if (fault_is("launch")) return STRATA_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  WindowBufs W = h->W;
  W.x = x;
  W.T = T;
  W.q_out = out->logits ? out->logits : h->logits;
  HeadArgs H = h->H;
  H.position = in->position;
  H.seed = reinterpret_cast<const unsigned long long*>(in->seed);
  H.temperature = in->temperature;
  H.fed = in->fed;
  H.tokens = out->tokens;
  H.n_emit = out->n_emit;
  const bool prof = h->profiling;
  cudaError_t e = prof ? cudaEventRecord(h->prof[0], s) : cudaSuccess;
  if (e == cudaSuccess) e = launch_head(h->L, W, h->cfg, H, h->nsm, s);
  if (e == cudaSuccess && prof) e = cudaEventRecord(h->prof[1], s);
  if (e == cudaSuccess) e = cudaEventRecord(h->done, s);
  if (e == cudaSuccess && prof) h->profiled_once = true;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

strata_status strata_head_sync(strata_head* h) {
  if (!h) return STRATA_EINVAL;
  if (cudaEventSynchronize(h->done) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  unsigned err = 0;
  if (cudaMemcpy(&err, h->W.err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  if (err != 0) {
    cudaMemset(h->W.err, 0, sizeof(unsigned));
    cudaMemset(h->W.gbar, 0, sizeof(unsigned long long));
    cudaDeviceSynchronize();
    cudaGetLastError();
    return STRATA_EDEVICE;
  }
  return STRATA_OK;
}

strata_status strata_head_set_profiling(strata_head* h, int32_t enable) {
  if (!h) return STRATA_EINVAL;
  if (enable && !h->prof[0]) {
    for (cudaEvent_t& ev : h->prof) {
      if (cudaEventCreate(&ev) != cudaSuccess) {
        cudaGetLastError();
        return STRATA_ECUDA;
      }
    }
  }
  h->profiling = enable != 0;
  return STRATA_OK;
}

strata_status strata_head_timings(strata_head* h, float* ms) {
  if (!h || !ms || !h->profiled_once) return STRATA_EINVAL;
  if (cudaEventSynchronize(h->prof[1]) != cudaSuccess ||
      cudaEventElapsedTime(ms, h->prof[0], h->prof[1]) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

strata_status strata_head_query(const strata_head* h, int64_t* head_bytes, int64_t* workspace_bytes) {
  if (!h) return STRATA_EINVAL;
  const strata_head_desc& d = h->desc;
  if (head_bytes)
    *head_bytes = (int64_t)d.vocab * ((int64_t)d.hidden * d.bits / 8 + 4LL * (d.hidden / d.block));
  if (workspace_bytes) *workspace_bytes = h->ws_bytes;
  return STRATA_OK;
}

strata_status strata_head_destroy(strata_head* h) {
  free_head(h);
  return STRATA_OK;
}

}  // extern "C"
