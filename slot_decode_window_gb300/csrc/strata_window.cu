// C ABI of the verify-window MoE step: argument checks, the handle's memory
// (kernel-ordered weights + window workspace), and the per-window launch of
// the persistent window kernel (one cooperative launch, one CTA per SM).
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "common.cuh"
#include "handle.h"
#include "kernels.h"
#include "strata_window.h"

using namespace strata;

bool strata::fault_is(const char* what) {
  const char* f = std::getenv("STRATA_FAULT");
  return f && std::strcmp(f, what) == 0;
}

long long strata::env_int(const char* name, long long dflt, long long lo, long long hi) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  const long long n = std::strtoll(v, &end, 10);
  if (*end != '\0' || n < lo || n > hi) return dflt;
  return n;
}

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int kstep_of(int bits) { return bits == 4 ? 64 : 128; }

strata_status check_desc(const strata_moe_desc* d) {
  if (!d) return STRATA_EINVAL;
  if (d->hidden <= 0 || d->n_experts <= 0 || d->top_k <= 0 || d->ffn <= 0 || d->shared_ffn < 0 || d->max_rows <= 0)
    return STRATA_EINVAL;
  if (d->top_k > d->n_experts) return STRATA_EINVAL;
  if (d->renorm_topk != 0 && d->renorm_topk != 1) return STRATA_EINVAL;
  if (d->max_rows > kMaxRows) return STRATA_EINVAL;
  if (!((d->bits == 4 && d->block == 32) || (d->bits == 2 && d->block == 16))) return STRATA_EUNSUPPORTED;
  if (d->n_experts > kMaxExperts || d->top_k > kMaxTopK) return STRATA_EUNSUPPORTED;
  const int ks = kstep_of(d->bits);
  if (d->hidden % ks != 0 || d->ffn % ks != 0 || (d->shared_ffn > 0 && d->shared_ffn % ks != 0))
    return STRATA_EUNSUPPORTED;
  if (d->hidden > 16384 || d->ffn > 16384 || d->shared_ffn > 16384) return STRATA_EUNSUPPORTED;
  return STRATA_OK;
}

bool qmat_ok(const strata_qmat& q) { return q.codes && q.scale && q.min; }

strata_status check_weights(const strata_moe_desc* d, const strata_moe_weights* w) {
  if (!w) return STRATA_EINVAL;
  if (!w->router_w || !qmat_ok(w->gate) || !qmat_ok(w->up) || !qmat_ok(w->down)) return STRATA_EINVAL;
  if (d->shared_ffn > 0 && (!qmat_ok(w->shared_gate) || !qmat_ok(w->shared_up) || !qmat_ok(w->shared_down)))
    return STRATA_EINVAL;
  return STRATA_OK;
}

long long qmat_bytes(int n, int rows, int cols, int bits, int block) {
  return (long long)n * rows * ((long long)cols * bits / 8 + 4LL * (cols / block));
}

void free_handle(strata_window* h) {
  if (!h) return;
  for (strata_graph_entry& g : h->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
  if (h->done) cudaEventDestroy(h->done);
  for (cudaEvent_t& ev : h->prof)
    if (ev) cudaEventDestroy(ev);
  if (h->wmem) cudaFree(h->wmem);
  if (h->ws) cudaFree(h->ws);
  delete h;
}

}  // namespace

extern "C" {

const char* strata_status_str(strata_status s) {
  switch (s) {
    case STRATA_OK: return "ok";
    case STRATA_EINVAL: return "invalid argument";
    case STRATA_ENOMEM: return "out of device memory";
    case STRATA_ECUDA: return "CUDA runtime error";
    case STRATA_EUNSUPPORTED: return "unsupported shape or format";
    case STRATA_EDEVICE: return "error flagged on the device";
  }
  return "unknown status";
}

// Dynamic shared memory left out of the window kernel's budget for its static
// shared memory, and the opt-in maximum of a GB300 (227 KB) that
// strata_window_plan assumes when given no limit.
constexpr int kStaticSmemReserve = 12288;
constexpr int kGb300SmemOptin = 232448;

strata_status strata_window_slots(int32_t n_slots, const int32_t* rows_per_slot, int32_t start, int32_t max_rows,
                                  int32_t* slots_out, int32_t* n_out, int32_t* next_start) {
  if (n_slots < 1 || !rows_per_slot || !slots_out || !n_out || !next_start) return STRATA_EINVAL;
  if (start < 0 || start >= n_slots || max_rows < 1 || max_rows > kMaxRows) return STRATA_EINVAL;
  for (int s = 0; s < n_slots; ++s)
    if (rows_per_slot[s] < 0 || rows_per_slot[s] > max_rows) return STRATA_EINVAL;
  int n = 0, used = 0, last = start - 1;
  for (int i = 0; i < n_slots; ++i) {
    const int s = (start + i) % n_slots;
    const int r = rows_per_slot[s];
    if (r == 0) continue;
    if (used + r > max_rows) break;
    slots_out[n++] = s;
    used += r;
    last = s;
  }
  *n_out = n;
  *next_start = ((last + 1) % n_slots + n_slots) % n_slots;
  return STRATA_OK;
}

strata_status strata_window_plan(const strata_moe_desc* desc, int32_t smem_limit, strata_window_info* info) {
  if (!info) return STRATA_EINVAL;
  std::memset(info, 0, sizeof(*info));
  const strata_status st = check_desc(desc);
  if (st != STRATA_OK) return st;
  if (smem_limit < 0) return STRATA_EINVAL;
  const int limit = smem_limit > 0 ? smem_limit : kGb300SmemOptin - kStaticSmemReserve;
  LayerDev L{};
  L.d = desc->hidden;
  L.E = desc->n_experts;
  L.k = desc->top_k;
  L.F = desc->ffn;
  L.Fs = desc->shared_ffn;
  L.bits = desc->bits;
  L.renorm = desc->renorm_topk;
  const KernelCfg C = window_cfg_direct(L, desc->max_rows, limit);
  if (!C.direct && C.nstages < 2) return STRATA_EUNSUPPORTED;
  info->stages = C.nstages;
  info->stage_bytes = C.stage_bytes;
  info->smem_bytes = C.total_bytes;
  return STRATA_OK;
}

strata_status strata_window_create(const strata_moe_desc* desc, const strata_moe_weights* weights, void* cuda_stream,
                                   strata_window** out) {
  if (!out) return STRATA_EINVAL;
  *out = nullptr;
  strata_status st = check_desc(desc);
  if (st != STRATA_OK) return st;
  st = check_weights(desc, weights);
  if (st != STRATA_OK) return st;
  if (fault_is("alloc")) return STRATA_ENOMEM;

  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  strata_window* h = new (std::nothrow) strata_window();
  if (!h) return STRATA_ENOMEM;
  h->desc = *desc;
  const int d = desc->hidden, E = desc->n_experts, k = desc->top_k, F = desc->ffn, Fs = desc->shared_ffn;
  const int bits = desc->bits, block = desc->block;

  int optin = 0;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->nsm, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return STRATA_ECUDA;
  }

  // ---- kernel-ordered weights + router copy ----
  const long long pg = packed_bytes(E, F, d, bits), pu = pg, pd = packed_bytes(E, d, F, bits);
  const long long psg = Fs > 0 ? packed_bytes(1, Fs, d, bits) : 0, psu = psg;
  const long long psd = Fs > 0 ? packed_bytes(1, d, Fs, bits) : 0;
  size_t off = 0;
  const size_t o_gate = off; off = align_up(off + pg, 256);
  const size_t o_up = off; off = align_up(off + pu, 256);
  const size_t o_down = off; off = align_up(off + pd, 256);
  const size_t o_sg = off; off = align_up(off + psg, 256);
  const size_t o_su = off; off = align_up(off + psu, 256);
  const size_t o_sd = off; off = align_up(off + psd, 256);
  const size_t o_rw = off; off = align_up(off + (size_t)E * d * 4, 256);
  const size_t o_rb = off; off = align_up(off + (size_t)E * 4, 256);
  h->packed = (long long)off;
  if (cudaMalloc(&h->wmem, off) != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return STRATA_ENOMEM;
  }
  uint8_t* wb = static_cast<uint8_t*>(h->wmem);

  // ---- workspace ----
  const int nmk_d = (d / block + 15) / 16;
  size_t w = 0;
  const int njb = (d + kRouterCols - 1) / kRouterCols;
  const size_t o_err = w; w = align_up(w + 8, 256);
  const size_t o_gbar = w; w = align_up(w + 8, 256);
  const size_t o_cnt = w; w = align_up(w + (size_t)(d / 16) * 4, 256);
  const size_t o_done = w; w = align_up(w + (size_t)(E + 1) * 4, 256);
  const size_t o_part = w; w = align_up(w + (size_t)njb * kMaxRows * E * 4, 256);
  const size_t o_xf = w; w = align_up(w + (size_t)kMaxRows * frag_halves(d, nmk_d) * 2, 256);
  const size_t o_hf = w; w = align_up(w + (size_t)kMaxEntries * 2 * F * 2, 256);
  const size_t o_hs = w; w = align_up(w + (size_t)kMaxEntries * (F / 16) * 4, 256);
  const size_t o_shf = w; w = align_up(w + (size_t)kMaxRows * 2 * Fs * 2, 256);
  const size_t o_shs = w; w = align_up(w + (size_t)kMaxRows * (Fs / 16) * 4, 256);
  const size_t o_ob = w; w = align_up(w + (size_t)kMaxEntries * d * 4, 256);
  const size_t o_sb = w; w = align_up(w + (size_t)kMaxRows * d * 4, 256);
  h->ws_bytes = (long long)w;
  if (cudaMalloc(&h->ws, w) != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return STRATA_ENOMEM;
  }
  uint8_t* wsb = static_cast<uint8_t*>(h->ws);

  // ---- fill ----
  cudaError_t e = cudaMemsetAsync(h->ws, 0, w, s);
  auto rp = [&](const strata_qmat& q, int n, int rows, int K, size_t o) {
    if (e == cudaSuccess)
      e = launch_repack(static_cast<const uint8_t*>(q.codes), q.scale, q.min, n, rows, K, bits, wb + o, s);
  };
  rp(weights->gate, E, F, d, o_gate);
  rp(weights->up, E, F, d, o_up);
  rp(weights->down, E, d, F, o_down);
  if (Fs > 0) {
    rp(weights->shared_gate, 1, Fs, d, o_sg);
    rp(weights->shared_up, 1, Fs, d, o_su);
    rp(weights->shared_down, 1, d, Fs, o_sd);
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(wb + o_rw, weights->router_w, (size_t)E * d * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && weights->router_b)
    e = cudaMemcpyAsync(wb + o_rb, weights->router_b, (size_t)E * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->done, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return STRATA_ECUDA;
  }

  LayerDev& L = h->L;
  L.d = d; L.E = E; L.k = k; L.F = F; L.Fs = Fs; L.bits = bits; L.renorm = desc->renorm_topk;
  L.router_w = reinterpret_cast<const float*>(wb + o_rw);
  L.router_b = weights->router_b ? reinterpret_cast<const float*>(wb + o_rb) : nullptr;
  L.gate = packed_desc(wb + o_gate, F, d, bits);
  L.up = packed_desc(wb + o_up, F, d, bits);
  L.down = packed_desc(wb + o_down, d, F, bits);
  if (Fs > 0) {
    L.sgate = packed_desc(wb + o_sg, Fs, d, bits);
    L.sup = packed_desc(wb + o_su, Fs, d, bits);
    L.sdown = packed_desc(wb + o_sd, d, Fs, bits);
  } else {
    L.sgate = L.sup = L.sdown = PackedMat{};
  }

  WindowBufs& W = h->W;
  W.err = reinterpret_cast<unsigned*>(wsb + o_err);
  W.gbar = reinterpret_cast<unsigned long long*>(wsb + o_gbar);
  W.counters = reinterpret_cast<int*>(wsb + o_cnt);
  W.done_gu = reinterpret_cast<int*>(wsb + o_done);
  h->partial = reinterpret_cast<float*>(wsb + o_part);
  W.partial = h->partial;
  W.njb = njb;
  // bounded device waits: 2^31 cycles (about a second) unless a diagnostic
  // override asks for a shorter limit; no extra grid-barrier arrivals unless a
  // failure test asks for some
  W.wait_cycles = env_int("STRATA_WAIT_CYCLES", 1LL << 31, 1000, 1LL << 40);
  W.bar_extra = (int)env_int("STRATA_TEST_BARRIER_EXTRA", 0, 0, 1 << 20);
  W.xfrag = reinterpret_cast<__half*>(wsb + o_xf);
  W.hfrag = reinterpret_cast<__half*>(wsb + o_hf);
  W.hsum = reinterpret_cast<float*>(wsb + o_hs);
  W.shfrag = reinterpret_cast<__half*>(wsb + o_shf);
  W.shsum = reinterpret_cast<float*>(wsb + o_shs);
  W.obuf = reinterpret_cast<float*>(wsb + o_ob);
  W.sbuf = reinterpret_cast<float*>(wsb + o_sb);

  const int limit = optin - kStaticSmemReserve;
  h->cfg = window_cfg_direct(L, desc->max_rows, limit);
  if (!h->cfg.direct && h->cfg.nstages < 2) {
    free_handle(h);
    return STRATA_EUNSUPPORTED;
  }
  if (window_set_attrs(bits, h->cfg.direct, h->cfg.total_bytes) != cudaSuccess) {
    cudaGetLastError();
    free_handle(h);
    return STRATA_ECUDA;
  }
  // the window kernel's CTAs wait on one another: all of them must be resident
  if (window_blocks_per_sm(bits, h->cfg.direct, h->cfg.total_bytes) < 1) {
    free_handle(h);
    return STRATA_EUNSUPPORTED;
  }
  *out = h;
  return STRATA_OK;
}

strata_status strata_moe_window_forward(strata_window* h, const float* x, int32_t T, float* y,
                                        const strata_routing_out* routing, void* cuda_stream) {
  if (!h || !x || !y) return STRATA_EINVAL;
  if (T < 1 || T > h->desc.max_rows) return STRATA_EINVAL;
  const size_t bytes = (size_t)T * h->desc.hidden * sizeof(float);
  const char* xb = reinterpret_cast<const char*>(x);
  const char* yb = reinterpret_cast<const char*>(y);
  if (xb < yb + bytes && yb < xb + bytes) return STRATA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % 16 != 0) return STRATA_EINVAL;
  if (fault_is("launch")) return STRATA_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  WindowBufs W = h->W;
  W.x = x;
  W.y = y;
  W.T = T;
  W.out_topk_idx = routing ? routing->topk_idx : nullptr;
  W.out_topk_w = routing ? routing->topk_w : nullptr;
  W.out_counts = routing ? routing->counts : nullptr;
  W.out_offsets = routing ? routing->offsets : nullptr;
  W.out_entries = routing ? routing->entries : nullptr;
  W.out_distinct = routing ? routing->distinct : nullptr;
  W.out_ndistinct = routing ? routing->n_distinct : nullptr;

  const bool prof = h->profiling;
  cudaError_t e = prof ? cudaEventRecord(h->prof[0], s) : cudaSuccess;
  if (e == cudaSuccess) e = launch_window(h->L, W, h->cfg, h->nsm, s);
  if (e == cudaSuccess && prof) e = cudaEventRecord(h->prof[1], s);
  if (e == cudaSuccess) e = cudaEventRecord(h->done, s);
  if (e == cudaSuccess && prof) h->profiled_once = true;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

strata_status strata_moe_window_forward_graph(strata_window* h, const float* x, int32_t T, float* y,
                                              void* cuda_stream) {
  if (!h || !x || !y) return STRATA_EINVAL;
  if (T < 1 || T > h->desc.max_rows) return STRATA_EINVAL;
  const size_t bytes = (size_t)T * h->desc.hidden * sizeof(float);
  const char* xb = reinterpret_cast<const char*>(x);
  const char* yb = reinterpret_cast<const char*>(y);
  if (xb < yb + bytes && yb < xb + bytes) return STRATA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % 16 != 0) return STRATA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  strata_graph_entry* hit = nullptr;
  strata_graph_entry* victim = &h->graphs[0];
  for (strata_graph_entry& g : h->graphs) {
    if (g.exec && g.T == T && g.x == x && g.y == y) {
      hit = &g;
      break;
    }
    if (!g.exec || (victim->exec && g.last_use < victim->last_use)) victim = &g;
  }
  if (!hit) {
    // capture the window launch on the handle's own stream and instantiate it
    if (!h->capture_stream && cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      return STRATA_ECUDA;
    }
    WindowBufs W = h->W;
    W.x = x;
    W.y = y;
    W.T = T;
    W.out_topk_idx = nullptr;
    W.out_topk_w = nullptr;
    W.out_counts = nullptr;
    W.out_offsets = nullptr;
    W.out_entries = nullptr;
    W.out_distinct = nullptr;
    W.out_ndistinct = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaError_t e = cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      const cudaError_t el = launch_window(h->L, W, h->cfg, h->nsm, h->capture_stream);
      e = cudaStreamEndCapture(h->capture_stream, &graph);
      if (el != cudaSuccess) e = el;
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return STRATA_ECUDA;
    }
    if (victim->exec) cudaGraphExecDestroy(victim->exec);
    victim->T = T;
    victim->x = x;
    victim->y = y;
    victim->exec = exec;
    hit = victim;
  }
  hit->last_use = ++h->graph_clock;
  cudaError_t e = cudaGraphLaunch(hit->exec, s);
  if (e == cudaSuccess) e = cudaEventRecord(h->done, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

strata_status strata_window_sync(strata_window* h) {
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
    // the window that failed may have left its grid-barrier count off a
    // multiple of the grid (CTAs that gave up before others arrived): start
    // the next window from zero
    cudaMemset(h->W.err, 0, sizeof(unsigned));
    cudaMemset(h->W.gbar, 0, sizeof(unsigned long long));
    cudaDeviceSynchronize();
    cudaGetLastError();
    return STRATA_EDEVICE;
  }
  return STRATA_OK;
}

strata_status strata_window_query(const strata_window* h, strata_window_info* info) {
  if (!h || !info) return STRATA_EINVAL;
  const strata_moe_desc& d = h->desc;
  info->n_sm = h->nsm;
  info->stages = h->cfg.nstages;
  info->stage_bytes = h->cfg.stage_bytes;
  info->smem_bytes = h->cfg.total_bytes;
  info->packed_bytes = h->packed;
  info->expert_bytes = qmat_bytes(2, d.ffn, d.hidden, d.bits, d.block) + qmat_bytes(1, d.hidden, d.ffn, d.bits, d.block);
  info->shared_bytes = d.shared_ffn > 0 ? qmat_bytes(2, d.shared_ffn, d.hidden, d.bits, d.block) +
                                              qmat_bytes(1, d.hidden, d.shared_ffn, d.bits, d.block)
                                        : 0;
  info->router_bytes = (long long)d.n_experts * d.hidden * 4 + (h->L.router_b ? d.n_experts * 4 : 0);
  info->workspace_bytes = h->ws_bytes;
  return STRATA_OK;
}

strata_status strata_window_set_profiling(strata_window* h, int32_t enable) {
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

strata_status strata_window_timings(strata_window* h, float* ms) {
  if (!h || !ms || !h->profiled_once) return STRATA_EINVAL;
  if (cudaEventSynchronize(h->prof[1]) != cudaSuccess ||
      cudaEventElapsedTime(ms, h->prof[0], h->prof[1]) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

strata_status strata_window_destroy(strata_window* h) {
  if (!h) return STRATA_OK;
  free_handle(h);
  return STRATA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// the window entry point that allocates nothing: one static scratch array
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) uint8_t g_window_scratch[STRATA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `dev` (the current device); looked
// up once per device.
void* scratch_on(int dev) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_window_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" strata_status strata_moe_window_forward_noalloc(strata_window* h, const float* x, int32_t T, float* y,
                                                           void* cuda_stream) {
  if (!h || !x || !y) return STRATA_EINVAL;
  if (T < 1 || T > h->desc.max_rows) return STRATA_EINVAL;
  const size_t bytes = (size_t)T * h->desc.hidden * sizeof(float);
  const char* xb = reinterpret_cast<const char*>(x);
  const char* yb = reinterpret_cast<const char*>(y);
  if (xb < yb + bytes && yb < xb + bytes) return STRATA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % 16 != 0) return STRATA_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  if (dev != h->device || dev < 0 || dev >= kMaxDevices) return STRATA_EINVAL;

  // Scratch layout: the zero-start parts first, so one memset clears them.
  const int d = h->desc.hidden, E = h->desc.n_experts, F = h->desc.ffn, Fs = h->desc.shared_ffn;
  const int nmk_d = (d / h->desc.block + 15) / 16;
  size_t w = 0;
  const size_t o_gbar = w; w = align_up(w + 8, 256);
  const size_t o_xf = w; w = align_up(w + (size_t)kMaxRows * frag_halves(d, nmk_d) * 2, 256);
  const size_t zero_end = w;
  const size_t o_cnt = w; w = align_up(w + (size_t)(d / 16) * 4, 256);
  const size_t o_done = w; w = align_up(w + (size_t)(E + 1) * 4, 256);
  const size_t o_part = w; w = align_up(w + (size_t)h->W.njb * kMaxRows * E * 4, 256);
  const size_t o_hf = w; w = align_up(w + (size_t)kMaxEntries * 2 * F * 2, 256);
  const size_t o_hs = w; w = align_up(w + (size_t)kMaxEntries * (F / 16) * 4, 256);
  const size_t o_shf = w; w = align_up(w + (size_t)kMaxRows * 2 * Fs * 2, 256);
  const size_t o_shs = w; w = align_up(w + (size_t)kMaxRows * (Fs / 16) * 4, 256);
  const size_t o_ob = w; w = align_up(w + (size_t)kMaxEntries * d * 4, 256);
  const size_t o_sb = w; w = align_up(w + (size_t)kMaxRows * d * 4, 256);
  if (w > (size_t)STRATA_NOALLOC_SCRATCH_BYTES) return STRATA_EUNSUPPORTED;

  uint8_t* base = static_cast<uint8_t*>(scratch_on(dev));
  if (!base) return STRATA_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  WindowBufs W = h->W;  // error word and router chunking stay the handle's
  W.gbar = reinterpret_cast<unsigned long long*>(base + o_gbar);
  W.xfrag = reinterpret_cast<__half*>(base + o_xf);
  W.counters = reinterpret_cast<int*>(base + o_cnt);
  W.done_gu = reinterpret_cast<int*>(base + o_done);
  W.partial = reinterpret_cast<float*>(base + o_part);
  W.hfrag = reinterpret_cast<__half*>(base + o_hf);
  W.hsum = reinterpret_cast<float*>(base + o_hs);
  W.shfrag = reinterpret_cast<__half*>(base + o_shf);
  W.shsum = reinterpret_cast<float*>(base + o_shs);
  W.obuf = reinterpret_cast<float*>(base + o_ob);
  W.sbuf = reinterpret_cast<float*>(base + o_sb);
  W.x = x;
  W.y = y;
  W.T = T;
  W.out_topk_idx = nullptr;
  W.out_topk_w = nullptr;
  W.out_counts = nullptr;
  W.out_offsets = nullptr;
  W.out_entries = nullptr;
  W.out_distinct = nullptr;
  W.out_ndistinct = nullptr;

  cudaError_t e = cudaMemsetAsync(base, 0, zero_end, s);
  if (e == cudaSuccess) e = launch_window(h->L, W, h->cfg, h->nsm, s);
  if (e == cudaSuccess) e = cudaEventRecord(h->done, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}
