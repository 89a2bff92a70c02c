// C ABI of the adaptive expert tier's bookkeeping: a tier object holds fp32
// routing counters, the set of experts in the fast tier and the last round's
// swaps on the device; the window kernel of a handle it is attached to adds
// each window's counts and runs the rounds (tier_count, tier_round_due in
// window.cu).
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "handle.h"
#include "kernels.h"
#include "strata_window.h"

using namespace strata;

struct strata_tier {
  strata_tier_desc desc;
  void* mem = nullptr;
  TierDev dev{};
};

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

strata_status check_tier_desc(const strata_tier_desc* d) {
  if (!d) return STRATA_EINVAL;
  if (d->n_experts < 1 || d->n_experts > kMaxExperts) return STRATA_EINVAL;
  if (d->capacity < 1 || d->capacity > d->n_experts) return STRATA_EINVAL;
  if (d->adapt_every < 1 || d->adapt_swaps < 0 || d->adapt_swaps > d->n_experts) return STRATA_EINVAL;
  if (!(d->decay > 0.f && d->decay <= 1.f)) return STRATA_EINVAL;
  if (!(d->min_gain >= 1.f && d->min_gain < 3.0e38f)) return STRATA_EINVAL;
  return STRATA_OK;
}

}  // namespace

extern "C" {

strata_status strata_tier_create(const strata_tier_desc* desc, const int32_t* initial, strata_tier** out) {
  if (!out) return STRATA_EINVAL;
  *out = nullptr;
  const strata_status st = check_tier_desc(desc);
  if (st != STRATA_OK) return st;
  const int E = desc->n_experts, cap = desc->capacity;
  std::vector<int> res(E, 0);
  for (int i = 0; i < cap; ++i) {
    const int e = initial ? initial[i] : i;
    if (e < 0 || e >= E || res[e]) return STRATA_EINVAL;  // out of range or listed twice
    res[e] = 1;
  }
  strata_tier* t = new (std::nothrow) strata_tier();
  if (!t) return STRATA_ENOMEM;
  t->desc = *desc;
  size_t w = 0;
  const size_t o_c = w; w = align_up(w + (size_t)E * 4, 256);
  const size_t o_r = w; w = align_up(w + (size_t)E * 4, 256);
  const size_t o_w = w; w = align_up(w + 8, 256);
  const size_t o_rd = w; w = align_up(w + 8, 256);
  const size_t o_n = w; w = align_up(w + 4, 256);
  const size_t o_in = w; w = align_up(w + (size_t)E * 4, 256);
  const size_t o_out = w; w = align_up(w + (size_t)E * 4, 256);
  if (cudaMalloc(&t->mem, w) != cudaSuccess) {
    cudaGetLastError();
    delete t;
    return STRATA_ENOMEM;
  }
  uint8_t* b = static_cast<uint8_t*>(t->mem);
  if (cudaMemset(t->mem, 0, w) != cudaSuccess ||
      cudaMemcpy(b + o_r, res.data(), (size_t)E * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(t->mem);
    delete t;
    return STRATA_ECUDA;
  }
  TierDev& d = t->dev;
  d.counters = reinterpret_cast<float*>(b + o_c);
  d.resident = reinterpret_cast<int*>(b + o_r);
  d.windows = reinterpret_cast<long long*>(b + o_w);
  d.rounds = reinterpret_cast<long long*>(b + o_rd);
  d.n_swaps = reinterpret_cast<int*>(b + o_n);
  d.swap_in = reinterpret_cast<int*>(b + o_in);
  d.swap_out = reinterpret_cast<int*>(b + o_out);
  d.adapt_every = desc->adapt_every;
  d.adapt_swaps = desc->adapt_swaps;
  d.decay = desc->decay;
  d.min_gain = desc->min_gain;
  *out = t;
  return STRATA_OK;
}

strata_status strata_window_set_tier(strata_window* h, strata_tier* t) {
  if (!h) return STRATA_EINVAL;
  if (t && t->desc.n_experts != h->desc.n_experts) return STRATA_EINVAL;
  // a due round keeps four expert arrays in the ring region beside stage R's
  // staged rows of x (8 rows x 512 floats)
  if (t && (long long)h->cfg.nstages * h->cfg.stage_bytes < 8 * 512 * 4 + 4 * kMaxExperts * 4)
    return STRATA_EUNSUPPORTED;
  // cached graphs hold the window's arguments by value: drop them
  for (strata_graph_entry& g : h->graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    g = strata_graph_entry{};
  }
  h->W.tier = t ? t->dev : TierDev{};
  return STRATA_OK;
}

strata_status strata_tier_read(strata_tier* t, float* counters, int32_t* resident, int32_t* swap_in,
                               int32_t* swap_out, strata_tier_stats* stats) {
  if (!t) return STRATA_EINVAL;
  const size_t E = (size_t)t->desc.n_experts;
  // a round that is due after the last window has not run yet (the next
  // window would run it before adding its own counts): run it now
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = launch_tier_round(t->dev, (int)E, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess && counters) e = cudaMemcpy(counters, t->dev.counters, E * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && resident) e = cudaMemcpy(resident, t->dev.resident, E * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && swap_in) e = cudaMemcpy(swap_in, t->dev.swap_in, E * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && swap_out) e = cudaMemcpy(swap_out, t->dev.swap_out, E * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && stats) {
    long long w = 0, r = 0;
    int n = 0;
    e = cudaMemcpy(&w, t->dev.windows, 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&r, t->dev.rounds, 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&n, t->dev.n_swaps, 4, cudaMemcpyDeviceToHost);
    stats->windows = w;
    stats->rounds = r;
    stats->n_swaps = n;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

strata_status strata_tier_destroy(strata_tier* t) {
  if (!t) return STRATA_OK;
  if (t->mem) cudaFree(t->mem);
  delete t;
  return STRATA_OK;
}

}  // extern "C"
