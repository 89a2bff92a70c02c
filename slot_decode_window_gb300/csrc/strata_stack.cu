// C ABI of a window through a stack of decoder layers: each layer's MoE part is
// a window handle (same checks, repack and workspace as strata_window_create);
// the stack adds the layers' kernel-ordered dense q/k/v/o weights, a device
// array of per-layer descriptors, and the residual-stream buffers, and runs
// every layer in one cooperative launch of the stack kernel.
#include <new>

#include "common.cuh"
#include "handle.h"
#include "kernels.h"
#include "strata_window.h"

using namespace strata;

struct strata_stack {
  int n_layers = 0;
  strata_moe_desc desc{};
  strata_attn_desc attn{};
  strata_window** layers = nullptr;  // one MoE window handle per layer
  void* dense = nullptr;             // kernel-ordered q/k/v (one matrix) and o of every layer
  LayerDev* dev_layers = nullptr;    // [n_layers] on the device
  float* extra = nullptr;            // v, x1, two ping-pong residual planes
  WindowBufs W{};
  KernelCfg cfg{};
  long long dense_bytes = 0;
  cudaEvent_t done = nullptr;
  bool profiling = false;
  bool profiled_once = false;
  cudaEvent_t prof[2] = {nullptr, nullptr};
  void* kvmem = nullptr;             // the cache attention's scratch (strata_stack_set_kv)
};

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
int log2i(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

strata_status check_attn(const strata_moe_desc* m, const strata_attn_desc* a) {
  if (!m || !a) return STRATA_EINVAL;
  if (a->heads <= 0 || a->kv_heads <= 0 || a->head_dim <= 0 || a->heads % a->kv_heads != 0) return STRATA_EINVAL;
  const int kstep = m->bits == 4 ? 64 : 128;
  if (a->head_dim % kstep != 0 || !pow2(a->head_dim / kstep) || !pow2(a->heads / a->kv_heads))
    return STRATA_EUNSUPPORTED;
  const long long dq = (long long)a->heads * a->head_dim;
  if (dq > 16384 || (long long)a->kv_heads * a->head_dim > m->hidden) return STRATA_EUNSUPPORTED;
  return STRATA_OK;
}

bool qmat_ok(const strata_qmat& q) { return q.codes && q.scale && q.min; }

void free_stack(strata_stack* s) {
  if (!s) return;
  if (s->layers) {
    for (int l = 0; l < s->n_layers; ++l) strata_window_destroy(s->layers[l]);
    delete[] s->layers;
  }
  if (s->dense) cudaFree(s->dense);
  if (s->dev_layers) cudaFree(s->dev_layers);
  if (s->extra) cudaFree(s->extra);
  if (s->kvmem) cudaFree(s->kvmem);
  if (s->done) cudaEventDestroy(s->done);
  for (cudaEvent_t& ev : s->prof)
    if (ev) cudaEventDestroy(ev);
  delete s;
}

}  // namespace

extern "C" {

strata_status strata_stack_create(int32_t n_layers, const strata_moe_desc* moe, const strata_attn_desc* attn,
                                  const strata_moe_weights* moe_w, const strata_attn_weights* attn_w,
                                  void* cuda_stream, strata_stack** out) {
  if (!out) return STRATA_EINVAL;
  *out = nullptr;
  if (n_layers < 1 || n_layers > 1024 || !moe_w || !attn_w) return STRATA_EINVAL;
  strata_status st = check_attn(moe, attn);
  if (st != STRATA_OK) return st;
  for (int l = 0; l < n_layers; ++l) {
    const strata_attn_weights& a = attn_w[l];
    if (!qmat_ok(a.q) || !qmat_ok(a.k) || !qmat_ok(a.v) || !qmat_ok(a.o)) return STRATA_EINVAL;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(cuda_stream);
  strata_stack* s = new (std::nothrow) strata_stack();
  if (!s) return STRATA_ENOMEM;
  s->desc = *moe;
  s->attn = *attn;
  s->layers = new (std::nothrow) strata_window*[n_layers]();
  if (!s->layers) {
    delete s;
    return STRATA_ENOMEM;
  }
  s->n_layers = n_layers;
  for (int l = 0; l < n_layers; ++l) {
    st = strata_window_create(moe, &moe_w[l], cuda_stream, &s->layers[l]);
    if (st != STRATA_OK) {
      free_stack(s);
      return st;
    }
  }
  const strata_window* h0 = s->layers[0];
  const int d = moe->hidden, bits = moe->bits, block = moe->block;
  const int dq = attn->heads * attn->head_dim, dkv = attn->kv_heads * attn->head_dim;

  // ---- dense weights: [Wq; Wk; Wv] as one tile matrix, then Wo, per layer ----
  const long long pq = packed_bytes(1, dq, d, bits), pk = packed_bytes(1, dkv, d, bits);
  const long long po = packed_bytes(1, d, dq, bits);
  const size_t per_layer = align_up((size_t)(pq + 2 * pk), 256) + align_up((size_t)po, 256);
  s->dense_bytes = (long long)(dq + 2LL * dkv) * ((long long)d * bits / 8 + 4LL * (d / block)) +
                   (long long)d * ((long long)dq * bits / 8 + 4LL * (dq / block));
  if (cudaMalloc(&s->dense, per_layer * n_layers) != cudaSuccess) {
    cudaGetLastError();
    free_stack(s);
    return STRATA_ENOMEM;
  }
  LayerDev* host_layers = new (std::nothrow) LayerDev[n_layers];
  if (!host_layers) {
    free_stack(s);
    return STRATA_ENOMEM;
  }
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
    uint8_t* base = static_cast<uint8_t*>(s->dense) + per_layer * l;
    uint8_t* ob = base + align_up((size_t)(pq + 2 * pk), 256);
    const strata_attn_weights& a = attn_w[l];
    auto rp = [&](const strata_qmat& q, int rows, int K, uint8_t* dst) {
      if (e == cudaSuccess)
        e = launch_repack(static_cast<const uint8_t*>(q.codes), q.scale, q.min, 1, rows, K, bits, dst, cs);
    };
    rp(a.q, dq, d, base);
    rp(a.k, dkv, d, base + pq);
    rp(a.v, dkv, d, base + pq + pk);
    rp(a.o, d, dq, ob);
    LayerDev L = s->layers[l]->L;
    L.qkv = packed_desc(base, dq + 2 * dkv, d, bits);
    L.o = packed_desc(ob, d, dq, bits);
    L.dq = dq;
    L.dkv = dkv;
    const int kstep = bits == 4 ? 64 : 128;
    L.kph_log2 = log2i(attn->head_dim / kstep);
    L.kpg_log2 = L.kph_log2 + log2i(attn->heads / attn->kv_heads);
    host_layers[l] = L;
  }
  if (e == cudaSuccess && cudaMalloc(&s->dev_layers, sizeof(LayerDev) * n_layers) != cudaSuccess) e = cudaErrorMemoryAllocation;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(s->dev_layers, host_layers, sizeof(LayerDev) * n_layers, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  const LayerDev L0 = host_layers[0];
  delete[] host_layers;
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_stack(s);
    return e == cudaErrorMemoryAllocation ? STRATA_ENOMEM : STRATA_ECUDA;
  }

  // ---- residual-stream buffers; the rest of the workspace is layer 0's ----
  // v, x1, two ping-pong residual planes, then v's block sums and v's B image
  const size_t n_v = (size_t)kMaxRows * dkv, n_x = (size_t)kMaxRows * d;
  const size_t n_vs = (size_t)kMaxRows * (dkv / 16), n_vi = (size_t)8 * dkv;  // n_vi floats = 16 dkv halves
  if (cudaMalloc(&s->extra, (n_v + 3 * n_x + n_vs + n_vi) * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    free_stack(s);
    return STRATA_ENOMEM;
  }
  s->W = h0->W;
  s->W.v = s->extra;
  s->W.x1 = s->extra + n_v;
  s->W.vsum = s->extra + n_v + 3 * n_x;
  s->W.vimg = reinterpret_cast<__half*>(s->W.vsum + n_vs);

  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h0->device) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->done, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    free_stack(s);
    return STRATA_ECUDA;
  }
  s->cfg = window_cfg(L0, moe->max_rows, optin - 12288, h0->nsm);
  if (s->cfg.nstages < 2) {
    free_stack(s);
    return STRATA_EUNSUPPORTED;
  }
  if (stack_set_attrs(bits, s->cfg.total_bytes) != cudaSuccess) {
    cudaGetLastError();
    free_stack(s);
    return STRATA_ECUDA;
  }
  if (stack_blocks_per_sm(bits, s->cfg.total_bytes) < 1) {
    free_stack(s);
    return STRATA_EUNSUPPORTED;
  }
  *out = s;
  return STRATA_OK;
}

strata_status strata_stack_set_kv(strata_stack* s, const strata_kv_cache* kv) {
  if (!s) return STRATA_EINVAL;
  if (!kv) {
    if (s->kvmem) cudaFree(s->kvmem);
    s->kvmem = nullptr;
    s->W.kv = KVDev{};
    return STRATA_OK;
  }
  const int hd = s->attn.head_dim, H = s->attn.heads, kvh = s->attn.kv_heads, grp = H / kvh;
  if (!kv->k || !kv->v || kv->n_slots < 1 || kv->max_ctx < 1 || kv->max_ctx > (1 << 20)) return STRATA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(kv->k) | reinterpret_cast<uintptr_t>(kv->v)) % 16 != 0) return STRATA_EINVAL;
  // the attention phase takes 32 to 128 head dimensions (whole lanes of a
  // warp) and keeps one chunk of keys and values, the rows' queries and their
  // scores in the shared-memory ring
  const long long need = 2LL * kAttnChunk * hd * 2 + (long long)kMaxRows * grp * hd * 4 +
                         (long long)kMaxRows * grp * kAttnChunk * 4;
  if (hd % 32 != 0 || hd > 128 || need > (long long)s->cfg.nstages * s->cfg.stage_bytes) return STRATA_EUNSUPPORTED;
  const int dq = H * hd, dkv = kvh * hd, block = s->desc.block;
  const int nch = (kv->max_ctx + kAttnChunk - 1) / kAttnChunk;
  size_t w = 0;
  const size_t o_q = w; w = align_up(w + (size_t)kMaxRows * dq * 4, 256);
  const size_t o_k = w; w = align_up(w + (size_t)kMaxRows * dkv * 4, 256);
  const size_t o_p = w; w = align_up(w + (size_t)kMaxRows * H * nch * (hd + 2) * 4, 256);
  const size_t o_a = w; w = align_up(w + (size_t)2 * 8 * dq * 2, 256);
  const size_t o_s = w; w = align_up(w + (size_t)kMaxRows * (dq / block) * 4, 256);
  void* mem = nullptr;
  if (cudaMalloc(&mem, w) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ENOMEM;
  }
  if (cudaMemset(mem, 0, w) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(mem);
    return STRATA_ECUDA;
  }
  if (s->kvmem) cudaFree(s->kvmem);
  s->kvmem = mem;
  uint8_t* b = static_cast<uint8_t*>(mem);
  KVDev& K = s->W.kv;
  K.k = reinterpret_cast<__half*>(kv->k);
  K.v = reinterpret_cast<__half*>(kv->v);
  K.n_slots = kv->n_slots;
  K.max_ctx = kv->max_ctx;
  K.head_dim = hd;
  K.nch = nch;
  K.slot = nullptr;
  K.pos = nullptr;
  K.qbuf = reinterpret_cast<float*>(b + o_q);
  K.kbuf = reinterpret_cast<float*>(b + o_k);
  K.part = reinterpret_cast<float*>(b + o_p);
  K.afrag = reinterpret_cast<__half*>(b + o_a);
  K.afrag_set = 8 * dq;
  K.asum = reinterpret_cast<float*>(b + o_s);
  return STRATA_OK;
}

}  // extern "C"

namespace {

strata_status stack_launch(strata_stack* s, const float* x, int32_t T, float* y, const strata_stack_out* out,
                           const int32_t* slot, const int32_t* position, void* cuda_stream) {
  if (!s || !x || !y) return STRATA_EINVAL;
  if (T < 1 || T > s->desc.max_rows) return STRATA_EINVAL;
  const size_t bytes = (size_t)T * s->desc.hidden * sizeof(float);
  const char* xb = reinterpret_cast<const char*>(x);
  const char* yb = reinterpret_cast<const char*>(y);
  if (xb < yb + bytes && yb < xb + bytes) return STRATA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % 16 != 0) return STRATA_EINVAL;
  cudaStream_t cs = static_cast<cudaStream_t>(cuda_stream);
  WindowBufs W = s->W;
  if (slot) {
    W.kv.slot = slot;
    W.kv.pos = position;
  } else {
    W.kv = KVDev{};  // the length-one reading
  }
  W.x = x;
  W.y = y;
  W.T = T;
  W.out_topk_idx = out ? out->topk_idx : nullptr;
  W.out_topk_w = out ? out->topk_w : nullptr;
  W.out_ndistinct = out ? out->n_distinct : nullptr;
  W.out_counts = W.out_offsets = W.out_entries = W.out_distinct = nullptr;
  float* ybuf = s->W.x1 + (size_t)kMaxRows * s->desc.hidden;
  const strata_window* h0 = s->layers[0];
  cudaError_t e = s->profiling ? cudaEventRecord(s->prof[0], cs) : cudaSuccess;
  if (e == cudaSuccess)
    e = launch_stack(s->dev_layers, s->n_layers, s->desc.bits, W, s->cfg, h0->nsm, x, y, ybuf, out ? out->q : nullptr,
                     out ? out->k : nullptr, cs);
  if (e == cudaSuccess && s->profiling) e = cudaEventRecord(s->prof[1], cs);
  if (e == cudaSuccess) e = cudaEventRecord(s->done, cs);
  if (e == cudaSuccess && s->profiling) s->profiled_once = true;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

}  // namespace

extern "C" {

strata_status strata_stack_forward(strata_stack* s, const float* x, int32_t T, float* y, const strata_stack_out* out,
                                   void* cuda_stream) {
  return stack_launch(s, x, T, y, out, nullptr, nullptr, cuda_stream);
}

strata_status strata_stack_forward_kv(strata_stack* s, const float* x, int32_t T, float* y, const int32_t* slot,
                                      const int32_t* position, const strata_stack_out* out, void* cuda_stream) {
  if (!s || !slot || !position || !s->W.kv.k) return STRATA_EINVAL;
  return stack_launch(s, x, T, y, out, slot, position, cuda_stream);
}

strata_status strata_stack_sync(strata_stack* s) {
  if (!s) return STRATA_EINVAL;
  if (cudaEventSynchronize(s->done) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  unsigned err = 0;
  if (cudaMemcpy(&err, s->W.err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  if (err != 0) {
    // as strata_window_sync: the failed window's grid-barrier count restarts at zero
    cudaMemset(s->W.err, 0, sizeof(unsigned));
    cudaMemset(s->W.gbar, 0, sizeof(unsigned long long));
    cudaDeviceSynchronize();
    cudaGetLastError();
    return STRATA_EDEVICE;
  }
  return STRATA_OK;
}

strata_status strata_stack_query(const strata_stack* s, strata_stack_info* info) {
  if (!s || !info) return STRATA_EINVAL;
  strata_window_info wi{};
  strata_status st = strata_window_query(s->layers[0], &wi);
  if (st != STRATA_OK) return st;
  info->n_layers = s->n_layers;
  info->n_sm = wi.n_sm;
  info->stages = s->cfg.nstages;
  info->stage_bytes = s->cfg.stage_bytes;
  info->smem_bytes = s->cfg.total_bytes;
  info->dense_bytes = s->dense_bytes;
  info->expert_bytes = wi.expert_bytes;
  info->shared_bytes = wi.shared_bytes;
  info->router_bytes = wi.router_bytes;
  return STRATA_OK;
}

strata_status strata_stack_set_profiling(strata_stack* s, int32_t enable) {
  if (!s) return STRATA_EINVAL;
  if (enable && !s->prof[0]) {
    if (cudaEventCreate(&s->prof[0]) != cudaSuccess || cudaEventCreate(&s->prof[1]) != cudaSuccess) {
      cudaGetLastError();
      return STRATA_ECUDA;
    }
  }
  s->profiling = enable != 0;
  return STRATA_OK;
}

strata_status strata_stack_timings(strata_stack* s, float* ms) {
  if (!s || !ms || !s->profiled_once) return STRATA_EINVAL;
  if (cudaEventSynchronize(s->prof[1]) != cudaSuccess || cudaEventElapsedTime(ms, s->prof[0], s->prof[1]) != cudaSuccess) {
    cudaGetLastError();
    return STRATA_ECUDA;
  }
  return STRATA_OK;
}

strata_status strata_stack_destroy(strata_stack* s) {
  if (!s) return STRATA_OK;
  free_stack(s);
  return STRATA_OK;
}

}  // extern "C"
