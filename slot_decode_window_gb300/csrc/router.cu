// Router + window preparation kernel.
//
// Each window's rows are routed (the Strata docs, "BATCHING.md", section
// "Several requests at once (batch slots)": every routed expert two
// conversations share is read once per window; the same page's adaptive-tier
// paragraph: batch windows count which experts they route to).  The pages
// give no router formula; this kernel computes the plain reading: fp32
// logits = Wr x + b, fp32 max-subtracted softmax over all experts, top-k by
// logit (descending, ties to the lower expert), gate weight = the selected
// expert's softmax probability (optionally renormalised over the k).
//
// Work split: CTA (eb, jb) computes partial logits of experts [8eb, 8eb+8)
// over columns [256jb, 256jb+256) with one warp per expert, x's column chunk
// staged in shared memory.  Every CTA also converts part of x into the
// activation fragment layout the expert kernels read.  The CTA that arrives
// last (one atomic ticket, no spinning) sums the partials in a fixed order,
// runs softmax/top-k per row, and groups the window's entries t*k+j by
// expert with a counting sort (bit-exact, no atomics).
#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace strata {

constexpr int kRouterCols = 256;
constexpr int kRouterExpertsPerCta = 8;

template <int BITS>
__device__ void write_x_frags(const LayerDev& L, const WindowBufs& W) {
  const int d = L.d;
  const int nblk = d / Fmt<BITS>::kBlock;
  const int nmk = (nblk + 15) / 16;
  const long long fh = frag_halves(d, nmk);
  const long long n_el = (long long)W.T * d;
  const long long n_sum = (long long)W.T * nmk * 16;
  const long long stride = (long long)gridDim.x * gridDim.y * blockDim.x;
  const long long tid = ((long long)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  for (long long i = tid; i < n_el; i += stride) {
    const int t = (int)(i / d), j = (int)(i % d);
    const float v = W.x[i];
    int off;
    float f;
    frag_main_pos<BITS>(j, off, f);
    __half hi, lo;
    split_hi_lo(v * f, hi, lo);
    __half* base = W.xfrag + t * fh;
    base[off] = hi;
    base[d + off] = lo;
  }
  for (long long i = tid; i < n_sum; i += stride) {
    const int t = (int)(i / (nmk * 16)), beta = (int)(i % (nmk * 16));
    float s = 0.f;
    if (beta < nblk) {
      const float* xr = W.x + (long long)t * d + beta * Fmt<BITS>::kBlock;
      for (int e = 0; e < Fmt<BITS>::kBlock; ++e) s += xr[e];
    }
    __half hi, lo;
    split_hi_lo(s, hi, lo);
    __half* base = W.xfrag + t * fh + 2 * d;
    const int off = frag_sum_pos(beta);
    base[off] = hi;
    base[nmk * 16 + off] = lo;
  }
}

__global__ void __launch_bounds__(kRouterThreads) router_kernel(LayerDev L, WindowBufs W, float* partial) {
  __shared__ __align__(16) float xs[kMaxRows][kRouterCols];
  __shared__ float lg[kMaxRows][kMaxExperts];
  __shared__ int sel[kMaxEntries];
  __shared__ int cnt[kMaxExperts];
  __shared__ int flag[kMaxExperts];
  __shared__ int is_last;

  // The expert kernel may start its prologue now; it waits for this grid's
  // completion before reading anything written here.
  griddep_launch_dependents();

  const int T = W.T, d = L.d, E = L.E, k = L.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int jb = blockIdx.y;
  const int j0 = jb * kRouterCols;
  const int ncol = min(kRouterCols, d - j0);

  // -- partial logits ------------------------------------------------------
  for (int i = tid; i < T * kRouterCols; i += blockDim.x) {
    const int t = i / kRouterCols, j = i % kRouterCols;
    xs[t][j] = (j < ncol) ? W.x[(long long)t * d + j0 + j] : 0.f;
  }
  __syncthreads();
  {
    const int e = blockIdx.x * kRouterExpertsPerCta + warp;
    if (e < E) {
      float acc[kMaxRows];
#pragma unroll
      for (int t = 0; t < kMaxRows; ++t) acc[t] = 0.f;
      const float* wr = L.router_w + (long long)e * d + j0;
      for (int j = lane * 4; j < ncol; j += 128) {
        const float4 w4 = *reinterpret_cast<const float4*>(wr + j);
#pragma unroll
        for (int t = 0; t < kMaxRows; ++t) {
          if (t < T) {
            const float4 x4 = *reinterpret_cast<const float4*>(&xs[t][j]);
            acc[t] = fmaf(w4.x, x4.x, acc[t]);
            acc[t] = fmaf(w4.y, x4.y, acc[t]);
            acc[t] = fmaf(w4.z, x4.z, acc[t]);
            acc[t] = fmaf(w4.w, x4.w, acc[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kMaxRows; ++t) {
        float v = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && t < T) partial[((long long)jb * kMaxRows + t) * E + e] = v;
      }
    }
  }

  // -- activation fragments of x, and this window's combine counters --------
  if (L.bits == 4) write_x_frags<4>(L, W); else write_x_frags<2>(L, W);
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = tid; i < d / 16; i += blockDim.x) W.counters[i] = 0;
  }

  // -- last CTA: softmax, top-k, grouping -----------------------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned total = gridDim.x * gridDim.y;
    is_last = (atomicAdd(W.ticket, 1u) == total - 1u);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  const int njb = gridDim.y;
  for (int i = tid; i < T * E; i += blockDim.x) {
    const int t = i / E, e = i % E;
    float v = 0.f;
    for (int b = 0; b < njb; ++b) v += __ldcg(partial + ((long long)b * kMaxRows + t) * E + e);
    if (L.router_b) v += L.router_b[e];
    lg[t][e] = v;
    W.logits[t * E + e] = v;
  }
  __syncthreads();

  Plan* P = W.plan;
  if (warp < T) {
    const int t = warp;
    float m = -INFINITY;
    bool finite = true;
    for (int e = lane; e < E; e += 32) {
      const float v = lg[t][e];
      finite &= isfinite(v);
      m = fmaxf(m, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!__all_sync(0xffffffffu, finite) && lane == 0) atomicOr(W.err, kErrNonFinite);
    float z = 0.f;
    for (int e = lane; e < E; e += 32) z += expf(lg[t][e] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    // top-k by logit, descending, ties -> lower expert index
    unsigned taken = 0u;  // bit i: expert lane + 32*i already selected
    float wsum = 0.f;
    float wsel[kMaxTopK];
    int esel[kMaxTopK];
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
      for (int i = 0, e = lane; e < E; ++i, e += 32) {
        const float v = lg[t][e];
        if (!((taken >> i) & 1u) && (v > bv || (v == bv && e < be))) { bv = v; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      if (be == 0x7fffffff) be = 0;  // only with non-finite logits
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      esel[j] = be;
      wsel[j] = expf(bv - m) / z;
      wsum += wsel[j];
    }
    if (lane == 0) {
      for (int j = 0; j < k; ++j) {
        const float g = L.renorm ? wsel[j] / wsum : wsel[j];
        sel[t * k + j] = esel[j];
        P->topk_idx[t * k + j] = esel[j];
        P->topk_w[t * k + j] = g;
        if (W.out_topk_idx) W.out_topk_idx[t * k + j] = esel[j];
        if (W.out_topk_w) W.out_topk_w[t * k + j] = g;
      }
    }
  }
  __syncthreads();

  // counting sort of entries by expert
  const int nent = T * k;
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int i = 0; i < nent; ++i) c += (sel[i] == e);
    cnt[e] = c;
    flag[e] = c > 0;
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0, nd = 0;
    for (int e = 0; e < E; ++e) {
      P->offsets[e] = off;
      if (W.out_offsets) W.out_offsets[e] = off;
      off += cnt[e];
      if (flag[e]) { P->distinct[nd] = e; if (W.out_distinct) W.out_distinct[nd] = e; ++nd; }
    }
    P->offsets[E] = off;
    if (W.out_offsets) W.out_offsets[E] = off;
    P->n_distinct = nd;
    P->T = T;
    if (W.out_ndistinct) *W.out_ndistinct = nd;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    P->counts[e] = cnt[e];
    if (W.out_counts) W.out_counts[e] = cnt[e];
    int pos = P->offsets[e];
    for (int i = 0; i < nent; ++i) {
      if (sel[i] == e) {
        P->entries[pos] = i;
        if (W.out_entries) W.out_entries[pos] = i;
        ++pos;
      }
    }
  }
  if (tid == 0) *W.ticket = 0u;
}

void launch_router(const LayerDev& L, const WindowBufs& W, float* partial, cudaStream_t s) {
  dim3 grid((L.E + kRouterExpertsPerCta - 1) / kRouterExpertsPerCta, (L.d + kRouterCols - 1) / kRouterCols);
  router_kernel<<<grid, kRouterThreads, 0, s>>>(L, W, partial);
}

int router_partial_floats(int d, int E) { return ((d + kRouterCols - 1) / kRouterCols) * kMaxRows * E; }

}  // namespace strata
