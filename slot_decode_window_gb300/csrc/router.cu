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
// activation fragment layout the expert kernels read (block sums by warp
// shuffles).  The partial logits are summed in a fixed order, and the
// softmax, top-k and grouping run, at the start of the gate/up kernel (see
// experts.cu), so this kernel has no serial tail.
#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace strata {

constexpr int kRouterCols = 256;
constexpr int kRouterExpertsPerCta = 8;

template <int BITS>
__device__ void write_x_frags(const LayerDev& L, const WindowBufs& W) {
  constexpr int B = Fmt<BITS>::kBlock;
  const int d = L.d;
  const int nmk = (d / B + 15) / 16;
  const long long fh = frag_halves(d, nmk);
  const long long n_el = (long long)W.T * d;  // a multiple of 64: warps never straddle a block or a row
  const long long stride = (long long)gridDim.x * gridDim.y * blockDim.x;
  const long long tid = ((long long)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  const long long n_iter = (n_el + stride - 1) / stride;
  for (long long it = 0; it < n_iter; ++it) {
    const long long i = tid + it * stride;
    const bool in = i < n_el;
    const int t = in ? (int)(i / d) : 0, j = in ? (int)(i % d) : 0;
    const float v = in ? W.x[i] : 0.f;
    __half* base = W.xfrag + t * fh;
    if (in) {
      int off;
      float f;
      frag_main_pos<BITS>(j, off, f);
      __half hi, lo;
      split_hi_lo(v * f, hi, lo);
      base[off] = hi;
      base[d + off] = lo;
    }
    float s = v;
#pragma unroll
    for (int o = B / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (in && (j % B) == 0) {
      __half hi, lo;
      split_hi_lo(s, hi, lo);
      const int off = frag_sum_pos(j / B);
      base[2 * d + off] = hi;
      base[2 * d + nmk * 16 + off] = lo;
    }
  }
}

__global__ void __launch_bounds__(kRouterThreads) router_kernel(LayerDev L, WindowBufs W, float* partial) {
  __shared__ __align__(16) float xs[kMaxRows][kRouterCols];

  // The expert kernel may start its prologue now; it waits for this grid's
  // completion before reading anything written here.
  griddep_launch_dependents();

  const int T = W.T, d = L.d, E = L.E;
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

}

void launch_router(const LayerDev& L, const WindowBufs& W, float* partial, cudaStream_t s) {
  dim3 grid((L.E + kRouterExpertsPerCta - 1) / kRouterExpertsPerCta, (L.d + kRouterCols - 1) / kRouterCols);
  router_kernel<<<grid, kRouterThreads, 0, s>>>(L, W, partial);
}

int router_partial_floats(int d, int E) { return ((d + kRouterCols - 1) / kRouterCols) * kMaxRows * E; }

}  // namespace strata
