// The verify-window MoE step as one persistent kernel.
//
// The Strata docs ("BATCHING.md", "Several requests at once (batch slots)",
// opening paragraph) state the scheme: a verify window carries one token of
// each open conversation, and the shared expert and every routed expert that
// rows of a window share are read once per window for all of them.  Here every
// distinct expert's packed tiles are streamed from HBM once and multiplied
// against all of that expert's rows (up to 8) in one pass.  The pages give no
// formulas; the kernel computes the plain reading stated in strata_window.h.
//
// One launch per window, one CTA per SM (cooperative launch, so all CTAs are
// resident and the few cross-CTA waits below always end):
//   R. router: each CTA stages one 512-column chunk of the rows of x and its
//      warps take that chunk's experts of the fp32 router GEMV, writing
//      partial logits; the CTA then turns its share of the chunk into the
//      activation fragments of the gate/up MMAs.  One grid barrier follows.
//   P. every CTA sums the partial logits in a fixed order and derives the same
//      routing plan: fp32 softmax, top-k by logit (ties to the lower expert),
//      gate weights, counting-sort row groups (bit-exact in every CTA).
//   0. gate/up: for the shared expert and each distinct routed expert e, for
//      each 16-row tile of Wg_e, Wu_e: gu = Wg_e x_t, uu = Wu_e x_t for every
//      row t of e's group, written in fp32.  Each finished task bumps its
//      group's completion counter.
//   1. down: a CTA starts a group's down tiles once that group's gate/up tasks
//      have all landed (bounded wait on the counter; the weights stream in
//      meanwhile); h = silu(gu) * uu is formed while staging the group; then
//      o = g_tj * (Wd_e h), or s_t = Wsd h_t for the shared expert.  The CTA
//      whose contribution to a 16-row slice of y lands last sums
//      y_t = s_t + sum_j o_tj in a fixed order.
//
// Within a CTA a producer warp streams k-chunks of each task's tiles into a
// shared-memory ring with bulk async copies; 16 consumer warps split the
// task's sub-tiles and k-steps.  A consumer turns packed codes into fp16
// subnormals (one AND per code pair), multiplies them against the rows'
// activations with mma.sync m16n8k16 (activations split into fp16 hi + lo
// parts so the products keep fp32-level accuracy), applies each block's scale
// to the fp32 accumulator fragment, and adds the min term with one more MMA
// against per-block activation sums.  Lanes whose activation columns are
// unused (groups of fewer than 4 or 8 rows) skip their operand loads.
#include <cstdlib>

#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace strata {

namespace {

constexpr int kMaxSub = 4;  // sub-tiles per task
// Where a due tier round keeps its arrays in the ring region while stage R's
// staged rows of x (kMaxRows x kRouterCols floats) still sit at its start.
constexpr int kTierScratchOff = kMaxRows * kRouterCols * 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;

// Stage timestamps for timing builds (-DSTRATA_STAMPS): one lane of the CTA
// records %globaltimer at stage boundaries into g_stamps[cta][slot].  The
// default build compiles these to nothing.
#ifdef STRATA_STAMPS
}  // namespace
__device__ unsigned long long g_stamps[1024][32];
namespace {
__device__ __forceinline__ void stamp(int slot) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  g_stamps[blockIdx.x][slot] = t;
}
#define STAMP(tid_, slot_) \
  do {                     \
    if (threadIdx.x == (tid_)) stamp(slot_); \
  } while (0)
// per-task trace: g_trace[cta][phase][task slot][event]
__device__ unsigned long long g_trace[1024][4][32][4];
__device__ unsigned long long g_ptrace[1024][4][64];  // producer: chunk issue times
__device__ __forceinline__ void trace(int phase, int slot, int ev) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  if (slot < 32) g_trace[blockIdx.x][phase][slot][ev] = t;
}
#define TRACE(tid_, ph_, slot_, ev_) \
  do {                               \
    if (threadIdx.x == (tid_)) trace(ph_, slot_, ev_); \
  } while (0)
#define PTRACE(ph_, n_)                                                   \
  do {                                                                    \
    unsigned long long t_;                                                \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                \
    if ((n_) < 64) g_ptrace[blockIdx.x][ph_][n_] = t_;                    \
  } while (0)
#else
#define TRACE(tid_, ph_, slot_, ev_) \
  do {                               \
  } while (0)
#define PTRACE(ph_, n_) \
  do {                  \
  } while (0)
#define STAMP(tid_, slot_) \
  do {                     \
  } while (0)
#endif

// Every wait below is bounded by W.wait_cycles (by default 2^31 cycles, about
// a second at GB300 clocks); one that gives up sets the error word and returns.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, unsigned* err, volatile int* abort_flag,
                                         long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) {
      atomicOr(err, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Shared-memory activation (B operand) layout, per set (hi, or lo when rows > 4):
//   main: k-step ks holds S/8 planes of 256 halves; in plane p, column col
//         (0..7) and lane quad c (0..3) own 8 halves at (col*4 + c)*8, so a
//         warp's 16-byte loads of one plane are contiguous (no bank conflicts).
//   sums: min group mk holds 16 halves per column: (mk*8 + col)*16 + c*4.
template <int BITS>
__device__ __forceinline__ int bmain_off(int ks, int p, int col, int c) {
  return ks * 32 * Fmt<BITS>::kBHalves + p * 256 + (col * 4 + c) * 8;
}

// One k-step of one sub-tile.  acc is in units of 2^-24 (subnormal codes).
// bk points at this lane's slot of plane 0 of the k-step (set 0); lanes whose
// MMA column is unused point at column 0 instead (same-address reads
// broadcast, and a column of the product depends only on that column of B).
// One k-step's A-side words of one lane: its 16 code bytes and the scale
// record(s) of its rows g and g + 8 (4-bit: 8 bytes; 2-bit: 32 bytes).
template <int BITS> struct KWords;
template <> struct KWords<4> {
  uint4 cw;
  uint2 sr;
};
template <> struct KWords<2> {
  uint4 cw;
  uint4 sa, sb;
};

template <int BITS>
__device__ __forceinline__ KWords<BITS> kwords_smem(const uint8_t* __restrict__ ch, int lane) {
  const int g = lane >> 2;
  KWords<BITS> kw;
  kw.cw = *reinterpret_cast<const uint4*>(ch + lane * 16);
  if constexpr (BITS == 4) {
    kw.sr = *reinterpret_cast<const uint2*>(ch + 512 + g * 8);
  } else {
    kw.sa = *reinterpret_cast<const uint4*>(ch + 512 + g * 32);       // s(g, b0..b7)
    kw.sb = *reinterpret_cast<const uint4*>(ch + 512 + g * 32 + 16);  // s(g+8, b0..b7)
  }
  return kw;
}

// A row's hi and lo parts run in separate MMA chains in both column layouts:
// paired, columns (2q, 2q + 1) are row q's (hi, lo), so a lane's d[0], d[1]
// (weight row g) and d[2], d[3] (row g + 8) pair up in place; two-set, the
// hi parts are one set of columns (d) and the lo parts the other (e).  Each
// block's t = d_hi + d_lo is then scaled into the accumulator, so a row's
// arithmetic is the same whether its group has 1 row or 8: the Strata docs
// ("BATCHING.md", section "Exactness") make a batch row's arithmetic the
// single-token window's.  acc: paired, [0] and [2] hold weight rows g and
// g + 8; two-set, [0..3] hold (rows 2q, 2q + 1) x (g, g + 8).
template <bool PAIRED>
__device__ __forceinline__ void scale_into(float (&acc)[4], const float (&d)[4], const float (&e)[4], float sg,
                                           float s8) {
  if constexpr (PAIRED) {
    acc[0] = fmaf(sg, d[0] + d[1], acc[0]);
    acc[2] = fmaf(s8, d[2] + d[3], acc[2]);
  } else {
    acc[0] = fmaf(sg, d[0] + e[0], acc[0]);
    acc[1] = fmaf(sg, d[1] + e[1], acc[1]);
    acc[2] = fmaf(s8, d[2] + e[2], acc[2]);
    acc[3] = fmaf(s8, d[3] + e[3], acc[3]);
  }
}

template <int BITS, bool PAIRED>
__device__ __forceinline__ void kstep_compute(const KWords<BITS>& kw, const __half* __restrict__ bk, int bm_set,
                                              int lane, float (&acc)[4]) {
  const float z4[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (BITS == 4) {
    const uint4 bA = *reinterpret_cast<const uint4*>(bk);
    const uint4 bB = *reinterpret_cast<const uint4*>(bk + 256);
    uint4 lA = bA, lB = bB;
    if constexpr (!PAIRED) {
      lA = *reinterpret_cast<const uint4*>(bk + bm_set);
      lB = *reinterpret_cast<const uint4*>(bk + bm_set + 256);
    }
    const uint4 cw = kw.cw;
    const uint2 sr = kw.sr;
    const float2 sg = __half22float2(*reinterpret_cast<const __half2*>(&sr.x));
    const float2 s8 = __half22float2(*reinterpret_cast<const __half2*>(&sr.y));
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint32_t wg = blk ? cw.z : cw.x, w8 = blk ? cw.w : cw.y;
      const uint32_t wg2 = wg >> 8, w82 = w8 >> 8;
      const uint4 b = blk ? bB : bA;
      float d[4], e[4];
      mma16816(d, dq_pair(wg, 0x000F000Fu), dq_pair(w8, 0x000F000Fu), dq_pair(wg2, 0x000F000Fu),
               dq_pair(w82, 0x000F000Fu), b.x, b.y, z4);
      mma16816(d, dq_pair(wg, 0x00F000F0u), dq_pair(w8, 0x00F000F0u), dq_pair(wg2, 0x00F000F0u),
               dq_pair(w82, 0x00F000F0u), b.z, b.w, d);
      if constexpr (!PAIRED) {
        const uint4 l = blk ? lB : lA;
        mma16816(e, dq_pair(wg, 0x000F000Fu), dq_pair(w8, 0x000F000Fu), dq_pair(wg2, 0x000F000Fu),
                 dq_pair(w82, 0x000F000Fu), l.x, l.y, z4);
        mma16816(e, dq_pair(wg, 0x00F000F0u), dq_pair(w8, 0x00F000F0u), dq_pair(wg2, 0x00F000F0u),
                 dq_pair(w82, 0x00F000F0u), l.z, l.w, e);
      }
      scale_into<PAIRED>(acc, d, e, blk ? sg.y : sg.x, blk ? s8.y : s8.x);
    }
  } else {
    const uint4 cw = kw.cw, sa = kw.sa, sb = kw.sb;
    const uint32_t cwv[4] = {cw.x, cw.y, cw.z, cw.w};
    const uint32_t sav[4] = {sa.x, sa.y, sa.z, sa.w};
    const uint32_t sbv[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 b = *reinterpret_cast<const uint4*>(bk + 256 * j);
      uint4 l = b;
      if constexpr (!PAIRED) l = *reinterpret_cast<const uint4*>(bk + bm_set + 256 * j);
      const uint32_t w = cwv[j], w2 = w >> 8;
      const float2 sgp = __half22float2(*reinterpret_cast<const __half2*>(&sav[j]));
      const float2 s8p = __half22float2(*reinterpret_cast<const __half2*>(&sbv[j]));
      float d[4], e[4];
      mma16816(d, dq_pair(w, 0x00030003u), dq_pair(w2, 0x00030003u), dq_pair(w, 0x000C000Cu),
               dq_pair(w2, 0x000C000Cu), b.x, b.y, z4);
      if constexpr (!PAIRED)
        mma16816(e, dq_pair(w, 0x00030003u), dq_pair(w2, 0x00030003u), dq_pair(w, 0x000C000Cu),
                 dq_pair(w2, 0x000C000Cu), l.x, l.y, z4);
      scale_into<PAIRED>(acc, d, e, sgp.x, s8p.x);
      mma16816(d, dq_pair(w, 0x00300030u), dq_pair(w2, 0x00300030u), dq_pair(w, 0x00C000C0u),
               dq_pair(w2, 0x00C000C0u), b.z, b.w, z4);
      if constexpr (!PAIRED)
        mma16816(e, dq_pair(w, 0x00300030u), dq_pair(w2, 0x00300030u), dq_pair(w, 0x00C000C0u),
                 dq_pair(w2, 0x00C000C0u), l.z, l.w, z4);
      scale_into<PAIRED>(acc, d, e, sgp.y, s8p.y);
    }
  }
}

// A warp's partial outputs of one task for the reduction buffer: per output
// fma(acc, 2^24, m_hi + m_lo), the min term's hi and lo chains (paired: accm
// columns 2q, 2q + 1; two-set: accm and accm2) added first.  Paired: the
// lane's two outputs (weight rows g, g + 8) land in .x and .z; two-set: its
// four outputs (rows 2q, 2q + 1 at g, g + 8) in .x .y .z .w.
template <bool PAIRED>
__device__ __forceinline__ float4 partials(const float (&acc)[4], const float (&accm)[4], const float (&accm2)[4]) {
  if constexpr (PAIRED) {
    return make_float4(fmaf(acc[0], kDqUnscale, accm[0] + accm[1]), 0.f,
                       fmaf(acc[2], kDqUnscale, accm[2] + accm[3]), 0.f);
  } else {
    return make_float4(fmaf(acc[0], kDqUnscale, accm[0] + accm2[0]), fmaf(acc[1], kDqUnscale, accm[1] + accm2[1]),
                       fmaf(acc[2], kDqUnscale, accm[2] + accm2[2]), fmaf(acc[3], kDqUnscale, accm[3] + accm2[3]));
  }
}

// One k-step of one sub-tile from a staged chunk in shared memory.
template <int BITS, bool PAIRED>
__device__ __forceinline__ void kstep_mma(const uint8_t* __restrict__ ch, const __half* __restrict__ bk, int bm_set,
                                          int lane, float (&acc)[4]) {
  kstep_compute<BITS, PAIRED>(kwords_smem<BITS>(ch, lane), bk, bm_set, lane, acc);
}

// This warp's share of one staged chunk of its sub-tile: k-steps [k0, k1)
// (chunk-local, tile k-step ks_base + kl) and min groups [m0, m1) (chunk-local,
// tile group mk_base + ml).
// VMAP: the activation is the grouped-query broadcast of v, so k-step ks of
// the 4096-wide input reads v's k-step (ks >> kpg) * 2^kph + (ks & (2^kph - 1))
// (kph, kpg: log2 of k-steps per head and per kv group).
template <int BITS, bool PAIRED, bool VMAP = false>
__device__ __forceinline__ void chunk_mma(const uint8_t* __restrict__ sub, int mins_off, int ks_base, int k0, int k1,
                                          int mk_base, int m0, int m1, const __half* __restrict__ bm,
                                          const __half* __restrict__ bs, int bm_set, int bs_set, int lane_b, int lane,
                                          float (&acc)[4], float (&accm)[4], float (&accm2)[4], int kph = 0,
                                          int kpg = 0) {
  constexpr int S = Fmt<BITS>::kBHalves;
  const uint8_t* a = sub + k0 * Fmt<BITS>::kChunk;
  const __half* bk = bm + (ks_base + k0) * 32 * S + lane_b * 8;
#pragma unroll 2
  for (int kl = k0; kl < k1; ++kl) {
    if constexpr (VMAP) {
      const int ks = ks_base + kl;
      bk = bm + (((ks >> kpg) << kph) + (ks & ((1 << kph) - 1))) * 32 * S + lane_b * 8;
    }
    kstep_mma<BITS, PAIRED>(a, bk, bm_set, lane, acc);
    a += Fmt<BITS>::kChunk;
    bk += 32 * S;
  }
  const uint8_t* am_p = sub + mins_off + m0 * 512 + lane * 16;
  const __half* sp = bs + (mk_base + m0) * 128 + lane_b * 4;
  for (int ml = m0; ml < m1; ++ml) {
    const uint2 b = *reinterpret_cast<const uint2*>(sp);
    const uint4 am = *reinterpret_cast<const uint4*>(am_p);
    mma16816(accm, am.x, am.y, am.z, am.w, b.x, b.y, accm);
    if constexpr (!PAIRED) {
      const uint2 l = *reinterpret_cast<const uint2*>(sp + bs_set);
      mma16816(accm2, am.x, am.y, am.z, am.w, l.x, l.y, accm2);
    }
    am_p += 512;
    sp += 128;
  }
}

// Task layout of one phase.
struct PhaseTasks {
  int ntask_s;  // tasks of the shared expert
  int ntask_e;  // tasks of each routed expert
  int mt;       // 16-row tiles per task
  int t0, t1;   // this CTA's task range
};

// Routing plan and task map, cached in shared memory for the whole kernel.
struct SPlan {
  int nd;
  int distinct[kMaxExperts];
  int counts[kMaxExperts];
  int offsets[kMaxExperts];
  int entries[kMaxEntries];
  int sel[kMaxEntries];
  float topk_w[kMaxEntries];
  int wscan[32];
  int wcnt[2][kMaxExperts];         // per-warp expert counts of the grouping pass
  int finish[kMaxEntries * 4];      // row slices this CTA combines
  int nfinish;
  int ok;                           // the grid barrier passed
  PhaseTasks pt[4];                 // gate/up, down, dense q/k/v, dense o
  alignas(8) uint64_t img_bar;      // completion of a bulk copy of a B image into B
  unsigned img_uses;                // copies completed so far (the wait's parity)
};

// The B-image copy barrier (thread 0, before the block barrier that follows
// the kernel's set-up).
__device__ __forceinline__ void init_img(SPlan& sp) {
  if (threadIdx.x == 0) {
    mbar_init(&sp.img_bar, 1);
    sp.img_uses = 0;
    fence_mbar_init();
  }
}

__device__ __forceinline__ unsigned ord_f32(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(unsigned u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// ---------------------------------------------------------------------------
// stage R: router partial logits and x fragments (all threads of all CTAs)
// ---------------------------------------------------------------------------
// The x fragments of a window live in global memory as the image of the
// shared-memory B operand of a group holding all T rows in order (the shared
// expert's group, and every dense phase's): set s of the main part at
// s * 8d halves, laid out as bmain_off; the sums after both sets, set s at
// 16d + s * 128 nmk halves, laid out as the B sums.  Rows > 4 use two sets
// (hi, lo); otherwise set 0 holds columns 2t (hi) and 2t + 1 (lo).  A group
// of all rows then stages with a plain copy; any other group gathers its
// rows' 16-byte pieces from their columns.
struct XImg {
  int set, col;  // row t's place for part (0: hi, 1: lo)
  __device__ __forceinline__ XImg(int T, int t, int part) {
    set = T <= 4 ? 0 : part;
    col = T <= 4 ? 2 * t + part : t;
  }
};
// Element with fragment offset off (frag_main_pos) of row t, part part.
template <int BITS>
__device__ __forceinline__ long long ximg_main(int T, int d, int t, int part, int off) {
  constexpr int S = Fmt<BITS>::kBHalves;
  const XImg q(T, t, part);
  return (long long)q.set * 8 * d + bmain_off<BITS>(off / (4 * S), (off % S) >> 3, q.col, (off / S) & 3) + (off & 7);
}
// Block sum with sum offset soff (frag_sum_pos) of row t, part part.
__device__ __forceinline__ long long ximg_sum(int T, int d, int nmk, int t, int part, int soff) {
  const XImg q(T, t, part);
  return 16LL * d + (long long)q.set * 128 * nmk + ((soff >> 4) * 8 + q.col) * 16 + ((soff >> 2) & 3) * 4 + (soff & 3);
}

template <int BITS>
__device__ void write_x_frags(const LayerDev& L, const WindowBufs& W) {
  constexpr int B = Fmt<BITS>::kBlock;
  const int d = L.d;
  const int nmk = (d / B + 15) / 16;
  const long long n_el = (long long)W.T * d;  // a multiple of 64: warps never straddle a block or a row
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long n_iter = (n_el + stride - 1) / stride;
  for (long long it = 0; it < n_iter; ++it) {
    const long long i = tid + it * stride;
    const bool in = i < n_el;
    const int t = in ? (int)(i / d) : 0, j = in ? (int)(i % d) : 0;
    const float v = in ? (W.rinv ? W.x[i] * W.rinv[t] : W.x[i]) : 0.f;
    if (in) {
      int off;
      float f;
      frag_main_pos<BITS>(j, off, f);
      __half hi, lo;
      split_hi_lo(v * f, hi, lo);
      W.xfrag[ximg_main<BITS>(W.T, d, t, 0, off)] = hi;
      W.xfrag[ximg_main<BITS>(W.T, d, t, 1, off)] = lo;
    }
    float s = v;
#pragma unroll
    for (int o = B / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (in && (j % B) == 0) {
      __half hi, lo;
      split_hi_lo(s, hi, lo);
      const int off = frag_sum_pos(j / B);
      W.xfrag[ximg_sum(W.T, d, nmk, t, 0, off)] = hi;
      W.xfrag[ximg_sum(W.T, d, nmk, t, 1, off)] = lo;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // the image is read by bulk copies
}

// 1 / sqrt(mean(x_t^2) + 1e-6) of every row (warp t sums row t in a fixed
// order, so every CTA gets the same bits).  Ends with a block barrier.
__device__ __noinline__ void row_rinv(const float* x, int T, int d, float* s_rinv) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < T) {
    const float4* xr = reinterpret_cast<const float4*>(x + (long long)warp * d);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < d / 4; j0 += 128) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * 32 + lane;
        if (j < d / 4) {
          const float4 v = __ldcg(xr + j);
          acc[u] = fmaf(v.x, v.x, acc[u]);
          acc[u] = fmaf(v.y, v.y, acc[u]);
          acc[u] = fmaf(v.z, v.z, acc[u]);
          acc[u] = fmaf(v.w, v.w, acc[u]);
        }
      }
    }
    float ss = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_rinv[warp] = 1.0f / sqrtf(ss / (float)d + 1e-6f);
  }
  __syncthreads();
}

// Sum of v[0..7] (one value per row t) over the 32 lanes of a warp, by
// halving: after the exchanges across lane bits 4, 3 and 2 every lane holds a
// partial sum of one row, t = 4*b4 + 2*b3 + b2 (its lane bits), and two more
// exchanges complete it.  9 shuffles instead of 8 x 5.
__device__ __forceinline__ float warp_sum8(float (&v)[kMaxRows], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? v[i] : v[i + 4], keep = b4 ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? v[i] : v[i + 2], keep = b3 ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const float send = b2 ? v[0] : v[1], keep = b2 ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  return v[0];
}

// Stage R.  The d columns are cut into njb chunks of kRouterCols; the CTAs
// are dealt out over the chunks (CTA c takes chunk c mod njb, together with
// the other CTAs of that chunk), so each CTA stages its chunk of the T rows of
// x in shared memory once.  Its warps then take the chunk's experts in turn:
// partial[jb][t][e] = sum over the chunk of Wr[e][j] x[t][j] (times 1/RMS of
// row t in a decoder layer).  Last, the CTA writes its share of the chunk's
// activation fragments (fp16 hi/lo and block sums) from the staged rows.
template <int BITS>
__device__ __noinline__ void router_stage(const LayerDev& L, const WindowBufs& W, float* xs) {
  constexpr int B = Fmt<BITS>::kBlock;
  const int T = W.T, d = L.d, E = L.E, njb = W.njb, G = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const bool spread = G >= njb;  // several CTAs per chunk (always, for the shapes here)
  const int nmk = (d / B + 15) / 16;
  for (int jb = spread ? (int)blockIdx.x % njb : (int)blockIdx.x; jb < njb; jb += spread ? njb : G) {
    const int cpc = spread ? G / njb + (jb < G % njb ? 1 : 0) : 1;  // CTAs on this chunk
    const int ci = spread ? (int)blockIdx.x / njb : 0;              // this CTA among them
    const int j0 = jb * kRouterCols, ncol = min(kRouterCols, d - j0);
    const int nq = ncol / 4;
    __syncthreads();  // xs is free (a previous chunk of this loop is done)
    for (int i = threadIdx.x; i < T * nq; i += blockDim.x) {
      const int t = i / nq, q = i - t * nq;
      cp_async16(xs + t * kRouterCols + 4 * q, W.x + (long long)t * d + j0 + 4 * q);
    }
    const int e0 = (int)((long long)E * ci / cpc), e1 = (int)((long long)E * (ci + 1) / cpc);
    // a warp's router row segment, loaded a row ahead (the first one while the
    // rows of x are still landing)
    constexpr int kJ = kRouterCols / 128;
    float4 w[kJ];
    auto load_w = [&](int e) {
      const float* wr = L.router_w + (long long)e * d + j0;
#pragma unroll
      for (int i = 0; i < kJ; ++i) {
        const int j = lane * 4 + 128 * i;
        w[i] = (e < e1 && j < ncol) ? __ldcs(reinterpret_cast<const float4*>(wr + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    load_w(e0 + warp);
    cp_async_wait_all();
    __syncthreads();
    for (int e = e0 + warp; e < e1; e += nwarps) {
      float acc[kMaxRows];
#pragma unroll
      for (int t = 0; t < kMaxRows; ++t) acc[t] = 0.f;
#pragma unroll
      for (int i = 0; i < kJ; ++i) {
        const int j = lane * 4 + 128 * i;
        if (j < ncol) {
#pragma unroll
          for (int t = 0; t < kMaxRows; ++t) {
            if (t < T) {
              const float4 x4 = *reinterpret_cast<const float4*>(xs + t * kRouterCols + j);
              acc[t] = fmaf(w[i].x, x4.x, acc[t]);
              acc[t] = fmaf(w[i].y, x4.y, acc[t]);
              acc[t] = fmaf(w[i].z, x4.z, acc[t]);
              acc[t] = fmaf(w[i].w, x4.w, acc[t]);
            }
          }
        }
      }
      load_w(e + nwarps);
      const float v = warp_sum8(acc, lane);
      const int t = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
      if ((lane & 3) == 0 && t < T)
        W.partial[((long long)jb * kMaxRows + t) * E + e] = W.rinv ? v * W.rinv[t] : v;
    }
    // this CTA's share of the chunk's activation fragments: units of 32
    // consecutive elements of one row (whole blocks), one per warp
    const int upr = ncol / 32, nu = T * upr;
    for (int u = ci + cpc * warp; u < nu; u += cpc * nwarps) {
      const int t = u / upr, jj = (u - t * upr) * 32 + lane, j = j0 + jj;
      const float v = W.rinv ? xs[t * kRouterCols + jj] * W.rinv[t] : xs[t * kRouterCols + jj];
      int off;
      float f;
      frag_main_pos<BITS>(j, off, f);
      __half hi, lo;
      split_hi_lo(v * f, hi, lo);
      W.xfrag[ximg_main<BITS>(T, d, t, 0, off)] = hi;
      W.xfrag[ximg_main<BITS>(T, d, t, 1, off)] = lo;
      float sm = v;
#pragma unroll
      for (int o = B / 2; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      if ((j % B) == 0) {
        split_hi_lo(sm, hi, lo);
        const int soff = frag_sum_pos(j / B);
        W.xfrag[ximg_sum(T, d, nmk, t, 0, soff)] = hi;
        W.xfrag[ximg_sum(T, d, nmk, t, 1, soff)] = lo;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // the image is read by bulk copies
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < d / 16; i += blockDim.x) W.counters[i] = 0;
    for (int i = threadIdx.x; i <= E; i += blockDim.x) W.done_gu[i] = 0;
  }
}

// All CTAs arrive; thread 0 waits (bounded) until every CTA of this window has.
// The counter only grows: the window's target is the next multiple of the grid
// (plus W.bar_extra, which is 0 except in tests that make the wait run out).
// grid_barrier_split arrives, runs `between` with all threads of the CTA when
// `run` (the same for every thread of the CTA), and then waits.
template <typename F>
__device__ bool grid_barrier_split(const WindowBufs& W, int* s_ok, bool run, F between) {
  __shared__ unsigned long long s_target;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long n = gridDim.x;
    const unsigned long long old = atomicAdd(W.gbar, 1ull);
    s_target = (old / n + 1) * n + (unsigned long long)W.bar_extra;
  }
  if (run) {
    between();
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const unsigned long long target = s_target;
    const long long t0 = clock64();
    int ok = 1;
    while (ld_acquire_u64(W.gbar) < target) {
      if (clock64() - t0 > W.wait_cycles) {
        atomicOr(W.err, kErrTimeout);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

__device__ __forceinline__ bool grid_barrier(const WindowBufs& W, int* s_ok) {
  return grid_barrier_split(W, s_ok, false, [] {});
}

// Row t (warp t; lane holds experts lane + 32 i): logits as the column-chunk
// partials summed in chunk order (four chunks' loads in flight at a time, so
// every CTA gets the same bits), top-k by logit (descending, ties to the lower
// expert), fp32 softmax over all E, and the selected experts' gate weights.
// NI: experts per lane, ceil(E / 32) rounded up to a power of two (the
// caller dispatches on E), so lanes scan no keys that cannot be experts.
template <int NI>
__device__ __forceinline__ void plan_row(const LayerDev& L, const WindowBufs& W, SPlan& sp, int t, int lane,
                                         bool pub) {
  const int E = L.E, k = L.k, njb = W.njb;
  float val[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) val[i] = 0.f;
  const float* pr = W.partial + (long long)t * E + lane;
  for (int b0 = 0; b0 < njb; b0 += 4) {
    float part[4][NI];
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int i = 0; i < NI; ++i)
        part[b][i] = (b0 + b < njb && lane + 32 * i < E) ? __ldcg(pr + (long long)(b0 + b) * kMaxRows * E + 32 * i)
                                                          : 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int i = 0; i < NI; ++i) val[i] += part[b][i];
  }
  unsigned key[NI];
  bool finite = true;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    if (e < E && L.router_b) val[i] += L.router_b[e];
    if (e < E) finite &= isfinite(val[i]);
    key[i] = e < E ? ord_f32(val[i]) : 0u;  // 0: below every real logit
  }
  if (!__all_sync(0xffffffffu, finite) && lane == 0 && pub) atomicOr(W.err, kErrNonFinite);
  int esel = 0;
  float lsel = 0.f, top = 0.f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    unsigned bk = 0u;
    int bi_l = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (key[i] > bk) {
        bk = key[i];
        bi_l = i;
      }
    const unsigned kmax = __reduce_max_sync(0xffffffffu, bk);
    const unsigned cand = (bk == kmax && bk != 0u) ? (unsigned)(lane + 32 * bi_l) : 0xffffffffu;
    int bi = (int)__reduce_min_sync(0xffffffffu, cand);
    if (bi < 0 || bi >= E) bi = 0;  // only with non-finite logits
    if ((bi & 31) == lane) {
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (i == (bi >> 5)) key[i] = 0u;
    }
    const float lv = unord_f32(kmax);
    if (j == 0) top = lv;
    if (lane == j) {
      esel = bi;
      lsel = lv;
    }
  }
  // softmax over all E logits, shifted by the largest
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < NI; ++i)
    if (lane + 32 * i < E) z += expf(val[i] - top);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float p = lane < k ? expf(lsel - top) / z : 0.f;
  float wsum = p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane < k) {
    const float g = L.renorm ? p / wsum : p;
    const int ent = t * k + lane;
    sp.sel[ent] = esel;
    sp.topk_w[ent] = g;
    if (pub) {
      if (W.out_topk_idx) W.out_topk_idx[ent] = esel;
      if (W.out_topk_w) W.out_topk_w[ent] = g;
    }
  }
}

// The adaptive tier's bookkeeping.  The Strata docs ("BATCHING.md", the
// adaptive expert tier paragraphs) have batch windows count the experts they
// route to and, every --adapt-every windows, swap the most-routed experts
// outside the fast tier with the least-routed ones inside, up to
// --adapt-swaps, a swap needing the incoming count to clear --adapt-min-gain
// times the outgoing one, with --adapt-decay aging the counts.  Here:
//   c_e += (entries routed to e in this window)            (fp32)
//   after every adapt_every-th window, a round: outside experts by c
//   descending and tier experts by c ascending (ties to the lower expert)
//   pair up in order; pair i swaps while i < adapt_swaps, c_in > c_out and
//   c_in >= min_gain * c_out (the first pair that fails ends the round); then
//   c_e *= decay.
// The counts are added by CTA 0 during the plan with fire-and-forget atomics
// (one adder per counter per window, so the fp32 sums are deterministic).  A
// round that is due runs in CTA 0 of the next window while that CTA waits at
// its first grid barrier (before the window's own counts are added), or in
// strata_tier_read's one-CTA launch, whichever comes first: the rounds
// counter says whether it has run.

// CTA 0, during the plan: add the window's counts (threads e < E).
__device__ __forceinline__ void tier_count(const TierDev& Tr, const SPlan& sp, int E) {
  const int tid = threadIdx.x;
  if (tid < E && sp.counts[tid] > 0) atomicAdd(Tr.counters + tid, (float)sp.counts[tid]);
  if (tid == 0) atomicAdd(reinterpret_cast<unsigned long long*>(Tr.windows), 1ull);
}

// All threads of one CTA: run the round that is due, if any.  scratch: four
// kMaxExperts-word arrays of shared memory nothing else uses meanwhile.
__device__ __noinline__ void tier_round_due(const TierDev& Tr, int E, uint8_t* scratch) {
  float* c = reinterpret_cast<float*>(scratch);
  int* res = reinterpret_cast<int*>(c + kMaxExperts);
  int* by_in = res + kMaxExperts;
  int* by_out = by_in + kMaxExperts;
  __shared__ int s_due;
  const int tid = threadIdx.x;
  if (tid == 0) {
    const long long w = *reinterpret_cast<volatile long long*>(Tr.windows);
    const long long r = *reinterpret_cast<volatile long long*>(Tr.rounds);
    s_due = (Tr.adapt_every > 0 && w / Tr.adapt_every > r) ? 1 : 0;
  }
  __syncthreads();
  if (!s_due) return;
  for (int e = tid; e < E; e += blockDim.x) {
    c[e] = __ldcg(Tr.counters + e);
    res[e] = __ldcg(Tr.resident + e);
  }
  __syncthreads();
  // ranks: four threads per expert, each counting a quarter of the others
  const int per = blockDim.x >> 2, q = tid & 3;
  const int iters = (E + per - 1) / per;
  for (int it = 0; it < iters; ++it) {
    const int e = it * per + (tid >> 2);
    const bool valid = (tid >> 2) < per && e < E;
    int rank = 0;
    if (valid) {
      const float ce = c[e];
      const int re = res[e];
      const int f0 = q * E / 4, f1 = (q + 1) * E / 4;
      for (int f = f0; f < f1; ++f) {
        if (res[f] != re) continue;
        const float cf = c[f];
        rank += re ? (cf < ce || (cf == ce && f < e)) : (cf > ce || (cf == ce && f < e));
      }
    }
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    rank += __shfl_xor_sync(0xffffffffu, rank, 2);
    if (valid && q == 0) (res[e] ? by_out : by_in)[rank] = e;
  }
  const int n_out = __syncthreads_count(tid < E && res[tid]);
  if (tid == 0) {
    const int n_in = E - n_out;
    const int lim = min(Tr.adapt_swaps, min(n_in, n_out));
    int n = 0;
    while (n < lim) {
      const float ca = c[by_in[n]], cb = c[by_out[n]];
      if (ca > cb && ca >= __fmul_rn(Tr.min_gain, cb)) ++n;
      else break;
    }
    for (int i = 0; i < n; ++i) {
      Tr.resident[by_in[i]] = 1;
      Tr.resident[by_out[i]] = 0;
      Tr.swap_in[i] = by_in[i];
      Tr.swap_out[i] = by_out[i];
    }
    *Tr.n_swaps = n;
    *Tr.rounds += 1;
  }
  for (int e = tid; e < E; e += blockDim.x) Tr.counters[e] = __fmul_rn(c[e], Tr.decay);
  __threadfence();
  __syncthreads();
}

// ---------------------------------------------------------------------------
// stage P: the routing plan (every CTA, same fixed-order arithmetic)
// ---------------------------------------------------------------------------
__device__ __noinline__ void compute_plan(const LayerDev& L, const WindowBufs& W, SPlan& sp) {
  const int T = W.T, E = L.E, k = L.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool pub = blockIdx.x == 0;
  // 1-2. row t (warp t): logits, top-k, softmax, gate weights
  if (warp < T) {
    if (E <= 32) plan_row<1>(L, W, sp, warp, lane, pub);
    else if (E <= 64) plan_row<2>(L, W, sp, warp, lane, pub);
    else if (E <= 128) plan_row<4>(L, W, sp, warp, lane, pub);
    else plan_row<8>(L, W, sp, warp, lane, pub);
  }
  __syncthreads();
  STAMP(0, 18);
  // 3. grouping: entries ordered by expert, then by entry index.  Warps 0 and 1
  //    hold entries 0..31 and 32..63; match_any gives each entry its rank among
  //    the same expert's entries of its warp and each warp's per-expert count.
  const int nent = T * k;
  const int n_me = warp * 32 + lane;
  const bool has_ent = warp < 2 && n_me < nent;
  const int e_me = has_ent ? sp.sel[n_me] : -1 - lane;  // distinct dummies never match
  int rank_me = 0;
  if (warp < 2) {
    const unsigned peers = __match_any_sync(0xffffffffu, e_me);
    rank_me = __popc(peers & ((1u << lane) - 1u));
    if (has_ent && rank_me == 0) sp.wcnt[warp][e_me] = __popc(peers);
  }
  __syncthreads();
  // counts (low 16 bits) and "used" flags (high 16 bits) scanned together
  const int e = tid;
  const int c = e < E ? sp.wcnt[0][e] + sp.wcnt[1][e] : 0;
  const int flag = c > 0 ? 1 : 0;
  int v = c | (flag << 16);
  if (tid < kMaxExperts) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) sp.wscan[warp] = v;
  }
  __syncthreads();
  if (e < E) {
    int before = 0;
#pragma unroll
    for (int w = 0; w < kMaxExperts / 32; ++w) before += w < warp ? sp.wscan[w] : 0;
    const int incl = v + before;
    const int off = (incl & 0xffff) - c, rank = (incl >> 16) - flag;
    sp.counts[e] = c;
    sp.offsets[e] = off;
    if (flag) sp.distinct[rank] = e;
    if (e == E - 1) sp.nd = incl >> 16;
    if (pub) {
      if (W.out_counts) W.out_counts[e] = c;
      if (W.out_offsets) W.out_offsets[e] = off;
      if (flag && W.out_distinct) W.out_distinct[rank] = e;
      if (e == E - 1) {
        if (W.out_offsets) W.out_offsets[E] = off + c;
        if (W.out_ndistinct) *W.out_ndistinct = incl >> 16;
      }
    }
  }
  __syncthreads();
  if (has_ent) {
    const int pos = sp.offsets[e_me] + (warp == 1 ? sp.wcnt[0][e_me] : 0) + rank_me;
    sp.entries[pos] = n_me;
    if (pub && W.out_entries) W.out_entries[pos] = n_me;
  }
  if (pub && W.tier.counters) tier_count(W.tier, sp, E);
}

struct Task {
  bool shared;
  int expert;
  int group;  // shared expert first (when present), then distinct experts ascending
  int tile;   // first row tile
};

__device__ __forceinline__ Task decode_task(int task, const PhaseTasks& pt, bool has_shared, const SPlan& sp) {
  Task t;
  if (task < pt.ntask_s) {
    t.shared = true;
    t.expert = -1;
    t.group = 0;
    t.tile = task * pt.mt;
  } else {
    const int q = task - pt.ntask_s;
    const int gi = q / pt.ntask_e;
    t.shared = false;
    t.expert = sp.distinct[gi];
    t.group = gi + (has_shared ? 1 : 0);
    t.tile = (q - gi * pt.ntask_e) * pt.mt;
  }
  return t;
}

// Estimated cost of one task of a group of R rows (groups of more than 4 rows
// take the two-set path: twice the MMAs and activation loads); a paired task
// costs 2, a two-set one two_set.
__device__ __forceinline__ int task_cost(int R, int two_set) { return R <= 4 ? 2 : two_set; }

// Contiguous task ranges of equal estimated cost (one warp): each lane takes a
// run of consecutive groups, a warp scan gives every group its starting cost
// position, and the lane whose groups hold a range boundary reports the task.
// group_cost: the estimated cost of staging a group's activations, in the
// same units, charged to the group's first task (measured per CTA on GB300:
// ~0.45 of a paired 4-bit task in both phases; small beside a 2-bit task).
__device__ __forceinline__ void split_tasks(const WindowBufs& W, SPlan& sp, bool has_shared, PhaseTasks& pt, int lane,
                                            int group_cost, int two_set) {
  const int hs = has_shared ? 1 : 0;
  const int ng = hs + sp.nd;
  const int ntotal = hs * pt.ntask_s + sp.nd * pt.ntask_e;
  const int per = (ng + 31) >> 5;
  const int g0 = lane * per;
  auto cost_of = [&](int g, int& nt, int& cst) {
    const bool sh = has_shared && g == 0;
    nt = sh ? pt.ntask_s : pt.ntask_e;
    cst = task_cost(sh ? W.T : sp.counts[sp.distinct[g - hs]], two_set);
  };
  int run = 0;
  for (int i = 0; i < per; ++i) {
    const int g = g0 + i;
    if (g < ng) {
      int nt, cst;
      cost_of(g, nt, cst);
      run += nt * cst + group_cost;
    }
  }
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int res[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int P = (int)((long long)total * (blockIdx.x + q) / gridDim.x);
    int found = -1, pos = incl - run;
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < ng) {
        int nt, cst;
        cost_of(g, nt, cst);
        const int len = nt * cst + group_cost;
        if (P >= pos && P < pos + len) {
          const int first = (g < hs) ? 0 : hs * pt.ntask_s + (g - hs) * pt.ntask_e;
          const int into = P - pos - group_cost;
          const int j = into <= 0 ? 0 : (into + cst - 1) / cst;
          found = first + (j < nt ? j : nt);
        }
        pos += len;
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, found >= 0);
    res[q] = bal ? __shfl_sync(0xffffffffu, found, __ffs(bal) - 1) : ntotal;
  }
  if (lane == 0) {
    pt.t0 = res[0];
    pt.t1 = res[1];
  }
  __syncwarp();
}

// Zero the sum slots of blocks nb .. 16 nmk - 1 (past the end of a K of nb
// blocks) in every column of a group of R rows (paired: 2R columns of one
// set; else R columns of both sets).
__device__ __forceinline__ void zero_padded_sums(__half* bs, const KernelCfg& C, int nb, int nmk, int R, bool paired,
                                                 int ctid) {
  const int npad = nmk * 16 - nb;
  if (npad <= 0) return;
  const int ncols = paired ? 2 * R : R;
  const __half z = __float2half_rn(0.f);
  for (int i = ctid; i < ncols * npad; i += kConsumerThreads) {
    const int col = i / npad, blk = nb + (i - col * npad);
    const int spos = frag_sum_pos(blk);
    const int mk = spos >> 4, c = (spos >> 2) & 3, slot = spos & 3;
    const int o = mk * 128 + col * 16 + c * 4 + slot;
    bs[o] = z;
    if (!paired) bs[C.bsum_halves + o] = z;
  }
}

// Copy a window's B image (global, set s of the main part at s * main_bytes,
// of the sums at s * sum_bytes) into B (all consumer threads): thread 0 issues
// one bulk copy per set and part, every thread waits (bounded) for them.  The
// image was written by other CTAs' generic stores before a grid barrier, and B
// last read by this CTA's generic loads before a consumer barrier: proxy
// fences order both before the bulk copies.
__device__ __forceinline__ void img_copy(SPlan& sp, __half* bm, __half* bs, int bmain_halves, int bsum_halves,
                                         const __half* main_src, uint32_t main_bytes, const __half* sum_src,
                                         uint32_t sum_bytes, int nsets, unsigned* err, long long wait_cycles, int ctid) {
  const uint32_t parity = sp.img_uses & 1u;
  if (ctid == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(&sp.img_bar, (uint32_t)nsets * (main_bytes + sum_bytes));
    for (int set = 0; set < nsets; ++set) {
      bulk_g2s(bm + set * bmain_halves, main_src + (size_t)set * (main_bytes / 2), main_bytes, &sp.img_bar);
      if (sum_bytes) bulk_g2s(bs + set * bsum_halves, sum_src + (size_t)set * (sum_bytes / 2), sum_bytes, &sp.img_bar);
    }
  }
  // bounded by wait_cycles alone (the copies are in flight; an abort elsewhere
  // does not stop them)
  if (!mbar_try_wait(&sp.img_bar, parity)) {
    const long long t0 = clock64();
    while (!mbar_try_wait(&sp.img_bar, parity)) {
      if (clock64() - t0 > wait_cycles) {
        atomicOr(err, kErrTimeout);
        break;
      }
    }
  }
  consumer_sync();  // every thread has seen this parity before the next copy flips it
  if (ctid == 0) sp.img_uses += 1;
}

// Stage one group's activations into shared memory (all consumer threads).
// Phases 0 and 2: copy x fragments (written by stage R or D0).  Phase 1: copy
// h fragments (written by the gate/up epilogue) and form the block sums from
// their 16-element partial sums.  The main-part copies are 16-byte cp.async
// pieces, all in flight before the one wait.  Phase 3 (the dense o
// projection) forms v's fragments here, since v is short.
template <int BITS, int PHASE>
__device__ void load_group_B(const LayerDev& L, const WindowBufs& W, SPlan& sp, const KernelCfg& C, __half* bm,
                             __half* bs, bool is_shared, int R, int ent_off, int K, int ctid) {
  constexpr int S = Fmt<BITS>::kBHalves;
  constexpr int B = Fmt<BITS>::kBlock;
  const int nks = K / Fmt<BITS>::kKstep;
  const int nmk = (K / B + 15) / 16;
  const bool paired = R <= 4;
  const int nsets = paired ? 1 : 2;
  const int ncols = paired ? 2 * R : R;
  if constexpr (PHASE == 0 || PHASE == 2) {
    // x fragments (the window's B image, K = d)
    TRACE(0, PHASE, 31, 0);
    const int T = W.T;
    if (PHASE == 2 || is_shared) {
      // all T rows in order: the image is this group's B as it stands, one
      // bulk copy per set of the main part and of the sums
      img_copy(sp, bm, bs, C.bmain_halves, C.bsum_halves, W.xfrag, 16u * K, W.xfrag + 16LL * K, 256u * nmk, nsets,
               W.err, W.wait_cycles, ctid);
      TRACE(0, PHASE, 31, 1);
    } else {
      // an expert's rows: each column's 16-byte pieces from its row's column
      // of the image
      const int per_col = nks * 4 * (S / 8);
      for (int i = ctid; i < nsets * ncols * per_col; i += kConsumerThreads) {
        const int cs = i / per_col, rem = i - cs * per_col;
        const int set = cs / ncols, col = cs - set * ncols;
        const int r = paired ? (col >> 1) : col;
        const int part = paired ? (col & 1) : set;
        const int ks = rem / (4 * (S / 8)), cp = rem - ks * 4 * (S / 8);
        const int c = cp / (S / 8), p = cp - c * (S / 8);
        const XImg q(T, sp.entries[ent_off + r] / L.k, part);
        cp_async16(bm + set * C.bmain_halves + bmain_off<BITS>(ks, p, col, c),
                   W.xfrag + (long long)q.set * 8 * K + bmain_off<BITS>(ks, p, q.col, c));
      }
      TRACE(0, PHASE, 31, 1);
      for (int i = ctid; i < nsets * ncols * nmk * 4; i += kConsumerThreads) {
        const int cs = i / (nmk * 4), rem = i - cs * nmk * 4;
        const int set = cs / ncols, col = cs - set * ncols;
        const int r = paired ? (col >> 1) : col;
        const int part = paired ? (col & 1) : set;
        const int mk = rem >> 2, c = rem & 3;
        const XImg q(T, sp.entries[ent_off + r] / L.k, part);
        const uint2 v = __ldcg(reinterpret_cast<const uint2*>(W.xfrag + 16LL * K + (long long)q.set * 128 * nmk +
                                                              (mk * 8 + q.col) * 16 + c * 4));
        *reinterpret_cast<uint2*>(bs + set * C.bsum_halves + (mk * 8 + col) * 16 + c * 4) = v;
      }
    }
    TRACE(0, PHASE, 31, 2);
    cp_async_wait_all();
    TRACE(0, PHASE, 31, 3);
  } else if constexpr (PHASE == 1) {
    // h fragments (one row of fragments per entry, or per row for the shared
    // expert), and the block sums formed from their 16-element partial sums
    auto row_base = [&](int r) -> const __half* {
      return is_shared ? W.shfrag + (long long)r * 2 * L.Fs : W.hfrag + (long long)sp.entries[ent_off + r] * 2 * L.F;
    };
    // main: 16-byte pieces (ks, c, plane) of each used column
    const int per_col = nks * 4 * (S / 8);
    for (int i = ctid; i < nsets * ncols * per_col; i += kConsumerThreads) {
      const int cs = i / per_col, rem = i - cs * per_col;
      const int set = cs / ncols, col = cs - set * ncols;
      const int r = paired ? (col >> 1) : col;
      const int part = paired ? (col & 1) : set;
      const int ks = rem / (4 * (S / 8)), cp = rem - ks * 4 * (S / 8);
      const int c = cp / (S / 8), p = cp - c * (S / 8);
      cp_async16(bm + set * C.bmain_halves + bmain_off<BITS>(ks, p, col, c),
                 row_base(r) + (long long)part * K + ks * 4 * S + c * S + p * 8);
    }
    // padded block slots of the last min group (blocks K/B .. 16 nmk - 1):
    // their min fragments are zero, but an earlier group may have left a
    // non-finite sum there (0 x NaN = NaN), so they are cleared for every
    // column this group uses
    zero_padded_sums(bs, C, K / B, nmk, R, paired, ctid);
    // block sums from the 16-element partial sums, split into hi/lo
    constexpr int kParts = B / 16;
    for (int i = ctid; i < R * (K / B); i += kConsumerThreads) {
      const int r = i / (K / B), blk = i - r * (K / B);
      const float* hs = is_shared ? W.shsum + (long long)r * (L.Fs / 16)
                                  : W.hsum + (long long)sp.entries[ent_off + r] * (L.F / 16);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kParts; ++j) sum += __ldcg(hs + blk * kParts + j);
      __half hi, lo;
      split_hi_lo(sum, hi, lo);
      const int spos = frag_sum_pos(blk);
      const int mk = spos >> 4, c = (spos >> 2) & 3, slot = spos & 3;
      const int o = mk * 128 + c * 4 + slot;
      if (paired) {
        bs[o + (2 * r) * 16] = hi;
        bs[o + (2 * r + 1) * 16] = lo;
      } else {
        bs[o + r * 16] = hi;
        bs[C.bsum_halves + o + r * 16] = lo;
      }
    }
    cp_async_wait_all();
    TRACE(0, PHASE, 31, 3);
  } else if (W.kv.k) {
    // the o projection's input is the cache attention's output: its main
    // fragments stay in global memory (kv_combine wrote them in this layout);
    // its block sums are split into hi/lo here (the padded sum slots were
    // cleared before the phase: dense_o_prologue)
    const int nb = L.dq / B;
    for (int i = ctid; i < R * nb; i += kConsumerThreads) {
      const int r = i / nb, blk = i - r * nb;
      __half hi, lo;
      split_hi_lo(__ldcg(W.kv.asum + (long long)r * nb + blk), hi, lo);
      const int spos = frag_sum_pos(blk);
      const int mk = spos >> 4, c = (spos >> 2) & 3, slot = spos & 3;
      const int o = mk * 128 + c * 4 + slot;
      if (paired) {
        bs[o + (2 * r) * 16] = hi;
        bs[o + (2 * r + 1) * 16] = lo;
      } else {
        bs[o + r * 16] = hi;
        bs[C.bsum_halves + o + r * 16] = lo;
      }
    }
  } else {
    // the length-one reading: v's fragments as the q/k/v epilogue left them
    // in the window's B image (K = dkv), and its block sums split into hi/lo,
    // each written for every block of the broadcast input that repeats that v
    // block (the padded sum slots were cleared before the phase:
    // dense_o_prologue)
    img_copy(sp, bm, nullptr, C.bmain_halves, 0, W.vimg, 16u * K, nullptr, 0u, nsets, W.err, W.wait_cycles, ctid);
    const int nbv = K / B;
    const int bph = (1 << L.kph_log2) * Fmt<BITS>::kBlocksPerKstep;
    const int ncopy = 1 << (L.kpg_log2 - L.kph_log2);
    for (int i = ctid; i < R * nbv; i += kConsumerThreads) {
      const int r = i / nbv, vb = i - r * nbv;
      __half hi, lo;
      split_hi_lo(__ldcg(W.vsum + (long long)r * nbv + vb), hi, lo);
      // v block vb = (kv group, block in head) -> broadcast blocks (group * G + head) * bph + j
      const int grp = vb / bph, j = vb - grp * bph;
      for (int hc = 0; hc < ncopy; ++hc) {
        const int spos = frag_sum_pos((grp * ncopy + hc) * bph + j);
        const int mk = spos >> 4, c = (spos >> 2) & 3, slot = spos & 3;
        const int o = mk * 128 + c * 4 + slot;
        if (paired) {
          bs[o + (2 * r) * 16] = hi;
          bs[o + (2 * r + 1) * 16] = lo;
        } else {
          bs[o + r * 16] = hi;
          bs[C.bsum_halves + o + r * 16] = lo;
        }
      }
    }
    cp_async_wait_all();
  }
}

// Ring state shared by the producer and the consumers.
struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  volatile int* abort_flag;
};

// Position in the stage ring: slot, parity of the current lap, slots passed.
struct RingPos {
  int stage = 0;
  uint32_t parity = 0;
  int n = 0;
  __device__ __forceinline__ void advance(int nstages) {
    ++n;
    if (++stage == nstages) {
      stage = 0;
      parity ^= 1u;
    }
  }
};

// Walks a CTA's contiguous task range without dividing: decode the first
// task once, then step through the groups' task lists.
struct TaskWalk {
  Task tk;
  int j;  // task index inside its group
  __device__ __forceinline__ void start(int task, const PhaseTasks& pt, bool has_shared, const SPlan& sp) {
    tk = decode_task(task, pt, has_shared, sp);
    j = tk.tile / pt.mt;
  }
  __device__ __forceinline__ void next(const PhaseTasks& pt, bool has_shared, const SPlan& sp) {
    ++j;
    if (tk.shared) {
      if (j == pt.ntask_s) {
        j = 0;
        tk.shared = false;
        tk.group = 1;
        tk.expert = sp.distinct[0];
      }
    } else if (j == pt.ntask_e) {
      j = 0;
      ++tk.group;
      const int gi = tk.group - (has_shared ? 1 : 0);
      tk.expert = gi < sp.nd ? sp.distinct[gi] : -1;
    }
    tk.tile = j * pt.mt;
  }
};

// ---------------------------------------------------------------------------
// producer: one thread streams every task's k-chunks, phase 0 then phase 1
// ---------------------------------------------------------------------------
// The packed matrix sub-tile s of a task reads (phase 0: kMT gate tiles, then
// kMT up tiles; the other phases: kMT tiles of one matrix): its base and the
// bytes of one expert's matrix.  Values, not references: a reference into the
// kernel's parameter struct would force a local copy of the whole struct.
struct MatRef {
  const uint8_t* base;
  long long mat_bytes;
};
__device__ __forceinline__ MatRef mat_ref(const PackedMat& M) { return MatRef{M.base, M.mat_bytes}; }

template <int PHASE, int kMT>
__device__ __forceinline__ MatRef task_mat(const LayerDev& L, bool shared, int s) {
  if constexpr (PHASE == 0) {
    const bool up = s >= kMT;
    const uint8_t* b = up ? (shared ? L.sup.base : L.up.base) : (shared ? L.sgate.base : L.gate.base);
    const long long mb = up ? (shared ? L.sup.mat_bytes : L.up.mat_bytes)
                            : (shared ? L.sgate.mat_bytes : L.gate.mat_bytes);
    return MatRef{b, mb};
  } else if constexpr (PHASE == 1) {
    return MatRef{shared ? L.sdown.base : L.down.base, shared ? L.sdown.mat_bytes : L.down.mat_bytes};
  } else if constexpr (PHASE == 2) {
    return mat_ref(L.qkv);
  } else {
    return mat_ref(L.o);
  }
}

template <int BITS, int PHASE>
__device__ __forceinline__ int task_k(const LayerDev& L, bool shared) {
  return PHASE == 0 ? L.d : PHASE == 1 ? (shared ? L.Fs : L.F) : PHASE == 2 ? L.d : L.dq;
}

template <int BITS>
__device__ __forceinline__ int tile_bytes_of(int K) {
  return (K / Fmt<BITS>::kKstep) * Fmt<BITS>::kChunk + ((K / Fmt<BITS>::kBlock + 15) / 16) * 512;
}

template <int BITS, int PHASE, int NS>
__device__ bool produce(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, const SPlan& sp, const Ring& rg,
                        RingPos& rp) {
  constexpr int kMT = PHASE == 0 ? NS / 2 : NS;
  const PhaseCfg& P = C.ph[PHASE];
  const PhaseTasks& pt = sp.pt[PHASE];
  const bool has_shared = L.Fs > 0;
  // the ring was last written through the generic proxy (staged router rows,
  // plan scratch): order that before the bulk copies
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  TaskWalk tw;
  if (pt.t0 < pt.t1) tw.start(pt.t0, pt, has_shared, sp);
  for (int task = pt.t0; task < pt.t1; ++task, tw.next(pt, has_shared, sp)) {
    const Task& tk = tw.tk;
    if (!tk.shared && (unsigned)tk.expert >= (unsigned)L.E) {
      atomicOr(W.err, kErrIndex);
      *rg.abort_flag = 1;
      return false;
    }
    const int K = task_k<BITS, PHASE>(L, tk.shared);
    const int nks = K / Fmt<BITS>::kKstep;
    const int tbytes = tile_bytes_of<BITS>(K);
    const int kv = (PHASE == 1 && tk.shared) ? 1 : 0;
    for (int ch = 0; ch < P.nchunks; ++ch) {
      const int ks0 = P.cks[kv][ch], ks1 = P.cks[kv][ch + 1];
      const int mk0 = P.cmk[kv][ch], mk1 = P.cmk[kv][ch + 1];
      const int stage = rp.stage;
      if (rp.n >= C.nstages && !wait_bar(&rg.empty[stage], rp.parity ^ 1u, W.err, rg.abort_flag, W.wait_cycles))
        return false;
      PTRACE(PHASE, (task - pt.t0) * P.nchunks + ch);
      const uint32_t cbytes = (uint32_t)((ks1 - ks0) * Fmt<BITS>::kChunk), mbytes = (uint32_t)((mk1 - mk0) * 512);
      uint8_t* dst = rg.base + (size_t)stage * C.stage_bytes;
      if (P.nchunks == 1 && tbytes == P.sub_stride) {
        // whole tiles, laid out in the stage as in memory: one copy per run
        // of consecutive tiles (phase 0: the gate run, then the up run)
        mbar_arrive_expect_tx(&rg.full[stage], NS * tbytes);
#pragma unroll
        for (int r = 0; r < (PHASE == 0 ? 2 : 1); ++r) {
          const MatRef M = task_mat<PHASE, kMT>(L, tk.shared, r * kMT);
          const uint8_t* src =
              M.base + (tk.shared ? 0LL : (long long)tk.expert * M.mat_bytes) + (long long)tk.tile * tbytes;
          bulk_g2s(dst + r * kMT * P.sub_stride, src, (uint32_t)(kMT * tbytes), &rg.full[stage]);
        }
        rp.advance(C.nstages);
        continue;
      }
      mbar_arrive_expect_tx(&rg.full[stage], NS * (cbytes + mbytes));
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const bool up = PHASE == 0 && s >= kMT;
        const MatRef M = task_mat<PHASE, kMT>(L, tk.shared, s);
        const int tile = tk.tile + (up ? s - kMT : s);
        const uint8_t* src =
            M.base + (tk.shared ? 0LL : (long long)tk.expert * M.mat_bytes) + (long long)tile * tbytes;
        uint8_t* dd = dst + s * P.sub_stride;
        if (cbytes) bulk_g2s(dd, src + (size_t)ks0 * Fmt<BITS>::kChunk, cbytes, &rg.full[stage]);
        if (mbytes) bulk_g2s(dd + P.mins_off, src + (size_t)nks * Fmt<BITS>::kChunk + mk0 * 512, mbytes, &rg.full[stage]);
      }
      rp.advance(C.nstages);
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// consumers: one phase's tasks (all 16 consumer warps)
// ---------------------------------------------------------------------------
// One output of a warp's partials (see partials): element idx, whose low
// bit is 0 in the paired layout.  Selects, not an indexed array, so the
// fragment stays in registers.
__device__ __forceinline__ float frag_pick(const float4 a, int idx, bool paired) {
  (void)paired;
  const float lo = (idx & 2) ? a.z : a.x, hi = (idx & 2) ? a.w : a.y;
  return (idx & 1) ? hi : lo;
}

// Group state of the consumer loop: rows of the current group and their MMA
// column layout (paired: 8 columns = 4 rows x (hi, lo); else two column sets).
struct GroupState {
  int cur = -2;
  int R = 0, ent_off = 0;
  bool paired = true, bon = true;
  int lane_b = 0;
  uint32_t inv_d = 0;  // ceil(2^16 / (16 R)): i / (16 R) == (i * inv_d) >> 16 for i < 512
};

// Enter task tk's group (all consumer threads): its rows, the bounded wait for
// its gate/up tasks (phase 1), and its activations staged in B.
template <int BITS, int PHASE>
__device__ __forceinline__ void enter_group(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, SPlan& sp,
                                            const Task& tk, int K, volatile int* abort_flag, __half* bm, __half* bs,
                                            GroupState& gs) {
  const int tid = threadIdx.x, lane = tid & 31, g = lane >> 2;
  if (tk.shared) {
    gs.R = W.T;
    gs.ent_off = 0;
  } else {
    gs.R = sp.counts[tk.expert];
    gs.ent_off = sp.offsets[tk.expert];
  }
  if (gs.R < 1 || gs.R > kMaxRows) {
    atomicOr(W.err, kErrIndex);
    gs.R = gs.R < 1 ? 1 : kMaxRows;
  }
  const int R = gs.R;
  gs.paired = R <= 4;
  gs.bon = gs.paired ? (g < 2 * R) : (g < R);
  gs.lane_b = gs.bon ? lane : (lane & 3);
  gs.inv_d = (65536u + 16u * R - 1u) / (16u * R);
  if (PHASE == 1) {
    // wait (bounded) until every gate/up task of this group has landed
    if (tid == 0) {
      const int need = tk.shared ? sp.pt[0].ntask_s : sp.pt[0].ntask_e;
      const long long t0 = clock64();
      while (!*abort_flag && ld_acquire(W.done_gu + tk.group) < need) {
        if (clock64() - t0 > W.wait_cycles) {
          atomicOr(W.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        __nanosleep(32);
      }
    }
    consumer_sync();
    if (gs.cur == -2) STAMP(0, 6);
  }
  // the previous task's barrier guarantees no warp still reads the old fragments
  load_group_B<BITS, PHASE>(L, W, sp, C, bm, bs, tk.shared, R, gs.ent_off, PHASE == 3 ? L.dkv : K, tid);
  consumer_sync();
  if (PHASE == 1 && gs.cur == -2) STAMP(0, 7);
  gs.cur = tk.group;
}

// The warps that share a task's outputs: in gate/up (phase 0) row tile m's
// gate and up sub-tiles, in the down phase one sub-tile.  On the warp-streamed
// path they meet after each task at their own named barrier (ids 2..5) and
// sum its partials among themselves, so the warps of other row tiles go on
// without waiting.  Warps of all groups still meet before a group's
// activations are restaged.  (The ring path keeps one barrier of all 16
// warps per task: there the groups gained nothing, and the decoder stack's
// dense phases lost time.)
template <int PHASE, int NS>
struct OutGroup {
  static constexpr int kWPS = kConsumerWarps / NS;
  static constexpr int kMT = PHASE == 0 ? NS / 2 : NS;
  static constexpr int kThreads = (PHASE == 0 ? 2 * kWPS : kWPS) * 32;
  int id;    // row tile (phase 0) or sub-tile
  int gtid;  // thread index inside the group
  __device__ __forceinline__ OutGroup(int sub, int kg, int lane) {
    id = PHASE == 0 ? sub % kMT : sub;
    gtid = (PHASE == 0 && sub >= kMT ? kWPS * 32 : 0) + kg * 32 + lane;
  }
  __device__ __forceinline__ void sync() const {
    asm volatile("bar.sync %0, %1;" ::"r"(2 + id), "n"(kThreads) : "memory");
  }
};

// One task's epilogue: the cross-warp sums of its partials (rb) in a fixed
// order for outputs i = i_first, i_first + stride, ... < i_end (output i is
// row r = (i mod 16R) / 16, element i mod 16 of sub-tile i / 16R).  Callers
// hand consecutive outputs to consecutive threads, starting at a warp that
// rotates with the task, so the other warps go straight on.
template <int BITS, int PHASE, int NS>
__device__ __forceinline__ void task_epilogue(const LayerDev& L, const WindowBufs& W, const SPlan& sp,
                                              const float4* rb, const Task& tk, const GroupState& gs, int i_first,
                                              int i_end, int stride) {
  constexpr int kMT = PHASE == 0 ? NS / 2 : NS;
  constexpr int kWPS = kConsumerWarps / NS;
  const int lane = threadIdx.x & 31;
  if (PHASE == 0) {
    for (int i = i_first; i < i_end; i += stride) {
      const int m = (int)(((uint32_t)i * gs.inv_d) >> 16), rem = i - m * 16 * gs.R;
      const int r = rem >> 4, row = rem & 15;
      const int src_lane = (row & 7) * 4 + (gs.paired ? r : (r >> 1));
      const int idx = ((row >> 3) << 1) + (gs.paired ? 0 : (r & 1));
      float gv = 0.f, uv = 0.f;
#pragma unroll
      for (int w = 0; w < kWPS; ++w) {
        gv += frag_pick(rb[(m * kWPS + w) * 32 + src_lane], idx, gs.paired);
        uv += frag_pick(rb[((kMT + m) * kWPS + w) * 32 + src_lane], idx, gs.paired);
      }
      // h = silu(gate) * up, stored as the down phase's activation fragments:
      // fp16 hi/lo parts at the element's fragment slot, and the sum of the 16
      // elements of this sub-tile (held by 16 consecutive lanes: i % 16 == row)
      const int f = (tk.tile + m) * 16 + row;
      const float h = silu_f32(gv) * uv;
      const int Kh = tk.shared ? L.Fs : L.F;
      const long long hrow = tk.shared ? r : sp.entries[gs.ent_off + r];
      __half* hb = (tk.shared ? W.shfrag : W.hfrag) + hrow * 2 * Kh;
      int off;
      float fac;
      frag_main_pos<BITS>(f, off, fac);
      __half hi, lo;
      split_hi_lo(h * fac, hi, lo);
      hb[off] = hi;
      hb[Kh + off] = lo;
      const unsigned half_mask = 0xffffu << (lane & 16);
      float ps = h;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) ps += __shfl_xor_sync(half_mask, ps, o);
      if (row == 0) (tk.shared ? W.shsum : W.hsum)[hrow * (Kh / 16) + f / 16] = ps;
    }
  } else {
    for (int i = i_first; i < i_end; i += stride) {
      const int s = (int)(((uint32_t)i * gs.inv_d) >> 16), rem = i - s * 16 * gs.R;
      const int r = rem >> 4, row = rem & 15;
      const int src_lane = (row & 7) * 4 + (gs.paired ? r : (r >> 1));
      const int idx = ((row >> 3) << 1) + (gs.paired ? 0 : (r & 1));
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWPS; ++w) v += frag_pick(rb[(s * kWPS + w) * 32 + src_lane], idx, gs.paired);
      const int drow = (tk.tile + s) * 16 + row;
      if constexpr (PHASE == 2) {
        // rows of [Wq; Wk; Wv] (q and k also kept for the cache attention)
        if (drow < L.dq) {
          if (W.q_out) W.q_out[(long long)r * L.dq + drow] = v;
          if (W.kv.qbuf) W.kv.qbuf[(long long)r * L.dq + drow] = v;
        } else if (drow < L.dq + L.dkv) {
          if (W.k_out) W.k_out[(long long)r * L.dkv + drow - L.dq] = v;
          if (W.kv.kbuf) W.kv.kbuf[(long long)r * L.dkv + drow - L.dq] = v;
        } else {
          const int f = drow - L.dq - L.dkv;
          W.v[(long long)r * L.dkv + f] = v;
          if (W.vimg && !W.kv.k) {
            // the length-one o phase's B operand: v's fragments in the
            // window's B image, and v's block sums (a 16-row tile holds half
            // a 4-bit block or one 2-bit block: at most two adds onto zero,
            // so the sum does not depend on their order)
            constexpr int B = Fmt<BITS>::kBlock;
            int off;
            float fac;
            frag_main_pos<BITS>(f, off, fac);
            __half hi, lo;
            split_hi_lo(v * fac, hi, lo);
            W.vimg[ximg_main<BITS>(W.T, L.dkv, r, 0, off)] = hi;
            W.vimg[ximg_main<BITS>(W.T, L.dkv, r, 1, off)] = lo;
            const unsigned half_mask = 0xffffu << (threadIdx.x & 16);
            float ps = v;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) ps += __shfl_xor_sync(half_mask, ps, o);
            if (row == 0) atomicAdd(W.vsum + (long long)r * (L.dkv / B) + f / B, ps);
            asm volatile("fence.proxy.async.global;" ::: "memory");  // the image is read by bulk copies
          }
        }
      } else if constexpr (PHASE == 3) {
        W.x1[(long long)r * L.d + drow] = W.x[(long long)r * L.d + drow] + v;
      } else if (tk.shared) {
        W.sbuf[(long long)r * L.d + drow] = v;
      } else {
        const int ent = sp.entries[gs.ent_off + r];
        W.obuf[(long long)ent * L.d + drow] = sp.topk_w[ent] * v;
      }
    }
  }
}

template <int BITS, int PHASE, int NS>
__device__ void consume(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, SPlan& sp, const Ring& rg,
                        __half* bm, __half* bs, float4* red, RingPos& rp, int& buf) {
  constexpr int kWPS = kConsumerWarps / NS;  // warps per sub-tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PhaseCfg& P = C.ph[PHASE];
  const PhaseTasks& pt = sp.pt[PHASE];
  const bool has_shared = L.Fs > 0;
  const int sub = warp / kWPS, kg = warp % kWPS;
  GroupState gs;
  TaskWalk tw;
  TRACE(0, PHASE, 30, 0);
  if (pt.t0 < pt.t1) tw.start(pt.t0, pt, has_shared, sp);
  for (int task = pt.t0; task < pt.t1; ++task, tw.next(pt, has_shared, sp)) {
    const Task& tk = tw.tk;
    if (!tk.shared && (unsigned)tk.expert >= (unsigned)L.E) break;  // flagged by the producer
    const int K = PHASE == 0 ? L.d : PHASE == 1 ? (tk.shared ? L.Fs : L.F) : PHASE == 2 ? L.d : L.dq;
    // the previous task's barrier guarantees no warp still reads the old activations
    if (tk.group != gs.cur) enter_group<BITS, PHASE>(L, W, C, sp, tk, K, rg.abort_flag, bm, bs, gs);
    const int kv = (PHASE == 1 && tk.shared) ? 1 : 0;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, accm[4] = {0.f, 0.f, 0.f, 0.f}, accm2[4] = {0.f, 0.f, 0.f, 0.f};
    TRACE(0, PHASE, task - pt.t0, 0);
    for (int ch = 0; ch < P.nchunks; ++ch) {
      const int ks0 = P.cks[kv][ch], ks1 = P.cks[kv][ch + 1];
      const int mk0 = P.cmk[kv][ch], mk1 = P.cmk[kv][ch + 1];
      const int nk = ks1 - ks0, nm = mk1 - mk0;
      const int k0 = (kg * nk) / kWPS, k1 = ((kg + 1) * nk) / kWPS;
      const int m0 = (kg * nm) / kWPS, m1 = ((kg + 1) * nm) / kWPS;
      const int stage = rp.stage;
      if (wait_bar(&rg.full[stage], rp.parity, W.err, rg.abort_flag, W.wait_cycles)) {
        if (ch == 0) TRACE(0, PHASE, task - pt.t0, 1);
        const uint8_t* st = rg.base + (size_t)stage * C.stage_bytes + sub * P.sub_stride;
        if (PHASE == 3 && !W.kv.k) {  // the length-one reading: v's fragments, k-steps remapped
          if (gs.paired)
            chunk_mma<BITS, true, true>(st, P.mins_off, ks0, k0, k1, mk0, m0, m1, bm, bs, C.bmain_halves,
                                        C.bsum_halves, gs.lane_b, lane, acc, accm, accm2, L.kph_log2,
                                        L.kpg_log2);
          else
            chunk_mma<BITS, false, true>(st, P.mins_off, ks0, k0, k1, mk0, m0, m1, bm, bs, C.bmain_halves,
                                         C.bsum_halves, gs.lane_b, lane, acc, accm, accm2, L.kph_log2,
                                         L.kpg_log2);
        } else {
          // (phase 3 with the cache attention: B is the attention output's
          // fragments in global memory, kv.afrag)
          const __half* bmx = PHASE == 3 ? W.kv.afrag : bm;
          const int bset = PHASE == 3 ? W.kv.afrag_set : C.bmain_halves;
          if (gs.paired)
            chunk_mma<BITS, true, false>(st, P.mins_off, ks0, k0, k1, mk0, m0, m1, bmx, bs, bset, C.bsum_halves,
                                         gs.lane_b, lane, acc, accm, accm2);
          else
            chunk_mma<BITS, false, false>(st, P.mins_off, ks0, k0, k1, mk0, m0, m1, bmx, bs, bset, C.bsum_halves,
                                          gs.lane_b, lane, acc, accm, accm2);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rg.empty[stage]);
      rp.advance(C.nstages);
    }
    TRACE(0, PHASE, task - pt.t0, 2);
    float4* rb = red + buf * (kConsumerWarps * 32);
    rb[warp * 32 + lane] = gs.paired ? partials<true>(acc, accm, accm2) : partials<false>(acc, accm, accm2);
    consumer_sync();  // all 16 warps: the ring path's warps stay in step
    TRACE(0, PHASE, task - pt.t0, 3);

    constexpr int kMT = PHASE == 0 ? NS / 2 : NS;
    task_epilogue<BITS, PHASE, NS>(L, W, sp, rb, tk, gs, (tid + 32 * (task & (kConsumerWarps - 1))) & (kConsumerThreads - 1),
                                   kMT * 16 * gs.R, kConsumerThreads);
    buf ^= 1;
  }
  TRACE(0, PHASE, 30, 1);
  if (PHASE == 0) {
    // publish this CTA's finished gate/up tasks: one fence, then per-group counts
    __threadfence();
    consumer_sync();
    for (int task = pt.t0 + tid; task < pt.t1; task += kConsumerThreads) {
      const Task tk = decode_task(task, pt, has_shared, sp);
      atomicAdd(W.done_gu + tk.group, 1);
    }
  }
}

// ---------------------------------------------------------------------------
// warp-streamed consumers (the window kernel): every warp copies its own share
// of each task into a private FIFO of shared-memory slots with 16-byte
// cp.async, kDepth items ahead; no producer warp and no CTA-wide stage ring
// ---------------------------------------------------------------------------
// FIFO depth in items per warp
template <int BITS> struct FifoDepth { static constexpr int value = 4; };

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A warp's items of one task of contraction length K: k-steps [k0, k0 + nk)
// then min groups [m0, m0 + n - nk) of its sub-tile.  An item is one k-step
// chunk (512 code bytes and the scale records, laid out as in the tile) or one
// 512-byte min fragment.  The copying side and the computing side of a warp
// both take the ranges from here, so they walk the same item sequence.
struct ItemRange {
  int k0, nk, m0, n;
};
template <int BITS, int NS>
__device__ __forceinline__ ItemRange item_range(int K, int kg) {
  constexpr int kWPS = kConsumerWarps / NS;
  const int nks = K / Fmt<BITS>::kKstep, nmk = (K / Fmt<BITS>::kBlock + 15) / 16;
  ItemRange r;
  r.k0 = kg * nks / kWPS;
  r.nk = (kg + 1) * nks / kWPS - r.k0;
  r.m0 = kg * nmk / kWPS;
  r.n = r.nk + (kg + 1) * nmk / kWPS - r.m0;
  return r;
}

template <int PHASE>
__device__ __forceinline__ int task_k(const LayerDev& L, const Task& tk) {
  return PHASE == 0 ? L.d : (tk.shared ? L.Fs : L.F);
}

// The copying side of a warp's item stream over its CTA's task range of one
// phase.  Every warp has at least one item in every task (the kernel is used
// only when each warp's k-range is non-empty); `set` checks this and, should
// it fail, flags the error word and stops the stream.
template <int BITS, int PHASE, int NS>
struct DStream {
  static constexpr int kMT = PHASE == 0 ? NS / 2 : NS;
  TaskWalk tw;
  int task, t1, i, n, nk;
  const uint8_t* kp;  // the next k-step chunk of the current task
  const uint8_t* mp;  // the next min fragment
  volatile int* abort_flag;

  __device__ __forceinline__ void set(const LayerDev& L, int sub, int kg, unsigned* err) {
    const Task& tk = tw.tk;
    if (!tk.shared && (unsigned)tk.expert >= (unsigned)L.E) {  // only with a corrupt plan
      atomicOr(err, kErrIndex);
      *abort_flag = 1;  // later waits give up at once
      task = t1;        // no further copies; the computing side stops at this task
      return;
    }
    const int K = task_k<PHASE>(L, tk);
    const ItemRange r = item_range<BITS, NS>(K, kg);
    if (r.n < 1) {
      // a warp with no item in this task would never reach the item that
      // moves its stream on, and would copy past the task's tile: stop
      // copying instead (the host's shape rule rules this out)
      atomicOr(err, kErrConfig);
      *abort_flag = 1;
      task = t1;
      return;
    }
    const int nks = K / Fmt<BITS>::kKstep, nmk = (K / Fmt<BITS>::kBlock + 15) / 16;
    const int tbytes = nks * Fmt<BITS>::kChunk + nmk * 512;
    const MatRef M = task_mat<PHASE, kMT>(L, tk.shared, sub);
    const int t = tk.tile + (PHASE == 0 && sub >= kMT ? sub - kMT : sub);
    const uint8_t* tile = M.base + (tk.shared ? 0LL : (long long)tk.expert * M.mat_bytes) + (long long)t * tbytes;
    kp = tile + (size_t)r.k0 * Fmt<BITS>::kChunk;
    mp = tile + (size_t)nks * Fmt<BITS>::kChunk + (size_t)r.m0 * 512;
    nk = r.nk;
    n = r.n;
    i = 0;
  }
  __device__ __forceinline__ void start(const LayerDev& L, const SPlan& sp, const PhaseTasks& pt, int sub, int kg,
                                        volatile int* abort, unsigned* err) {
    abort_flag = abort;
    task = pt.t0;
    t1 = pt.t1;
    if (task < t1) {
      tw.start(task, pt, L.Fs > 0, sp);
      set(L, sub, kg, err);
    }
  }
  // copy the next item into `dst` (this warp's slot; not waited for); past
  // the range's last item nothing is copied
  __device__ __forceinline__ void issue(uint8_t* dst, const LayerDev& L, const SPlan& sp, const PhaseTasks& pt,
                                        int sub, int kg, int lane, unsigned* err) {
    if (task >= t1) return;
    if (i < nk) {
      constexpr int kScaleBytes = Fmt<BITS>::kChunk - 512;
      cp_async16(dst + lane * 16, kp + lane * 16);
      if (lane * 16 < kScaleBytes) cp_async16(dst + 512 + lane * 16, kp + 512 + lane * 16);
      kp += Fmt<BITS>::kChunk;
    } else {
      cp_async16(dst + lane * 16, mp + lane * 16);
      mp += 512;
    }
    if (++i == n && ++task < t1) {
      tw.next(pt, L.Fs > 0, sp);
      set(L, sub, kg, err);
    }
  }
};

// One phase's tasks on the warp-streamed path (all 16 warps).  Warp w keeps
// kDepth items of its stream in flight in its FIFO slots (one cp.async group
// per item); items are consumed in order, across task and group boundaries,
// so a phase's first copies are in flight while its first group's
// activations are staged.  The computing side tracks its own place in each
// task's item range.  After an abort (a timed-out wait) the warps still walk
// every task, so that all of them meet every barrier; the results are then
// discarded by the caller through the error word.
template <int BITS, int PHASE, int NS>
__device__ void consume_direct(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, SPlan& sp,
                               volatile int* abort_flag, __half* bm, __half* bs, float4* red, uint8_t* fifo,
                               int& buf) {
  constexpr int kDepth = FifoDepth<BITS>::value;
  constexpr int kSlot = Fmt<BITS>::kChunk;
  constexpr int S = Fmt<BITS>::kBHalves;
  constexpr int kWPS = kConsumerWarps / NS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PhaseTasks& pt = sp.pt[PHASE];
  const bool has_shared = L.Fs > 0;
  const int sub = warp / kWPS, kg = warp % kWPS;
  if (pt.t0 < pt.t1) {
    uint8_t* const slots = fifo + (size_t)warp * kDepth * kSlot;
    uint8_t* const slots_end = slots + kDepth * kSlot;
    DStream<BITS, PHASE, NS> ds;
    ds.start(L, sp, pt, sub, kg, abort_flag, W.err);
#pragma unroll
    for (int q = 0; q < kDepth; ++q) {
      ds.issue(slots + q * kSlot, L, sp, pt, sub, kg, lane, W.err);
      cp_async_commit();
    }
    const OutGroup<PHASE, NS> og(sub, kg, lane);
    GroupState gs;
    TaskWalk tw;
    tw.start(pt.t0, pt, has_shared, sp);
    int task = pt.t0;
    uint8_t* it = slots;
    while (true) {
      const Task& tk = tw.tk;
      if (!tk.shared && (unsigned)tk.expert >= (unsigned)L.E) break;  // flagged by the copying side
      const int K = task_k<PHASE>(L, tk);
      if (tk.group != gs.cur) {
        consumer_sync();  // no warp still reads the previous group's activations
        enter_group<BITS, PHASE>(L, W, C, sp, tk, K, abort_flag, bm, bs, gs);
      }
      const ItemRange r = item_range<BITS, NS>(K, kg);
      TRACE(0, PHASE, task - pt.t0, 0);
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, accm[4] = {0.f, 0.f, 0.f, 0.f}, accm2[4] = {0.f, 0.f, 0.f, 0.f};
      const __half* bk = bm + r.k0 * 32 * S + gs.lane_b * 8;
      const __half* bsm = bs + r.m0 * 128 + gs.lane_b * 4;
      // refill the slot just used with the stream's next item, then move on
      auto next_slot = [&]() {
        __syncwarp();  // every lane is done with the slot before it is refilled
        ds.issue(it, L, sp, pt, sub, kg, lane, W.err);
        cp_async_commit();
        it += kSlot;
        if (it == slots_end) it = slots;
      };
      // k-steps first, then min groups; the item's copies are this lane's
      // oldest group in flight
      if (gs.paired) {
        for (int ci = 0; ci < r.nk; ++ci) {
          cp_async_wait_group<kDepth - 1>();
          __syncwarp();
          kstep_mma<BITS, true>(it, bk, C.bmain_halves, lane, acc);
          bk += 32 * S;
          next_slot();
        }
      } else {
        for (int ci = 0; ci < r.nk; ++ci) {
          cp_async_wait_group<kDepth - 1>();
          __syncwarp();
          kstep_mma<BITS, false>(it, bk, C.bmain_halves, lane, acc);
          bk += 32 * S;
          next_slot();
        }
      }
      for (int ci = r.nk; ci < r.n; ++ci) {
        cp_async_wait_group<kDepth - 1>();
        __syncwarp();
        const uint4 am = *reinterpret_cast<const uint4*>(it + lane * 16);
        const uint2 b = *reinterpret_cast<const uint2*>(bsm);
        mma16816(accm, am.x, am.y, am.z, am.w, b.x, b.y, accm);
        if (!gs.paired) {
          const uint2 l = *reinterpret_cast<const uint2*>(bsm + C.bsum_halves);
          mma16816(accm2, am.x, am.y, am.z, am.w, l.x, l.y, accm2);
        }
        bsm += 128;
        next_slot();
      }
      TRACE(0, PHASE, task - pt.t0, 2);
      float4* rb = red + buf * (kConsumerWarps * 32);
      rb[warp * 32 + lane] = gs.paired ? partials<true>(acc, accm, accm2) : partials<false>(acc, accm, accm2);
      og.sync();
      TRACE(0, PHASE, task - pt.t0, 3);
      {
        constexpr int kGT = OutGroup<PHASE, NS>::kThreads;
        const int i0 = og.id * 16 * gs.R;
        task_epilogue<BITS, PHASE, NS>(L, W, sp, rb, tk, gs, i0 + ((og.gtid + 32 * task) & (kGT - 1)),
                                       i0 + 16 * gs.R, kGT);
      }
      buf ^= 1;
      if (++task == pt.t1) break;
      tw.next(pt, has_shared, sp);
    }
    cp_async_wait_all();  // nothing of this phase may land in the FIFO later
    __syncwarp();
  }
  if (PHASE == 0) {
    // publish this CTA's finished gate/up tasks: one fence, then per-group counts
    __threadfence();
    consumer_sync();
    for (int task = pt.t0 + tid; task < pt.t1; task += kConsumerThreads) {
      const Task tk = decode_task(task, pt, has_shared, sp);
      atomicAdd(W.done_gu + tk.group, 1);
    }
  }
}

// Count this CTA's finished row slices of y; the CTA that completes a slice's
// count sums it in a fixed order (consumer threads).
template <int NS>
__device__ void combine(const LayerDev& L, const WindowBufs& W, SPlan& sp) {
  const int tid = threadIdx.x;
  const PhaseTasks& pt = sp.pt[1];
  const bool has_shared = L.Fs > 0;
  __threadfence();
  consumer_sync();
  if (tid == 0) sp.nfinish = 0;
  consumer_sync();
  const int ngroups = (has_shared ? 1 : 0) + sp.nd;
  const int ntiles = (pt.t1 - pt.t0) * NS;
  // y over 4 consecutive outputs of row t: shared expert first, then the
  // k weighted expert outputs in entry order (all loads issued up front)
  auto sum_quad = [&](int tile, int u) {
    const int t = u >> 2, rr = tile * 16 + (u & 3) * 4;
    float4 y = has_shared ? __ldcg(reinterpret_cast<const float4*>(W.sbuf + (long long)t * L.d + rr))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    if (W.resid) {
      const float4 x1 = __ldcg(reinterpret_cast<const float4*>(W.resid + (long long)t * L.d + rr));
      y.x += x1.x;
      y.y += x1.y;
      y.z += x1.z;
      y.w += x1.w;
    }
    float4 o[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      o[j] = j < L.k ? __ldcg(reinterpret_cast<const float4*>(W.obuf + (long long)(t * L.k + j) * L.d + rr))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < L.k) {
        y.x += o[j].x;
        y.y += o[j].y;
        y.z += o[j].z;
        y.w += o[j].w;
      }
    }
    *reinterpret_cast<float4*>(W.y + (long long)t * L.d + rr) = y;
  };
  for (int i = tid; i < ntiles; i += kConsumerThreads) {
    const Task tk = decode_task(pt.t0 + i / NS, pt, has_shared, sp);
    const int tile = tk.tile + i % NS;
    if (atomicAdd(W.counters + tile, 1) == ngroups - 1) {
      const int slot = atomicAdd(&sp.nfinish, 1);
      if (slot < kMaxEntries * 4) {
        sp.finish[slot] = tile;
      } else {  // list full: this thread sums the slice itself
        __threadfence();
        for (int u = 0; u < W.T * 4; ++u) sum_quad(tile, u);
      }
    }
  }
  consumer_sync();
  __threadfence();
  const int nf = min(sp.nfinish, kMaxEntries * 4);
  for (int i = tid; i < nf * W.T * 4; i += kConsumerThreads) sum_quad(sp.finish[i / (W.T * 4)], i % (W.T * 4));
}

// The combine for windows of kGridCombineRows rows or more, after a grid
// barrier that follows every CTA's down tasks: y = s + x1 + sum_j o[t k + j]
// (shared expert first, the residual if any, then the k weighted expert
// outputs in entry order), four outputs per thread, each CTA a contiguous
// range, every load issued before the sums.  Smaller windows keep the
// per-slice combine above: with few rows its tail is shorter than a barrier.
constexpr int kGridCombineRows = 4;

__device__ __noinline__ void combine_all(const LayerDev& L, const WindowBufs& W) {
  const int nq = W.T * (L.d / 4);
  const int q0 = (int)((long long)nq * blockIdx.x / gridDim.x), q1 = (int)((long long)nq * (blockIdx.x + 1) / gridDim.x);
  const bool has_shared = L.Fs > 0;
  for (int q = q0 + (int)threadIdx.x; q < q1; q += blockDim.x) {
    const int t = q / (L.d / 4), rr = (q - t * (L.d / 4)) * 4;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 y = has_shared ? __ldcg(reinterpret_cast<const float4*>(W.sbuf + (long long)t * L.d + rr)) : z;
    const float4 x1 = W.resid ? __ldcg(reinterpret_cast<const float4*>(W.resid + (long long)t * L.d + rr)) : z;
    float4 o[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      o[j] = j < L.k ? __ldcg(reinterpret_cast<const float4*>(W.obuf + (long long)(t * L.k + j) * L.d + rr)) : z;
    y.x += x1.x;
    y.y += x1.y;
    y.z += x1.z;
    y.w += x1.w;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < L.k) {
        y.x += o[j].x;
        y.y += o[j].y;
        y.z += o[j].z;
        y.w += o[j].w;
      }
    }
    *reinterpret_cast<float4*>(W.y + (long long)t * L.d + rr) = y;
  }
}

// The producer thread's drain after an abort: every copy it issued lands
// before the CTA may move on or exit.
__device__ __noinline__ void drain_ring(const Ring& rg, const KernelCfg& C, const RingPos& rp, long long limit) {
  const int it = rp.n;
  for (int j = (it > C.nstages ? it - C.nstages : 0); j < it; ++j) {
    const long long tw = clock64();
    while (!mbar_try_wait(&rg.full[j % C.nstages], (j / C.nstages) & 1)) {
      if (clock64() - tw > limit) break;
    }
  }
}

// Shared-memory carve-up common to both kernels.
struct Smem {
  uint8_t* ring;
  __half* bm;
  __half* bs;
  float4* red;
  uint64_t* full;
  uint64_t* empty;
};
__device__ __forceinline__ Smem carve(uint8_t* smem, const KernelCfg& C) {
  Smem m;
  m.ring = smem;
  m.bm = reinterpret_cast<__half*>(smem + (size_t)C.nstages * C.stage_bytes);
  m.bs = m.bm + (size_t)C.nsets * C.bmain_halves;
  m.red = reinterpret_cast<float4*>(m.bs + (size_t)C.nsets * C.bsum_halves);
  m.full = reinterpret_cast<uint64_t*>(m.red + 2 * kConsumerWarps * 32);
  m.empty = m.full + kMaxStages;
  return m;
}

__device__ __forceinline__ void init_cta(const KernelCfg& C, const Smem& m, volatile int* s_abort) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < C.nstages; ++s) {
      mbar_init(&m.full[s], 1);
      mbar_init(&m.empty[s], kConsumerWarps);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  // padded block-sum slots are never written: zero the sums region once
  for (int i = threadIdx.x; i < C.nsets * C.bsum_halves / 2; i += blockDim.x) reinterpret_cast<uint32_t*>(m.bs)[i] = 0u;
}

// After stage R and its grid barrier: the routing plan, gate/up and down of one
// MoE layer, and for windows of fewer than kGridCombineRows rows the per-slice
// combine (larger windows combine after a grid barrier, in the caller).
// Returns false when the plan is unusable (the error word says why); every
// CTA sees the same plan, so all return alike.
template <int BITS, bool DIRECT = false>
__device__ __forceinline__ bool moe_block(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, SPlan& sp,
                                          const Ring& rg, const Smem& m, RingPos& rp, int& buf) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // P: the routing plan (the ring is free until the producer starts: logits scratch)
  compute_plan(L, W, sp);
  STAMP(0, 3);
  const int nd = sp.nd;
  if (nd < 0 || nd > L.E) {
    if (tid == 0) atomicOr(W.err, kErrIndex);
    return false;
  }
  const bool has_shared = L.Fs > 0;
  // Task widths depend on the layer shape only, never on the window's
  // routing: a task's sub-tile count fixes how its K is split over the warps
  // (and so the order of a row's fp32 sums), and a row must get the same bits
  // whatever other rows share its window (the Strata docs, "BATCHING.md",
  // section "Exactness": a batch row's arithmetic is the single-token
  // window's).
  if (warp == 0) {
    // gate/up: 2 row tiles per task (the gate and up sub-tiles of each)
    PhaseTasks& p0 = sp.pt[0];
    const int tiles_e = L.F / 16, tiles_s = has_shared ? L.Fs / 16 : 0;
    p0.mt = (C.ph[0].max_sub >= 4 && tiles_e % 2 == 0 && tiles_s % 2 == 0) ? 2 : 1;
    p0.ntask_s = tiles_s / p0.mt;
    p0.ntask_e = tiles_e / p0.mt;
    split_tasks(W, sp, has_shared, p0, lane, BITS == 4 ? 2 : 0, 3);
  } else if (warp == 1) {
    // down: as many row tiles per task (up to 4) as the stage plan allows and
    // the d / 16 row tiles divide into (a down task is short, and its fixed
    // cost outweighs finer balance); the warp-streamed path's plan allows 4,
    // so every warp there has a k-step of each task
    PhaseTasks& p1 = sp.pt[1];
    const int tiles_g = L.d / 16;
    int mt = C.ph[1].max_sub;
    while (mt > 1 && tiles_g % mt != 0) mt >>= 1;
    p1.mt = mt;
    p1.ntask_s = has_shared ? tiles_g / mt : 0;
    p1.ntask_e = tiles_g / mt;
    // (a two-set down task costs ~1.9 paired ones on the ring path, ~1.5 on
    // the warp-streamed one: measured per CTA)
    split_tasks(W, sp, has_shared, p1, lane, BITS == 4 ? 2 : 0, DIRECT ? 3 : 4);
  }
  __syncthreads();
#ifdef STRATA_STAMPS
  if (tid == 0) {
    g_stamps[blockIdx.x][13] = (unsigned long long)(sp.pt[0].t1 - sp.pt[0].t0);
    g_stamps[blockIdx.x][14] = (unsigned long long)(sp.pt[1].t1 - sp.pt[1].t0);
    g_stamps[blockIdx.x][15] = (unsigned long long)(sp.pt[0].mt * 100 + sp.pt[1].mt);
  }
#endif
  STAMP(0, 4);

  const int ns0 = 2 * sp.pt[0].mt, ns1 = sp.pt[1].mt;
  if constexpr (DIRECT) {
    if (ns0 == 4) consume_direct<BITS, 0, 4>(L, W, C, sp, rg.abort_flag, m.bm, m.bs, m.red, m.ring, buf);
    else consume_direct<BITS, 0, 2>(L, W, C, sp, rg.abort_flag, m.bm, m.bs, m.red, m.ring, buf);
    STAMP(0, 5);
    const bool slices = W.T < kGridCombineRows;  // else the caller combines after a grid barrier
    if (ns1 == 4) {
      consume_direct<BITS, 1, 4>(L, W, C, sp, rg.abort_flag, m.bm, m.bs, m.red, m.ring, buf);
      STAMP(0, 8);
      if (slices) combine<4>(L, W, sp);
    } else {
      consume_direct<BITS, 1, 2>(L, W, C, sp, rg.abort_flag, m.bm, m.bs, m.red, m.ring, buf);
      STAMP(0, 8);
      if (slices) combine<2>(L, W, sp);
    }
    STAMP(0, 9);
    return true;
  }
  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const bool ok = ns0 == 4 ? produce<BITS, 0, 4>(L, W, C, sp, rg, rp) : produce<BITS, 0, 2>(L, W, C, sp, rg, rp);
      STAMP(kConsumerThreads, 11);
      if (ok) {
        if (ns1 == 4) produce<BITS, 1, 4>(L, W, C, sp, rg, rp);
        else if (ns1 == 2) produce<BITS, 1, 2>(L, W, C, sp, rg, rp);
        else produce<BITS, 1, 1>(L, W, C, sp, rg, rp);
      }
      STAMP(kConsumerThreads, 12);
      if (*rg.abort_flag) drain_ring(rg, C, rp, W.wait_cycles);
    }
    return true;
  }
  if (ns0 == 4) consume<BITS, 0, 4>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
  else consume<BITS, 0, 2>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
  STAMP(0, 5);
  const bool slices = W.T < kGridCombineRows;  // else the caller combines after a grid barrier
  if (ns1 == 4) {
    consume<BITS, 1, 4>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
    STAMP(0, 8);
    if (slices) combine<4>(L, W, sp);
  } else if (ns1 == 2) {
    consume<BITS, 1, 2>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
    STAMP(0, 8);
    if (slices) combine<2>(L, W, sp);
  } else {
    consume<BITS, 1, 1>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
    STAMP(0, 8);
    if (slices) combine<1>(L, W, sp);
  }
  STAMP(0, 9);
  return true;
}

// Before the dense o phase (all threads): its input is dq wide, and when dq /
// block is not a multiple of 16 the last min group has padded block slots
// whose min fragments are zero; an earlier phase may have left a non-finite
// sum there (0 x NaN = NaN), so they are cleared in every column of both
// sets.  The phase stages one group (all rows) and writes only real blocks,
// so they stay clear through it.  (Clearing them inside the staging itself
// slowed the stack's dense phases by a sixth.)
__device__ __noinline__ void dense_o_prologue(const LayerDev& L, const KernelCfg& C, __half* bs, int bits) {
  const int nb = L.dq / (bits == 4 ? 32 : 16), nmk = (nb + 15) / 16, npad = nmk * 16 - nb;
  if (npad <= 0) return;
  const __half z = __float2half_rn(0.f);
  for (int i = threadIdx.x; i < 16 * npad; i += blockDim.x) {
    const int col = i / npad, blk = nb + (i - col * npad);
    const int spos = frag_sum_pos(blk);
    const int o = (spos >> 4) * 128 + col * 16 + ((spos >> 2) & 3) * 4 + (spos & 3);
    bs[o] = z;
    bs[C.bsum_halves + o] = z;
  }
}

// One dense projection phase (2: [Wq; Wk; Wv] a, 3: x + Wo att) over all T
// rows, its row tiles split evenly over the CTAs.
template <int BITS, int PHASE>
__device__ __forceinline__ void dense_phase(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, SPlan& sp,
                                            const Ring& rg, const Smem& m, RingPos& rp, int& buf) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rows = PHASE == 2 ? L.dq + 2 * L.dkv : L.d;
  if (tid == 0) {
    PhaseTasks& p = sp.pt[PHASE];
    const int tiles = rows / 16;
    int mt = C.ph[PHASE].max_sub;
    while (mt > 1 && (tiles % mt != 0 || tiles / mt < 2 * (int)gridDim.x)) mt >>= 1;
    p.mt = mt;
    p.ntask_s = tiles / mt;
    p.ntask_e = 0;
    p.t0 = (int)((long long)p.ntask_s * blockIdx.x / gridDim.x);
    p.t1 = (int)((long long)p.ntask_s * (blockIdx.x + 1) / gridDim.x);
  }
  __syncthreads();
  const int ns = sp.pt[PHASE].mt;
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      if (ns == 4) produce<BITS, PHASE, 4>(L, W, C, sp, rg, rp);
      else if (ns == 2) produce<BITS, PHASE, 2>(L, W, C, sp, rg, rp);
      else produce<BITS, PHASE, 1>(L, W, C, sp, rg, rp);
      if (*rg.abort_flag) drain_ring(rg, C, rp, W.wait_cycles);
    }
    return;
  }
  if (ns == 4) consume<BITS, PHASE, 4>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
  else if (ns == 2) consume<BITS, PHASE, 2>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
  else consume<BITS, PHASE, 1>(L, W, C, sp, rg, m.bm, m.bs, m.red, rp, buf);
  TRACE(0, PHASE, 30, 2);
}

}  // namespace

// Shared memory: [ring: nstages x stage_bytes][B main: nsets][B sums: nsets]
// [red: 2 x 16 warps x 32 lanes float4][full/empty mbarriers]; static: SPlan.
template <int BITS>
__global__ void __launch_bounds__(kExpertThreads, 1) window_kernel(LayerDev L, WindowBufs W, KernelCfg C) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ SPlan sp;
  const Smem m = carve(smem, C);
  const Ring rg{m.ring, m.full, m.empty, &s_abort};
  init_cta(C, m, &s_abort);
  init_img(sp);
  for (int i = threadIdx.x; i < 2 * kMaxExperts; i += blockDim.x) (&sp.wcnt[0][0])[i] = 0;
  STAMP(0, 0);

  // R: router partial logits, x fragments; then every CTA waits for all
  router_stage<BITS>(L, W, reinterpret_cast<float*>(m.ring));
  STAMP(0, 1);
#ifdef STRATA_STAMPS
  __syncthreads();
  STAMP(0, 19);
#endif
  if (!grid_barrier_split(W, &sp.ok, blockIdx.x == 0 && W.tier.counters != nullptr,
                          [&] { tier_round_due(W.tier, L.E, m.ring + kTierScratchOff); }))
    return;  // timed out: the error word says so
  STAMP(0, 2);
  RingPos rp;
  int buf = 0;
  if (!moe_block<BITS>(L, W, C, sp, rg, m, rp, buf)) return;
  if (W.T >= kGridCombineRows) {
    if (!grid_barrier(W, &sp.ok) || s_abort) return;
    STAMP(0, 10);
    combine_all(L, W);
    STAMP(0, 16);
  }
}

// The window kernel on the register-fed path: 16 warps, no producer warp and
// no stage ring (the ring's place holds only stage R's staged rows of x).
template <int BITS>
__global__ void __launch_bounds__(kConsumerThreads, 1) window_kernel_direct(LayerDev L, WindowBufs W, KernelCfg C) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ SPlan sp;
  const Smem m = carve(smem, C);
  const Ring rg{m.ring, m.full, m.empty, &s_abort};
  init_cta(C, m, &s_abort);
  init_img(sp);
  for (int i = threadIdx.x; i < 2 * kMaxExperts; i += blockDim.x) (&sp.wcnt[0][0])[i] = 0;
  STAMP(0, 0);
  router_stage<BITS>(L, W, reinterpret_cast<float*>(m.ring));
  STAMP(0, 1);
  if (!grid_barrier_split(W, &sp.ok, blockIdx.x == 0 && W.tier.counters != nullptr,
                          [&] { tier_round_due(W.tier, L.E, m.ring + kTierScratchOff); }))
    return;  // timed out: the error word says so
  STAMP(0, 2);
  RingPos rp;
  int buf = 0;
  if (!moe_block<BITS, true>(L, W, C, sp, rg, m, rp, buf)) return;
  if (W.T >= kGridCombineRows) {
    if (!grid_barrier(W, &sp.ok) || s_abort) return;
    STAMP(0, 10);
    combine_all(L, W);
    STAMP(0, 16);
  }
}

// ---------------------------------------------------------------------------
// attention over each slot's KV cache (stack kernel)
// ---------------------------------------------------------------------------
// The Strata docs ("BATCHING.md", "Several requests at once (batch slots)")
// keep one KV cache per slot; a verify window carries one row per slot, plus
// the slot's MTP proposal as a second row at the next position.  Here a row t
// of slot s_t at position p_t stores its k and v (fp16) at p_t, and then
// attends, for query head h, over positions 0..p_t of its slot with kv head
// h / (heads / kv_heads): softmax_j(q_h . K_j / sqrt(head_dim)) applied to the
// V_j.  No position encoding (the pages name none).

__device__ __forceinline__ bool kv_row_ok(const KVDev& K, int t) {
  const int s = K.slot[t], p = K.pos[t];
  return s >= 0 && s < K.n_slots && p >= 0 && p < K.max_ctx;
}

__device__ __forceinline__ long long kv_base(const KVDev& K, int layer, int kvh, int slot, int g) {
  return (((long long)layer * K.n_slots + slot) * kvh + g) * K.max_ctx * K.head_dim;
}

// A0 (all CTAs): every row's k and v to position p_t of slot s_t, in fp16.
// A row whose slot or position is out of range is flagged and left out.
__device__ __noinline__ void kv_append(const LayerDev& L, const WindowBufs& W, int layer) {
  const KVDev& K = W.kv;
  const int hd = K.head_dim, kvh = L.dkv / hd;
  const int n = W.T * L.dkv;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int t = i / L.dkv, f = i - t * L.dkv, g = f / hd, e = f - g * hd;
    if (!kv_row_ok(K, t)) {
      if (f == 0) atomicOr(W.err, kErrIndex);
      continue;
    }
    const long long o = kv_base(K, layer, kvh, K.slot[t], g) + (long long)K.pos[t] * hd + e;
    K.k[o] = __float2half_rn(K.kbuf[(long long)t * L.dkv + f]);
    K.v[o] = __float2half_rn(W.v[(long long)t * L.dkv + f]);
  }
}

// The window's valid rows grouped by slot, in first-row order: each group's
// slot, row mask and largest position (every CTA computes the same).
struct SlotGroups {
  int n;
  int slot[kMaxRows];
  unsigned rows[kMaxRows];
  int pmax[kMaxRows];
};

__device__ void group_slots(const WindowBufs& W, SlotGroups& G) {
  const KVDev& K = W.kv;
  G.n = 0;
  for (int t = 0; t < W.T; ++t) {
    if (!kv_row_ok(K, t)) continue;
    const int s = K.slot[t], p = K.pos[t];
    int i = 0;
    while (i < G.n && G.slot[i] != s) ++i;
    if (i == G.n) {
      G.slot[i] = s;
      G.rows[i] = 0u;
      G.pmax[i] = p;
      ++G.n;
    }
    G.rows[i] |= 1u << t;
    G.pmax[i] = max(G.pmax[i], p);
  }
}

// A1: per-chunk partials.  An item is (slot group, kv head g, chunk c of
// kAttnChunk positions up to the group's largest position); it serves every
// row of the group, so the two rows of a slot read its cache once.  For each
// row r and query head h of kv head g: m = the largest score over the chunk's
// positions j <= p_r, l = sum exp(s_j - m), o = sum exp(s_j - m) V_j (fp32,
// fixed orders), written to kv.part.  Items are dealt out over the CTAs.
// smem: K and V chunk (fp16), the rows' q, the scores / weights.
__device__ __noinline__ void kv_partials(const LayerDev& L, const WindowBufs& W, int layer, uint8_t* smem) {
  const KVDev& K = W.kv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  const int hd = K.head_dim, kvh = L.dkv / hd, H = L.dq / hd, grp = H / kvh, dpl = hd / 32;
  constexpr int C = kAttnChunk;
  __shared__ SlotGroups G;
  __shared__ int s_rows[kMaxRows];
  if (tid == 0) group_slots(W, G);
  __syncthreads();
  __half* Ks = reinterpret_cast<__half*>(smem);
  __half* Vs = Ks + C * hd;
  float* qs = reinterpret_cast<float*>(Vs + C * hd);
  float* sc = qs + kMaxRows * grp * hd;
  const float scale = 1.0f / sqrtf((float)hd);
  int n_items = 0;
  for (int i = 0; i < G.n; ++i) n_items += kvh * ((G.pmax[i] + C) / C);
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    int i = 0, rem = item;
    while (rem >= kvh * ((G.pmax[i] + C) / C)) {
      rem -= kvh * ((G.pmax[i] + C) / C);
      ++i;
    }
    const int nch_i = (G.pmax[i] + C) / C;
    const int g = rem / nch_i, c = rem - g * nch_i;
    const int j0 = c * C, n = min(C, G.pmax[i] + 1 - j0);
    const unsigned rows = G.rows[i];
    const int R = __popc(rows);
    if (tid == 0) {
      int r = 0;
      for (int t = 0; t < W.T; ++t)
        if (rows & (1u << t)) s_rows[r++] = t;
    }
    // K and V of positions j0 .. j0 + n - 1 (contiguous for one slot and head)
    const long long base = kv_base(K, layer, kvh, G.slot[i], g) + (long long)j0 * hd;
    const int pieces = n * hd / 8;
    for (int q = tid; q < 2 * pieces; q += blockDim.x) {
      const bool isv = q >= pieces;
      const int qq = isv ? q - pieces : q;
      cp_async16((isv ? Vs : Ks) + qq * 8, (isv ? K.v : K.k) + base + qq * 8);
    }
    __syncthreads();  // s_rows
    for (int q = tid; q < R * grp * hd; q += blockDim.x) {
      const int pr = q / hd, e = q - pr * hd, r = pr / grp, hh = pr - r * grp;
      qs[q] = __ldcg(K.qbuf + (long long)s_rows[r] * L.dq + (g * grp + hh) * hd + e);
    }
    cp_async_wait_all();
    __syncthreads();
    // scores: warp per position, lanes over the head dimension
    for (int j = warp; j < n; j += nw) {
      float kk[4];
#pragma unroll
      for (int d = 0; d < 4; ++d) kk[d] = d < dpl ? __half2float(Ks[j * hd + lane * dpl + d]) : 0.f;
      for (int pr = 0; pr < R * grp; ++pr) {
        const float* qp = qs + pr * hd + lane * dpl;
        float v = 0.f;
#pragma unroll
        for (int d = 0; d < 4; ++d)
          if (d < dpl) v = fmaf(qp[d], kk[d], v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sc[pr * C + j] = v * scale;
      }
    }
    __syncthreads();
    // softmax statistics per (row, head) over the positions the row sees
    for (int pr = warp; pr < R * grp; pr += nw) {
      const int r = pr / grp, hh = pr - r * grp, t = s_rows[r];
      const int jmax = K.pos[t] - j0;  // positions j <= jmax are the row's
      float m = -INFINITY;
      for (int j = lane; j < n; j += 32)
        if (j <= jmax) m = fmaxf(m, sc[pr * C + j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float l = 0.f;
      for (int j = lane; j < n; j += 32) {
        const float w = (j <= jmax && m != -INFINITY) ? expf(sc[pr * C + j] - m) : 0.f;
        sc[pr * C + j] = w;
        l += w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) {
        float* pp = K.part + (((long long)t * H + g * grp + hh) * K.nch + c) * (hd + 2);
        pp[hd] = m;
        pp[hd + 1] = l;
      }
    }
    __syncthreads();
    // o = sum_j w_j V_j
    for (int q = tid; q < R * grp * hd; q += blockDim.x) {
      const int pr = q / hd, e = q - pr * hd, r = pr / grp, hh = pr - r * grp;
      float o = 0.f;
      for (int j = 0; j < n; ++j) o = fmaf(sc[pr * C + j], __half2float(Vs[j * hd + e]), o);
      K.part[(((long long)s_rows[r] * H + g * grp + hh) * K.nch + c) * (hd + 2) + e] = o;
    }
    __syncthreads();  // the chunk buffers are reused by the next item
  }
}

// A2: each row's attention output from its chunks' partials, written as the
// o projection's B operand (fp16 hi/lo fragments in the shared-memory B
// layout, kv.afrag) and per-block sums (kv.asum).  (row, head) pairs are dealt
// out over the CTAs; thread e < head_dim takes element e of the head.
template <int BITS>
__device__ __noinline__ void kv_combine(const LayerDev& L, const WindowBufs& W) {
  const KVDev& K = W.kv;
  constexpr int S = Fmt<BITS>::kBHalves, B = Fmt<BITS>::kBlock;
  const int tid = threadIdx.x, T = W.T, hd = K.head_dim, H = L.dq / hd;
  constexpr int C = kAttnChunk;
  const bool paired = T <= 4;
  for (int q = blockIdx.x; q < T * H; q += gridDim.x) {
    const int t = q / H, h = q - t * H;
    if (tid >= hd) continue;
    const int e = tid, f = h * hd + e;
    float a = 0.f;
    if (kv_row_ok(K, t)) {
      const int nc = (K.pos[t] + C) / C;
      const float* pp = K.part + ((long long)t * H + h) * K.nch * (hd + 2);
      float M = -INFINITY;
      for (int c = 0; c < nc; ++c) M = fmaxf(M, __ldcg(pp + c * (hd + 2) + hd));
      float lsum = 0.f, o = 0.f;
      for (int c = 0; c < nc; ++c) {
        const float mc = __ldcg(pp + c * (hd + 2) + hd);
        if (mc == -INFINITY) continue;
        const float w = expf(mc - M);
        lsum = fmaf(w, __ldcg(pp + c * (hd + 2) + hd + 1), lsum);
        o = fmaf(w, __ldcg(pp + c * (hd + 2) + e), o);
      }
      a = lsum > 0.f ? o / lsum : 0.f;
    }
    int off;
    float fac;
    frag_main_pos<BITS>(f, off, fac);
    const int ks = off / (4 * S), cq = (off / S) & 3, slot = off % S;
    __half hi, lo;
    split_hi_lo(a * fac, hi, lo);
    if (paired) {
      K.afrag[bmain_off<BITS>(ks, slot >> 3, 2 * t, cq) + (slot & 7)] = hi;
      K.afrag[bmain_off<BITS>(ks, slot >> 3, 2 * t + 1, cq) + (slot & 7)] = lo;
    } else {
      K.afrag[bmain_off<BITS>(ks, slot >> 3, t, cq) + (slot & 7)] = hi;
      K.afrag[K.afrag_set + bmain_off<BITS>(ks, slot >> 3, t, cq) + (slot & 7)] = lo;
    }
    // block sums: B consecutive elements of the head in B consecutive lanes
    float sm = a;
    const unsigned mask = B == 32 ? 0xffffffffu : (0xffffu << (tid & 16));
#pragma unroll
    for (int o = B / 2; o > 0; o >>= 1) sm += __shfl_xor_sync(mask, sm, o);
    if ((f % B) == 0) K.asum[(long long)t * (L.dq / B) + f / B] = sm;
  }
}

// A window through n decoder layers in one launch.  Per layer:
//   D0. every CTA: 1/RMS of each row of x; all CTAs write the fragments of
//       x / RMS(x);  grid barrier
//   D1. [q; k; v] = [Wq; Wk; Wv] a;  grid barrier
//   D2. x1 = x + Wo att, att = the grouped-query broadcast of v (a context of
//       one position: every query head's softmax weight is 1);  grid barrier
//   M.  the MoE window on x1 / RMS(x1) (stage R, grid barrier, plan, gate/up,
//       down), its combine adding x1;  grid barrier
// Layer l reads x from the previous layer's output (ping-pong buffers ybuf)
// and the last layer writes y.
template <int BITS>
__global__ void __launch_bounds__(kExpertThreads, 1)
    stack_kernel(const LayerDev* __restrict__ layers, int n_layers, WindowBufs Wp, KernelCfg C, const float* x_in,
                 float* y_out, float* ybuf, float* q_all, float* k_all) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ SPlan sp;
  __shared__ LayerDev sL;
  __shared__ WindowBufs sW;
  __shared__ float s_rinv[kMaxRows];
  const int tid = threadIdx.x;
  const Smem m = carve(smem, C);
  const Ring rg{m.ring, m.full, m.empty, &s_abort};
  init_cta(C, m, &s_abort);
  init_img(sp);
  RingPos rp;
  int buf = 0;
  for (int l = 0; l < n_layers; ++l) {
    if (tid == 0) {
      sL = layers[l];
      WindowBufs w = Wp;
      const long long plane = (long long)kMaxRows * sL.d;
      w.x = l == 0 ? x_in : ybuf + ((l - 1) & 1) * plane;
      w.y = l == n_layers - 1 ? y_out : ybuf + (l & 1) * plane;
      w.q_out = q_all ? q_all + (long long)l * Wp.T * sL.dq : nullptr;
      w.k_out = k_all ? k_all + (long long)l * Wp.T * sL.dkv : nullptr;
      w.rinv = s_rinv;
      w.resid = nullptr;
      const long long tk = (long long)l * Wp.T * sL.k;
      w.out_topk_idx = Wp.out_topk_idx ? Wp.out_topk_idx + tk : nullptr;
      w.out_topk_w = Wp.out_topk_w ? Wp.out_topk_w + tk : nullptr;
      w.out_ndistinct = Wp.out_ndistinct ? Wp.out_ndistinct + l : nullptr;
      w.out_counts = w.out_offsets = w.out_entries = w.out_distinct = nullptr;
      sW = w;
    }
    for (int i = tid; i < 2 * kMaxExperts; i += blockDim.x) (&sp.wcnt[0][0])[i] = 0;
    __syncthreads();
    STAMP(0, 20);
    const LayerDev& L = sL;
    // D0
    row_rinv(sW.x, sW.T, L.d, s_rinv);
    write_x_frags<BITS>(L, sW);
    if (blockIdx.x == 0 && sW.vimg && !sW.kv.k) {  // v's block sums start at zero (D1 adds into them)
      const int n = sW.T * (L.dkv / Fmt<BITS>::kBlock);
      for (int i = tid; i < n; i += blockDim.x) sW.vsum[i] = 0.f;
    }
    STAMP(0, 21);
    if (!grid_barrier(sW, &sp.ok)) return;
    STAMP(0, 22);
    // D1
    dense_phase<BITS, 2>(L, sW, C, sp, rg, m, rp, buf);
    STAMP(0, 23);
    if (!grid_barrier(sW, &sp.ok) || s_abort) return;
    STAMP(0, 24);
    if (sW.kv.k) {
      // A0-A2: attention over each slot's KV cache
      kv_append(L, sW, l);
      if (!grid_barrier(sW, &sp.ok)) return;
      kv_partials(L, sW, l, m.ring);
      if (!grid_barrier(sW, &sp.ok)) return;
      kv_combine<BITS>(L, sW);
      if (!grid_barrier(sW, &sp.ok)) return;
    }
    // D2
    dense_o_prologue(L, C, m.bs, BITS);
    dense_phase<BITS, 3>(L, sW, C, sp, rg, m, rp, buf);
    STAMP(0, 25);
    if (!grid_barrier(sW, &sp.ok) || s_abort) return;
    STAMP(0, 26);
    // M
    if (tid == 0) {
      sW.x = sW.x1;
      sW.resid = sW.x1;
    }
    __syncthreads();
    row_rinv(sW.x, sW.T, L.d, s_rinv);
    router_stage<BITS>(L, sW, reinterpret_cast<float*>(m.ring));
    STAMP(0, 27);
    if (!grid_barrier(sW, &sp.ok)) return;
    STAMP(0, 28);
    if (!moe_block<BITS>(L, sW, C, sp, rg, m, rp, buf)) return;
    if (sW.T >= kGridCombineRows) {
      if (!grid_barrier(sW, &sp.ok) || s_abort) return;
      STAMP(0, 29);
      combine_all(L, sW);
    }
    STAMP(0, 30);
    if (!grid_barrier(sW, &sp.ok) || s_abort) return;
    STAMP(0, 31);
  }
}

// ---------------------------------------------------------------------------
// the output head: logits = W_head RMSNorm(x) for the window's rows, each
// row's token (greedy or drawn), and each slot's proposal check
// ---------------------------------------------------------------------------

// Word 0 of Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011) for counter (pos, 0, 0, 0) and key
// (seed, 0): ten rounds of two 64 x 64 -> 128-bit products of words 0 and 2
// by the method's two multipliers, the new block (hi(M1 c2) ^ c1 ^ k0,
// lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)), and the key bumped by its two
// Weyl increments before every round but the first.
__device__ __noinline__ unsigned long long philox4x64_word0(unsigned long long pos, unsigned long long seed) {
  constexpr unsigned long long M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  constexpr unsigned long long W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
  unsigned long long c0 = pos, c1 = 0, c2 = 0, c3 = 0, k0 = seed, k1 = 0;
#pragma unroll 1
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += W0;
      k1 += W1;
    }
    const unsigned long long hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
    const unsigned long long hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  return c0;
}

// The row's uniform in [0, 1): the top 24 bits of the Philox word times 2^-24
// (exact in fp32).
__device__ __forceinline__ float row_uniform(unsigned long long pos, unsigned long long seed) {
  return (float)(philox4x64_word0(pos, seed) >> 40) * 5.9604644775390625e-8f;
}

// Argmax order: the larger value, then the lower token.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

// Probability weight of logit l in a row of maximum M at temperature tau.
__device__ __forceinline__ float draw_weight(float l, float M, float tau) {
  return expf(__fdiv_rn(__fsub_rn(l, M), tau));
}

// Inclusive prefix sums over the block's threads in thread order (warp
// Kogge-Stone scans, then the warp totals added one after another by thread
// 0), each thread's result also left in s_incl[tid]; the same arithmetic every
// time it runs on the same values.  s_w: one float per warp.
__device__ float block_incl_scan(float v, float* s_incl, float* s_w) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = __fadd_rn(v, n);
  }
  if (lane == 31) s_w[warp] = v;
  __syncthreads();
  if (tid == 0) {
    float run = 0.f;
    for (int w = 0; w < nw; ++w) {
      const float tw = s_w[w];
      s_w[w] = run;
      run = __fadd_rn(run, tw);
    }
  }
  __syncthreads();
  const float incl = warp ? __fadd_rn(s_w[warp], v) : v;
  s_incl[tid] = incl;
  __syncthreads();
  return incl;
}

// This thread's chunk of the CTA's vocabulary slice [v0, v1).
__device__ __forceinline__ void chunk_of(int v0, int v1, int& a, int& b) {
  const long long n = v1 - v0;
  a = v0 + (int)(n * threadIdx.x / blockDim.x);
  b = v0 + (int)(n * (threadIdx.x + 1) / blockDim.x);
}

// Sequential sum of the weights of this thread's chunk of row t.
__device__ __forceinline__ float chunk_weight(const float* lg, int a, int b, float M, float tau) {
  float s = 0.f;
  for (int v = a; v < b; ++v) s = __fadd_rn(s, draw_weight(__ldcg(lg + v), M, tau));
  return s;
}

// The slices' weight sums of row t in slice (CTA) order, one running fp32
// sum: warp t loads the G sums into shared memory (all lanes, one round trip),
// then lane 0 adds them one after another; the total goes to every lane.  The
// chain is the same arithmetic wherever it runs, so every CTA gets the same
// total and the same slice boundaries.
__device__ __forceinline__ float slice_total(const float* part_sum, int t, int G, float* s_row, int lane) {
  for (int q = lane; q < G; q += 32) s_row[q] = __ldcg(part_sum + q * kMaxRows + t);
  __syncwarp();
  float Z = 0.f;
  if (lane == 0) {
#pragma unroll 8
    for (int q = 0; q < G; ++q) Z = __fadd_rn(Z, s_row[q]);
  }
  return __shfl_sync(0xffffffffu, Z, 0);
}

// The token of every row from the logits [T][V] (all CTAs; ends with CTA 0
// writing tokens and the slots' emitted counts).
//   greedy rows (temperature <= 0): the argmax, ties to the lower token;
//   sampled rows: u from Philox4x64-10(seed, position); the first token whose
//   cumulative softmax(logits / temperature) weight exceeds u times the total,
//   the vocabulary summed slice by slice (CTA order), each slice chunk by
//   chunk (thread order) and each chunk token by token; should rounding leave
//   no token above it, the greedy token.
//   proposal check: a slot's first row (fed < 0) emits its token; each next
//   row of the slot adds its token while the previous row's token equals the
//   proposal the row was fed.
__device__ __noinline__ bool head_select(const WindowBufs& W, const HeadArgs& H, const float* logits, int* s_ok,
                                         uint8_t* scratch) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = W.T, V = H.V, G = gridDim.x, c = blockIdx.x;
  float* s_bv = reinterpret_cast<float*>(scratch);               // [2][8]
  int* s_bi = reinterpret_cast<int*>(s_bv + 2 * kMaxRows);         // [2][8]
  float* s_M = reinterpret_cast<float*>(s_bi + 2 * kMaxRows);      // [8]
  float* s_tgt = s_M + kMaxRows;                                   // [8] target within the chosen slice
  int* s_cs = reinterpret_cast<int*>(s_tgt + kMaxRows);            // [8] the chosen slice
  float* s_w = reinterpret_cast<float*>(s_cs + kMaxRows);          // [32]
  float* s_incl = s_w + 32;                                        // [blockDim]
  int* s_any = reinterpret_cast<int*>(s_incl + blockDim.x);
  float* s_ps = reinterpret_cast<float*>(s_any + 4);               // [8][G] the slices' sums of each row
  int v0, v1;
  {
    v0 = (int)((long long)V * c / G);
    v1 = (int)((long long)V * (c + 1) / G);
  }
  if (tid == 0) {
    int any = 0;
    for (int t = 0; t < T; ++t) any |= H.temperature[t] > 0.f ? 1 : 0;
    *s_any = any;
  }
  // A: this slice's maximum and its token, per row (warp w: row w % 8, half w / 8)
  if (warp < 2 * kMaxRows) {
    const int t = warp & 7, h = warp >> 3;
    if (t < T) {
      const int mid = v0 + (v1 - v0) / 2, lo = h ? mid : v0, hi = h ? v1 : mid;
      const float* lg = logits + (long long)t * V;
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      bool fin = true;
      for (int vb = lo; vb < hi; vb += 8 * 32) {  // eight loads in flight per lane
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = vb + u * 32 + lane;
          x[u] = v < hi ? __ldcg(lg + v) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = vb + u * 32 + lane;
          if (v < hi) {
            fin &= isfinite(x[u]);
            if (x[u] > bv) {
              bv = x[u];
              bi = v;
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (!__all_sync(0xffffffffu, fin) && lane == 0) atomicOr(W.err, kErrNonFinite);
      if (lane == 0) {
        s_bv[h * kMaxRows + t] = bv;
        s_bi[h * kMaxRows + t] = bi;
      }
    }
  }
  __syncthreads();
  if (tid < T) {
    float bv = s_bv[tid];
    int bi = s_bi[tid];
    if (better(s_bv[kMaxRows + tid], s_bi[kMaxRows + tid], bv, bi)) {
      bv = s_bv[kMaxRows + tid];
      bi = s_bi[kMaxRows + tid];
    }
    H.part_max[c * kMaxRows + tid] = bv;
    H.part_arg[c * kMaxRows + tid] = bi;
  }
  const bool sampled = *s_any != 0;
  if (!grid_barrier(W, s_ok)) return false;
  if (sampled) {
    // B: every CTA takes each row's maximum; this slice's sum of weights
    if (warp < T) {  // each row's maximum over the slices (warp t)
      float M = -INFINITY;
      for (int q = lane; q < G; q += 32) M = fmaxf(M, __ldcg(H.part_max + q * kMaxRows + warp));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      if (lane == 0) s_M[warp] = M;
    }
    __syncthreads();
    int a, b;
    chunk_of(v0, v1, a, b);
    for (int t = 0; t < T; ++t) {
      const float tau = H.temperature[t];
      if (!(tau > 0.f)) continue;
      const float incl = block_incl_scan(chunk_weight(logits + (long long)t * V, a, b, s_M[t], tau), s_incl, s_w);
      if (tid == blockDim.x - 1) H.part_sum[c * kMaxRows + t] = incl;
    }
    if (!grid_barrier(W, s_ok)) return false;
    // C: every CTA finds each sampled row's slice: the first whose running
    // total passes u x (the total); that CTA finds the token inside it
    if (warp < T) {  // row t = warp
      int cs = -1;
      float tl = 0.f;
      if (H.temperature[warp] > 0.f) {
        float* s_row = s_ps + warp * G;
        const float Z = slice_total(H.part_sum, warp, G, s_row, lane);
        if (lane == 0) {
          const float tgt = __fmul_rn(row_uniform((unsigned long long)(long long)H.position[warp], H.seed[warp]), Z);
          float P = 0.f;
          for (int q = 0; q < G; ++q) {
            const float Pn = __fadd_rn(P, s_row[q]);
            if (Pn > tgt) {
              cs = q;
              tl = __fsub_rn(tgt, P);
              break;
            }
            P = Pn;
          }
        }
      }
      if (lane == 0) {
        s_cs[warp] = cs;
        s_tgt[warp] = tl;
      }
    }
    __syncthreads();
    for (int t = 0; t < T; ++t) {
      if (s_cs[t] != c) continue;
      const float tau = H.temperature[t], M = s_M[t], tl = s_tgt[t];
      const float* lg = logits + (long long)t * V;
      const float incl = block_incl_scan(chunk_weight(lg, a, b, M, tau), s_incl, s_w);
      const float excl = tid ? s_incl[tid - 1] : 0.f;
      const float total = s_incl[blockDim.x - 1];
      if (tl >= total) {
        if (tid == 0) H.tokens[t] = v1 - 1;  // rounding: the slice's last token
      } else if (excl <= tl && tl < incl) {
        int tok = b - 1;
        float run = 0.f;
        for (int v = a; v < b; ++v) {
          run = __fadd_rn(run, draw_weight(__ldcg(lg + v), M, tau));
          if (__fadd_rn(excl, run) > tl) {
            tok = v;
            break;
          }
        }
        H.tokens[t] = tok;
      }
      __syncthreads();
    }
    if (!grid_barrier(W, s_ok)) return false;
  } else if (!grid_barrier(W, s_ok)) {
    return false;
  }
  // final: CTA 0 writes the greedy tokens (and a sampled row's when no slice
  // passed its target), then each slot's emitted count
  if (c != 0) return true;
  if (warp < T) {  // row t = warp
    const bool greedy = !(H.temperature[warp] > 0.f);
    bool need = greedy;
    if (!greedy) {
      const float Z = slice_total(H.part_sum, warp, G, s_ps + warp * G, lane);
      const float tgt = __fmul_rn(row_uniform((unsigned long long)(long long)H.position[warp], H.seed[warp]), Z);
      need = !(Z > tgt);
    }
    if (need) {  // the argmax over the slices' maxima (ties to the lower token: any order gives the same)
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int q = lane; q < G; q += 32) {
        const float v = __ldcg(H.part_max + q * kMaxRows + warp);
        const int i = __ldcg(H.part_arg + q * kMaxRows + warp);
        if (better(v, i, bv, bi)) {
          bv = v;
          bi = i;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (lane == 0) H.tokens[warp] = (bi >= 0 && bi < V) ? bi : 0;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    int start = 0, emit = 1;
    bool ok = true;
    for (int t = 1; t < T; ++t) {
      if (H.fed[t] < 0) {  // a new slot
        H.n_emit[start] = emit;
        start = t;
        emit = 1;
        ok = true;
      } else {
        if (ok && __ldcg(H.tokens + t - 1) == H.fed[t]) ++emit;
        else ok = false;
        H.n_emit[t] = 0;
      }
    }
    H.n_emit[start] = emit;
  }
  return true;
}

// The head of a window: D0 (1/RMS of each row, the fragments of x / RMS(x);
// grid barrier), the head GEMV as the dense phase over the V rows of the head
// matrix (logits to W.q_out; grid barrier), then head_select.
template <int BITS>
__global__ void __launch_bounds__(kExpertThreads, 1) head_kernel(LayerDev L, WindowBufs Wp, KernelCfg C, HeadArgs H) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ SPlan sp;
  __shared__ WindowBufs sW;
  __shared__ float s_rinv[kMaxRows];
  const Smem m = carve(smem, C);
  const Ring rg{m.ring, m.full, m.empty, &s_abort};
  init_cta(C, m, &s_abort);
  init_img(sp);
  if (threadIdx.x == 0) {
    sW = Wp;
    sW.rinv = s_rinv;
  }
  __syncthreads();
  STAMP(0, 0);
  row_rinv(sW.x, sW.T, L.d, s_rinv);
  write_x_frags<BITS>(L, sW);
  STAMP(0, 1);
  if (!grid_barrier(sW, &sp.ok)) return;
  STAMP(0, 2);
  RingPos rp;
  int buf = 0;
  dense_phase<BITS, 2>(L, sW, C, sp, rg, m, rp, buf);
  STAMP(0, 3);
  if (!grid_barrier(sW, &sp.ok) || s_abort) return;
  STAMP(0, 4);
  head_select(sW, H, sW.q_out, &sp.ok, m.ring);
  STAMP(0, 5);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Cut one phase's tiles into ring stages: the task width (sub-tiles 4, 2 or 1;
// gate/up need >= 2) and the fewest k-chunks per tile that fit the stage
// budget, scored by k-steps per warp per chunk (each chunk costs one wait and
// one release per warp).
static PhaseCfg phase_cfg(int phase, int bits, int Kv0, int Kv1, int stage_budget, int& stage_bytes, int ns_only = 0) {
  const int kstep = bits == 4 ? 64 : 128, block = bits == 4 ? 32 : 16, chunk = bits == 4 ? 576 : 768;
  const int Kmax = Kv0 > Kv1 ? Kv0 : Kv1;
  const int nks = Kmax / kstep, nmk = (Kmax / block + 15) / 16;
  const int ns_min = phase == 0 ? 2 : 1;
  PhaseCfg best{};
  int best_score = -1;
  stage_bytes = 0;
  for (int ns = kMaxSub; ns >= ns_min; ns >>= 1) {
    if (ns_only && ns != ns_only) continue;
    const int wps = kConsumerWarps / ns;
    for (int nc = 1; nc <= nks && nc <= kMaxChunks; ++nc) {
      const int cks = (nks + nc - 1) / nc, cmk = (nmk + nc - 1) / nc;
      const int sub_stride = cks * chunk + cmk * 512;
      if (ns * sub_stride > stage_budget) continue;
      const int per_warp = (nks / nc) / wps;
      const int score = (per_warp > 8 ? 8 : per_warp) * 1000 + ns * 100;
      if (score > best_score) {
        best_score = score;
        best.nchunks = nc;
        best.sub_stride = sub_stride;
        best.mins_off = cks * chunk;
        best.max_sub = ns;
        stage_bytes = ns * sub_stride;
      }
      break;
    }
  }
  if (best_score < 0) {  // even one k-step per chunk does not fit: smallest possible stage
    best.nchunks = nks < kMaxChunks ? nks : kMaxChunks;
    const int cks = (nks + best.nchunks - 1) / best.nchunks, cmk = (nmk + best.nchunks - 1) / best.nchunks;
    best.sub_stride = cks * chunk + cmk * 512;
    best.mins_off = cks * chunk;
    best.max_sub = ns_only ? ns_only : ns_min;
    stage_bytes = best.max_sub * best.sub_stride;
  }
  for (int v = 0; v < 2; ++v) {
    const int K = v == 0 ? Kv0 : Kv1;
    const int nks_v = K / kstep, nmk_v = (K / block + 15) / 16;
    for (int ch = 0; ch <= best.nchunks; ++ch) {
      best.cks[v][ch] = (short)(ch * nks_v / best.nchunks);
      best.cmk[v][ch] = (short)(ch * nmk_v / best.nchunks);
    }
  }
  return best;
}

// The task width (row tiles per task) of a dense phase over `tiles` row
// tiles on `grid` CTAs: the widest of 4, 2, 1 that divides the tiles and
// still gives every CTA two tasks -- the rule dense_phase applies.
static int dense_width(int tiles, int grid) {
  int mt = kMaxSub;
  while (mt > 1 && (tiles % mt != 0 || tiles / mt < 2 * grid)) mt >>= 1;
  return mt;
}

KernelCfg window_cfg(const LayerDev& L, int max_rows, int smem_limit, int grid) {
  KernelCfg C{};
  const int bits = L.bits;
  const int block = bits == 4 ? 32 : 16;
  // B main holds the widest activation vector a phase stages (the dense o
  // projection stages v and remaps k-steps); B sums cover the widest input
  int Kmax = L.d > (L.F > L.Fs ? L.F : L.Fs) ? L.d : (L.F > L.Fs ? L.F : L.Fs);
  if (L.dkv > Kmax) Kmax = L.dkv;
  const int Ksum = L.dq > Kmax ? L.dq : Kmax;
  const int nmk = (Ksum / block + 15) / 16;
  C.bmain_halves = 8 * Kmax;
  C.bsum_halves = nmk * 8 * 4 * 4;
  C.nsets = max_rows > 4 ? 2 : 1;
  const int fixed = C.nsets * (C.bmain_halves + C.bsum_halves) * 2 + 2 * kConsumerWarps * 32 * 16 + 2 * kMaxStages * 8;
  const int ring = smem_limit - fixed;
  const int budget = ring / 3;  // at least three stages in flight
  int sb0 = 0, sb1 = 0;
  C.ph[0] = phase_cfg(0, bits, L.d, L.d, budget, sb0);
  C.ph[1] = phase_cfg(1, bits, L.F, L.Fs > 0 ? L.Fs : L.F, budget, sb1);
  C.stage_bytes = sb0 > sb1 ? sb0 : sb1;
  if (L.dq > 0) {
    // decoder layer: the dense q/k/v and o phases, cut into chunks for the
    // task width they run at on this grid (a chunking made for 4-tile tasks
    // leaves a 1-tile task with a quarter-full stage and more waits)
    int sb2 = 0, sb3 = 0;
    const int w2 = grid > 0 ? dense_width((L.dq + 2 * L.dkv) / 16, grid) : 0;
    const int w3 = grid > 0 ? dense_width(L.d / 16, grid) : 0;
    C.ph[2] = phase_cfg(1, bits, L.d, L.d, budget, sb2, w2);
    C.ph[3] = phase_cfg(1, bits, L.dq, L.dq, budget, sb3, w3);
    if (sb2 > C.stage_bytes) C.stage_bytes = sb2;
    if (sb3 > C.stage_bytes) C.stage_bytes = sb3;
  }
  int st = C.stage_bytes > 0 ? ring / C.stage_bytes : 0;
  C.nstages = st > kMaxStages ? kMaxStages : st;
  C.total_bytes = C.nstages * C.stage_bytes + fixed;
  C.direct = 0;
  return C;
}

// The window kernel's register-fed configuration: no stage ring, only stage
// R's staged rows of x in its place.  Usable when every warp gets at least one
// k-step of every task (phase 0: K = d over up to 8 warps; phase 1: K = F or
// Fs over up to 8 warps) and the down matrix splits into 2-tile tasks.
KernelCfg window_cfg_direct(const LayerDev& L, int max_rows, int smem_limit) {
  KernelCfg C = window_cfg(L, max_rows, smem_limit, 0);
  const int kstep = L.bits == 4 ? 64 : 128;
  // measured: faster than the ring for 2-bit layers (their k-steps carry
  // twice the arithmetic) and for 4-bit layers whose wide activations leave a
  // ring of less than three 32 KB stages (d = 4096: 115 against 123 us per
  // eight-row window); the ring wins where it is longer (d = 2048: 74 against
  // 84 us).  STRATA_WINDOW_RING=1 forces the ring and STRATA_WINDOW_DIRECT=1
  // this path wherever its shape conditions hold, for comparisons and tests.
  const bool short_ring = C.nstages * C.stage_bytes < 96 * 1024;
  const bool force = std::getenv("STRATA_WINDOW_DIRECT") != nullptr;
  const bool ok = (L.bits == 2 || short_ring || force) && L.dq == 0 && L.d / kstep >= 8 && L.F / kstep >= 8 &&
                  (L.Fs == 0 || L.Fs / kstep >= 8) && (L.d / 16) % 2 == 0 &&
                  std::getenv("STRATA_WINDOW_RING") == nullptr;
  if (!ok) return C;
  const int fixed = C.total_bytes - C.nstages * C.stage_bytes;
  // the ring's place holds stage R's staged rows of x, later the warps' FIFOs
  const int fifo = kConsumerWarps * (L.bits == 4 ? FifoDepth<4>::value * Fmt<4>::kChunk : FifoDepth<2>::value * Fmt<2>::kChunk);
  const int region = fifo > kMaxRows * kRouterCols * 4 ? fifo : kMaxRows * kRouterCols * 4;
  if (region + fixed > smem_limit) return C;
  C.direct = 1;
  C.nstages = 1;
  C.stage_bytes = region;
  C.total_bytes = C.stage_bytes + fixed;
  C.ph[0].max_sub = 4;
  C.ph[1].max_sub = 4;
  return C;
}

static const void* window_fn(int bits, int direct) {
  if (direct) return bits == 4 ? (const void*)window_kernel_direct<4> : (const void*)window_kernel_direct<2>;
  return bits == 4 ? (const void*)window_kernel<4> : (const void*)window_kernel<2>;
}

cudaError_t window_set_attrs(int bits, int direct, int smem_bytes) {
  return cudaFuncSetAttribute(window_fn(bits, direct), cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

int window_blocks_per_sm(int bits, int direct, int smem_bytes) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, window_fn(bits, direct), direct ? kConsumerThreads : kExpertThreads,
                                                    smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_window(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C.direct ? kConsumerThreads : kExpertThreads);
  cfg.dynamicSmemBytes = C.total_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (C.direct)
    return L.bits == 4 ? cudaLaunchKernelEx(&cfg, window_kernel_direct<4>, L, W, C)
                       : cudaLaunchKernelEx(&cfg, window_kernel_direct<2>, L, W, C);
  if (L.bits == 4) return cudaLaunchKernelEx(&cfg, window_kernel<4>, L, W, C);
  return cudaLaunchKernelEx(&cfg, window_kernel<2>, L, W, C);
}

// One CTA: the round that is due, if any (strata_tier_read).
__global__ void __launch_bounds__(kExpertThreads, 1) tier_round_kernel(TierDev Tr, int E) {
  __shared__ __align__(16) uint8_t scratch[4 * kMaxExperts * 4];
  tier_round_due(Tr, E, scratch);
}

cudaError_t launch_tier_round(const TierDev& Tr, int E, cudaStream_t s) {
  tier_round_kernel<<<1, kExpertThreads, 0, s>>>(Tr, E);
  return cudaGetLastError();
}

KernelCfg head_cfg(int d, int bits, int max_rows, int smem_limit) {
  // the activation buffers of a layer whose inputs are all d wide; phase 2
  // (the head rows, K = d) cut into ring stages like the dense projections
  LayerDev L{};
  L.d = d;
  L.F = d;
  L.Fs = 0;
  L.bits = bits;
  KernelCfg C = window_cfg(L, max_rows, smem_limit, 0);
  const int fixed = C.total_bytes - C.nstages * C.stage_bytes;
  const int ring = smem_limit - fixed;
  int sb2 = 0;
  C.ph[2] = phase_cfg(1, bits, d, d, ring / 3, sb2);
  C.stage_bytes = sb2;
  const int st = sb2 > 0 ? ring / sb2 : 0;
  C.nstages = st > kMaxStages ? kMaxStages : st;
  C.total_bytes = C.nstages * C.stage_bytes + fixed;
  C.direct = 0;
  return C;
}

static const void* head_fn(int bits) {
  return bits == 4 ? (const void*)head_kernel<4> : (const void*)head_kernel<2>;
}

cudaError_t head_set_attrs(int bits, int smem_bytes) {
  return cudaFuncSetAttribute(head_fn(bits), cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

int head_blocks_per_sm(int bits, int smem_bytes) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, head_fn(bits), kExpertThreads, smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_head(const LayerDev& L, const WindowBufs& W, const KernelCfg& C, const HeadArgs& H, int grid,
                        cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kExpertThreads);
  cfg.dynamicSmemBytes = C.total_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.bits == 4) return cudaLaunchKernelEx(&cfg, head_kernel<4>, L, W, C, H);
  return cudaLaunchKernelEx(&cfg, head_kernel<2>, L, W, C, H);
}

static const void* stack_fn(int bits) {
  return bits == 4 ? (const void*)stack_kernel<4> : (const void*)stack_kernel<2>;
}

cudaError_t stack_set_attrs(int bits, int smem_bytes) {
  return cudaFuncSetAttribute(stack_fn(bits), cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

int stack_blocks_per_sm(int bits, int smem_bytes) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, stack_fn(bits), kExpertThreads, smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_stack(const LayerDev* layers, int n_layers, int bits, const WindowBufs& W, const KernelCfg& C,
                         int grid, const float* x, float* y, float* ybuf, float* q_all, float* k_all,
                         cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kExpertThreads);
  cfg.dynamicSmemBytes = C.total_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bits == 4) return cudaLaunchKernelEx(&cfg, stack_kernel<4>, layers, n_layers, W, C, x, y, ybuf, q_all, k_all);
  return cudaLaunchKernelEx(&cfg, stack_kernel<2>, layers, n_layers, W, C, x, y, ybuf, q_all, k_all);
}

}  // namespace strata

#ifdef STRATA_STAMPS
// Timing builds only: copy the stage timestamps of the first n CTAs to host.
extern "C" int strata_probe_stamps(void* host, int n) {
  return (int)cudaMemcpyFromSymbol(host, strata::g_stamps, (size_t)n * 32 * sizeof(unsigned long long));
}
extern "C" int strata_probe_trace(void* host, int n) {
  return (int)cudaMemcpyFromSymbol(host, strata::g_trace, (size_t)n * 4 * 32 * 4 * sizeof(unsigned long long));
}
extern "C" int strata_probe_ptrace(void* host, int n) {
  return (int)cudaMemcpyFromSymbol(host, strata::g_ptrace, (size_t)n * 4 * 64 * sizeof(unsigned long long));
}
extern "C" int strata_probe_trace_clear() {
  static unsigned long long zero[1024 * 4 * 32 * 4];
  return (int)cudaMemcpyToSymbol(strata::g_trace, zero, sizeof(zero));
}
#endif
