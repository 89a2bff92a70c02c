// Grouped expert kernels of the verify window.
//
// The Strata docs ("BATCHING.md", "Several requests at once (batch slots)",
// opening paragraph) state the scheme: the shared expert and every routed
// expert that rows of a window share are read once per window for all of
// them.  Here every distinct expert's packed tiles are streamed from HBM once
// and multiplied against all of that expert's rows (up to 8) in one pass.
//
// Phase 0 (gate/up): first every CTA turns the router's partial logits into
//   the window's routing plan (fp32 softmax, top-k, counting-sort groups; the
//   same fixed-order arithmetic in every CTA, so all agree bit for bit).  Then
//   for the shared expert and each distinct routed expert e, for each 16-row
//   tile of Wg_e and Wu_e: gu = Wg_e x_t and uu = Wu_e x_t for all rows t of
//   e's group, written out in fp32.
// Phase 1 (down + combine): h = silu(gu) * uu is formed while a group's rows
//   are staged (fp16 hi/lo fragments + block sums); for each 16-row tile of
//   Wd_e: o = g_tj * (Wd_e h); the shared expert writes s_t = Wsd h_t.  For
//   each 16-row slice of y, the CTA whose contribution lands last (one atomic
//   per slice, no spinning) sums y_t = s_t + sum_j o_tj in a fixed order.
//
// Structure: one persistent CTA per SM; a producer warp streams k-chunks of a
// task's tiles into a shared-memory ring with bulk async copies; 16 consumer
// warps, split over the task's NS sub-tiles (gate/up of 1-2 row tiles, or 1-4
// down tiles) and, within a sub-tile, over its k-steps.  A consumer turns
// packed codes into fp16 subnormals (one AND per code pair), multiplies them
// against the rows' activations with mma.sync m16n8k16 (activations split into
// fp16 hi + lo parts so the products keep fp32-level accuracy), applies each
// block's scale to the fp32 accumulator fragment, and adds the min term with
// one more MMA against per-block activation sums.  Lanes whose activation
// columns are unused (groups of fewer than 4 or 8 rows) skip their operand
// loads.  Tasks are split across CTAs in contiguous ranges of equal estimated
// cost, so a CTA meets few expert changes.
#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace strata {

namespace {

constexpr int kMaxSub = 4;      // sub-tiles per task
constexpr int kMaxChunks = 32;  // k-chunks per tile
constexpr int kConsumerThreads = kConsumerWarps * 32;

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > (1LL << 31)) {
      atomicOr(err, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
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
// bk points at this lane's slot of plane 0 of the k-step (set 0).
template <int BITS, bool PAIRED>
__device__ __forceinline__ void kstep_mma(const uint8_t* __restrict__ ch, const __half* __restrict__ bk, int bm_set,
                                          bool bon, int lane, float (&acc)[4]) {
  const int g = lane >> 2;
  const float z4[4] = {0.f, 0.f, 0.f, 0.f};
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  if constexpr (BITS == 4) {
    const uint4 bA = bon ? *reinterpret_cast<const uint4*>(bk) : z;
    const uint4 bB = bon ? *reinterpret_cast<const uint4*>(bk + 256) : z;
    uint4 lA = bA, lB = bB;
    if constexpr (!PAIRED) {
      lA = bon ? *reinterpret_cast<const uint4*>(bk + bm_set) : z;
      lB = bon ? *reinterpret_cast<const uint4*>(bk + bm_set + 256) : z;
    }
    const uint4 cw = *reinterpret_cast<const uint4*>(ch + lane * 16);
    const uint2 sr = *reinterpret_cast<const uint2*>(ch + 512 + g * 8);
    const float2 sg = __half22float2(*reinterpret_cast<const __half2*>(&sr.x));
    const float2 s8 = __half22float2(*reinterpret_cast<const __half2*>(&sr.y));
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint32_t wg = blk ? cw.z : cw.x, w8 = blk ? cw.w : cw.y;
      const uint32_t wg2 = wg >> 8, w82 = w8 >> 8;
      const uint4 b = blk ? bB : bA;
      float d[4];
      mma16816(d, dq_pair(wg, 0x000F000Fu), dq_pair(w8, 0x000F000Fu), dq_pair(wg2, 0x000F000Fu),
               dq_pair(w82, 0x000F000Fu), b.x, b.y, z4);
      mma16816(d, dq_pair(wg, 0x00F000F0u), dq_pair(w8, 0x00F000F0u), dq_pair(wg2, 0x00F000F0u),
               dq_pair(w82, 0x00F000F0u), b.z, b.w, d);
      if constexpr (!PAIRED) {
        const uint4 l = blk ? lB : lA;
        mma16816(d, dq_pair(wg, 0x000F000Fu), dq_pair(w8, 0x000F000Fu), dq_pair(wg2, 0x000F000Fu),
                 dq_pair(w82, 0x000F000Fu), l.x, l.y, d);
        mma16816(d, dq_pair(wg, 0x00F000F0u), dq_pair(w8, 0x00F000F0u), dq_pair(wg2, 0x00F000F0u),
                 dq_pair(w82, 0x00F000F0u), l.z, l.w, d);
      }
      const float sgv = blk ? sg.y : sg.x, s8v = blk ? s8.y : s8.x;
      acc[0] = fmaf(sgv, d[0], acc[0]);
      acc[1] = fmaf(sgv, d[1], acc[1]);
      acc[2] = fmaf(s8v, d[2], acc[2]);
      acc[3] = fmaf(s8v, d[3], acc[3]);
    }
  } else {
    const uint4 cw = *reinterpret_cast<const uint4*>(ch + lane * 16);
    const uint4 sa = *reinterpret_cast<const uint4*>(ch + 512 + g * 32);       // s(g, b0..b7)
    const uint4 sb = *reinterpret_cast<const uint4*>(ch + 512 + g * 32 + 16);  // s(g+8, b0..b7)
    const uint32_t cwv[4] = {cw.x, cw.y, cw.z, cw.w};
    const uint32_t sav[4] = {sa.x, sa.y, sa.z, sa.w};
    const uint32_t sbv[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 b = bon ? *reinterpret_cast<const uint4*>(bk + 256 * j) : z;
      uint4 l = b;
      if constexpr (!PAIRED) l = bon ? *reinterpret_cast<const uint4*>(bk + bm_set + 256 * j) : z;
      const uint32_t w = cwv[j], w2 = w >> 8;
      const float2 sgp = __half22float2(*reinterpret_cast<const __half2*>(&sav[j]));
      const float2 s8p = __half22float2(*reinterpret_cast<const __half2*>(&sbv[j]));
      float d[4];
      mma16816(d, dq_pair(w, 0x00030003u), dq_pair(w2, 0x00030003u), dq_pair(w, 0x000C000Cu),
               dq_pair(w2, 0x000C000Cu), b.x, b.y, z4);
      if constexpr (!PAIRED)
        mma16816(d, dq_pair(w, 0x00030003u), dq_pair(w2, 0x00030003u), dq_pair(w, 0x000C000Cu),
                 dq_pair(w2, 0x000C000Cu), l.x, l.y, d);
      acc[0] = fmaf(sgp.x, d[0], acc[0]);
      acc[1] = fmaf(sgp.x, d[1], acc[1]);
      acc[2] = fmaf(s8p.x, d[2], acc[2]);
      acc[3] = fmaf(s8p.x, d[3], acc[3]);
      mma16816(d, dq_pair(w, 0x00300030u), dq_pair(w2, 0x00300030u), dq_pair(w, 0x00C000C0u),
               dq_pair(w2, 0x00C000C0u), b.z, b.w, z4);
      if constexpr (!PAIRED)
        mma16816(d, dq_pair(w, 0x00300030u), dq_pair(w2, 0x00300030u), dq_pair(w, 0x00C000C0u),
                 dq_pair(w2, 0x00C000C0u), l.z, l.w, d);
      acc[0] = fmaf(sgp.y, d[0], acc[0]);
      acc[1] = fmaf(sgp.y, d[1], acc[1]);
      acc[2] = fmaf(s8p.y, d[2], acc[2]);
      acc[3] = fmaf(s8p.y, d[3], acc[3]);
    }
  }
}

// This warp's share of one staged chunk of its sub-tile: k-steps [k0, k1)
// (chunk-local, tile k-step ks_base + kl) and min groups [m0, m1) (chunk-local,
// tile group mk_base + ml).
template <int BITS, bool PAIRED>
__device__ __forceinline__ void chunk_mma(const uint8_t* __restrict__ sub, int mins_off, int ks_base, int k0, int k1,
                                          int mk_base, int m0, int m1, const __half* __restrict__ bm,
                                          const __half* __restrict__ bs, int bm_set, int bs_set, bool bon, int lane,
                                          float (&acc)[4], float (&accm)[4]) {
  constexpr int S = Fmt<BITS>::kBHalves;
  const uint8_t* a = sub + k0 * Fmt<BITS>::kChunk;
  const __half* bk = bm + (ks_base + k0) * 32 * S + lane * 8;
#pragma unroll 2
  for (int kl = k0; kl < k1; ++kl) {
    kstep_mma<BITS, PAIRED>(a, bk, bm_set, bon, lane, acc);
    a += Fmt<BITS>::kChunk;
    bk += 32 * S;
  }
  const uint8_t* am_p = sub + mins_off + m0 * 512 + lane * 16;
  const __half* sp = bs + (mk_base + m0) * 128 + lane * 4;
  const uint2 z = make_uint2(0u, 0u);
  for (int ml = m0; ml < m1; ++ml) {
    const uint2 b = bon ? *reinterpret_cast<const uint2*>(sp) : z;
    const uint4 am = *reinterpret_cast<const uint4*>(am_p);
    mma16816(accm, am.x, am.y, am.z, am.w, b.x, b.y, accm);
    if constexpr (!PAIRED) {
      const uint2 l = bon ? *reinterpret_cast<const uint2*>(sp + bs_set) : z;
      mma16816(accm, am.x, am.y, am.z, am.w, l.x, l.y, accm);
    }
    am_p += 512;
    sp += 128;
  }
}

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
  long long cpos[kMaxExperts + 2];   // cost position of each group's first task
  int finish[kMaxEntries * 4];       // row slices this CTA combines (phase 1)
  int nfinish;
  int t0, t1;                        // this CTA's task range
  short cks[2][kMaxChunks + 1];      // k-chunk bounds: [0] routed K, [1] shared K
  short cmk[2][kMaxChunks + 1];
};

__device__ __forceinline__ unsigned ord_f32(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(unsigned u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// The window's routing from the router kernel's partial logits.  Every CTA runs
// this same fixed-order arithmetic; CTA 0 also publishes the plan and the
// caller's routing outputs.
__device__ void compute_plan(const LayerDev& L, const WindowBufs& W, SPlan& sp, float* lg) {
  const int T = W.T, E = L.E, k = L.k, njb = W.njb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool pub = blockIdx.x == 0;
  Plan* P = W.plan;
  for (int i = tid; i < T * E; i += blockDim.x) {
    const int t = i / E, e = i - t * E;
    const float* pp = W.partial + (long long)t * E + e;
    float part[8];
    float v = 0.f;
    for (int b0 = 0; b0 < njb; b0 += 8) {
#pragma unroll
      for (int b = 0; b < 8; ++b)
        part[b] = (b0 + b < njb) ? __ldcg(pp + (long long)(b0 + b) * kMaxRows * E) : 0.f;
#pragma unroll
      for (int b = 0; b < 8; ++b) v += part[b];
    }
    if (L.router_b) v += L.router_b[e];
    lg[t * E + e] = v;
    if (pub) W.logits[t * E + e] = v;
  }
  __syncthreads();
  if (warp < T) {
    const int t = warp;
    const float* lr = lg + t * E;
    float m = -INFINITY;
    bool finite = true;
    for (int e = lane; e < E; e += 32) {
      const float v = lr[e];
      finite &= isfinite(v);
      m = fmaxf(m, v);
    }
    m = unord_f32(__reduce_max_sync(0xffffffffu, ord_f32(m)));
    if (!__all_sync(0xffffffffu, finite) && lane == 0 && pub) atomicOr(W.err, kErrNonFinite);
    float z = 0.f;
    for (int e = lane; e < E; e += 32) z += expf(lr[e] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    // top-k by logit, descending, ties -> lower expert index
    unsigned taken = 0u;  // bit i: expert lane + 32*i already selected
    float wsum = 0.f, wsel = 0.f;
    int esel = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
      for (int i = 0, e = lane; e < E; ++i, e += 32) {
        const float v = lr[e];
        if (!((taken >> i) & 1u) && (v > bv || be == 0x7fffffff)) { bv = v; be = e; }
      }
      const unsigned key = be == 0x7fffffff ? 0u : ord_f32(bv);
      const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
      int bi = (int)__reduce_min_sync(0xffffffffu, (key == kmax && be != 0x7fffffff) ? (unsigned)be : 0xffffffffu);
      if (bi < 0 || bi >= E) bi = 0;  // only with non-finite logits
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      const float p = expf(unord_f32(kmax) - m) / z;
      wsum += p;
      if (lane == j) { esel = bi; wsel = p; }
    }
    if (lane < k) {
      const float g = L.renorm ? wsel / wsum : wsel;
      const int ent = t * k + lane;
      sp.sel[ent] = esel;
      sp.topk_w[ent] = g;
      if (pub) {
        P->topk_idx[ent] = esel;
        P->topk_w[ent] = g;
        if (W.out_topk_idx) W.out_topk_idx[ent] = esel;
        if (W.out_topk_w) W.out_topk_w[ent] = g;
      }
    }
  }
  __syncthreads();
  // counting sort of entries by expert: thread e < 256 owns expert e; the
  // counts (low 16 bits) and the "used" flags (high 16 bits) are scanned together
  const int nent = T * k;
  const int e = tid;
  int c = 0;
  if (e < E)
    for (int i = 0; i < nent; ++i) c += (sp.sel[i] == e);
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
  if (warp == 0) {
    int tv = lane < kMaxExperts / 32 ? sp.wscan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, tv, o);
      if (lane >= o) tv += n;
    }
    sp.wscan[lane] = tv;  // inclusive prefix over warps
  }
  __syncthreads();
  if (e < E) {
    const int incl = v + (warp > 0 ? sp.wscan[warp - 1] : 0);
    const int off = (incl & 0xffff) - c, rank = (incl >> 16) - flag;
    sp.counts[e] = c;
    sp.offsets[e] = off;
    if (flag) sp.distinct[rank] = e;
    int pos = off;
    for (int i = 0; i < nent && pos < off + c; ++i)
      if (sp.sel[i] == e) sp.entries[pos++] = i;
    if (e == E - 1) sp.nd = (incl >> 16);
    if (pub) {
      P->counts[e] = c;
      P->offsets[e] = off;
      if (W.out_counts) W.out_counts[e] = c;
      if (W.out_offsets) W.out_offsets[e] = off;
      if (flag) {
        P->distinct[rank] = e;
        if (W.out_distinct) W.out_distinct[rank] = e;
      }
      if (e == E - 1) {
        P->offsets[E] = off + c;
        P->n_distinct = incl >> 16;
        P->T = T;
        if (W.out_offsets) W.out_offsets[E] = off + c;
        if (W.out_ndistinct) *W.out_ndistinct = incl >> 16;
      }
    }
  }
  __syncthreads();
  if (pub) {
    for (int i = tid; i < nent; i += blockDim.x) {
      P->entries[i] = sp.entries[i];
      if (W.out_entries) W.out_entries[i] = sp.entries[i];
    }
  }
}

struct Task {
  bool shared;
  int expert;
  int tile;  // first row tile
};

__device__ __forceinline__ Task decode_task(int task, int ntask_s, int ntask_e, int tiles_per_task, const SPlan& sp) {
  Task t;
  if (task < ntask_s) {
    t.shared = true;
    t.expert = -1;
    t.tile = task * tiles_per_task;
  } else {
    const int q = task - ntask_s;
    const int gi = q / ntask_e;
    t.shared = false;
    t.expert = sp.distinct[gi];
    t.tile = (q - gi * ntask_e) * tiles_per_task;
  }
  return t;
}

// Estimated cost of one task of a group of R rows (groups of more than 4 rows
// take the two-set path: twice the MMAs and activation loads).
__device__ __forceinline__ int task_cost(int R) { return R <= 4 ? 2 : 3; }

// Contiguous task ranges of equal estimated cost (thread 0 only): fills the
// group cost prefix and this CTA's [t0, t1).
__device__ void split_tasks(const WindowBufs& W, SPlan& sp, bool has_shared, int ntask_s, int ntask_e) {
  const int ng = (has_shared ? 1 : 0) + sp.nd;
  auto rows_of = [&](int g) -> int {
    return (has_shared && g == 0) ? W.T : sp.counts[sp.distinct[g - (has_shared ? 1 : 0)]];
  };
  auto ntask_of = [&](int g) -> int { return (has_shared && g == 0) ? ntask_s : ntask_e; };
  long long pos = 0;
  for (int g = 0; g < ng; ++g) {
    sp.cpos[g] = pos;
    pos += (long long)ntask_of(g) * task_cost(rows_of(g));
  }
  sp.cpos[ng] = pos;
  auto task_at = [&](long long p) -> int {  // first task whose start position is >= p
    int task = 0;
    for (int g = 0; g < ng; ++g) {
      const int nt = ntask_of(g);
      if (p <= sp.cpos[g]) return task;
      if (p < sp.cpos[g + 1]) {
        const int cst = task_cost(rows_of(g));
        const long long i = (p - sp.cpos[g] + cst - 1) / cst;
        return task + (int)(i < nt ? i : nt);
      }
      task += nt;
    }
    return task;
  };
  const long long total = sp.cpos[ng];
  sp.t0 = task_at(total * blockIdx.x / gridDim.x);
  sp.t1 = task_at(total * (blockIdx.x + 1) / gridDim.x);
}

// Stage one group's activations into shared memory (all consumer threads).
// Phase 0: copy the router's x fragments.  Phase 1: form h = silu(gu) * uu,
// its fp16 hi/lo fragments and its block sums.
template <int BITS, int PHASE>
__device__ void load_group_B(const LayerDev& L, const WindowBufs& W, const SPlan& sp, const SmemCfg& C, __half* bm,
                             __half* bs, bool is_shared, int R, int ent_off, int K, int ctid) {
  constexpr int S = Fmt<BITS>::kBHalves;
  constexpr int B = Fmt<BITS>::kBlock;
  const int nks = K / Fmt<BITS>::kKstep;
  const int nmk = (K / B + 15) / 16;
  const bool paired = R <= 4;
  if (PHASE == 0) {
    const long long fh = frag_halves(K, nmk);
    const int nsets = paired ? 1 : 2;
    const int ncols = paired ? 2 * R : R;
    // main: 16-byte pieces (ks, c, plane) of each used column
    const int per_col = nks * 4 * (S / 8);
    for (int i = ctid; i < nsets * ncols * per_col; i += kConsumerThreads) {
      const int cs = i / per_col, rem = i - cs * per_col;
      const int set = cs / ncols, col = cs - set * ncols;
      const int r = paired ? (col >> 1) : col;
      const int part = paired ? (col & 1) : set;
      const int xrow = is_shared ? r : sp.entries[ent_off + r] / L.k;
      const int ks = rem / (4 * (S / 8)), cp = rem - ks * 4 * (S / 8);
      const int c = cp / (S / 8), p = cp - c * (S / 8);
      const uint4 v = __ldcg(reinterpret_cast<const uint4*>(W.xfrag + xrow * fh + (long long)part * K + ks * 4 * S +
                                                            c * S + p * 8));
      *reinterpret_cast<uint4*>(bm + set * C.bmain_halves + bmain_off<BITS>(ks, p, col, c)) = v;
    }
    // sums: 8-byte pieces (mk, c)
    for (int i = ctid; i < nsets * ncols * nmk * 4; i += kConsumerThreads) {
      const int cs = i / (nmk * 4), rem = i - cs * nmk * 4;
      const int set = cs / ncols, col = cs - set * ncols;
      const int r = paired ? (col >> 1) : col;
      const int part = paired ? (col & 1) : set;
      const int xrow = is_shared ? r : sp.entries[ent_off + r] / L.k;
      const int mk = rem >> 2, c = rem & 3;
      const uint2 v = __ldcg(reinterpret_cast<const uint2*>(W.xfrag + xrow * fh + 2LL * K +
                                                            (long long)part * 16 * nmk + mk * 16 + c * 4));
      *reinterpret_cast<uint2*>(bs + set * C.bsum_halves + (mk * 8 + col) * 16 + c * 4) = v;
    }
  } else {
    // one element per thread and step; a warp covers 32 consecutive elements of
    // one row (K is a multiple of 64), so block sums come from lane shuffles
    for (int i0 = 0; i0 < R * K; i0 += kConsumerThreads) {
      const int i = i0 + ctid;
      const bool in = i < R * K;
      const int r = in ? i / K : 0, f = in ? i - r * K : 0;
      float h = 0.f;
      if (in) {
        const float2* src = is_shared ? W.sgu + (long long)r * L.Fs : W.gu + (long long)sp.entries[ent_off + r] * L.F;
        const float2 gu = __ldcg(src + f);
        h = silu_f32(gu.x) * gu.y;
        int off;
        float fac;
        frag_main_pos<BITS>(f, off, fac);
        const int ks = off / (4 * S), c = (off / S) & 3, slot = off % S;
        __half hi, lo;
        split_hi_lo(h * fac, hi, lo);
        const int o = bmain_off<BITS>(ks, slot >> 3, 0, c) + (slot & 7);
        if (paired) {
          bm[o + (2 * r) * 32] = hi;
          bm[o + (2 * r + 1) * 32] = lo;
        } else {
          bm[o + r * 32] = hi;
          bm[C.bmain_halves + o + r * 32] = lo;
        }
      }
      float s = h;
#pragma unroll
      for (int o = B / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (in && (f % B) == 0) {
        const int spos = frag_sum_pos(f / B);
        const int mk = spos >> 4, c = (spos >> 2) & 3, slot = spos & 3;
        __half hi, lo;
        split_hi_lo(s, hi, lo);
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
  }
}

}  // namespace

// Shared memory: [ring: nstages x stage_bytes][B main: nsets][B sums: nsets]
// [red: 2 x 16 warps x 32 lanes float4][full/empty mbarriers]; static: SPlan.
template <int BITS, int PHASE, int NS>
__device__ __forceinline__ void run_tasks(const LayerDev& L, const WindowBufs& W, const SmemCfg& C, SPlan& sp,
                                          uint8_t* ring, __half* bm, __half* bs, float4* red, uint64_t* full,
                                          uint64_t* empty, volatile int* s_abort, int ntask_s, int ntask_e, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int kMT = PHASE == 0 ? NS / 2 : NS;  // row tiles per task
  constexpr int kWPS = kConsumerWarps / NS;      // warps per sub-tile
  const bool has_shared = L.Fs > 0;
  const int t0 = sp.t0, t1 = sp.t1;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int task = t0; task < t1 && ok; ++task) {
        const Task tk = decode_task(task, ntask_s, ntask_e, kMT, sp);
        if (!tk.shared && (unsigned)tk.expert >= (unsigned)L.E) {
          atomicOr(W.err, kErrIndex);
          *s_abort = 1;
          break;
        }
        const int K = PHASE == 0 ? L.d : (tk.shared ? L.Fs : L.F);
        const int nks = K / Fmt<BITS>::kKstep, nmk = (K / Fmt<BITS>::kBlock + 15) / 16;
        const int tbytes = nks * Fmt<BITS>::kChunk + nmk * 512;
        const int kv = (PHASE == 1 && tk.shared) ? 1 : 0;
        for (int ch = 0; ch < C.nchunks; ++ch) {
          const int ks0 = sp.cks[kv][ch], ks1 = sp.cks[kv][ch + 1];
          const int mk0 = sp.cmk[kv][ch], mk1 = sp.cmk[kv][ch + 1];
          const int stage = it % C.nstages;
          if (it >= C.nstages && !wait_bar(&empty[stage], ((it / C.nstages) - 1) & 1, W.err, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t cbytes = (uint32_t)((ks1 - ks0) * Fmt<BITS>::kChunk), mbytes = (uint32_t)((mk1 - mk0) * 512);
          mbar_arrive_expect_tx(&full[stage], NS * (cbytes + mbytes));
          uint8_t* dst = ring + (size_t)stage * C.stage_bytes;
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            const bool up = PHASE == 0 && s >= kMT;
            const PackedMat& M = PHASE == 0 ? (up ? (tk.shared ? L.sup : L.up) : (tk.shared ? L.sgate : L.gate))
                                            : (tk.shared ? L.sdown : L.down);
            const int tile = tk.tile + (up ? s - kMT : s);
            const uint8_t* src = M.base + (tk.shared ? 0LL : (long long)tk.expert * M.mat_bytes) +
                                 (long long)tile * tbytes;
            uint8_t* d = dst + s * C.sub_stride;
            if (cbytes) bulk_g2s(d, src + (size_t)ks0 * Fmt<BITS>::kChunk, cbytes, &full[stage]);
            if (mbytes) bulk_g2s(d + C.mins_off, src + (size_t)nks * Fmt<BITS>::kChunk + mk0 * 512, mbytes, &full[stage]);
          }
          ++it;
        }
      }
      if (*s_abort) {
        // Let every copy this warp issued land before the CTA can exit.
        for (int j = (it > C.nstages ? it - C.nstages : 0); j < it; ++j) {
          const long long tw = clock64();
          while (!mbar_try_wait(&full[j % C.nstages], (j / C.nstages) & 1)) {
            if (clock64() - tw > (1LL << 31)) break;
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int sub = warp / kWPS, kg = warp % kWPS;
  const int g = lane >> 2;
  int it = 0;
  int cur = -2;
  int R = 0, ent_off = 0;
  bool paired = true, bon = true;
  int buf = 0;
  for (int task = t0; task < t1; ++task) {
    const Task tk = decode_task(task, ntask_s, ntask_e, kMT, sp);
    const int group = tk.shared ? -1 : tk.expert;
    if ((unsigned)(group + 1) > (unsigned)L.E) break;  // guarded by the producer too
    const int K = PHASE == 0 ? L.d : (tk.shared ? L.Fs : L.F);
    if (group != cur) {
      if (tk.shared) {
        R = W.T;
        ent_off = 0;
      } else {
        R = sp.counts[tk.expert];
        ent_off = sp.offsets[tk.expert];
      }
      if (R < 1 || R > kMaxRows) {
        atomicOr(W.err, kErrIndex);
        R = R < 1 ? 1 : kMaxRows;
      }
      paired = R <= 4;
      bon = paired ? (g < 2 * R) : (g < R);
      // the previous task's barrier guarantees no warp still reads the old fragments
      load_group_B<BITS, PHASE>(L, W, sp, C, bm, bs, tk.shared, R, ent_off, K, tid);
      consumer_sync();
      cur = group;
    }
    const int kv = (PHASE == 1 && tk.shared) ? 1 : 0;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, accm[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ch = 0; ch < C.nchunks; ++ch) {
      const int ks0 = sp.cks[kv][ch], ks1 = sp.cks[kv][ch + 1];
      const int mk0 = sp.cmk[kv][ch], mk1 = sp.cmk[kv][ch + 1];
      const int nk = ks1 - ks0, nm = mk1 - mk0;
      const int k0 = (kg * nk) / kWPS, k1 = ((kg + 1) * nk) / kWPS;
      const int m0 = (kg * nm) / kWPS, m1 = ((kg + 1) * nm) / kWPS;
      const int stage = it % C.nstages;
      if (wait_bar(&full[stage], (it / C.nstages) & 1, W.err, s_abort)) {
        const uint8_t* st = ring + (size_t)stage * C.stage_bytes + sub * C.sub_stride;
        if (paired)
          chunk_mma<BITS, true>(st, C.mins_off, ks0, k0, k1, mk0, m0, m1, bm, bs, C.bmain_halves, C.bsum_halves,
                                bon, lane, acc, accm);
        else
          chunk_mma<BITS, false>(st, C.mins_off, ks0, k0, k1, mk0, m0, m1, bm, bs, C.bmain_halves, C.bsum_halves,
                                 bon, lane, acc, accm);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      ++it;
    }
    float4* rb = red + buf * (kConsumerWarps * 32);
    rb[warp * 32 + lane] = make_float4(fmaf(acc[0], kDqUnscale, accm[0]), fmaf(acc[1], kDqUnscale, accm[1]),
                                       fmaf(acc[2], kDqUnscale, accm[2]), fmaf(acc[3], kDqUnscale, accm[3]));
    consumer_sync();

    // ---------------- epilogue: cross-warp sums in a fixed order ----------------
    if (PHASE == 0) {
      for (int i = tid; i < kMT * 16 * R; i += kConsumerThreads) {
        const int m = i / (16 * R), rem = i - m * 16 * R;
        const int r = rem >> 4, row = rem & 15;
        const int src_lane = (row & 7) * 4 + (paired ? r : (r >> 1));
        const int idx = ((row >> 3) << 1) + (paired ? 0 : (r & 1));
        float gv = 0.f, uv = 0.f;
#pragma unroll
        for (int w = 0; w < kWPS; ++w) {
          const float4 a = rb[(m * kWPS + w) * 32 + src_lane];
          const float4 b = rb[((kMT + m) * kWPS + w) * 32 + src_lane];
          const float* af = reinterpret_cast<const float*>(&a);
          const float* bf = reinterpret_cast<const float*>(&b);
          gv += paired ? (af[idx] + af[idx + 1]) : af[idx];
          uv += paired ? (bf[idx] + bf[idx + 1]) : bf[idx];
        }
        const int f = (tk.tile + m) * 16 + row;
        float2* dst = tk.shared ? W.sgu + (long long)r * L.Fs : W.gu + (long long)sp.entries[ent_off + r] * L.F;
        dst[f] = make_float2(gv, uv);
      }
    } else {
      for (int i = tid; i < NS * 16 * R; i += kConsumerThreads) {
        const int s = i / (16 * R), rem = i - s * 16 * R;
        const int r = rem >> 4, row = rem & 15;
        const int src_lane = (row & 7) * 4 + (paired ? r : (r >> 1));
        const int idx = ((row >> 3) << 1) + (paired ? 0 : (r & 1));
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWPS; ++w) {
          const float4 a = rb[(s * kWPS + w) * 32 + src_lane];
          const float* af = reinterpret_cast<const float*>(&a);
          v += paired ? (af[idx] + af[idx + 1]) : af[idx];
        }
        const int drow = (tk.tile + s) * 16 + row;
        if (tk.shared) {
          W.sbuf[(long long)r * L.d + drow] = v;
        } else {
          const int ent = sp.entries[ent_off + r];
          W.obuf[(long long)ent * L.d + drow] = sp.topk_w[ent] * v;
        }
      }
    }
    buf ^= 1;
  }

  if (PHASE == 1) {
    // Count this CTA's finished row slices; the CTA that completes a slice's
    // count sums y for it in a fixed order.
    __threadfence();
    consumer_sync();
    if (tid == 0) sp.nfinish = 0;
    consumer_sync();
    const int ngroups = (has_shared ? 1 : 0) + sp.nd;
    const int ntiles = (t1 - t0) * NS;
    for (int i = tid; i < ntiles; i += kConsumerThreads) {
      const Task tk = decode_task(t0 + i / NS, ntask_s, ntask_e, NS, sp);
      const int tile = tk.tile + i % NS;
      if (atomicAdd(W.counters + tile, 1) == ngroups - 1) {
        const int slot = atomicAdd(&sp.nfinish, 1);
        if (slot < kMaxEntries * 4) {
          sp.finish[slot] = tile;
        } else {  // list full: this thread sums the slice itself
          __threadfence();
          for (int e = 0; e < W.T * 16; ++e) {
            const int t = e >> 4, rr = tile * 16 + (e & 15);
            float y = has_shared ? __ldcg(W.sbuf + (long long)t * L.d + rr) : 0.f;
            for (int j = 0; j < L.k; ++j) y += __ldcg(W.obuf + (long long)(t * L.k + j) * L.d + rr);
            W.y[(long long)t * L.d + rr] = y;
          }
        }
      }
    }
    consumer_sync();
    __threadfence();
    const int nf = min(sp.nfinish, kMaxEntries * 4);
    const int T = W.T, k = L.k;
    for (int i = tid; i < nf * T * 16; i += kConsumerThreads) {
      const int f = i / (T * 16), rem = i % (T * 16);
      const int t = rem >> 4, rr = sp.finish[f] * 16 + (rem & 15);
      float y = has_shared ? __ldcg(W.sbuf + (long long)t * L.d + rr) : 0.f;
      for (int j = 0; j < k; ++j) y += __ldcg(W.obuf + (long long)(t * k + j) * L.d + rr);
      W.y[(long long)t * L.d + rr] = y;
    }
  }
}

template <int BITS, int PHASE>
__global__ void __launch_bounds__(kExpertThreads, 1) expert_kernel(LayerDev L, WindowBufs W, SmemCfg C) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ SPlan sp;
  const int tid = threadIdx.x;
  uint8_t* ring = smem;
  __half* bm = reinterpret_cast<__half*>(smem + (size_t)C.nstages * C.stage_bytes);
  __half* bs = bm + (size_t)C.nsets * C.bmain_halves;
  float4* red = reinterpret_cast<float4*>(bs + (size_t)C.nsets * C.bsum_halves);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 2 * kConsumerWarps * 32);
  uint64_t* empty = full + kMaxStages;

  if (tid == 0) {
    for (int s = 0; s < C.nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    s_abort = 0;
    fence_mbar_init();
    for (int v = 0; v < 2; ++v) {
      const int K = PHASE == 0 ? L.d : (v == 0 ? L.F : L.Fs);
      const int nks = K / Fmt<BITS>::kKstep, nmk = (K / Fmt<BITS>::kBlock + 15) / 16;
      for (int ch = 0; ch <= C.nchunks; ++ch) {
        sp.cks[v][ch] = (short)(ch * nks / C.nchunks);
        sp.cmk[v][ch] = (short)(ch * nmk / C.nchunks);
      }
    }
  }
  // padded block-sum slots are never written: zero the sums region once
  for (int i = tid; i < C.nsets * C.bsum_halves / 2; i += blockDim.x) reinterpret_cast<uint32_t*>(bs)[i] = 0u;
  griddep_launch_dependents();
  griddep_wait();

  if (PHASE == 0) {
    // the ring is free until the producer starts: use it for the logits
    compute_plan(L, W, sp, reinterpret_cast<float*>(ring));
  } else {
    const Plan* P = W.plan;
    const int E = L.E, nent = W.T * L.k;
    if (tid == 0) sp.nd = __ldcg(&P->n_distinct);
    for (int i = tid; i < E; i += blockDim.x) {
      sp.distinct[i] = __ldcg(P->distinct + i);
      sp.counts[i] = __ldcg(P->counts + i);
      sp.offsets[i] = __ldcg(P->offsets + i);
    }
    for (int i = tid; i < nent; i += blockDim.x) {
      sp.entries[i] = __ldcg(P->entries + i);
      sp.topk_w[i] = __ldcg(P->topk_w + i);
    }
  }
  __syncthreads();
  const int nd = sp.nd;
  if (nd < 0 || nd > L.E) {
    if (tid == 0) atomicOr(W.err, kErrIndex);
    return;
  }

  const bool has_shared = L.Fs > 0;
  const int ngroups = (has_shared ? 1 : 0) + nd;
  int mt, ntask_s, ntask_e;
  if (PHASE == 0) {
    // gate/up row tiles per task: 2 when that still leaves >= 3 tasks per CTA
    const int tiles_e = L.F / 16, tiles_s = has_shared ? L.Fs / 16 : 0;
    const long long all_tiles = tiles_s + (long long)nd * tiles_e;
    mt = (C.max_sub >= 4 && tiles_e % 2 == 0 && tiles_s % 2 == 0 && all_tiles / 2 >= 3LL * gridDim.x) ? 2 : 1;
    ntask_s = tiles_s / mt;
    ntask_e = tiles_e / mt;
  } else {
    // down row tiles per task: as many as keep >= 3 tasks per CTA (up to 4)
    const int tiles_g = L.d / 16;
    const long long all_tiles = (long long)ngroups * tiles_g;
    mt = C.max_sub;
    while (mt > 1 && (tiles_g % mt != 0 || all_tiles / mt < 3LL * gridDim.x)) mt >>= 1;
    ntask_s = has_shared ? tiles_g / mt : 0;
    ntask_e = tiles_g / mt;
  }
  if (tid == 0) split_tasks(W, sp, has_shared, ntask_s, ntask_e);
  __syncthreads();
  if (PHASE == 0) {
    if (mt == 2)
      run_tasks<BITS, 0, 4>(L, W, C, sp, ring, bm, bs, red, full, empty, &s_abort, ntask_s, ntask_e, tid);
    else
      run_tasks<BITS, 0, 2>(L, W, C, sp, ring, bm, bs, red, full, empty, &s_abort, ntask_s, ntask_e, tid);
  } else {
    if (mt == 4)
      run_tasks<BITS, 1, 4>(L, W, C, sp, ring, bm, bs, red, full, empty, &s_abort, ntask_s, ntask_e, tid);
    else if (mt == 2)
      run_tasks<BITS, 1, 2>(L, W, C, sp, ring, bm, bs, red, full, empty, &s_abort, ntask_s, ntask_e, tid);
    else
      run_tasks<BITS, 1, 1>(L, W, C, sp, ring, bm, bs, red, full, empty, &s_abort, ntask_s, ntask_e, tid);
  }
}

SmemCfg expert_smem_cfg(const LayerDev& L, int phase, int max_rows, int smem_limit) {
  SmemCfg C{};
  const int bits = L.bits;
  const int kstep = bits == 4 ? 64 : 128, block = bits == 4 ? 32 : 16, chunk = bits == 4 ? 576 : 768;
  const int S = bits == 4 ? 16 : 32;
  int Kmax = phase == 0 ? L.d : (L.Fs > L.F ? L.Fs : L.F);
  const int nks = Kmax / kstep;
  const int nmk = (Kmax / block + 15) / 16;
  C.bmain_halves = nks * 8 * 4 * S;
  C.bsum_halves = nmk * 8 * 4 * 4;
  C.nsets = max_rows > 4 ? 2 : 1;
  const int fixed = C.nsets * (C.bmain_halves + C.bsum_halves) * 2 + 2 * kConsumerWarps * 32 * 16 + 2 * kMaxStages * 8;
  // Pick the task width (sub-tiles: 4, 2, or 1; gate/up need >= 2) and the
  // k-chunks per tile: the fewest chunks that leave >= 3 ring stages, scored by
  // k-steps per warp per chunk (each chunk costs a wait and a release).
  const int ns_min = phase == 0 ? 2 : 1;
  int best_score = -1;
  SmemCfg best = C;
  for (int ns = kMaxSub; ns >= ns_min; ns >>= 1) {
    const int wps = kConsumerWarps / ns;
    for (int nc = 1; nc <= nks && nc <= kMaxChunks; ++nc) {
      const int cks = (nks + nc - 1) / nc, cmk = (nmk + nc - 1) / nc;
      SmemCfg t = C;
      t.mins_off = cks * chunk;
      t.sub_stride = t.mins_off + cmk * 512;
      t.stage_bytes = ns * t.sub_stride;
      t.nchunks = nc;
      t.max_sub = ns;
      int st = (smem_limit - fixed) / t.stage_bytes;
      if (st > kMaxStages) st = kMaxStages;
      t.nstages = st;
      if (st < 3) continue;
      const int per_warp = (nks / nc) / wps;
      const int score = (per_warp > 8 ? 8 : per_warp) * 1000 + ns * 100 + st;
      if (score > best_score) {
        best_score = score;
        best = t;
      }
      break;
    }
  }
  if (best_score < 0) {  // not even 3 stages: the narrowest task, small chunks
    best = C;
    best.nchunks = nks < kMaxChunks ? nks : kMaxChunks;
    const int cks = (nks + best.nchunks - 1) / best.nchunks, cmk = (nmk + best.nchunks - 1) / best.nchunks;
    best.mins_off = cks * chunk;
    best.sub_stride = best.mins_off + cmk * 512;
    best.max_sub = ns_min;
    best.stage_bytes = ns_min * best.sub_stride;
    best.nstages = (smem_limit - fixed) / best.stage_bytes;
    if (best.nstages > kMaxStages) best.nstages = kMaxStages;
  }
  C = best;
  C.total_bytes = C.nstages * C.stage_bytes + fixed;
  return C;
}

static const void* expert_fn(int bits, int phase) {
  if (bits == 4) return phase == 0 ? (const void*)expert_kernel<4, 0> : (const void*)expert_kernel<4, 1>;
  return phase == 0 ? (const void*)expert_kernel<2, 0> : (const void*)expert_kernel<2, 1>;
}

cudaError_t expert_set_attrs(int bits, int phase, int smem_bytes) {
  return cudaFuncSetAttribute(expert_fn(bits, phase), cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t launch_expert(const LayerDev& L, const WindowBufs& W, const SmemCfg& C, int phase, int grid,
                          cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kExpertThreads);
  cfg.dynamicSmemBytes = C.total_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (L.bits == 4) {
    if (phase == 0) return cudaLaunchKernelEx(&cfg, expert_kernel<4, 0>, L, W, C);
    return cudaLaunchKernelEx(&cfg, expert_kernel<4, 1>, L, W, C);
  }
  if (phase == 0) return cudaLaunchKernelEx(&cfg, expert_kernel<2, 0>, L, W, C);
  return cudaLaunchKernelEx(&cfg, expert_kernel<2, 1>, L, W, C);
}

}  // namespace strata
