// Grouped expert kernels of the verify window.
//
// The Strata docs ("BATCHING.md", "Several requests at once (batch slots)",
// opening paragraph) state the scheme: the shared expert and every routed
// expert that rows of a window share are read once per window for all of
// them.  Here every distinct expert's packed tiles are streamed from HBM once
// and multiplied against all of that expert's rows (up to 8) in one pass.
//
// Phase 0 (gate/up): for the shared expert and each distinct routed expert e,
//   for each 16-row tile of Wg_e and Wu_e: gu = Wg_e x_t, uu = Wu_e x_t for all
//   rows t of e's group; h = silu(gu) * uu is written as down-projection
//   activation fragments (fp16 hi/lo) plus per-16 partial sums.
// Phase 1 (down + combine): for each 16-row tile of Wd_e: o = g_tj * (Wd_e h);
//   the shared expert writes s_t = Wsd h_t.  The CTA that finishes a row tile
//   last (one atomic per tile, no spinning) sums y_t = s_t + sum_j o_tj in a
//   fixed order.
//
// Structure: one persistent CTA per SM, a producer warp streaming whole tiles
// (16 rows x full K) into a shared-memory ring with bulk async copies, and 8
// consumer warps splitting each tile's K range.  A consumer turns packed codes
// into exact fp16 integers (lop3 + sub), multiplies them against the rows'
// activations with mma.sync m16n8k16 (activations split into fp16 hi + lo
// parts so the products keep fp32-level accuracy), applies each block's scale
// to the fp32 accumulator fragment, and adds the min term with one more MMA
// against per-block activation sums.  Tasks (tiles) are split evenly and
// contiguously across CTAs so a CTA meets few expert changes.
#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace strata {

namespace {

__device__ __forceinline__ bool wait_full(uint64_t* bar, uint32_t parity, unsigned* err, volatile int* abort_flag) {
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

template <int BITS>
__host__ __device__ inline int tile_bytes_of(int K) {
  const int nks = K / Fmt<BITS>::kKstep;
  const int nmk = (K / Fmt<BITS>::kBlock + 15) / 16;
  return nks * Fmt<BITS>::kChunk + nmk * 512;
}

// One 16-row tile, this warp's share of K.  acc layout: paired (rows <= 4):
// [row g, (r=c) hi], [row g, (r=c) lo], [row g+8, hi], [row g+8, lo];
// unpaired: [row g, r=2c], [row g, r=2c+1], [row g+8, r=2c], [row g+8, r=2c+1].
template <int BITS, bool PAIRED>
__device__ __forceinline__ void tile_mma(const uint8_t* __restrict__ st, const __half* __restrict__ bm,
                                         const __half* __restrict__ bs, int bm_set, int bs_set, int nks, int k0,
                                         int k1, int m0, int m1, int lane, float (&acc)[4]) {
  const int g = lane >> 2, c = lane & 3;
  const float z4[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (BITS == 4) {
#pragma unroll 2
    for (int ks = k0; ks < k1; ++ks) {
      const uint8_t* ch = st + ks * Fmt<4>::kChunk;
      const uint4 cw = *reinterpret_cast<const uint4*>(ch + lane * 16);
      const uint2 sr = *reinterpret_cast<const uint2*>(ch + 512 + g * 8);
      const float2 sg = __half22float2(*reinterpret_cast<const __half2*>(&sr.x));  // s(g,b0), s(g,b1)
      const float2 s8 = __half22float2(*reinterpret_cast<const __half2*>(&sr.y));  // s(g+8,b0), s(g+8,b1)
      const __half* bp = bm + ((ks * 8 + g) * 4 + c) * 16;
      const uint4 bA = *reinterpret_cast<const uint4*>(bp);
      const uint4 bB = *reinterpret_cast<const uint4*>(bp + 8);
      uint4 lA, lB;
      if constexpr (!PAIRED) {
        lA = *reinterpret_cast<const uint4*>(bp + bm_set);
        lB = *reinterpret_cast<const uint4*>(bp + bm_set + 8);
      }
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint32_t wg = blk ? cw.z : cw.x, w8 = blk ? cw.w : cw.y;
        const uint32_t wg2 = wg >> 8, w82 = w8 >> 8;
        const uint32_t a0 = dq_pair(wg, 0x000F000Fu), a1 = dq_pair(w8, 0x000F000Fu);
        const uint32_t a2 = dq_pair(wg2, 0x000F000Fu), a3 = dq_pair(w82, 0x000F000Fu);
        const uint32_t e0 = dq_pair(wg, 0x00F000F0u), e1 = dq_pair(w8, 0x00F000F0u);
        const uint32_t e2 = dq_pair(wg2, 0x00F000F0u), e3 = dq_pair(w82, 0x00F000F0u);
        const uint4 b = blk ? bB : bA;
        float d[4];
        mma16816(d, a0, a1, a2, a3, b.x, b.y, z4);
        mma16816(d, e0, e1, e2, e3, b.z, b.w, d);
        if constexpr (!PAIRED) {
          const uint4 l = blk ? lB : lA;
          mma16816(d, a0, a1, a2, a3, l.x, l.y, d);
          mma16816(d, e0, e1, e2, e3, l.z, l.w, d);
        }
        const float sgv = blk ? sg.y : sg.x, s8v = blk ? s8.y : s8.x;
        acc[0] = fmaf(sgv, d[0], acc[0]);
        acc[1] = fmaf(sgv, d[1], acc[1]);
        acc[2] = fmaf(s8v, d[2], acc[2]);
        acc[3] = fmaf(s8v, d[3], acc[3]);
      }
    }
  } else {
#pragma unroll 1
    for (int ks = k0; ks < k1; ++ks) {
      const uint8_t* ch = st + ks * Fmt<2>::kChunk;
      const uint4 cw = *reinterpret_cast<const uint4*>(ch + lane * 16);
      const uint4 sa = *reinterpret_cast<const uint4*>(ch + 512 + g * 32);       // s(g, b0..b7)
      const uint4 sb = *reinterpret_cast<const uint4*>(ch + 512 + g * 32 + 16);  // s(g+8, b0..b7)
      const uint32_t cwv[4] = {cw.x, cw.y, cw.z, cw.w};
      const uint32_t sav[4] = {sa.x, sa.y, sa.z, sa.w};
      const uint32_t sbv[4] = {sb.x, sb.y, sb.z, sb.w};
      const __half* bp = bm + ((ks * 8 + g) * 4 + c) * 32;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = cwv[j], w2 = w >> 8;
        const uint4 b = *reinterpret_cast<const uint4*>(bp + 8 * j);
        const float2 sgp = __half22float2(*reinterpret_cast<const __half2*>(&sav[j]));
        const float2 s8p = __half22float2(*reinterpret_cast<const __half2*>(&sbv[j]));
        float d[4];
        {
          const uint32_t a0 = dq_pair(w, 0x00030003u), a1 = dq_pair(w2, 0x00030003u);
          const uint32_t a2 = dq_pair(w, 0x000C000Cu), a3 = dq_pair(w2, 0x000C000Cu);
          mma16816(d, a0, a1, a2, a3, b.x, b.y, z4);
          if constexpr (!PAIRED) {
            const uint4 l = *reinterpret_cast<const uint4*>(bp + bm_set + 8 * j);
            mma16816(d, a0, a1, a2, a3, l.x, l.y, d);
          }
          acc[0] = fmaf(sgp.x, d[0], acc[0]);
          acc[1] = fmaf(sgp.x, d[1], acc[1]);
          acc[2] = fmaf(s8p.x, d[2], acc[2]);
          acc[3] = fmaf(s8p.x, d[3], acc[3]);
        }
        {
          const uint32_t a0 = dq_pair(w, 0x00300030u), a1 = dq_pair(w2, 0x00300030u);
          const uint32_t a2 = dq_pair(w, 0x00C000C0u), a3 = dq_pair(w2, 0x00C000C0u);
          mma16816(d, a0, a1, a2, a3, b.z, b.w, z4);
          if constexpr (!PAIRED) {
            const uint4 l = *reinterpret_cast<const uint4*>(bp + bm_set + 8 * j);
            mma16816(d, a0, a1, a2, a3, l.z, l.w, d);
          }
          acc[0] = fmaf(sgp.y, d[0], acc[0]);
          acc[1] = fmaf(sgp.y, d[1], acc[1]);
          acc[2] = fmaf(s8p.y, d[2], acc[2]);
          acc[3] = fmaf(s8p.y, d[3], acc[3]);
        }
      }
    }
  }
  // min term: sum over blocks of min(row, block) * (activation block sum)
  const uint8_t* mins = st + nks * Fmt<BITS>::kChunk;
  for (int mk = m0; mk < m1; ++mk) {
    const uint4 am = *reinterpret_cast<const uint4*>(mins + mk * 512 + lane * 16);
    const __half* sp = bs + ((mk * 8 + g) * 4 + c) * 4;
    const uint2 b = *reinterpret_cast<const uint2*>(sp);
    mma16816(acc, am.x, am.y, am.z, am.w, b.x, b.y, acc);
    if constexpr (!PAIRED) {
      const uint2 l = *reinterpret_cast<const uint2*>(sp + bs_set);
      mma16816(acc, am.x, am.y, am.z, am.w, l.x, l.y, acc);
    }
  }
}

struct Task {
  bool shared;
  int expert;   // routed expert id (unused for shared)
  int tile;
};

__device__ __forceinline__ Task decode_task(long long task, int ntile_s, int ntile_e, const int* distinct) {
  Task t;
  if (task < ntile_s) {
    t.shared = true;
    t.expert = -1;
    t.tile = (int)task;
  } else {
    const long long q = task - ntile_s;
    t.shared = false;
    t.expert = __ldcg(distinct + q / ntile_e);
    t.tile = (int)(q % ntile_e);
  }
  return t;
}

// Copy the activation fragments of one group's rows into shared memory.
template <int BITS, int PHASE>
__device__ void load_group_B(const LayerDev& L, const WindowBufs& W, const Plan* P, const SmemCfg& C, __half* bm,
                             __half* bs, bool is_shared, int R, int ent_off, int K, int ctid) {
  constexpr int S = Fmt<BITS>::kBHalves;
  const int nks = K / Fmt<BITS>::kKstep;
  const int nblk = K / Fmt<BITS>::kBlock;
  const int nmk = (nblk + 15) / 16;
  const bool paired = R <= 4;
  const int nsets = paired ? 1 : 2;
  const long long fh = frag_halves(K, nmk);
  auto vec_index = [&](int r) -> int {
    if (is_shared) return r;
    const int ent = __ldcg(P->entries + ent_off + r);
    return PHASE == 0 ? ent / L.k : ent;
  };
  auto vec_base = [&](int r) -> const __half* {
    const int v = vec_index(r);
    if (PHASE == 0) return W.xfrag + v * fh;
    return (is_shared ? W.shfrag : W.hfrag) + v * fh;
  };
  constexpr int per = 4 * S / 8;  // uint4 per (k-step, column)
  const int total = nsets * 8 * nks * per;
  for (int i = ctid; i < total; i += kConsumerWarps * 32) {
    const int q = i % per;
    int rest = i / per;
    const int ks = rest % nks;
    rest /= nks;
    const int col = rest % 8, set = rest / 8;
    const int r = paired ? (col >> 1) : col;
    const int part = paired ? (col & 1) : set;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < R) v = __ldcg(reinterpret_cast<const uint4*>(vec_base(r) + (long long)part * K + ks * 4 * S) + q);
    *(reinterpret_cast<uint4*>(bm + set * C.bmain_halves + (ks * 8 + col) * 4 * S) + q) = v;
  }
  if (PHASE == 0) {
    const int tot = nsets * 8 * nmk * 2;
    for (int i = ctid; i < tot; i += kConsumerWarps * 32) {
      const int q = i & 1;
      int rest = i >> 1;
      const int mk = rest % nmk;
      rest /= nmk;
      const int col = rest % 8, set = rest / 8;
      const int r = paired ? (col >> 1) : col;
      const int part = paired ? (col & 1) : set;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < R)
        v = __ldcg(reinterpret_cast<const uint4*>(vec_base(r) + 2LL * K + (long long)part * 16 * nmk + mk * 16) + q);
      *(reinterpret_cast<uint4*>(bs + set * C.bsum_halves + (mk * 8 + col) * 16) + q) = v;
    }
  } else {
    // block sums of h from the per-16 partial sums written by phase 0
    const int nparts = (is_shared ? L.Fs : L.F) / 16;
    const int tot = nsets * 8 * nmk * 16;
    for (int i = ctid; i < tot; i += kConsumerWarps * 32) {
      const int slot = i & 3, c = (i >> 2) & 3;
      int rest = i >> 4;
      const int mk = rest % nmk;
      rest /= nmk;
      const int col = rest % 8, set = rest / 8;
      const int r = paired ? (col >> 1) : col;
      const int part = paired ? (col & 1) : set;
      const int beta = frag_sum_block(mk, c, slot);
      float s = 0.f;
      if (r < R && beta < nblk) {
        const float* pp = (is_shared ? W.shpart : W.hpart) + (long long)vec_index(r) * nparts;
        if (BITS == 4) s = __ldcg(pp + 2 * beta) + __ldcg(pp + 2 * beta + 1);
        else s = __ldcg(pp + beta);
      }
      __half hi, lo;
      split_hi_lo(s, hi, lo);
      bs[set * C.bsum_halves + ((mk * 8 + col) * 4 + c) * 4 + slot] = part ? lo : hi;
    }
  }
}

}  // namespace

template <int BITS, int PHASE>
__global__ void __launch_bounds__(kExpertThreads, 1) expert_kernel(LayerDev L, WindowBufs W, SmemCfg C) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  }
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();

  const Plan* P = W.plan;
  const int nd = __ldcg(&P->n_distinct);
  const bool has_shared = L.Fs > 0;
  const int ntile_s = has_shared ? (PHASE == 0 ? L.Fs : L.d) / 16 : 0;
  const int ntile_e = (PHASE == 0 ? L.F : L.d) / 16;
  const long long ntask = ntile_s + (long long)nd * ntile_e;
  const long long t0 = ntask * blockIdx.x / gridDim.x;
  const long long t1 = ntask * (blockIdx.x + 1) / gridDim.x;
  constexpr int kTilesPerTask = PHASE == 0 ? 2 : 1;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (long long task = t0; task < t1 && ok; ++task) {
        const Task tk = decode_task(task, ntile_s, ntile_e, P->distinct);
        if (!tk.shared && (unsigned)tk.expert >= (unsigned)L.E) {
          atomicOr(W.err, kErrIndex);
          s_abort = 1;
          ok = false;
          break;
        }
        for (int h = 0; h < kTilesPerTask; ++h) {
          const PackedMat& M = PHASE == 0 ? (h == 0 ? (tk.shared ? L.sgate : L.gate) : (tk.shared ? L.sup : L.up))
                                          : (tk.shared ? L.sdown : L.down);
          const int stage = it % C.nstages;
          if (it >= C.nstages) {
            if (!wait_full(&empty[stage], ((it / C.nstages) - 1) & 1, W.err, &s_abort)) {
              ok = false;
              break;
            }
          }
          const uint8_t* src = M.base + (tk.shared ? 0LL : (long long)tk.expert * M.mat_bytes) +
                               (long long)tk.tile * M.tile_bytes;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)M.tile_bytes);
          bulk_g2s(ring + (size_t)stage * C.stage_bytes, src, (uint32_t)M.tile_bytes, &full[stage]);
          ++it;
        }
      }
      if (s_abort) {
        // Let every copy this warp issued land before the CTA can exit.
        for (int j = (it > C.nstages ? it - C.nstages : 0); j < it; ++j) {
          const int stage = j % C.nstages;
          const long long tw = clock64();
          while (!mbar_try_wait(&full[stage], (j / C.nstages) & 1)) {
            if (clock64() - tw > (1LL << 31)) break;
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp;
  int it = 0;
  int cur = -2;
  int R = 0, ent_off = 0;
  bool paired = true;
  for (long long task = t0; task < t1; ++task) {
    const Task tk = decode_task(task, ntile_s, ntile_e, P->distinct);
    const int group = tk.shared ? -1 : tk.expert;
    if ((unsigned)(group + 1) > (unsigned)L.E) break;  // guarded by the producer too
    const int K = PHASE == 0 ? L.d : (tk.shared ? L.Fs : L.F);
    if (group != cur) {
      consumer_sync();
      if (tk.shared) {
        R = W.T;
        ent_off = 0;
      } else {
        R = __ldcg(P->counts + tk.expert);
        ent_off = __ldcg(P->offsets + tk.expert);
      }
      if (R < 1 || R > kMaxRows) { atomicOr(W.err, kErrIndex); R = R < 1 ? 1 : kMaxRows; }
      paired = R <= 4;
      load_group_B<BITS, PHASE>(L, W, P, C, bm, bs, tk.shared, R, ent_off, K, tid);
      consumer_sync();
      cur = group;
    }
    const int nks = K / Fmt<BITS>::kKstep;
    const int nmk = (K / Fmt<BITS>::kBlock + 15) / 16;
    const int k0 = cw * nks / kConsumerWarps, k1 = (cw + 1) * nks / kConsumerWarps;
    const int m0 = cw * nmk / kConsumerWarps, m1 = (cw + 1) * nmk / kConsumerWarps;
#pragma unroll 1
    for (int h = 0; h < kTilesPerTask; ++h) {
      const int stage = it % C.nstages;
      const bool ok = wait_full(&full[stage], (it / C.nstages) & 1, W.err, &s_abort);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (ok) {
        const uint8_t* st = ring + (size_t)stage * C.stage_bytes;
        if (paired)
          tile_mma<BITS, true>(st, bm, bs, C.bmain_halves, C.bsum_halves, nks, k0, k1, m0, m1, lane, acc);
        else
          tile_mma<BITS, false>(st, bm, bs, C.bmain_halves, C.bsum_halves, nks, k0, k1, m0, m1, lane, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      red[(h * kConsumerWarps + cw) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      ++it;
    }
    consumer_sync();

    // ---------------- epilogue: cross-warp sums in a fixed order ----------------
    const int r = tid >> 4, row = tid & 15;
    const bool valid = tid < 128 && r < R;
    float v0 = 0.f, v1 = 0.f;
    if (valid) {
      const int src_lane = (row & 7) * 4 + (paired ? r : (r >> 1));
      const int idx = ((row >> 3) << 1) + (paired ? 0 : (r & 1));
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float4 a = red[w * 32 + src_lane];
        const float* af = reinterpret_cast<const float*>(&a);
        v0 += paired ? (af[idx] + af[idx + 1]) : af[idx];
        if (PHASE == 0) {
          const float4 b = red[(kConsumerWarps + w) * 32 + src_lane];
          const float* bf = reinterpret_cast<const float*>(&b);
          v1 += paired ? (bf[idx] + bf[idx + 1]) : bf[idx];
        }
      }
    }
    if (PHASE == 0) {
      if (tid < 128) {
        const float hval = valid ? silu_f32(v0) * v1 : 0.f;
        const int Kd = tk.shared ? L.Fs : L.F;
        const int nmk_d = (Kd / Fmt<BITS>::kBlock + 15) / 16;
        const long long fh = frag_halves(Kd, nmk_d);
        int vec = 0;
        if (valid) {
          vec = tk.shared ? r : __ldcg(P->entries + ent_off + r);
          __half* base = (tk.shared ? W.shfrag : W.hfrag) + vec * fh;
          int off;
          float fac;
          frag_main_pos<BITS>(tk.tile * 16 + row, off, fac);
          __half hi, lo;
          split_hi_lo(hval * fac, hi, lo);
          base[off] = hi;
          base[Kd + off] = lo;
        }
        float s = hval;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (valid && row == 0) {
          float* part = tk.shared ? W.shpart + (long long)vec * (L.Fs / 16) : W.hpart + (long long)vec * (L.F / 16);
          part[tk.tile] = s;
        }
      }
    } else {
      const int drow = tk.tile * 16 + row;
      if (valid) {
        if (tk.shared) {
          W.sbuf[(long long)r * L.d + drow] = v0;
        } else {
          const int ent = __ldcg(P->entries + ent_off + r);
          W.obuf[(long long)ent * L.d + drow] = __ldcg(P->topk_w + ent) * v0;
        }
        __threadfence();
      }
      consumer_sync();
      if (tid == 0) {
        const int ngroups = (has_shared ? 1 : 0) + nd;
        s_last = (atomicAdd(W.counters + tk.tile, 1) == ngroups - 1);
      }
      consumer_sync();
      if (s_last) {
        __threadfence();
        const int T = W.T, k = L.k;
        for (int i = tid; i < T * 16; i += kConsumerWarps * 32) {
          const int t = i >> 4, rr = tk.tile * 16 + (i & 15);
          float y = has_shared ? __ldcg(W.sbuf + (long long)t * L.d + rr) : 0.f;
          for (int j = 0; j < k; ++j) y += __ldcg(W.obuf + (long long)(t * k + j) * L.d + rr);
          W.y[(long long)t * L.d + rr] = y;
        }
      }
    }
    consumer_sync();
  }
}

SmemCfg expert_smem_cfg(const LayerDev& L, int phase, int max_rows, int smem_limit) {
  SmemCfg C{};
  const int bits = L.bits;
  const int kstep = bits == 4 ? 64 : 128, block = bits == 4 ? 32 : 16;
  const int S = bits == 4 ? 16 : 32;
  auto tb = [&](int K) { return bits == 4 ? tile_bytes_of<4>(K) : tile_bytes_of<2>(K); };
  int Kmax;
  if (phase == 0) {
    Kmax = L.d;
    C.stage_bytes = tb(L.d);
  } else {
    Kmax = L.Fs > L.F ? L.Fs : L.F;
    C.stage_bytes = tb(L.F);
    if (L.Fs > 0 && tb(L.Fs) > C.stage_bytes) C.stage_bytes = tb(L.Fs);
  }
  const int nks = Kmax / kstep;
  const int nmk = (Kmax / block + 15) / 16;
  C.bmain_halves = nks * 8 * 4 * S;
  C.bsum_halves = nmk * 8 * 4 * 4;
  C.nsets = max_rows > 4 ? 2 : 1;
  const int fixed = C.nsets * (C.bmain_halves + C.bsum_halves) * 2 + 2 * kConsumerWarps * 32 * 16 + 2 * kMaxStages * 8;
  int ns = (smem_limit - fixed) / C.stage_bytes;
  if (ns > kMaxStages) ns = kMaxStages;
  C.nstages = ns;
  C.total_bytes = ns * C.stage_bytes + fixed;
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
