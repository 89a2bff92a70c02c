// Device-side definitions shared by the window kernels: packed tile format,
// window workspace layout, and thin PTX wrappers (mbarrier, bulk async copy,
// programmatic dependent launch, mma.sync, lop3).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace strata {

constexpr int kMaxRows = 8;       // a verify window holds at most 8 rows
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 256;
constexpr int kMaxEntries = kMaxRows * kMaxTopK;
constexpr int kConsumerWarps = 16;
constexpr int kExpertThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kRouterThreads = 256;
constexpr int kMaxStages = 8;

// Bits of the device error word.
enum : uint32_t {
  kErrTimeout = 1u,     // a bounded wait gave up
  kErrIndex = 2u,       // an index derived from routing was out of range
  kErrNonFinite = 4u,   // a router logit was not finite
  kErrConfig = 8u,      // a launch saw an impossible configuration
};

// ---------------------------------------------------------------------------
// Packed tile format.
//
// A quantized matrix [rows][K] (rows % 16 == 0, K % kstep == 0) is stored as
// rows/16 tiles of 16 rows.  A tile is nks "k-steps" followed by nmk min
// fragments:
//   k-step (576 B for 4-bit, 768 B for 2-bit):
//     512 B codes: 32 lanes x 16 B, lane (g = lane/4, c = lane%4) holds the
//                  A-operand codes of rows g and g+8 for its k-slots;
//     scales: 8 records (one per g): 4-bit: s(g,b0) s(g,b1) s(g+8,b0) s(g+8,b1)
//             2-bit: s(g,b0..b7) then s(g+8,b0..b7)   (fp16)
//   min fragment (512 B per 16 blocks): lane (g,c) holds the mins of rows
//     g, g+8 for blocks 2c, 2c+1, 2c+8, 2c+9 in mma A-fragment order (fp16,
//     blocks past the end are zero).
// Code words: each 32-bit word holds pairs of codes at bits (p, p+16) so that
// one AND yields an fp16x2 of subnormals f*q*2^-24 (see dq_pair).
//   4-bit word (one row, one block, lane c covers elements 8c..8c+7):
//     bits 0/16: e0,e1   4/20: e2,e3 (x16)   8/24: e4,e5   12/28: e6,e7 (x16)
//   2-bit word (rows g and g+8, two blocks b0,b1, lane c covers elements 4c..4c+3):
//     pair p at bits (2p, 2p+16): p=0 g/b0 e0,e1; p=1 g/b0 e2,e3 (x4);
//     p=2 g/b1 e0,e1 (x16); p=3 g/b1 e2,e3 (x64); p=4..7 the same for row g+8.
// The activation (B operand) records carry the inverse power-of-two factors.
// ---------------------------------------------------------------------------
template <int BITS> struct Fmt;
template <> struct Fmt<4> {
  static constexpr int kBlock = 32, kKstep = 64, kBlocksPerKstep = 2;
  static constexpr int kScaleRec = 8;      // bytes per g in a k-step
  static constexpr int kChunk = 512 + 8 * kScaleRec;   // 576
  static constexpr int kBHalves = 16;      // B halves per (k-step, lane c)
};
template <> struct Fmt<2> {
  static constexpr int kBlock = 16, kKstep = 128, kBlocksPerKstep = 8;
  static constexpr int kScaleRec = 32;
  static constexpr int kChunk = 512 + 8 * kScaleRec;   // 768
  static constexpr int kBHalves = 32;
};

// One packed matrix stack [n][rows][K].
struct PackedMat {
  const uint8_t* base;
  int rows, K, nks, nmk;
  int tile_bytes;          // nks*chunk + nmk*512
  long long mat_bytes;     // (rows/16) * tile_bytes
};

// Activation fragments of one vector of length K:
//   main hi [nks][4][S] halves, main lo [nks][4][S], sums hi [nmk][4][4],
//   sums lo [nmk][4][4].  Size in halves: 2*K + 32*nmk.
__host__ __device__ inline long long frag_halves(int K, int nmk) { return 2LL * K + 32LL * nmk; }

struct LayerDev {
  int d, E, k, F, Fs, bits, renorm;
  const float* router_w;   // [E][d]
  const float* router_b;   // [E] or null
  PackedMat gate, up, down, sgate, sup, sdown;
  // dense attention projections of a decoder layer (stack kernel only):
  // qkv = [Wq; Wk; Wv] as one [dq + 2 dkv][d] matrix, o = Wo [d][dq]
  PackedMat qkv, o;
  int dq, dkv;             // query width (heads x head_dim) and kv width
  int kph_log2, kpg_log2;  // log2 of the o-projection k-steps per head / per kv group
};

// Adaptive expert tier state that windows update (device pointers; a null
// `counters` means no tier is attached).  Counters are fp32 routed-entry
// counts aged by `decay` after every round; a round every `adapt_every`
// windows swaps up to `adapt_swaps` experts between the tier and the rest.
struct TierDev {
  float* counters;          // [E]
  int* resident;            // [E] 1 = in the tier
  long long* windows;       // windows counted so far
  long long* rounds;        // rounds run so far
  int* n_swaps;             // swaps made by the last round
  int* swap_in;             // [E] experts the last round moved in (first n_swaps)
  int* swap_out;            // [E] experts it moved out, pairwise with swap_in
  int adapt_every, adapt_swaps;
  float decay, min_gain;
};

// A stack window's attention over each slot's KV cache (stack kernel only; a
// null k means the length-one reading: every query head outputs v of its kv
// head).  The caches are the caller's; the rest is the stack's scratch.
struct KVDev {
  __half* k;               // [n_layers][n_slots][kv_heads][max_ctx][head_dim] fp16
  __half* v;               // the same for values
  int n_slots, max_ctx, head_dim;
  int nch;                 // chunks of kAttnChunk positions in max_ctx (rounded up)
  const int* slot;         // [T] each row's slot
  const int* pos;          // [T] each row's position
  float* qbuf;             // [kMaxRows][dq] the rows' q
  float* kbuf;             // [kMaxRows][dkv] the rows' k
  float* part;             // [kMaxRows][heads][nch][head_dim + 2] per-chunk partials (o, max, sum)
  __half* afrag;           // the o projection's B operand (att), in the shared-memory B layout, 2 sets
  int afrag_set;           // halves per set of afrag (8 x dq)
  float* asum;             // [kMaxRows][dq / block] block sums of att
};
constexpr int kAttnChunk = 64;  // cache positions per attention work item

struct WindowBufs {
  const float* x;          // [T][d]
  float* y;                // [T][d]
  int T;
  // caller's optional routing outputs (device pointers, each may be null)
  int* out_topk_idx; float* out_topk_w; int* out_counts; int* out_offsets;
  int* out_entries; int* out_distinct; int* out_ndistinct;
  // workspace
  __half* xfrag;           // x fragments of the T rows as one B image (16 d + 256 nmk halves)
  // h = silu(Wg x) * (Wu x) of each routed entry, written by the gate/up
  // epilogue already in activation-fragment form: fp16 hi then lo parts of
  // F elements each (the x-fragment main layout), plus fp32 sums of h over
  // every 16 consecutive elements (block sums are 1 or 2 of these)
  __half* hfrag;           // [kMaxEntries][2F]
  float* hsum;             // [kMaxEntries][F/16]
  __half* shfrag;          // [kMaxRows][2Fs] the same for the shared expert
  float* shsum;            // [kMaxRows][Fs/16]
  float* obuf;             // [kMaxEntries][d]
  float* sbuf;             // [kMaxRows][d]
  int* counters;           // [d/16] contributions landed per 16-row slice of y
  int* done_gu;            // [E+1] finished gate/up tasks per group (shared first)
  unsigned long long* gbar;  // grid barrier arrivals (monotonic across windows)
  float* partial;          // router partial logits [njb][kMaxRows][E]
  int njb;                 // column chunks of the router GEMV
  unsigned* err;
  TierDev tier;            // adaptive tier bookkeeping (single-layer windows; counters null = none)
  KVDev kv;                // attention over KV caches (stack kernel; k null = the length-one reading)
  long long wait_cycles;   // limit of every bounded device wait, in SM clock cycles
  int bar_extra;           // arrivals a grid barrier expects beyond the grid (0; > 0 only in failure tests)
  // decoder-layer extras (stack kernel only; null in the single-layer kernel)
  const float* rinv;       // [T] 1 / RMS of each row of x (inputs are x * rinv)
  const float* resid;      // [T][d] added to y in the combine
  float* v;                // [kMaxRows][dkv] value projection
  float* x1;               // [kMaxRows][d] x + Wo att
  __half* vimg;            // the o phase's length-one B operand: v as one B image (16 dkv halves), or null
  float* vsum;             // [kMaxRows][dkv / block] v's block sums (zeroed in D0, added by D1's epilogue)
  float* q_out;            // [T][dq] or null
  float* k_out;            // [T][dkv] or null
};

// Per-row token draw of the output head and its proposal check (head kernel
// only; all device pointers, arrays of the window's T rows).
struct HeadArgs {
  const int* position;               // [T] position whose token the row draws (Philox counter)
  const unsigned long long* seed;    // [T] the row's seed (Philox key)
  const float* temperature;          // [T] <= 0: greedy
  const int* fed;                    // [T] the proposal the row was fed; -1 for a slot's first row
  int* tokens;                       // [T] out: the row's token
  int* n_emit;                       // [T] out: tokens the slot emits, at its first row (0 elsewhere)
  float* part_max;                   // [grid][kMaxRows] scratch: per-CTA slice maxima
  int* part_arg;                     // [grid][kMaxRows] scratch: their tokens
  float* part_sum;                   // [grid][kMaxRows] scratch: per-CTA slice sums of exp
  int V;                             // vocabulary (rows of the head matrix)
};

constexpr int kMaxChunks = 32;  // k-chunks per tile

// How one phase (0 gate/up, 1 down, 2 dense q/k/v, 3 dense o) cuts its tiles
// into ring stages.
struct PhaseCfg {
  int nchunks;             // k-chunks per tile
  int sub_stride;          // bytes per sub-tile inside a stage
  int mins_off;            // offset of the mins part inside a sub-tile slot
  int max_sub;             // most sub-tiles a task may hold (stage sizing)
  short cks[2][kMaxChunks + 1];  // k-step bounds of each chunk: [0] routed K, [1] shared K
  short cmk[2][kMaxChunks + 1];  // min-group bounds of each chunk
};

// Shared-memory plan of the window kernel.
struct KernelCfg {
  int nstages;
  int stage_bytes;         // one stage: up to max_sub sub-tiles' k-chunk (codes+scales, then mins)
  int bmain_halves;        // B main halves per set: 8 * max K
  int bsum_halves;         // B sums halves per set: nmk_max*8*4*4
  int nsets;               // 1 (rows <= 4) or 2
  int total_bytes;
  int direct;              // window kernel on the register-fed path (no producer, no ring)
  PhaseCfg ph[4];
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (L2 only), and the wait for all
// of this thread's outstanding ones.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// The waiting thread may be suspended (up to ~0.1 ms per call) instead of
// spinning, so waiting warps leave the issue slots to the working ones.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
#ifdef STRATA_TRYWAIT_NOHINT
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(100000u)
      : "memory");
#endif
  return ok != 0;
}
// Bounded wait: gives up after ~2^31 cycles (about a second), sets the error
// word and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1LL << 31)) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// Bulk async copy global -> this CTA's shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Named barrier among the consumer warps only (the producer warp keeps running).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Two codes at bits (p, p+16) -> an fp16x2 of exact subnormals f*q*2^-24
// (exponent field zero, the code in the low mantissa bits).  The tensor cores
// take fp16 subnormal operands exactly, so one AND dequantizes a pair; the
// 2^-24 is undone once per output.
__device__ __forceinline__ uint32_t dq_pair(uint32_t w, uint32_t mask) { return w & mask; }
constexpr float kDqUnscale = 16777216.0f;  // 2^24

// D = A * B + C, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// hi = fp16(v), lo = fp16(v - hi)
__device__ __forceinline__ void split_hi_lo(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

}  // namespace strata
