/*
 * strata_window.h -- C ABI of a GB300 (sm_103a) library that runs the batched
 * verify-window MoE decode step.
 *
 * What a window is (the Strata docs, "BATCHING.md", section "Several requests
 * at once (batch slots)", opening paragraph): every verify window carries one
 * token of each open conversation, so the dense weights, the shared expert and
 * every routed expert two conversations share are read once per window for all
 * of them.  A window holds at most 8 rows (same page, option table: "a window
 * holds 8 rows"); with --batch-mtp each slot adds its MTP proposal as a second
 * row (same page, --batch-mtp paragraph).  Section "Exactness": a batch row's
 * arithmetic is the single-token window's.
 *
 * One MoE layer of a window, as this library computes it (the pages give no
 * formulas; these are the readings the library implements):
 *   logit[t][e] = sum_j Wr[e][j] x[t][j] + b[e]                 (fp32)
 *   p[t]        = softmax(logit[t]) over all E experts           (fp32)
 *   sel[t]      = the top_k experts by logit, descending, ties to the lower id
 *   g[t][j]     = p[t][sel[t][j]]  (or renormalised over the k when renorm_topk)
 *   h           = silu(Wg_e x_t) * (Wu_e x_t),  silu(z) = z / (1 + e^-z)
 *   y[t]        = shared(x_t) + sum_j g[t][j] * Wd_e h          (e = sel[t][j])
 * where shared() is the same SwiGLU FFN with weight 1 and no gate.
 *
 * Block format of a quantized matrix [rows][cols]: blocks of `block` elements
 * along cols; per block `block*bits/8` code bytes (element i of a row in byte
 * i*bits/8, least-significant bits first: for 4-bit the even element is the
 * low nibble), one fp16 scale and one fp16 min; weight = scale*q + min.  Codes
 * are row-major [rows][cols*bits/8]; scale and min are fp16 bit patterns
 * [rows][cols/block].  Supported: bits=4 with block=32, bits=2 with block=16.
 *
 * Errors: every call returns a status and never aborts.  Argument errors are
 * found on the host before any GPU work.  Errors the GPU detects (a bounded
 * wait that gave up, an index guard, a non-finite router logit) are recorded
 * in a device error word and returned by the next strata_window_sync().
 */
#ifndef STRATA_WINDOW_H
#define STRATA_WINDOW_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  STRATA_OK = 0,
  STRATA_EINVAL = 1,        /* a bad argument; nothing was launched */
  STRATA_ENOMEM = 2,        /* a device allocation failed */
  STRATA_ECUDA = 3,         /* a CUDA runtime call failed */
  STRATA_EUNSUPPORTED = 4,  /* a valid but unsupported shape or format */
  STRATA_EDEVICE = 5        /* the GPU flagged an error during an earlier call */
} strata_status;

typedef struct strata_window strata_window; /* opaque handle */

/* One stack of quantized matrices in the block format above.  All three are
 * device pointers.  For a stack of n matrices the arrays are the n matrices
 * back to back ([n][rows][...]). */
typedef struct {
  const void* codes;      /* uint8 [n][rows][cols*bits/8] */
  const uint16_t* scale;  /* fp16 bits [n][rows][cols/block] */
  const uint16_t* min;    /* fp16 bits [n][rows][cols/block] */
} strata_qmat;

/* Shape of one MoE layer. */
typedef struct {
  int32_t hidden;       /* d: multiple of 64 (4-bit) or 128 (2-bit) */
  int32_t n_experts;    /* E: 1..256 */
  int32_t top_k;        /* k: 1..min(E, 8) */
  int32_t ffn;          /* F: routed expert width, multiple of 64 (4-bit) or 128 (2-bit) */
  int32_t shared_ffn;   /* Fs: shared expert width (same rule), 0 = no shared expert */
  int32_t bits;         /* 4 or 2 */
  int32_t block;        /* 32 (with bits=4) or 16 (with bits=2) */
  int32_t max_rows;     /* largest window this handle serves: 1..8 */
  int32_t renorm_topk;  /* 0: gate = softmax prob over all E; 1: renormalised over the k */
} strata_moe_desc;

/* Weights of one layer (device pointers).  They are read during
 * strata_window_create only: create copies them into the handle's own
 * kernel-ordered layout, so the caller may free them once create returns. */
typedef struct {
  const float* router_w;    /* fp32 [E][d] */
  const float* router_b;    /* fp32 [E], or NULL for no bias */
  strata_qmat gate;         /* [E][F][d] */
  strata_qmat up;           /* [E][F][d] */
  strata_qmat down;         /* [E][d][F] */
  strata_qmat shared_gate;  /* [1][Fs][d]  (ignored when shared_ffn == 0) */
  strata_qmat shared_up;    /* [1][Fs][d] */
  strata_qmat shared_down;  /* [1][d][Fs] */
} strata_moe_weights;

/* Optional routing outputs of a forward call (device pointers; each may be
 * NULL).  Entries are numbered t*k + j (row t, j-th selected expert). */
typedef struct {
  int32_t* topk_idx;    /* [T][k] selected experts, descending logit */
  float* topk_w;        /* [T][k] gate weights */
  int32_t* counts;      /* [E] entries per expert */
  int32_t* offsets;     /* [E+1] exclusive prefix sum of counts */
  int32_t* entries;     /* [T*k] entries grouped by expert (ascending), ascending within an expert */
  int32_t* distinct;    /* [E] experts with count > 0, ascending (first n_distinct valid) */
  int32_t* n_distinct;  /* [1] */
} strata_routing_out;

/* Sizes a handle chose (for measurement and tests). */
typedef struct {
  int32_t n_sm;               /* SMs of the device (CTAs of the window kernel) */
  int32_t stages;             /* shared-memory ring stages of the window kernel; 1 when the handle uses the
                                 warp-streamed path (no ring, per-warp copy FIFOs: 2-bit layers, and 4-bit
                                 layers whose activations leave a ring under three 32 KB stages) */
  int32_t stage_bytes;        /* bytes per ring stage (warp-streamed path: the FIFO region) */
  int32_t smem_bytes;         /* dynamic shared memory bytes per CTA */
  int64_t packed_bytes;       /* bytes of the handle's kernel-ordered weights */
  int64_t expert_bytes;       /* block-format bytes of one routed expert (gate+up+down) */
  int64_t shared_bytes;       /* block-format bytes of the shared expert */
  int64_t router_bytes;       /* router weight (+ bias) bytes */
  int64_t workspace_bytes;    /* handle scratch bytes */
} strata_window_info;

/* Create a handle for one MoE layer on the current CUDA device.
 *   desc, weights: as above; weights are read on `cuda_stream` (a cudaStream_t,
 *   or NULL for the default stream) and create waits for that work to finish.
 *   out: receives the handle; set to NULL on failure.
 * The handle picks its window kernel here (see strata_window_info.stages).
 * Two environment variables, read at this call, override the choice for
 * comparisons: STRATA_WINDOW_RING (any value) forces the ring path;
 * STRATA_WINDOW_DIRECT (any value) forces the warp-streamed path where the
 * shape allows it (every warp gets a k-step of each task).  Results of the two
 * paths agree within the output tolerance, not bit for bit.
 * Two more variables, also read here, bound the device's waits:
 * STRATA_WAIT_CYCLES (an integer from 1000 to 2^40; default 2^31, about a
 * second at GB300 clocks) is the limit of every bounded wait of the kernel,
 * in SM clock cycles; STRATA_TEST_BARRIER_EXTRA (default 0) makes every grid
 * barrier wait for that many arrivals that never come.  They exist so that
 * failure tests can make a wait run out: each CTA then gives up after the
 * limit, records EDEVICE and returns.  Malformed values are ignored.
 * Returns EINVAL (bad pointer or shape), EUNSUPPORTED (bits/block pair or size
 * limits), ENOMEM, ECUDA. */
strata_status strata_window_create(const strata_moe_desc* desc, const strata_moe_weights* weights,
                                   void* cuda_stream, strata_window** out);

/* The window-kernel plan a handle for this layer shape would choose, computed
 * on the host with no device and no CUDA call: fills stages, stage_bytes and
 * smem_bytes of *info as strata_window_query would report them (stages = 1:
 * the warp-streamed path); every other field is set to 0.
 *   smem_limit: dynamic shared memory the window kernel may use per CTA, in
 *   bytes; 0 = what strata_window_create grants on a GB300 (the 232,448-byte
 *   opt-in maximum less 12,288 bytes kept for the kernel's static shared
 *   memory).  Create takes the device's own opt-in maximum instead.
 * Reads the same environment overrides as strata_window_create.
 * Returns EINVAL (NULL pointer, bad shape, negative limit) or EUNSUPPORTED
 * (no plan fits the limit: create would fail the same way). */
strata_status strata_window_plan(const strata_moe_desc* desc, int32_t smem_limit, strata_window_info* info);

/* The slots of the next window when more slots are open than one window
 * holds.  The Strata docs ("BATCHING.md", --batch-mtp paragraph): a window
 * carries each active slot's rows (its token, and its MTP proposal with
 * --batch-mtp), at most 8 rows, so at most four slots with proposals are in
 * one window, and more slots rotate through.  The rule here (a reading):
 * starting at slot `start`, slots are taken in cyclic order, each at most
 * once, while their rows still fit in max_rows; a slot with no rows is
 * skipped; the next window starts at the slot after the last one taken.  The
 * window's rows are the taken slots' rows in this order, each slot's rows
 * consecutive (token row, then proposal row), which is the layout
 * strata_head_forward's proposal check reads.
 *   rows_per_slot: host [n_slots], each 0..max_rows; slots_out: host
 *   [n_slots] receives the window's slots, *n_out their number;
 *   *next_start the next window's start.  Host only: no device is touched.
 * Returns EINVAL for a bad argument. */
strata_status strata_window_slots(int32_t n_slots, const int32_t* rows_per_slot, int32_t start, int32_t max_rows,
                                  int32_t* slots_out, int32_t* n_out, int32_t* next_start);

/* Run one window: y = MoE(x) for T rows.
 *   x: device fp32 [T][d], caller-owned; y: device fp32 [T][d], caller-owned,
 *   must not overlap x; both 16-byte aligned.  1 <= T <= desc.max_rows.
 *   routing: NULL, or a struct of optional device outputs.
 *   cuda_stream: the stream to enqueue on (NULL = default stream).
 * Asynchronous: returns once the work is enqueued.  One handle serves one
 * stream at a time (calls on the same handle must not overlap on the GPU). */
strata_status strata_moe_window_forward(strata_window* h, const float* x, int32_t T, float* y,
                                        const strata_routing_out* routing, void* cuda_stream);

/* Run one window like strata_moe_window_forward (no routing outputs) by
 * replaying a CUDA graph of the window launch.  The handle keeps a bounded
 * cache of 16 instantiated graphs keyed by (T, x, y): the first call with a
 * key captures and instantiates its graph (on a stream the handle owns),
 * later calls only launch it; the least recently used graph is evicted when
 * the cache is full.  The Strata pages' pull request on windows with MTP rows
 * describes eight-row windows run through a bounded batch graph cache; this
 * is that cache for the one-launch window.  Returns EINVAL as the plain
 * forward, ECUDA if capture, instantiation or launch fails. */
strata_status strata_moe_window_forward_graph(strata_window* h, const float* x, int32_t T, float* y,
                                              void* cuda_stream);

/* Wait for the handle's last forward call to finish; report (and clear) any
 * error the GPU recorded: EDEVICE in that case.  After an error the handle's
 * grid-barrier count is reset too (a window that gave up part way may have
 * left it off a multiple of the grid), so the next window starts clean. */
strata_status strata_window_sync(strata_window* h);

/* Fill *info with the sizes the handle chose. */
strata_status strata_window_query(const strata_window* h, strata_window_info* info);

/* Measurement aid.  With enable != 0 every later forward call also records
 * CUDA events on its stream right before and after its window kernel.
 * enable = 0 turns it off. */
strata_status strata_window_set_profiling(strata_window* h, int32_t enable);

/* Device time (ms) of the window kernel of the last profiled forward call;
 * waits for that call.  Returns EINVAL if profiling was never enabled. */
strata_status strata_window_timings(strata_window* h, float* ms);

/* ---------------------------------------------------------------------------
 * A window through a stack of decoder layers.
 *
 * Each layer: a = RMSNorm(x); q = Wq a, k = Wk a, v = Wv a; attention over a
 * context of one position, so query head h outputs v of kv head
 * h / (heads / kv_heads); x1 = x + Wo att; x_next = x1 + MoE(RMSNorm(x1)).
 * RMSNorm(x) = x / sqrt(mean(x^2) + 1e-6) with unit gain.  The Strata docs
 * ("BATCHING.md", "Several requests at once (batch slots)", opening
 * paragraph) name the dense weights among what a window reads once for all of
 * its rows; the pages give no attention or norm formulas, so these are the
 * plain readings (pre-norm, residual adds, no final norm).
 * ------------------------------------------------------------------------- */
typedef struct strata_stack strata_stack;

/* Dense attention shapes; the weights use the MoE desc's bits/block format.
 * heads % kv_heads == 0, (heads / kv_heads) and (head_dim / k-step) powers of
 * two, head_dim a multiple of the k-step (64 for 4-bit, 128 for 2-bit). */
typedef struct {
  int32_t heads, kv_heads, head_dim;
} strata_attn_desc;

typedef struct {
  strata_qmat q;  /* [heads*head_dim][hidden] */
  strata_qmat k;  /* [kv_heads*head_dim][hidden] */
  strata_qmat v;  /* [kv_heads*head_dim][hidden] */
  strata_qmat o;  /* [hidden][heads*head_dim] */
} strata_attn_weights;

/* Optional per-layer outputs of a stack window (device pointers, each may be NULL). */
typedef struct {
  float* q;              /* [n_layers][T][heads*head_dim] */
  float* k;              /* [n_layers][T][kv_heads*head_dim] */
  int32_t* topk_idx;     /* [n_layers][T][top_k] */
  float* topk_w;         /* [n_layers][T][top_k] */
  int32_t* n_distinct;   /* [n_layers] */
} strata_stack_out;

typedef struct {
  int32_t n_layers;
  int32_t n_sm, stages, stage_bytes, smem_bytes;
  int64_t dense_bytes;   /* block-format bytes of one layer's q, k, v, o */
  int64_t expert_bytes;  /* per routed expert, as strata_window_info */
  int64_t shared_bytes;
  int64_t router_bytes;
} strata_stack_info;

/* Create a stack of n_layers decoder layers, all with the shapes of `moe` and
 * `attn`; moe_w and attn_w point to n_layers weight sets (borrowed for the
 * duration of the call: the handle keeps its own kernel-ordered copies).
 * Returns EINVAL (bad pointer or shape), EUNSUPPORTED, ENOMEM, ECUDA. */
strata_status strata_stack_create(int32_t n_layers, const strata_moe_desc* moe, const strata_attn_desc* attn,
                                  const strata_moe_weights* moe_w, const strata_attn_weights* attn_w,
                                  void* cuda_stream, strata_stack** out);

/* Run one window of T rows through every layer: x device fp32 [T][hidden]
 * (caller-owned, 16-byte aligned), y device fp32 [T][hidden] (must not
 * overlap x, 16-byte aligned); out may be NULL.  One cooperative launch,
 * asynchronous on cuda_stream. */
strata_status strata_stack_forward(strata_stack* s, const float* x, int32_t T, float* y, const strata_stack_out* out,
                                   void* cuda_stream);

/* Attention over each slot's KV cache instead of the length-one reading.
 *
 * The Strata docs ("BATCHING.md", "Several requests at once (batch slots)")
 * keep one KV cache per conversation slot; a verify window carries one row per
 * slot, plus the slot's MTP proposal as a second row at the next position.
 * With a cache set, each layer of strata_stack_forward_kv does, after the
 * q/k/v projections: every row t (slot s_t, position p_t) stores its k and v,
 * rounded to fp16, at position p_t of its slot in that layer's cache; then
 * row t attends, for query head h, over positions 0..p_t of its slot with kv
 * head h / (heads / kv_heads): softmax_j(q_h . K_j / sqrt(head_dim)) applied
 * to the V_j (fp32 arithmetic; no position encoding, the pages name none).
 * A proposal row at p + 1 thus sees its token row's entry at p written in the
 * same window.  The o projection then reads this output in place of the
 * length-one broadcast of v.
 *   k, v: device fp16 bit patterns [n_layers][n_slots][kv_heads][max_ctx]
 *   [head_dim], caller-owned and 16-byte aligned; positions below a row's are
 *   the conversation's history, which the caller writes; the window writes
 *   its rows' entries.  The caches must outlive their use.
 * Requires head_dim a multiple of 32 and at most 128 (EUNSUPPORTED
 * otherwise).  The stack allocates its attention scratch here (ENOMEM).  NULL
 * drops the caches and frees that scratch. */
typedef struct {
  uint16_t* k;
  uint16_t* v;
  int32_t n_slots;
  int32_t max_ctx;
} strata_kv_cache;

strata_status strata_stack_set_kv(strata_stack* s, const strata_kv_cache* kv);

/* A window through every layer with attention over the caches set by
 * strata_stack_set_kv (EINVAL when none is set): slot and position are
 * device int32 [T].  Rows must have distinct (slot, position) pairs.  A row
 * whose slot or position is out of range is left out of the caches, attends
 * to nothing (zero attention output) and makes the next strata_stack_sync
 * report EDEVICE.  Otherwise as strata_stack_forward (which always uses the
 * length-one reading). */
strata_status strata_stack_forward_kv(strata_stack* s, const float* x, int32_t T, float* y, const int32_t* slot,
                                      const int32_t* position, const strata_stack_out* out, void* cuda_stream);

/* Wait for the last stack_forward; EDEVICE if the GPU recorded an error. */
strata_status strata_stack_sync(strata_stack* s);

strata_status strata_stack_query(const strata_stack* s, strata_stack_info* info);

/* Measurement aid, as strata_window_set_profiling / strata_window_timings. */
strata_status strata_stack_set_profiling(strata_stack* s, int32_t enable);
strata_status strata_stack_timings(strata_stack* s, float* ms);

/* Free the stack and everything it owns.  NULL is accepted. */
strata_status strata_stack_destroy(strata_stack* s);

/* Size of the one static scratch array that strata_moe_window_forward_noalloc
 * uses for every window on a device. */
#define STRATA_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Run one window like strata_moe_window_forward, but allocate nothing and use
 * none of the handle's workspace: the window's scratch (router partial logits,
 * x fragments, gate/up and down results, counters, the grid barrier word)
 * lives in one file-scope static device array of STRATA_NOALLOC_SCRATCH_BYTES
 * bytes.  The source pages describe no counterpart of this call; it exists
 * for callers that may not allocate device memory at call time.
 *   h: a handle created on the current device (EINVAL otherwise); its
 *   kernel-ordered weights are read, its error word records device errors
 *   (reported by strata_window_sync(h)) and its completion event is recorded.
 *   x, y, T, cuda_stream: as for strata_moe_window_forward; no routing outputs.
 * The scratch the handle's layer shape needs is computed on the host; above
 * STRATA_NOALLOC_SCRATCH_BYTES the call returns EUNSUPPORTED and launches
 * nothing.  The first call on a device looks the array's address up with
 * cudaGetSymbolAddress while that device is current; make that first call
 * before any stream capture.  Every call on a device shares the one array: the
 * parts that must start at zero (the grid barrier word and the x fragments)
 * are cleared by each call on its stream, and calls that overlap on the GPU
 * (any handle, any stream) race on the array. */
strata_status strata_moe_window_forward_noalloc(strata_window* h, const float* x, int32_t T, float* y,
                                                void* cuda_stream);

/* ---------------------------------------------------------------------------
 * The window's output head, each row's token and each slot's proposal check.
 *
 * The Strata docs ("BATCHING.md", "Several requests at once (batch slots)"):
 * the head is among the weights a verify window reads once for all of its
 * rows (opening paragraph); sampled requests draw every row with the solo
 * window's counter-based draw, Philox(seed, position) (section "Exactness");
 * with --batch-mtp a window carries two rows per slot, its token and its MTP
 * proposal, and checks the proposal (--batch-mtp paragraph).  The readings
 * this library implements (the pages give no formulas):
 *   logits[t] = W_head RMSNorm(x_t), RMSNorm(x) = x / sqrt(mean(x^2) + 1e-6)
 *   temperature <= 0: token = argmax (ties to the lower token)
 *   temperature > 0: u = (Philox4x64-10(counter (position, 0, 0, 0),
 *     key (seed, 0)) word 0 >> 40) * 2^-24; token = the first v whose
 *     cumulative softmax(logits / temperature) weight exceeds u times the
 *     total (fp32, the vocabulary summed in fixed slices); the greedy token
 *     should rounding leave no token above it
 *   a slot's rows are consecutive; its first row has fed = -1, each later row
 *   was fed a proposal; the slot emits its first row's token and then, while
 *   the previous row's token equals the proposal a row was fed, that row's
 *   token too (n_emit at the slot's first row; 0 at its other rows).
 * ------------------------------------------------------------------------- */
typedef struct strata_head strata_head;

typedef struct {
  int32_t hidden;    /* d: multiple of 64 (4-bit) or 128 (2-bit) */
  int32_t vocab;     /* V: multiple of 16, at most 2^22 */
  int32_t bits;      /* 4 (block 32) or 2 (block 16) */
  int32_t block;
  int32_t max_rows;  /* 1..8 */
} strata_head_desc;

/* Per-row draw inputs (device arrays of the window's T rows). */
typedef struct {
  const int32_t* position;     /* the position whose token the row draws (Philox counter) */
  const uint64_t* seed;        /* the row's seed (Philox key) */
  const float* temperature;    /* <= 0: greedy */
  const int32_t* fed;          /* the proposal the row was fed, -1 for a slot's first row */
} strata_draw_in;

/* Per-row outputs (device arrays). */
typedef struct {
  int32_t* tokens;   /* [T] each row's token */
  int32_t* n_emit;   /* [T] tokens each slot emits, at its first row; 0 at its other rows */
  float* logits;     /* [T][V] the logits, or NULL (then they stay in the handle's workspace) */
} strata_draw_out;

/* Create a head on the current device.  weight: device block-format matrix
 * [1][V][d] (copied into the handle's kernel-ordered layout; the caller may
 * free it once create returns), read on cuda_stream.  Returns EINVAL,
 * EUNSUPPORTED, ENOMEM, ECUDA. */
strata_status strata_head_create(const strata_head_desc* desc, const strata_qmat* weight, void* cuda_stream,
                                 strata_head** out);

/* One window's head: x device fp32 [T][d] (16-byte aligned), 1 <= T <=
 * max_rows; in and out as above.  Asynchronous on cuda_stream; one
 * cooperative launch.  Device errors (a non-finite logit, a wait that gave up)
 * are reported by strata_head_sync.  Returns EINVAL before any launch for bad
 * arguments, ECUDA if the launch fails. */
strata_status strata_head_forward(strata_head* h, const float* x, int32_t T, const strata_draw_in* in,
                                  const strata_draw_out* out, void* cuda_stream);

/* Wait for the last head_forward; EDEVICE (once) if the GPU recorded an error. */
strata_status strata_head_sync(strata_head* h);

/* Block-format bytes of the head matrix and the handle's workspace bytes
 * (either pointer may be NULL). */
strata_status strata_head_query(const strata_head* h, int64_t* head_bytes, int64_t* workspace_bytes);

/* Measurement aid, as strata_window_set_profiling / strata_window_timings. */
strata_status strata_head_set_profiling(strata_head* h, int32_t enable);
strata_status strata_head_timings(strata_head* h, float* ms);

/* Free a head.  NULL is accepted. */
strata_status strata_head_destroy(strata_head* h);

/* ---------------------------------------------------------------------------
 * Routing counters of an adaptive expert tier.
 *
 * The Strata docs ("BATCHING.md", "Several requests at once (batch slots)",
 * the adaptive expert tier paragraphs): batch windows count which experts
 * they route to, and every --adapt-every windows (default 4) the engine swaps
 * the most-routed experts that are not in the fast tier into it in place of
 * the least-routed resident ones; --adapt-swaps bounds a round's swaps,
 * --adapt-decay ages the counts, and --adapt-min-gain F (default 1.5) is the
 * bar a swap must clear (incoming count against outgoing count).  A tier
 * matters where the experts do not all fit the fast memory; this library keeps
 * every expert in HBM and computes the same window either way, so a tier here
 * is the bookkeeping a caller uses to place experts elsewhere.
 *
 * The readings this library implements (the pages leave them open):
 *   c_e += entries routed to e by the window                      (fp32)
 *   after the counts of every adapt_every-th window, a round: experts outside
 *   the tier by c descending and tier experts by c ascending (ties to the
 *   lower expert) pair up in order; pair i swaps while i < adapt_swaps and
 *   c_in > c_out and c_in >= min_gain * c_out (fp32); the first pair that
 *   fails ends the round; then every c_e *= decay                 (fp32)
 * All of it runs on the device, in the window kernel of a handle the tier is
 * attached to (strata_window_set_tier): its first CTA adds the window's
 * counts while it forms the routing plan, and runs a round that is due while
 * it waits at the next window's first grid barrier, before that window's
 * counts; strata_tier_read runs a due round itself before it copies, so what
 * it reports is always the state after the rounds of the windows so far.
 * ------------------------------------------------------------------------- */
typedef struct strata_tier strata_tier;

typedef struct {
  int32_t n_experts;    /* E of the layer it follows: 1..256 */
  int32_t capacity;     /* experts the tier holds: 1..E */
  int32_t adapt_every;  /* a round after every this many windows: >= 1 */
  int32_t adapt_swaps;  /* most swaps per round: 0..E */
  float decay;          /* every counter is multiplied by this after a round: (0, 1] */
  float min_gain;       /* the swap bar: finite, >= 1 */
} strata_tier_desc;

typedef struct {
  int64_t windows;      /* windows counted */
  int64_t rounds;       /* rounds run */
  int32_t n_swaps;      /* swaps made by the last round */
} strata_tier_stats;

/* Create a tier on the current device with zero counters.
 *   initial: host array of `capacity` distinct experts the tier starts with,
 *   or NULL for experts 0..capacity-1.
 * Returns EINVAL (bad field or initial list), ENOMEM, ECUDA. */
strata_status strata_tier_create(const strata_tier_desc* desc, const int32_t* initial, strata_tier** out);

/* Attach a tier to a window handle (NULL detaches).  Every later window of
 * the handle (plain, graph-cache and allocation-free entry points) updates it;
 * the handle's cached graphs are dropped.  One tier per handle; the tier must
 * outlive the attachment.  Returns EINVAL if n_experts differs from the
 * handle's E. */
/* (EUNSUPPORTED if the handle's shared-memory ring is too small to hold a
 * round's arrays beside the staged rows of x; no layer shape here comes near.) */
strata_status strata_window_set_tier(strata_window* h, strata_tier* tier);

/* Wait for the device, run the round that is due (if the last window
 * completed a multiple of adapt_every windows and its round has not run yet),
 * then copy the tier's state to host arrays (each may be NULL): counters
 * float [E], resident int32 [E] (1 = in the tier), swap_in / swap_out int32
 * [E] (the last round's swaps, pairwise, first stats->n_swaps valid), stats.
 * No window of the attached handle may run meanwhile. */
strata_status strata_tier_read(strata_tier* tier, float* counters, int32_t* resident, int32_t* swap_in,
                               int32_t* swap_out, strata_tier_stats* stats);

/* Free a tier (detach it from its handle first).  NULL is accepted. */
strata_status strata_tier_destroy(strata_tier* tier);

/* Free the handle and everything it owns.  NULL is accepted (returns OK). */
strata_status strata_window_destroy(strata_window* h);

/* A static, human-readable name of a status. */
const char* strata_status_str(strata_status s);

#ifdef __cplusplus
}
#endif

#endif /* STRATA_WINDOW_H */
