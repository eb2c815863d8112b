/*
 * confkv.h -- C ABI of the CONF-KV decode-step library for GB300 (sm_103a).
 *
 * Method: "CONF-KV: Confidence-Aware KV Cache Eviction with Mixed-Precision
 * Storage for Long-Horizon LLM" (gist.science summaries of paper 2605.24786,
 * "Technische Samenvatting" / "Riepilogo Tecnico" / "기술 요약").  Section
 * names below are those of the Dutch page.
 *
 * One context manages the KV cache of every (layer, sequence) of a batch.
 * Each decode step:
 *   1. reduces each sequence's logits to a confidence
 *        c = 0.4 (1 - H^) + 0.3 sigma(m) + 0.3 p(1)        [Vertrouwensschatting]
 *   2. picks the budget N_high if c >= tau, else N_low   [Adaptieve Budgetselectie]
 *      (optionally scaled per layer, CONF-KV-L)           [Pyramidale Budgetten]
 *   3. updates each cached token's EMA attention mass, ranks tokens by
 *      EMA mass + recency, keeps the best N, never evicting the newest P
 *                                                         [Tokenrangschikking]
 *   4. compacts the survivors contiguously and stores tokens older than the
 *      newest W as INT8 (absmax, per token and KV head; optionally also a
 *      power-of-two factor per KV head and channel)      [Mixed-Precision Opslag,
 *                                                          Implementatie]
 *   5. runs block-wise online-softmax decode attention with the INT8
 *      dequantisation fused into the block reads           [Implementatie]
 *
 * Conventions for every call:
 *   - fp16 tensors are IEEE binary16 bit patterns (uint16_t); fp32 is float.
 *   - Tensor arguments of confkv_prefill / confkv_step are DEVICE pointers on
 *     the context's GPU, contiguous, row-major in the stated layout, owned by
 *     the caller, and only touched by work enqueued on `stream` during the
 *     call.  `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - The context owns all cache memory; it is single-threaded: calls on one
 *     context must not run concurrently from several host threads.  The GPU
 *     work of successive calls on one context must be ordered: the same
 *     stream, or streams ordered by events (a call's inputs may come from
 *     the kernel right before it in its stream, even one that lets its
 *     dependents start early through programmatic dependent launch).
 *   - Calls return CONFKV_OK (0) or a negative CONFKV_ERR_* code.  Argument
 *     errors are detected on the host before any work is enqueued; the
 *     message is available from confkv_last_error().  Errors the GPU detects
 *     (non-finite logits, a wait that timed out) are latched in device memory
 *     and returned by the next confkv_stats() call.  No exception crosses the
 *     ABI; no call traps the GPU.
 *   - confkv_step, confkv_step_begin and confkv_step_layer never synchronise
 *     the host with the GPU and allocate nothing, so a decode step (one
 *     confkv_step, or a confkv_step_begin followed by every layer's
 *     confkv_step_layer) can be captured in a CUDA graph once the context has
 *     been prefilled.  All step state, the position included, lives in device
 *     memory: each replay of the graph is one further decode step that reads
 *     the buffers captured (the caller writes the next step's inputs into
 *     them before the replay), and replays mix freely with eager steps.
 *     Only the host-side argument checks (the per-layer order, the position
 *     overflow check) see the capture and not the replays.
 */
#ifndef CONFKV_H_
#define CONFKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CONFKV_OK 0
#define CONFKV_ERR_INVALID_ARG (-1)   /* bad argument; nothing enqueued */
#define CONFKV_ERR_CUDA (-2)          /* a CUDA runtime call failed */
#define CONFKV_ERR_OOM (-3)           /* device allocation failed */
#define CONFKV_ERR_CAPACITY (-4)      /* prefill longer than max_context */
#define CONFKV_ERR_NONFINITE_LOGITS (-5) /* a NaN/+inf (or no finite) logit was seen */
#define CONFKV_ERR_STATE (-6)         /* call out of order (e.g. prefill after steps) */
#define CONFKV_ERR_DEVICE (-7)        /* a device-side wait gave up */

/* device-side error flags (bit mask, confkv_stats_t.error_flags) */
#define CONFKV_FLAG_NONFINITE 1
#define CONFKV_FLAG_CAPACITY 2
#define CONFKV_FLAG_TIMEOUT 4

typedef struct confkv_ctx confkv_ctx;

/*
 * Ranking policies (confkv_opts.policy).  CONF-KV is the method; the others
 * are the comparison points its pages name, run on the same cache, kernels
 * and storage rule (tokens older than the newest W are INT8):
 *   CONFKV  budget from the confidence; key = EMA mass + 1/(1 + age)
 *                                                     [Tokenrangschikking]
 *   WINDOW  fixed budget N_low, the newest tokens are kept (a sliding
 *           window; with N_low and W at least the context length it is the
 *           full FP16 cache).  No confidence is computed: conf_out and
 *           budget_out are not written and logits may be NULL.
 *   H2O     budget from the confidence; key = accumulated attention mass
 *           (acc <- acc + a, fp32), the newest P protected: heavy hitters
 *           plus a recent window
 *   RANDOM  budget from the confidence; key = a uniform draw in [0, 1) per
 *           (step, sequence, token): random eviction at CONF-KV's rate (the
 *           pages' ablation).  The draw is the top 24 bits of SplitMix64
 *           applied as h = mix(mix(mix(mix(seed) ^ t) ^ (l*B + b)) ^ pos),
 *           with mix(x): x += 0x9E3779B97F4A7C15; x = (x ^ x>>30) *
 *           0xBF58476D1CE4E5B9; x = (x ^ x>>27) * 0x94D049BB133111EB;
 *           x ^ x>>31 (Steele, Lea and Flood's SplitMix64 finaliser).
 * Ties between equal keys keep the newer position under every policy.
 */
#define CONFKV_POLICY_CONFKV 0
#define CONFKV_POLICY_WINDOW 1
#define CONFKV_POLICY_H2O 2
#define CONFKV_POLICY_RANDOM 3

/* Optional settings of confkv_create (all fields may be zero = default). */
typedef struct confkv_opts {
  int batch;         /* B sequences decoded together (default 1) */
  int vocab;         /* V, logits per sequence (required, >= 2) */
  int max_context;   /* longest prefill T accepted by confkv_prefill (default 0) */
  float pyramid_min; /* CONF-KV-L: budget factor of the last layer; the factor
                        falls linearly from 1 at layer 0 (0 or 1 = uniform) */
  int device;        /* CUDA device ordinal; negative = the current device
                        (a NULL opts also means the current device) */
  int attn_splits;   /* split-K factor of the attention (0 = automatic) */
  int attn_kernel;   /* 0 automatic (tensor cores when Hq/Hkv <= 8), 1 CUDA
                        cores, 2 tensor cores (requires Hq/Hkv <= 8) */
  int attn_tma;      /* tensor-core attention stages K/V tiles with TMA
                        (0, default) or with cp.async (-1) */
  int policy;        /* CONFKV_POLICY_* (default CONFKV) */
  int int8_channel;  /* INT8 storage [Mixed-Precision Opslag: "per head and
                        channel"]: 0 (default) one absmax scale per (token, KV
                        head, K or V); 1 adds one power-of-two factor 2^f_c per
                        (layer, sequence, KV head, K or V, channel c), fixed by
                        confkv_prefill from the prompt's channel maxima:
                        E_c = ceil(log2 max_t |x_tc|),
                        f_c = max(-8, E_c - max_c E_c), f_c = 0 for a channel
                        that is zero in the prompt and for every channel when
                        there is no prompt.  A row is stored as
                        code_c = round-half-even(x_c 2^-f_c / s) with s the
                        absmax/127 of x 2^-f, and read as code_c s 2^f_c (round
                        trip within s 2^f_c / 2).  The factors belong to the
                        head, so compaction moves tokens without re-quantising.
                        Other values: CONFKV_ERR_INVALID_ARG. */
  uint64_t seed;     /* RANDOM policy: seed of the draws */
} confkv_opts;

/* Counters read back by confkv_stats (cumulative since create unless noted). */
typedef struct confkv_stats_t {
  int64_t steps;            /* decode steps run, graph replays included (a
                               per-layer step counts from confkv_step_begin) */
  int64_t position;         /* position of the next arriving token */
  int32_t error_flags;      /* CONFKV_FLAG_* bits latched since the last call */
  int32_t reserved;
  int64_t tokens_evicted;   /* over all (layer, sequence) */
  int64_t tokens_quantized; /* FP16 -> INT8 conversions (prefill included) */
  int64_t tokens_moved;     /* compaction moves */
  int64_t cache_tokens;     /* current sum over (layer, sequence) of cached tokens */
  int64_t attn_kv_bytes;    /* algorithmic KV + scale bytes read by attention */
  int64_t logits_bytes;     /* logits bytes read by the confidence reduction */
  int64_t budget_high_steps;/* (sequence, step) pairs that chose N_high */
  double cache_bytes;       /* current bytes of cached K/V + scales */
  int64_t kernel_launches;  /* kernels this context has enqueued, counted on
                               the host at each launch (a captured graph's
                               replays add none) */
} confkv_stats_t;

/* Per-kernel device time, accumulated while profiling is enabled. */
typedef struct confkv_profile_t {
  int32_t n_kernels;        /* entries used below */
  int32_t launches[8];
  double total_ms[8];
  const char* names[8];     /* static strings */
} confkv_profile_t;

/*
 * confkv_create -- allocate the cache manager of L layers x B sequences.
 *   layers (L >= 1), heads (Hq query heads), kv_heads (Hkv; Hq % Hkv == 0,
 *   Hq / Hkv <= 16), head_dim (d = 64 or 128).
 *   N_low: budget chosen when c < tau; N_high: budget when c >= tau
 *     [Adaptieve Budgetselectie]; both >= P.
 *   tau: confidence threshold.
 *   P: protected window, the newest P tokens are never evicted (P >= 1)
 *     [Tokenrangschikking].
 *   W: the newest W tokens stay FP16, older kept tokens are INT8 (W >= P)
 *     [Mixed-Precision Opslag].
 *   ema_decay: beta of ema <- beta*ema + (1-beta)*mass, in [0, 1].
 *   opts: see confkv_opts (vocab is required).
 *   *out receives the context.  Returns CONFKV_ERR_INVALID_ARG or
 *   CONFKV_ERR_OOM on failure (then *out is NULL).
 */
int confkv_create(int layers, int heads, int kv_heads, int head_dim, int N_low,
                  int N_high, float tau, int P, int W, float ema_decay,
                  const confkv_opts* opts, confkv_ctx** out);

/*
 * confkv_prefill -- store a prompt of T tokens (positions 0..T-1) in every
 * (layer, sequence) cache.  No token is evicted; tokens whose age T-1-pos is
 * >= W are stored as INT8.  Optional q_last seeds the attention mass that the
 * first decode step folds into the EMA (the EMA itself stays 0).
 *   k, v:   fp16 [L][B][Hkv][T][d] (device)
 *   q_last: fp16 [L][B][Hq][d] (device) or NULL
 * Must precede the first confkv_step; T <= max_context (else
 * CONFKV_ERR_CAPACITY).  T == 0 is a no-op.
 */
int confkv_prefill(confkv_ctx* ctx, const uint16_t* k, const uint16_t* v, int T,
                   const uint16_t* q_last, void* stream);

/*
 * confkv_step -- one decode step of every (layer, sequence): confidence,
 * budget, EMA + ranking, eviction, compaction + INT8 aging, attention.
 *   logits:  fp32 [B][V]          this step's next-token logits
 *   q:       fp16 [L][B][Hq][d]   queries of the new token (16-byte aligned)
 *   k_new:   fp16 [L][B][Hkv][d]  key of the new token (appended, FP16;
 *                                 16-byte aligned, as is v_new)
 *   v_new:   fp16 [L][B][Hkv][d]
 *   out:     fp32 [L][B][Hq][d]   attention output over the kept cache
 *   kept_pos:   int32 [L][B][N_max], N_max = max(N_low, N_high): positions of
 *               the kept tokens, in cache slot order (INT8 region first);
 *               entries past kept_count are left untouched.  May be NULL.
 *   kept_count: int32 [L][B] tokens kept.  May be NULL.
 *   conf_out:   fp32 [B] confidence c (NULL allowed)
 *   budget_out: int32 [B] budget N of the sequence before the per-layer
 *               pyramid factor (NULL allowed)
 * Non-finite logits latch CONFKV_FLAG_NONFINITE and the step proceeds with
 * c = 0 (budget N_low).
 */
int confkv_step(confkv_ctx* ctx, const float* logits, const uint16_t* q,
                const uint16_t* k_new, const uint16_t* v_new, float* out,
                int32_t* kept_pos, int32_t* kept_count, float* conf_out,
                int32_t* budget_out, void* stream);

/*
 * Per-layer stepping, for a model that produces one layer's q / k / v at a
 * time (the layers of a decode step are not all known up front):
 *
 * confkv_step_begin -- first stage of a decode step: the attention mass the
 * previous per-layer step deferred (a no-op where nothing is pending), the
 * confidence and the budget of every sequence from this step's logits (as in
 * confkv_step), then
 * the EMA update, ranking, eviction, compaction and INT8 aging of every
 * layer's caches in one launch (none of it depends on the new token's K/V),
 * reserving each layer's FP16 slot for its arriving token.
 *   logits fp32 [B][V]; conf_out fp32 [B] and budget_out int32 [B] may be NULL.
 * CONFKV_ERR_STATE if the previous begun step still has layers to run.
 *
 * confkv_step_layer -- the rest of the step for one layer `layer`: the
 * arriving token's K/V rows go to the reserved slots, then the attention of
 * that layer's B caches.  Buffers hold that layer only:
 *   q fp16 [B][Hq][d]; k_new, v_new fp16 [B][Hkv][d] (all three 16-byte aligned);
 *   out fp32 [B][Hq][d]; kept_pos int32 [B][N_max] and kept_count int32 [B]
 *   may be NULL.
 * Every layer must be run exactly once, in any order; the step (and the
 * position) advances after the last one.  Until a layer has run, its caches
 * hold the step's compacted state without the arriving token's K/V rows.
 * On the tensor-core attention a layer's launch ends with its output and
 * keeps the raw scores and each query head's (max, sum); the per-token
 * attention mass that the next step ranks by is computed from them by the
 * next confkv_step_begin (or confkv_step, confkv_step_host, or a
 * confkv_read_cache that asks for the mass), with the same arithmetic as a
 * whole step, so the results stay bitwise equal.
 * CONFKV_ERR_STATE without a begun step or for a layer already run;
 * CONFKV_ERR_INVALID_ARG for a bad layer.  The results equal confkv_step's
 * for the same inputs.
 */
int confkv_step_begin(confkv_ctx* ctx, const float* logits, float* conf_out,
                      int32_t* budget_out, void* stream);
int confkv_step_layer(confkv_ctx* ctx, int layer, const uint16_t* q, const uint16_t* k_new,
                      const uint16_t* v_new, float* out, int32_t* kept_pos,
                      int32_t* kept_count, void* stream);

/*
 * confkv_step_host -- confkv_step with HOST buffers of the same layouts.
 * Copies the inputs to context-owned device staging buffers, runs the step
 * and returns the outputs, then waits for all of it.  The copies overlap the
 * compute: logits go first on `stream`; q, k_new and v_new travel on a
 * context-owned copy stream while the confidence and the selection (which do
 * not read them) run; the kept lists go back during the attention.  When
 * `out` (and conf_out and budget_out, if given) is 4-byte-aligned
 * page-locked host memory mapped into the device's address space
 * (cudaHostAlloc / cudaMallocHost memory under unified addressing), the
 * kernels write those outputs into it directly as they produce them, and
 * the attention is one launch.
 * Otherwise those outputs go through staging too: large steps then run the
 * attention as two launches over consecutive (layer, sequence) ranges (the
 * second on a second context-owned stream, so the grids overlap), the first
 * range's outputs copied back while the second computes.  Pinned host
 * memory makes the copies asynchronous DMA; pageable memory works but is
 * slower.  NULL optional
 * outputs are skipped.  The results equal confkv_step's bit for bit, except
 * that kept_pos entries past kept_count are unspecified here (the whole
 * staging row is copied back).  The call synchronises, so it cannot be
 * captured in a CUDA graph.  The first call allocates the staging buffers
 * (the inputs' and outputs' sizes), a copy stream, a second attention stream
 * and their events.
 */
int confkv_step_host(confkv_ctx* ctx, const float* logits, const uint16_t* q,
                     const uint16_t* k_new, const uint16_t* v_new, float* out,
                     int32_t* kept_pos, int32_t* kept_count, float* conf_out,
                     int32_t* budget_out, void* stream);

/*
 * confkv_stats -- synchronise the context's device and read the counters.
 * Returns the first latched device error (CONFKV_ERR_NONFINITE_LOGITS or
 * CONFKV_ERR_DEVICE) and clears the flags, else CONFKV_OK.
 */
int confkv_stats(confkv_ctx* ctx, confkv_stats_t* out);

/*
 * confkv_read_cache -- copy the cache of one (layer l, sequence b) to host
 * memory for inspection (synchronises).  Rows are in slot order: INT8 slots
 * first (n8 of them), then FP16 slots (n16).  Any pointer may be NULL.
 *   pos [n], ema [n]  (int32, fp32)
 *   k8, v8 [n8][Hkv][d] int8;  ks, vs [n8][Hkv] fp32 scales (an INT8 element
 *   reads as code * scale, times 2^f_c of confkv_read_channel_exponents under
 *   int8_channel = 1)
 *   k16, v16 [n16][Hkv][d] fp16 bits
 *   mass [n] fp32: the attention mass of the last attention (mean over the
 *   query heads), which the next step folds into the EMA
 * *n8 and *n16 receive the region sizes; `cap` bounds n8 + n16 rows written.
 */
int confkv_read_cache(confkv_ctx* ctx, int l, int b, int cap, int* n8, int* n16,
                      int32_t* pos, float* ema, int8_t* k8, int8_t* v8, float* ks,
                      float* vs, uint16_t* k16, uint16_t* v16, float* mass);

/*
 * confkv_read_channel_exponents -- copy the channel exponents f_c of one
 * (layer l, sequence b) to host memory (synchronises) [Mixed-Precision
 * Opslag, per head and channel]: k_exp, v_exp int8 [Hkv][d] (either may be
 * NULL).  All zero (factor 1) under int8_channel = 0 or before a prompt.
 * CONFKV_ERR_INVALID_ARG for a bad (l, b).
 */
int confkv_read_channel_exponents(confkv_ctx* ctx, int l, int b, int8_t* k_exp,
                                  int8_t* v_exp);

/*
 * Per-kernel CUDA-event timing of the step kernels (0 confidence, 1 select:
 * EMA, ranking, eviction, compaction and INT8 aging, 2 append: the arriving
 * token of one layer under per-layer stepping, 3 attention).  confkv_profile_enable(ctx, mask) synchronises,
 * clears the totals and records an event pair around every launch of each
 * kernel whose bit is set in `mask` (0 disables).  confkv_profile_read
 * synchronises and returns launches and total milliseconds per kernel.
 * Timing adds event records to the stream; leave it off in production.
 */
int confkv_profile_enable(confkv_ctx* ctx, int kernel_mask);
int confkv_profile_read(confkv_ctx* ctx, confkv_profile_t* out);

/*
 * confkv_confidence_noalloc -- the confidence c and budget of each of `batch`
 * sequences, like the first stage of confkv_step, for callers that cannot
 * allocate device memory: code that runs inside a fixed device-memory budget
 * owned by someone else, a host process whose allocator must not be re-entered
 * from this call, or a latency-critical loop that cannot absorb an
 * allocation's cost or failure.  It needs no context and allocates nothing.
 * The CONF-KV pages have no counterpart to this call; it is an engineering
 * variant of the confidence reduction.
 *   logits:     fp32 [batch][vocab] (device)
 *   conf_out:   fp32 [batch] (device, required)
 *   budget_out: int32 [batch] (device, may be NULL): N_high if c >= tau else N_low
 *   flags_out:  int32 [batch] (device, may be NULL): CONFKV_FLAG_NONFINITE for a
 *               row with a NaN/+inf logit or no finite logit (its c is 0)
 * Work is enqueued on `stream` on the current device.  The cross-CTA scratch
 * is a fixed device array inside the library (about 45 KB, held by every GPU
 * that loads the library until the process exits): batch <= 1024 and at most
 * 2048 CTAs per call, else CONFKV_ERR_CAPACITY before anything is enqueued.
 * Every call shares that array, so calls whose work overlaps on the GPU (on
 * different streams, or from several host threads) race; serialise them.
 * The first call on each device looks up the array's device address (a
 * one-time set-up with that device current); make that first call before any
 * stream capture.  Returns CONFKV_OK, CONFKV_ERR_INVALID_ARG,
 * CONFKV_ERR_CAPACITY or CONFKV_ERR_CUDA.
 */
int confkv_confidence_noalloc(const float* logits, int batch, int vocab, float tau,
                              int N_low, int N_high, float* conf_out, int32_t* budget_out,
                              int32_t* flags_out, void* stream);

/*
 * Which attention kernel the context's steps run (fixed at create):
 * CONFKV_ATTN_CUDA_CORE (Hq/Hkv > 8 or forced), CONFKV_ATTN_TENSOR_CP_ASYNC
 * (tensor cores, K/V tiles staged with cp.async), CONFKV_ATTN_TENSOR_TMA
 * (tensor cores, K/V tiles by TMA); CONFKV_ERR_INVALID_ARG for NULL.
 */
#define CONFKV_ATTN_CUDA_CORE 0
#define CONFKV_ATTN_TENSOR_CP_ASYNC 1
#define CONFKV_ATTN_TENSOR_TMA 2
int confkv_attention_path(const confkv_ctx* ctx);

/*
 * confkv_selftest_bounded_wait -- checks the device-side failure path of the
 * attention's tile waits without any fault: on `device`, one thread waits
 * with the same bounded mbarrier wait, limited to `timeout_us`, on a phase
 * that nothing completes.  *gave_up receives 1 when the wait gave up (the
 * expected result), *waited_us the device time it waited.  Synchronous;
 * allocates 16 bytes of device memory for the call.  timeout_us must be in
 * [1, 1000000], else CONFKV_ERR_INVALID_ARG; CONFKV_ERR_CUDA on a CUDA error.
 * The attention kernel's own limit is 2 s per wait, after which it flags
 * CONFKV_FLAG_TIMEOUT (returned by confkv_stats) and leaves the unit.
 */
int confkv_selftest_bounded_wait(int device, int timeout_us, int* gave_up, double* waited_us);

/* Message of the last error of this context (never NULL). */
const char* confkv_last_error(const confkv_ctx* ctx);

/* Release the context and all its device memory (NULL is a no-op). */
void confkv_free(confkv_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* CONFKV_H_ */
