// Internal device-side layout of the CONF-KV cache and launch wrappers.
//
// HBM layout of one context (lb = l*B + b, h = KV head):
//   INT8 region   k8, v8  int8  [L*B][Hkv][cap8][d]    (slots 0..n8-1 live; each
//                 byte holds code + 128 (offset binary), code in [-127, 127])
//                 ks, vs  fp32  [L*B][Hkv][cap8]       one absmax scale per row
//   FP16 region   k16,v16 fp16  [L*B][Hkv][Wr][d]      (slots 0..n16-1 live;
//                 Wr = W rounded up to 16, so whole 16-token chunks stay in bounds)
//   metadata      pos8, ema8 [L*B][cap8]; pos16, ema16 [L*B][Wr]   (cap8 % 32 == 0)
//   chexp         int8 [L*B][Hkv][2][d]    channel exponents f_c of K, then V
//                 (per-(head, channel) storage mode only; else null): an INT8
//                 element reads as code * scale * 2^f_c
//   mass          fp32 [L*B][Hkv][slots]   attention mass of the last
//                 attention summed over the query heads of one KV head;
//                 slot id = INT8 slot, or cap8 + FP16 slot; slots = cap8 + Wr
//   scores        fp32 [L*B][Hq][slots]    raw scores of the last attention
//   fin           fp32 [L*B][Hq][2]        (max, sum) of each query head's last
//                 attention, kept when a per-layer launch defers the mass
//   mass_pending  int32 [L*B][Hkv]         1: the unit's mass is still to be
//                 computed from scores and fin (deferred by per-layer launches);
//                 cleared by the CTA that computes it, so finalising twice is a no-op
// Both regions are dense (contiguous compaction): live slots are always
// [0, n8) and [0, n16), so the attention streams them without any indirection.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

namespace confkv {

// Drops one 128-byte line from L2 without writing it back: for scratch that
// has been read for the last time before its next full rewrite (PTX
// `discard.global.L2`; the line's contents become undefined).  `p` must be
// 128-byte aligned and the line must hold nothing else that is still live.
__device__ __forceinline__ void l2_discard_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;\n" ::"l"(p) : "memory");
}

// Programmatic dependent launch.  The step kernels are launched so that each
// may start while its predecessor in the stream is still running: a kernel
// calls pdl_wait() before it touches anything the predecessor writes (the
// wait returns once that grid has completed and its memory is visible), and
// pdl_trigger() once its own dependents may be scheduled.  Without the launch
// attribute both are no-ops.  Every kernel waits before it completes, so a
// grid's completion implies that of every earlier kernel in the stream.  The
// confidence kernel triggers right after its own wait and the attention after
// its main loop; the selection and append kernels trigger at their start,
// which is safe because the attention reads nothing but its caller's queries
// before its wait.  The selection reads the previous step's state before its
// own wait: its predecessor is the confidence kernel (which has waited for
// the previous attention) or, under the WINDOW policy, the previous step's
// attention, whose trigger comes after every read of the cache data the
// selection moves.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kMaxGroup = 16;   // query heads per KV head supported

struct DevStats {
  unsigned long long evicted;
  unsigned long long quantized;
  unsigned long long moved;
  unsigned long long kv_bytes;
  unsigned long long logits_bytes;
  unsigned long long hi_steps;
  unsigned long long steps;   // decode steps whose selection has run
};

struct ConfPart {       // partial confidence state of one CTA
  float m1, m2, S, T;
  int bad;
};

struct Cache {
  int L, B, Hq, Hkv, d, g, W, Wr, P, cap8, slots, Ncap;
  int8_t* k8;
  int8_t* v8;
  float* ks;
  float* vs;
  __half* k16;
  __half* v16;
  int32_t* pos8;
  int32_t* pos16;
  float* ema8;
  float* ema16;
  float* mass;
  float* scores;
  float* keys;      // [L*B][slots] ranking keys of the current step
  int32_t* n8;
  int32_t* n16;
  int32_t* tstep;     // [L*B] decode steps run since the prefill; the arriving
                      // token's position is t0 + tstep (kept on the device so
                      // that a captured step can be replayed)
  int32_t* new_slot;  // [L*B] FP16 slot reserved for the arriving token when the
                      // selection runs ahead of the layer's K/V (per-layer steps)
  int8_t* chexp;      // [L*B*Hkv][2][d] channel exponents, or null (per-token scales only)
  float* fin;         // [L*B][Hq][2] per-head (max, sum) of a deferred mass
  int32_t* mass_pending;  // [L*B*Hkv] the unit's mass awaits launch_mass_finalise
  DevStats* stats;
  int32_t* err;
};

struct StepParams {
  int lb0, nlb;          // (layer, sequence) range of this launch: [lb0, lb0 + nlb);
                         // the caller's buffers below start at lb0
  int t0;                // prefill length: position of the first decoded token
  float beta, omb;       // EMA decay and 1 - decay (fp32)
  const int32_t* btab;   // [L][2] per-layer budget for (N_low, N_high)
  const int32_t* hi;     // [B] 1 if the sequence chose N_high
  int32_t* kept_pos;     // [L*B][Ncap] or null
  int32_t* kept_count;   // [L*B] or null
  const __half* k_new;   // [L*B][Hkv][d] key / value of the new token
  const __half* v_new;
  int policy;            // CONFKV_POLICY_*: ranking key and EMA rule
  int defer_new;         // 1: reserve the arriving token's FP16 slot in new_slot and
                         // leave its K/V rows and the kept lists to launch_append
  uint64_t seed;         // RANDOM policy draws
};

struct AttnParams {
  int lb0, nlb;          // (layer, sequence) range; q and out start at lb0
  int kernel;             // 0 auto, 1 CUDA-core, 2 tensor-core
  const void* tmaps;     // host pointer to 4 CUtensorMap (K8, V8, K16, V16) or null
  const __half* q;       // [L*B][Hq][d]
  float* out;            // [L*B][Hq][d]
  int splits;
  float* part_ml;        // [L*B*Hq][splits][2]
  float* part_acc;       // [L*B*Hq][splits][d]
  unsigned int* ticket;  // [L*B*Hkv]
  float scale;           // 1/sqrt(d)
  int mass;              // 1: write the per-token attention mass (EMA / H2O policies)
  int defer_mass;        // 1: keep the raw scores and each head's (max, sum) instead
                         // and flag the lane; launch_mass_finalise computes the mass
  int cluster;           // set by the launcher: the splits of a unit are one cluster
  // Per-layer steps on the tensor-core path (else null): the arriving token's
  // K/V [nlb][Hkv][d], stored into the FP16 slot the selection reserved
  // (new_slot) before that slot is read, and the kept positions [nlb][Ncap] /
  // counts [nlb] of the range (either may be null).
  const __half* k_new;
  const __half* v_new;
  int32_t* kept_pos;
  int32_t* kept_count;
  // Per-layer calls: the caller's q, k_new and v_new may come from the kernel
  // right before this launch, so they are read only after the dependency
  // wait (q_late = 1).  A layer launch that is not the step's first may also
  // read its own layer's cache (region sizes, reserved slot, tiles) before
  // the wait (early = 1, tensor-core TMA path): that cache is written only by
  // the step's selection, which is complete by then -- the step's first
  // layer launch passes its own wait (the selection done) before it
  // triggers, and every later launch in the stream starts after that trigger.
  int q_late;
  int early;
};

// ---- launch wrappers (each file owns its kernels) ----
int confidence_ctas_per_seq(int B, int V);
cudaError_t launch_confidence(const float* logits, int B, int V, float tau, int N_low,
                              int N_high, float* conf, int32_t* hi, float* conf_out,
                              int32_t* budget_out, int32_t* err, DevStats* st, ConfPart* part,
                              unsigned int* ticket, cudaStream_t s);
cudaError_t launch_select(const Cache& c, const StepParams& sp, cudaStream_t s);
// Second half of a deferred selection for (layer, sequence) range [lb0, lb0 + nlb):
// stores the arriving token's K/V rows (k_new, v_new) in the reserved FP16
// slots and writes kept_pos / kept_count when given.
cudaError_t launch_append(const Cache& c, const StepParams& sp, cudaStream_t s);
cudaError_t launch_prefill_store(const Cache& c, const __half* k, const __half* v, int T,
                                 cudaStream_t s);
// Channel exponents of every (unit, K or V) from the prompt's T rows (before
// launch_prefill_store; c.chexp must be set).
cudaError_t launch_prefill_exponents(const Cache& c, const __half* k, const __half* v, int T,
                                     cudaStream_t s);

// 2^-f as a float for a channel exponent f in [-8, 0] (exact): the factor a
// value is divided by before the absmax quantiser.
__device__ __forceinline__ float chan_inv_factor(int f) {
  return __uint_as_float(static_cast<uint32_t>(127 - f) << 23);
}
// 2^f as a float (f in [-8, 0]): the factor a dequantised value is multiplied by.
__device__ __forceinline__ float chan_factor(int f) {
  return __uint_as_float(static_cast<uint32_t>(127 + f) << 23);
}
cudaError_t launch_attention(const Cache& c, const AttnParams& ap, cudaStream_t s);
// true if launch_attention runs the tensor-core kernel for this cache and
// AttnParams::kernel (only that kernel handles AttnParams::k_new)
bool attention_uses_mma(const Cache& c, int kernel);
cudaError_t launch_attention_mma(const Cache& c, const AttnParams& ap, cudaStream_t s);
// The per-token attention mass of every lane whose attention deferred it
// (mass_pending), from the raw scores and per-head (max, sum) the attention
// kept, with the same arithmetic as the attention's own mass epilogue.
cudaError_t launch_mass_finalise(const Cache& c, cudaStream_t s);
// Encodes the four tensor maps of the TMA attention path into `out`
// (kTmaMapsBytes bytes, 64-byte aligned); returns false if the driver cannot
// or the cache is too large for 32-bit tile coordinates.
constexpr int kTmaMapsBytes = 512;
bool encode_attention_maps(const Cache& c, void* out);
// One thread waits, with the attention's bounded mbarrier wait and limit
// limit_ns, on a phase nothing completes; *gave_up = 1 when it gave up,
// *waited_ns the device time it waited (device pointers).
cudaError_t selftest_bounded_wait(unsigned long long limit_ns, int* gave_up,
                                  unsigned long long* waited_ns, cudaStream_t s);

}  // namespace confkv
