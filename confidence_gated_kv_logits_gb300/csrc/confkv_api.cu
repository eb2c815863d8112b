// Host side of the CONF-KV C ABI (include/confkv.h): context lifetime,
// argument validation, launch sequencing of the per-step kernels, counters
// and inspection.  No host/device synchronisation happens on the step path.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/confkv.h"
#include "confkv_internal.cuh"

using confkv::AttnParams;
using confkv::Cache;
using confkv::DevStats;
using confkv::StepParams;

namespace {

constexpr int kSmCountDefault = 152;   // GB300; the context reads the device's own count
// resident tensor-core attention CTAs per SM (register-bound): 3 at head_dim
// 128, 4 at head_dim 64
int attn_ctas_per_sm(int d) { return d == 64 ? 4 : 3; }
constexpr int kProfKernels = 4;
constexpr int kHostGroups = 2;   // most attention launches of one host step
// "select" covers ranking, eviction, compaction moves and INT8 aging;
// "append" is the arriving token's store under per-layer stepping (a kernel
// of its own only with the CUDA-core attention).
const char* const kProfNames[kProfKernels] = {"confidence", "select", "append", "attention"};

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (dev >= 0 && dev != prev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

}  // namespace

struct confkv_ctx {
  int L = 0, B = 0, Hq = 0, Hkv = 0, d = 0, g = 0, V = 0;
  int N_low = 0, N_high = 0, P = 0, W = 0, Wr = 0, Ncap = 0, cap8 = 0, slots = 0;
  int max_context = 0, device = 0, splits = 1, splits_layer = 1, attn_kernel = 0;
  int sms = kSmCountDefault;   // the device's SM count (launch-shape heuristics)
  // per-layer stepping (confkv_step_begin / confkv_step_layer)
  bool step_open = false;
  bool layered = false;       // a per-layer step has been begun: masses may be deferred
  int layers_left = 0;
  std::vector<unsigned char> layer_done;
  float tau = 0.f, beta = 0.f, omb = 0.f, pyramid_min = 1.f;
  int policy = CONFKV_POLICY_CONFKV;
  int int8_channel = 0;       // per-(head, channel) power-of-two factors on INT8 rows
  uint64_t seed = 0;
  int64_t t = 0, steps = 0;   // host view: steps launched eagerly (a replayed
                              // graph advances only the device counters)
  int64_t t0 = 0;             // prefill length
  int64_t launches = 0;       // kernels enqueued by this context
  bool prefilled = false;
  Cache cache{};
  float* conf = nullptr;
  int32_t* hi = nullptr;
  confkv::ConfPart* conf_part = nullptr;
  unsigned int* conf_ticket = nullptr;
  int32_t* btab = nullptr;
  float* part_ml = nullptr;
  float* part_acc = nullptr;
  unsigned int* ticket = nullptr;

  float* seed_out = nullptr;
  std::vector<void*> allocs;
  // staging of confkv_step_host
  float* st_logits = nullptr;
  uint16_t* st_q = nullptr;
  uint16_t* st_k = nullptr;
  uint16_t* st_v = nullptr;
  float* st_out = nullptr;
  int32_t* st_kp = nullptr;
  int32_t* st_kc = nullptr;
  float* st_conf = nullptr;
  int32_t* st_bud = nullptr;
  // copy stream, second attention stream and events of confkv_step_host
  // (created with the staging): [0] call start, [1] selection done, [2]
  // cache ready for the attention, [3 + g] inputs of range g on the device,
  // [3 + kHostGroups + g] attention of range g done
  cudaStream_t cp_stream = nullptr;
  cudaStream_t k_stream = nullptr;
  cudaEvent_t cp_ev[3 + 2 * kHostGroups] = {};
  bool cp_ready = false;
  bool staged = false;        // every staging buffer allocated
  std::string msg = "ok";
  alignas(64) unsigned char tmaps[confkv::kTmaMapsBytes];          // tensor maps of the TMA attention path
  bool has_tmaps = false;
  // profiling
  int prof = 0;                                 // kernel bit mask
  std::vector<cudaEvent_t> ev[kProfKernels];   // start/stop pairs
  double prof_ms[kProfKernels] = {0, 0, 0, 0};
  long long prof_n[kProfKernels] = {0, 0, 0, 0};
};

namespace {

int fail(confkv_ctx* c, int code, const std::string& m) {
  if (c) c->msg = m;
  return code;
}

template <typename T>
cudaError_t dalloc(confkv_ctx* c, T** p, size_t count) {
  void* q = nullptr;
  const cudaError_t e = cudaMalloc(&q, std::max<size_t>(count, 1) * sizeof(T));
  if (e != cudaSuccess) return e;
  c->allocs.push_back(q);
  *p = static_cast<T*>(q);
  return cudaMemset(q, 0, std::max<size_t>(count, 1) * sizeof(T));
}

void free_all(confkv_ctx* c) {
  for (void* p : c->allocs) cudaFree(p);
  c->allocs.clear();
  for (cudaEvent_t& e : c->cp_ev)
    if (e) { cudaEventDestroy(e); e = nullptr; }
  if (c->cp_stream) { cudaStreamDestroy(c->cp_stream); c->cp_stream = nullptr; }
  if (c->k_stream) { cudaStreamDestroy(c->k_stream); c->k_stream = nullptr; }
  c->cp_ready = false;
  for (int k = 0; k < kProfKernels; ++k) {
    for (cudaEvent_t e : c->ev[k]) cudaEventDestroy(e);
    c->ev[k].clear();
  }
}

// CONF-KV-L: linear per-layer factor from 1 (layer 0) to pyramid_min (last
// layer), rounded to nearest, never below the protected window.
int layer_budget(int N, int l, int L, double pmin, int P) {
  const double f = (L > 1) ? 1.0 - (1.0 - pmin) * static_cast<double>(l) / static_cast<double>(L - 1)
                           : 1.0;
  const int n = static_cast<int>(std::floor(static_cast<double>(N) * f + 0.5));
  return std::max(P, n);
}

void prof_mark(confkv_ctx* c, int k, cudaStream_t s) {
  if (!(c->prof & (1 << k))) return;
  cudaEvent_t e;
  if (cudaEventCreate(&e) != cudaSuccess) return;
  cudaEventRecord(e, s);
  c->ev[k].push_back(e);
}

void prof_collect(confkv_ctx* c) {
  for (int k = 0; k < kProfKernels; ++k) {
    std::vector<cudaEvent_t>& v = c->ev[k];
    for (size_t i = 0; i + 1 < v.size(); i += 2) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, v[i], v[i + 1]) == cudaSuccess) {
        c->prof_ms[k] += ms;
        c->prof_n[k] += 1;
      }
    }
    for (cudaEvent_t e : v) cudaEventDestroy(e);
    v.clear();
  }
}

// WINDOW keeps a fixed budget (N_low) and computes no confidence
bool uses_confidence(const confkv_ctx* c) { return c->policy != CONFKV_POLICY_WINDOW; }

// Largest power of two <= x (x >= 1): odd split counts measured slower (their
// clusters and chunk shares are uneven).
int floor_pow2(int x) {
  int p = 1;
  while (2 * p <= x) p *= 2;
  return p;
}

// Split-K count of a whole-step attention launch: as many splits as still
// fit every CTA in one wave (3 or 4 resident CTAs per SM), at least ~512
// cached tokens per split (by the budget), at most one cluster (8), a power
// of two.
// Measured on GB300: a second wave, or splits of a few chunks per warp, cost
// more than the idle SMs they would fill (Qwen-14B shape, 384 units: 1 split
// 48 us, 2 splits 60 us; gpt-oss shape, 192 units: 2 splits 31 us, 3 splits
// 43 us, 4 splits 39 us).
int auto_splits(int units, int ncap, int d, int sms) {
  const int want = std::max(1, attn_ctas_per_sm(d) * sms / units);
  const int tok_lim = std::max(1, (ncap + 1) / 512);
  return floor_pow2(std::max(1, std::min(std::min(want, tok_lim), 8)));
}

// One layer's launch holds few units, so its time is one CTA's latency: as
// many splits as still fit one wave, at least ~256 budget tokens per split,
// at most 8, an even count (Qwen-32B shape, 64 units per layer, per-layer
// step: 4 splits 927 us, 5: 883, 6: 884, 7: 1403 -- a 7-CTA cluster).
int auto_splits_layer(int units, int ncap, int d, int sms) {
  const int want = std::max(1, attn_ctas_per_sm(d) * sms / units);
  const int tok_lim = std::max(1, (ncap + 1) / 256);
  const int n = std::max(1, std::min(std::min(want, tok_lim), 8));
  return n > 1 ? (n & ~1) : 1;
}

// layer_call: 0 not a per-layer call; 1 the first layer launch of a
// per-layer step; 2 a later one (which may read its cache before its wait)
int run_attention(confkv_ctx* c, const __half* q, float* out, cudaStream_t s, int lb0, int nlb,
                  int splits, const StepParams* fused = nullptr, bool defer_mass = false,
                  int layer_call = 0) {
  AttnParams ap{};
  ap.q_late = layer_call != 0 ? 1 : 0;
  ap.early = layer_call == 2 ? 1 : 0;
  if (fused) {
    ap.k_new = fused->k_new;
    ap.v_new = fused->v_new;
    ap.kept_pos = fused->kept_pos;
    ap.kept_count = fused->kept_count;
  }
  ap.lb0 = lb0;
  ap.nlb = nlb;
  ap.q = q;
  ap.out = out;
  ap.kernel = c->attn_kernel;
  ap.tmaps = c->has_tmaps ? c->tmaps : nullptr;
  ap.splits = splits;
  ap.part_ml = c->part_ml;
  ap.part_acc = c->part_acc;
  ap.ticket = c->ticket;
  ap.scale = 1.0f / std::sqrt(static_cast<float>(c->d));
  // the per-token attention mass feeds only the EMA (CONF-KV) and the
  // accumulated mass (H2O); per-layer launches defer it to the next step
  const bool uses = c->policy == CONFKV_POLICY_CONFKV || c->policy == CONFKV_POLICY_H2O;
  ap.mass = (uses && !defer_mass) ? 1 : 0;
  ap.defer_mass = (uses && defer_mass) ? 1 : 0;
  const cudaError_t e = confkv::launch_attention(c->cache, ap, s);
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("attention launch: ") + cudaGetErrorString(e));
  c->launches += 1;
  return CONFKV_OK;
}

}  // namespace

extern "C" {

int confkv_create(int layers, int heads, int kv_heads, int head_dim, int N_low, int N_high,
                  float tau, int P, int W, float ema_decay, const confkv_opts* opts,
                  confkv_ctx** out) {
  if (!out) return CONFKV_ERR_INVALID_ARG;
  *out = nullptr;
  confkv_opts o{};
  if (opts) o = *opts;
  if (o.batch == 0) o.batch = 1;
  const float pmin = (o.pyramid_min == 0.0f) ? 1.0f : o.pyramid_min;
  if (layers < 1 || heads < 1 || kv_heads < 1 || heads % kv_heads != 0 ||
      heads / kv_heads > confkv::kMaxGroup || (head_dim != 64 && head_dim != 128) || P < 1 ||
      W < P || N_low < P || N_high < P || !(ema_decay >= 0.0f && ema_decay <= 1.0f) ||
      !std::isfinite(tau) || o.batch < 1 || o.vocab < 2 || o.max_context < 0 ||
      !(pmin > 0.0f && pmin <= 1.0f) || o.attn_splits < 0 || o.attn_splits > 64 ||
      o.attn_kernel < 0 || o.attn_kernel > 2 || o.attn_tma < -1 || o.attn_tma > 0 ||
      (o.attn_kernel == 2 && heads / kv_heads > 8) || o.policy < CONFKV_POLICY_CONFKV ||
      o.policy > CONFKV_POLICY_RANDOM || o.int8_channel < 0 || o.int8_channel > 1)
    return CONFKV_ERR_INVALID_ARG;
  int dev = o.device;
  if (!opts || dev < 0) cudaGetDevice(&dev);
  DeviceGuard guard(dev);
  confkv_ctx* c = new confkv_ctx();
  c->L = layers;
  c->B = o.batch;
  c->Hq = heads;
  c->Hkv = kv_heads;
  c->d = head_dim;
  c->g = heads / kv_heads;
  c->V = o.vocab;
  c->N_low = N_low;
  c->N_high = N_high;
  c->P = P;
  c->W = W;
  c->tau = tau;
  c->beta = ema_decay;
  c->omb = 1.0f - ema_decay;
  c->pyramid_min = pmin;
  c->max_context = o.max_context;
  c->device = dev;
  {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
      c->sms = sms;
    else
      (void)cudaGetLastError();
  }
  c->attn_kernel = o.attn_kernel;
  c->policy = o.policy;
  c->int8_channel = o.int8_channel;
  c->seed = o.seed;
  c->Ncap = std::max(N_low, N_high);
  // INT8 slots: the prefill's tokens older than W, and the kept tokens older
  // than W (under WINDOW the kept tokens are the newest N_low)
  const int kept_old = (o.policy == CONFKV_POLICY_WINDOW) ? std::max(0, N_low - W) : c->Ncap;
  c->cap8 = std::max(std::max(0, o.max_context - W), std::max(kept_old, 32));
  c->cap8 = (c->cap8 + 31) / 32 * 32;
  c->Wr = (W + 15) / 16 * 16;
  c->slots = c->cap8 + c->Wr;

  const size_t LB = static_cast<size_t>(c->L) * c->B;
  const size_t U = LB * c->Hkv;
  const int units = static_cast<int>(U);
  if (o.attn_splits > 0) {
    c->splits = c->splits_layer = o.attn_splits;
  } else {
    c->splits = auto_splits(units, c->Ncap, c->d, c->sms);
    c->splits_layer = auto_splits_layer(c->B * c->Hkv, c->Ncap, c->d, c->sms);
  }
  const int max_splits = std::max(c->splits, c->splits_layer);

  Cache& k = c->cache;
  k.L = c->L; k.B = c->B; k.Hq = c->Hq; k.Hkv = c->Hkv; k.d = c->d; k.g = c->g;
  k.W = c->W; k.Wr = c->Wr; k.P = c->P; k.cap8 = c->cap8; k.slots = c->slots; k.Ncap = c->Ncap;
  cudaError_t e = cudaSuccess;
  auto A = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  A(dalloc(c, &k.k8, U * c->cap8 * c->d));
  A(dalloc(c, &k.v8, U * c->cap8 * c->d));
  A(dalloc(c, &k.ks, U * c->cap8));
  A(dalloc(c, &k.vs, U * c->cap8));
  A(dalloc(c, &k.k16, U * c->Wr * c->d));
  A(dalloc(c, &k.v16, U * c->Wr * c->d));
  A(dalloc(c, &k.pos8, LB * c->cap8));
  A(dalloc(c, &k.pos16, LB * c->Wr));
  A(dalloc(c, &k.ema8, LB * c->cap8));
  A(dalloc(c, &k.ema16, LB * c->Wr));
  A(dalloc(c, &k.mass, U * c->slots));
  A(dalloc(c, &k.scores, LB * c->Hq * c->slots));
  A(dalloc(c, &k.keys, LB * c->slots));
  A(dalloc(c, &k.n8, LB));
  A(dalloc(c, &k.n16, LB));
  A(dalloc(c, &k.new_slot, LB));
  A(dalloc(c, &k.tstep, LB));
  A(dalloc(c, &k.fin, LB * c->Hq * 2));
  A(dalloc(c, &k.mass_pending, U));
  k.chexp = nullptr;
  if (c->int8_channel) A(dalloc(c, &k.chexp, U * 2 * c->d));    // zero: every factor 1
  A(dalloc(c, &k.stats, 1));
  A(dalloc(c, &k.err, 1));
  A(dalloc(c, &c->conf, c->B));
  A(dalloc(c, &c->hi, c->B));
  A(dalloc(c, &c->conf_part, static_cast<size_t>(c->B) * confkv::confidence_ctas_per_seq(c->B, c->V)));
  A(dalloc(c, &c->conf_ticket, c->B));
  A(dalloc(c, &c->btab, static_cast<size_t>(c->L) * 2));
  A(dalloc(c, &c->part_ml, LB * c->Hq * max_splits * 2));
  A(dalloc(c, &c->part_acc, LB * c->Hq * max_splits * c->d));
  A(dalloc(c, &c->ticket, U));

  A(dalloc(c, &c->seed_out, LB * c->Hq * c->d));
  if (e == cudaSuccess) {
    std::vector<int32_t> bt(static_cast<size_t>(c->L) * 2);
    for (int l = 0; l < c->L; ++l) {
      bt[l * 2] = layer_budget(N_low, l, c->L, pmin, P);
      bt[l * 2 + 1] = layer_budget(N_high, l, c->L, pmin, P);
    }
    e = cudaMemcpy(c->btab, bt.data(), bt.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess && o.attn_tma >= 0) c->has_tmaps = confkv::encode_attention_maps(c->cache, c->tmaps);
  if (e != cudaSuccess) {
    const bool oom = (e == cudaErrorMemoryAllocation);
    cudaGetLastError();
    free_all(c);
    delete c;
    return oom ? CONFKV_ERR_OOM : CONFKV_ERR_CUDA;
  }
  c->layer_done.assign(c->L, 0);
  *out = c;
  return CONFKV_OK;
}

int confkv_prefill(confkv_ctx* c, const uint16_t* k, const uint16_t* v, int T,
                   const uint16_t* q_last, void* stream) {
  if (!c) return CONFKV_ERR_INVALID_ARG;
  if (c->steps > 0 || c->prefilled || c->step_open)
    return fail(c, CONFKV_ERR_STATE, "prefill must precede every step and happen once");
  if (T < 0) return fail(c, CONFKV_ERR_INVALID_ARG, "T < 0");
  if (T > c->max_context) return fail(c, CONFKV_ERR_CAPACITY, "T exceeds max_context");
  if (T > 0 && (!k || !v)) return fail(c, CONFKV_ERR_INVALID_ARG, "null k or v");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & (c->int8_channel ? 15u : 1u))
    return fail(c, CONFKV_ERR_INVALID_ARG,
                c->int8_channel ? "k and v must be 16-byte aligned" : "misaligned k or v");
  DeviceGuard guard(c->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->prefilled = true;
  c->t = T;
  c->t0 = T;
  if (T == 0) return CONFKV_OK;
  cudaError_t e = cudaSuccess;
  if (c->int8_channel) {
    // the channel factors first: the store quantises with them
    e = confkv::launch_prefill_exponents(c->cache, reinterpret_cast<const __half*>(k),
                                         reinterpret_cast<const __half*>(v), T, s);
    if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("prefill exponents: ") + cudaGetErrorString(e));
    c->launches += 1;
  }
  e = confkv::launch_prefill_store(c->cache, reinterpret_cast<const __half*>(k),
                                   reinterpret_cast<const __half*>(v), T, s);
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("prefill: ") + cudaGetErrorString(e));
  c->launches += 1;
  if (q_last)
    return run_attention(c, reinterpret_cast<const __half*>(q_last), c->seed_out, s, 0,
                         c->L * c->B, c->splits);
  return CONFKV_OK;
}

}  // extern "C"

namespace {

int check_layer_args(confkv_ctx* c, const uint16_t* q, const uint16_t* k_new,
                     const uint16_t* v_new, float* out) {
  if (!q || !k_new || !v_new || !out)
    return fail(c, CONFKV_ERR_INVALID_ARG, "null q, k_new, v_new or out");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return fail(c, CONFKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(q) & 15u)
    return fail(c, CONFKV_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(out) & 3u)
    return fail(c, CONFKV_ERR_INVALID_ARG, "misaligned out");
  return CONFKV_OK;
}

int run_confidence(confkv_ctx* c, const float* logits, float* conf_out, int32_t* budget_out,
                   cudaStream_t s) {
  if (reinterpret_cast<uintptr_t>(logits) & 3u)
    return fail(c, CONFKV_ERR_INVALID_ARG, "misaligned logits");
  prof_mark(c, 0, s);
  const cudaError_t e = confkv::launch_confidence(
      logits, c->B, c->V, c->tau, c->N_low, c->N_high, c->conf, c->hi, conf_out, budget_out,
      c->cache.err, c->cache.stats, c->conf_part, c->conf_ticket, s);
  prof_mark(c, 0, s);
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("confidence: ") + cudaGetErrorString(e));
  c->launches += 1;
  return CONFKV_OK;
}

StepParams step_params(const confkv_ctx* c, int lb0, int nlb, const uint16_t* k_new,
                       const uint16_t* v_new, int32_t* kept_pos, int32_t* kept_count) {
  StepParams sp{};
  sp.lb0 = lb0;
  sp.nlb = nlb;
  sp.t0 = static_cast<int>(c->t0);
  sp.beta = c->beta;
  sp.omb = c->omb;
  sp.btab = c->btab;
  sp.hi = c->hi;
  sp.kept_pos = kept_pos;
  sp.kept_count = kept_count;
  sp.k_new = reinterpret_cast<const __half*>(k_new);
  sp.v_new = reinterpret_cast<const __half*>(v_new);
  sp.policy = c->policy;
  sp.seed = c->seed;
  return sp;
}

// The masses that per-layer attention launches deferred, computed before
// anything reads them (a no-op on the device for lanes with nothing pending).
int run_mass_finalise(confkv_ctx* c, cudaStream_t s) {
  // only the tensor-core attention defers the mass (per-layer launches)
  if (!confkv::attention_uses_mma(c->cache, c->attn_kernel)) return CONFKV_OK;
  const cudaError_t e = confkv::launch_mass_finalise(c->cache, s);
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("mass finalise: ") + cudaGetErrorString(e));
  c->launches += 1;
  return CONFKV_OK;
}

bool uses_mass(const confkv_ctx* c) {
  return c->policy == CONFKV_POLICY_CONFKV || c->policy == CONFKV_POLICY_H2O;
}

int run_select(confkv_ctx* c, const StepParams& sp, cudaStream_t s) {
  prof_mark(c, 1, s);
  const cudaError_t e = confkv::launch_select(c->cache, sp, s);
  prof_mark(c, 1, s);
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("select: ") + cudaGetErrorString(e));
  c->launches += 1;
  return CONFKV_OK;
}

int run_attention_timed(confkv_ctx* c, const uint16_t* q, float* out, cudaStream_t s, int lb0,
                        int nlb, int splits, const StepParams* fused = nullptr,
                        bool defer_mass = false, int layer_call = 0) {
  prof_mark(c, 3, s);
  const int rc = run_attention(c, reinterpret_cast<const __half*>(q), out, s, lb0, nlb, splits, fused,
                               defer_mass, layer_call);
  prof_mark(c, 3, s);
  return rc;
}

// The (layer, sequence) lanes of a host step cut into consecutive ranges,
// one attention launch each: cuts[0] = 0 < ... < cuts[G] = L*B; returns G.
// The outputs of range 0 are copied back while range 1 computes, so the
// exposed copy is range 1's; a launch boundary costs about one partial wave,
// so there are two ranges, the first ending on a whole CTA wave near 78% of
// the step (the output copy runs at ~0.3x the attention's rate per lane).
// Steps of fewer than 6 waves run as one launch.
int host_ranges(const confkv_ctx* c, size_t* cuts) {
  const size_t LB = static_cast<size_t>(c->L) * c->B;
  const size_t per_lane = static_cast<size_t>(c->Hkv) * c->splits;        // CTAs
  const size_t wave = static_cast<size_t>(attn_ctas_per_sm(c->d)) * c->sms;
  const double waves = static_cast<double>(LB * per_lane) / static_cast<double>(wave);
  cuts[0] = 0;
  if (waves < 6.0 || LB < 2) {
    cuts[1] = LB;
    return 1;
  }
  const size_t w0 = static_cast<size_t>(waves * 0.78 + 0.5);
  cuts[1] = std::max<size_t>(1, std::min(LB - 1, w0 * wave / per_lane));
  cuts[2] = LB;
  return 2;
}

}  // namespace

extern "C" {

int confkv_step(confkv_ctx* c, const float* logits, const uint16_t* q, const uint16_t* k_new,
                const uint16_t* v_new, float* out, int32_t* kept_pos, int32_t* kept_count,
                float* conf_out, int32_t* budget_out, void* stream) {
  if (!c) return CONFKV_ERR_INVALID_ARG;
  if (!logits && uses_confidence(c)) return fail(c, CONFKV_ERR_INVALID_ARG, "null logits");
  int rc = check_layer_args(c, q, k_new, v_new, out);
  if (rc != CONFKV_OK) return rc;
  if (c->step_open) return fail(c, CONFKV_ERR_STATE, "a per-layer step is open");
  if (c->t >= 0x7fffffffLL) return fail(c, CONFKV_ERR_STATE, "position overflow");
  DeviceGuard guard(c->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c->layered && uses_mass(c)) {
    rc = run_mass_finalise(c, s);
    if (rc != CONFKV_OK) return rc;
  }
  if (uses_confidence(c)) {
    rc = run_confidence(c, logits, conf_out, budget_out, s);
    if (rc != CONFKV_OK) return rc;
  }
  rc = run_select(c, step_params(c, 0, c->L * c->B, k_new, v_new, kept_pos, kept_count), s);
  if (rc != CONFKV_OK) return rc;
  rc = run_attention_timed(c, q, out, s, 0, c->L * c->B, c->splits);
  if (rc != CONFKV_OK) return rc;
  c->t += 1;
  c->steps += 1;
  return CONFKV_OK;
}

int confkv_step_begin(confkv_ctx* c, const float* logits, float* conf_out, int32_t* budget_out,
                      void* stream) {
  if (!c) return CONFKV_ERR_INVALID_ARG;
  if (!logits && uses_confidence(c)) return fail(c, CONFKV_ERR_INVALID_ARG, "null logits");
  if (c->step_open) return fail(c, CONFKV_ERR_STATE, "the previous step still has layers to run");
  if (c->t >= 0x7fffffffLL) return fail(c, CONFKV_ERR_STATE, "position overflow");
  DeviceGuard guard(c->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the previous per-layer step's layers deferred their attention mass; it is
  // computed here, before the selection folds it into the EMA (always
  // launched, so that a captured step does it on every replay)
  c->layered = true;
  if (uses_mass(c)) {
    const int rc = run_mass_finalise(c, s);
    if (rc != CONFKV_OK) return rc;
  }
  if (uses_confidence(c)) {
    const int rc = run_confidence(c, logits, conf_out, budget_out, s);
    if (rc != CONFKV_OK) return rc;
  }
  // the selection of every layer needs nothing of this step but the budgets:
  // it runs here in one launch and reserves each arriving token's FP16 slot
  StepParams sp = step_params(c, 0, c->L * c->B, nullptr, nullptr, nullptr, nullptr);
  sp.defer_new = 1;
  const int rc = run_select(c, sp, s);
  if (rc != CONFKV_OK) return rc;
  c->step_open = true;
  c->layers_left = c->L;
  std::fill(c->layer_done.begin(), c->layer_done.end(), 0);
  return CONFKV_OK;
}

int confkv_step_layer(confkv_ctx* c, int layer, const uint16_t* q, const uint16_t* k_new,
                      const uint16_t* v_new, float* out, int32_t* kept_pos, int32_t* kept_count,
                      void* stream) {
  if (!c) return CONFKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= c->L) return fail(c, CONFKV_ERR_INVALID_ARG, "layer out of range");
  int rc = check_layer_args(c, q, k_new, v_new, out);
  if (rc != CONFKV_OK) return rc;
  if (!c->step_open) return fail(c, CONFKV_ERR_STATE, "no step begun (confkv_step_begin)");
  if (c->layer_done[layer]) return fail(c, CONFKV_ERR_STATE, "layer already run in this step");
  DeviceGuard guard(c->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const StepParams sp = step_params(c, layer * c->B, c->B, k_new, v_new, kept_pos, kept_count);
  // the tensor-core attention stores the arriving token itself; the CUDA-core
  // one runs after a separate append launch
  const bool fused = confkv::attention_uses_mma(c->cache, c->attn_kernel);
  if (!fused) {
    prof_mark(c, 2, s);
    const cudaError_t e = confkv::launch_append(c->cache, sp, s);
    prof_mark(c, 2, s);
    if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("append: ") + cudaGetErrorString(e));
    c->launches += 1;
  }
  // the tensor-core attention defers this layer's mass to the next step's
  // first kernel, so that the layer's launch ends with its output
  // the step's first layer launch finds the selection possibly still running;
  // every later one starts after that launch has waited for it
  rc = run_attention_timed(c, q, out, s, layer * c->B, c->B, c->splits_layer, fused ? &sp : nullptr,
                           fused, c->layers_left == c->L ? 1 : 2);
  if (rc != CONFKV_OK) return rc;
  c->layer_done[layer] = 1;
  if (--c->layers_left == 0) {
    c->step_open = false;
    c->t += 1;
    c->steps += 1;
  }
  return CONFKV_OK;
}

int confkv_step_host(confkv_ctx* c, const float* logits, const uint16_t* q,
                     const uint16_t* k_new, const uint16_t* v_new, float* out,
                     int32_t* kept_pos, int32_t* kept_count, float* conf_out,
                     int32_t* budget_out, void* stream) {
  if (!c) return CONFKV_ERR_INVALID_ARG;
  if ((!logits && uses_confidence(c)) || !q || !k_new || !v_new || !out)
    return fail(c, CONFKV_ERR_INVALID_ARG, "null logits, q, k_new, v_new or out");
  if (c->step_open) return fail(c, CONFKV_ERR_STATE, "a per-layer step is open");
  if (c->t >= 0x7fffffffLL) return fail(c, CONFKV_ERR_STATE, "position overflow");
  DeviceGuard guard(c->device);
  const size_t LB = static_cast<size_t>(c->L) * c->B;
  const size_t nlog = static_cast<size_t>(c->B) * c->V, nq = LB * c->Hq * c->d,
               nkv = LB * c->Hkv * c->d, nkp = LB * c->Ncap;
  cudaError_t e = cudaSuccess;
  auto A = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  if (!c->staged) {
    // each buffer once (a call after a failed allocation completes the set)
    auto once = [&](auto** p, size_t n) { if (!*p) A(dalloc(c, p, n)); };
    once(&c->st_logits, nlog);
    once(&c->st_q, nq);
    once(&c->st_k, nkv);
    once(&c->st_v, nkv);
    once(&c->st_out, nq);
    once(&c->st_kp, nkp);
    once(&c->st_kc, LB);
    once(&c->st_conf, static_cast<size_t>(c->B));
    once(&c->st_bud, static_cast<size_t>(c->B));
    if (e != cudaSuccess) return fail(c, e == cudaErrorMemoryAllocation ? CONFKV_ERR_OOM : CONFKV_ERR_CUDA, "staging allocation");
    c->staged = true;
  }
  if (!c->cp_ready) {
    if (!c->cp_stream) A(cudaStreamCreateWithFlags(&c->cp_stream, cudaStreamNonBlocking));
    if (!c->k_stream) A(cudaStreamCreateWithFlags(&c->k_stream, cudaStreamNonBlocking));
    for (cudaEvent_t& ev : c->cp_ev)
      if (!ev) A(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("copy stream: ") + cudaGetErrorString(e));
    c->cp_ready = true;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = c->cp_stream, ks = c->k_stream;
  // When `out` (and c and the budgets, if asked for) are page-locked host
  // memory mapped into the device's address space (cudaHostAlloc /
  // cudaMallocHost memory under unified addressing), the kernels write them
  // directly while the step runs, so no copy trails the attention and the
  // attention is one launch; otherwise they go through the device staging
  // buffers and copies back.  The kept lists always go through staging:
  // the selection writes them at its very end, and waiting for them to cross
  // the host link would hold back the attention, which waits for that grid.
  auto mapped = [](void* p) -> void* {
    // (the kernels store 4-byte words: a misaligned buffer goes through staging)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 3u)) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
  };
  float* out_d = static_cast<float*>(mapped(out));
  float* cf_d = static_cast<float*>(mapped(conf_out));
  int32_t* bd_d = static_cast<int32_t*>(mapped(budget_out));
  const bool direct = out_d && (!conf_out || cf_d) && (!budget_out || bd_d);
  // once copies are enqueued, no return may leave one in flight (the
  // caller's host buffers are only borrowed for the call)
  auto drain = [&](int code) {
    cudaStreamSynchronize(cs);
    cudaStreamSynchronize(ks);
    cudaStreamSynchronize(s);
    return code;
  };
  size_t cuts[kHostGroups + 1] = {0, LB};
  // direct outputs leave nothing to overlap with a second range
  const int G = direct ? 1 : host_ranges(c, cuts);
  cudaEvent_t ev_start = c->cp_ev[0], ev_sel = c->cp_ev[1], ev_ready = c->cp_ev[2];
  const cudaEvent_t* ev_in = c->cp_ev + 3;
  const cudaEvent_t* ev_out = c->cp_ev + 3 + kHostGroups;
  // the logits first (the confidence waits for them); q, k_new and v_new
  // follow range by range on the copy stream (after the work already on
  // `stream`) while the confidence and the selection run: neither reads them
  A(cudaEventRecord(ev_start, s));
  if (logits) A(cudaMemcpyAsync(c->st_logits, logits, nlog * sizeof(float), cudaMemcpyHostToDevice, s));
  A(cudaStreamWaitEvent(cs, ev_start, 0));
  for (int gi = 0; gi < G; ++gi) {
    const size_t lb0 = cuts[gi], nlb = cuts[gi + 1] - lb0;
    const size_t oq = lb0 * c->Hq * c->d, okv = lb0 * c->Hkv * c->d;
    A(cudaMemcpyAsync(c->st_q + oq, q + oq, nlb * c->Hq * c->d * 2, cudaMemcpyHostToDevice, cs));
    A(cudaMemcpyAsync(c->st_k + okv, k_new + okv, nlb * c->Hkv * c->d * 2, cudaMemcpyHostToDevice, cs));
    A(cudaMemcpyAsync(c->st_v + okv, v_new + okv, nlb * c->Hkv * c->d * 2, cudaMemcpyHostToDevice, cs));
    A(cudaEventRecord(ev_in[gi], cs));
  }
  if (e != cudaSuccess) return drain(fail(c, CONFKV_ERR_CUDA, std::string("H2D: ") + cudaGetErrorString(e)));
  int rc;
  if (c->layered && uses_mass(c)) {
    rc = run_mass_finalise(c, s);
    if (rc != CONFKV_OK) return drain(rc);
  }
  if (uses_confidence(c)) {
    rc = run_confidence(c, c->st_logits, conf_out ? (direct ? cf_d : c->st_conf) : nullptr,
                        budget_out ? (direct ? bd_d : c->st_bud) : nullptr, s);
    if (rc != CONFKV_OK) return drain(rc);
  }
  // the selection of every (layer, sequence), reserving the new tokens'
  // slots; the kept lists are final here and go back during the attention
  int32_t* kp = kept_pos ? c->st_kp : nullptr;
  int32_t* kc = kept_count ? c->st_kc : nullptr;
  StepParams sel = step_params(c, 0, static_cast<int>(LB), nullptr, nullptr, kp, kc);
  sel.defer_new = 1;
  rc = run_select(c, sel, s);
  if (rc != CONFKV_OK) return drain(rc);
  A(cudaEventRecord(ev_sel, s));
  A(cudaStreamWaitEvent(cs, ev_sel, 0));
  if (kept_pos)
    A(cudaMemcpyAsync(kept_pos, c->st_kp, nkp * sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
  if (kept_count)
    A(cudaMemcpyAsync(kept_count, c->st_kc, LB * sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
  if (!direct && conf_out && uses_confidence(c))
    A(cudaMemcpyAsync(conf_out, c->st_conf, c->B * sizeof(float), cudaMemcpyDeviceToHost, cs));
  if (!direct && budget_out && uses_confidence(c))
    A(cudaMemcpyAsync(budget_out, c->st_bud, c->B * sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
  const bool fused = confkv::attention_uses_mma(c->cache, c->attn_kernel);
  if (!fused) {
    A(cudaStreamWaitEvent(s, ev_in[G - 1], 0));
    const StepParams ap = step_params(c, 0, static_cast<int>(LB), c->st_k, c->st_v, nullptr, nullptr);
    prof_mark(c, 2, s);
    A(confkv::launch_append(c->cache, ap, s));
    prof_mark(c, 2, s);
    if (e != cudaSuccess) return drain(fail(c, CONFKV_ERR_CUDA, std::string("append: ") + cudaGetErrorString(e)));
    c->launches += 1;
  }
  // one attention launch per range, as soon as its inputs are on the device:
  // the first on `stream`, the second on a second stream, so that the two
  // grids overlap (no launch-boundary tail); each range's outputs go back on
  // the copy stream as soon as it is done
  A(cudaEventRecord(ev_ready, s));
  for (int gi = 0; gi < G; ++gi) {
    const size_t lb0 = cuts[gi], nlb = cuts[gi + 1] - lb0;
    cudaStream_t as = gi == 0 ? s : ks;
    if (gi > 0) A(cudaStreamWaitEvent(as, ev_ready, 0));
    A(cudaStreamWaitEvent(as, ev_in[gi], 0));
    const StepParams f = step_params(c, static_cast<int>(lb0), static_cast<int>(nlb),
                                     c->st_k + lb0 * c->Hkv * c->d, c->st_v + lb0 * c->Hkv * c->d,
                                     nullptr, nullptr);
    float* dst = (direct ? out_d : c->st_out) + lb0 * c->Hq * c->d;
    rc = run_attention_timed(c, c->st_q + lb0 * c->Hq * c->d, dst, as, static_cast<int>(lb0),
                             static_cast<int>(nlb), c->splits, fused ? &f : nullptr);
    if (rc != CONFKV_OK) return drain(rc);
    if (!direct) {
      A(cudaEventRecord(ev_out[gi], as));
      A(cudaStreamWaitEvent(cs, ev_out[gi], 0));
      const size_t oq = lb0 * c->Hq * c->d;
      A(cudaMemcpyAsync(out + oq, c->st_out + oq, nlb * c->Hq * c->d * sizeof(float),
                        cudaMemcpyDeviceToHost, cs));
    }
  }
  if (G > 1) A(cudaStreamWaitEvent(s, ev_out[G - 1], 0));     // `stream` covers every range
  c->t += 1;
  c->steps += 1;
  A(cudaStreamSynchronize(cs));
  A(cudaStreamSynchronize(s));
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("D2H: ") + cudaGetErrorString(e));
  return CONFKV_OK;
}

int confkv_stats(confkv_ctx* c, confkv_stats_t* out) {
  if (!c || !out) return CONFKV_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("sync: ") + cudaGetErrorString(e));
  DevStats ds{};
  int32_t err = 0;
  const size_t LB = static_cast<size_t>(c->L) * c->B;
  std::vector<int32_t> n8(LB), n16(LB);
  e = cudaMemcpy(&ds, c->cache.stats, sizeof(ds), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&err, c->cache.err, sizeof(err), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(n8.data(), c->cache.n8, LB * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(n16.data(), c->cache.n16, LB * 4, cudaMemcpyDeviceToHost);
  int32_t tstep0 = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&tstep0, c->cache.tstep, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(c->cache.err, 0, sizeof(int32_t));
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, std::string("stats: ") + cudaGetErrorString(e));
  std::memset(out, 0, sizeof(*out));
  out->steps = static_cast<int64_t>(ds.steps);
  out->position = c->t0 + tstep0;
  out->error_flags = err;
  out->tokens_evicted = static_cast<int64_t>(ds.evicted);
  out->tokens_quantized = static_cast<int64_t>(ds.quantized);
  out->tokens_moved = static_cast<int64_t>(ds.moved);
  out->attn_kv_bytes = static_cast<int64_t>(ds.kv_bytes);
  out->logits_bytes = static_cast<int64_t>(ds.logits_bytes);
  out->budget_high_steps = static_cast<int64_t>(ds.hi_steps);
  int64_t tok = 0;
  double bytes = 0.0;
  for (size_t i = 0; i < LB; ++i) {
    tok += n8[i] + n16[i];
    bytes += static_cast<double>(c->Hkv) * (n8[i] * (2.0 * c->d + 8.0) + n16[i] * 4.0 * c->d);
  }
  out->cache_tokens = tok;
  out->cache_bytes = bytes;
  out->kernel_launches = c->launches;
  if (err & CONFKV_FLAG_TIMEOUT) return fail(c, CONFKV_ERR_DEVICE, "a device-side wait gave up");
  if (err & CONFKV_FLAG_NONFINITE) return fail(c, CONFKV_ERR_NONFINITE_LOGITS, "non-finite logits seen");
  if (err & CONFKV_FLAG_CAPACITY) return fail(c, CONFKV_ERR_CAPACITY, "cache capacity exceeded");
  return CONFKV_OK;
}

int confkv_read_cache(confkv_ctx* c, int l, int b, int cap, int* n8o, int* n16o, int32_t* pos,
                      float* ema, int8_t* k8, int8_t* v8, float* ks, float* vs, uint16_t* k16,
                      uint16_t* v16, float* mass) {
  if (!c || l < 0 || l >= c->L || b < 0 || b >= c->B || cap < 0)
    return fail(c, CONFKV_ERR_INVALID_ARG, "bad (l, b) or cap");
  DeviceGuard guard(c->device);
  cudaError_t e = cudaDeviceSynchronize();     // the caller's steps may be on any stream
  if (e == cudaSuccess && mass && c->layered && uses_mass(c) && !c->step_open) {
    const int rc = run_mass_finalise(c, nullptr);     // deferred masses first
    if (rc != CONFKV_OK) return rc;
    e = cudaDeviceSynchronize();
  }
  const size_t lb = static_cast<size_t>(l) * c->B + b;
  int n8 = 0, n16 = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&n8, c->cache.n8 + lb, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&n16, c->cache.n16 + lb, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, cudaGetErrorString(e));
  if (n8o) *n8o = n8;
  if (n16o) *n16o = n16;
  const int r8 = std::min(n8, cap), r16 = std::max(0, std::min(n16, cap - r8));
  const int d = c->d, H = c->Hkv;
  auto cp = [&](void* dst, const void* src, size_t bytes) {
    if (e == cudaSuccess && bytes) e = cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost);
  };
  if (pos) {
    cp(pos, c->cache.pos8 + lb * c->cap8, r8 * 4);
    cp(pos + r8, c->cache.pos16 + lb * c->Wr, r16 * 4);
  }
  if (ema) {
    cp(ema, c->cache.ema8 + lb * c->cap8, r8 * 4);
    cp(ema + r8, c->cache.ema16 + lb * c->Wr, r16 * 4);
  }
  std::vector<int8_t> t8(static_cast<size_t>(std::max(r8, 1)) * d);
  std::vector<float> tf(std::max(r8, 1));
  std::vector<uint16_t> t16(static_cast<size_t>(std::max(r16, 1)) * d);
  for (int h = 0; h < H; ++h) {
    const size_t u = lb * H + h;
    for (int which = 0; which < 2; ++which) {
      int8_t* dst8 = which ? v8 : k8;
      if (dst8 && r8) {
        cp(t8.data(), (which ? c->cache.v8 : c->cache.k8) + u * c->cap8 * d, static_cast<size_t>(r8) * d);
        for (int i = 0; i < r8; ++i)
          for (int x = 0; x < d; ++x)   // stored offset binary (code + 128)
            dst8[(static_cast<size_t>(i) * H + h) * d + x] =
                static_cast<int8_t>(t8[static_cast<size_t>(i) * d + x] ^ 0x80);
      }
      float* dsts = which ? vs : ks;
      if (dsts && r8) {
        cp(tf.data(), (which ? c->cache.vs : c->cache.ks) + u * c->cap8, static_cast<size_t>(r8) * 4);
        for (int i = 0; i < r8; ++i) dsts[static_cast<size_t>(i) * H + h] = tf[i];
      }
      uint16_t* dst16 = which ? v16 : k16;
      if (dst16 && r16) {
        cp(t16.data(), reinterpret_cast<const uint16_t*>(which ? c->cache.v16 : c->cache.k16) + u * c->Wr * d,
           static_cast<size_t>(r16) * d * 2);
        for (int i = 0; i < r16; ++i)
          std::memcpy(dst16 + (static_cast<size_t>(i) * H + h) * d, t16.data() + static_cast<size_t>(i) * d, d * 2);
      }
    }
  }
  if (mass) {
    std::vector<float> m(static_cast<size_t>(c->slots));
    for (int i = 0; i < r8 + r16; ++i) mass[i] = 0.0f;
    for (int h = 0; h < H; ++h) {
      cp(m.data(), c->cache.mass + (lb * H + h) * c->slots, static_cast<size_t>(c->slots) * 4);
      for (int i = 0; i < r8; ++i) mass[i] += m[i];
      for (int i = 0; i < r16; ++i) mass[r8 + i] += m[c->cap8 + i];
    }
    for (int i = 0; i < r8 + r16; ++i) mass[i] /= static_cast<float>(c->Hq);
  }
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, cudaGetErrorString(e));
  return CONFKV_OK;
}

int confkv_read_channel_exponents(confkv_ctx* c, int l, int b, int8_t* k_exp, int8_t* v_exp) {
  if (!c || l < 0 || l >= c->L || b < 0 || b >= c->B)
    return fail(c, CONFKV_ERR_INVALID_ARG, "bad (l, b)");
  const size_t row = static_cast<size_t>(c->d);
  const size_t lb = static_cast<size_t>(l) * c->B + b;
  if (!c->cache.chexp) {
    if (k_exp) std::memset(k_exp, 0, c->Hkv * row);
    if (v_exp) std::memset(v_exp, 0, c->Hkv * row);
    return CONFKV_OK;
  }
  DeviceGuard guard(c->device);
  std::vector<int8_t> t(static_cast<size_t>(c->Hkv) * 2 * row);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(t.data(), c->cache.chexp + lb * c->Hkv * 2 * row, t.size(), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(c, CONFKV_ERR_CUDA, cudaGetErrorString(e));
  for (int h = 0; h < c->Hkv; ++h) {
    if (k_exp) std::memcpy(k_exp + h * row, t.data() + (2 * h) * row, row);
    if (v_exp) std::memcpy(v_exp + h * row, t.data() + (2 * h + 1) * row, row);
  }
  return CONFKV_OK;
}

int confkv_profile_enable(confkv_ctx* c, int kernel_mask) {
  if (!c || kernel_mask < 0) return CONFKV_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  cudaDeviceSynchronize();
  prof_collect(c);
  for (int k = 0; k < kProfKernels; ++k) { c->prof_ms[k] = 0.0; c->prof_n[k] = 0; }
  c->prof = kernel_mask & ((1 << kProfKernels) - 1);
  return CONFKV_OK;
}

int confkv_profile_read(confkv_ctx* c, confkv_profile_t* out) {
  if (!c || !out) return CONFKV_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  cudaDeviceSynchronize();
  prof_collect(c);
  std::memset(out, 0, sizeof(*out));
  out->n_kernels = kProfKernels;
  for (int k = 0; k < kProfKernels; ++k) {
    out->launches[k] = static_cast<int32_t>(c->prof_n[k]);
    out->total_ms[k] = c->prof_ms[k];
    out->names[k] = kProfNames[k];
  }
  return CONFKV_OK;
}

int confkv_selftest_bounded_wait(int device, int timeout_us, int* gave_up, double* waited_us) {
  if (!gave_up || !waited_us || timeout_us < 1 || timeout_us > 1000000) return CONFKV_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  void* buf = nullptr;
  if (cudaMalloc(&buf, 16) != cudaSuccess) return CONFKV_ERR_CUDA;
  unsigned long long* d_ns = static_cast<unsigned long long*>(buf);
  int* d_flag = reinterpret_cast<int*>(d_ns + 1);
  cudaError_t e = confkv::selftest_bounded_wait(static_cast<unsigned long long>(timeout_us) * 1000ull,
                                                d_flag, d_ns, nullptr);
  unsigned long long ns = 0;
  int flag = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&ns, d_ns, sizeof(ns), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&flag, d_flag, sizeof(flag), cudaMemcpyDeviceToHost);
  cudaFree(buf);
  if (e != cudaSuccess) return CONFKV_ERR_CUDA;
  *gave_up = flag;
  *waited_us = static_cast<double>(ns) * 1e-3;
  return CONFKV_OK;
}

int confkv_attention_path(const confkv_ctx* c) {
  if (!c) return CONFKV_ERR_INVALID_ARG;
  if (!confkv::attention_uses_mma(c->cache, c->attn_kernel)) return CONFKV_ATTN_CUDA_CORE;
  return c->has_tmaps ? CONFKV_ATTN_TENSOR_TMA : CONFKV_ATTN_TENSOR_CP_ASYNC;
}

const char* confkv_last_error(const confkv_ctx* c) { return c ? c->msg.c_str() : "null context"; }

void confkv_free(confkv_ctx* c) {
  if (!c) return;
  DeviceGuard guard(c->device);
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
}

}  // extern "C"
