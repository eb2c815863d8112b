// K1: vocabulary-wide confidence reduction and budget choice.
//
// CONF-KV page, Technische Samenvatting, Methodologie:
//   Vertrouwensschatting  c = 0.4 (1 - H^) + 0.3 sigma(m) + 0.3 p(1), where H^
//                         is the normalised entropy of the next-token
//                         distribution, m the log-probability margin of the two
//                         top tokens and p(1) the top probability;
//   Adaptieve Budgetselectie  c >= tau -> N_high, else N_low.
//
// Each sequence's V logits are split over enough CTAs to cover every SM
// (each thread kBatch coalesced loads in flight).  Each thread reduces its
// registers to a state (top-1, top-2, S = sum e^(z-top1),
// T = sum e^(z-top1)(z-top1)); states are merged by warp shuffles and shared
// memory, stored per CTA, and the CTA that takes the last ticket of its
// sequence (an atomic counter; no CTA waits) merges them and picks the
// budget.  The sums are fp32 (exponentials by ex2.approx: ~1e-7 relative),
// well inside the 1e-5 tolerance on c.  With p_i = e^(z_i - z*)/S:
//   H = ln S - T/S,  p(1) = 1/S,  m = z(1) - z(2).
#include <cfloat>
#include <cmath>
#include <mutex>

#include "../../include/confkv.h"

#include "confkv_internal.cuh"

namespace confkv {
namespace {

struct ConfState {
  float m1, m2, S, T;
  int bad;
};

constexpr float kL2E = 1.4426950408889634f;
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ ConfState merge(const ConfState& a, const ConfState& b) {
  ConfState r;
  r.bad = a.bad | b.bad;
  r.m1 = fmaxf(a.m1, b.m1);
  r.m2 = fmaxf(fminf(a.m1, b.m1), fmaxf(a.m2, b.m2));
  r.S = 0.0f;
  r.T = 0.0f;
  if (a.S > 0.0f) {
    const float dlt = a.m1 - r.m1;
    const float f = ex2(dlt * kL2E);
    r.S += f * a.S;
    r.T += f * (a.T + dlt * a.S);
  }
  if (b.S > 0.0f) {
    const float dlt = b.m1 - r.m1;
    const float f = ex2(dlt * kL2E);
    r.S += f * b.S;
    r.T += f * (b.T + dlt * b.S);
  }
  return r;
}

__device__ __forceinline__ ConfState shfl_xor(const ConfState& s, int o) {
  ConfState r;
  r.m1 = __shfl_xor_sync(0xffffffffu, s.m1, o);
  r.m2 = __shfl_xor_sync(0xffffffffu, s.m2, o);
  r.S = __shfl_xor_sync(0xffffffffu, s.S, o);
  r.T = __shfl_xor_sync(0xffffffffu, s.T, o);
  r.bad = __shfl_xor_sync(0xffffffffu, s.bad, o);
  return r;
}

constexpr int kThreads = 512;
constexpr int kBatch = 8;      // logits per thread in flight per batch

// The reduction both confidence kernels share.  CTA rk of the cps CTAs of
// sequence b reduces its slice of the row to a state, stores it in part[] and
// takes a ticket; the CTA that takes the sequence's last ticket merges every
// slice's state (no CTA waits) and resets the ticket.  Returns true in lane 0
// of warp 0 of that CTA only, with the merged state in *out.
__device__ __forceinline__ bool reduce_sequence(const float* __restrict__ logits, int V, int cps,
                                                ConfPart* part, unsigned int* ticket,
                                                ConfState* out) {
  const int b = blockIdx.x / cps;
  const int rk = blockIdx.x - b * cps;
  const long long lo = static_cast<long long>(V) * rk / cps;
  const long long hi_ = static_cast<long long>(V) * (rk + 1) / cps;
  const float* z = logits + static_cast<size_t>(b) * V + lo;
  const int Vc = static_cast<int>(hi_ - lo);
  ConfState s{-INFINITY, -INFINITY, 0.0f, 0.0f, 0};
  for (int base = 0; base < Vc; base += kBatch * kThreads) {
    float x[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = base + k * kThreads + threadIdx.x;
      x[k] = (i < Vc) ? __ldcs(z + i) : -INFINITY;      // -inf: outside the slice
    }
    // top-1 / top-2 (ties count twice) and the NaN / +inf test, branch-free
    ConfState bs{-INFINITY, -INFINITY, 0.0f, 0.0f, 0};
    int bad = 0;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      bad |= !(x[k] < INFINITY) && !(x[k] == -INFINITY);
      bs.m2 = fmaxf(bs.m2, fminf(bs.m1, x[k]));
      bs.m1 = fmaxf(bs.m1, x[k]);
    }
    bs.bad = bad;
    if (bs.m1 > -INFINITY) {
      const float ml = bs.m1 * kL2E;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float xc = fmaxf(x[k], -3.0e38f);            // masked tokens -> weight 0
        const float e = ex2(fmaf(xc, kL2E, -ml));
        bs.S += e;
        bs.T = fmaf(e, xc - bs.m1, bs.T);
      }
    }
    s = merge(s, bs);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = merge(s, shfl_xor(s, o));
  __shared__ ConfState sh[kThreads / 32];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh[warp] = s;
  __syncthreads();
  if (warp == 0) {
    s = (lane < kThreads / 32) ? sh[lane] : ConfState{-INFINITY, -INFINITY, 0.0f, 0.0f, 0};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = merge(s, shfl_xor(s, o));
    if (lane == 0) {
      part[blockIdx.x] = ConfPart{s.m1, s.m2, s.S, s.T, s.bad};
      __threadfence();
      s_last = (atomicAdd(&ticket[b], 1u) == static_cast<unsigned>(cps - 1));
    }
  }
  __syncthreads();
  if (!s_last || warp != 0) return false;
  // last CTA of sequence b: merge every CTA's state
  __threadfence();
  s = ConfState{-INFINITY, -INFINITY, 0.0f, 0.0f, 0};
  for (int i = lane; i < cps; i += 32) {
    const ConfPart* pp = part + static_cast<size_t>(b) * cps + i;
    ConfState q{__ldcg(&pp->m1), __ldcg(&pp->m2), __ldcg(&pp->S), __ldcg(&pp->T), __ldcg(&pp->bad)};
    s = merge(s, q);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = merge(s, shfl_xor(s, o));
  if (lane != 0) return false;
  ticket[b] = 0u;
  *out = s;
  return true;
}

// c of a merged state (0 and *bad = true for a row with a NaN / +inf logit or
// no finite logit): H = ln S - T/S, H^ = H / ln V, m = z(1) - z(2), p(1) = 1/S.
__device__ __forceinline__ float confidence_of(const ConfState& s, int V, bool* bad) {
  *bad = s.bad || !(s.S > 0.0f);
  if (*bad) return 0.0f;
  const float H = logf(s.S) - s.T / s.S;
  const float Hn = H / logf(static_cast<float>(V));
  const float m = s.m1 - s.m2;                      // +inf when one finite logit
  const float sig = 1.0f / (1.0f + expf(-m));
  return 0.4f * (1.0f - Hn) + 0.3f * sig + 0.3f / s.S;
}

__global__ void __launch_bounds__(kThreads)
k_confidence(const float* __restrict__ logits, int V, int cps, float tau, int N_low, int N_high,
             float* conf, int32_t* hi, float* conf_out, int32_t* budget_out, int32_t* err,
             DevStats* st, ConfPart* part, unsigned int* ticket) {
  pdl_wait();        // the logits (and the previous step) are complete
  pdl_trigger();     // the selection may start its EMA pass meanwhile
  ConfState s;
  if (!reduce_sequence(logits, V, cps, part, ticket, &s)) return;
  const int b = blockIdx.x / cps;
  bool bad;
  const float c = confidence_of(s, V, &bad);
  if (bad) atomicOr(err, 1);
  const int h = (!bad && c >= tau) ? 1 : 0;
  conf[b] = c;
  hi[b] = h;
  if (conf_out) conf_out[b] = c;
  if (budget_out) budget_out[b] = h ? N_high : N_low;
  atomicAdd(&st->logits_bytes, static_cast<unsigned long long>(V) * 4ull);
  if (h) atomicAdd(&st->hi_steps, 1ull);
}

}  // namespace

// CTAs per sequence: enough to fill the GPU twice, but no fewer than one full
// batch of kBatch logits per thread each (smaller CTAs cost more in the
// cross-CTA merge than they save: batch-1 gpt-oss shape, V = 201088, 49 CTAs
// instead of 197: step 28.2 vs 31.0 us).
int confidence_ctas_per_seq(int B, int V) {
  const int want = (2 * 152 + B - 1) / B;
  const int by_size = (V + kThreads * kBatch - 1) / (kThreads * kBatch);
  return max(1, min(want, by_size));
}

cudaError_t launch_confidence(const float* logits, int B, int V, float tau, int N_low,
                              int N_high, float* conf, int32_t* hi, float* conf_out,
                              int32_t* budget_out, int32_t* err, DevStats* st, ConfPart* part,
                              unsigned int* ticket, cudaStream_t s) {
  const int cps = confidence_ctas_per_seq(B, V);
  const cudaError_t e = launch_pdl(k_confidence, dim3(B * cps), dim3(kThreads), 0, s, logits, V,
                                   cps, tau, N_low, N_high, conf, hi, conf_out, budget_out, err,
                                   st, part, ticket);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the confidence and budget of a batch of logits
// without a context and without any device allocation.  Its cross-CTA scratch
// (one partial state per CTA and one ticket per sequence) lives in a
// file-scope device array that every GPU loading this library holds until the
// process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxBatch = 1024;           // sequences per call
constexpr int kNoAllocMaxParts = 2048;           // CTAs per call (batch x CTAs per sequence)
constexpr size_t kNoAllocBytes =
    sizeof(ConfPart) * kNoAllocMaxParts + sizeof(unsigned int) * kNoAllocMaxBatch;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_conf_scratch[kNoAllocBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_conf_scratch on the current device: looked up once per
// device with that device current (host code cannot use the symbol itself).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_conf_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

__global__ void __launch_bounds__(kThreads)
k_confidence_noalloc(const float* __restrict__ logits, int V, int cps, float tau, int N_low,
                     int N_high, float* conf_out, int32_t* budget_out, int32_t* flags_out,
                     ConfPart* part, unsigned int* ticket) {
  ConfState s;
  if (!reduce_sequence(logits, V, cps, part, ticket, &s)) return;
  const int b = blockIdx.x / cps;
  bool bad;
  const float c = confidence_of(s, V, &bad);
  conf_out[b] = c;
  if (budget_out) budget_out[b] = (!bad && c >= tau) ? N_high : N_low;
  if (flags_out) flags_out[b] = bad ? CONFKV_FLAG_NONFINITE : 0;
}

}  // namespace

}  // namespace confkv

extern "C" int confkv_confidence_noalloc(const float* logits, int batch, int vocab, float tau,
                                         int N_low, int N_high, float* conf_out,
                                         int32_t* budget_out, int32_t* flags_out, void* stream) {
  using namespace confkv;
  if (!logits || !conf_out || batch < 1 || vocab < 2 || !std::isfinite(tau))
    return CONFKV_ERR_INVALID_ARG;
  const int cps = confidence_ctas_per_seq(batch, vocab);
  if (batch > kNoAllocMaxBatch || static_cast<long long>(batch) * cps > kNoAllocMaxParts)
    return CONFKV_ERR_CAPACITY;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return CONFKV_ERR_CUDA;
  ConfPart* part = static_cast<ConfPart*>(base);
  unsigned int* ticket = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(base) +
                                                         sizeof(ConfPart) * kNoAllocMaxParts);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the tickets must start at zero; the partial states are written before read
  if (cudaMemsetAsync(ticket, 0, sizeof(unsigned int) * batch, s) != cudaSuccess)
    return CONFKV_ERR_CUDA;
  k_confidence_noalloc<<<batch * cps, kThreads, 0, s>>>(logits, vocab, cps, tau, N_low, N_high,
                                                        conf_out, budget_out, flags_out, part,
                                                        ticket);
  return cudaGetLastError() == cudaSuccess ? CONFKV_OK : CONFKV_ERR_CUDA;
}
