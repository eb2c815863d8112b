// K1: vocabulary-wide confidence reduction and budget choice.
//
// CONF-KV page, Technische Samenvatting, Methodologie:
//   Vertrouwensschatting  c = 0.4 (1 - H^) + 0.3 sigma(m) + 0.3 p(1), where H^
//                         is the normalised entropy of the next-token
//                         distribution, m the log-probability margin of the two
//                         top tokens and p(1) the top probability;
//   Adaptieve Budgetselectie  c >= tau -> N_high, else N_low.
//
// One thread-block cluster of kClusterCtas CTAs per sequence streams its V
// logits once with 128-bit loads (each CTA one contiguous chunk).  Each thread
// keeps an online state (top-1, top-2, S = sum e^(z-top1),
// T = sum e^(z-top1)(z-top1)); states are merged by warp shuffles, shared
// memory and, across the cluster, distributed shared memory read by CTA rank
// 0 after a hardware cluster barrier.  With p_i = e^(z_i - z*)/S:
//   H = ln S - T/S,  p(1) = 1/S,  m = z(1) - z(2).
#include <cooperative_groups.h>

#include <cfloat>

#include "confkv_internal.cuh"

namespace confkv {
namespace {

struct ConfState {
  float m1, m2, S, T;
  int bad;
};

__device__ __forceinline__ void add_elem(ConfState& st, float x) {
  if (isnan(x) || x == INFINITY) { st.bad = 1; return; }
  if (x == -INFINITY) return;                       // masked token
  if (x > st.m1) {
    if (st.S > 0.0f) {
      const float dlt = st.m1 - x;                  // < 0
      const float f = expf(dlt);
      st.T = f * (st.T + dlt * st.S);
      st.S = f * st.S;
    }
    st.m2 = st.m1;
    st.m1 = x;
    st.S += 1.0f;
  } else {
    if (x > st.m2) st.m2 = x;
    const float dlt = x - st.m1;
    const float e = expf(dlt);
    st.S += e;
    st.T = fmaf(e, dlt, st.T);
  }
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
    const float f = expf(dlt);
    r.S += f * a.S;
    r.T += f * (a.T + dlt * a.S);
  }
  if (b.S > 0.0f) {
    const float dlt = b.m1 - r.m1;
    const float f = expf(dlt);
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

constexpr int kThreads = 1024;
constexpr int kClusterCtas = 8;

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kThreads)
k_confidence(const float* __restrict__ logits, int V, float tau, int N_low, int N_high,
             float* conf, int32_t* hi, float* conf_out, int32_t* budget_out, int32_t* err,
             DevStats* st) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int b = blockIdx.x / kClusterCtas;
  const int rank = static_cast<int>(cluster.block_rank());
  // chunk of this CTA: multiples of 4 elements so that the 128-bit body stays aligned
  const int per = ((V + kClusterCtas - 1) / kClusterCtas + 3) & ~3;
  const int lo = min(V, rank * per), hi_ = min(V, lo + per);
  const float* z = logits + static_cast<size_t>(b) * V + lo;
  const int Vc = hi_ - lo;
  ConfState s{-INFINITY, -INFINITY, 0.0f, 0.0f, 0};

  // 128-bit loads over the 16-byte aligned body, scalar head and tail.
  const uintptr_t addr = reinterpret_cast<uintptr_t>(z);
  int head = static_cast<int>(((16 - (addr & 15)) & 15) / 4);
  if (head > Vc) head = Vc;
  for (int i = threadIdx.x; i < head; i += kThreads) add_elem(s, z[i]);
  const int nvec = (Vc - head) / 4;
  const float4* zv = reinterpret_cast<const float4*>(z + head);
  for (int i = threadIdx.x; i < nvec; i += kThreads) {
    const float4 x = __ldcs(zv + i);
    add_elem(s, x.x);
    add_elem(s, x.y);
    add_elem(s, x.z);
    add_elem(s, x.w);
  }
  for (int i = head + nvec * 4 + threadIdx.x; i < Vc; i += kThreads) add_elem(s, z[i]);

#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = merge(s, shfl_xor(s, o));

  __shared__ ConfState sh[kThreads / 32];
  __shared__ ConfState cta_state;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh[warp] = s;
  __syncthreads();
  if (warp == 0) {
    s = (lane < kThreads / 32) ? sh[lane] : ConfState{-INFINITY, -INFINITY, 0.0f, 0.0f, 0};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = merge(s, shfl_xor(s, o));
    if (lane == 0) cta_state = s;
  }
  cluster.sync();                        // every CTA's state is visible cluster-wide
  if (rank == 0 && warp == 0) {
    s = (lane < kClusterCtas) ? *cluster.map_shared_rank(&cta_state, lane)
                              : ConfState{-INFINITY, -INFINITY, 0.0f, 0.0f, 0};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = merge(s, shfl_xor(s, o));
    if (lane == 0) {
      double c = 0.0;
      const bool bad = s.bad || !(s.S > 0.0f);
      if (!bad) {
        const double S = s.S, T = s.T;
        const double H = log(S) - T / S;
        const double Hn = H / log(static_cast<double>(V));
        const double m = static_cast<double>(s.m1) - static_cast<double>(s.m2);
        const double sig = 1.0 / (1.0 + exp(-m));
        c = 0.4 * (1.0 - Hn) + 0.3 * sig + 0.3 / S;
      } else {
        atomicOr(err, 1);
      }
      const float cf = static_cast<float>(c);
      const int h = (!bad && cf >= tau) ? 1 : 0;
      conf[b] = cf;
      hi[b] = h;
      if (conf_out) conf_out[b] = cf;
      if (budget_out) budget_out[b] = h ? N_high : N_low;
      atomicAdd(&st->logits_bytes, static_cast<unsigned long long>(V) * 4ull);
      if (h) atomicAdd(&st->hi_steps, 1ull);
    }
  }
  cluster.sync();                        // keep remote shared memory alive until read
}

}  // namespace

cudaError_t launch_confidence(const float* logits, int B, int V, float tau, int N_low,
                              int N_high, float* conf, int32_t* hi, float* conf_out,
                              int32_t* budget_out, int32_t* err, DevStats* st,
                              cudaStream_t s) {
  k_confidence<<<B * kClusterCtas, kThreads, 0, s>>>(logits, V, tau, N_low, N_high, conf, hi, conf_out,
                                      budget_out, err, st);
  return cudaGetLastError();
}

}  // namespace confkv
