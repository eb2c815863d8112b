// K3: contiguous compaction of the KV data, and the prefill store.
//
// CONF-KV page, Technische Samenvatting, Systeemintegratie:
//   Implementatie  continuous compaction keeps a dense layout for the
//     attention kernels (no indirection tables); its gather cost is paid
//     here, once per eviction, instead of on every attention read.
//   Mixed-Precision Opslag  the newest W tokens FP16, older ones INT8.
//
// The selection kernel has already planned every move (hole <- mover) and
// quantised the token that aged out of W; all moves read slots at or beyond
// the new region end and write slots below it, so they are independent and
// run fully parallel: one CTA per (layer, sequence, KV head), one thread per
// 16-byte chunk.
#include "confkv_internal.cuh"

namespace confkv {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads)
k_compact(Cache c, const __half* __restrict__ k_new, const __half* __restrict__ v_new) {
  const int unit = blockIdx.x;
  const int lb = unit / c.Hkv;
  const int d = c.d;
  const int nj8 = c.njobs[lb * 2], nj16 = c.njobs[lb * 2 + 1];
  const int2* j8 = c.jobs8 + static_cast<size_t>(lb) * c.cap8;
  const int2* j16 = c.jobs16 + static_cast<size_t>(lb) * c.Wr;

  // INT8 moves: 16-byte chunks of the K and V rows
  const int cpr8 = d / 16;
  int8_t* K8 = c.k8 + static_cast<size_t>(unit) * c.cap8 * d;
  int8_t* V8 = c.v8 + static_cast<size_t>(unit) * c.cap8 * d;
  for (int idx = threadIdx.x; idx < nj8 * 2 * cpr8; idx += kThreads) {
    const int r = idx / (2 * cpr8);
    const int rem = idx - r * 2 * cpr8;
    const bool isv = rem >= cpr8;
    const int ch = isv ? rem - cpr8 : rem;
    const int2 jb = j8[r];
    int8_t* base = isv ? V8 : K8;
    reinterpret_cast<int4*>(base + static_cast<size_t>(jb.x) * d)[ch] =
        reinterpret_cast<const int4*>(base + static_cast<size_t>(jb.y) * d)[ch];
  }
  float* KS = c.ks + static_cast<size_t>(unit) * c.cap8;
  float* VS = c.vs + static_cast<size_t>(unit) * c.cap8;
  for (int r = threadIdx.x; r < nj8; r += kThreads) {
    const int2 jb = j8[r];
    KS[jb.x] = KS[jb.y];
    VS[jb.x] = VS[jb.y];
  }
  // FP16 moves and the new token: 16-byte chunks (8 halves)
  const int cpr16 = d / 8;
  __half* K16 = c.k16 + static_cast<size_t>(unit) * c.Wr * d;
  __half* V16 = c.v16 + static_cast<size_t>(unit) * c.Wr * d;
  const __half* kn = k_new + static_cast<size_t>(unit) * d;
  const __half* vn = v_new + static_cast<size_t>(unit) * d;
  for (int idx = threadIdx.x; idx < nj16 * 2 * cpr16; idx += kThreads) {
    const int r = idx / (2 * cpr16);
    const int rem = idx - r * 2 * cpr16;
    const bool isv = rem >= cpr16;
    const int ch = isv ? rem - cpr16 : rem;
    const int2 jb = j16[r];
    __half* base = isv ? V16 : K16;
    const __half* src = (jb.y >= 0) ? base + static_cast<size_t>(jb.y) * d : (isv ? vn : kn);
    reinterpret_cast<int4*>(base + static_cast<size_t>(jb.x) * d)[ch] =
        reinterpret_cast<const int4*>(src)[ch];
  }
}

// Prefill: one warp per (token, K or V) row.  Token i of T has age T-1-i; the
// first max(0, T-W) tokens go to INT8 slots 0.., the rest to FP16 slots 0...
__global__ void __launch_bounds__(256)
k_prefill_store(Cache c, const __half* __restrict__ k, const __half* __restrict__ v, int T) {
  const int unit = blockIdx.x;
  const int lb = unit / c.Hkv, h = unit - lb * c.Hkv;
  const int d = c.d;
  const int n8p = max(0, T - c.W);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_cta = 8;            // warps
  const int per = d / 32;
  for (int i = blockIdx.y * rows_per_cta + warp; i < T; i += gridDim.y * rows_per_cta) {
    for (int isv = 0; isv < 2; ++isv) {
      const __half* src = (isv ? v : k) + (static_cast<size_t>(unit) * T + i) * d;
      if (i < n8p) {
        float x[4];
        float amax = 0.0f;
        for (int j = 0; j < per; ++j) {
          x[j] = __half2float(src[lane * per + j]);
          amax = fmaxf(amax, fabsf(x[j]));
        }
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(amax, 127.0f);
        int8_t* dst = (isv ? c.v8 : c.k8) + (static_cast<size_t>(unit) * c.cap8 + i) * d;
        for (int j = 0; j < per; ++j) {
          int q = 0;
          if (s != 0.0f) q = max(-127, min(127, __float2int_rn(__fdiv_rn(x[j], s))));
          dst[lane * per + j] = static_cast<int8_t>(q);
        }
        if (lane == 0) (isv ? c.vs : c.ks)[static_cast<size_t>(unit) * c.cap8 + i] = s;
      } else {
        __half* dst = (isv ? c.v16 : c.k16) + (static_cast<size_t>(unit) * c.Wr + (i - n8p)) * d;
        for (int j = lane; j < d; j += 32) dst[j] = src[j];
      }
    }
    if (h == 0 && lane == 0) {
      if (i < n8p) {
        c.pos8[static_cast<size_t>(lb) * c.cap8 + i] = i;
        c.ema8[static_cast<size_t>(lb) * c.cap8 + i] = 0.0f;
      } else {
        c.pos16[static_cast<size_t>(lb) * c.Wr + (i - n8p)] = i;
        c.ema16[static_cast<size_t>(lb) * c.Wr + (i - n8p)] = 0.0f;
      }
    }
  }
  if (h == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    c.n8[lb] = n8p;
    c.n16[lb] = T - n8p;
    if (n8p > 0) atomicAdd(&c.stats->quantized, static_cast<unsigned long long>(n8p));
  }
}

}  // namespace

cudaError_t launch_compact(const Cache& c, const __half* k_new, const __half* v_new,
                           cudaStream_t s) {
  k_compact<<<c.L * c.B * c.Hkv, kThreads, 0, s>>>(c, k_new, v_new);
  return cudaGetLastError();
}

cudaError_t launch_prefill_store(const Cache& c, const __half* k, const __half* v, int T,
                                 cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int units = c.L * c.B * c.Hkv;
  int ychunks = (T + 7) / 8;
  const int max_ctas = 152 * 32;
  if (static_cast<long long>(units) * ychunks > max_ctas) ychunks = max(1, max_ctas / units);
  if (ychunks > 65535) ychunks = 65535;
  k_prefill_store<<<dim3(units, ychunks), 256, 0, s>>>(c, k, v, T);
  return cudaGetLastError();
}

}  // namespace confkv
