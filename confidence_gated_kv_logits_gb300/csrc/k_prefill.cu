// Prefill store: the prompt's K/V rows go to the dense cache regions.
//
// CONF-KV page, Technische Samenvatting, Systeemintegratie:
//   Mixed-Precision Opslag  the newest W tokens are kept in FP16, older
//     ones as INT8 (absmax, one scale per token and KV head).
// No token is evicted at prefill: the first decode step applies the budget.
#include "confkv_internal.cuh"

namespace confkv {
namespace {

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
          dst[lane * per + j] = static_cast<int8_t>(q ^ 0x80);   // offset binary: code + 128
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
