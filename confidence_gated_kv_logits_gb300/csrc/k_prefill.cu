// Prefill store: the prompt's K/V rows go to the dense cache regions.
//
// CONF-KV page, Technische Samenvatting, Systeemintegratie:
//   Mixed-Precision Opslag  the newest W tokens are kept in FP16, older
//     ones as INT8 (absmax, one scale per token and KV head; in the
//     per-(head, channel) mode also one power-of-two factor per channel,
//     fixed here from the prompt).
// No token is evicted at prefill: the first decode step applies the budget.
#include <climits>

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
        const int8_t* fe = c.chexp ? c.chexp + (static_cast<size_t>(unit) * 2 + isv) * d : nullptr;
        for (int j = 0; j < per; ++j) {
          x[j] = __half2float(src[lane * per + j]);
          if (fe) x[j] *= chan_inv_factor(fe[lane * per + j]);     // exact: x * 2^-f
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

// Channel exponents of one (unit, K or V): the prompt's T rows are streamed
// (kRowsPar rows in parallel, 16-byte pieces of 8 channels per thread, 4
// loads in flight) to the per-channel max |x| (exact in fp32), then
// E_c = ceil(log2 cmax_c) from the exact binary exponent, and
// f_c = max(-8, E_c - max E) over the channels with cmax_c > 0 (0 otherwise).
template <int D>
__global__ void __launch_bounds__(256)
k_prefill_exponents(Cache c, const __half* __restrict__ k, const __half* __restrict__ v, int T) {
  constexpr int kPieces = D / 8;                 // 16-byte pieces per row
  constexpr int kRowsPar = 256 / kPieces;        // rows in flight per pass
  const int unit = blockIdx.x, isv = blockIdx.y;
  const int tid = threadIdx.x, pc = tid % kPieces, r0 = tid / kPieces;
  const __half* src = (isv ? v : k) + static_cast<size_t>(unit) * T * D;
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int base = r0; base < T; base += 4 * kRowsPar) {
    int4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int row = base + u * kRowsPar;
      w[u] = row < T ? reinterpret_cast<const int4*>(src + static_cast<size_t>(row) * D)[pc]
                     : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __half2* h2 = reinterpret_cast<const __half2*>(&w[u]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h2[e]);
        m[2 * e] = fmaxf(m[2 * e], fabsf(f.x));
        m[2 * e + 1] = fmaxf(m[2 * e + 1], fabsf(f.y));
      }
    }
  }
  __shared__ float sm[kRowsPar][D];
  __shared__ int sE[D];
  __shared__ int s_emax;
#pragma unroll
  for (int e = 0; e < 8; ++e) sm[r0][pc * 8 + e] = m[e];
  if (tid == 0) s_emax = INT_MIN;
  __syncthreads();
  for (int ch = tid; ch < D; ch += 256) {
    float cm = 0.0f;
    for (int r = 0; r < kRowsPar; ++r) cm = fmaxf(cm, sm[r][ch]);
    int E = INT_MIN;
    if (cm > 0.0f) {
      int ex;
      const float fr = frexpf(cm, &ex);          // cm = fr * 2^ex, fr in [0.5, 1): exact
      E = (fr == 0.5f) ? ex - 1 : ex;
      atomicMax(&s_emax, E);
    }
    sE[ch] = E;
  }
  __syncthreads();
  for (int ch = tid; ch < D; ch += 256) {
    const int E = sE[ch];
    c.chexp[(static_cast<size_t>(unit) * 2 + isv) * D + ch] =
        static_cast<int8_t>(E == INT_MIN ? 0 : max(-8, E - s_emax));
  }
}

}  // namespace

cudaError_t launch_prefill_exponents(const Cache& c, const __half* k, const __half* v, int T,
                                     cudaStream_t s) {
  if (T <= 0 || !c.chexp) return cudaSuccess;
  const int units = c.L * c.B * c.Hkv;
  if (c.d == 128) k_prefill_exponents<128><<<dim3(units, 2), 256, 0, s>>>(c, k, v, T);
  else if (c.d == 64) k_prefill_exponents<64><<<dim3(units, 2), 256, 0, s>>>(c, k, v, T);
  else return cudaErrorInvalidValue;
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
