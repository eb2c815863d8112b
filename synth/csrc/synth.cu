// Device twin of synth/gen.py: the seeded counter-based input generator.
// Holds no cache-manager arithmetic.  Every floating-point operation is an
// explicit round-to-nearest intrinsic in the same order as the numpy code, so
// the values are bit-identical to the host generator's.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr unsigned long long kG = 0x9E3779B97F4A7C15ull;
constexpr unsigned long long kMul1 = 0xBF58476D1CE4E5B9ull;
constexpr unsigned long long kMul2 = 0x94D049BB133111EBull;
constexpr int kLogTerms = 13;
constexpr int kTrigTerms = 13;
constexpr double kLn2 = 0.6931471805599453;
constexpr double kSqrtHalf = 0.7071067811865476;
constexpr double kHalfPi = 1.5707963267948966;

struct Tables {
  double inv_odd[kLogTerms];
  double cos_c[kTrigTerms];
  double sin_c[kTrigTerms];
};
__constant__ Tables c_tab;

__device__ __forceinline__ unsigned long long fmix(unsigned long long z) {
  z = (z ^ (z >> 30)) * kMul1;
  z = (z ^ (z >> 27)) * kMul2;
  return z ^ (z >> 31);
}

__device__ double ln01(double x) {
  int e;
  double m = frexp(x, &e);
  if (m < kSqrtHalf) {
    m = __dmul_rn(m, 2.0);
    e -= 1;
  }
  const double s = __ddiv_rn(__dsub_rn(m, 1.0), __dadd_rn(m, 1.0));
  const double s2 = __dmul_rn(s, s);
  double acc = c_tab.inv_odd[kLogTerms - 1];
  for (int j = kLogTerms - 2; j >= 0; --j) acc = __dadd_rn(__dmul_rn(acc, s2), c_tab.inv_odd[j]);
  const double lnm = __dmul_rn(__dmul_rn(2.0, s), acc);
  return __dadd_rn(lnm, __dmul_rn(static_cast<double>(e), kLn2));
}

__device__ double poly(double t, const double* c) {
  double acc = c[kTrigTerms - 1];
  for (int j = kTrigTerms - 2; j >= 0; --j) acc = __dadd_rn(__dmul_rn(acc, t), c[j]);
  return acc;
}

__device__ double cos2pi(double u) {
  const double v = __dmul_rn(u, 4.0);
  const double q = floor(v);
  const double f = __dsub_rn(v, q);
  const double th = __dmul_rn(f, kHalfPi);
  const double t = __dmul_rn(th, th);
  const double c = poly(t, c_tab.cos_c);
  const double s = __dmul_rn(th, poly(t, c_tab.sin_c));
  const int qi = static_cast<int>(q);
  return qi == 0 ? c : (qi == 1 ? -s : (qi == 2 ? -c : s));
}

__device__ double normal(unsigned long long key, unsigned long long i) {
  const unsigned long long r = fmix(key + (i + 1ull) * kG);
  const double hi = static_cast<double>(r >> 32);
  const double lo = static_cast<double>(r & 0xffffffffull);
  const double u1 = __dmul_rn(__dadd_rn(hi, 1.0), 0x1p-32);
  const double u2 = __dmul_rn(lo, 0x1p-32);
  const double rad = __dsqrt_rn(__dmul_rn(-2.0, ln01(u1)));
  return __dmul_rn(rad, cos2pi(u2));
}

__global__ void k_fill_f16(__half* out, long long n, unsigned long long key, long long inner,
                           long long tlen, long long pos0, int heavy) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    double z = normal(key, static_cast<unsigned long long>(i));
    if (heavy) {
      const long long pos = pos0 + (i / inner) % tlen;
      z = __dmul_rn(z, (pos % 97 == 96) ? 4.0 : 1.0);
    }
    out[i] = __float2half_rn(__double2float_rn(z));
  }
}

__global__ void k_fill_logits(float* out, long long n, unsigned long long key, double temp) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    out[i] = __double2float_rn(__ddiv_rn(normal(key, static_cast<unsigned long long>(i)), temp));
}

int init_tables() {
  static bool done = false;
  if (done) return 0;
  Tables t;
  for (int j = 0; j < kLogTerms; ++j) t.inv_odd[j] = 1.0 / static_cast<double>(2 * j + 1);
  t.cos_c[0] = 1.0;
  t.sin_c[0] = 1.0;
  for (int k = 1; k < kTrigTerms; ++k) {
    t.cos_c[k] = -t.cos_c[k - 1] / static_cast<double>((2 * k - 1) * (2 * k));
    t.sin_c[k] = -t.sin_c[k - 1] / static_cast<double>((2 * k) * (2 * k + 1));
  }
  if (cudaMemcpyToSymbol(c_tab, &t, sizeof(t)) != cudaSuccess) return -1;
  done = true;
  return 0;
}

int grid_for(long long n) {
  long long g = (n + 255) / 256;
  if (g > 152 * 64) g = 152 * 64;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Measurement helper (not an input generator): streams a buffer once with
// 128-bit loads, four in flight per thread, and keeps the loads live through
// a data-dependent store that never happens for real data.  bench.py times
// it to report the achievable HBM read rate beside the copy peak.
__global__ void __launch_bounds__(256) k_read_probe(const int4* __restrict__ p, long long n16,
                                                    unsigned* sink) {
  unsigned acc = 0u;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += 4 * stride) {
    int4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long j = i + u * stride;
      v[u] = (j < n16) ? __ldcs(p + j) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) acc ^= static_cast<unsigned>(v[u].x ^ v[u].y ^ v[u].z ^ v[u].w);
  }
  if (acc == 0x9E3779B9u && threadIdx.x == 0) sink[blockIdx.x & 63] = acc;
}

}  // namespace

extern "C" {

// Reads `bytes` (a multiple of 16) from `buf` once; sink: 64 words of scratch.
int synth_read_probe(const void* buf, long long bytes, unsigned* sink, int blocks, void* stream) {
  if (!buf || !sink || bytes <= 0 || (bytes & 15) || blocks < 1) return -1;
  k_read_probe<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const int4*>(buf), bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int synth_fill_f16(void* out, long long n, unsigned long long key, long long inner,
                   long long tlen, long long pos0, int heavy, void* stream) {
  if (init_tables()) return -2;
  if (n <= 0) return 0;
  if (heavy && (inner <= 0 || tlen <= 0)) return -1;
  k_fill_f16<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<__half*>(out), n, key, inner, tlen, pos0, heavy);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int synth_fill_logits(void* out, long long n, unsigned long long key, double temperature,
                      void* stream) {
  if (init_tables()) return -2;
  if (n <= 0) return 0;
  k_fill_logits<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<float*>(out), n, key, temperature);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // extern "C"
