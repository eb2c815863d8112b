// K2: EMA attention mass update, ranking, exact top-N selection with the
// protected window, and the contiguous-compaction plan.
//
// CONF-KV page, Technische Samenvatting, Methodologie:
//   Tokenrangschikking en Evictie  tokens are ranked by a score combining the
//     EMA of the attention mass they receive and their recency; the newest P
//     tokens are never evicted; the best N within the budget are kept.
//   Pyramidale Budgetten  optional per-layer budgets (folded into btab).
//   Implementatie  survivors are compacted contiguously (no indirection).
//   Mixed-Precision Opslag  the token leaving the newest W is stored as INT8.
//   Betekenis en Beweringen  forward-only: an evicted token never returns.
//
// Readings (the pages give the ingredients, not the formulas):
//   a_i  = (sum over query heads of the previous attention probability) / Hq
//   ema  = beta*ema + (1-beta)*a_i                 (fp32, one rounding per op)
//   key  = ema + 1/(1 + age)                       (fp32, one rounding per op)
//   order: key descending, then position descending (newer wins a tie)
//   protected: age < P (the new token included); append, then evict.
// The fp32 operations use explicit _rn intrinsics so that no contraction
// changes the rounding: the decision is taken in fp32 on exact fp32 values.
//
// One CTA of kThreads per (layer, sequence).  Selection: the need-th largest
// 64-bit key (key bits << 32 | position; unique) is found by an 8-bit MSB
// radix select over the candidates (early exit once the boundary bucket is
// taken whole); a single eviction, the steady state, is one arg-min.
#include <cfloat>

#include "confkv_internal.cuh"

namespace confkv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ unsigned long long key64(float key, int pos) {
  return (static_cast<unsigned long long>(__float_as_uint(key)) << 32) |
         static_cast<unsigned int>(pos);
}

// Block-wide exclusive scan of two flags; returns the ranks, accumulates totals.
struct Scan2 {
  int* wsum;  // smem [2][kWarps]
};

__device__ __forceinline__ void block_scan2(bool fa, bool fb, int* wsum, int& ra, int& rb,
                                            int& tota, int& totb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned ba = __ballot_sync(0xffffffffu, fa);
  const unsigned bb = __ballot_sync(0xffffffffu, fb);
  const unsigned lt = (1u << lane) - 1u;
  if (lane == 0) {
    wsum[warp] = __popc(ba);
    wsum[kWarps + warp] = __popc(bb);
  }
  __syncthreads();
  int offa = 0, offb = 0, sa = 0, sb = 0;
  for (int w = 0; w < kWarps; ++w) {
    const int xa = wsum[w], xb = wsum[kWarps + w];
    if (w < warp) { offa += xa; offb += xb; }
    sa += xa;
    sb += xb;
  }
  ra = tota + offa + __popc(ba & lt);
  rb = totb + offb + __popc(bb & lt);
  tota += sa;
  totb += sb;
  __syncthreads();
}

__device__ __forceinline__ unsigned long long block_min_u64(unsigned long long v,
                                                            unsigned long long* sh) {
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long x = __shfl_xor_sync(0xffffffffu, v, o);
    v = x < v ? x : v;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  unsigned long long r = sh[0];
  for (int w = 1; w < kWarps; ++w) r = sh[w] < r ? sh[w] : r;
  __syncthreads();
  return r;
}

// warp-level INT8 absmax quantisation of one fp16 row of d elements
__device__ void quantize_row_warp(const __half* src, int8_t* dst, float* scale_out, int d) {
  const int lane = threadIdx.x & 31;
  const int per = d / 32;                 // 2 or 4
  float x[4];
  float amax = 0.0f;
  for (int j = 0; j < per; ++j) {
    x[j] = __half2float(src[lane * per + j]);
    amax = fmaxf(amax, fabsf(x[j]));
  }
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
  for (int j = 0; j < per; ++j) {
    int q = 0;
    if (s != 0.0f) {
      q = __float2int_rn(__fdiv_rn(x[j], s));
      q = max(-127, min(127, q));
    }
    dst[lane * per + j] = static_cast<int8_t>(q);
  }
  if (lane == 0) *scale_out = s;
}

__global__ void __launch_bounds__(kThreads) k_select(Cache c, StepParams sp) {
  const int lb = blockIdx.x;
  const int l = lb / c.B, b = lb % c.B;
  const int tid = threadIdx.x;
  const int n8 = c.n8[lb], n16 = c.n16[lb];
  const int N = sp.btab[l * 2 + (sp.hi[b] ? 1 : 0)];
  const int t = sp.t;
  const int Hkv = c.Hkv, cap8 = c.cap8, W = c.W, P = c.P;
  const size_t lbs = static_cast<size_t>(lb) * c.slots;
  int32_t* pos8 = c.pos8 + static_cast<size_t>(lb) * cap8;
  int32_t* pos16 = c.pos16 + static_cast<size_t>(lb) * c.Wr;
  float* ema8 = c.ema8 + static_cast<size_t>(lb) * cap8;
  float* ema16 = c.ema16 + static_cast<size_t>(lb) * c.Wr;
  float* keys = c.keys + lbs;
  const float* mass = c.mass + static_cast<size_t>(lb) * Hkv * c.slots;

  __shared__ int s_prot, s_jage, s_D, s_k, s_cnt;
  __shared__ int s_hist[256];
  __shared__ int s_wsum[2 * kWarps];
  __shared__ unsigned long long s_min[kWarps];
  if (tid == 0) { s_prot = 0; s_jage = -1; }
  __syncthreads();

  // ---- phase A: EMA update and ranking keys of every cached token ----
  const float hqf = static_cast<float>(c.Hq);
  for (int i = tid; i < n8 + n16; i += kThreads) {
    const bool is8 = i < n8;
    const int j = is8 ? i : i - n8;
    const int sid = is8 ? j : cap8 + j;
    float asum = 0.0f;
    for (int h = 0; h < Hkv; ++h) asum = __fadd_rn(asum, mass[static_cast<size_t>(h) * c.slots + sid]);
    const float a = __fdiv_rn(asum, hqf);
    float* ep = is8 ? ema8 + j : ema16 + j;
    const float e = __fadd_rn(__fmul_rn(sp.beta, *ep), __fmul_rn(sp.omb, a));
    *ep = e;
    const int age = t - (is8 ? pos8[j] : pos16[j]);
    keys[sid] = __fadd_rn(e, __fdiv_rn(1.0f, static_cast<float>(1 + age)));
    if (!is8) {
      if (age < P) atomicAdd(&s_prot, 1);
      if (age == W) s_jage = j;
    }
  }
  __syncthreads();
  const int pcount = s_prot + 1;            // + the new token
  const int jage = s_jage;
  const int n_tot = n8 + n16 + 1;
  // candidate test: INT8 slots always, FP16 slots when age >= P
  // keep rule: mode 0 keep all, 1 keep none, 2 (k & mask) >= prefix, 3 k != kmin
  int mode = 0;
  unsigned long long mask = 0, prefix = 0, kmin = 0;
  if (n_tot > N) {
    const int ncand = n_tot - pcount;
    const int need = N - pcount;            // >= 0: N >= P >= pcount
    if (need <= 0) {
      mode = 1;
    } else if (ncand - need == 1) {
      unsigned long long v = ~0ull;
      for (int i = tid; i < n8 + n16; i += kThreads) {
        const bool is8 = i < n8;
        const int j = is8 ? i : i - n8;
        const int p = is8 ? pos8[j] : pos16[j];
        if (!is8 && t - p < P) continue;
        const unsigned long long k = key64(keys[is8 ? j : cap8 + j], p);
        v = k < v ? k : v;
      }
      kmin = block_min_u64(v, s_min);
      mode = 3;
    } else {
      mode = 2;
      int k = need;
      for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        for (int i = tid; i < 256; i += kThreads) s_hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < n8 + n16; i += kThreads) {
          const bool is8 = i < n8;
          const int j = is8 ? i : i - n8;
          const int p = is8 ? pos8[j] : pos16[j];
          if (!is8 && t - p < P) continue;
          const unsigned long long kk = key64(keys[is8 ? j : cap8 + j], p);
          if ((kk & mask) == prefix) atomicAdd(&s_hist[(kk >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid == 0) {
          int cum = 0, D = 0;
          for (D = 255; D > 0; --D) {
            if (cum + s_hist[D] >= k) break;
            cum += s_hist[D];
          }
          s_D = D;
          s_k = k - cum;
          s_cnt = s_hist[D];
        }
        __syncthreads();
        prefix |= static_cast<unsigned long long>(s_D) << shift;
        mask |= 255ull << shift;
        k = s_k;
        const bool done = (s_cnt == k);
        __syncthreads();
        if (done) break;
      }
    }
  }
  auto kept = [&](bool is8, int j) -> bool {
    const int p = is8 ? pos8[j] : pos16[j];
    if (!is8 && t - p < P) return true;
    if (mode == 0) return true;
    if (mode == 1) return false;
    const unsigned long long kk = key64(keys[is8 ? j : cap8 + j], p);
    if (mode == 2) return (kk & mask) >= prefix;
    return kk != kmin;
  };

  // ---- phase B: compaction plan of the INT8 region ----
  const bool keptA = (jage >= 0) && kept(false, jage);
  int k8 = 0;
  {
    int dummy = 0, tot = 0, tot2 = 0;
    for (int base = 0; base < n8; base += kThreads) {
      const int j = base + tid;
      int r1, r2;
      block_scan2(j < n8 && kept(true, j), false, s_wsum, r1, r2, tot, tot2);
      (void)r1; (void)r2; (void)dummy;
    }
    k8 = tot;
  }
  const int n8n = k8 + (keptA ? 1 : 0);
  int nmov8 = 0;
  {
    int toth = 0, totm = 0;
    const int lim = max(n8, n8n);
    int2* jobs = c.jobs8 + static_cast<size_t>(lb) * cap8;
    for (int base = 0; base < lim; base += kThreads) {
      const int j = base + tid;
      const bool hole = (j < n8n) && (j >= n8 || !kept(true, j));
      const bool mover = (j >= n8n) && (j < n8) && kept(true, j);
      int rh, rm;
      block_scan2(hole, mover, s_wsum, rh, rm, toth, totm);
      if (hole) jobs[rh].x = j;
      if (mover) jobs[rm].y = j;
    }
    nmov8 = totm;
  }
  // ---- FP16 region ----
  int k16 = 0;
  {
    int tot = 0, tot2 = 0;
    for (int base = 0; base < n16; base += kThreads) {
      const int j = base + tid;
      int r1, r2;
      block_scan2(j < n16 && j != jage && kept(false, j), false, s_wsum, r1, r2, tot, tot2);
    }
    k16 = tot;
  }
  const int n16n = k16 + 1;
  int nmov16 = 0;
  {
    int toth = 0, totm = 0;
    const int lim = max(n16, n16n);
    int2* jobs = c.jobs16 + static_cast<size_t>(lb) * c.Wr;
    for (int base = 0; base < lim; base += kThreads) {
      const int j = base + tid;
      const bool kn = (j < n16) && j != jage && kept(false, j);
      const bool hole = (j < n16n) && !kn;
      const bool mover = (j >= n16n) && kn;
      int rh, rm;
      block_scan2(hole, mover, s_wsum, rh, rm, toth, totm);
      if (hole) jobs[rh].x = j;
      if (mover) jobs[rm].y = j;
    }
    nmov16 = totm;
    if (tid == 0) jobs[nmov16].y = -1;      // the new token fills the last hole
  }
  __syncthreads();

  // ---- phase C: metadata moves (INT8 destinations first: the aging token is
  // read from its FP16 slot before any FP16 slot is overwritten) ----
  const int2* j8 = c.jobs8 + static_cast<size_t>(lb) * cap8;
  const int2* j16 = c.jobs16 + static_cast<size_t>(lb) * c.Wr;
  for (int r = tid; r < nmov8; r += kThreads) {
    const int2 jb = j8[r];
    pos8[jb.x] = pos8[jb.y];
    ema8[jb.x] = ema8[jb.y];
  }
  int hage = -1;
  if (keptA) hage = j8[nmov8].x;
  if (keptA && tid == 0) {
    pos8[hage] = pos16[jage];
    ema8[hage] = ema16[jage];
  }
  // the aging token's K/V rows: quantise FP16 slot jage into INT8 slot hage
  if (keptA) {
    const int warp = tid >> 5;
    for (int row = warp; row < 2 * Hkv; row += kWarps) {
      const int h = row >> 1;
      const bool isv = row & 1;
      const size_t u8 = static_cast<size_t>(lb) * Hkv + h;
      const __half* src = (isv ? c.v16 : c.k16) + (u8 * c.Wr + jage) * c.d;
      int8_t* dst = (isv ? c.v8 : c.k8) + (u8 * cap8 + hage) * c.d;
      float* sc = (isv ? c.vs : c.ks) + u8 * cap8 + hage;
      quantize_row_warp(src, dst, sc, c.d);
    }
  }
  __syncthreads();
  for (int r = tid; r < nmov16; r += kThreads) {
    const int2 jb = j16[r];
    pos16[jb.x] = pos16[jb.y];
    ema16[jb.x] = ema16[jb.y];
  }
  if (tid == 0) {
    const int hn = j16[nmov16].x;
    pos16[hn] = t;
    ema16[hn] = 0.0f;
  }
  __syncthreads();

  // ---- outputs ----
  if (sp.kept_pos) {
    int32_t* kp = sp.kept_pos + static_cast<size_t>(lb) * c.Ncap;
    for (int j = tid; j < n8n; j += kThreads) kp[j] = pos8[j];
    for (int j = tid; j < n16n; j += kThreads) kp[n8n + j] = pos16[j];
  }
  if (tid == 0) {
    if (sp.kept_count) sp.kept_count[lb] = n8n + n16n;
    c.n8[lb] = n8n;
    c.n16[lb] = n16n;
    c.njobs[lb * 2] = nmov8;
    c.njobs[lb * 2 + 1] = nmov16 + 1;
    atomicAdd(&c.stats->evicted, static_cast<unsigned long long>(n_tot - n8n - n16n));
    atomicAdd(&c.stats->quantized, keptA ? 1ull : 0ull);
    atomicAdd(&c.stats->moved, static_cast<unsigned long long>(nmov8 + nmov16));
    atomicAdd(&c.stats->kv_bytes,
              static_cast<unsigned long long>(Hkv) *
                  (static_cast<unsigned long long>(n8n) * (2ull * c.d + 8ull) +
                   static_cast<unsigned long long>(n16n) * 4ull * c.d));
  }
}

}  // namespace

cudaError_t launch_select(const Cache& c, const StepParams& sp, cudaStream_t s) {
  k_select<<<c.L * c.B, kThreads, 0, s>>>(c, sp);
  return cudaGetLastError();
}

}  // namespace confkv
