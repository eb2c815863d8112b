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
// One CTA of kThreads per (layer, sequence).  The same CTA then applies the
// compaction: metadata and K/V data moves of every KV head, the INT8
// quantisation of the aging token and the write of the new token.  Selection: the need-th largest
// 64-bit key (key bits << 32 | position; unique) is found by an 8-bit MSB
// radix select over the candidates (early exit once the boundary bucket is
// taken whole); a single eviction, the steady state, is one arg-min.
#include <cfloat>

#include "confkv_internal.cuh"

namespace confkv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kReg = 4;        // slots per thread held in registers

__device__ __forceinline__ unsigned long long key64(float key, int pos) {
  return (static_cast<unsigned long long>(__float_as_uint(key)) << 32) |
         static_cast<unsigned int>(pos);
}

// Block-wide exclusive scan of two per-thread counts (ranks in thread order).
__device__ __forceinline__ void block_scan2(int& a, int& b, int* wsum, int& tot_a, int& tot_b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
  for (int o = 1; o < 32; o <<= 1) {
    const int xa = __shfl_up_sync(0xffffffffu, ia, o);
    const int xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += xa; ib += xb; }
  }
  if (lane == 31) {
    wsum[warp] = ia;
    wsum[kWarps + warp] = ib;
  }
  __syncthreads();
  int oa = 0, ob = 0, ta = 0, tb = 0;
  for (int w = 0; w < kWarps; ++w) {
    const int xa = wsum[w], xb = wsum[kWarps + w];
    if (w < warp) { oa += xa; ob += xb; }
    ta += xa;
    tb += xb;
  }
  a = oa + ia - a;
  b = ob + ib - b;
  tot_a = ta;
  tot_b = tb;
  __syncthreads();
}

// Plan of one dense region of n live slots that keeps nn of them: the slots
// below nn that are not kept (holes) are filled, in rank order, by the kept
// slots at or above nn (movers).  jobs[r].x = hole r, jobs[r].y = mover r.
// Each thread scans 8 consecutive slots per pass.  Returns the mover count.
__device__ int plan_region(const unsigned char* f, int n, int nn, int2* jobs, int* wsum) {
  constexpr int kPer = 8;
  const int lim = max(n, nn);
  int hbase = 0, mbase = 0;
  for (int base = 0; base < lim; base += kThreads * kPer) {
    const int j0 = base + threadIdx.x * kPer;
    int hc = 0, mc = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int j = j0 + e;
      if (j < nn) hc += (j >= n || !f[j]) ? 1 : 0;
      else if (j < n) mc += f[j] ? 1 : 0;
    }
    int th, tm;
    block_scan2(hc, mc, wsum, th, tm);
    int rh = hbase + hc, rm = mbase + mc;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int j = j0 + e;
      if (j < nn) {
        if (j >= n || !f[j]) jobs[rh++].x = j;
      } else if (j < n && f[j]) {
        jobs[rm++].y = j;
      }
    }
    hbase += th;
    mbase += tm;
  }
  return mbase;
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
    dst[lane * per + j] = static_cast<int8_t>(q ^ 0x80);   // offset binary: code + 128
  }
  if (lane == 0) *scale_out = s;
}

__global__ void __launch_bounds__(kThreads, 2) k_select(Cache c, StepParams sp) {
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

  // ---- phase A: EMA update and ranking keys of every cached token.
  // Slots are taken kReg per thread per round with all loads issued first;
  // when n <= kReg * kThreads the 64-bit keys stay in registers for the
  // selection and the flag pass (otherwise they are re-read from `keys`).
  const int ntok = n8 + n16;
  const bool in_regs = ntok <= kReg * kThreads;
  unsigned long long rkey[kReg];
  bool rcand[kReg];
  unsigned long long lmin = ~0ull;
  int lprot = 0;
  const float hqf = static_cast<float>(c.Hq);
  for (int base = 0; base < ntok; base += kReg * kThreads) {
    int sid[kReg], pv[kReg];
    float ev[kReg], asum[kReg];
#pragma unroll
    for (int r = 0; r < kReg; ++r) {
      const int i = base + r * kThreads + tid;
      const bool is8 = i < n8;
      const int j = is8 ? i : i - n8;
      sid[r] = (i < ntok) ? (is8 ? j : cap8 + j) : -1;
      pv[r] = (i < ntok) ? (is8 ? pos8[j] : pos16[j]) : 0;
      ev[r] = (i < ntok) ? (is8 ? ema8[j] : ema16[j]) : 0.0f;
      asum[r] = 0.0f;
    }
    for (int h = 0; h < Hkv; ++h) {
      const float* mh = mass + static_cast<size_t>(h) * c.slots;
#pragma unroll
      for (int r = 0; r < kReg; ++r)
        if (sid[r] >= 0) asum[r] = __fadd_rn(asum[r], mh[sid[r]]);
    }
#pragma unroll
    for (int r = 0; r < kReg; ++r) {
      rcand[r] = false;
      if (sid[r] < 0) continue;
      const int i = base + r * kThreads + tid;
      const bool is8 = i < n8;
      const int j = is8 ? i : i - n8;
      const float a = __fdiv_rn(asum[r], hqf);
      const float e = __fadd_rn(__fmul_rn(sp.beta, ev[r]), __fmul_rn(sp.omb, a));
      if (is8) ema8[j] = e; else ema16[j] = e;
      const int age = t - pv[r];
      const float key = __fadd_rn(e, __fdiv_rn(1.0f, static_cast<float>(1 + age)));
      keys[sid[r]] = key;
      const bool prot = !is8 && age < P;
      if (prot) ++lprot;
      if (!is8 && age == W) s_jage = j;
      const unsigned long long k64 = key64(key, pv[r]);
      rkey[r] = k64;
      rcand[r] = !prot;
      if (!prot) lmin = k64 < lmin ? k64 : lmin;
    }
  }
  for (int o = 16; o > 0; o >>= 1) lprot += __shfl_xor_sync(0xffffffffu, lprot, o);
  if ((tid & 31) == 0 && lprot) atomicAdd(&s_prot, lprot);
  __syncthreads();
  const int pcount = s_prot + 1;            // + the new token
  const int jage = s_jage;
  const int n_tot = n8 + n16 + 1;
  // keep rule for candidates: mode 0 keep all, 1 keep none,
  // 2 (key & mask) >= prefix, 3 key != kmin (exactly one eviction)
  int mode = 0;
  unsigned long long mask = 0, prefix = 0, kmin = 0;
  // candidate key of slot i (unified order), or false if protected
  auto cand_key = [&](int i, unsigned long long& k64) -> bool {
    const bool is8 = i < n8;
    const int j = is8 ? i : i - n8;
    const int p = is8 ? pos8[j] : pos16[j];
    if (!is8 && t - p < P) return false;
    k64 = key64(keys[is8 ? j : cap8 + j], p);
    return true;
  };
  if (n_tot > N) {
    const int ncand = n_tot - pcount;
    const int need = N - pcount;            // >= 0: N >= P >= pcount
    if (need <= 0) {
      mode = 1;
    } else if (ncand - need == 1) {
      if (!in_regs) {
        lmin = ~0ull;
        for (int i = tid; i < ntok; i += kThreads) {
          unsigned long long k64;
          if (cand_key(i, k64)) lmin = k64 < lmin ? k64 : lmin;
        }
      }
      kmin = block_min_u64(lmin, s_min);
      mode = 3;
    } else {
      mode = 2;
      int k = need;
      for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        for (int i = tid; i < 256; i += kThreads) s_hist[i] = 0;
        __syncthreads();
        if (in_regs) {
#pragma unroll
          for (int r = 0; r < kReg; ++r)
            if (rcand[r] && (rkey[r] & mask) == prefix)
              atomicAdd(&s_hist[(rkey[r] >> shift) & 255u], 1);
        } else {
          for (int i = tid; i < ntok; i += kThreads) {
            unsigned long long kk;
            if (cand_key(i, kk) && (kk & mask) == prefix)
              atomicAdd(&s_hist[(kk >> shift) & 255u], 1);
          }
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
  auto keep_key = [&](unsigned long long kk) -> bool {
    if (mode == 0) return true;
    if (mode == 1) return false;
    if (mode == 2) return (kk & mask) >= prefix;
    return kk != kmin;
  };

  // ---- keep flags in shared memory: one pass over the slots ----
  // fl8[j]: INT8 slot j kept; fl16[j]: FP16 slot j kept and staying FP16
  extern __shared__ __align__(16) unsigned char fl[];
  unsigned char* fl8 = fl;
  unsigned char* fl16 = fl + cap8;
  int2* sj8 = reinterpret_cast<int2*>(fl + ((cap8 + c.Wr + 15) & ~15));   // [Ncap + 1]
  int2* sj16 = sj8 + c.Ncap + 1;                                            // [Wr]
  __shared__ int s_k8, s_k16, s_keptA;
  if (tid == 0) {
    s_k8 = 0;
    s_k16 = 0;
    s_keptA = 0;
  }
  __syncthreads();
  {
    int c8 = 0, c16 = 0;
    auto flag = [&](int i, bool cand, unsigned long long kk) {
      const bool k = !cand || keep_key(kk);
      if (i < n8) {
        fl8[i] = k;
        c8 += k;
      } else {
        const int j = i - n8;
        if (j == jage) {
          s_keptA = k;
          fl16[j] = 0;
        } else {
          fl16[j] = k;
          c16 += k;
        }
      }
    };
    if (in_regs) {
#pragma unroll
      for (int r = 0; r < kReg; ++r) {
        const int i = r * kThreads + tid;
        if (i < ntok) flag(i, rcand[r], rkey[r]);
      }
    } else {
      for (int i = tid; i < ntok; i += kThreads) {
        unsigned long long kk = 0;
        const bool cand = cand_key(i, kk);
        flag(i, cand, kk);
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      c8 += __shfl_xor_sync(0xffffffffu, c8, o);
      c16 += __shfl_xor_sync(0xffffffffu, c16, o);
    }
    if ((tid & 31) == 0) {
      atomicAdd(&s_k8, c8);
      atomicAdd(&s_k16, c16);
    }
  }
  __syncthreads();
  const bool keptA = s_keptA != 0;
  const int n8n = s_k8 + (keptA ? 1 : 0);
  const int n16n = s_k16 + 1;
  // ---- compaction plans: hole of rank r <- mover of rank r ----
  const int nmov8 = plan_region(fl8, n8, n8n, sj8, s_wsum);
  const int nmov16 = plan_region(fl16, n16, n16n, sj16, s_wsum);
  if (tid == 0) sj16[nmov16].y = -1;        // the new token fills the last FP16 hole
  __syncthreads();

  // ---- phase C: data and metadata moves.  INT8 destinations first: the
  // aging token is read from its FP16 slot before FP16 slots are rewritten ----
  const int2* j8 = sj8;
  const int2* j16 = sj16;
  const int d = c.d;
  const int warp = tid >> 5, lane = tid & 31;
  {
    // one warp per (move, KV head): lanes copy the 16-byte pieces of the K and
    // V rows, two more lanes the two scales
    const int cpr = d / 16;
    for (int p = warp; p < nmov8 * Hkv; p += kWarps) {
      const int r = p / Hkv, h = p - r * Hkv;
      const int2 jb = j8[r];
      const size_t u8 = (static_cast<size_t>(lb) * Hkv + h) * cap8;
      if (lane < 2 * cpr) {
        int8_t* base = (lane < cpr ? c.k8 : c.v8) + u8 * d;
        const int ch = lane < cpr ? lane : lane - cpr;
        reinterpret_cast<int4*>(base + static_cast<size_t>(jb.x) * d)[ch] =
            reinterpret_cast<const int4*>(base + static_cast<size_t>(jb.y) * d)[ch];
      } else if (lane < 2 * cpr + 2) {
        float* sc = (lane == 2 * cpr) ? c.ks : c.vs;
        sc[u8 + jb.x] = sc[u8 + jb.y];
      }
    }
  }
  for (int r = tid; r < nmov8; r += kThreads) {
    const int2 jb = j8[r];
    pos8[jb.x] = pos8[jb.y];
    ema8[jb.x] = ema8[jb.y];
  }
  if (keptA) {
    const int hage = j8[nmov8].x;
    if (tid == 0) {
      pos8[hage] = pos16[jage];
      ema8[hage] = ema16[jage];
    }
    // the aging token's K/V rows: quantise FP16 slot jage into INT8 slot hage
    for (int row = warp; row < 2 * Hkv; row += kWarps) {
      const int h = row >> 1;
      const bool isv = row & 1;
      const size_t u8 = static_cast<size_t>(lb) * Hkv + h;
      const __half* src = (isv ? c.v16 : c.k16) + (u8 * c.Wr + jage) * d;
      int8_t* dst = (isv ? c.v8 : c.k8) + (u8 * cap8 + hage) * d;
      float* sc = (isv ? c.vs : c.ks) + u8 * cap8 + hage;
      quantize_row_warp(src, dst, sc, d);
    }
  }
  __syncthreads();
  {
    // one warp per (FP16 move or new token, KV head): one lane per 16-byte piece
    const int cpr = d / 8;
    for (int p = warp; p < (nmov16 + 1) * Hkv; p += kWarps) {
      const int r = p / Hkv, h = p - r * Hkv;
      if (lane < 2 * cpr) {
        const int2 jb = j16[r];
        const size_t u8 = static_cast<size_t>(lb) * Hkv + h;
        const bool isv = lane >= cpr;
        const int ch = isv ? lane - cpr : lane;
        __half* base = (isv ? c.v16 : c.k16) + u8 * c.Wr * d;
        const __half* src = (jb.y >= 0) ? base + static_cast<size_t>(jb.y) * d
                                        : (isv ? sp.v_new : sp.k_new) + u8 * d;
        reinterpret_cast<int4*>(base + static_cast<size_t>(jb.x) * d)[ch] =
            reinterpret_cast<const int4*>(src)[ch];
      }
    }
  }
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
    int32_t* __restrict__ kp = sp.kept_pos + static_cast<size_t>(lb) * c.Ncap;
    for (int base = 0; base < n8n + n16n; base += 4 * kThreads) {
      int v[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = base + r * kThreads + tid;
        v[r] = (i < n8n) ? pos8[i] : (i < n8n + n16n ? pos16[i - n8n] : 0);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = base + r * kThreads + tid;
        if (i < n8n + n16n) kp[i] = v[r];
      }
    }
  }
  if (tid == 0) {
    if (sp.kept_count) sp.kept_count[lb] = n8n + n16n;
    c.n8[lb] = n8n;
    c.n16[lb] = n16n;
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
  const size_t smem = ((static_cast<size_t>(c.cap8) + c.Wr + 15) & ~static_cast<size_t>(15)) +
                      (static_cast<size_t>(c.Ncap) + 1 + c.Wr) * sizeof(int2);
  static size_t attr = 48 * 1024;
  if (smem > attr) {
    const cudaError_t e = cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = smem;
  }
  k_select<<<c.L * c.B, kThreads, smem, s>>>(c, sp);
  return cudaGetLastError();
}

}  // namespace confkv
