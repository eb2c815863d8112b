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
// Comparison policies (same selection, compaction and storage): WINDOW key
// 0 (the newest are kept), H2O acc = acc + a_i and key = acc, RANDOM key = a
// SplitMix64 draw in [0, 1) per (step, sequence, token).
// The fp32 operations use explicit _rn intrinsics so that no contraction
// changes the rounding: the decision is taken in fp32 on exact fp32 values.
//
// One CTA of kThreads per (layer, sequence), small enough for every CTA of
// the grid to be resident at once.  Keys stay in registers (kReg per thread).
// Selection: the need-th largest 64-bit key (key bits << 32 | position;
// unique) by an 8-bit MSB radix select over the candidates (early exit once
// the boundary bucket is taken whole); a single eviction, the steady state,
// is one arg-min.  Keep flags become 32-bit ballot masks; one warp per region
// turns them into the compaction plan with popc / ffs.  The same CTA then
// applies the compaction: metadata and K/V data moves of every KV head, the
// INT8 quantisation of the aging token and the write of the new token.  In
// the deferred form (per-layer steps, host-buffer steps) the new token's K/V
// rows are not yet known: the CTA only reserves their FP16 slot (new_slot)
// and the attention, or k_append, stores them.  The step position is the
// prefill length plus a per-(layer, sequence) device counter this kernel
// advances, so a captured step replays as the next one.
#include <cfloat>

#include "../../include/confkv.h"

#include "confkv_internal.cuh"

namespace confkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kReg = 8;        // slots per thread held in registers (n <= 2048)

// RANDOM policy: a uniform draw in [0, 1) per (step, sequence, token), the
// top 24 bits of the SplitMix64 finaliser (Steele, Lea and Flood) chained
// over (seed, t, l*B + b, position); exact in fp32.
__device__ __forceinline__ uint64_t splitmix_mix(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}
__device__ __forceinline__ float random_key(uint64_t seed, int t, int lb, int pos) {
  uint64_t h = splitmix_mix(seed);
  h = splitmix_mix(h ^ static_cast<uint64_t>(static_cast<uint32_t>(t)));
  h = splitmix_mix(h ^ static_cast<uint64_t>(static_cast<uint32_t>(lb)));
  h = splitmix_mix(h ^ static_cast<uint64_t>(static_cast<uint32_t>(pos)));
  return static_cast<float>(static_cast<uint32_t>(h >> 40)) * 0x1p-24f;
}

__device__ __forceinline__ unsigned long long key64(float key, int pos) {
  return (static_cast<unsigned long long>(__float_as_uint(key)) << 32) |
         static_cast<unsigned int>(pos);
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

// bits [0, k) set (k clamped to [0, 32])
__device__ __forceinline__ unsigned lowmask(int k) {
  return k >= 32 ? 0xffffffffu : (k <= 0 ? 0u : ((1u << k) - 1u));
}

// Compaction plan of one dense region, by one warp.  bits: word q holds the
// keep flags of slots [32q, 32q + 32) (bits at or beyond n are ignored).
// The region keeps kc + extra slots (extra: tokens that arrive in it);
// holes = slots below min(n, nn) not kept, then slot n when nn > n;
// movers = kept slots in [nn, n).  jobs[r].x = hole r, jobs[r].y = mover r,
// both in slot order.  Returns the mover count; *nn_out = nn.
__device__ int plan_warp(const unsigned* bits, int n, int extra, int2* jobs, int* nn_out) {
  const int lane = threadIdx.x & 31;
  const int nw = (n + 31) >> 5;
  const int per = (nw + 31) >> 5;
  const int w0 = min(nw, lane * per), w1 = min(nw, w0 + per);
  int kc = 0;
  for (int q = w0; q < w1; ++q) kc += __popc(bits[q] & lowmask(n - 32 * q));
  for (int o = 16; o > 0; o >>= 1) kc += __shfl_xor_sync(0xffffffffu, kc, o);
  const int nn = kc + extra;
  const int hl = min(n, nn);
  int hc = 0, mc = 0;
  for (int q = w0; q < w1; ++q) {
    const unsigned kb = bits[q];
    hc += __popc(~kb & lowmask(hl - 32 * q));
    mc += __popc(kb & lowmask(n - 32 * q) & ~lowmask(nn - 32 * q));
  }
  int hs = hc, ms = mc;                     // inclusive scans over lanes
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, hs, o);
    const int y = __shfl_up_sync(0xffffffffu, ms, o);
    if (lane >= o) { hs += x; ms += y; }
  }
  const int htot = __shfl_sync(0xffffffffu, hs, 31), mtot = __shfl_sync(0xffffffffu, ms, 31);
  hs -= hc;
  ms -= mc;
  for (int q = w0; q < w1; ++q) {
    const unsigned kb = bits[q];
    unsigned hm = ~kb & lowmask(hl - 32 * q);
    unsigned mm = kb & lowmask(n - 32 * q) & ~lowmask(nn - 32 * q);
    while (hm) {
      const int bit = __ffs(hm) - 1;
      jobs[hs++].x = 32 * q + bit;
      hm &= hm - 1u;
    }
    while (mm) {
      const int bit = __ffs(mm) - 1;
      jobs[ms++].y = 32 * q + bit;
      mm &= mm - 1u;
    }
  }
  if (nn > n && lane == 0) jobs[htot].x = n;  // the arriving token's slot past the end
  *nn_out = nn;
  return mtot;
}

// The fp32 steps of the INT8 absmax quantiser of one fp16 row of d = 32 * per
// elements, lane holding elements lane * per + j: amax over the row, scale =
// amax / 127, code = round-half-even(x / scale) clamped to +-127, stored
// offset-binary (code + 128).  Byte j of the result is element lane*per + j.
__device__ __forceinline__ uint32_t quantize_lane(const float (&x)[4], int per, float& scale) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < per) amax = fmaxf(amax, fabsf(x[j]));
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
  uint32_t packed = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int q = 0;
    if (j < per && s != 0.0f) {
      q = __float2int_rn(__fdiv_rn(x[j], s));
      q = max(-127, min(127, q));
    }
    packed |= static_cast<uint32_t>((q ^ 0x80) & 0xff) << (8 * j);
  }
  scale = s;
  return packed;
}

// warp-level INT8 absmax quantisation of one fp16 row of d elements; fe
// (null: none) holds the row's channel exponents (x_c is divided by 2^f_c)
__device__ void quantize_row_warp(const __half* src, int8_t* dst, float* scale_out, int d,
                                  const int8_t* fe) {
  const int lane = threadIdx.x & 31;
  const int per = d / 32;                 // 2 or 4
  float x[4];
  float amax = 0.0f;
  for (int j = 0; j < per; ++j) {
    x[j] = __half2float(src[lane * per + j]);
    if (fe) x[j] *= chan_inv_factor(fe[lane * per + j]);       // exact: x * 2^-f
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

template <int kPolicy>
__global__ void __launch_bounds__(kThreads, 4) k_select(Cache c, StepParams sp) {
  const int lb = sp.lb0 + blockIdx.x;
  const int lbu = blockIdx.x;                 // index into the caller's buffers
  const int l = lb / c.B, b = lb % c.B;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();     // the attention may be scheduled (it waits for this grid)
  // n8, n16, the step count, positions, EMA and mass come from the previous
  // step, which the confidence kernel has already waited for; the budget is
  // read after pdl_wait() below
  const int n8 = c.n8[lb], n16 = c.n16[lb];
  const int nstep = c.tstep[lb];
  const int t = sp.t0 + nstep;
  const int Hkv = c.Hkv, cap8 = c.cap8, W = c.W, P = c.P, d = c.d;
  int32_t* pos8 = c.pos8 + static_cast<size_t>(lb) * cap8;
  int32_t* pos16 = c.pos16 + static_cast<size_t>(lb) * c.Wr;
  float* ema8 = c.ema8 + static_cast<size_t>(lb) * cap8;
  float* ema16 = c.ema16 + static_cast<size_t>(lb) * c.Wr;
  float* keys = c.keys + static_cast<size_t>(lb) * c.slots;
  const float* mass = c.mass + static_cast<size_t>(lb) * Hkv * c.slots;

  // dynamic shared memory: unified keep mask | FP16 keep mask | INT8 jobs | FP16 jobs
  extern __shared__ __align__(16) unsigned char dsm[];
  const int uwords = (cap8 + c.Wr) / 32 + 2;
  const int fwords = c.Wr / 32 + 2;
  unsigned* ubits = reinterpret_cast<unsigned*>(dsm);
  unsigned* fbits = ubits + uwords;
  int2* sj8 = reinterpret_cast<int2*>(dsm + ((static_cast<size_t>(uwords + fwords) * 4 + 15) & ~static_cast<size_t>(15)));
  int2* sj16 = sj8 + c.Ncap + 1;

  __shared__ int s_prot, s_jage, s_D, s_k, s_cnt, s_keptA, s_nn8, s_nn16, s_mov8, s_mov16;
  __shared__ int s_hist[256];
  __shared__ unsigned long long s_min[kWarps];
  if (tid == 0) { s_prot = 0; s_jage = -1; s_keptA = 0; }
  __syncthreads();

  // ---- phase A: EMA update and ranking keys of every cached token.
  // Slot i (unified order: INT8 slots, then FP16 slots) of round `base` is
  // base + r * kThreads + tid; all loads of a half-round are issued first.
  const int ntok = n8 + n16;
  const bool in_regs = ntok <= kReg * kThreads;
  unsigned long long rkey[kReg];
  unsigned rcand = 0;                       // bit r: slot of register r is a candidate
  unsigned long long lmin = ~0ull;
  int lprot = 0;
  const float hqf = static_cast<float>(c.Hq);
  // the EMA (CONF-KV) and the accumulated mass (H2O) read the previous
  // attention's per-token mass; WINDOW and RANDOM rank without it
  constexpr bool use_mass = kPolicy == CONFKV_POLICY_CONFKV || kPolicy == CONFKV_POLICY_H2O;
for (int base = 0; base < ntok; base += kReg * kThreads) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      constexpr int kH = kReg / 2;
      int sid[kH], pv[kH];
      float ev[kH], asum[kH];
#pragma unroll
      for (int r = 0; r < kH; ++r) {
        const int i = base + (half * kH + r) * kThreads + tid;
        const bool is8 = i < n8;
        const int j = is8 ? i : i - n8;
        sid[r] = (i < ntok) ? (is8 ? j : cap8 + j) : -1;
        pv[r] = (i < ntok) ? (is8 ? pos8[j] : pos16[j]) : 0;
        if constexpr (use_mass) {
          ev[r] = (i < ntok) ? (is8 ? ema8[j] : ema16[j]) : 0.0f;
        } else {
          ev[r] = 0.0f;
        }
        asum[r] = 0.0f;
      }
      if constexpr (use_mass) {
        for (int h = 0; h < Hkv; ++h) {
          const float* mh = mass + static_cast<size_t>(h) * c.slots;
#pragma unroll
          for (int r = 0; r < kH; ++r)
            if (sid[r] >= 0) asum[r] = __fadd_rn(asum[r], mh[sid[r]]);
        }
      }
#pragma unroll
      for (int r = 0; r < kH; ++r) {
        const int rr = half * kH + r;
        if (sid[r] < 0) { rkey[rr] = 0; continue; }
        const int i = base + rr * kThreads + tid;
        const bool is8 = i < n8;
        const int j = is8 ? i : i - n8;
        const int age = t - pv[r];
        float key;
        if constexpr (kPolicy == CONFKV_POLICY_CONFKV) {
          const float a = __fdiv_rn(asum[r], hqf);
          const float e = __fadd_rn(__fmul_rn(sp.beta, ev[r]), __fmul_rn(sp.omb, a));
          if (is8) ema8[j] = e; else ema16[j] = e;
          key = __fadd_rn(e, __fdiv_rn(1.0f, static_cast<float>(1 + age)));
        } else if constexpr (kPolicy == CONFKV_POLICY_H2O) {
          const float e = __fadd_rn(ev[r], __fdiv_rn(asum[r], hqf));   // accumulated mass
          if (is8) ema8[j] = e; else ema16[j] = e;
          key = e;
        } else if constexpr (kPolicy == CONFKV_POLICY_RANDOM) {
          key = random_key(sp.seed, t, lb, pv[r]);
        } else {
          key = 0.0f;                                                   // WINDOW
        }
        keys[sid[r]] = key;
        const bool prot = !is8 && age < P;
        if (prot) ++lprot;
        if (!is8 && age == W) s_jage = j;
        const unsigned long long k64 = key64(key, pv[r]);
        rkey[rr] = k64;
        if (!prot) {
          rcand |= 1u << rr;
          lmin = k64 < lmin ? k64 : lmin;
        }
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) lprot += __shfl_xor_sync(0xffffffffu, lprot, o);
  if (lane == 0 && lprot) atomicAdd(&s_prot, lprot);
  pdl_wait();        // the confidence kernel's budget flags are complete
  const int N = sp.btab[l * 2 + (sp.hi[b] ? 1 : 0)];
  __syncthreads();
  // Every thread has read the previous attention's per-token mass, which this
  // step's attention rewrites for every live slot before the next read: drop
  // its whole 128-byte lines from L2 without a write-back.
  if constexpr (use_mass) {
    const int l8 = n8 >> 5, l16 = n16 >> 5, per = l8 + l16;
    for (int x = tid; x < Hkv * per; x += kThreads) {
      const int h = x / per, r = x - h * per;
      const float* line = mass + static_cast<size_t>(h) * c.slots + (r < l8 ? 32 * r : cap8 + 32 * (r - l8));
      if ((reinterpret_cast<uintptr_t>(line) & 127u) == 0) l2_discard_line(line);
    }
  }
  const int pcount = s_prot + 1;            // + the new token
  const int jage = s_jage;
  // The token leaving the FP16 window (age W) is quantised now, before the
  // selection decides whether it stays, so that its row loads and divisions
  // overlap the selection; its codes are stored once its INT8 slot is known.
  // Warp w takes rows w and w + kWarps of the 2 * Hkv (K, V) rows.
  constexpr int kQRows = 2;
  const bool early_q = jage >= 0 && 2 * Hkv <= kWarps * kQRows;
  uint32_t qcode[kQRows] = {0u, 0u};
  float qscale[kQRows] = {0.0f, 0.0f};
  if (early_q) {
    const int per = d / 32;                 // 2 or 4
    float xr[kQRows][4];
#pragma unroll
    for (int rr = 0; rr < kQRows; ++rr) {
      const int row = warp + rr * kWarps;
      const int h = row >> 1;
      const __half* src = ((row & 1) ? c.v16 : c.k16) +
                          ((static_cast<size_t>(lb) * Hkv + h) * c.Wr + jage) * d + lane * per;
      const int8_t* fe = (c.chexp && row < 2 * Hkv)
                             ? c.chexp + ((static_cast<size_t>(lb) * Hkv + h) * 2 + (row & 1)) * d +
                                   lane * per
                             : nullptr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xr[rr][j] = (row < 2 * Hkv && j < per) ? __half2float(src[j]) : 0.0f;
        if (fe && j < per) xr[rr][j] *= chan_inv_factor(fe[j]);   // exact: x * 2^-f
      }
    }
#pragma unroll
    for (int rr = 0; rr < kQRows; ++rr) qcode[rr] = quantize_lane(xr[rr], per, qscale[rr]);
  }
  const int n_tot = ntok + 1;
  // keep rule for candidates: mode 0 keep all, 1 keep none,
  // 2 (key & mask) >= prefix, 3 key != kmin (exactly one eviction)
  int mode = 0;
  unsigned long long mask = 0, prefix = 0, kmin = 0;
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
            if (((rcand >> r) & 1u) && (rkey[r] & mask) == prefix)
              atomicAdd(&s_hist[(rkey[r] >> shift) & 255u], 1);
        } else {
          for (int i = tid; i < ntok; i += kThreads) {
            unsigned long long kk;
            if (cand_key(i, kk) && (kk & mask) == prefix)
              atomicAdd(&s_hist[(kk >> shift) & 255u], 1);
          }
        }
        __syncthreads();
        if (warp == 0) {
          // the highest bucket D whose count from the top reaches k: lane q
          // holds buckets 255 - 8q .. 248 - 8q; scan across lanes, then within
          // the first lane whose running total reaches k (one always does:
          // the candidates under the prefix number at least k)
          int h8[8], sum = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            h8[j] = s_hist[255 - 8 * lane - j];
            sum += h8[j];
          }
          int incl = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
          }
          const unsigned reach = __ballot_sync(0xffffffffu, incl >= k);
          const int first = reach ? __ffs(reach) - 1 : 31;
          if (lane == first) {
            int cum = incl - sum, D = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (cum + h8[j] >= k || 8 * lane + j == 255) {     // bucket 0 is the last resort
                D = 255 - 8 * lane - j;
                break;
              }
              cum += h8[j];
            }
            s_D = D;
            s_k = k - cum;
            s_cnt = s_hist[D];
          }
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

  // ---- keep masks: bit i of ubits = unified slot i kept (and, for the FP16
  // region, staying FP16: the aging token's bit is cleared) ----
  {
    auto put = [&](int rr, int i, bool cand, unsigned long long kk) {
      bool k = false;
      if (i < ntok) {
        k = !cand || keep_key(kk);
        if (i >= n8 && i - n8 == jage) {
          s_keptA = k;
          k = false;
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, k);
      if (lane == 0) ubits[rr * kWarps + warp] = m;
    };
    if (in_regs) {
#pragma unroll
      for (int rr = 0; rr < kReg; ++rr) {
        const int i = rr * kThreads + tid;
        if (rr * kThreads < ntok) put(rr, i, (rcand >> rr) & 1u, rkey[rr]);
      }
    } else {
      const int rounds = (ntok + kThreads - 1) / kThreads;
      for (int rr = 0; rr < rounds; ++rr) {
        const int i = rr * kThreads + tid;
        unsigned long long kk = 0;
        const bool cand = (i < ntok) ? cand_key(i, kk) : false;
        put(rr, i, cand, kk);
      }
    }
    const int nw = (ntok + 31) / 32;
    for (int q = nw + tid; q < uwords; q += kThreads) ubits[q] = 0u;
  }
  __syncthreads();
  // FP16 keep mask: unified bits [n8, n8 + n16) shifted down to slot 0
  for (int q = tid; q < (n16 + 31) / 32; q += kThreads) {
    const int bit0 = n8 + 32 * q;
    fbits[q] = __funnelshift_r(ubits[bit0 >> 5], ubits[(bit0 >> 5) + 1], bit0 & 31);
  }
  __syncthreads();
  const bool keptA = s_keptA != 0;
  // ---- compaction plans: warp 0 the INT8 region, warp 1 the FP16 region ----
  if (warp == 0) {
    int nn;
    const int mv = plan_warp(ubits, n8, keptA ? 1 : 0, sj8, &nn);
    if (lane == 0) { s_nn8 = nn; s_mov8 = mv; }
  } else if (warp == 1) {
    int nn;
    const int mv = plan_warp(fbits, n16, 1, sj16, &nn);
    if (lane == 0) {
      s_nn16 = nn;
      s_mov16 = mv;
      sj16[mv].y = -1;                      // the new token fills the last FP16 hole
    }
  }
  __syncthreads();
  const int n8n = s_nn8, n16n = s_nn16, nmov8 = s_mov8, nmov16 = s_mov16;

  // ---- data and metadata moves.  INT8 destinations first: the aging token
  // is read from its FP16 slot before FP16 slots are rewritten ----
  {
    // INT8 moves: every (move, KV head, 16-byte piece of K or V) is one item;
    // each thread loads 4 items before storing them (4 loads in flight)
    const int cpr = d / 16, per = 2 * cpr, items = nmov8 * Hkv * per;
    for (int base = 0; base < items; base += 4 * kThreads) {
      int4 v[4];
      int8_t* dst[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * kThreads + tid;
        dst[u] = nullptr;
        if (it < items) {
          const int r = it / (Hkv * per);
          const int rem = it - r * Hkv * per;
          const int h = rem / per, pc = rem - h * per;
          const int2 jb = sj8[r];
          int8_t* rows = (pc < cpr ? c.k8 : c.v8) + (static_cast<size_t>(lb) * Hkv + h) * cap8 * d;
          const int ch = pc < cpr ? pc : pc - cpr;
          v[u] = reinterpret_cast<const int4*>(rows + static_cast<size_t>(jb.y) * d)[ch];
          dst[u] = rows + static_cast<size_t>(jb.x) * d + 16 * ch;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (dst[u]) *reinterpret_cast<int4*>(dst[u]) = v[u];
    }
    for (int it = tid; it < nmov8 * Hkv; it += kThreads) {
      const int r = it / Hkv, h = it - r * Hkv;
      const int2 jb = sj8[r];
      const size_t u8 = (static_cast<size_t>(lb) * Hkv + h) * cap8;
      const float ksv = c.ks[u8 + jb.y], vsv = c.vs[u8 + jb.y];
      c.ks[u8 + jb.x] = ksv;
      c.vs[u8 + jb.x] = vsv;
    }
  }
  for (int r = tid; r < nmov8; r += kThreads) {
    const int2 jb = sj8[r];
    pos8[jb.x] = pos8[jb.y];
    ema8[jb.x] = ema8[jb.y];
  }
  if (keptA) {
    const int hage = sj8[nmov8].x;
    if (tid == 0) {
      pos8[hage] = pos16[jage];
      ema8[hage] = ema16[jage];
    }
    // the aging token's K/V rows: FP16 slot jage -> INT8 slot hage
    if (early_q) {
      const int per = d / 32;
#pragma unroll
      for (int rr = 0; rr < kQRows; ++rr) {
        const int row = warp + rr * kWarps;
        if (row < 2 * Hkv) {
          const bool isv = row & 1;
          const size_t u8 = static_cast<size_t>(lb) * Hkv + (row >> 1);
          int8_t* dst = (isv ? c.v8 : c.k8) + (u8 * cap8 + hage) * d + lane * per;
          if (per == 4) *reinterpret_cast<uint32_t*>(dst) = qcode[rr];
          else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(qcode[rr]);
          if (lane == 0) ((isv ? c.vs : c.ks) + u8 * cap8)[hage] = qscale[rr];
        }
      }
    } else {
      for (int row = warp; row < 2 * Hkv; row += kWarps) {
        const int h = row >> 1;
        const bool isv = row & 1;
        const size_t u8 = static_cast<size_t>(lb) * Hkv + h;
        const __half* src = (isv ? c.v16 : c.k16) + (u8 * c.Wr + jage) * d;
        int8_t* dst = (isv ? c.v8 : c.k8) + (u8 * cap8 + hage) * d;
        float* sc = (isv ? c.vs : c.ks) + u8 * cap8 + hage;
        quantize_row_warp(src, dst, sc, d, c.chexp ? c.chexp + (u8 * 2 + (isv ? 1 : 0)) * d : nullptr);
      }
    }
  }
  __syncthreads();
  {
    // FP16 moves and the new token: (move, KV head, 16-byte piece) items,
    // 4 loads in flight per thread
    const int cpr = d / 8, per = 2 * cpr,
              items = (nmov16 + (sp.defer_new ? 0 : 1)) * Hkv * per;
    for (int base = 0; base < items; base += 4 * kThreads) {
      int4 v[4];
      __half* dst[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * kThreads + tid;
        dst[u] = nullptr;
        if (it < items) {
          const int r = it / (Hkv * per);
          const int rem = it - r * Hkv * per;
          const int h = rem / per, pc = rem - h * per;
          const int2 jb = sj16[r];
          const size_t u8 = static_cast<size_t>(lb) * Hkv + h;
          const bool isv = pc >= cpr;
          const int ch = isv ? pc - cpr : pc;
          __half* rows = (isv ? c.v16 : c.k16) + u8 * c.Wr * d;
          const __half* src = (jb.y >= 0) ? rows + static_cast<size_t>(jb.y) * d
                                          : (isv ? sp.v_new : sp.k_new) +
                                                (static_cast<size_t>(lbu) * Hkv + h) * d;
          v[u] = reinterpret_cast<const int4*>(src)[ch];
          dst[u] = rows + static_cast<size_t>(jb.x) * d + 8 * ch;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (dst[u]) *reinterpret_cast<int4*>(dst[u]) = v[u];
    }
  }
  for (int r = tid; r < nmov16; r += kThreads) {
    const int2 jb = sj16[r];
    pos16[jb.x] = pos16[jb.y];
    ema16[jb.x] = ema16[jb.y];
  }
  if (tid == 0) {
    const int hn = sj16[nmov16].x;
    pos16[hn] = t;
    ema16[hn] = 0.0f;
    if (sp.defer_new) c.new_slot[lb] = hn;
    c.tstep[lb] = nstep + 1;
    if (lb == 0) c.stats->steps += 1ull;
  }
  __syncthreads();

  // ---- outputs ----
  if (sp.kept_pos) {
    int32_t* __restrict__ kp = sp.kept_pos + static_cast<size_t>(lbu) * c.Ncap;
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
    if (sp.kept_count) sp.kept_count[lbu] = n8n + n16n;
    c.n8[lb] = n8n;
    c.n16[lb] = n16n;
    atomicAdd(&c.stats->evicted, static_cast<unsigned long long>(n_tot - n8n - n16n));
    atomicAdd(&c.stats->quantized, keptA ? 1ull : 0ull);
    atomicAdd(&c.stats->moved, static_cast<unsigned long long>(nmov8 + nmov16));
    atomicAdd(&c.stats->kv_bytes,
              static_cast<unsigned long long>(Hkv) *
                  (static_cast<unsigned long long>(n8n) * (2ull * d + 8ull) +
                   static_cast<unsigned long long>(n16n) * 4ull * d));
  }
}

// The arriving token of a deferred selection, one CTA per (layer, sequence):
// its K/V rows go to the FP16 slot the selection reserved, then the kept
// positions (INT8 slots, then FP16 slots) are reported.
__global__ void __launch_bounds__(kThreads) k_append(Cache c, StepParams sp) {
  const int lb = sp.lb0 + blockIdx.x;
  const int lbu = blockIdx.x;                 // index into the caller's buffers
  const int tid = threadIdx.x;
  pdl_trigger();     // the attention reads only its queries before its own wait
  pdl_wait();        // the selection that reserved the slot is complete
  const int Hkv = c.Hkv, d = c.d, hn = c.new_slot[lb];
  const int cpr = d / 8, items = Hkv * 2 * cpr;    // 16-byte pieces of K and V
  for (int it = tid; it < items; it += kThreads) {
    const int h = it / (2 * cpr), pc = it - h * 2 * cpr;
    const bool isv = pc >= cpr;
    const int ch = isv ? pc - cpr : pc;
    const size_t u = static_cast<size_t>(lb) * Hkv + h;
    const int4 v = reinterpret_cast<const int4*>((isv ? sp.v_new : sp.k_new) +
                                                 (static_cast<size_t>(lbu) * Hkv + h) * d)[ch];
    reinterpret_cast<int4*>((isv ? c.v16 : c.k16) + (u * c.Wr + hn) * d)[ch] = v;
  }
  const int n8 = c.n8[lb], n16 = c.n16[lb];
  if (sp.kept_pos) {
    const int32_t* pos8 = c.pos8 + static_cast<size_t>(lb) * c.cap8;
    const int32_t* pos16 = c.pos16 + static_cast<size_t>(lb) * c.Wr;
    int32_t* __restrict__ kp = sp.kept_pos + static_cast<size_t>(lbu) * c.Ncap;
    for (int i = tid; i < n8 + n16; i += kThreads) kp[i] = (i < n8) ? pos8[i] : pos16[i - n8];
  }
  if (sp.kept_count && tid == 0) sp.kept_count[lbu] = n8 + n16;
}

}  // namespace

size_t select_smem_bytes(const Cache& c) {
  const size_t uwords = (static_cast<size_t>(c.cap8) + c.Wr) / 32 + 2;
  const size_t fwords = static_cast<size_t>(c.Wr) / 32 + 2;
  return (((uwords + fwords) * 4 + 15) & ~static_cast<size_t>(15)) +
         (static_cast<size_t>(c.Ncap) + 1 + c.Wr) * sizeof(int2);
}

namespace {

template <int kPolicy>
cudaError_t launch_select_p(const Cache& c, const StepParams& sp, size_t smem, cudaStream_t s) {
  // the largest dynamic shared memory set so far, per device (the same
  // process may drive several devices; devices past the bound are not cached)
  constexpr int kMaxDevicesCached = 64;
  static size_t attr[kMaxDevicesCached] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesCached) dev = -1;
  const size_t have = dev >= 0 ? attr[dev] : 0;
  if (smem > 48 * 1024 && smem > have) {
    const cudaError_t e = cudaFuncSetAttribute(k_select<kPolicy>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0) attr[dev] = smem;
  }
  const cudaError_t e = launch_pdl(k_select<kPolicy>, dim3(sp.nlb), dim3(kThreads), smem, s, c, sp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const Cache& c, const StepParams& sp, cudaStream_t s) {
  const size_t smem = select_smem_bytes(c);
  switch (sp.policy) {
    case CONFKV_POLICY_CONFKV: return launch_select_p<CONFKV_POLICY_CONFKV>(c, sp, smem, s);
    case CONFKV_POLICY_WINDOW: return launch_select_p<CONFKV_POLICY_WINDOW>(c, sp, smem, s);
    case CONFKV_POLICY_H2O: return launch_select_p<CONFKV_POLICY_H2O>(c, sp, smem, s);
    case CONFKV_POLICY_RANDOM: return launch_select_p<CONFKV_POLICY_RANDOM>(c, sp, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_append(const Cache& c, const StepParams& sp, cudaStream_t s) {
  const cudaError_t e = launch_pdl(k_append, dim3(sp.nlb), dim3(kThreads), 0, s, c, sp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace confkv
