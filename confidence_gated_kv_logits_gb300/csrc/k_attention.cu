// K4: split-K decode attention over the INT8 and FP16 regions, with the INT8
// dequantisation fused into the block reads and an online-softmax merge; it
// also produces the per-token attention mass the next step's EMA needs.
//
// CONF-KV page, Technische Samenvatting:
//   Implementatie  dequantisation is fused with block-wise attention reads.
//   Belangrijkste Bijdragen / Systeemontwerp  block-wise online-softmax
//     attention over mixed FP16/INT8 storage.
//   Tokenrangschikking  the EMA attention mass of each cached token.
//
// Work unit: one (layer, sequence, KV head) -- the whole GQA group of g query
// heads shares each K/V row read -- split over `splits` CTAs along the token
// axis (INT8 slots first, then FP16 slots).  Each warp runs an online softmax
// over 32-token tiles; warps and then splits are merged with the usual
// (max, sum, acc) rescaling.  A split-K unit is finished by whichever CTA
// takes the last ticket (an atomic counter; no CTA ever waits).
//
// The raw scores s_{h,i} are written to `scores`; once the final (max, sum)
// of every head is known the finishing CTA turns them into the per-token mass
// sum_h exp(s_{h,i} - max_h) / sum_h, summed over the group.
//
// Per-(head, channel) storage mode (c.chexp set): an INT8 element reads as
// code * s * 2^f_c; the INT8 keys meet a copy of the query whose channel c is
// multiplied by 2^f_c (fp32, exact), and the INT8 values are multiplied by
// 2^f_c as they are dequantised.
#include <cfloat>

#include "confkv_internal.cuh"

namespace confkv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float rescale(float m_old, float m_new) {
  return (m_old == -INFINITY) ? 0.0f : expf(m_old - m_new);
}

template <int D>
__global__ void __launch_bounds__(kThreads) k_attn_simple(Cache c, AttnParams ap) {
  constexpr int DPL = D / 32;
  const int unit = ap.lb0 * c.Hkv + blockIdx.x, split = blockIdx.y;
  const int lb = unit / c.Hkv, kvh = unit - lb * c.Hkv, g = c.g;
  const int lbu = lb - ap.lb0;                // index into the caller's q / out
  const int n8 = c.n8[lb], n16 = c.n16[lb], n = n8 + n16;
  const int ntiles = (n + kTile - 1) / kTile;
  const int tps = (ntiles + ap.splits - 1) / ap.splits;
  const int t0 = min(ntiles, split * tps), t1 = min(ntiles, t0 + tps);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ float smem[];
  float* qs = smem;                         // [g][D]
  float* qs8 = qs + g * D;                  // [g][D] query of the INT8 keys (channel factors)
  float* wm = c.chexp ? qs8 + g * D : qs8;  // [kWarps][g]
  float* wl = wm + kWarps * g;              // [kWarps][g]
  float* fin = wl + kWarps * g;             // [2][g] final max, sum
  float* wacc = fin + 2 * g;                // [kWarps][g][D]

  const size_t qbase = (static_cast<size_t>(lbu) * c.Hq + kvh * g) * D;
  const int8_t* fk = c.chexp ? c.chexp + static_cast<size_t>(unit) * 2 * D : nullptr;
  for (int i = tid; i < g * D; i += kThreads) {
    qs[i] = __half2float(ap.q[qbase + i]);
    if (fk) qs8[i] = qs[i] * chan_factor(fk[i % D]);
  }
  const float* qk8 = fk ? qs8 : qs;
  float vfac[DPL];                           // V channel factors of this lane's channels
#pragma unroll
  for (int k = 0; k < DPL; ++k) vfac[k] = fk ? chan_factor(fk[D + lane + 32 * k]) : 1.0f;
  __syncthreads();

  float m[kMaxGroup], lsum[kMaxGroup], acc[kMaxGroup][DPL];
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    m[h] = -INFINITY;
    lsum[h] = 0.0f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[h][k] = 0.0f;
  }

  const int8_t* K8 = c.k8 + static_cast<size_t>(unit) * c.cap8 * D;
  const int8_t* V8 = c.v8 + static_cast<size_t>(unit) * c.cap8 * D;
  const float* KS = c.ks + static_cast<size_t>(unit) * c.cap8;
  const float* VS = c.vs + static_cast<size_t>(unit) * c.cap8;
  const __half* K16 = c.k16 + static_cast<size_t>(unit) * c.Wr * D;
  const __half* V16 = c.v16 + static_cast<size_t>(unit) * c.Wr * D;
  float* SC = c.scores + (static_cast<size_t>(lb) * c.Hq + kvh * g) * c.slots;

  for (int tile = t0 + warp; tile < t1; tile += kWarps) {
    const int u = tile * kTile + lane;
    const bool valid = u < n;
    const bool is8 = u < n8;
    const int j = is8 ? u : u - n8;
    const int sid = is8 ? j : c.cap8 + j;
    float s[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) s[h] = 0.0f;
    if (valid) {
      if (is8) {
        const int4* row = reinterpret_cast<const int4*>(K8 + static_cast<size_t>(j) * D);
        for (int ch = 0; ch < D / 16; ++ch) {
          const int4 w = row[ch];
          const int ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float x = static_cast<float>(static_cast<int>((ws[e >> 2] >> (8 * (e & 3))) & 0xff) - 128);
#pragma unroll
            for (int h = 0; h < kMaxGroup; ++h)
              if (h < g) s[h] = fmaf(x, qk8[h * D + ch * 16 + e], s[h]);
          }
        }
        const float sc = KS[j] * ap.scale;
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) s[h] *= sc;
      } else {
        const int4* row = reinterpret_cast<const int4*>(K16 + static_cast<size_t>(j) * D);
        for (int ch = 0; ch < D / 8; ++ch) {
          const int4 w = row[ch];
          const __half2* hp = reinterpret_cast<const __half2*>(&w);
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const float2 f = __half22float2(hp[e2]);
#pragma unroll
            for (int h = 0; h < kMaxGroup; ++h)
              if (h < g) {
                s[h] = fmaf(f.x, qs[h * D + ch * 8 + 2 * e2], s[h]);
                s[h] = fmaf(f.y, qs[h * D + ch * 8 + 2 * e2 + 1], s[h]);
              }
          }
        }
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) s[h] *= ap.scale;
      }
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h)
        if (h < g && ap.mass) SC[static_cast<size_t>(h) * c.slots + sid] = s[h];
    }
    // online softmax update of the tile, per head
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h < g) {
        const float tmax = warp_max(valid ? s[h] : -INFINITY);
        const float mnew = fmaxf(m[h], tmax);
        const float corr = rescale(m[h], mnew);
        const float p = valid ? expf(s[h] - mnew) : 0.0f;
        lsum[h] = lsum[h] * corr + warp_sum(p);
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[h][k] *= corr;
        m[h] = mnew;
        s[h] = p;
      }
    }
    // P . V over the tile: lane owns channels lane + 32k
    const int nvalid = min(kTile, n - tile * kTile);
    for (int jj = 0; jj < nvalid; ++jj) {
      const int uu = tile * kTile + jj;
      float v[DPL];
      if (uu < n8) {
        const float vsc = VS[uu];
        const int8_t* vr = V8 + static_cast<size_t>(uu) * D;
#pragma unroll
        for (int k = 0; k < DPL; ++k)
          v[k] = static_cast<float>(static_cast<int>(static_cast<uint8_t>(vr[lane + 32 * k])) - 128) * vsc *
                 vfac[k];
      } else {
        const __half* vr = V16 + static_cast<size_t>(uu - n8) * D;
#pragma unroll
        for (int k = 0; k < DPL; ++k) v[k] = __half2float(vr[lane + 32 * k]);
      }
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) {
        if (h < g) {
          const float ph = __shfl_sync(0xffffffffu, s[h], jj);
#pragma unroll
          for (int k = 0; k < DPL; ++k) acc[h][k] = fmaf(ph, v[k], acc[h][k]);
        }
      }
    }
  }

  // ---- merge the warps of this CTA ----
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    if (h < g) {
      if (lane == 0) {
        wm[warp * g + h] = m[h];
        wl[warp * g + h] = lsum[h];
      }
#pragma unroll
      for (int k = 0; k < DPL; ++k) wacc[(warp * g + h) * D + lane + 32 * k] = acc[h][k];
    }
  }
  __syncthreads();
  const size_t obase = (static_cast<size_t>(lb) * c.Hq + kvh * g);   // split-K scratch
  float* outp = ap.out + (static_cast<size_t>(lbu) * c.Hq + kvh * g) * D;
  for (int idx = tid; idx < g * D; idx += kThreads) {
    const int h = idx / D, dd = idx - h * D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * g + h]);
    float Ls = 0.0f, A = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      const float f = rescale(wm[w * g + h], M);
      Ls += wl[w * g + h] * f;
      A += wacc[(w * g + h) * D + dd] * f;
    }
    if (ap.splits == 1) {
      outp[h * D + dd] = A / Ls;
      if (dd == 0) { fin[h] = M; fin[g + h] = Ls; }
    } else {
      const size_t pi = (obase + h) * ap.splits + split;
      ap.part_acc[pi * D + dd] = A;
      if (dd == 0) { ap.part_ml[pi * 2] = M; ap.part_ml[pi * 2 + 1] = Ls; }
    }
  }

  int tok_lo = t0 * kTile, tok_hi = min(n, t1 * kTile);
  if (ap.splits > 1) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&ap.ticket[unit], 1u) == static_cast<unsigned>(ap.splits - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int idx = tid; idx < g * D; idx += kThreads) {
      const int h = idx / D, dd = idx - h * D;
      const size_t pb = (obase + h) * ap.splits;
      float M = -INFINITY;
      for (int sp = 0; sp < ap.splits; ++sp) M = fmaxf(M, __ldcg(&ap.part_ml[(pb + sp) * 2]));
      float Ls = 0.0f, A = 0.0f;
      for (int sp = 0; sp < ap.splits; ++sp) {
        const float f = rescale(__ldcg(&ap.part_ml[(pb + sp) * 2]), M);
        Ls += __ldcg(&ap.part_ml[(pb + sp) * 2 + 1]) * f;
        A += __ldcg(&ap.part_acc[(pb + sp) * D + dd]) * f;
      }
      outp[h * D + dd] = A / Ls;
      if (dd == 0) { fin[h] = M; fin[g + h] = Ls; }
    }
    if (tid == 0) ap.ticket[unit] = 0u;
    tok_lo = 0;
    tok_hi = n;
  }
  if (!ap.mass) return;       // the policy ranks without the attention mass
  __syncthreads();
  // ---- attention mass of every token of the finished unit ----
  float* MS = c.mass + (static_cast<size_t>(lb) * c.Hkv + kvh) * c.slots;
  for (int u = tok_lo + tid; u < tok_hi; u += kThreads) {
    const int sid = (u < n8) ? u : c.cap8 + (u - n8);
    float a = 0.0f;
    for (int h = 0; h < g; ++h)
      a += expf(__ldcg(&SC[static_cast<size_t>(h) * c.slots + sid]) - fin[h]) / fin[g + h];
    MS[sid] = a;
  }
}

template <int D>
cudaError_t launch_simple(const Cache& c, const AttnParams& ap, cudaStream_t s) {
  const size_t smem = sizeof(float) * ((c.chexp ? 2 : 1) * c.g * D + 2 * kWarps * c.g + 2 * c.g +
                                       kWarps * c.g * D);
  if (smem > 48 * 1024) {          // above the default dynamic shared-memory limit
    const cudaError_t e = cudaFuncSetAttribute(k_attn_simple<D>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  k_attn_simple<D><<<dim3(ap.nlb * c.Hkv, ap.splits), kThreads, smem, s>>>(c, ap);
  return cudaGetLastError();
}

}  // namespace

bool attention_uses_mma(const Cache& c, int kernel) {
  return kernel != 1 && c.g >= 1 && c.g <= 8;
}

cudaError_t launch_attention(const Cache& c, const AttnParams& ap, cudaStream_t s) {
  const bool mma_ok = c.g >= 1 && c.g <= 8;
  if (ap.kernel == 2 && !mma_ok) return cudaErrorInvalidValue;
  if (attention_uses_mma(c, ap.kernel)) return launch_attention_mma(c, ap, s);
  if (ap.k_new || ap.kept_pos || ap.kept_count) return cudaErrorInvalidValue;
  if (c.d == 64) return launch_simple<64>(c, ap, s);
  if (c.d == 128) return launch_simple<128>(c, ap, s);
  return cudaErrorInvalidValue;
}

}  // namespace confkv
