// CONF-KV decode-step oracle: TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU statement of what one CONF-KV decode
// step computes, used by the tests, by the package's smoke check and by the
// benchmark's CPU-baseline leg.  Nothing in the product path may link or call
// it.  It shares no code with the CUDA library.
//
// Source: "CONF-KV: Confidence-Aware KV Cache Eviction with Mixed-Precision
// Storage for Long-Horizon LLM" as summarised on gist.science (paper
// 2605.24786; Dutch page "Technische Samenvatting", Italian page "Riepilogo
// Tecnico", Korean page "기술 요약" -- the three state the same method).
// Sections cited below by their Dutch names:
//   [Vertrouwensschatting]  confidence estimation and its one equation
//   [Adaptieve Budgetselectie] threshold tau -> N_high / N_low
//   [Tokenrangschikking]    EMA attention mass + recency ranking, window P
//   [Mixed-Precision Opslag] most recent W tokens FP16, older INT8
//   [Pyramidale Budgetten]  optional per-layer budgets (CONF-KV-L)
//   [Implementatie]         contiguous compaction, block-wise attention
//   [Betekenis]             forward-only (no re-admission), short-context no-op
//
// Precision: fp64 everywhere, except the quantities whose rounding decides an
// integer on both sides and that the cache stores in fp32: the INT8 quantiser
// (scale, codes) and the EMA / ranking key.  Those are evaluated here in IEEE
// fp32 with one rounding per operation (build with -ffp-contract=off), so the
// ranking and the codes are decided in the same precision as the kernels'.
//
// Readings of points the pages leave open (the plainest reading each time):
//   * normalised entropy: H / ln V (natural log); V >= 2
//   * margin m = log p(1) - log p(2) = z(1) - z(2) (top two with multiplicity)
//   * sigma = logistic function
//   * NaN / +inf logits, or no finite logit: flagged, c := 0 (-> N_low);
//     -inf logits are masked tokens and contribute nothing
//   * c >= tau selects N_high (the tighter budget)
//   * EMA: ema <- beta*ema + (1-beta)*a, a = mean over all query heads of the
//     previous step's attention probability of the token (0 before any)
//   * ranking key s = ema + 1/(1+age), ties broken by the newer position
//   * protected = age < P (includes the new token); append, then evict
//   * FP16 region = kept tokens with age < W; older kept tokens are INT8 with
//     one absmax scale per (token, KV head, K or V) over the head's d channels,
//     scale = amax/127, code = round-half-even(x/scale) clamped to [-127,127]
//   * optional per-(head, channel) storage mode (int8_channel = 1): each
//     (layer, sequence, KV head, K or V) also has one power-of-two factor
//     2^f_c per channel, fixed at prefill from the prompt's channel maxima:
//     E_c = ceil(log2 max_t |x_tc|), f_c = max(-8, E_c - max_c E_c) (0 for a
//     channel that is zero throughout the prompt, and for every channel when
//     there is no prompt).  A row is quantised as y_c = x_c * 2^-f_c (exact
//     in fp32) with the per-token absmax scale s of y, and read back as
//     code_c * s * 2^f_c; the round trip is within s * 2^f_c / 2 per element.
//     The factors belong to the head, not to a token, so compaction (which
//     moves single tokens) never re-quantises anything.
//   * pyramid: N_l = max(P, floor(N*(1 - (1-pmin)*l/(L-1)) + 0.5))
//   * prefill: no eviction; age >= W quantised; an optional last query seeds
//     the attention mass, the EMA stays 0
//
// Comparison policies the pages name, on the same cache and storage rule
// (the method's own budget, selection and compaction unless noted):
//   * WINDOW: fixed budget N_low (per-layer factor applied), key 0, so the
//     newest tokens are kept: the sliding-window baseline; with N_low and W at
//     least the context length it is the full FP16 cache.  No EMA.
//   * H2O: acc <- acc + a (fp32), key = acc: heavy hitters by accumulated
//     attention mass, plus the protected recent window P.
//   * RANDOM: key = a uniform draw in [0, 1) per (step, sequence, token): the
//     top 24 bits of the SplitMix64 finaliser chained over
//     (seed, t, l*B + b, position); random eviction at CONF-KV's rate.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// IEEE binary16 bit pattern -> double (exact).
double half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int expo = (h >> 10) & 0x1f;
  const int mant = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(mant), -24);           // subnormal / zero
  } else if (expo == 31) {
    v = mant ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(mant | 0x400), expo - 25);
  }
  return sign ? -v : v;
}

// Round half to even of an fp32 value (|y| <= 2^23 here).
float round_half_even(float y) {
  float fl = std::floor(y);
  float fr = y - fl;                     // exact
  if (fr > 0.5f) return fl + 1.0f;
  if (fr < 0.5f) return fl;
  return (std::fmod(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

struct Params {
  int L, B, Hq, Hkv, d, V, N_low, N_high, P, W;
  float tau, beta;
  double pyramid_min;
  int policy;
  int int8_channel;
  uint64_t seed;
};

constexpr int kChannelExpMin = -8;   // smallest channel exponent f_c

enum { kConfKV = 0, kWindow = 1, kH2O = 2, kRandom = 3 };

struct Tok {
  int32_t pos = 0;
  float ema = 0.0f;
  float a_prev = 0.0f;
  bool q8 = false;
  std::vector<uint16_t> k16, v16;  // [Hkv*d] while FP16
  std::vector<int8_t> k8, v8;      // [Hkv*d] once INT8
  std::vector<float> ks, vs;       // [Hkv] INT8 scales
};

struct Lane {
  std::vector<Tok> toks;           // any order: attention is order-free
  std::vector<int8_t> fexp;        // [2][Hkv][d] channel exponents of K, then V
                                   // (all 0 unless int8_channel and a prompt)
  // diagnostics of the last selection
  std::vector<float> key;
  std::vector<int32_t> key_pos;
  std::vector<uint8_t> key_prot;
  int last_budget = 0;
  int last_evicted = 0;
};

}  // namespace

struct orc_ctx {
  Params p;
  std::vector<Lane> lanes;         // [L*B]
  std::vector<uint8_t> active;     // [L*B]
  int64_t t = 0;                   // position of the next token
  bool started = false;
};

extern "C" {

struct orc_params {
  int L, B, Hq, Hkv, d, V, N_low, N_high, P, W;
  float tau, beta;
  double pyramid_min;
  int policy;               // 0 CONF-KV, 1 WINDOW, 2 H2O, 3 RANDOM
  int int8_channel;         // 1: per-(head, channel) power-of-two factors
  uint64_t seed;            // RANDOM draws
};

// ---------------------------------------------------------------------------
// [Vertrouwensschatting] c = 0.4(1 - H^) + 0.3 sigma(m) + 0.3 p(1).
// Plain definition: softmax over the vocabulary, entropy -sum p ln p,
// normalised by ln V; top-two logits from a full sort.
// comps (nullable) receives {H^, m, p(1), nonfinite}.
// ---------------------------------------------------------------------------
double orc_confidence(const float* z, int V, double* comps) {
  bool bad = (V < 2);
  double zmax = -INFINITY;
  for (int i = 0; i < V && !bad; ++i) {
    const double x = z[i];
    if (std::isnan(x) || x == INFINITY) bad = true;
    else if (x > zmax) zmax = x;
  }
  if (!bad && zmax == -INFINITY) bad = true;                 // nothing finite
  if (bad) {
    if (comps) { comps[0] = 1.0; comps[1] = 0.0; comps[2] = 0.0; comps[3] = 1.0; }
    return 0.0;
  }
  std::vector<double> e(V);
  double S = 0.0;
  for (int i = 0; i < V; ++i) {
    e[i] = (z[i] == -INFINITY) ? 0.0 : std::exp(static_cast<double>(z[i]) - zmax);
    S += e[i];
  }
  double H = 0.0;
  for (int i = 0; i < V; ++i) {
    const double pi = e[i] / S;
    if (pi > 0.0) H -= pi * std::log(pi);
  }
  const double Hn = H / std::log(static_cast<double>(V));
  std::vector<double> srt(z, z + V);
  std::sort(srt.begin(), srt.end(), [](double a, double b) { return a > b; });
  const double m = srt[0] - srt[1];                         // log p(1) - log p(2)
  const double p1 = 1.0 / S;                                 // exp(0) / S
  const double sig = 1.0 / (1.0 + std::exp(-m));
  if (comps) { comps[0] = Hn; comps[1] = m; comps[2] = p1; comps[3] = 0.0; }
  return 0.4 * (1.0 - Hn) + 0.3 * sig + 0.3 * p1;
}

// [Adaptieve Budgetselectie] c >= tau -> N_high, else N_low.
int orc_budget(double c, float tau, int N_low, int N_high) {
  return (c >= static_cast<double>(tau)) ? N_high : N_low;
}

// [Pyramidale Budgetten] linear per-layer factor from 1 down to pyramid_min.
int orc_layer_budget(int N, int l, int L, double pyramid_min, int P) {
  const double f = (L > 1)
      ? 1.0 - (1.0 - pyramid_min) * static_cast<double>(l) / static_cast<double>(L - 1)
      : 1.0;
  const int n = static_cast<int>(std::floor(static_cast<double>(N) * f + 0.5));
  return std::max(P, n);
}

// [Mixed-Precision Opslag] one absmax INT8 row (fp32 arithmetic).  f (null:
// all 0) holds the row's channel exponents: channel c is divided by 2^f_c
// before the absmax and the rounding (exact: f_c in [-8, 0]).
void orc_quantize_ch(const uint16_t* x, int d, const int8_t* f, int8_t* codes, float* scale) {
  std::vector<float> y(d);
  float amax = 0.0f;
  for (int c = 0; c < d; ++c) {
    const float v = static_cast<float>(half_to_double(x[c]));
    y[c] = f ? std::ldexp(v, -f[c]) : v;
    amax = std::max(amax, std::fabs(y[c]));
  }
  const float s = amax / 127.0f;
  *scale = s;
  for (int c = 0; c < d; ++c) {
    if (s == 0.0f) { codes[c] = 0; continue; }
    float r = round_half_even(y[c] / s);
    r = std::min(127.0f, std::max(-127.0f, r));
    codes[c] = static_cast<int8_t>(r);
  }
}

void orc_quantize(const uint16_t* x, int d, int8_t* codes, float* scale) {
  orc_quantize_ch(x, d, nullptr, codes, scale);
}

// [Mixed-Precision Opslag], per head and channel: the channel exponents of
// one KV head's K (or V) from the prompt's T rows x[T][d] (fp16 bits).
// cmax_c = max_t |x_tc| (exact); E_c = ceil(log2 cmax_c) from the exact
// binary exponent; f_c = max(-8, E_c - max E) over the channels with
// cmax_c > 0, and f_c = 0 for the others.  T = 0 gives all zeros.
void orc_channel_exponents(const uint16_t* x, int T, int d, int8_t* f) {
  std::vector<double> cmax(d, 0.0);
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < d; ++c)
      cmax[c] = std::max(cmax[c], std::fabs(half_to_double(x[static_cast<size_t>(t) * d + c])));
  std::vector<int> E(d, 0);
  bool any = false;
  int emax = 0;
  for (int c = 0; c < d; ++c) {
    if (cmax[c] == 0.0) continue;
    int ex = 0;
    const double fr = std::frexp(cmax[c], &ex);       // cmax = fr * 2^ex, fr in [0.5, 1)
    E[c] = (fr == 0.5) ? ex - 1 : ex;                 // ceil(log2 cmax)
    emax = any ? std::max(emax, E[c]) : E[c];
    any = true;
  }
  for (int c = 0; c < d; ++c)
    f[c] = static_cast<int8_t>(cmax[c] == 0.0 ? 0 : std::max(kChannelExpMin, E[c] - emax));
}

// [Tokenrangschikking] EMA update and ranking key, fp32 with single roundings.
float orc_ema_update(float ema, float a, float beta) {
  const float omb = 1.0f - beta;
  const float t1 = beta * ema;
  const float t2 = omb * a;
  return t1 + t2;
}

float orc_rank_key(float ema, int64_t age) {
  const float r = 1.0f / static_cast<float>(1 + age);
  return ema + r;
}

// H2O comparison: accumulated attention mass, fp32.
float orc_h2o_update(float acc, float a) { return acc + a; }

// RANDOM comparison: SplitMix64's output function (Steele, Lea and Flood,
// "Fast splittable pseudorandom number generators", 2014), applied to
// (seed, t, lb, pos) one word at a time; the top 24 bits of the result as a
// fraction in [0, 1).
uint64_t orc_splitmix(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

float orc_random_key(uint64_t seed, int64_t t, int64_t lb, int32_t pos) {
  uint64_t h = orc_splitmix(seed);
  h = orc_splitmix(h ^ static_cast<uint64_t>(static_cast<uint32_t>(t)));
  h = orc_splitmix(h ^ static_cast<uint64_t>(static_cast<uint32_t>(lb)));
  h = orc_splitmix(h ^ static_cast<uint64_t>(static_cast<uint32_t>(pos)));
  return static_cast<float>(h >> 40) / 16777216.0f;
}

// [Tokenrangschikking] keep every protected token and the best
// (N - #protected) others by (key desc, pos desc).  keep[i] receives 0/1.
// Returns the number of kept tokens.
int orc_select(int n, const float* key, const int32_t* pos, const uint8_t* prot,
               int N, uint8_t* keep) {
  int nprot = 0;
  for (int i = 0; i < n; ++i) { keep[i] = prot[i] ? 1 : 0; nprot += prot[i] ? 1 : 0; }
  if (n <= N) { for (int i = 0; i < n; ++i) keep[i] = 1; return n; }
  std::vector<int> cand;
  for (int i = 0; i < n; ++i) if (!prot[i]) cand.push_back(i);
  std::sort(cand.begin(), cand.end(), [&](int a, int b) {
    if (key[a] != key[b]) return key[a] > key[b];
    return pos[a] > pos[b];
  });
  const int room = std::max(0, N - nprot);
  for (int j = 0; j < static_cast<int>(cand.size()) && j < room; ++j) keep[cand[j]] = 1;
  return nprot + std::min(room, static_cast<int>(cand.size()));
}

// [Implementatie] textbook softmax attention of one query head over n keys
// (fp64).  k, v: [n][d] dequantised values; out[d]; prob[n] (nullable).
void orc_attention_head(const double* q, const double* k, const double* v, int n, int d,
                        double* out, double* prob) {
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (n == 0) return;
  const double inv = 1.0 / std::sqrt(static_cast<double>(d));
  std::vector<double> s(n);
  double mx = -INFINITY;
  for (int i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += q[c] * k[static_cast<size_t>(i) * d + c];
    s[i] = acc * inv;
    mx = std::max(mx, s[i]);
  }
  double den = 0.0;
  for (int i = 0; i < n; ++i) { s[i] = std::exp(s[i] - mx); den += s[i]; }
  for (int i = 0; i < n; ++i) {
    const double p = s[i] / den;
    if (prob) prob[i] = p;
    for (int c = 0; c < d; ++c) out[c] += p * v[static_cast<size_t>(i) * d + c];
  }
}

// ---------------------------------------------------------------------------
// Whole-cache oracle.
// ---------------------------------------------------------------------------
orc_ctx* orc_create(const orc_params* prm) {
  if (!prm) return nullptr;
  const orc_params& q = *prm;
  if (q.L < 1 || q.B < 1 || q.Hkv < 1 || q.Hq < q.Hkv || q.Hq % q.Hkv || q.d < 1 ||
      q.V < 2 || q.P < 1 || q.W < q.P || q.N_low < q.P || q.N_high < q.P || q.policy < 0 ||
      q.policy > 3 || q.int8_channel < 0 || q.int8_channel > 1)
    return nullptr;
  orc_ctx* c = new orc_ctx();
  c->p = Params{q.L, q.B, q.Hq, q.Hkv, q.d, q.V, q.N_low, q.N_high, q.P, q.W,
                q.tau, q.beta, q.pyramid_min, q.policy, q.int8_channel ? 1 : 0, q.seed};
  c->lanes.resize(static_cast<size_t>(q.L) * q.B);
  for (Lane& ln : c->lanes) ln.fexp.assign(static_cast<size_t>(2) * q.Hkv * q.d, 0);
  c->active.assign(static_cast<size_t>(q.L) * q.B, 1);
  return c;
}

void orc_free(orc_ctx* c) { delete c; }

void orc_set_active(orc_ctx* c, const uint8_t* act) {
  for (size_t i = 0; i < c->active.size(); ++i) c->active[i] = act[i];
}

namespace {

// the channel exponents of KV head h's K (isk) or V in a lane
const int8_t* lane_fexp(const Params& p, const Lane& ln, int h, bool isk) {
  return ln.fexp.data() + (static_cast<size_t>(isk ? 0 : 1) * p.Hkv + h) * p.d;
}

void quantize_tok(const Params& p, const Lane& ln, Tok& tk) {
  const int d = p.d;
  tk.k8.assign(static_cast<size_t>(p.Hkv) * d, 0);
  tk.v8.assign(static_cast<size_t>(p.Hkv) * d, 0);
  tk.ks.assign(p.Hkv, 0.0f);
  tk.vs.assign(p.Hkv, 0.0f);
  for (int h = 0; h < p.Hkv; ++h) {
    orc_quantize_ch(&tk.k16[static_cast<size_t>(h) * d], d, lane_fexp(p, ln, h, true),
                    &tk.k8[static_cast<size_t>(h) * d], &tk.ks[h]);
    orc_quantize_ch(&tk.v16[static_cast<size_t>(h) * d], d, lane_fexp(p, ln, h, false),
                    &tk.v8[static_cast<size_t>(h) * d], &tk.vs[h]);
  }
  tk.q8 = true;
  tk.k16.clear();
  tk.v16.clear();
}

// dequantised value of channel c of KV head h (K if isk): code * scale (the
// fp32 product) times the channel factor 2^f_c (exact)
double deq(const Params& p, const Lane& ln, const Tok& tk, int h, int c, bool isk) {
  const int d = p.d;
  if (!tk.q8) return half_to_double((isk ? tk.k16 : tk.v16)[static_cast<size_t>(h) * d + c]);
  const int8_t code = (isk ? tk.k8 : tk.v8)[static_cast<size_t>(h) * d + c];
  const float s = (isk ? tk.ks : tk.vs)[h];
  return std::ldexp(static_cast<double>(static_cast<float>(code) * s), lane_fexp(p, ln, h, isk)[c]);
}

// attention of all query heads of one lane; sets a_prev; out [Hq][d] (nullable)
void lane_attention(const Params& p, Lane& ln, const uint16_t* qlb, double* out) {
  const int n = static_cast<int>(ln.toks.size());
  const int d = p.d, g = p.Hq / p.Hkv;
  std::vector<double> K(static_cast<size_t>(n) * d), Vv(static_cast<size_t>(n) * d);
  std::vector<double> q(d), o(d), prob(n), mass(n, 0.0);
  for (int h = 0; h < p.Hkv; ++h) {
    for (int i = 0; i < n; ++i)
      for (int c = 0; c < d; ++c) {
        K[static_cast<size_t>(i) * d + c] = deq(p, ln, ln.toks[i], h, c, true);
        Vv[static_cast<size_t>(i) * d + c] = deq(p, ln, ln.toks[i], h, c, false);
      }
    for (int j = 0; j < g; ++j) {
      const int hq = h * g + j;
      for (int c = 0; c < d; ++c) q[c] = half_to_double(qlb[static_cast<size_t>(hq) * d + c]);
      orc_attention_head(q.data(), K.data(), Vv.data(), n, d, o.data(), prob.data());
      if (out) for (int c = 0; c < d; ++c) out[static_cast<size_t>(hq) * d + c] = o[c];
      for (int i = 0; i < n; ++i) mass[i] += prob[i];
    }
  }
  for (int i = 0; i < n; ++i)
    ln.toks[i].a_prev = static_cast<float>(mass[i] / static_cast<double>(p.Hq));
}

}  // namespace

// Prefill of one (layer l, sequence b): T tokens at positions 0..T-1.
// k, v: [Hkv][T][d] fp16 bits; q_last: [Hq][d] or null.  No eviction; tokens
// with age >= W (age measured from T-1) are stored as INT8.
int orc_prefill_lb(orc_ctx* c, int l, int b, const uint16_t* k, const uint16_t* v, int T,
                   const uint16_t* q_last) {
  const Params& p = c->p;
  if (l < 0 || l >= p.L || b < 0 || b >= p.B || T < 0) return -1;
  Lane& ln = c->lanes[static_cast<size_t>(l) * p.B + b];
  ln.toks.clear();
  const int d = p.d;
  std::fill(ln.fexp.begin(), ln.fexp.end(), 0);
  if (p.int8_channel && T > 0)
    for (int h = 0; h < p.Hkv; ++h) {
      orc_channel_exponents(k + static_cast<size_t>(h) * T * d, T, d,
                            ln.fexp.data() + static_cast<size_t>(h) * d);
      orc_channel_exponents(v + static_cast<size_t>(h) * T * d, T, d,
                            ln.fexp.data() + (static_cast<size_t>(p.Hkv) + h) * d);
    }
  for (int i = 0; i < T; ++i) {
    Tok tk;
    tk.pos = i;
    tk.k16.resize(static_cast<size_t>(p.Hkv) * d);
    tk.v16.resize(static_cast<size_t>(p.Hkv) * d);
    for (int h = 0; h < p.Hkv; ++h)
      for (int x = 0; x < d; ++x) {
        const size_t src = (static_cast<size_t>(h) * T + i) * d + x;
        tk.k16[static_cast<size_t>(h) * d + x] = k[src];
        tk.v16[static_cast<size_t>(h) * d + x] = v[src];
      }
    if ((T - 1) - i >= p.W) quantize_tok(p, ln, tk);
    ln.toks.push_back(std::move(tk));
  }
  if (q_last && T > 0) lane_attention(p, ln, q_last, nullptr);
  c->t = T;
  c->started = true;
  return 0;
}

// Sets the position of the next decode token (for a decode-only start).
void orc_set_position(orc_ctx* c, int64_t t) { c->t = t; c->started = true; }

// One decode step for every active (layer, sequence).
//   logits [B][V] fp32; q [L][B][Hq][d], k_new / v_new [L][B][Hkv][d] fp16 bits
//   out [L][B][Hq][d] fp64; kept_pos [L][B][cap] (any order); kept_count [L][B]
//   conf [B], budget [B], flags [B] (1 = non-finite logits)
int orc_step(orc_ctx* c, const float* logits, const uint16_t* q, const uint16_t* k_new,
             const uint16_t* v_new, double* out, int32_t* kept_pos, int32_t* kept_count,
             int cap, double* conf, int32_t* budget, int32_t* flags) {
  const Params& p = c->p;
  const int64_t t = c->t;
  const int d = p.d;
  std::vector<int> Nb(p.B);
  for (int b = 0; b < p.B; ++b) {
    double comps[4];
    const double cb = orc_confidence(logits + static_cast<size_t>(b) * p.V, p.V, comps);
    Nb[b] = (p.policy == kWindow) ? p.N_low : orc_budget(cb, p.tau, p.N_low, p.N_high);
    if (conf) conf[b] = cb;
    if (budget) budget[b] = Nb[b];
    if (flags) flags[b] = comps[3] != 0.0 ? 1 : 0;
  }
  for (int l = 0; l < p.L; ++l) {
    for (int b = 0; b < p.B; ++b) {
      const size_t lb = static_cast<size_t>(l) * p.B + b;
      if (!c->active[lb]) continue;
      Lane& ln = c->lanes[lb];
      // EMA update (H2O: accumulation) from the previous step's attention mass
      for (Tok& tk : ln.toks) {
        if (p.policy == kConfKV) tk.ema = orc_ema_update(tk.ema, tk.a_prev, p.beta);
        if (p.policy == kH2O) tk.ema = orc_h2o_update(tk.ema, tk.a_prev);
        tk.a_prev = 0.0f;
      }
      // append the new token (FP16, ema 0)
      Tok nt;
      nt.pos = static_cast<int32_t>(t);
      nt.k16.assign(k_new + lb * p.Hkv * d, k_new + (lb + 1) * p.Hkv * d);
      nt.v16.assign(v_new + lb * p.Hkv * d, v_new + (lb + 1) * p.Hkv * d);
      ln.toks.push_back(std::move(nt));
      // rank and evict
      const int n = static_cast<int>(ln.toks.size());
      const int N = orc_layer_budget(Nb[b], l, p.L, p.pyramid_min, p.P);
      ln.key.resize(n); ln.key_pos.resize(n); ln.key_prot.resize(n);
      for (int i = 0; i < n; ++i) {
        const int64_t age = t - ln.toks[i].pos;
        switch (p.policy) {
          case kConfKV: ln.key[i] = orc_rank_key(ln.toks[i].ema, age); break;
          case kH2O: ln.key[i] = ln.toks[i].ema; break;
          case kRandom:
            ln.key[i] = orc_random_key(p.seed, t, static_cast<int64_t>(lb), ln.toks[i].pos);
            break;
          default: ln.key[i] = 0.0f; break;     // WINDOW: the newest win the tie
        }
        ln.key_pos[i] = ln.toks[i].pos;
        ln.key_prot[i] = age < p.P ? 1 : 0;
      }
      std::vector<uint8_t> keep(n);
      orc_select(n, ln.key.data(), ln.key_pos.data(), ln.key_prot.data(), N, keep.data());
      ln.last_budget = N;
      std::vector<Tok> kept;
      kept.reserve(n);
      for (int i = 0; i < n; ++i) if (keep[i]) kept.push_back(std::move(ln.toks[i]));
      ln.last_evicted = n - static_cast<int>(kept.size());
      ln.toks.swap(kept);
      // tokens leaving the most recent W are stored as INT8
      for (Tok& tk : ln.toks)
        if (!tk.q8 && t - tk.pos >= p.W) quantize_tok(p, ln, tk);
      // attention over the kept tokens
      lane_attention(p, ln, q + lb * p.Hq * d, out ? out + lb * p.Hq * d : nullptr);
      if (kept_count) kept_count[lb] = static_cast<int32_t>(ln.toks.size());
      if (kept_pos) {
        const int m = std::min(cap, static_cast<int>(ln.toks.size()));
        for (int i = 0; i < m; ++i) kept_pos[lb * cap + i] = ln.toks[i].pos;
      }
    }
  }
  c->t = t + 1;
  return 0;
}

// Number of tokens cached for (l, b).
int orc_count(const orc_ctx* c, int l, int b) {
  return static_cast<int>(c->lanes[static_cast<size_t>(l) * c->p.B + b].toks.size());
}

// Keys of the last selection of (l, b): key[n], pos[n], prot[n]; returns n,
// *budget = N_l used, *evicted = tokens dropped.
int orc_last_keys(const orc_ctx* c, int l, int b, float* key, int32_t* pos, uint8_t* prot,
                  int cap, int* budget, int* evicted) {
  const Lane& ln = c->lanes[static_cast<size_t>(l) * c->p.B + b];
  const int n = static_cast<int>(ln.key.size());
  for (int i = 0; i < n && i < cap; ++i) { key[i] = ln.key[i]; pos[i] = ln.key_pos[i]; prot[i] = ln.key_prot[i]; }
  if (budget) *budget = ln.last_budget;
  if (evicted) *evicted = ln.last_evicted;
  return n;
}

// Cached state of (l, b), one row per token (any order):
//   pos[n], is8[n], ema[n], a_prev[n]; k16/v16 [n][Hkv][d] (fp16 tokens, else 0);
//   k8/v8 [n][Hkv][d] and ks/vs [n][Hkv] (INT8 tokens, else 0).  Returns n.
int orc_get_tokens(const orc_ctx* c, int l, int b, int cap, int32_t* pos, uint8_t* is8,
                   float* ema, float* a_prev, uint16_t* k16, uint16_t* v16, int8_t* k8,
                   int8_t* v8, float* ks, float* vs) {
  const Params& p = c->p;
  const Lane& ln = c->lanes[static_cast<size_t>(l) * p.B + b];
  const int n = std::min(cap, static_cast<int>(ln.toks.size()));
  const size_t row = static_cast<size_t>(p.Hkv) * p.d;
  for (int i = 0; i < n; ++i) {
    const Tok& tk = ln.toks[i];
    if (pos) pos[i] = tk.pos;
    if (is8) is8[i] = tk.q8 ? 1 : 0;
    if (ema) ema[i] = tk.ema;
    if (a_prev) a_prev[i] = tk.a_prev;
    for (size_t x = 0; x < row; ++x) {
      if (k16) k16[i * row + x] = tk.q8 ? 0 : tk.k16[x];
      if (v16) v16[i * row + x] = tk.q8 ? 0 : tk.v16[x];
      if (k8) k8[i * row + x] = tk.q8 ? tk.k8[x] : 0;
      if (v8) v8[i * row + x] = tk.q8 ? tk.v8[x] : 0;
    }
    for (int h = 0; h < p.Hkv; ++h) {
      if (ks) ks[static_cast<size_t>(i) * p.Hkv + h] = tk.q8 ? tk.ks[h] : 0.0f;
      if (vs) vs[static_cast<size_t>(i) * p.Hkv + h] = tk.q8 ? tk.vs[h] : 0.0f;
    }
  }
  return n;
}

// Channel exponents of (l, b): fk, fv [Hkv][d] (K, V).
void orc_get_exponents(const orc_ctx* c, int l, int b, int8_t* fk, int8_t* fv) {
  const Params& p = c->p;
  const Lane& ln = c->lanes[static_cast<size_t>(l) * p.B + b];
  const size_t n = static_cast<size_t>(p.Hkv) * p.d;
  for (size_t i = 0; i < n; ++i) {
    if (fk) fk[i] = ln.fexp[i];
    if (fv) fv[i] = ln.fexp[n + i];
  }
}

double orc_half_to_double(uint16_t h) { return half_to_double(h); }

}  // extern "C"
