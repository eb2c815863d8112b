"""Counter-based seeded input generator (host side, numpy).

This module produces the synthetic inputs of the decode workloads: fp16
queries / keys / values drawn from N(0, 1), fp32 logits drawn from N(0, 1)
and divided by a temperature, the heavy-hitter keys (every 97th position
scaled by 4), and the needle keys of the long-context workload.  It holds
none of the cache manager's arithmetic.  The same generator is implemented
for the GPU in ``synth/csrc/synth.cu``; every operation below is an IEEE
operation with a single rounding (integer mixing, +, -, *, /, sqrt, frexp),
so both implementations produce bit-identical values.

Definition
----------
* ``fmix(z)`` is the output function of SplitMix64 (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* A stream is addressed by ``(seed, kind, step)``:
  ``key = fmix(fmix(fmix(seed) + kind*G) + step*G)``, G = 0x9E3779B97F4A7C15.
* Element ``i`` of a stream is ``r = fmix(key + (i + 1)*G)`` (the i-th
  SplitMix64 output from state ``key``).
* A normal deviate uses Box-Muller on the two 32-bit halves of ``r``:
  ``u1 = (hi + 1) / 2^32`` in (0, 1], ``u2 = lo / 2^32`` in [0, 1),
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``.  ``ln`` and ``cos`` are evaluated
  by the fixed series below (atanh series after frexp range reduction;
  Taylor series after quadrant reduction), accurate to ~1e-16, so the
  deviate is a proper normal and is reproducible bit for bit.
* fp16 values are ``float16(float32(z * mult))``; fp32 logits are
  ``float32(z / temperature)``.
"""
import math

import numpy as np

G = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1
MUL1 = 0xBF58476D1CE4E5B9
MUL2 = 0x94D049BB133111EB

# stream kinds
KIND_Q = 1
KIND_KNEW = 2
KIND_VNEW = 3
KIND_LOGITS = 4
KIND_KPRE = 5
KIND_VPRE = 6
KIND_NEEDLE_POS = 8
KIND_NEEDLE_DIR = 9

HEAVY_PERIOD = 97     # every 97th key (1-based: position % 97 == 96) ...
HEAVY_MULT = 4.0      # ... is scaled by 4

LN2 = 0.6931471805599453
SQRT_HALF = 0.7071067811865476
HALF_PI = 1.5707963267948966
_LOG_TERMS = 13       # atanh series terms: s^2 <= 0.0295, 0.0295^13 < 1e-19
_TRIG_TERMS = 13      # Taylor terms on [0, pi/2): (pi/2)^26 / 26! < 1e-21


def _inv_odd():
    return [1.0 / float(2 * j + 1) for j in range(_LOG_TERMS)]


def _cos_coef():
    c = [1.0]
    for k in range(1, _TRIG_TERMS):
        c.append(-c[-1] / float((2 * k - 1) * (2 * k)))
    return c


def _sin_coef():
    c = [1.0]
    for k in range(1, _TRIG_TERMS):
        c.append(-c[-1] / float((2 * k) * (2 * k + 1)))
    return c


INV_ODD = _inv_odd()
COS_C = _cos_coef()
SIN_C = _sin_coef()


def fmix_int(z):
    """SplitMix64 output function on a Python int (mod 2^64)."""
    z &= M64
    z = ((z ^ (z >> 30)) * MUL1) & M64
    z = ((z ^ (z >> 27)) * MUL2) & M64
    return z ^ (z >> 31)


def stream_key(seed, kind, step):
    k = fmix_int(seed)
    k = fmix_int(k + kind * G)
    return fmix_int(k + step * G)


def _fmix_arr(z):
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(MUL1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(MUL2)
    return z ^ (z >> np.uint64(31))


def raw_u64(key, idx):
    """r_i = fmix(key + (i+1)*G) for an array of indices (uint64 wraparound)."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        s = (idx + np.uint64(1)) * np.uint64(G) + np.uint64(key & M64)
        return _fmix_arr(s)


def _ln(x):
    """Natural log on (0, 1] by frexp + atanh series (plain IEEE ops)."""
    m, e = np.frexp(x)
    small = m < SQRT_HALF
    m = np.where(small, m * 2.0, m)
    e = np.where(small, e - 1, e).astype(np.float64)
    s = (m - 1.0) / (m + 1.0)
    s2 = s * s
    acc = np.full_like(s, INV_ODD[_LOG_TERMS - 1])
    for j in range(_LOG_TERMS - 2, -1, -1):
        acc = acc * s2
        acc = acc + INV_ODD[j]
    lnm = (2.0 * s) * acc
    return lnm + e * LN2


def _poly(t, coef):
    acc = np.full_like(t, coef[-1])
    for j in range(len(coef) - 2, -1, -1):
        acc = acc * t
        acc = acc + coef[j]
    return acc


def _cos2pi(u):
    """cos(2*pi*u) for dyadic u in [0, 1): exact quadrant split + Taylor."""
    v = u * 4.0
    q = np.floor(v)
    f = v - q
    th = f * HALF_PI
    t = th * th
    c = _poly(t, COS_C)
    s = th * _poly(t, SIN_C)
    qi = q.astype(np.int64)
    return np.select([qi == 0, qi == 1, qi == 2], [c, -s, -c], s)


def normal_f64(key, idx):
    """Standard-normal deviates (float64) of stream `key` at indices `idx`."""
    r = raw_u64(key, idx)
    hi = (r >> np.uint64(32)).astype(np.float64)
    lo = (r & np.uint64(0xFFFFFFFF)).astype(np.float64)
    u1 = (hi + 1.0) * (2.0 ** -32)
    u2 = lo * (2.0 ** -32)
    rad = np.sqrt(-2.0 * _ln(u1))
    return rad * _cos2pi(u2)


def to_f16(x64):
    """float64 -> float32 (RN) -> float16 (RN)."""
    return np.asarray(x64, dtype=np.float64).astype(np.float32).astype(np.float16)


def heavy_mult(pos):
    pos = np.asarray(pos)
    return np.where(pos % HEAVY_PERIOD == HEAVY_PERIOD - 1, HEAVY_MULT, 1.0)


# ---------------------------------------------------------------------------
# Tensors of the decode workloads (flat index = C-order index of the shape).
# ---------------------------------------------------------------------------

def gen_f16(seed, kind, step, shape, idx_lo=0, idx_hi=None, inner=None,
            tlen=None, pos0=0, heavy=False):
    """fp16 tensor from stream (seed, kind, step).

    The full tensor has C-order `shape`; this returns the flat range
    [idx_lo, idx_hi).  With `heavy`, element i sits at position
    pos0 + (i // inner) % tlen and is scaled by 4 when that position is a
    heavy-hitter position.
    """
    total = int(np.prod(shape))
    if idx_hi is None:
        idx_hi = total
    idx = np.arange(idx_lo, idx_hi, dtype=np.uint64)
    z = normal_f64(stream_key(seed, kind, step), idx)
    if heavy:
        pos = pos0 + (idx.astype(np.int64) // inner) % tlen
        z = z * heavy_mult(pos)
    return to_f16(z)


def gen_logits(seed, step, B, V, temperature):
    key = stream_key(seed, KIND_LOGITS, step)
    z = normal_f64(key, np.arange(B * V, dtype=np.uint64))
    return (z / float(temperature)).astype(np.float32).reshape(B, V)


def gen_u64(seed, kind, step, n):
    return raw_u64(stream_key(seed, kind, step), np.arange(n, dtype=np.uint64))


def needle_positions(seed, b, T, W, count):
    """`count` distinct positions uniform in [0, T-W) for sequence b."""
    span = T - W
    if span <= 0 or count <= 0:
        return np.zeros(0, dtype=np.int64)
    key = stream_key(seed, KIND_NEEDLE_POS, b)
    out, seen, j = [], set(), 0
    while len(out) < min(count, span):
        r = int(raw_u64(key, np.array([j], dtype=np.uint64))[0])
        j += 1
        p = r % span
        if p not in seen:
            seen.add(p)
            out.append(p)
    return np.array(out, dtype=np.int64)


def needle_direction(seed, L, Hkv, d):
    """Unit direction u[l, kvh, :] (float64)."""
    key = stream_key(seed, KIND_NEEDLE_DIR, 0)
    g = normal_f64(key, np.arange(L * Hkv * d, dtype=np.uint64)).reshape(L, Hkv, d)
    nrm = np.sqrt(np.sum(g * g, axis=-1, keepdims=True))
    return g / nrm
