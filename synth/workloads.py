"""Synthetic decode workloads and their seeded inputs (no cache arithmetic).

Shapes follow the model families the CONF-KV pages evaluate (GPT-2,
Qwen-14B/32B, gpt-oss-20b; "Technische Samenvatting", Experimentele
Resultaten).  Model weights, corpora and benchmark items are not used: the
inputs are seeded synthetic tensors of the same shapes:

* q / k / v: fp16 ~ N(0, 1); every key at a position p with p % 97 == 96 is
  scaled by 4 so that it becomes a heavy hitter.
* logits: fp32, N(0, 1) divided by a temperature that alternates in 64-step
  segments between 0.3 (confident) and 3.0 (uncertain), so that the budget
  switches between N_high and N_low.
* long-context workload: 16 needle keys per sequence at seeded positions in
  [0, T - W), each of norm equal to the key it replaces and pointing along a
  seeded unit direction u[l, kv_head]; the prefill's last query is sqrt(d)*u.
"""
from dataclasses import dataclass, field, replace

import numpy as np

from . import gen


@dataclass(frozen=True)
class Workload:
    name: str
    L: int
    B: int
    Hq: int
    Hkv: int
    d: int
    V: int
    prefill: int
    steps: int
    N_high: int
    N_low: int
    P: int
    W: int
    tau: float = 0.5
    beta: float = 0.9
    pyramid_min: float = 1.0
    needles: int = 0
    seed: int = 0
    temps: tuple = (0.3, 3.0)
    segment: int = 64
    int8_channel: int = 0      # storage mode flag passed to the cache (not an input)

    @property
    def g(self):
        return self.Hq // self.Hkv

    def temperature(self, s):
        return self.temps[(s // self.segment) % 2]

    def position(self, s):
        return self.prefill + s

    def capacity(self):
        """Token slots one (layer, sequence) cache must hold."""
        return max(self.prefill, self.N_low, self.N_high) + 1

    def with_(self, **kw):
        return replace(self, **kw)


GPT2_L1 = Workload("gpt2-small-1layer", L=1, B=1, Hq=12, Hkv=12, d=64, V=50257,
                   prefill=0, steps=2048, N_high=384, N_low=768, P=64, W=128)
GPT2_FULL = Workload("gpt2-small-12layer-b8-pyramid", L=12, B=8, Hq=12, Hkv=12, d=64,
                     V=50257, prefill=0, steps=2048, N_high=384, N_low=768, P=64,
                     W=128, pyramid_min=0.5)
QWEN14B = Workload("qwen14b-shaped-b1-p32768", L=48, B=1, Hq=40, Hkv=8, d=128,
                   V=152064, prefill=32768, steps=256, N_high=2048, N_low=4096,
                   P=128, W=512, needles=16)
QWEN32B = Workload("qwen32b-shaped-b8-p8192", L=64, B=8, Hq=40, Hkv=8, d=128,
                   V=152064, prefill=8192, steps=512, N_high=1024, N_low=2048,
                   P=128, W=256)


def gptoss(B, prefill):
    n_low = prefill // 4
    return Workload(f"gptoss20b-shaped-b{B}-p{prefill}", L=24, B=B, Hq=64, Hkv=8,
                    d=64, V=201088, prefill=prefill, steps=256, N_high=n_low // 2,
                    N_low=n_low, P=128, W=512)


GPTOSS_SWEEP = [gptoss(B, p) for B in (1, 8, 32) for p in (4096, 16384, 32768)]

ALL = {w.name: w for w in [GPT2_L1, GPT2_FULL, QWEN14B, QWEN32B] + GPTOSS_SWEEP}


# ---------------------------------------------------------------------------
# per-step inputs (host, numpy)
# ---------------------------------------------------------------------------

def step_logits(w, s):
    return gen.gen_logits(w.seed, s, w.B, w.V, w.temperature(s))


def step_q(w, s):
    return gen.gen_f16(w.seed, gen.KIND_Q, s, (w.L, w.B, w.Hq, w.d)).reshape(
        w.L, w.B, w.Hq, w.d)


def step_k(w, s):
    return gen.gen_f16(w.seed, gen.KIND_KNEW, s, (w.L, w.B, w.Hkv, w.d), heavy=True,
                       inner=w.d, tlen=1, pos0=w.position(s)).reshape(
        w.L, w.B, w.Hkv, w.d)


def step_v(w, s):
    return gen.gen_f16(w.seed, gen.KIND_VNEW, s, (w.L, w.B, w.Hkv, w.d)).reshape(
        w.L, w.B, w.Hkv, w.d)


def step_inputs(w, s):
    return step_logits(w, s), step_q(w, s), step_k(w, s), step_v(w, s)


# ---------------------------------------------------------------------------
# prefill (host, numpy); one (layer, sequence) slice at a time
# ---------------------------------------------------------------------------

def prefill_kv_lb(w, l, b):
    """k, v of shape [Hkv, T, d] for layer l, sequence b (needles applied)."""
    T = w.prefill
    n = w.Hkv * T * w.d
    lo = (l * w.B + b) * n
    shape = (w.L, w.B, w.Hkv, T, w.d)
    k = gen.gen_f16(w.seed, gen.KIND_KPRE, 0, shape, lo, lo + n, inner=w.d, tlen=T,
                    pos0=0, heavy=True).reshape(w.Hkv, T, w.d)
    v = gen.gen_f16(w.seed, gen.KIND_VPRE, 0, shape, lo, lo + n).reshape(w.Hkv, T, w.d)
    if w.needles:
        k = k.copy()
        pos, vals = needle_keys_lb(w, l, b, k)
        for j, p in enumerate(pos):
            k[:, p, :] = vals[j]
    return k, v


def needle_keys_lb(w, l, b, k_lb):
    """Needle positions of sequence b and their fp16 keys [n, Hkv, d] in layer l.

    k_lb: the generated (pre-needle) keys [Hkv, T, d] of that (layer, sequence).
    """
    pos = gen.needle_positions(w.seed, b, w.prefill, w.W, w.needles)
    u = gen.needle_direction(w.seed, w.L, w.Hkv, w.d)[l]          # [Hkv, d]
    vals = np.zeros((len(pos), w.Hkv, w.d), dtype=np.float16)
    for j, p in enumerate(pos):
        orig = k_lb[:, p, :].astype(np.float64)                  # [Hkv, d]
        nrm = np.sqrt(np.sum(orig * orig, axis=-1, keepdims=True))
        vals[j] = gen.to_f16(nrm * u)
    return pos, vals


def q_last(w):
    """Last prefill query [L, B, Hq, d] (long-context workload) or None."""
    if not w.needles:
        return None
    u = gen.needle_direction(w.seed, w.L, w.Hkv, w.d)            # [L, Hkv, d]
    qh = np.repeat(u, w.g, axis=1) * np.sqrt(float(w.d))          # [L, Hq, d]
    q = gen.to_f16(qh)
    return np.ascontiguousarray(np.broadcast_to(q[:, None], (w.L, w.B, w.Hq, w.d)))


def q_last_lb(w, l, b):
    q = q_last(w)
    return None if q is None else q[l, b]


def step_inputs_lanes(w, s, lbs):
    """Inputs of decode step s with q / k_new / v_new filled for the (l, b)
    lanes in `lbs` only (other lanes zero) and the full logits."""
    lg = step_logits(w, s)
    q = np.zeros((w.L, w.B, w.Hq, w.d), np.float16)
    k = np.zeros((w.L, w.B, w.Hkv, w.d), np.float16)
    v = np.zeros((w.L, w.B, w.Hkv, w.d), np.float16)
    nq, nk = w.Hq * w.d, w.Hkv * w.d
    for l, b in lbs:
        lb = l * w.B + b
        q[l, b] = gen.gen_f16(w.seed, gen.KIND_Q, s, q.shape, lb * nq, (lb + 1) * nq).reshape(
            w.Hq, w.d)
        k[l, b] = gen.gen_f16(w.seed, gen.KIND_KNEW, s, k.shape, lb * nk, (lb + 1) * nk,
                              heavy=True, inner=w.d, tlen=1, pos0=w.position(s)).reshape(w.Hkv, w.d)
        v[l, b] = gen.gen_f16(w.seed, gen.KIND_VNEW, s, v.shape, lb * nk, (lb + 1) * nk).reshape(
            w.Hkv, w.d)
    return lg, q, k, v


def step_inputs_lane(w, s, l, b):
    """Inputs of decode step s with q / k_new / v_new filled for (l, b) only
    (other lanes zero) and the full logits: enough for an oracle that
    simulates just that lane."""
    lg = step_logits(w, s)
    q = np.zeros((w.L, w.B, w.Hq, w.d), np.float16)
    k = np.zeros((w.L, w.B, w.Hkv, w.d), np.float16)
    v = np.zeros((w.L, w.B, w.Hkv, w.d), np.float16)
    lb = l * w.B + b
    nq, nk = w.Hq * w.d, w.Hkv * w.d
    q[l, b] = gen.gen_f16(w.seed, gen.KIND_Q, s, q.shape, lb * nq, (lb + 1) * nq).reshape(w.Hq, w.d)
    k[l, b] = gen.gen_f16(w.seed, gen.KIND_KNEW, s, k.shape, lb * nk, (lb + 1) * nk, heavy=True,
                          inner=w.d, tlen=1, pos0=w.position(s)).reshape(w.Hkv, w.d)
    v[l, b] = gen.gen_f16(w.seed, gen.KIND_VNEW, s, v.shape, lb * nk, (lb + 1) * nk).reshape(
        w.Hkv, w.d)
    return lg, q, k, v
