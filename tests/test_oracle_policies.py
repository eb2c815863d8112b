"""Pins of the oracle's comparison policies (WINDOW, H2O, RANDOM).

The CONF-KV pages compare the method with a fixed sliding window, full KV,
H2O-style heavy hitters and random eviction at the same rate (CONF-KV page,
Technische Samenvatting: Resultaten and Ablatie).  Each policy is pinned to
something other than the oracle itself:
* WINDOW: the kept set is the newest N_low positions whatever the confidence
  (closed form); its output is full attention over that window on
  numpy-quantised INT8 values; with N_low, W >= context it is plain full
  attention over FP16 (the full-KV baseline);
* RANDOM: the draw is SplitMix64, pinned to the published output sequence of
  the generator seeded with 0; the kept set equals a brute-force top-N over
  an independent Python restatement of the draws;
* H2O: the kept set equals a brute-force numpy simulation (scipy softmax for
  the attention mass, fp32 accumulation, top-N by accumulated mass).
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle
from synth import workloads as wl

M64 = (1 << 64) - 1


def small(**kw):
    base = dict(name="tiny", L=2, B=2, Hq=4, Hkv=2, d=16, V=300, prefill=0, steps=50,
                N_high=10, N_low=16, P=3, W=6, beta=0.9)
    base.update(kw)
    return wl.Workload(**base)


def np_quant(x16):
    xf = x16.astype(np.float32)
    amax = np.max(np.abs(xf), axis=-1, keepdims=True)
    s = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.where(s > 0, np.clip(np.rint(xf / s), -127, 127), 0)
    return (c.astype(np.float32) * s).astype(np.float64)


def attn(q16, K, V):
    """q16 [Hq, d]; K, V [n, Hkv, d] float64 -> out [Hq, d], mass [n]."""
    Hq, d = q16.shape
    g = Hq // K.shape[1]
    out = np.zeros((Hq, d))
    mass = np.zeros(K.shape[0])
    for h in range(Hq):
        p = sp_softmax(K[:, h // g, :] @ q16[h].astype(np.float64) / math.sqrt(d))
        out[h] = p @ V[:, h // g, :]
        mass += p
    return out, mass / Hq


def py_splitmix(x):
    z = (x + 0x9E3779B97F4A7C15) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def py_random_key(seed, t, lb, pos):
    h = py_splitmix(seed & M64)
    for w in (t, lb, pos):
        h = py_splitmix(h ^ (w & 0xFFFFFFFF))
    return np.float32((h >> 40) / 16777216.0)


def test_splitmix_published_sequence():
    # SplitMix64 seeded with 0: the first three outputs
    gamma = 0x9E3779B97F4A7C15
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [oracle.splitmix(k * gamma & M64) for k in range(3)] == want
    assert [py_splitmix(k * gamma & M64) for k in range(3)] == want


def test_random_key_is_the_24_bit_draw():
    rng = np.random.default_rng(0)
    for _ in range(200):
        seed, t, lb, pos = (int(rng.integers(0, 2**63)), int(rng.integers(0, 10**6)),
                            int(rng.integers(0, 4096)), int(rng.integers(0, 10**6)))
        k = oracle.random_key(seed, t, lb, pos)
        assert k == py_random_key(seed, t, lb, pos)
        assert 0.0 <= k < 1.0


def run(w, policy, seed=0, fn=None):
    o = oracle.Oracle.for_workload(w, policy, seed)
    o.set_position(0)
    hist = {"k": [], "v": []}
    for s in range(w.steps):
        lg, q, k, v = wl.step_inputs(w, s)
        hist["k"].append(k)
        hist["v"].append(v)
        r = o.step(lg, q, k, v)
        if fn:
            fn(o, s, (lg, q, k, v), r, hist)
    return o


def test_window_keeps_the_newest_n_low_whatever_the_confidence():
    w = small(steps=60, W=5, P=3, N_high=8, N_low=13, tau=0.3)
    budgets = set()

    def chk(o, s, inp, r, hist):
        K16 = np.stack(hist["k"], axis=2)
        V16 = np.stack(hist["v"], axis=2)
        budgets.update(r["budget"].tolist())
        for l in range(w.L):
            for b in range(w.B):
                n = min(w.N_low, s + 1)
                kept = list(range(s - n + 1, s + 1))
                assert sorted(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist()) == kept
                ages = s - np.array(kept)
                Kd = np.where((ages >= w.W)[:, None, None], np_quant(K16[l, b, kept]),
                              K16[l, b, kept].astype(np.float64))
                Vd = np.where((ages >= w.W)[:, None, None], np_quant(V16[l, b, kept]),
                              V16[l, b, kept].astype(np.float64))
                out, _ = attn(inp[1][l, b], Kd, Vd)
                assert np.allclose(r["out"][l, b], out, rtol=1e-12, atol=1e-12)
    run(w, oracle.POLICY_WINDOW, fn=chk)
    assert budgets == {w.N_low}


def test_window_wide_enough_is_full_fp16_attention():
    w = small(steps=40, W=64, P=3, N_high=64, N_low=64)

    def chk(o, s, inp, r, hist):
        K = np.stack(hist["k"], axis=2).astype(np.float64)
        V = np.stack(hist["v"], axis=2).astype(np.float64)
        for l in range(w.L):
            for b in range(w.B):
                assert r["kept_count"][l, b] == s + 1
                out, _ = attn(inp[1][l, b], K[l, b], V[l, b])
                assert np.allclose(r["out"][l, b], out, rtol=1e-12, atol=1e-12)
    run(w, oracle.POLICY_WINDOW, fn=chk)


def brute_kept(keys, pos, prot, N):
    """top-N by (key desc, pos desc) among unprotected, plus the protected"""
    n = len(pos)
    if n <= N:
        return set(pos)
    kept = {p for p, pr in zip(pos, prot) if pr}
    cand = sorted([(k, p) for k, p, pr in zip(keys, pos, prot) if not pr], reverse=True)
    kept |= {p for _, p in cand[:max(0, N - len(kept))]}
    return kept


def test_random_policy_is_top_n_of_the_draws():
    w = small(steps=50, W=5, P=3, N_high=7, N_low=11, tau=0.3)
    seed = 0x1234_5678_9ABC
    cache = {(l, b): [] for l in range(w.L) for b in range(w.B)}
    evicted = [0]

    def chk(o, s, inp, r, hist):
        for l in range(w.L):
            for b in range(w.B):
                N = oracle.layer_budget(int(r["budget"][b]), l, w.L, w.pyramid_min, w.P)
                toks = cache[(l, b)] + [s]
                keys = [py_random_key(seed, s, l * w.B + b, p) for p in toks]
                prot = [s - p < w.P for p in toks]
                kept = brute_kept(keys, toks, prot, N)
                got = set(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist())
                assert got == kept, (s, l, b)
                evicted[0] += len(toks) - len(kept)
                cache[(l, b)] = sorted(kept)
    run(w, oracle.POLICY_RANDOM, seed, fn=chk)
    assert evicted[0] > 100


def test_h2o_is_top_n_by_accumulated_mass():
    w = small(steps=45, W=5, P=3, N_high=7, N_low=11, tau=0.3)
    st = {(l, b): {"pos": [], "acc": {}, "a": {}} for l in range(w.L) for b in range(w.B)}
    div = [0]

    def chk(o, s, inp, r, hist):
        K16 = np.stack(hist["k"], axis=2)
        V16 = np.stack(hist["v"], axis=2)
        for l in range(w.L):
            for b in range(w.B):
                S = st[(l, b)]
                for p in S["pos"]:                       # acc <- acc + a (fp32)
                    S["acc"][p] = np.float32(S["acc"][p] + S["a"][p])
                toks = S["pos"] + [s]
                S["acc"][s] = np.float32(0.0)
                N = oracle.layer_budget(int(r["budget"][b]), l, w.L, w.pyramid_min, w.P)
                keys = [S["acc"][p] for p in toks]
                prot = [s - p < w.P for p in toks]
                kept = brute_kept(keys, toks, prot, N)
                got = set(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist())
                if got != kept:
                    # only a near tie at the cut may differ (fp64 mass sums)
                    cut = min(S["acc"][p] for p in kept if s - p >= w.P)
                    for p in got ^ kept:
                        assert abs(S["acc"][p] - cut) <= 1e-6 * abs(cut), (s, l, b, p)
                    div[0] += 1
                    kept = got
                S["pos"] = sorted(kept)
                ages = s - np.array(S["pos"])
                Kd = np.where((ages >= w.W)[:, None, None], np_quant(K16[l, b, S["pos"]]),
                              K16[l, b, S["pos"]].astype(np.float64))
                Vd = np.where((ages >= w.W)[:, None, None], np_quant(V16[l, b, S["pos"]]),
                              V16[l, b, S["pos"]].astype(np.float64))
                out, mass = attn(inp[1][l, b], Kd, Vd)
                assert np.allclose(r["out"][l, b], out, rtol=1e-12, atol=1e-12)
                S["a"] = {p: np.float32(m) for p, m in zip(S["pos"], mass)}
    run(w, oracle.POLICY_H2O, fn=chk)
    assert div[0] <= 2


def test_h2o_keeps_a_heavy_hitter_that_recency_would_drop():
    d = 16
    o = oracle.Oracle(L=1, B=1, Hq=2, Hkv=1, d=d, V=16, N_low=8, N_high=8, tau=0.5,
                      P=2, W=4, beta=0.9, policy=oracle.POLICY_H2O)
    o.set_position(0)
    rng = np.random.default_rng(5)
    e0 = np.zeros(d)
    e0[0] = 1.0
    lg = np.zeros((1, 16), dtype=np.float32)
    for s in range(40):
        k = (8 * e0 if s == 0 else 0.1 * rng.standard_normal(d)).astype(np.float16)
        v = rng.standard_normal(d).astype(np.float16)
        q = np.tile(4 * e0, (2, 1)).astype(np.float16)
        r = o.step(lg, q.reshape(1, 1, 2, d), k.reshape(1, 1, 1, d), v.reshape(1, 1, 1, d))
        kept = set(r["kept_pos"][0, 0, :r["kept_count"][0, 0]].tolist())
        assert 0 in kept and len(kept) == min(s + 1, 8)
    tk = o.tokens(0, 0)
    i0 = int(np.nonzero(tk["pos"] == 0)[0][0])
    assert tk["ema"][i0] > 30.0          # accumulated over ~39 steps of mass ~1


def test_policy_out_of_range_is_rejected():
    with pytest.raises(ValueError):
        oracle.Oracle(L=1, B=1, Hq=2, Hkv=1, d=16, V=16, N_low=8, N_high=8, tau=0.5,
                      P=2, W=4, beta=0.9, policy=4)
