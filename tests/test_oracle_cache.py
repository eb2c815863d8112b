"""Whole-step pins of the oracle: special cases with closed forms and invariants.

* short-context no-op (CONF-KV page, Betekenis en Beweringen: no effect when
  the context never exceeds the eviction threshold) -> plain full attention;
* beta = 1 freezes the EMA, so the ranking is pure recency -> the kept set is
  the newest positions (a sliding window), and the output is full attention
  over that window on numpy-quantised INT8 values;
* invariants: |cache| <= N, the newest P always kept, no re-admission
  (forward-only), INT8 exactly for age >= W, attention mass sums to one.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle
from synth import workloads as wl


def small(**kw):
    base = dict(name="tiny", L=2, B=2, Hq=4, Hkv=2, d=16, V=300, prefill=0, steps=60,
                N_high=12, N_low=20, P=4, W=8, beta=0.9)
    base.update(kw)
    return wl.Workload(**base)


def np_quant(x16):
    """numpy fp32 absmax quantiser (independent restatement for the pins)."""
    xf = x16.astype(np.float32)
    amax = np.max(np.abs(xf), axis=-1, keepdims=True)
    s = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.where(s > 0, np.clip(np.rint(xf / s), -127, 127), 0)
    return (c.astype(np.float32) * s).astype(np.float64)


def full_attention(q16, K, V):
    """q16 [Hq, d]; K, V [n, Hkv, d] float64 -> out [Hq, d], mass [n]."""
    Hq, d = q16.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    out = np.zeros((Hq, d))
    mass = np.zeros(K.shape[0])
    for h in range(Hq):
        p = sp_softmax(K[:, h // g, :] @ q16[h].astype(np.float64) / math.sqrt(d))
        out[h] = p @ V[:, h // g, :]
        mass += p
    return out, mass / Hq


def run(w, fn):
    o = oracle.Oracle.for_workload(w)
    o.set_position(0)
    hist = {"k": [], "v": []}
    for s in range(w.steps):
        lg, q, k, v = wl.step_inputs(w, s)
        hist["k"].append(k)
        hist["v"].append(v)
        r = o.step(lg, q, k, v)
        fn(o, s, (lg, q, k, v), r, hist)
    return o


def test_short_context_noop_equals_full_attention():
    w = small(N_high=80, N_low=80, P=4, W=80, steps=40)

    def chk(o, s, inp, r, hist):
        K = np.stack(hist["k"], axis=2).astype(np.float64)    # [L,B,n,Hkv,d]
        V = np.stack(hist["v"], axis=2).astype(np.float64)
        for l in range(w.L):
            for b in range(w.B):
                assert sorted(r["kept_pos"][l, b, :r["kept_count"][l, b]]) == list(range(s + 1))
                out, _ = full_attention(inp[1][l, b], K[l, b], V[l, b])
                assert np.allclose(r["out"][l, b], out, rtol=1e-12, atol=1e-12)
    run(w, chk)


def test_beta_one_is_sliding_window_with_int8():
    w = small(beta=1.0, steps=70, W=6, P=3, N_high=9, N_low=15)
    state = {"n": np.zeros((w.L, w.B), int)}

    def chk(o, s, inp, r, hist):
        K16 = np.stack(hist["k"], axis=2)
        V16 = np.stack(hist["v"], axis=2)
        for l in range(w.L):
            for b in range(w.B):
                N = oracle.layer_budget(r["budget"][b], l, w.L, w.pyramid_min, w.P)
                n = min(N, state["n"][l, b] + 1)
                state["n"][l, b] = n
                kept = list(range(s - n + 1, s + 1))
                got = sorted(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist())
                assert got == kept
                ages = s - np.array(kept)
                Kd = np.where((ages >= w.W)[:, None, None], np_quant(K16[l, b, kept]),
                              K16[l, b, kept].astype(np.float64))
                Vd = np.where((ages >= w.W)[:, None, None], np_quant(V16[l, b, kept]),
                              V16[l, b, kept].astype(np.float64))
                out, _ = full_attention(inp[1][l, b], Kd, Vd)
                assert np.allclose(r["out"][l, b], out, rtol=1e-12, atol=1e-12)
    run(w, chk)


@pytest.mark.parametrize("pyr", [1.0, 0.5])
def test_free_run_invariants(pyr):
    w = small(steps=90, pyramid_min=pyr, L=3)
    prev = {}

    def chk(o, s, inp, r, hist):
        for l in range(w.L):
            for b in range(w.B):
                N = oracle.layer_budget(r["budget"][b], l, w.L, w.pyramid_min, w.P)
                kept = set(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist())
                assert len(kept) <= N
                assert set(range(max(0, s - w.P + 1), s + 1)) <= kept      # protected
                assert kept <= prev.get((l, b), set()) | {s}              # no re-admission
                prev[(l, b)] = kept
                tk = o.tokens(l, b)
                ages = s - tk["pos"]
                assert np.array_equal(tk["is8"], ages >= w.W)
                assert abs(tk["a_prev"].astype(np.float64).sum() - 1.0) < 1e-6
                # INT8 round trip against the generated fp16 values
                for i in np.nonzero(tk["is8"])[0]:
                    p = tk["pos"][i]
                    x = hist["k"][p][l, b].astype(np.float32)           # [Hkv, d]
                    err = np.abs(x - tk["k8"][i].astype(np.float32) * tk["ks"][i][:, None])
                    assert np.all(err <= tk["ks"][i][:, None] * (0.5 + 2.0 ** -16))
    run(w, chk)


def test_budgets_follow_confidence_and_sawtooth():
    w = small(steps=200, V=64)
    seen = set()

    def chk(o, s, inp, r, hist):
        for b in range(w.B):
            c = oracle.confidence(inp[0][b])[0]
            assert r["conf"][b] == c
            assert r["budget"][b] == (w.N_high if c >= w.tau else w.N_low)
            seen.add(int(r["budget"][b]))
    run(w, chk)
    assert seen == {w.N_high, w.N_low}


def test_prefill_int8_split_and_q_last_seed():
    w = small(prefill=50, W=8, P=4, steps=0)
    o = oracle.Oracle.for_workload(w)
    rng = np.random.default_rng(0)
    for l in range(w.L):
        for b in range(w.B):
            k = rng.standard_normal((w.Hkv, 50, w.d)).astype(np.float16)
            v = rng.standard_normal((w.Hkv, 50, w.d)).astype(np.float16)
            q = rng.standard_normal((w.Hq, w.d)).astype(np.float16)
            o.prefill_lb(l, b, k, v, q if b == 0 else None)
            tk = o.tokens(l, b)
            assert np.array_equal(tk["pos"], np.arange(50))
            assert np.array_equal(tk["is8"], (49 - tk["pos"]) >= w.W)
            assert not tk["ema"].any()
            if b == 0:
                Kd = np.where(tk["is8"][:, None, None],
                              tk["k8"].astype(np.float32) * tk["ks"][:, :, None],
                              tk["k16"].view(np.float16).astype(np.float32)).astype(np.float64)
                Vd = np.zeros_like(Kd)
                _, mass = full_attention(q, Kd, Vd)
                assert np.allclose(tk["a_prev"], mass, rtol=1e-6, atol=1e-9)
            else:
                assert not tk["a_prev"].any()


def test_heavy_hitter_survives_by_ema_mass():
    # One old key takes nearly all attention (q aligned with it): its EMA mass
    # keeps it cached far beyond the window; recency alone would drop it.
    d, steps = 16, 60
    o = oracle.Oracle(L=1, B=1, Hq=2, Hkv=1, d=d, V=16, N_low=10, N_high=10, tau=0.5,
                      P=2, W=4, beta=0.9)
    o.set_position(0)
    rng = np.random.default_rng(2)
    e0 = np.zeros(d)
    e0[0] = 1.0
    lg = np.zeros((1, 16), dtype=np.float32)
    for s in range(steps):
        k = (8 * e0 if s == 0 else 0.1 * rng.standard_normal(d)).astype(np.float16)
        v = rng.standard_normal(d).astype(np.float16)
        q = np.tile(4 * e0, (2, 1)).astype(np.float16)
        r = o.step(lg, q.reshape(1, 1, 2, d), k.reshape(1, 1, 1, d), v.reshape(1, 1, 1, d))
        kept = set(r["kept_pos"][0, 0, :r["kept_count"][0, 0]].tolist())
        assert 0 in kept
        assert len(kept) == min(s + 1, 10)
    tk = o.tokens(0, 0)
    i0 = int(np.nonzero(tk["pos"] == 0)[0][0])
    assert tk["ema"][i0] > 0.9 and tk["a_prev"][i0] > 0.9
