"""Pins of the oracle's per-(head, channel) INT8 storage mode.

CONF-KV page, Technische Samenvatting, Systeemintegratie, Mixed-Precision
Opslag: older tokens are stored as INT8 per head and channel.  The mode
gives every (layer, sequence, KV head, K or V) one power-of-two factor 2^f_c
per channel, fixed at prefill from the prompt's channel maxima
(E_c = ceil(log2 max_t |x_tc|), f_c = max(-8, E_c - max_c E_c), 0 for a
channel that is zero in the prompt), on top of the per-token absmax scale s:
code_c = rint(x_c 2^-f_c / s), read back as code_c s 2^f_c.

Pins: hand values of the exponents; an independent numpy restatement of the
exponents and of the quantiser; the round trip within s 2^f_c / 2; the
largest |x_c / 2^f_c| maps to +-127; f = 0 reduces to the per-token
quantiser; a prompt whose channels share one binary exponent gives all-zero
factors and the same step results as the mode off; a beta = 1 run (pure
recency, a sliding window) with the mode on equals full attention over the
numpy-dequantised window; the factors stay fixed while tokens are compacted.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle
from synth import workloads as wl


def np_exponents(x16):
    """numpy restatement: x16 [T, d] fp16 -> int8 [d]."""
    a = np.abs(x16.astype(np.float64))
    cmax = a.max(axis=0) if a.shape[0] else np.zeros(x16.shape[-1])
    f = np.zeros(cmax.size, np.int8)
    nz = cmax > 0
    if nz.any():
        m, e = np.frexp(cmax[nz])
        E = np.where(m == 0.5, e - 1, e)
        f[nz] = np.maximum(-8, E - E.max()).astype(np.int8)
    return f


def np_quant_ch(x16, f):
    """numpy fp32 quantiser with channel exponents: (codes int8, scale f32)."""
    y = np.ldexp(x16.astype(np.float32), -f.astype(np.int32)).astype(np.float32)
    s = np.float32(np.max(np.abs(y)) / np.float32(127.0))
    if s == 0:
        return np.zeros(x16.size, np.int8), s
    return np.clip(np.rint(y / s), -127, 127).astype(np.int8), s


def np_deq_ch(codes, s, f):
    return np.ldexp((codes.astype(np.float32) * np.float32(s)).astype(np.float64),
                    f.astype(np.int32))


def test_exponent_hand_values():
    x = np.array([[1.0, 0.5, 0.3, 4.0, 0.0, 2.0 ** -10, -6.0],
                  [0.5, -0.25, 0.1, -3.0, 0.0, 0.0009, 0.0]], np.float16)
    # cmax = 1, .5, .3, 4, 0, 2^-10, 6 -> E = 0, -1, -1, 2, -, -10, 3; max E = 3
    assert oracle.channel_exponents(x).tolist() == [-3, -4, -4, -1, 0, -8, 0]
    # an exact power of two is its own ceiling; just above it rounds up
    assert oracle.channel_exponents(np.array([[4.0, 4.0039]], np.float16)).tolist() == [-1, 0]
    # fp16 subnormals: 2^-24 (E = -24) and 3 * 2^-24 (E = -22)
    sub = np.array([[2.0 ** -24, 3 * 2.0 ** -24, 2.0 ** -17]], np.float16)
    assert oracle.channel_exponents(sub).tolist() == [-7, -5, 0]
    # no prompt rows, or an all-zero prompt: every factor is 1
    assert not oracle.channel_exponents(np.zeros((0, 5), np.float16)).any()
    assert not oracle.channel_exponents(np.zeros((3, 5), np.float16)).any()


def test_exponents_match_numpy_restatement():
    rng = np.random.default_rng(11)
    for d in (4, 64, 128):
        for T in (1, 7, 300):
            x = rng.standard_normal((T, d)) * np.exp(rng.uniform(-9, 4, size=d))
            x = x.astype(np.float16)
            assert np.array_equal(oracle.channel_exponents(x), np_exponents(x))


def test_channel_quantizer_matches_numpy_and_round_trip():
    rng = np.random.default_rng(5)
    for d in (8, 64, 128):
        for _ in range(150):
            x = (rng.standard_normal(d) * np.exp(rng.uniform(-6, 3, size=d))).astype(np.float16)
            f = rng.integers(-8, 1, size=d).astype(np.int8)
            codes, s = oracle.quantize(x, f)
            rc, rs = np_quant_ch(x, f)
            assert s == rs and np.array_equal(codes, rc)
            if s == 0:
                continue
            # the channel of largest |x_c / 2^f_c| maps to +-127 exactly
            y = np.abs(np.ldexp(x.astype(np.float64), -f.astype(np.int32)))
            assert abs(int(codes[int(np.argmax(y))])) == 127
            # round trip within half of the effective step s * 2^f_c per element
            err = np.abs(x.astype(np.float64) - np_deq_ch(codes, s, f))
            step = np.ldexp(float(s), f.astype(np.int32))
            assert np.all(err <= step * (0.5 + 2.0 ** -16))


def test_zero_exponents_reduce_to_per_token_quantizer():
    rng = np.random.default_rng(6)
    for _ in range(100):
        x = (rng.standard_normal(64) * 3).astype(np.float16)
        c0, s0 = oracle.quantize(x)
        c1, s1 = oracle.quantize(x, np.zeros(64, np.int8))
        assert s0 == s1 and np.array_equal(c0, c1)
    c, s = oracle.quantize(np.zeros(16, np.float16), np.full(16, -3, np.int8))
    assert s == 0 and not c.any()


def test_outlier_channel_error_drops():
    # one channel 64x larger than the rest: the per-token scale is set by it,
    # so the other channels lose ~6 bits; the channel factors give them back
    rng = np.random.default_rng(7)
    prompt = rng.standard_normal((256, 64))
    prompt[:, 5] *= 64
    f = np_exponents(prompt.astype(np.float16))
    assert f[5] == 0 and np.all(f[np.arange(64) != 5] <= -5)
    e_tok = e_ch = 0.0
    for _ in range(200):
        x = rng.standard_normal(64)
        x[5] *= 64
        x = x.astype(np.float16)
        mask = np.arange(64) != 5
        c0, s0 = oracle.quantize(x)
        c1, s1 = oracle.quantize(x, f)
        xf = x.astype(np.float64)
        e_tok += np.abs(xf - c0.astype(np.float32) * np.float32(s0))[mask].mean()
        e_ch += np.abs(xf - np_deq_ch(c1, s1, f))[mask].mean()
    assert e_ch < e_tok / 8


def tiny(**kw):
    base = dict(name="tiny-ch", L=2, B=2, Hq=4, Hkv=2, d=16, V=300, prefill=24, steps=40,
                N_high=12, N_low=20, P=4, W=8, beta=0.9, int8_channel=1)
    base.update(kw)
    return wl.Workload(**base)


def prompt(w, scale):
    """A prompt [L, B, Hkv, T, d] whose channel c is scaled by scale[c]."""
    rng = np.random.default_rng(21)
    K = rng.standard_normal((w.L, w.B, w.Hkv, w.prefill, w.d)) * scale
    V = rng.standard_normal((w.L, w.B, w.Hkv, w.prefill, w.d)) * scale[::-1]
    return K.astype(np.float16), V.astype(np.float16)


def full_attention(q16, K, V):
    Hq, d = q16.shape
    g = Hq // K.shape[1]
    out = np.zeros((Hq, d))
    for h in range(Hq):
        p = sp_softmax(K[:, h // g, :] @ q16[h].astype(np.float64) / math.sqrt(d))
        out[h] = p @ V[:, h // g, :]
    return out


def test_prefill_exponents_per_head_and_fixed_over_steps():
    w = tiny()
    scale = np.exp2(np.arange(w.d) % 7 - 4.0)
    K, V = prompt(w, scale)
    o = oracle.Oracle.for_workload(w)
    for l in range(w.L):
        for b in range(w.B):
            o.prefill_lb(l, b, K[l, b], V[l, b])
    want = {(l, b): (np.stack([np_exponents(K[l, b, h]) for h in range(w.Hkv)]),
                     np.stack([np_exponents(V[l, b, h]) for h in range(w.Hkv)]))
            for l in range(w.L) for b in range(w.B)}
    for s in range(w.steps):
        o.step(*wl.step_inputs(w, s))
        for (l, b), (fk, fv) in want.items():
            gk, gv = o.exponents(l, b)
            assert np.array_equal(gk, fk) and np.array_equal(gv, fv)
            tk = o.tokens(l, b)
            for i in np.nonzero(tk["is8"])[0]:          # stored codes = numpy quantiser
                p = tk["pos"][i]
                for h in range(w.Hkv):
                    xk = K[l, b, h, p] if p < w.prefill else None
                    if xk is None:
                        continue
                    ck, sk = np_quant_ch(xk, fk[h])
                    assert np.array_equal(tk["k8"][i, h], ck) and tk["ks"][i, h] == sk


def test_shared_binary_exponent_gives_the_mode_off_results():
    # every channel's prompt maximum is exactly 1.0: all E_c = 0, all f_c = 0,
    # so the channel mode must reproduce the per-token mode bit for bit
    w = tiny(steps=30)
    K, V = prompt(w, np.full(w.d, 0.2))
    K[..., 0, :] = 1.0
    V[..., 0, :] = -1.0
    K = np.clip(K, -1, 1).astype(np.float16)
    V = np.clip(V, -1, 1).astype(np.float16)
    a = oracle.Oracle.for_workload(w)
    b_ = oracle.Oracle.for_workload(w.with_(int8_channel=0))
    for l in range(w.L):
        for b in range(w.B):
            a.prefill_lb(l, b, K[l, b], V[l, b])
            b_.prefill_lb(l, b, K[l, b], V[l, b])
            assert not any(x.any() for x in a.exponents(l, b))
    for s in range(w.steps):
        inp = wl.step_inputs(w, s)
        ra, rb = a.step(*inp), b_.step(*inp)
        assert np.array_equal(ra["out"], rb["out"])
        assert np.array_equal(ra["kept_pos"], rb["kept_pos"])


def test_beta_one_window_with_channel_factors_is_full_attention():
    # beta = 1: keys are pure recency, so the kept set is the newest n tokens;
    # the output must be full attention over them, INT8 ones dequantised by
    # the numpy restatement with the prompt's channel factors
    w = tiny(beta=1.0, steps=45, W=6, P=3, N_high=9, N_low=15)
    scale = np.exp2((np.arange(w.d) * 5) % 11 - 6.0)
    K, V = prompt(w, scale)
    o = oracle.Oracle.for_workload(w)
    for l in range(w.L):
        for b in range(w.B):
            o.prefill_lb(l, b, K[l, b], V[l, b])
    hk = [K[:, :, :, t] for t in range(w.prefill)]          # [L, B, Hkv, d] per position
    hv = [V[:, :, :, t] for t in range(w.prefill)]
    n = np.full((w.L, w.B), w.prefill)
    for s in range(w.steps):
        lg, q, k, v = wl.step_inputs(w, s)
        hk.append(k)
        hv.append(v)
        t = w.prefill + s
        r = o.step(lg, q, k, v)
        for l in range(w.L):
            for b in range(w.B):
                N = oracle.layer_budget(r["budget"][b], l, w.L, w.pyramid_min, w.P)
                n[l, b] = min(N, n[l, b] + 1)
                kept = list(range(t - n[l, b] + 1, t + 1))
                assert sorted(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist()) == kept
                Kd = np.zeros((len(kept), w.Hkv, w.d))
                Vd = np.zeros_like(Kd)
                for i, p in enumerate(kept):
                    for h in range(w.Hkv):
                        xk, xv = hk[p][l, b, h], hv[p][l, b, h]
                        if t - p >= w.W:
                            fk = np_exponents(K[l, b, h])
                            fv = np_exponents(V[l, b, h])
                            Kd[i, h] = np_deq_ch(*np_quant_ch(xk, fk), fk)
                            Vd[i, h] = np_deq_ch(*np_quant_ch(xv, fv), fv)
                        else:
                            Kd[i, h], Vd[i, h] = xk, xv
                out = full_attention(q[l, b], Kd, Vd)
                assert np.allclose(r["out"][l, b], out, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("prefill", [0, 30])
def test_free_run_invariants_with_channel_factors(prefill):
    w = tiny(prefill=prefill, steps=60, L=3)
    scale = np.exp2(np.arange(w.d) % 5 - 2.0)
    o = oracle.Oracle.for_workload(w)
    hk = {}
    if prefill:
        K, V = prompt(w, scale)
        for l in range(w.L):
            for b in range(w.B):
                o.prefill_lb(l, b, K[l, b], V[l, b])
        for t in range(prefill):
            hk[t] = K[:, :, :, t]
    else:
        o.set_position(0)
    prev = {}
    for s in range(w.steps):
        lg, q, k, v = wl.step_inputs(w, s)
        t = prefill + s
        hk[t] = k
        r = o.step(lg, q, k, v)
        for l in range(w.L):
            for b in range(w.B):
                N = oracle.layer_budget(r["budget"][b], l, w.L, w.pyramid_min, w.P)
                kept = set(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist())
                assert len(kept) <= N
                assert set(range(max(0, t - w.P + 1), t + 1)) <= kept
                if (l, b) in prev:
                    assert kept <= prev[(l, b)] | {t}
                prev[(l, b)] = kept
                tk = o.tokens(l, b)
                assert np.array_equal(tk["is8"], t - tk["pos"] >= w.W)
                fk, _ = o.exponents(l, b)
                if not prefill:
                    assert not fk.any()
                for i in np.nonzero(tk["is8"])[0]:
                    x = hk[tk["pos"][i]][l, b].astype(np.float64)     # [Hkv, d]
                    deq = np.ldexp((tk["k8"][i].astype(np.float32) *
                                    tk["ks"][i][:, None]).astype(np.float64), fk.astype(np.int32))
                    step = np.ldexp(tk["ks"][i][:, None].astype(np.float64), fk.astype(np.int32))
                    assert np.all(np.abs(x - deq) <= step * (0.5 + 2.0 ** -16))
