"""Pins of the CPU oracle against what the CONF-KV pages and mathematics fix.

None of these re-types the oracle's own formulas: each value comes from a
closed form, an invariant, a special case that reduces to a library routine
(numpy / scipy), or brute force on tiny inputs.  The pages print no worked
example, so there is no printed vector to compare against.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax
from scipy.stats import entropy as sp_entropy

import oracle


# ---------------------------------------------------------------------------
# fp16 decoding
# ---------------------------------------------------------------------------

def test_half_decode_matches_numpy_all_patterns():
    lib = oracle.lib()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.orc_half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------------------
# confidence  c = 0.4(1 - H^) + 0.3 sigma(m) + 0.3 p(1)
# (CONF-KV page, Technische Samenvatting, Vertrouwensschatting)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("V", [2, 7, 50257, 152064])
def test_confidence_uniform_closed_form(V):
    # uniform: H^ = 1, m = 0, p(1) = 1/V  ->  c = 0.15 + 0.3/V
    c, Hn, m, p1, bad = oracle.confidence(np.full(V, 1.25, dtype=np.float32))
    assert not bad
    assert abs(Hn - 1.0) < 1e-10 and m == 0.0 and abs(p1 - 1.0 / V) < 1e-15
    assert abs(c - (0.15 + 0.3 / V)) < 1e-10


def test_confidence_uniform_gpt2_vocab_value():
    # 0.15 + 0.3/50257 = 0.15000596931... (hand value)
    c = oracle.confidence(np.zeros(50257, dtype=np.float32))[0]
    assert abs(c - 0.1500059693177) < 1e-11


def test_confidence_near_one_hot_is_one():
    z = np.zeros(50257, dtype=np.float32)
    z[123] = 60.0
    c, Hn, m, p1, _ = oracle.confidence(z)
    assert abs(c - 1.0) < 1e-12 and m == 60.0


@pytest.mark.parametrize("a", [0.0, 0.25, 1.0, math.log(3.0), 2.5, 7.0, -1.5])
def test_confidence_two_token_closed_form(a):
    # V = 2, z = (a, 0): p = sigma(|a|), H = binary entropy, m = |a|.
    # c = 0.4 (1 - h2(p)/ln 2) + 0.3 sigma(|a|) + 0.3 p   (hand derivation)
    af = float(np.float32(a))
    p = 1.0 / (1.0 + math.exp(-abs(af)))
    h2 = -(p * math.log(p) + (1 - p) * math.log(1 - p))
    want = 0.4 * (1 - h2 / math.log(2.0)) + 0.3 * p + 0.3 * p
    c = oracle.confidence(np.array([af, 0.0], dtype=np.float32))[0]
    assert abs(c - want) < 1e-13


def test_confidence_two_token_ln3_hand_value():
    # z = (ln 3, 0) -> p = (3/4, 1/4): H = 0.5623351446, H^ = 0.8112781245,
    # c = 0.4*0.1887218755 + 0.6*0.75 = 0.5254887502 (fp32 ln 3 moves it < 1e-7)
    c = oracle.confidence(np.array([math.log(3.0), 0.0], dtype=np.float32))[0]
    assert abs(c - 0.5254887502) < 1e-7


def test_confidence_uniform_over_finite_subset_with_masking():
    # V' finite equal logits, the rest -inf: H = ln V', normalised by ln V
    V, Vp = 1000, 37
    z = np.full(V, -np.inf, dtype=np.float32)
    z[np.random.default_rng(1).choice(V, Vp, replace=False)] = -3.0
    want = 0.4 * (1 - math.log(Vp) / math.log(V)) + 0.15 + 0.3 / Vp
    assert abs(oracle.confidence(z)[0] - want) < 1e-12


def test_confidence_entropy_matches_scipy_and_invariances():
    rng = np.random.default_rng(7)
    for V in (3, 100, 5000):
        z = (rng.standard_normal(V) / 0.3).astype(np.float32)
        c, Hn, m, p1, _ = oracle.confidence(z)
        p = sp_softmax(z.astype(np.float64))
        assert abs(Hn - sp_entropy(p) / math.log(V)) < 1e-12
        assert abs(p1 - p.max()) < 1e-14
        zs = np.sort(z.astype(np.float64))[::-1]
        assert m == zs[0] - zs[1]
        # shift / permutation invariance; range [0.15, 1]
        c2 = oracle.confidence((z + np.float32(5.0)).astype(np.float32))[0]
        c3 = oracle.confidence(rng.permutation(z))[0]
        assert abs(c - c2) < 1e-6 and abs(c - c3) < 1e-13
        assert 0.15 < c <= 1.0


def test_confidence_tied_top_two_margin_zero():
    z = np.array([1.0, 3.0, 3.0, -2.0], dtype=np.float32)
    assert oracle.confidence(z)[2] == 0.0


@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_confidence_nonfinite_flagged(bad):
    z = np.zeros(10, dtype=np.float32)
    z[4] = bad
    c, *_, flag = oracle.confidence(z)
    assert flag and c == 0.0


def test_confidence_all_masked_flagged():
    assert oracle.confidence(np.full(8, -np.inf, dtype=np.float32))[4]


# ---------------------------------------------------------------------------
# budget (Adaptieve Budgetselectie) and pyramid (Pyramidale Budgetten)
# ---------------------------------------------------------------------------

def test_budget_threshold_semantics():
    tau = np.float32(0.5)
    assert oracle.budget(0.5, tau, 768, 384) == 384          # c == tau -> N_high
    assert oracle.budget(np.nextafter(0.5, 0), tau, 768, 384) == 768
    assert oracle.budget(0.9, tau, 768, 384) == 384
    assert oracle.budget(0.15, tau, 768, 384) == 768


@pytest.mark.parametrize("N,l,L,want", [
    (768, 0, 12, 768), (768, 11, 12, 384),
    (768, 5, 12, 593),     # 768*(1-0.5*5/11) = 593.45
    (384, 3, 12, 332),     # 384*(1-0.5*3/11) = 331.64
    (384, 7, 12, 262),     # 384*(1-0.5*7/11) = 261.82
    (100, 11, 12, 64),     # floor by P = 64
    (500, 0, 1, 500),      # single layer: factor 1
])
def test_layer_budget_hand_values(N, l, L, want):
    assert oracle.layer_budget(N, l, L, 0.5, 64) == want


def test_layer_budget_uniform_when_pyramid_off():
    assert all(oracle.layer_budget(768, l, 12, 1.0, 64) == 768 for l in range(12))


# ---------------------------------------------------------------------------
# INT8 quantiser (Mixed-Precision Opslag)
# ---------------------------------------------------------------------------

def test_quantizer_matches_numpy_fp32_and_round_trip():
    rng = np.random.default_rng(3)
    for d in (1, 8, 64, 128):
        for _ in range(200):
            x = (rng.standard_normal(d) * rng.choice([1e-3, 1.0, 4.0, 300.0])).astype(np.float16)
            codes, s = oracle.quantize(x)
            xf = x.astype(np.float32)
            amax = np.max(np.abs(xf))
            s_ref = np.float32(amax / np.float32(127.0))
            assert s == s_ref
            if s_ref == 0:
                assert not codes.any()
                continue
            ref = np.clip(np.rint(xf / s_ref), -127, 127).astype(np.int8)  # RN-even
            assert np.array_equal(codes, ref)
            # amax element -> +-127 exactly
            i = int(np.argmax(np.abs(xf)))
            assert abs(int(codes[i])) == 127
            # round trip within half a step (plus the fp32 quotient rounding)
            err = np.abs(xf.astype(np.float64) - codes.astype(np.float64) * float(s))
            assert np.all(err <= float(s) * (0.5 + 2.0 ** -16))


def test_quantizer_zero_row_and_half_ties():
    codes, s = oracle.quantize(np.zeros(16, dtype=np.float16))
    assert s == 0 and not codes.any()
    # x = (127, 0.5, 1.5, 2.5): scale 1 -> ties go to even: 0, 2, 2
    codes, s = oracle.quantize(np.array([127, 0.5, 1.5, 2.5, -0.5, -1.5], dtype=np.float16))
    assert s == 1.0 and list(codes) == [127, 0, 2, 2, 0, -2]


# ---------------------------------------------------------------------------
# EMA and ranking key (Tokenrangschikking)
# ---------------------------------------------------------------------------

def test_ema_closed_form_constant_input():
    beta, a = 0.9, 0.0123
    e = np.float32(0.0)
    for k in range(1, 60):
        e = oracle.ema_update(e, a, beta)
        assert abs(float(e) - a * (1 - 0.9 ** k)) < 1e-6 * a * k + 1e-9


def test_ema_beta_one_stays_zero_and_key_is_recency():
    e = np.float32(0.0)
    for _ in range(10):
        e = oracle.ema_update(e, 0.7, 1.0)
    assert e == 0.0
    assert oracle.rank_key(0.0, 0) == 1.0 and oracle.rank_key(0.0, 1) == 0.5
    assert oracle.rank_key(0.0, 3) == 0.25


# ---------------------------------------------------------------------------
# selection: brute force on tiny inputs
# ---------------------------------------------------------------------------

def _brute_select(key, pos, prot, N):
    n = len(key)
    if n <= N:
        return set(range(n))
    must = {i for i in range(n) if prot[i]}
    rest = [i for i in range(n) if not prot[i]]
    room = max(0, N - len(must))
    best, best_sig = None, None
    for comb in itertools.combinations(rest, min(room, len(rest))):
        # lexicographic signature: the kept keys sorted best-first
        sig = sorted(((key[i], pos[i]) for i in comb), reverse=True)
        if best_sig is None or sig > best_sig:
            best, best_sig = set(comb), sig
    return must | best


def test_select_brute_force_tiny():
    rng = np.random.default_rng(11)
    for trial in range(400):
        n = int(rng.integers(1, 11))
        key = rng.choice([0.1, 0.2, 0.25, 0.5, 0.7], size=n).astype(np.float32)  # ties
        pos = rng.permutation(100)[:n].astype(np.int32)
        prot = rng.random(n) < 0.25
        N = int(rng.integers(max(1, prot.sum()), n + 2))
        keep = oracle.select(key, pos, prot, N)
        want = _brute_select(key.tolist(), pos.tolist(), prot.tolist(), N)
        assert set(np.nonzero(keep)[0].tolist()) == want
        assert keep.sum() <= max(N, prot.sum()) and keep[prot].all()


# ---------------------------------------------------------------------------
# attention (block-wise online softmax reaches the plain softmax exactly)
# ---------------------------------------------------------------------------

def test_attention_head_matches_scipy_softmax():
    rng = np.random.default_rng(5)
    for n, d in [(1, 4), (5, 8), (37, 64), (300, 128)]:
        q = rng.standard_normal(d)
        k = rng.standard_normal((n, d)) * 2
        v = rng.standard_normal((n, d))
        out, prob = oracle.attention_head(q, k, v)
        p = sp_softmax(k @ q / math.sqrt(d))
        assert np.allclose(prob, p, rtol=1e-12, atol=1e-15)
        assert abs(prob.sum() - 1.0) < 1e-12
        assert np.allclose(out, p @ v, rtol=1e-11, atol=1e-13)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((6, 16))
    out, prob = oracle.attention_head(rng.standard_normal(16), np.ones((6, 16)), v)
    assert np.allclose(prob, 1 / 6) and np.allclose(out, v.mean(0), atol=1e-14)
    out, prob = oracle.attention_head(rng.standard_normal(16), np.ones((1, 16)), v[:1])
    assert prob[0] == 1.0 and np.array_equal(out, v[0])


def _printed_constants():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "conf_kv_printed_constants.txt")
    out = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, value = line.split()[:2]
        out[key] = value
    return out


@pytest.mark.parametrize("a", [0.0, 0.7, 2.5, -4.0])
def test_confidence_uses_the_printed_weights(a):
    # the weights as the pages print them (golden fixture), applied to the
    # two-token closed form: p = sigma(|a|), H^ = h2(p) / ln 2, m = |a|
    k = _printed_constants()
    w1, w2, w3 = (float(k[x]) for x in ("weight_one_minus_entropy", "weight_sigma_margin",
                                        "weight_top1_probability"))
    assert abs(w1 + w2 + w3 - 1.0) < 1e-15
    af = float(np.float32(a))
    p = 1.0 / (1.0 + math.exp(-abs(af)))
    h2 = -(p * math.log(p) + (1 - p) * math.log(1 - p))
    want = w1 * (1 - h2 / math.log(2.0)) + w2 * p + w3 * p
    c = oracle.confidence(np.array([af, 0.0], dtype=np.float32))[0]
    assert abs(c - want) < 1e-13


def test_budget_rule_as_printed():
    # c >= tau -> the tight budget N_high; c < tau -> N_low (golden fixture)
    assert _printed_constants()["high_confidence_rule"] == "ge"
    z = np.array([math.log(3.0), 0.0], dtype=np.float32)
    c = np.float32(oracle.confidence(z)[0])          # c and tau compare in fp32
    assert oracle.budget(c, tau=c, n_low=64, n_high=16) == 16
    above = np.nextafter(c, np.float32(2.0))
    assert oracle.budget(c, tau=above, n_low=64, n_high=16) == 64
