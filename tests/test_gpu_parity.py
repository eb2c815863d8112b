"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (from the method's contract): INT8 codes, budgets and kept sets
bit-exact (a near-tie -- the oracle's keys at the cut, or its c and tau,
within 1e-6 relative -- is a counted divergence, and every test here requires
none); c within 1e-5 absolute; attention outputs within 1e-3 max-abs.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import gen, workloads as wl

from . import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def small(**kw):
    base = dict(name="small", L=2, B=3, Hq=8, Hkv=2, d=128, V=3000, prefill=0, steps=80,
                N_high=48, N_low=72, P=8, W=24)
    base.update(kw)
    return wl.Workload(**base)


# ---------------------------------------------------------------------------
# input generator: device twin bit-identical to the host generator
# ---------------------------------------------------------------------------

def test_device_generator_bit_exact():
    from synth import device as sd
    shape = (3, 2, 5, 97, 64)
    t = torch.empty(shape, dtype=torch.float16, device=DEV)
    sd.fill_f16(t, 0, gen.KIND_KPRE, 0, heavy=True, inner=64, tlen=97, pos0=0)
    ref = gen.gen_f16(0, gen.KIND_KPRE, 0, shape, inner=64, tlen=97, heavy=True).reshape(shape)
    assert np.array_equal(t.cpu().numpy().view(np.uint16), ref.view(np.uint16))
    lg = torch.empty(4, 50257, dtype=torch.float32, device=DEV)
    sd.fill_logits(lg, 0, 7, 0.3)
    ref = gen.gen_logits(0, 7, 4, 50257, 0.3)
    assert np.array_equal(lg.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    w = wl.QWEN32B.with_(L=2, B=2, prefill=300)
    dl, dq, dk, dv = sd.step_inputs(w, 5)
    hl, hq, hk, hv = wl.step_inputs(w, 5)
    for a, b in ((dl, hl), (dq, hq), (dk, hk), (dv, hv)):
        assert np.array_equal(a.cpu().numpy(), b)


# ---------------------------------------------------------------------------
# confidence reduction and budget
# ---------------------------------------------------------------------------

def _conf_case(V, logits):
    import confidence_gated_kv_logits_gb300 as pkg
    B = logits.shape[0]
    kv = pkg.ConfKV(1, 2, 1, 64, 8, 4, 0.5, 2, 4, 0.9, batch=B, vocab=V, device=0)
    lg = torch.from_numpy(np.ascontiguousarray(logits)).to(DEV)
    q = torch.zeros(1, B, 2, 64, dtype=torch.float16, device=DEV)
    k = torch.zeros(1, B, 1, 64, dtype=torch.float16, device=DEV)
    out = torch.zeros(1, B, 2, 64, device=DEV)
    cf = torch.zeros(B, device=DEV)
    bd = torch.zeros(B, dtype=torch.int32, device=DEV)
    kv.step(lg, q, k, k, out, conf=cf, budget=bd)
    st, rc = kv.stats(check=False)
    kv.close()
    return cf.cpu().numpy(), bd.cpu().numpy(), st, rc


@pytest.mark.parametrize("V", [2, 7, 1000, 50257, 152064, 201088])
def test_confidence_parity(V):
    rng = np.random.default_rng(V)
    B = 8
    lg = np.empty((B, V), np.float32)
    temps = [0.05, 0.1, 0.3, 0.3, 1.0, 3.0, 0.02, 10.0]
    for b in range(B):
        lg[b] = rng.standard_normal(V) / temps[b] + rng.uniform(-50, 50)
    if V > 10:
        lg[6, rng.choice(V, V // 3, replace=False)] = -np.inf      # masked tokens
        lg[7, :] = 1.5                                              # uniform
    c, bud, st, rc = _conf_case(V, lg)
    assert rc == 0
    for b in range(B):
        co = oracle.confidence(lg[b])[0]
        assert abs(c[b] - co) < 1e-5, (b, c[b], co)
        if abs(co - 0.5) > 1e-5:
            assert bud[b] == (4 if co >= 0.5 else 8)


def test_confidence_nonfinite_is_flagged_not_fatal():
    import confidence_gated_kv_logits_gb300 as pkg
    lg = np.zeros((3, 100), np.float32)
    lg[1, 5] = np.nan
    lg[2, :] = -np.inf
    c, bud, st, rc = _conf_case(100, lg)
    assert rc == pkg.ERR_NONFINITE_LOGITS and st["error_flags"] & pkg.FLAG_NONFINITE
    assert c[1] == 0 and c[2] == 0 and bud[1] == 8 and bud[2] == 8
    assert abs(c[0] - oracle.confidence(lg[0])[0]) < 1e-5


# ---------------------------------------------------------------------------
# whole-step parity on small shapes (several tiles, ragged tails)
# ---------------------------------------------------------------------------

def _check(rep):
    """Every lane-step compared with the oracle, no near-tie divergence."""
    return parity.check(rep)


def test_gqa_d128_decode_from_empty():
    _check(parity.run(small(steps=120)))


def test_gqa_d128_prefill_and_budget_drops():
    w = small(prefill=150, L=2, B=3, Hq=40, Hkv=8, N_high=40, N_low=70, P=8, W=20, steps=60,
              V=64)
    rep = _check(parity.run(w))
    assert rep.stats["tokens_evicted"] > 0 and rep.stats["tokens_moved"] > 0


def test_mha_d64_gpt2_shape_1layer():
    w = wl.GPT2_L1.with_(steps=900)
    rep = _check(parity.run(w, check_codes_every=100))
    assert rep.stats["tokens_evicted"] > 0


def test_gqa8_d64_pyramid():
    w = small(L=4, B=2, Hq=64, Hkv=8, d=64, pyramid_min=0.5, prefill=100, steps=50,
              N_high=30, N_low=60, P=6, W=12, V=500)
    _check(parity.run(w))


# 2..8 splits merge inside a thread-block cluster, 12 through global memory;
# tma 0: TMA tiles (128-byte swizzle at d = 128, 64-byte INT8 swizzle at
# d = 64), -1: cp.async staging
@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("splits", [1, 3, 8, 12])
@pytest.mark.parametrize("kernel,tma", [(1, 0), (2, 0), (2, -1)])
def test_forced_split_counts_and_kernels(splits, kernel, tma, d):
    w = small(prefill=90, steps=40, V=64, d=d)
    _check(parity.run(w, splits=splits, kernel=kernel, tma=tma))


@pytest.mark.parametrize("kernel,tma", [(1, 0), (2, 0), (2, -1)])
@pytest.mark.parametrize("Hq,Hkv,d", [(12, 12, 64), (40, 8, 128), (64, 8, 64), (6, 2, 128),
                                      (7, 1, 64), (16, 2, 128)])
def test_attention_kernels_over_group_sizes(kernel, tma, Hq, Hkv, d):
    w = small(L=1, B=2, Hq=Hq, Hkv=Hkv, d=d, prefill=77, steps=25, N_high=40, N_low=60,
              P=5, W=19, V=64)
    _check(parity.run(w, kernel=kernel, tma=tma))


def test_large_values_and_scale_extremes():
    # keys/values far from N(0,1): exercises the per-chunk power-of-two scaling
    rng = np.random.default_rng(9)
    w = small(L=1, B=1, prefill=100, steps=20, V=64)

    def big(s, lg):
        return lg
    import confidence_gated_kv_logits_gb300 as pkg
    kv = pkg.ConfKV.for_workload(w, device=0)
    orc = oracle.Oracle.for_workload(w)
    k = (rng.standard_normal((w.Hkv, 100, w.d)) * 300).astype(np.float16)
    v = (rng.standard_normal((w.Hkv, 100, w.d)) * np.logspace(-4, 2, 100)[None, :, None]
         ).astype(np.float16)
    orc.prefill_lb(0, 0, k, v)
    kv.prefill(torch.from_numpy(k[None, None]).to(DEV), torch.from_numpy(v[None, None]).to(DEV), 100)
    out = torch.zeros(1, 1, w.Hq, w.d, device=DEV)
    for s in range(w.steps):
        lg, q, kn, vn = wl.step_inputs(w, s)
        q = (q.astype(np.float32) * 0.01).astype(np.float16)
        kv.step(*(torch.from_numpy(np.ascontiguousarray(x)).to(DEV) for x in (lg, q, kn, vn)), out)
        r = orc.step(lg, q, kn, vn)
        torch.cuda.synchronize()
        o = out.cpu().numpy()
        assert np.max(np.abs(o - r["out"])) < 1e-3 * max(1.0, np.max(np.abs(r["out"])))
    kv.close()


def test_sliding_window_special_case_is_exact():
    # beta = 1 freezes the EMA: keys are pure recency, identical in both precisions
    w = small(beta=1.0, prefill=60, steps=60, V=64)
    rep = _check(parity.run(w))
    assert rep.kept_div == 0


@pytest.mark.parametrize("P,W,N_high,N_low", [(1, 1, 1, 2), (5, 5, 5, 9), (8, 40, 8, 8),
                                              (16, 16, 20, 17)])
def test_edge_windows_and_budgets(P, W, N_high, N_low):
    w = small(P=P, W=W, N_high=N_high, N_low=N_low, prefill=33, steps=45, V=64, L=1, B=2)
    _check(parity.run(w))


def test_short_context_noop():
    w = small(N_high=500, N_low=500, W=500, P=8, prefill=70, steps=40)
    rep = _check(parity.run(w))
    assert rep.stats["tokens_evicted"] == 0


def test_prefill_shorter_than_window_and_empty_prefill():
    _check(parity.run(small(prefill=10, W=24, steps=50)))
    _check(parity.run(small(prefill=0, W=24, steps=30)))


def test_needles_q_last_seed():
    w = wl.QWEN14B.with_(L=2, B=1, prefill=2000, W=128, P=32, N_high=256, N_low=512,
                         steps=12, needles=16, V=5000)
    _check(parity.run(w))


# ---------------------------------------------------------------------------
# full-size shapes in the benchmark's launch configuration, sampled (l, b)
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_full_size_qwen32b_sampled():
    # the benchmark's workload over its first 160 decode steps: the budget
    # drop right after the 8192-token prefill, steady-state EMA eviction, the
    # temperature switch at step 64 and the one-token-per-step regrowth after
    # each drop to N_high
    w = wl.QWEN32B
    lbs = [(0, 0), (31, 5), (63, 7)]
    rep = _check(parity.run(w, steps=160, lbs=lbs, device_inputs=True, check_codes_every=20))
    assert rep.stats["tokens_evicted"] > 0 and rep.steps == 160


# ---------------------------------------------------------------------------
# comparison policies on the same kernels (WINDOW, H2O, RANDOM)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("policy", [1, 2, 3])
@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (12, 12, 64)])
def test_policies_parity(policy, Hq, Hkv, d):
    w = small(L=2, B=3, Hq=Hq, Hkv=Hkv, d=d, prefill=90, steps=60, N_high=40, N_low=70,
              P=8, W=20, V=64)
    rep = _check(parity.run(w, policy=policy, seed=0xC0FFEE))
    assert rep.stats["tokens_evicted"] > 0


def test_window_full_kv_configuration():
    # budget and FP16 window at least the context: nothing evicted, nothing
    # quantised, attention over the full FP16 cache
    w = small(L=2, B=2, prefill=100, steps=40, N_high=160, N_low=160, P=8, W=160, V=64)
    rep = _check(parity.run(w, policy=1))
    assert rep.stats["tokens_evicted"] == 0 and rep.stats["tokens_quantized"] == 0


@pytest.mark.parametrize("d", [128, 64])
def test_attention_path_reported(d):
    import confidence_gated_kv_logits_gb300 as pkg
    w = small(d=d)
    for kw, want in ((dict(), "tensor-core TMA"), (dict(attn_tma=-1), "tensor-core cp.async"),
                     (dict(attn_kernel=1), "cuda-core")):
        kv = pkg.ConfKV.for_workload(w, device=0, **kw)
        assert kv.attention_path() == want
        kv.close()


def test_bounded_wait_gives_up_and_device_stays_usable():
    # the attention's tile wait on a phase that nothing completes gives up
    # after its limit (no fault, no hang), and the GPU keeps working
    import confidence_gated_kv_logits_gb300 as pkg
    gave_up, waited_us = pkg.selftest_bounded_wait(0, timeout_us=2000)
    assert gave_up
    assert 2000.0 <= waited_us < 200000.0
    w = small(steps=6)
    _check(parity.run(w))


# ---------------------------------------------------------------------------
# per-(head, channel) INT8 storage (Mixed-Precision Opslag, "per head and
# channel"): power-of-two channel factors fixed at prefill, on every kernel
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("kernel,tma", [(0, 0), (2, -1), (1, 0)])
def test_channel_mode_parity(d, splits, kernel, tma):
    w = small(prefill=120, steps=50, V=64, d=d, int8_channel=1)
    rep = _check(parity.run(w, splits=splits, kernel=kernel, tma=tma,
                            spread=parity.channel_spread(d), check_codes_every=7))
    assert rep.code_checks > 0 and rep.stats["tokens_quantized"] > 0


def test_channel_mode_exponents_are_nontrivial_and_fixed():
    import confidence_gated_kv_logits_gb300 as pkg
    w = small(prefill=64, steps=10, V=64, int8_channel=1)
    sc = parity.channel_spread(w.d)
    kv = pkg.ConfKV.for_workload(w, device=0)
    K = np.zeros((w.L, w.B, w.Hkv, w.prefill, w.d), np.float16)
    V = np.zeros_like(K)
    for l in range(w.L):
        for b in range(w.B):
            k, v = wl.prefill_kv_lb(w, l, b)
            K[l, b], V[l, b] = parity._spread_host(k, sc), parity._spread_host(v, sc[::-1].copy())
    kv.prefill(parity.to_dev(K, DEV), parity.to_dev(V, DEV), w.prefill)
    fk0, fv0 = kv.read_channel_exponents(1, 2)
    want = np.stack([oracle.channel_exponents(K[1, 2, h]) for h in range(w.Hkv)])
    assert np.array_equal(fk0, want) and len(set(fk0.ravel().tolist())) >= 4
    out = torch.zeros(w.L, w.B, w.Hq, w.d, device=DEV)
    for s in range(w.steps):
        lg, q, k, v = (parity.to_dev(x, DEV) for x in wl.step_inputs(w, s))
        kv.step(lg, q, k, v, out)
    fk1, fv1 = kv.read_channel_exponents(1, 2)
    assert np.array_equal(fk0, fk1) and np.array_equal(fv0, fv1)
    kv.close()
    # without the mode, or without a prompt, every factor is 1
    w0 = small(prefill=0, steps=3, V=64, int8_channel=1)
    kv = pkg.ConfKV.for_workload(w0, device=0)
    assert not any(x.any() for x in kv.read_channel_exponents(0, 0))
    kv.close()


def test_channel_mode_mha_and_decode_from_empty():
    # 12 KV heads: the selection quantises the aging token row by row (the
    # warp-per-row path); no prompt: every factor is 1
    _check(parity.run(wl.GPT2_L1.with_(steps=300, prefill=200, int8_channel=1),
                      spread=parity.channel_spread(64), check_codes_every=50))
    _check(parity.run(small(prefill=0, steps=60, V=64, int8_channel=1)))


def test_channel_mode_per_layer_and_policies():
    w = small(L=3, B=2, Hq=40, Hkv=8, prefill=70, steps=25, V=64, int8_channel=1)
    _check(parity.run(w, per_layer=True, spread=parity.channel_spread(w.d)))
    _check(parity.run(w, policy=2, spread=parity.channel_spread(w.d)))


@pytest.mark.slow
def test_full_size_qwen32b_channel_mode_sampled():
    w = wl.QWEN32B.with_(int8_channel=1)
    rep = _check(parity.run(w, steps=40, lbs=[(0, 0), (40, 3)], device_inputs=True,
                            check_codes_every=13, spread=parity.channel_spread(w.d)))
    assert rep.stats["tokens_evicted"] > 0
