"""GPU-vs-oracle comparison driver shared by the parity tests.

Both sides run free from the same seeded inputs; the oracle never receives a
value computed on the GPU.  Per step and per (layer, sequence):
  * confidence c within 1e-5 absolute; budget decisions identical, except where
    the oracle's c and tau differ by less than 1e-6 relative (counted as a
    budget divergence);
  * kept-position sets identical, except where every differing token's oracle
    ranking key lies within 1e-6 relative of the oracle's cut (counted);
  * attention outputs within 1e-3 max-abs while the kept sets agree;
  * INT8 codes, scales and FP16 rows bit-exact (by position) on checked steps.
A (layer, sequence) that diverged legitimately can no longer be compared with
the oracle (the two caches differ from then on, and the oracle is never fed
GPU state); its GPU-only invariants are still checked every step, and the
lane-steps left uncompared are counted.  Every report is kept in RECORDS so
that the test session can print the divergence counts it saw; the tests
require zero divergences unless they say otherwise.
"""
import numpy as np
import torch

import oracle
from synth import workloads as wl

import os

TOL_C = 1e-5
TOL_OUT = 1e-3
TOL_KEY_REL = 1e-6

RECORDS = []        # (test id, Report) of every run in this process


def to_dev(a, dev):
    # a writable, contiguous host copy: some generators hand out read-only views
    return torch.from_numpy(np.require(a, requirements=("C", "W"))).to(dev)


class Report:
    def __init__(self):
        self.compared = 0       # lane-steps whose kept set, output and c matched
        self.total = 0          # lane-steps run
        self.kept_div = 0       # legitimate kept-set near-tie divergences
        self.budget_div = 0     # legitimate budget near-tie divergences
        self.uncompared = 0     # lane-steps after a divergence (invariants only)
        self.code_checks = 0
        self.max_out_err = 0.0
        self.max_c_err = 0.0
        self.steps = 0

    def __repr__(self):
        return (f"compared={self.compared}/{self.total} kept_div={self.kept_div} "
                f"budget_div={self.budget_div} uncompared={self.uncompared} "
                f"code_checks={self.code_checks} max_out_err={self.max_out_err:.2e} "
                f"max_c_err={self.max_c_err:.2e}")


def budget_near_tie(c_oracle, tau):
    """A budget decision may differ only where the oracle's c and tau differ by
    less than 1e-6 relative (the same rule as the ranking keys)."""
    return abs(c_oracle - tau) < TOL_KEY_REL * max(abs(c_oracle), abs(tau))


def _legit_kept_divergence(keys, kept_o, kept_g):
    """Every differing token's oracle key within 1e-6 relative of the cut."""
    key, pos, prot = keys["key"], keys["pos"], keys["prot"]
    by_pos = {int(p): float(k) for p, k in zip(pos, key)}
    cand_kept = [by_pos[p] for p in kept_o if p in by_pos and not prot[list(pos).index(p)]]
    if not cand_kept:
        return False
    cut = min(cand_kept)
    for p in kept_o ^ kept_g:
        if p not in by_pos:
            return False
        if abs(by_pos[p] - cut) > TOL_KEY_REL * abs(cut):
            return False
    return True


def compare_cache(kv, orc, l, b, rep):
    g = kv.read_cache(l, b)
    o = orc.tokens(l, b)
    if orc.int8_channel:                     # per-(head, channel) exponents, bit-exact
        gk, gv = kv.read_channel_exponents(l, b)
        ok, ov = orc.exponents(l, b)
        assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
    assert sorted(g["pos"].tolist()) == sorted(o["pos"].tolist())
    oi = {int(p): i for i, p in enumerate(o["pos"])}
    for i in range(g["n8"]):
        j = oi[int(g["pos"][i])]
        assert o["is8"][j], "GPU INT8 token is FP16 in the oracle"
        assert np.array_equal(g["k8"][i], o["k8"][j]) and np.array_equal(g["v8"][i], o["v8"][j])
        assert np.array_equal(g["ks"][i], o["ks"][j]) and np.array_equal(g["vs"][i], o["vs"][j])
    for i in range(g["n16"]):
        j = oi[int(g["pos"][g["n8"] + i])]
        assert not o["is8"][j], "GPU FP16 token is INT8 in the oracle"
        assert np.array_equal(g["k16"][i], o["k16"][j]) and np.array_equal(g["v16"][i], o["v16"][j])
    rep.code_checks += 1


def channel_spread(d, seed=3):
    """Per-channel powers of two in [2^-7, 1] (K; V uses them reversed): the
    unequal channel magnitudes that the per-(head, channel) INT8 mode is for."""
    rng = np.random.default_rng(seed)
    return np.exp2(-rng.integers(0, 8, size=d)).astype(np.float32)


def _spread_host(x, sc):
    """fp16 x times per-channel powers of two, one rounding to fp16."""
    return (x.astype(np.float32) * sc).astype(np.float16)


def _spread_dev(x, sc):
    """The same on the device: the fp16 product of x and a power of two is
    exact in fp32, so torch's fp16 multiply rounds it once, like numpy."""
    return x * torch.from_numpy(sc.astype(np.float16)).to(x.device)


def run(w, steps=None, lbs=None, device_inputs=False, check_codes_every=16, splits=0,
        logits_override=None, kernel=0, tma=0, per_layer=False, policy=0, seed=0, spread=None):
    """Run workload `w` on the GPU and in the oracle; return a Report.

    lbs: iterable of (l, b) the oracle simulates (default: all).
    device_inputs: generate the GPU's inputs with the device generator (large
      workloads); the oracle always uses the host generator.
    logits_override: optional fn(s, logits) -> logits applied to both sides.
    spread: optional per-channel powers of two (length d) multiplying every
      K (and, reversed, every V) row of the prefill and of each step, on both
      sides identically.
    per_layer: True runs every step through confkv_step_begin + one
      confkv_step_layer per layer (reversed order); a callable s -> bool
      chooses per step (mixed per-layer and whole steps).
    """
    sk = None if spread is None else np.asarray(spread, np.float32)
    sv = None if spread is None else sk[::-1].copy()
    import confidence_gated_kv_logits_gb300 as pkg
    dev = torch.device("cuda", 0)
    steps = w.steps if steps is None else steps
    kv = pkg.ConfKV.for_workload(w, device=0, attn_splits=splits, attn_kernel=kernel,
                                attn_tma=tma, policy=policy, seed=seed)
    orc = oracle.Oracle.for_workload(w, policy, seed)
    fixed_budget = policy == oracle.POLICY_WINDOW      # no confidence computed
    all_lbs = [(l, b) for l in range(w.L) for b in range(w.B)]
    lbs = all_lbs if lbs is None else list(lbs)
    mask = np.zeros((w.L, w.B), np.uint8)
    for l, b in lbs:
        mask[l, b] = 1
    orc.set_active(mask)
    rep = Report()
    test_id = os.environ.get("PYTEST_CURRENT_TEST", w.name).rsplit(" (", 1)[0]
    RECORDS.append((test_id, rep))      # recorded first: a failing run still shows its counts
    # ---- prefill ----
    if w.prefill:
        if device_inputs:
            from synth import device as sd
            K, V = sd.prefill_kv(w)
            if sk is not None:
                K, V = _spread_dev(K, sk), _spread_dev(V, sv)
        else:
            K = np.zeros((w.L, w.B, w.Hkv, w.prefill, w.d), np.float16)
            V = np.zeros_like(K)
        ql = wl.q_last(w)
        for l, b in (lbs if device_inputs else all_lbs):
            k, v = wl.prefill_kv_lb(w, l, b)
            if sk is not None:
                k, v = _spread_host(k, sk), _spread_host(v, sv)
            if not device_inputs:
                K[l, b], V[l, b] = k, v
            if mask[l, b]:
                orc.prefill_lb(l, b, k, v, None if ql is None else ql[l, b])
        if not device_inputs:
            K, V = to_dev(K, dev), to_dev(V, dev)
        kv.prefill(K, V, w.prefill, None if ql is None else to_dev(ql, dev))
        del K, V
    else:
        orc.set_position(0)
    out = torch.zeros(w.L, w.B, w.Hq, w.d, device=dev)
    kp = torch.full((w.L, w.B, kv.Ncap), -1, dtype=torch.int32, device=dev)
    kc = torch.zeros(w.L, w.B, dtype=torch.int32, device=dev)
    cf = torch.zeros(w.B, device=dev)
    bd = torch.zeros(w.B, dtype=torch.int32, device=dev)
    diverged = set()
    prev = {}
    for s in range(steps):
        if device_inputs and lbs is not all_lbs:
            lg, q, k, v = wl.step_inputs_lanes(w, s, lbs)     # host inputs of the sampled lanes
        else:
            lg, q, k, v = wl.step_inputs(w, s)
        if logits_override is not None:
            lg = logits_override(s, lg)
        if sk is not None:
            k, v = _spread_host(k, sk), _spread_host(v, sv)
        if device_inputs and logits_override is None:
            from synth import device as sd
            glg, gq, gk, gv = sd.step_inputs(w, s)
            if sk is not None:
                gk, gv = _spread_dev(gk, sk), _spread_dev(gv, sv)
        else:
            glg, gq, gk, gv = (to_dev(x, dev) for x in (lg, q, k, v))
        if per_layer is True or (callable(per_layer) and per_layer(s)):
            # confkv_step_begin + one confkv_step_layer per layer, reversed
            kv.step_begin(glg, cf, bd)
            for l in reversed(range(w.L)):
                ol = torch.empty(w.B, w.Hq, w.d, device=dev)
                kpl = torch.full((w.B, kv.Ncap), -1, dtype=torch.int32, device=dev)
                kcl = torch.zeros(w.B, dtype=torch.int32, device=dev)
                kv.step_layer(l, gq[l].contiguous(), gk[l].contiguous(), gv[l].contiguous(), ol,
                              kpl, kcl)
                out[l], kp[l], kc[l] = ol, kpl, kcl
        else:
            kv.step(glg, gq, gk, gv, out, kp, kc, cf, bd)
        r = orc.step(lg, q, k, v, cap=kv.Ncap)
        torch.cuda.synchronize()
        g_out, g_kp, g_kc = out.cpu().numpy(), kp.cpu().numpy(), kc.cpu().numpy()
        g_cf, g_bd = cf.cpu().numpy(), bd.cpu().numpy()
        t = w.position(s)
        if fixed_budget:
            g_bd = np.full(w.B, w.N_low, np.int32)
        for b in range(w.B):
            if fixed_budget:
                break
            rep.max_c_err = max(rep.max_c_err, abs(float(g_cf[b]) - r["conf"][b]))
            assert abs(float(g_cf[b]) - r["conf"][b]) < TOL_C, (s, b, g_cf[b], r["conf"][b])
            if g_bd[b] != r["budget"][b]:          # c depends on the logits only
                assert budget_near_tie(r["conf"][b], w.tau), (s, b, g_cf[b], r["conf"][b])
                rep.budget_div += 1
                diverged |= {(l, b) for l in range(w.L)}
        for l, b in lbs:
            rep.total += 1
            n = int(g_kc[l, b])
            kept_g = set(g_kp[l, b, :n].tolist())
            N = oracle.layer_budget(int(g_bd[b]), l, w.L, w.pyramid_min, w.P)
            # GPU-only invariants
            assert len(kept_g) == n <= max(N, 1)
            assert set(range(max(0, t - w.P + 1), t + 1)) <= kept_g
            if (l, b) in prev:
                assert kept_g <= prev[(l, b)] | {t}
            prev[(l, b)] = kept_g
            if (l, b) in diverged:
                rep.uncompared += 1
                continue
            kept_o = set(r["kept_pos"][l, b, :r["kept_count"][l, b]].tolist())
            if kept_g != kept_o:
                assert _legit_kept_divergence(orc.last_keys(l, b), kept_o, kept_g), (
                    s, l, b, sorted(kept_g ^ kept_o))
                rep.kept_div += 1
                rep.uncompared += 1
                diverged.add((l, b))
                continue
            err = float(np.max(np.abs(g_out[l, b] - r["out"][l, b])))
            rep.max_out_err = max(rep.max_out_err, err)
            assert err < TOL_OUT, (s, l, b, err)
            rep.compared += 1
            if check_codes_every and (s % check_codes_every == 0 or s == steps - 1):
                compare_cache(kv, orc, l, b, rep)
        rep.steps += 1
    st, rc = kv.stats(check=False)
    kv.close()
    rep.stats = st
    rep.rc = rc
    return rep


def check(rep, allowed_divergences=0):
    """Every lane-step compared unless a counted near-tie divergence stopped a
    lane; at most `allowed_divergences` of them (0 unless a test is about
    near-ties)."""
    assert rep.rc == 0, rep.rc
    assert rep.kept_div + rep.budget_div <= allowed_divergences, rep
    if allowed_divergences == 0:
        assert rep.compared == rep.total and rep.uncompared == 0, rep
    else:
        assert rep.compared + rep.uncompared == rep.total, rep
    return rep
