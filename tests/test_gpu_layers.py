"""Per-layer stepping (confkv_step_begin + confkv_step_layer) on the GPU.

The per-layer calls must give what one confkv_step gives: bit-identical
outputs for the same split-K factor, and parity with the oracle.
"""
import numpy as np
import pytest
import torch

from synth import workloads as wl

from . import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def small(**kw):
    base = dict(name="layers", L=3, B=2, Hq=8, Hkv=2, d=128, V=500, prefill=60, steps=30,
                N_high=40, N_low=56, P=6, W=20)
    base.update(kw)
    return wl.Workload(**base)


def _T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("d,splits,kernel", [(128, 1, 0), (128, 3, 0), (64, 2, 0), (128, 5, 0),
                                             (128, 2, 1), (64, 1, 1)])
def test_per_layer_equals_full_step_bitwise(d, splits, kernel):
    # kernel 0: the tensor-core attention stores the arriving token itself;
    # kernel 1: the CUDA-core attention after a separate append launch
    import confidence_gated_kv_logits_gb300 as pkg
    w = small(d=d)
    a = pkg.ConfKV.for_workload(w, device=0, attn_splits=splits, attn_kernel=kernel)
    b = pkg.ConfKV.for_workload(w, device=0, attn_splits=splits, attn_kernel=kernel)
    kvs = [[wl.prefill_kv_lb(w, l, bb) for bb in range(w.B)] for l in range(w.L)]
    K = np.stack([np.stack([x[0] for x in row]) for row in kvs])
    V = np.stack([np.stack([x[1] for x in row]) for row in kvs])
    a.prefill(_T(K), _T(V), w.prefill)
    b.prefill(_T(K), _T(V), w.prefill)
    for s in range(w.steps):
        lg, q, k, v = (_T(x) for x in wl.step_inputs(w, s))
        oa = torch.empty(w.L, w.B, w.Hq, w.d, device=DEV)
        kpa = torch.full((w.L, w.B, a.Ncap), -1, dtype=torch.int32, device=DEV)
        kca = torch.zeros(w.L, w.B, dtype=torch.int32, device=DEV)
        a.step(lg, q, k, v, oa, kpa, kca)
        b.step_begin(lg)
        order = np.random.default_rng(s).permutation(w.L)
        for l in order:
            ob = torch.empty(w.B, w.Hq, w.d, device=DEV)
            kpb = torch.full((w.B, b.Ncap), -1, dtype=torch.int32, device=DEV)
            kcb = torch.zeros(w.B, dtype=torch.int32, device=DEV)
            b.step_layer(int(l), q[l].contiguous(), k[l].contiguous(), v[l].contiguous(), ob, kpb, kcb)
            assert torch.equal(ob, oa[l]) and torch.equal(kcb, kca[l])
            assert torch.equal(kpb, kpa[l])
    sa, _ = a.stats()
    sb, _ = b.stats()
    assert sa["position"] == sb["position"] == w.prefill + w.steps
    a.close()
    b.close()


@pytest.mark.parametrize("policy", [0, 2])
def test_per_layer_parity_with_oracle(policy):
    # both policies that rank by the attention mass (CONF-KV's EMA, H2O's
    # accumulated mass) defer it under per-layer stepping
    parity.check(parity.run(small(L=4, Hq=40, Hkv=8, steps=25), per_layer=True, policy=policy,
                            seed=7))


@pytest.mark.parametrize("splits", [0, 1, 12])
def test_mixed_per_layer_and_whole_steps(splits):
    # per-layer launches defer each layer's attention mass to the next step's
    # first kernel; whole steps after per-layer steps (and the reverse) must
    # fold it in exactly as if every step had been whole
    w = small(L=3, Hq=40, Hkv=8, steps=30)
    parity.check(parity.run(w, splits=splits, per_layer=lambda s: (s // 4) % 2 == 0))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g,splits", [(1, 2), (3, 4), (5, 6), (8, 7), (8, 8), (5, 3), (1, 8)])
def test_per_layer_cluster_merge_shapes(d, g, splits):
    # A per-layer launch merges the splits of a unit by sending each CTA of
    # the cluster the bytes it needs -- every split's per-head (max, sum) and
    # the partials of the output blocks it finishes -- and each CTA waits for
    # exactly that many.  Every group size, head dim and split count must
    # deliver them all (a short count would end the wait and flag the step),
    # including splits left without any chunk and partial output blocks.
    Hkv = 2
    w = small(L=2, Hq=g * Hkv, Hkv=Hkv, d=d, prefill=90, steps=8, N_high=60, N_low=80, W=24)
    parity.check(parity.run(w, splits=splits, per_layer=True))


def test_per_layer_state_errors():
    import confidence_gated_kv_logits_gb300 as pkg
    w = small()
    kv = pkg.ConfKV.for_workload(w, device=0)
    q = torch.zeros(w.B, w.Hq, w.d, dtype=torch.float16, device=DEV)
    k = torch.zeros(w.B, w.Hkv, w.d, dtype=torch.float16, device=DEV)
    o = torch.zeros(w.B, w.Hq, w.d, device=DEV)
    lg = torch.zeros(w.B, w.V, device=DEV)
    with pytest.raises(pkg.ConfKVError) as e:
        kv.step_layer(0, q, k, k, o)                       # no begun step
    assert e.value.code == pkg.ERR_STATE
    kv.step_begin(lg)
    with pytest.raises(pkg.ConfKVError) as e:
        kv.step_begin(lg)                                   # layers still to run
    assert e.value.code == pkg.ERR_STATE
    with pytest.raises(pkg.ConfKVError) as e:
        kv.step_layer(w.L, q, k, k, o)                     # bad layer
    assert e.value.code == pkg.ERR_INVALID_ARG
    qbuf = torch.zeros(q.numel() + 8, dtype=torch.float16, device=DEV)
    q_mis = qbuf[4:4 + q.numel()].view(q.shape)            # 8-byte aligned only
    with pytest.raises(pkg.ConfKVError) as e:
        kv.step_layer(1, q_mis, k, k, o)                   # q must be 16-byte aligned
    assert e.value.code == pkg.ERR_INVALID_ARG
    kv.step_layer(1, q, k, k, o)
    with pytest.raises(pkg.ConfKVError) as e:
        kv.step_layer(1, q, k, k, o)                       # layer twice
    assert e.value.code == pkg.ERR_STATE
    kv.step_layer(0, q, k, k, o)
    kv.step_layer(2, q, k, k, o)
    st, rc = kv.stats()
    assert rc == 0 and st["steps"] == 1 and st["position"] == 1     # no prefill here
    kv.close()


def _eager_and_graph(w, per_layer, n_eager, n_replay, policy=0):
    """Runs n_eager eager steps, then n_replay more either eagerly or as
    replays of one captured step; returns the last outputs of each run."""
    import confidence_gated_kv_logits_gb300 as pkg
    results = []
    for graph in (False, True):
        kv = pkg.ConfKV.for_workload(w, device=0, policy=policy, seed=11)
        kvs = [[wl.prefill_kv_lb(w, l, bb) for bb in range(w.B)] for l in range(w.L)]
        K = np.stack([np.stack([x[0] for x in row]) for row in kvs])
        V = np.stack([np.stack([x[1] for x in row]) for row in kvs])
        kv.prefill(_T(K), _T(V), w.prefill)
        # the buffers a captured step reads and writes
        lg = torch.zeros(w.B, w.V, device=DEV)
        q = torch.zeros(w.L, w.B, w.Hq, w.d, dtype=torch.float16, device=DEV)
        k = torch.zeros(w.L, w.B, w.Hkv, w.d, dtype=torch.float16, device=DEV)
        v = torch.zeros_like(k)
        out = torch.zeros(w.L, w.B, w.Hq, w.d, device=DEV)
        kp = torch.full((w.L, w.B, kv.Ncap), -1, dtype=torch.int32, device=DEV)
        kc = torch.zeros(w.L, w.B, dtype=torch.int32, device=DEV)
        conf = torch.zeros(w.B, device=DEV)
        bud = torch.zeros(w.B, dtype=torch.int32, device=DEV)

        def load(s):
            for dst, src in zip((lg, q, k, v), wl.step_inputs(w, s)):
                dst.copy_(torch.from_numpy(np.ascontiguousarray(src)))

        def one_step(stream=None):
            if not per_layer:
                kv.step(lg, q, k, v, out, kp, kc, conf, bud, stream=stream)
                return
            kv.step_begin(lg, conf, bud, stream=stream)
            for l in range(w.L):
                kv.step_layer(l, q[l], k[l], v[l], out[l], kp[l], kc[l], stream=stream)

        for s in range(n_eager):
            load(s)
            one_step()
        g = None
        for s in range(n_eager, n_eager + n_replay):
            load(s)
            if not graph:
                one_step()
            elif g is None:
                # capturing enqueues nothing: the first replay is this step
                torch.cuda.synchronize()
                stream = torch.cuda.Stream()
                stream.wait_stream(torch.cuda.current_stream())
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    one_step(stream)
                g.replay()
            else:
                g.replay()
        torch.cuda.synchronize()
        st, rc = kv.stats()
        assert rc == 0
        assert st["steps"] == n_eager + n_replay
        assert st["position"] == w.prefill + n_eager + n_replay
        results.append([x.cpu().numpy() for x in (out, kp, kc, conf, bud)])
        kv.close()
    return results


@pytest.mark.parametrize("per_layer,policy", [(False, 0), (True, 0), (False, 1), (True, 3),
                                              (False, 2)])
def test_step_graph_replayed_equals_eager(per_layer, policy):
    # one captured step replayed for several decode steps (new inputs written
    # into the captured buffers before each replay) gives the same bits as
    # the same steps run eagerly: the position and all state are on the
    # device (policy 3 draws its keys from the position; 1 has no confidence)
    w = small(L=3, B=2, steps=20)
    eager, graph = _eager_and_graph(w, per_layer, n_eager=4, n_replay=14, policy=policy)
    for a, b in zip(eager, graph):
        if a.dtype == np.float32:
            a, b = a.view(np.uint32), b.view(np.uint32)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("ch,splits", [(0, 1), (1, 1), (0, 2), (1, 2)])
def test_per_layer_cache_state_equals_whole_step(ch, splits):
    # Per-layer launches defer each layer's attention mass to the next
    # step's first kernel (or to an inspection of the cache).  Reading the
    # caches lane by lane between steps finalises the masses repeatedly,
    # which must change nothing: every lane's positions, EMA, mass, codes,
    # scales and FP16 rows equal those of whole steps on the same inputs.
    import confidence_gated_kv_logits_gb300 as pkg
    w = small(L=3, Hq=40, Hkv=8, prefill=70, steps=8, int8_channel=ch)
    a = pkg.ConfKV.for_workload(w, device=0, attn_splits=splits)
    b = pkg.ConfKV.for_workload(w, device=0, attn_splits=splits)
    kvs = [[wl.prefill_kv_lb(w, l, bb) for bb in range(w.B)] for l in range(w.L)]
    K = np.stack([np.stack([x[0] for x in row]) for row in kvs])
    V = np.stack([np.stack([x[1] for x in row]) for row in kvs])
    a.prefill(_T(K), _T(V), w.prefill)
    b.prefill(_T(K), _T(V), w.prefill)
    for s in range(w.steps):
        lg, q, k, v = (_T(x) for x in wl.step_inputs(w, s))
        oa = torch.empty(w.L, w.B, w.Hq, w.d, device=DEV)
        a.step(lg, q, k, v, oa)
        b.step_begin(lg)
        for l in reversed(range(w.L)):
            ob = torch.empty(w.B, w.Hq, w.d, device=DEV)
            b.step_layer(l, q[l].contiguous(), k[l].contiguous(), v[l].contiguous(), ob)
            assert torch.equal(ob, oa[l]), (s, l)
        for l in range(w.L):
            for bb in range(w.B):
                ra, rb = a.read_cache(l, bb), b.read_cache(l, bb)
                for key in ("pos", "ema", "mass", "k8", "v8", "ks", "vs", "k16", "v16"):
                    assert np.array_equal(ra[key], rb[key]), (s, l, bb, key)
    a.close()
    b.close()


def test_read_cache_after_per_layer_steps_on_a_side_stream():
    # the caller's per-layer steps run on a non-blocking stream; reading the
    # caches right after them (no host synchronisation in between) must see
    # the finished step, its deferred masses included
    import confidence_gated_kv_logits_gb300 as pkg
    w = small(L=2, Hq=40, Hkv=8, prefill=70, steps=5)
    a = pkg.ConfKV.for_workload(w, device=0)
    b = pkg.ConfKV.for_workload(w, device=0)
    kvs = [[wl.prefill_kv_lb(w, l, bb) for bb in range(w.B)] for l in range(w.L)]
    K = _T(np.stack([np.stack([x[0] for x in row]) for row in kvs]))
    V = _T(np.stack([np.stack([x[1] for x in row]) for row in kvs]))
    a.prefill(K, V, w.prefill)
    b.prefill(K, V, w.prefill)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    for s in range(w.steps):
        lg, q, k, v = (_T(x) for x in wl.step_inputs(w, s))
        oa = torch.empty(w.L, w.B, w.Hq, w.d, device=DEV)
        a.step(lg, q, k, v, oa)
        side.wait_stream(torch.cuda.current_stream())      # the inputs are ready
        with torch.cuda.stream(side):
            ob = torch.empty(w.L, w.B, w.Hq, w.d, device=DEV)
            b.step_begin(lg, stream=side)
            for l in range(w.L):
                b.step_layer(l, q[l].contiguous(), k[l].contiguous(), v[l].contiguous(), ob[l],
                             stream=side)
        for l in range(w.L):
            for bb in range(w.B):
                ra, rb = a.read_cache(l, bb), b.read_cache(l, bb)
                for key in ("pos", "ema", "mass", "k8", "ks", "k16"):
                    assert np.array_equal(ra[key], rb[key]), (s, l, bb, key)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
    a.close()
    b.close()
