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


@pytest.mark.parametrize("d,splits", [(128, 1), (128, 3), (64, 2)])
def test_per_layer_equals_full_step_bitwise(d, splits):
    import confidence_gated_kv_logits_gb300 as pkg
    w = small(d=d)
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


def test_per_layer_parity_with_oracle():
    rep = parity.run(small(L=4, Hq=40, Hkv=8, steps=25), per_layer=True)
    print(rep)
    assert rep.rc == 0 and rep.compared >= 0.6 * rep.total


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


def test_step_captured_in_cuda_graph_equals_eager():
    # a step captured in a CUDA graph (allocation-free, no host sync) and
    # replayed once gives the same bits as the same step run eagerly
    import confidence_gated_kv_logits_gb300 as pkg
    w = small(L=2, B=2, steps=12)
    outs = []
    for graph in (False, True):
        kv = pkg.ConfKV.for_workload(w, device=0)
        out = torch.zeros(w.L, w.B, w.Hq, w.d, device=DEV)
        kp = torch.full((w.L, w.B, kv.Ncap), -1, dtype=torch.int32, device=DEV)
        kc = torch.zeros(w.L, w.B, dtype=torch.int32, device=DEV)
        inputs = [tuple(torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
                        for x in wl.step_inputs(w, s)) for s in range(w.steps)]
        torch.cuda.synchronize()
        for s in range(w.steps - 1):
            kv.step(*inputs[s], out, kp, kc)
        last = inputs[-1]
        if graph:
            stream = torch.cuda.Stream()
            stream.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                kv.step(*last, out, kp, kc, stream=stream)
            g.replay()
        else:
            kv.step(*last, out, kp, kc)
        torch.cuda.synchronize()
        st, rc = kv.stats()
        assert rc == 0 and st["steps"] == w.steps
        outs.append((out.cpu().numpy(), kp.cpu().numpy(), kc.cpu().numpy()))
        kv.close()
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                              b.view(np.uint32) if b.dtype == np.float32 else b)
