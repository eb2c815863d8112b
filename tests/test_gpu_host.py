"""confkv_step_host (host buffers, copies inside the call) on the GPU.

The host path overlaps the input copy with the confidence and selection
kernels and cuts the attention into ranges whose outputs are copied back
while the next range computes; its results must be bitwise those of
confkv_step on device buffers.
"""
import numpy as np
import pytest
import torch

from synth import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _prefilled(w, **kw):
    import confidence_gated_kv_logits_gb300 as pkg
    kv = pkg.ConfKV.for_workload(w, device=0, **kw)
    if w.prefill:
        kvs = [[wl.prefill_kv_lb(w, l, b) for b in range(w.B)] for l in range(w.L)]
        K = np.stack([np.stack([x[0] for x in row]) for row in kvs])
        V = np.stack([np.stack([x[1] for x in row]) for row in kvs])
        kv.prefill(torch.from_numpy(K).to(DEV), torch.from_numpy(V).to(DEV), w.prefill)
    return kv


def _pinned(shape, dtype):
    return torch.zeros(shape, dtype=dtype).pin_memory().numpy()


def _pageable(shape, dtype):
    return torch.zeros(shape, dtype=dtype).numpy()


@pytest.mark.parametrize("shape", [
    dict(L=3, B=2, Hq=8, Hkv=2, d=128, V=500, prefill=60, steps=12, N_high=40, N_low=56, P=6, W=20),
    dict(L=2, B=3, Hq=16, Hkv=2, d=64, V=300, prefill=30, steps=10, N_high=24, N_low=40, P=4, W=12),
    # 4096 units at d = 128: with pageable outputs the attention runs as two
    # ranges with overlapped copies; pinned outputs are written directly
    dict(L=32, B=16, Hq=16, Hkv=8, d=128, V=64, prefill=40, steps=5, N_high=24, N_low=36, P=4, W=12),
])
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("outs", ["pinned", "pageable"])
def test_step_host_equals_device_step(shape, kernel, outs):
    # pinned (mapped) outputs are written by the kernels directly; pageable
    # ones go through device staging buffers and copies
    alloc = _pinned if outs == "pinned" else _pageable
    w = wl.Workload(name="host", **shape)
    a = _prefilled(w, attn_kernel=kernel)
    b = _prefilled(w, attn_kernel=kernel)
    for s in range(w.steps):
        lg, q, k, v = (np.ascontiguousarray(x) for x in wl.step_inputs(w, s))
        dev_in = [torch.from_numpy(x).to(DEV) for x in (lg, q, k, v)]
        oa = torch.zeros(w.L, w.B, w.Hq, w.d, device=DEV)
        kpa = torch.full((w.L, w.B, a.Ncap), -1, dtype=torch.int32, device=DEV)
        kca = torch.zeros(w.L, w.B, dtype=torch.int32, device=DEV)
        cfa = torch.zeros(w.B, device=DEV)
        bda = torch.zeros(w.B, dtype=torch.int32, device=DEV)
        a.step(*dev_in, oa, kpa, kca, cfa, bda)
        hin = []
        for x in (lg, q, k, v):
            h = _pinned(x.shape, torch.float32 if x.dtype == np.float32 else torch.float16)
            h[...] = x
            hin.append(h)
        ob = alloc((w.L, w.B, w.Hq, w.d), torch.float32)
        kpb = alloc((w.L, w.B, b.Ncap), torch.int32)
        kpb[...] = -1
        kcb = alloc((w.L, w.B), torch.int32)
        cfb = alloc((w.B,), torch.float32)
        bdb = alloc((w.B,), torch.int32)
        b.step_host(*hin, ob, kpb, kcb, cfb, bdb)
        assert np.array_equal(ob.view(np.uint32), oa.cpu().numpy().view(np.uint32))
        assert np.array_equal(kcb, kca.cpu().numpy())
        # entries past kept_count are unspecified (the staging keeps old ones)
        kpa_h = kpa.cpu().numpy()
        for l in range(w.L):
            for bb in range(w.B):
                n = kcb[l, bb]
                assert np.array_equal(kpb[l, bb, :n], kpa_h[l, bb, :n])
        assert np.array_equal(cfb.view(np.uint32), cfa.cpu().numpy().view(np.uint32))
        assert np.array_equal(bdb, bda.cpu().numpy())
    sa, ra = a.stats()
    sb, rb = b.stats()
    # the host step may run its attention as two launches (copy overlap), so
    # only the launch counts may differ
    la, lb_ = sa.pop("kernel_launches"), sb.pop("kernel_launches")
    assert ra == rb == 0 and sa == sb
    assert la >= 3 * w.steps and lb_ >= la
    a.close()
    b.close()


def test_step_host_optional_outputs_null():
    w = wl.Workload(name="host", L=2, B=2, Hq=8, Hkv=2, d=128, V=200, prefill=30, steps=4,
                    N_high=24, N_low=32, P=4, W=12)
    a = _prefilled(w)
    b = _prefilled(w)
    for s in range(w.steps):
        lg, q, k, v = (np.ascontiguousarray(x) for x in wl.step_inputs(w, s))
        oa = torch.zeros(w.L, w.B, w.Hq, w.d, device=DEV)
        a.step(*(torch.from_numpy(x).to(DEV) for x in (lg, q, k, v)), oa)
        ob = _pinned((w.L, w.B, w.Hq, w.d), torch.float32)
        b.step_host(lg, q, k, v, ob)                  # pageable inputs, no optional outputs
        assert np.array_equal(ob.view(np.uint32), oa.cpu().numpy().view(np.uint32))
    a.close()
    b.close()


@pytest.mark.parametrize("policy", [1, 2, 3])
def test_step_host_policies(policy):
    # WINDOW runs without logits (NULL) and writes no c / budget; H2O and
    # RANDOM as CONF-KV: the host path equals the device step bit for bit
    w = wl.Workload(name="host", L=2, B=2, Hq=8, Hkv=2, d=128, V=200, prefill=50, steps=8,
                    N_high=24, N_low=40, P=4, W=12)
    a = _prefilled(w, policy=policy, seed=5)
    b = _prefilled(w, policy=policy, seed=5)
    for s in range(w.steps):
        lg, q, k, v = (np.ascontiguousarray(x) for x in wl.step_inputs(w, s))
        oa = torch.zeros(w.L, w.B, w.Hq, w.d, device=DEV)
        kca = torch.zeros(w.L, w.B, dtype=torch.int32, device=DEV)
        dl = None if policy == 1 else torch.from_numpy(lg).to(DEV)
        a.step(dl, *(torch.from_numpy(x).to(DEV) for x in (q, k, v)), oa, None, kca)
        ob = _pinned((w.L, w.B, w.Hq, w.d), torch.float32)
        kcb = _pinned((w.L, w.B), torch.int32)
        b.step_host(None if policy == 1 else lg, q, k, v, ob, None, kcb)
        assert np.array_equal(ob.view(np.uint32), oa.cpu().numpy().view(np.uint32))
        assert np.array_equal(kcb, kca.cpu().numpy())
    a.close()
    b.close()


def test_step_host_misaligned_pinned_output():
    # A pinned output that is not 4-byte aligned cannot take the kernels'
    # direct 4-byte stores: the call must route it through staging (checked
    # on the host before anything is enqueued) and return the same bits.
    w = wl.Workload(name="host", L=2, B=2, Hq=8, Hkv=2, d=128, V=300, prefill=30, steps=4,
                    N_high=24, N_low=32, P=4, W=12)
    a = _prefilled(w)
    b = _prefilled(w)
    n = w.L * w.B * w.Hq * w.d
    raw = torch.zeros(4 * n + 8, dtype=torch.uint8).pin_memory().numpy()
    ob = np.frombuffer(raw, dtype=np.float32, count=n, offset=2).reshape(w.L, w.B, w.Hq, w.d)
    assert ob.ctypes.data % 4 == 2 and ob.flags.c_contiguous
    for s in range(w.steps):
        lg, q, k, v = (np.ascontiguousarray(x) for x in wl.step_inputs(w, s))
        oa = torch.zeros(w.L, w.B, w.Hq, w.d, device=DEV)
        a.step(*[torch.from_numpy(x).to(DEV) for x in (lg, q, k, v)], oa)
        b.step_host(lg, q, k, v, ob)
        assert np.array_equal(ob.view(np.uint32), oa.cpu().numpy().view(np.uint32))
    assert a.stats()[1] == b.stats()[1] == 0
    a.close()
    b.close()
