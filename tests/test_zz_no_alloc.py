"""The allocation-free confidence entry point against the context-based step
and the CPU oracle.

Runs last (file name) so that a failure here leaves every other test already
run.  Calls go through the C ABI (ctypes) on device buffers that the test
allocates itself; the entry point must give the same c (within the 1e-5
tolerance the parity tests use) and the same budgets as confkv_step's conf /
budget outputs and as the oracle's confidence, on two calls in a row.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL_C = 1e-5


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _step_conf(pkg, logits, tau, n_low, n_high):
    """c and budgets from the existing entry point (confkv_step on a context)."""
    B, V = logits.shape
    kv = pkg.ConfKV(1, 2, 1, 64, n_low, n_high, tau, 2, 4, 0.9, batch=B, vocab=V, device=0)
    q = torch.zeros(1, B, 2, 64, dtype=torch.float16, device=DEV)
    k = torch.zeros(1, B, 1, 64, dtype=torch.float16, device=DEV)
    out = torch.zeros(1, B, 2, 64, device=DEV)
    cf = torch.zeros(B, device=DEV)
    bd = torch.zeros(B, dtype=torch.int32, device=DEV)
    kv.step(logits, q, k, k, out, conf=cf, budget=bd)
    torch.cuda.synchronize()
    kv.close()
    return cf.cpu().numpy(), bd.cpu().numpy()


def _noalloc(lib, logits, tau, n_low, n_high):
    B, V = logits.shape
    cf = torch.full((B,), -1.0, device=DEV)
    bd = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    fl = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    rc = lib.confkv_confidence_noalloc(_ptr(logits), B, V, tau, n_low, n_high, _ptr(cf), _ptr(bd),
                                       _ptr(fl), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, cf.cpu().numpy(), bd.cpu().numpy(), fl.cpu().numpy()


@pytest.mark.parametrize("B,V", [(8, 152064), (3, 50257), (1, 201088)])
def test_noalloc_matches_step_on_two_calls(B, V):
    import confidence_gated_kv_logits_gb300 as pkg
    lib = pkg.load_library()
    rng = np.random.default_rng(B * 7 + V)
    tau, n_low, n_high = 0.5, 64, 32
    batches = []
    for _ in range(2):
        lg = (rng.standard_normal((B, V)) / rng.choice([0.05, 0.3, 3.0], size=(B, 1))).astype(np.float32)
        batches.append(torch.from_numpy(lg).to(DEV))
    for lg in batches:                       # two calls in a row, different logits
        c_ref, b_ref = _step_conf(pkg, lg, tau, n_low, n_high)
        rc, c, bud, fl = _noalloc(lib, lg, tau, n_low, n_high)
        assert rc == pkg.OK
        assert np.max(np.abs(c - c_ref)) < TOL_C
        assert np.array_equal(bud, b_ref) and not fl.any()
        lg_h = lg.cpu().numpy()
        for b in range(B):
            c_orc = oracle.confidence(lg_h[b])[0]
            assert abs(float(c[b]) - c_orc) < TOL_C, (b, c[b], c_orc)
            if abs(c_orc - tau) > TOL_C:
                assert bud[b] == oracle.budget(c_orc, tau, n_low, n_high)
    rc, c2, bud2, _ = _noalloc(lib, batches[1], tau, n_low, n_high)   # and again on the same input
    assert rc == pkg.OK and np.array_equal(c2, c) and np.array_equal(bud2, bud)


def test_noalloc_flags_and_limits():
    import confidence_gated_kv_logits_gb300 as pkg
    lib = pkg.load_library()
    lg = torch.zeros(4, 1000, device=DEV)
    lg[1, 3] = float("nan")
    lg[2, :] = float("-inf")
    rc, c, bud, fl = _noalloc(lib, lg, 0.5, 64, 32)
    assert rc == pkg.OK
    assert list(fl) == [0, pkg.FLAG_NONFINITE, pkg.FLAG_NONFINITE, 0]
    assert c[1] == 0 and c[2] == 0 and bud[1] == 64 and bud[2] == 64
    c_ref, _ = _step_conf(pkg, lg[[0]].contiguous(), 0.5, 64, 32)
    assert abs(c[0] - c_ref[0]) < TOL_C
    assert abs(c[0] - oracle.confidence(lg[0].cpu().numpy())[0]) < TOL_C
    assert abs(c[3] - oracle.confidence(lg[3].cpu().numpy())[0]) < TOL_C
    big = torch.zeros(1025, 4, device=DEV)                 # batch beyond the scratch limit
    cf = torch.zeros(1025, device=DEV)
    assert lib.confkv_confidence_noalloc(_ptr(big), 1025, 4, 0.5, 64, 32, _ptr(cf), None, None,
                                         None) == pkg.ERR_CAPACITY
