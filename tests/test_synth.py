"""The seeded input generator: distribution, determinism, workload structure."""
import numpy as np

from synth import gen, workloads as wl


def test_normal_moments_and_determinism():
    key = gen.stream_key(0, gen.KIND_Q, 3)
    z = gen.normal_f64(key, np.arange(400_000))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs((z ** 4).mean() - 3) < 0.05
    assert np.array_equal(z[1000:2000], gen.normal_f64(key, np.arange(1000, 2000)))
    other = gen.normal_f64(gen.stream_key(0, gen.KIND_Q, 4), np.arange(1000))
    assert not np.array_equal(z[:1000], other)


def test_series_accuracy():
    x = np.random.default_rng(0).random(50_000) + 1e-12
    assert np.max(np.abs(gen._ln(x) - np.log(x))) < 1e-14
    u = np.arange(0, 1 << 16, dtype=np.float64) / (1 << 16)
    assert np.max(np.abs(gen._cos2pi(u) - np.cos(2 * np.pi * u))) < 1e-14


def test_heavy_keys_and_temperature_segments():
    w = wl.GPT2_L1
    k95, k96 = wl.step_k(w, 95), wl.step_k(w, 96)
    raw96 = gen.gen_f16(w.seed, gen.KIND_KNEW, 96, (1, 1, 12, 64)).reshape(k96.shape)
    assert np.array_equal(k96.astype(np.float32), 4 * raw96.astype(np.float32))
    assert w.temperature(0) == 0.3 and w.temperature(64) == 3.0 and w.temperature(128) == 0.3


def test_prefill_slice_matches_full_tensor_and_needles():
    w = wl.QWEN14B.with_(L=2, B=2, Hkv=2, Hq=4, d=8, prefill=700, W=64, needles=4)
    full = gen.gen_f16(w.seed, gen.KIND_KPRE, 0, (2, 2, 2, 700, 8), inner=8, tlen=700,
                       heavy=True).reshape(2, 2, 2, 700, 8)
    k, v = wl.prefill_kv_lb(w, 1, 0, )
    pos = gen.needle_positions(w.seed, 0, 700, 64, 4)
    assert len(set(pos.tolist())) == 4 and pos.max() < 700 - 64
    mask = np.ones(700, bool)
    mask[pos] = False
    assert np.array_equal(k[:, mask], full[1, 0][:, mask])
    u = gen.needle_direction(w.seed, 2, 2, 8)[1]
    for p in pos:
        nk = k[:, p].astype(np.float64)
        cos = np.sum(nk * u, -1) / np.linalg.norm(nk, axis=-1)
        assert np.all(cos > 0.999)
    assert wl.q_last(w).shape == (2, 2, 4, 8)


def test_lane_inputs_match_full_inputs():
    w = wl.QWEN32B.with_(L=3, B=2, V=500, prefill=100)
    full = wl.step_inputs(w, 7)
    lane = wl.step_inputs_lane(w, 7, 2, 1)
    assert np.array_equal(full[0], lane[0])
    for a, b in zip(full[1:], lane[1:]):
        assert np.array_equal(a[2, 1], b[2, 1]) and not b[0].any()
