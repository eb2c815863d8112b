"""Full-size parity: every workload shape of the benchmark suite at its full
size (layers, batch, heads, vocabulary, prefill, budgets), in the launch
configuration the benchmark times (device-generated inputs, automatic split
and kernel choice), against the oracle on sampled (layer, sequence) lanes.
The oracle receives the host generator's inputs for those lanes only.  Step
counts are bounded so the oracle finishes in about a minute per workload;
the first steps after a long prefill include the large budget drop.
"""
import pytest

from synth import workloads as wl

from . import parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _check(rep):
    """Every lane-step compared with the oracle, no near-tie divergence."""
    return parity.check(rep)


def test_gpt2_single_layer_all_2048_steps():
    w = wl.GPT2_L1
    rep = _check(parity.run(w, steps=w.steps, device_inputs=True, check_codes_every=256))
    assert rep.stats["tokens_evicted"] > 0 and rep.stats["tokens_quantized"] > 0


def test_gpt2_full_model_pyramid_sampled():
    w = wl.GPT2_FULL
    rep = _check(parity.run(w, steps=512, lbs=[(0, 0), (6, 3), (11, 7)], device_inputs=True,
                            check_codes_every=128))
    assert rep.stats["tokens_evicted"] > 0


def test_qwen14b_needles_prefill_32768_sampled():
    w = wl.QWEN14B
    rep = _check(parity.run(w, steps=48, lbs=[(0, 0), (47, 0)], device_inputs=True,
                            check_codes_every=16))
    assert rep.stats["tokens_evicted"] > 0


def test_gptoss_sweep_point_sampled():
    w = wl.ALL["gptoss20b-shaped-b8-p16384"]
    rep = _check(parity.run(w, steps=48, lbs=[(0, 0), (23, 7)], device_inputs=True,
                            check_codes_every=16))
    assert rep.stats["tokens_evicted"] > 0


def test_gptoss_longest_context_sampled():
    # the largest kept context of the suite (N_low = 8192 tokens): the output
    # error of the INT8 path must stay well inside the 1e-3 tolerance
    w = wl.ALL["gptoss20b-shaped-b8-p32768"]
    rep = _check(parity.run(w, steps=24, lbs=[(0, 0), (23, 7)], device_inputs=True,
                            check_codes_every=12))
    assert rep.max_out_err < 5e-4
