"""The seeded input generator against the recipe of each workload.

The workloads stand in for the pages' evaluation settings (Qwen3-4B- and DeepSeek-V4-shaped
vocabularies and widths, a mixed-difficulty batch, a long block): these tests fix their shapes,
random laws, noise groups, cost curves and graph tiers, so that a changed generator cannot
silently change what the parity tests and the benchmark run on.  Laws are checked on reduced
sizes (the generator's laws do not depend on the sizes) against sampling error bounds."""
import math

import numpy as np
import pytest

from speculative_decoding_draft_markov_gb300 import inputs as I

# name -> (bs, gamma, V, r, d, dtype, U std, W std, noise stds, seed, tier step, largest tier)
RECIPE = {
    "tiny_fp32": (4, 7, 1024, 32, 64, "f32", math.sqrt(2.0), 0.1, (0.5, 1.0, 1.5, 2.0), 0, 0, 64),
    "qwen3_4b": (64, 7, 151936, 256, 2560, "bf16", 3.0, 0.05, (1.0,), 1, 16, 512),
    "mixed_bs256": (256, 7, 151936, 256, 4096, "bf16", 3.0, 0.05, (0.5, 1.0, 2.0), 2, 64, 2048),
    "dsv4_sweep": (256, 5, 129280, 256, 7168, "bf16", 3.0, 0.05, (1.0,), 3, 16, 1536),
    "long_block": (128, 15, 151936, 256, 4096, "bf16", 3.0, 0.05, (1.25,), 4, 128, 2048),
}


@pytest.mark.parametrize("name", list(RECIPE))
def test_workload_fields(name):
    wl = I.WORKLOADS[name]
    bs, gamma, V, r, d, dtype, u_std, w_std, sigmas, seed, step, tmax = RECIPE[name]
    assert (wl.bs, wl.gamma, wl.V, wl.r, wl.d, wl.dtype, wl.seed) == (bs, gamma, V, r, d, dtype, seed)
    assert wl.u_std == pytest.approx(u_std) and wl.w_std == pytest.approx(w_std)
    assert tuple(wl.sigmas) == sigmas
    assert wl.temperature == 1.0
    assert (wl.tier_step, wl.tier_max) == (step, tmax)


def test_dsv4_sweep_points():
    """Batch sizes 1 .. 256, tiers padded up to (gamma + 1) bs."""
    assert I.DSV4_BATCHES == (1, 8, 32, 128, 256)
    for bs in I.DSV4_BATCHES:
        wl = I.dsv4(bs)
        assert wl.bs == bs and wl.gamma == 5 and wl.V == 129280
        t = I.tiers_for(wl)
        assert t[-1] == 6 * bs and np.all(np.diff(t) > 0) and np.all(t > 0)


@pytest.mark.parametrize("name", list(RECIPE))
def test_tiers_and_cost_curve(name):
    wl = I.WORKLOADS[name]
    t = I.tiers_for(wl)
    T = I.cost_curve_ms(wl)
    assert T.shape == (wl.tier_max + 1,)
    assert np.all(np.diff(T) > 0)  # a monotone profile
    if wl.tier_step == 0:
        assert t.size == 0
        np.testing.assert_allclose(1.0 / T, 1.0 / (1.0 + 0.002 * np.arange(wl.tier_max + 1)))  # SPS = 1/(1+0.002M)
    else:
        np.testing.assert_array_equal(t, np.arange(wl.tier_step, wl.tier_max + 1, wl.tier_step))
        assert T[0] == 5.0 and T[100] == pytest.approx(6.0)  # 5 ms plus a per-token slope


def _within(sample: np.ndarray, std: float, n_sigma: float = 5.0):
    """Sample std within n_sigma standard errors of std (normal law: se(s) ~ std / sqrt(2n)), and
    the mean within n_sigma std / sqrt(n)."""
    n = sample.size
    assert abs(sample.mean()) < n_sigma * std / math.sqrt(n), (sample.mean(), std)
    assert abs(sample.std() - std) < n_sigma * std / math.sqrt(2 * n) + 2e-3 * std, (sample.std(), std)


def _host(wl):
    x = I.make_host_inputs(wl)
    f = (lambda a: np.asarray(a, np.float64)) if wl.dtype == "f32" else (lambda a: I.bf16_bits_to_f32(a).astype(np.float64))
    return x, f


def _torch(wl):
    """The generator the benchmark and the full-size tests use (torch's, here on the CPU)."""
    torch = pytest.importorskip("torch")
    x = I.make_device_inputs(wl, torch.device("cpu"))
    x = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    x["anchor"] = x["anchor"].numpy()
    x["sts_T"] = x["sts_T"].numpy()
    return x, (lambda a: a.float().numpy().astype(np.float64) if isinstance(a, torch.Tensor) else np.asarray(a, np.float64))


@pytest.mark.parametrize("gen", ["numpy", "torch"])
@pytest.mark.parametrize("name", list(RECIPE))
def test_laws_of_the_generated_inputs(name, gen):
    wl = I.WORKLOADS[name]
    small = wl.with_(bs=24, V=4096, d=256)
    x, f = _host(small) if gen == "numpy" else _torch(small)
    U, W1, W2t, h, target = f(x["U"]), f(x["W1"]), f(x["W2t"]), f(x["h"]), f(x["target"])
    assert U.shape == (24, wl.gamma, 4096) and target.shape == (24, wl.gamma + 1, 4096)
    assert W1.shape == W2t.shape == (4096, wl.r) and h.shape == (24, wl.gamma, 256)
    _within(U, wl.u_std)
    _within(W1, wl.w_std)
    _within(W2t, wl.w_std)
    _within(h, 1.0)
    w = x["w"].numpy() if hasattr(x["w"], "numpy") else x["w"]  # float32 in both generators
    _within(np.asarray(w, np.float64), 1.0 / math.sqrt(256 + wl.r), n_sigma=6.0)
    assert x["b"] == 0.0
    np.testing.assert_allclose(x["sts_T"], 1.0 + 0.1 * np.arange(1, wl.gamma + 1), rtol=1e-7)
    assert x["anchor"].min() >= 0 and x["anchor"].max() < 4096
    # target rows 0 .. gamma-1 = U of the scored position + noise (per request group); the bonus
    # row gamma = a fresh base draw + noise.  (In bf16 each target value is rounded once more,
    # by at most 2^-9 of its size: negligible against these noise levels.)
    sig = I.sigma_per_request(24, wl.sigmas)
    for s in sorted(set(sig)):
        grp = sig == s
        _within(target[grp, :wl.gamma] - U[grp], s, n_sigma=6.0)
        _within(target[grp, wl.gamma], math.sqrt(wl.u_std ** 2 + s ** 2), n_sigma=6.0)


def test_noise_groups_are_contiguous_thirds():
    """The mixed-difficulty batch: three contiguous groups of requests with noise std 0.5, 1, 2."""
    sig = I.sigma_per_request(256, (0.5, 1.0, 2.0))
    assert (sig[:85] == 0.5).all() and (sig[85:170] == 1.0).all() and (sig[170:] == 2.0).all()


def test_generator_is_seeded():
    wl = I.WORKLOADS["qwen3_4b"].with_(bs=3, V=512, d=64)
    a, b = I.make_host_inputs(wl), I.make_host_inputs(wl)
    for k in ("U", "W1", "W2t", "anchor", "target", "h", "w"):
        np.testing.assert_array_equal(a[k], b[k])
    c = I.make_host_inputs(wl.with_(seed=wl.seed + 1))
    assert not np.array_equal(a["U"], c["U"]) and not np.array_equal(a["target"], c["target"])
