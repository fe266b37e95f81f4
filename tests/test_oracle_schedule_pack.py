"""Pins of the oracle's S2 (confidence), S3 (scheduler), cost table and S4 (packing).

- confidence: which features enter z (h_k and W1[x_{k-1}] with x_0 = anchor), sigmoid
  special values, STS order preservation, survival is a non-increasing running product;
- scheduler: equals exhaustive search over every prefix-length assignment (exact rational
  arithmetic) -- always for GLOBAL_ARGMAX, and for EARLY_STOP whenever Theta(K) is
  unimodal; admitted sets are contiguous prefixes; tie order;
- cost table: running-max monotone forcing and the 121 -> 128 graph-tier staircase;
- packing: the 121 -> 128 example, sum n_r = bs + K, the static layout, pad rows."""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- confidence

def _conf_inputs(bs=3, gamma=4, d=5, r=3, V=9, seed=0):
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(bs, gamma, d)).astype(np.float32)
    W1 = rng.normal(size=(V, r)).astype(np.float32)
    anchor = rng.integers(0, V, size=bs).astype(np.int32)
    tokens = rng.integers(0, V, size=(bs, gamma)).astype(np.int32)
    return h, W1, anchor, tokens


def test_confidence_feature_indexing():
    h, W1, anchor, tokens = _conf_inputs()
    bs, gamma, d = h.shape
    r = W1.shape[1]
    T = np.ones(gamma, dtype=np.float32)
    for j in (0, d - 1):
        w = np.zeros(d + r, dtype=np.float32); w[j] = 1.0
        _, _, z = O.confidence(h, W1, anchor, tokens, w, 0.0, T, dtype="f32")
        np.testing.assert_array_equal(z, h[:, :, j].astype(np.float64))
    for i in range(r):
        w = np.zeros(d + r, dtype=np.float32); w[d + i] = 1.0
        _, _, z = O.confidence(h, W1, anchor, tokens, w, 0.0, T, dtype="f32")
        for b in range(bs):
            assert z[b, 0] == W1[anchor[b], i]            # position 1 conditions on the anchor
            for k in range(1, gamma):
                assert z[b, k] == W1[tokens[b, k - 1], i]  # position k+1 on x_k


def test_confidence_special_values():
    h, W1, anchor, tokens = _conf_inputs()
    gamma = h.shape[1]
    w0 = np.zeros(h.shape[2] + W1.shape[1], dtype=np.float32)
    c, a, _ = O.confidence(h, W1, anchor, tokens, w0, 0.0, np.ones(gamma), dtype="f32")
    assert np.all(c == 0.5)
    np.testing.assert_array_equal(a, 0.5 ** np.arange(1, gamma + 1)[None, :].repeat(3, 0))
    # bias only: z = b; sigmoid(b / T_k); sigmoid(-x) = 1 - sigmoid(x)
    T = 1.0 + 0.1 * np.arange(1, gamma + 1)
    c1, _, _ = O.confidence(h, W1, anchor, tokens, w0, 2.0, T, dtype="f32")
    c2, _, _ = O.confidence(h, W1, anchor, tokens, w0, -2.0, T, dtype="f32")
    np.testing.assert_allclose(c1 + c2, 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(c1[0]) < 0)  # larger T_k pulls a positive logit towards 1/2


def test_sts_preserves_rank_and_survival_is_monotone():
    wl = I.WORKLOADS["tiny_fp32"].with_(bs=40)
    x = I.make_host_inputs(wl, with_target=False)
    tokens = I.random_tokens(wl.bs, wl.gamma, wl.V, 1)
    c, a, z = O.confidence(x["h"], x["W1"], x["anchor"], tokens, x["w"], 0.0, x["sts_T"], dtype="f32")
    for k in range(wl.gamma):
        np.testing.assert_array_equal(np.argsort(z[:, k], kind="stable"), np.argsort(c[:, k], kind="stable"))
    assert np.all(np.diff(a, axis=1) <= 0)
    np.testing.assert_allclose(a[:, 1:] / a[:, :-1], c[:, 1:], rtol=1e-12)
    np.testing.assert_array_equal(a[:, 0], c[:, 0])


# ---------------------------------------------------------------- cost table

def test_sps_monotone_forcing_and_tier_staircase():
    g = json.load(open(os.path.join(GOLDEN, "tier_padding.json")))
    tiers = list(range(g["tiers_every"], g["tier_max"] + 1, g["tiers_every"]))
    rng = np.random.default_rng(0)
    T = 5.0 + 0.01 * np.arange(g["tier_max"] + 1) + rng.normal(0, 0.02, g["tier_max"] + 1)  # noisy profile
    sps = O.build_sps(T, tiers)
    assert np.all(np.diff(sps) <= 0)  # non-increasing after forcing
    for case in g["cases"]:
        assert O.tier_of(case["total"], tiers) == case["tier"]
        assert sps[case["total"]] == sps[case["tier"]] == 1.0 / np.maximum.accumulate(T)[case["tier"]]
    # a table longer than the last tier: totals beyond it are never admitted
    sps2 = O.build_sps(np.ones(40), [8, 16, 24])
    assert np.all(sps2[25:] == 0) and sps2[24] == 1.0
    # no tiers: every total is its own graph
    np.testing.assert_array_equal(O.build_sps(np.array([1.0, 3.0, 2.0]), []), [1.0, 1 / 3, 1 / 3])


# ---------------------------------------------------------------- scheduler

def _exhaustive(a: np.ndarray, sps: np.ndarray):
    """Best Theta over every assignment of prefix lengths, exact rational arithmetic."""
    bs, gamma = a.shape
    af = [[Fraction(float(a[r, j])) for j in range(gamma)] for r in range(bs)]
    prefix = [[sum(af[r][:l], Fraction(0)) for l in range(gamma + 1)] for r in range(bs)]
    best, best_l = None, None
    for ls in itertools.product(range(gamma + 1), repeat=bs):
        M = bs + sum(ls)
        if M >= len(sps):
            continue
        th = (bs + sum(prefix[r][ls[r]] for r in range(bs))) * Fraction(float(sps[M]))
        if best is None or th > best:
            best, best_l = th, ls
    return best, best_l


def _random_case(bs, gamma, seed, steep=False):
    a = I.random_survival(bs, gamma, seed)
    rng = np.random.default_rng(seed + 1000)
    m_max = bs * (gamma + 1)
    base = 1.0 + rng.random() * 3.0
    slope = rng.random() * (0.9 if steep else 0.2)
    noise = 0.0 if seed >= 12 else 0.01
    T = base + slope * np.arange(m_max + 1) + rng.normal(0, noise, m_max + 1)
    step = 1 if seed >= 12 else int(rng.integers(1, 4))   # seeds >= 12: smooth, unimodal tables
    tiers = list(range(step, m_max, step)) + [m_max]
    return a, O.build_sps(T, tiers)


@pytest.mark.parametrize("seed", range(18))
def test_scheduler_equals_exhaustive_search(seed):
    bs, gamma = (3, 5) if seed % 2 else (4, 4)
    a, sps = _random_case(bs, gamma, seed, steep=seed % 3 == 0)
    best, best_l = _exhaustive(a, sps)
    win, K, th, theta = O.schedule(a, sps, O.GLOBAL_ARGMAX)
    # the greedy optimum reaches the exhaustive optimum up to the 2^-40 fixed-point quantum
    exact_greedy = (bs + sum(Fraction(float(a[r, j])) for r in range(bs) for j in range(win[r]))) \
        * Fraction(float(sps[bs + K]))
    assert abs(float(exact_greedy - best)) <= bs * gamma * 2.0 ** -40 * float(sps.max()) + 1e-15
    if abs(float(best)) > 0 and sorted(theta)[-1] - sorted(theta)[-2] > 1e-9:
        assert tuple(int(v) for v in win) == tuple(best_l)
    # early stop is the same whenever Theta(K) is unimodal
    d = np.sign(np.diff(theta))
    unimodal = not np.any((d[1:] > 0) & (d[:-1] <= 0))
    win2, K2, _, _ = O.schedule(a, sps, O.EARLY_STOP)
    if unimodal:
        assert K2 == K and np.array_equal(win2, win)
    else:
        assert K2 <= K


def test_scheduler_windows_are_contiguous_prefixes_and_top_k():
    a, sps = _random_case(16, 7, 77)
    win, K, _, _ = O.schedule(a, sps, O.GLOBAL_ARGMAX)
    assert win.sum() == K and np.all(win <= 7)
    admitted = np.concatenate([a[r, :win[r]] for r in range(16)])
    rejected = np.concatenate([a[r, win[r]:] for r in range(16)])
    if admitted.size and rejected.size:
        assert admitted.min() >= rejected.max()


def test_scheduler_tie_order_and_fixed_point():
    a = np.array([[0.5, 0.5, 0.25], [0.5, 0.25, 0.25]], dtype=np.float32)
    sps = np.array([1.0, 1.0, 1.0, 1.0, 0.9, 0.85, 0.6, 0.5, 0.1])
    win, K, th, theta = O.schedule(a, sps, O.EARLY_STOP)
    # Theta(0)=2*1.0, Theta(1)=2.5*1.0, Theta(2)=3.0*0.9=2.7, Theta(3)=3.5*0.85=2.975,
    # Theta(4)=3.75*0.6=2.25 -> stop at K=3: slots (0,0), (0,1), (1,0) by the tie order
    np.testing.assert_array_equal(theta[:5], [2.0, 2.5, 2.7, 3.5 * 0.85, 3.75 * 0.6])
    assert K == 3 and list(win) == [2, 1] and th == 3.5 * 0.85
    # fixed-point survival sums: tiny values below 2^-40 do not count
    a2 = np.array([[2.0 ** -41, 0.0]], dtype=np.float32)
    _, _, _, th2 = O.schedule(a2, np.ones(4), O.GLOBAL_ARGMAX)
    assert th2[1] == 1.0


def test_scheduler_zero_admission_when_table_is_steep():
    a = np.full((3, 4), 0.9, dtype=np.float32)
    a = np.cumprod(a, axis=1).astype(np.float32)
    sps = np.concatenate([np.ones(4), np.full(20, 0.01)])
    win, K, th, _ = O.schedule(a, sps, O.EARLY_STOP)
    assert K == 0 and th == 3.0 and not win.any()


# ---------------------------------------------------------------- packing

def test_pack_121_to_128():
    g = json.load(open(os.path.join(GOLDEN, "tier_padding.json")))
    tiers = list(range(g["tiers_every"], g["tier_max"] + 1, g["tiers_every"]))
    bs, gamma = 20, 7
    rng = np.random.default_rng(1)
    win = np.full(bs, 5, dtype=np.int32)
    win[:1] = 0
    win[1:7] = 6  # 1 + 6*7 + 13*6 = 121 packed tokens
    assert int(np.sum(win + 1)) == 121
    tokens = rng.integers(0, 100, size=(bs, gamma)).astype(np.int32)
    anchor = rng.integers(0, 100, size=bs).astype(np.int32)
    cu, ids, req, pos, padded = O.pack(win, anchor, tokens, tiers, cap=512)
    assert cu[-1] == 121 and padded == 128
    assert np.all(ids[121:128] == -1) and np.all(req[121:128] == -1) and np.all(pos[121:128] == -1)


def test_pack_layout_and_static():
    bs, gamma = 6, 4
    rng = np.random.default_rng(2)
    tokens = rng.integers(0, 50, size=(bs, gamma)).astype(np.int32)
    anchor = rng.integers(0, 50, size=bs).astype(np.int32)
    win = I.random_windows(bs, gamma, 3)
    cu, ids, req, pos, padded = O.pack(win, anchor, tokens, [], cap=64)
    assert padded == bs + win.sum() == cu[-1]
    for r in range(bs):
        assert cu[r + 1] - cu[r] == win[r] + 1
        assert ids[cu[r]] == anchor[r] and pos[cu[r]] == 0
        np.testing.assert_array_equal(ids[cu[r] + 1:cu[r + 1]], tokens[r, :win[r]])
        assert np.all(req[cu[r]:cu[r + 1]] == r)
    cu_s, ids_s, _, _, padded_s = O.pack(None, anchor, tokens, [], cap=64)
    np.testing.assert_array_equal(cu_s, np.arange(bs + 1) * (gamma + 1))
    # the static layout of the bs=256, gamma=7 workload fills the largest capture exactly
    c = json.load(open(os.path.join(GOLDEN, "page_constants.json")))["max_capture"]
    wl = I.WORKLOADS["mixed_bs256"]
    assert (wl.gamma + 1) * wl.bs == c["value"] == I.tiers_for(wl)[-1]


def test_pack_errors():
    tokens = np.zeros((2, 3), dtype=np.int32)
    with pytest.raises(ValueError):
        O.pack(np.array([3, 3]), np.zeros(2, np.int32), tokens, [4, 6], cap=16)   # M = 8 > 6
    with pytest.raises(ValueError):
        O.pack(np.array([1, 1]), np.zeros(2, np.int32), tokens, [4, 8], cap=3)    # tier 4 > cap


def test_scheduler_does_not_admit_a_slot_with_zero_gain():
    # Theta(0) = 1 * 1.5 = 1.5 and Theta(1) = (1 + 0.5) * 1.0 = 1.5: admitting the slot does
    # not raise the expected throughput, so it is not admitted (positive expected gain only)
    a = np.array([[0.5]], dtype=np.float32)
    sps = np.array([9.0, 1.5, 1.0])
    for mode in (O.EARLY_STOP, O.GLOBAL_ARGMAX):
        win, K, th, theta = O.schedule(a, sps, mode)
        assert theta[0] == theta[1] == 1.5
        assert K == 0 and win[0] == 0


def test_pruning_is_a_large_batch_effect():
    """[SGLANG, "A preliminary look at dynamic vs static scheduling", Fig. 3]: at batch 1 the
    verify step barely slows with more tokens, so pruning saves little; as concurrency rises the
    dynamic budget prunes, and (two workloads of different acceptance) more so where acceptance
    is low.  With the sweep's cost curve (5 ms + 0.01 ms per token, graph tiers every 16) the
    global search admits every slot at bs 1, and its admitted fraction falls with the batch and
    with the acceptance level."""
    fracs = {"high": [], "low": []}
    for bs in I.DSV4_BATCHES:
        wl = I.dsv4(bs)
        sps = O.build_sps(I.cost_curve_ms(wl), I.tiers_for(wl))
        for name, cmean in (("high", 0.9), ("low", 0.6)):
            rng = np.random.default_rng(bs)
            c = np.clip(rng.normal(cmean, 0.05, (bs, wl.gamma)), 0.01, 0.999).astype(np.float32)
            a = np.cumprod(c, axis=1).astype(np.float32)
            _, K, _, _ = O.schedule(a, sps, O.GLOBAL_ARGMAX)
            fracs[name].append(K / (bs * wl.gamma))
    for name in fracs:
        assert fracs[name][0] == 1.0                                   # bs 1: nothing pruned
        assert all(x >= y for x, y in zip(fracs[name], fracs[name][1:]))  # more pruning with load
    assert fracs["high"][-1] > 0.75 and fracs["low"][-1] < 0.35        # bs 256
    assert all(lo <= hi for lo, hi in zip(fracs["low"], fracs["high"]))
    assert fracs["low"][-1] < fracs["high"][-1] - 0.4
