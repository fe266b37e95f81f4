"""Pins of the oracle's observability records and its sequential temperature scaling fit.

- ECE: hand-computed cases, the closed form |p - c| for a constant score, and agreement with
  an independent library routine (scikit-learn's calibration curve, bin-weighted);
- prefix outcomes: hand cases with and without a ceiling (what compact can and cannot see);
- observe / report: sums, histograms, utilisation = accepted / ceiling by hand; cap-accept's
  ceiling recovers the labels compact hides;
- STS fit: recovers the temperatures of a known law, leaves a calibrated law at T = 1,
  preserves each position's order, and its per-position ECE is the grid minimum."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import inputs as I


def test_ece_by_hand():
    e, cnt, lab, sc = O.ece(np.float32([0.1, 0.4, 0.6, 0.9]), [0, 0, 1, 1], 10)
    # one score per bin: (0.1 + 0.4 + 0.4 + 0.1) / 4
    assert e == pytest.approx(0.25, abs=1e-7)
    assert list(np.nonzero(cnt)[0]) == [1, 4, 6, 9]
    e2, cnt2, _, _ = O.ece(np.float32([0.1, 0.4, 0.6, 0.9]), [0, 0, 1, 1], 2)
    assert list(cnt2) == [2, 2] and e2 == pytest.approx(0.25, abs=1e-7)   # |0 - 0.5| + |2 - 1.5|
    e3, _, _, _ = O.ece(np.float32([0.3, 0.3, 0.3, 0.3]), [1, 1, 1, 0], 10)
    assert e3 == pytest.approx(0.45, abs=1e-7)                            # |3/4 - 0.3|
    # bin edges: 1.0 falls in the last bin, 0 in the first
    _, cnt4, _, _ = O.ece(np.float32([0.0, 1.0, 0.5]), [0, 1, 1], 4)
    assert list(cnt4) == [1, 0, 1, 1]
    assert O.ece(np.zeros(0, np.float32), [], 10)[0] == 0.0


def test_ece_closed_form_constant_score():
    rng = np.random.default_rng(0)
    for c, p in [(0.2, 0.5), (0.9, 0.9), (0.55, 0.1)]:
        y = (rng.random(5000) < p).astype(np.int64)
        e, _, _, _ = O.ece(np.full(5000, c, np.float32), y, 15)
        assert e == pytest.approx(abs(y.mean() - np.float32(c)), abs=1e-9)


def test_ece_equals_library_calibration_curve():
    calib = pytest.importorskip("sklearn.calibration")
    rng = np.random.default_rng(1)
    a = rng.random(4000).astype(np.float32)
    y = (rng.random(4000) < a ** 1.5).astype(np.int64)
    for M in (5, 10, 20):
        prob_true, prob_pred = calib.calibration_curve(y, a, n_bins=M, strategy="uniform")
        counts = np.histogram(a, bins=np.linspace(0, 1, M + 1))[0]
        counts = counts[counts > 0]
        ref = float(np.sum(counts / a.size * np.abs(prob_true - prob_pred)))
        assert O.ece(a, y, M)[0] == pytest.approx(ref, abs=1e-6)


def test_prefix_labels_with_and_without_ceiling():
    # gamma 4; request 0: window 2, accepted 2 (whole window passed; beyond unknown)
    #          request 1: window 3, accepted 1 (rejected at 2: everything after is 0)
    #          request 2: window 0, accepted 0
    lab, known = O.prefix_labels([2, 3, 0], [2, 1, 0], None, 4)
    assert lab.tolist() == [[1, 1, 0, 0], [1, 0, 0, 0], [0, 0, 0, 0]]
    assert known.tolist() == [[True, True, False, False], [True, True, True, True],
                              [False, False, False, False]]
    # the ceiling of a full-block verification settles every position
    lab, known = O.prefix_labels([2, 3, 0], [2, 1, 0], [3, 1, 4], 4)
    assert lab.tolist() == [[1, 1, 1, 0], [1, 0, 0, 0], [1, 1, 1, 1]] and known.all()


def test_observe_and_report_by_hand():
    surv = np.float32([[0.9, 0.5, 0.2], [0.8, 0.7, 0.1]])
    st = O.observe(surv, [2, 3], [2, 1], [3, 1], n_bins=10)
    assert st["sum_window"] == 5 and st["sum_accepted"] == 3 and st["sum_ceiling"] == 4
    assert st["window_hist"][2] == 1 and st["window_hist"][3] == 1
    assert st["ceiling_hist"][1] == 1 and st["ceiling_hist"][3] == 1
    # outcomes: request 0 [1, 1, 1], request 1 [1, 0, 0]
    assert st["pos_count"].tolist() == [2, 2, 2] and st["pos_label"].tolist() == [2, 1, 1]
    rep = O.obs_report(st)
    assert rep["utilisation"] == pytest.approx(3 / 4)
    assert rep["mean_window"] == 2.5 and rep["mean_accepted"] == 1.5 and rep["mean_ceiling"] == 2.0
    # ECE over six scores: |1-0.9| + |1-0.8| + |1-0.5| + |0-0.7| + |1-0.2| + |0-0.1|, each alone in its bin
    assert rep["ece"] == pytest.approx((0.1 + 0.2 + 0.5 + 0.7 + 0.8 + 0.1) / 6, abs=1e-7)
    np.testing.assert_allclose(rep["pos_mean_survival"], [0.85, 0.6, 0.15], rtol=1e-6)


def test_cap_accept_ceiling_recovers_what_compact_hides():
    """Compact sees outcomes only inside the window when the window passes; a ceiling run
    labels every position and counts more of them."""
    rng = np.random.default_rng(3)
    bs, gamma = 64, 7
    surv = I.random_survival(bs, gamma, 9)
    ceiling = rng.integers(0, gamma + 1, bs)
    window = rng.integers(0, gamma + 1, bs)
    acc = np.minimum(ceiling, window)          # what a compact run with these uniforms accepts
    c = O.observe(surv, window, acc, None)
    f = O.observe(surv, window, acc, ceiling)
    assert int(np.sum(f["bin_count"])) == bs * gamma >= int(np.sum(c["bin_count"]))
    # where compact knows the outcome it agrees with the ceiling's
    lab_c, known = O.prefix_labels(window, acc, None, gamma)
    lab_f, _ = O.prefix_labels(window, acc, ceiling, gamma)
    assert np.array_equal(lab_c[known], lab_f[known])


def test_sts_fit_recovers_a_known_law():
    T_true = [1.6, 1.9, 1.3, 2.2, 1.0]
    z, ceiling = I.calibration_steps(40000, 5, T_true, seed=11)
    grid = np.round(np.arange(0.5, 3.01, 0.1), 6)
    T, best, table = O.sts_fit(z, ceiling, grid, n_bins=15)
    for k in range(4):   # the last position has few surviving prefixes; looser there
        assert abs(T[k] - T_true[k]) <= 0.2 + 1e-9, (k, T[k], T_true[k])
    assert abs(T[4] - T_true[4]) <= 0.5
    for k in range(5):
        assert best[k] == table[k].min() and T[k] == grid[int(np.argmin(table[k]))]
    # fitted survival is better calibrated than the raw (T = 1) one at every position
    _, best_raw, _ = O.sts_fit(z, ceiling, [1.0], n_bins=15)
    assert np.all(best <= best_raw + 1e-12) and best.mean() < 0.5 * best_raw.mean()


def test_sts_fit_keeps_a_calibrated_law_and_order():
    z, ceiling = I.calibration_steps(30000, 3, [1.0, 1.0, 1.0], seed=12)
    grid = np.round(np.arange(0.5, 2.01, 0.1), 6)
    T, best, _ = O.sts_fit(z, ceiling, grid, n_bins=10)
    assert np.all(np.abs(T - 1.0) <= 0.2 + 1e-9)
    assert np.all(best < 0.02)
    # each position's scores keep the order of its logits
    c = 1.0 / (1.0 + np.exp(-z[:, 0].astype(np.float64) / T[0]))
    assert np.array_equal(np.argsort(c, kind="stable"), np.argsort(z[:, 0].astype(np.float64), kind="stable"))


def test_sts_fit_uses_the_prefix_outcome_not_the_position_outcome():
    """Planted-mistake guard: labelling position k by [ceiling > k] (off by one) or by the
    position alone would change the fit on this hand case."""
    z = np.float32([[3.0, 0.0], [3.0, 0.0], [-3.0, 0.0], [-3.0, 0.0]])
    ceiling = np.int32([2, 1, 0, 0])
    T, best, table = O.sts_fit(z, ceiling, [0.5, 1.0, 100.0], n_bins=10)
    # position 1 outcomes [1, 1, 0, 0]: the sharpest grid value fits best
    assert T[0] == 0.5
    # position 2: survival = s1 * 0.5 with outcomes [1, 0, 0, 0]
    s1 = 1.0 / (1.0 + np.exp(-np.array([3.0, 3.0, -3.0, -3.0]) / 0.5))
    a2 = (s1 * 0.5).astype(np.float32)
    assert table[1, 0] == pytest.approx(O.ece(a2, [1, 0, 0, 0], 10)[0], abs=1e-12)
