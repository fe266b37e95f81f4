"""Pins of the oracle's samplers and of S1 (Markov block draft).

- the two-level Gumbel sampler draws exactly from softmax (chi-square, ragged chunks);
- the inverse-CDF step takes hand-computed ids on boundary and zero-weight cases, and the map
  u -> id partitions (0, 1) into intervals of length w_j / S (brute force over a fine u grid);
- the two-level chunk + inverse-CDF sampler of the draft draws exactly from softmax, its chunk
  marginal is the chunk mass, and its level-2 uniform is the element purpose's word 0;
- Markov logits equal a brute-force triple loop;
- the drafted joint distribution of (x_1, x_2) is p_1(x_1) p_2(x_2 | x_1) with the bias of
  position 2 taken from x_1 (catches an off-by-one in the conditioning token);
- temperature divides the logits; temperature 0 is the argmax."""
import numpy as np
from scipy import stats
from scipy.special import logsumexp as sp_lse, softmax

from oracle import dspark_oracle as O


def _chi2_ok(counts, probs, pmin=1e-4):
    counts = np.asarray(counts, dtype=np.float64)
    exp = probs * counts.sum()
    keep = exp > 0
    return stats.chisquare(counts[keep], exp[keep] * counts[keep].sum() / exp[keep].sum()).pvalue > pmin


def test_two_level_sampler_matches_softmax_with_ragged_chunks():
    rng = np.random.default_rng(3)
    logw = rng.normal(0, 1.5, size=13)
    logw[5] = -np.inf  # never drawn
    p = softmax(np.where(np.isfinite(logw), logw, -1e300))
    counts = np.zeros(13)
    for s in range(30000):
        v, _ = O.two_level_gumbel(logw, 9, s, 0, 1, O.P_DRAFT_CHUNK, O.P_DRAFT_ELEM, chunk=4)
        counts[v] += 1
    assert counts[5] == 0
    assert _chi2_ok(counts, p)


def test_two_level_sampler_chunk_marginal_is_chunk_mass():
    rng = np.random.default_rng(4)
    logw = rng.normal(0, 2.0, size=40)
    chunk = 8
    p = softmax(logw)
    mass = p.reshape(5, 8).sum(axis=1)
    counts = np.zeros(5)
    for s in range(20000):
        v, _ = O.two_level_gumbel(logw, 1, s, 3, 2, O.P_DECIDE_CHUNK, O.P_DECIDE_ELEM, chunk=chunk)
        counts[v // chunk] += 1
    assert _chi2_ok(counts, mass)
    np.testing.assert_allclose(np.exp(O.chunk_log_mass(logw, chunk)), np.exp(logw).reshape(5, 8).sum(1), rtol=1e-12)


def test_inverse_cdf_by_hand():
    # w = [1, 1, 2]: partial sums 1, 2, 4 (S = 4); the first j with C_j > u S
    w = [1.0, 1.0, 2.0]
    assert O.inverse_cdf(w, 0.1)[0] == 0      # u S = 0.4 < 1
    assert O.inverse_cdf(w, 0.25)[0] == 1     # u S = 1 = C_0: not > , so the next id
    assert O.inverse_cdf(w, 0.3)[0] == 1      # 1.2
    assert O.inverse_cdf(w, 0.5)[0] == 2      # 2 = C_1
    assert O.inverse_cdf(w, 0.99)[0] == 2
    j, m = O.inverse_cdf(w, 0.3)
    assert abs(m - 0.05) < 1e-12              # min(1.2 - 1, 2 - 1.2) / 4
    # zero weights are never drawn
    z = [0.0, 1.0, 0.0, 1.0]
    assert O.inverse_cdf(z, 0.2)[0] == 1 and O.inverse_cdf(z, 0.7)[0] == 3
    assert O.inverse_cdf([0.0, 0.0, 5.0], 0.01)[0] == 2


def test_inverse_cdf_partitions_the_unit_interval():
    rng = np.random.default_rng(12)
    w = rng.exponential(size=9)
    w[4] = 0.0
    n = 200_000
    us = (np.arange(n) + 0.5) / n
    ids = np.array([O.inverse_cdf(w, u)[0] for u in us])
    assert np.all(np.diff(ids) >= 0)          # monotone in u
    frac = np.bincount(ids, minlength=9) / n
    np.testing.assert_allclose(frac, w / w.sum(), atol=2.0 / n)


def test_chunk_cdf_sampler_matches_softmax_with_ragged_chunks():
    rng = np.random.default_rng(13)
    logw = rng.normal(0, 1.5, size=13)
    logw[6] = -np.inf
    p = softmax(np.where(np.isfinite(logw), logw, -1e300))
    counts = np.zeros(13)
    for s in range(30000):
        v, _ = O.two_level_cdf(logw, 9, s, 0, 1, O.P_DRAFT_CHUNK, O.P_DRAFT_ELEM, chunk=4)
        counts[v] += 1
    assert counts[6] == 0
    assert _chi2_ok(counts, p)


def test_chunk_cdf_sampler_levels():
    rng = np.random.default_rng(14)
    logw = rng.normal(0, 2.0, size=40)
    chunk = 8
    mass = softmax(logw).reshape(5, 8).sum(axis=1)
    counts = np.zeros(5)
    for s in range(20000):
        v, _ = O.two_level_cdf(logw, 2, s, 1, 3, O.P_DRAFT_CHUNK, O.P_DRAFT_ELEM, chunk=chunk)
        counts[v // chunk] += 1
    assert _chi2_ok(counts, mass)
    # inside the drawn chunk, the id is the inverse CDF of the element purpose's word 0
    for s in range(50):
        v, _ = O.two_level_cdf(logw, 2, s, 1, 3, O.P_DRAFT_CHUNK, O.P_DRAFT_ELEM, chunk=chunk)
        c = v // chunk
        u = O.uniform(2, s, O.P_DRAFT_ELEM, 1, 3, np.array([0]))[0]
        seg = logw[c * chunk:(c + 1) * chunk]
        p_in = np.exp(seg - seg.max())
        edges = np.concatenate([[0.0], np.cumsum(p_in)]) / p_in.sum()
        assert edges[v % chunk] <= u < edges[v % chunk + 1]


def test_markov_logits_brute_force():
    rng = np.random.default_rng(5)
    bs, V, r = 3, 11, 4
    U = rng.normal(size=(bs, V))
    W1 = rng.normal(size=(V, r))
    W2t = rng.normal(size=(V, r))
    x = np.array([2, 10, 0])
    got = O.markov_logits(U, W1, W2t, x)
    for b in range(bs):
        for v in range(V):
            acc = U[b, v]
            for i in range(r):
                acc += W1[x[b], i] * W2t[v, i]
            assert abs(got[b, v] - acc) < 1e-12


def _tiny_draft_inputs(V=6, r=3, gamma=2, seed=0):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 1.0, size=(1, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.8, size=(V, r)).astype(np.float32)
    W2t = rng.normal(0, 0.8, size=(V, r)).astype(np.float32)
    return U, W1, W2t


def test_draft_joint_distribution_of_first_two_tokens():
    V = 6
    U, W1, W2t = _tiny_draft_inputs(V=V)
    anchor = np.array([4], dtype=np.int32)
    U64, W164, W2t64 = (a.astype(np.float64) for a in (U, W1, W2t))
    p1 = softmax(U64[0, 0] + W164[4] @ W2t64.T)
    joint = np.zeros((V, V))
    for a in range(V):
        joint[a] = p1[a] * softmax(U64[0, 1] + W164[a] @ W2t64.T)
    counts = np.zeros((V, V))
    for s in range(12000):
        tok, lx, lse, _ = O.draft_block(U, W1, W2t, anchor, 1.0, 21, s, dtype="f32", chunk=4)
        counts[tok[0, 0], tok[0, 1]] += 1
    assert _chi2_ok(counts.ravel(), joint.ravel())


def test_draft_outputs_logit_and_lse():
    U, W1, W2t = _tiny_draft_inputs(V=300, r=5, gamma=3, seed=2)
    anchor = np.array([17], dtype=np.int32)
    tau = 0.7
    tok, lx, lse, _ = O.draft_block(U, W1, W2t, anchor, tau, 5, 0, dtype="f32")
    prev = 17
    for k in range(3):
        ell = U[0, k].astype(np.float64) + W1[prev].astype(np.float64) @ W2t.astype(np.float64).T
        assert abs(lx[0, k] - ell[tok[0, k]] / tau) < 1e-12
        assert abs(lse[0, k] - sp_lse(ell / tau)) < 1e-12
        prev = tok[0, k]


def test_draft_temperature_scales_logits():
    V = 5
    U, W1, W2t = _tiny_draft_inputs(V=V, gamma=1, seed=3)
    anchor = np.array([1], dtype=np.int32)
    ell = U[0, 0].astype(np.float64) + W1[1].astype(np.float64) @ W2t.astype(np.float64).T
    counts = np.zeros(V)
    for s in range(15000):
        tok, *_ = O.draft_block(U, W1, W2t, anchor, 0.5, 2, s, dtype="f32")
        counts[tok[0, 0]] += 1
    assert _chi2_ok(counts, softmax(ell / 0.5))


def test_draft_greedy_is_argmax():
    U, W1, W2t = _tiny_draft_inputs(V=50, r=4, gamma=4, seed=6)
    U = np.repeat(U, 3, axis=0)
    anchor = np.array([0, 7, 49], dtype=np.int32)
    tok, lx, lse, _ = O.draft_block(U, W1, W2t, anchor, 0.0, 1, 0, dtype="f32")
    for b in range(3):
        prev = anchor[b]
        for k in range(4):
            ell = U[b, k].astype(np.float64) + W1[prev].astype(np.float64) @ W2t.astype(np.float64).T
            assert tok[b, k] == int(np.argmax(ell))
            assert lx[b, k] == ell.max() and lse[b, k] == 0.0
            prev = tok[b, k]


def test_greedy_ties_go_to_lowest_index():
    U = np.zeros((1, 1, 8), dtype=np.float32)
    U[0, 0, [2, 5, 7]] = 3.0
    W1 = np.zeros((8, 2), dtype=np.float32)
    W2t = np.zeros((8, 2), dtype=np.float32)
    tok, *_ = O.draft_block(U, W1, W2t, np.array([0], dtype=np.int32), 0.0, 0, 0, dtype="f32")
    assert tok[0, 0] == 2
