"""Pins of the oracle's S5 (rejection-sampling verification).

- Monte-Carlo acceptance of position 1 equals 1 - 1/2 ||p_d - p_t||_1 (the analytic
  per-position acceptance of the technical summary's confidence-head section), and the
  acceptance of position 2 given position 1 equals its exact conditional value;
- the first committed token is distributed as p_t (lossless), also under random windows
  and in cap-accept mode (non-anticipating truncation);
- cap-accept commits bit-identically to compact and its ceiling equals static's count;
- greedy verification accepts exactly the argmax-matching prefix;
- with the draft's logits given explicitly: the same decisions as the recompute path, full
  acceptance when the draft equals the target, and losslessness for a non-Markov draft."""
import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import inputs as I


def _setup(V=16, r=3, gamma=2, reps=200, seed=0, noise=1.0):
    rng = np.random.default_rng(seed)
    U1 = rng.normal(0, 1.2, size=(1, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.7, size=(V, r)).astype(np.float32)
    W2t = rng.normal(0, 0.7, size=(V, r)).astype(np.float32)
    base = np.concatenate([U1, rng.normal(0, 1.2, size=(1, 1, V)).astype(np.float32)], axis=1)
    target1 = (base + rng.normal(0, noise, size=base.shape)).astype(np.float32)
    anchor1 = np.array([int(rng.integers(0, V))], dtype=np.int32)
    U = np.repeat(U1, reps, 0)
    target = np.repeat(target1, reps, 0)
    anchor = np.repeat(anchor1, reps)
    return U, W1, W2t, target, anchor


def _run_step(U, W1, W2t, target, anchor, window, mode, step, tau=1.0, seed=5):
    bs, gamma, V = U.shape
    tok, lx, lse, _ = O.draft_block(U, W1, W2t, anchor, tau, seed, step, dtype="f32")
    pack_win = window if mode == O.COMPACT else None
    cu, ids, req, pos, padded = O.pack(pack_win, anchor, tok, [], cap=bs * (gamma + 1))
    packed = I.gather_packed_target(target, req, pos, padded)
    out, acc, ceil, _ = O.verify(packed, cu, window, mode, anchor, tok, lx, lse, U, W1, W2t,
                                 tau, seed, step, dtype="f32")
    return tok, out, acc, ceil


@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_monte_carlo_acceptance_equals_one_minus_tv(tau):
    """At temperature tau both distributions are the tempered softmaxes: p_d = softmax(l / tau),
    p_t = softmax(t / tau), and the acceptance is 1 - TV between them."""
    U, W1, W2t, target, anchor = _setup()
    bs, gamma, V = U.shape
    f = lambda a: a.astype(np.float64)
    pd1 = softmax((f(U[0, 0]) + f(W1[anchor[0]]) @ f(W2t).T) / tau)
    pt1 = softmax(f(target[0, 0]) / tau)
    pt2 = softmax(f(target[0, 1]) / tau)
    acc1 = 1.0 - 0.5 * np.abs(pd1 - pt1).sum()
    # P(accept 2 | accept 1) = sum_x1 min(pd1, pt1)(x1) / acc1 * (1 - TV(pd2(.|x1), pt2))
    cond = 0.0
    for x1 in range(V):
        pd2 = softmax((f(U[0, 1]) + f(W1[x1]) @ f(W2t).T) / tau)
        cond += min(pd1[x1], pt1[x1]) / acc1 * (1.0 - 0.5 * np.abs(pd2 - pt2).sum())
    window = np.full(bs, gamma, dtype=np.int32)
    n1 = n2 = n = 0
    for step in range(60):
        _, _, acc, _ = _run_step(U, W1, W2t, target, anchor, window, O.COMPACT, step, tau=tau)
        n += bs
        n1 += int(np.sum(acc >= 1))
        n2 += int(np.sum(acc >= 2))
    p1 = n1 / n
    assert abs(p1 - acc1) < 4 * np.sqrt(acc1 * (1 - acc1) / n)
    p21 = n2 / n1
    assert abs(p21 - cond) < 4 * np.sqrt(cond * (1 - cond) / n1)


@pytest.mark.parametrize("tau", [1.0, 0.7])
@pytest.mark.parametrize("mode", ["compact_random", "static", "cap_accept"])
def test_first_committed_token_is_target_distributed(mode, tau):
    """Lossless at any temperature: the first committed token follows softmax(t / tau) -- through
    an accepted draft token, the residual after a rejection, or the bonus after an empty or
    fully accepted window."""
    U, W1, W2t, target, anchor = _setup(seed=1, noise=1.5)
    bs, gamma, V = U.shape
    pt1 = softmax(target[0, 0].astype(np.float64) / tau)
    counts = np.zeros(V)
    for step in range(60):
        window = I.random_windows(bs, gamma, 1000 + step)
        m = {"compact_random": O.COMPACT, "static": O.STATIC, "cap_accept": O.CAP_ACCEPT}[mode]
        _, out, _, _ = _run_step(U, W1, W2t, target, anchor, window, m, step, tau=tau)
        np.add.at(counts, out[:, 0], 1)
    assert stats.chisquare(counts, pt1 * counts.sum()).pvalue > 1e-4


@pytest.mark.parametrize("tau", [0.7, 1.6])
def test_second_committed_token_given_first_accepted_is_target_distributed(tau):
    """Given that x_1 was accepted, the next committed token follows the target's row 2 at the
    same temperature (accepted x_2, residual at position 2, or the bonus of a one-token window),
    so every position's tempering is exercised."""
    U, W1, W2t, target, anchor = _setup(seed=6, noise=0.8, reps=300)
    bs, gamma, V = U.shape
    pt2 = softmax(target[0, 1].astype(np.float64) / tau)
    counts = np.zeros(V)
    for step in range(40):
        window = np.where(I.random_windows(bs, gamma, 500 + step) > 0, gamma, 1).astype(np.int32)
        tok, out, acc, _ = _run_step(U, W1, W2t, target, anchor, window, O.COMPACT, step, tau=tau)
        sel = acc >= 1
        np.add.at(counts, out[sel, 1], 1)
    assert counts.sum() > 3000
    assert stats.chisquare(counts, pt2 * counts.sum()).pvalue > 1e-4


def test_cap_accept_commits_like_compact_and_exposes_static_ceiling():
    U, W1, W2t, target, anchor = _setup(V=40, gamma=5, reps=30, seed=3, noise=0.6)
    bs, gamma, V = U.shape
    for step in range(10):
        window = I.random_windows(bs, gamma, 77 + step)
        _, out_c, acc_c, _ = _run_step(U, W1, W2t, target, anchor, window, O.COMPACT, step)
        _, out_a, acc_a, ceil_a = _run_step(U, W1, W2t, target, anchor, window, O.CAP_ACCEPT, step)
        _, out_s, acc_s, _ = _run_step(U, W1, W2t, target, anchor, window, O.STATIC, step)
        np.testing.assert_array_equal(out_a, out_c)
        np.testing.assert_array_equal(acc_a, acc_c)
        np.testing.assert_array_equal(ceil_a, acc_s)
        assert np.all(ceil_a >= acc_a) and np.all(acc_a <= window)


def test_static_equals_compact_with_full_windows():
    U, W1, W2t, target, anchor = _setup(V=40, gamma=4, reps=20, seed=4)
    bs, gamma, V = U.shape
    full = np.full(bs, gamma, dtype=np.int32)
    _, out_c, acc_c, _ = _run_step(U, W1, W2t, target, anchor, full, O.COMPACT, 3)
    _, out_s, acc_s, _ = _run_step(U, W1, W2t, target, anchor, full, O.STATIC, 3)
    np.testing.assert_array_equal(out_c, out_s)
    np.testing.assert_array_equal(acc_c, acc_s)


def test_greedy_accepts_argmax_prefix():
    V, gamma, r = 30, 4, 2
    rng = np.random.default_rng(9)
    U = rng.normal(size=(1, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.3, size=(V, r)).astype(np.float32)
    W2t = rng.normal(0, 0.3, size=(V, r)).astype(np.float32)
    anchor = np.array([3], dtype=np.int32)
    tok, lx, lse, _ = O.draft_block(U, W1, W2t, anchor, 0.0, 0, 0, dtype="f32")
    target = rng.normal(size=(1, gamma + 1, V)).astype(np.float32)
    for k in range(2):                      # positions 1 and 2 agree with the draft
        target[0, k, tok[0, k]] = 10.0
    wrong = (tok[0, 2] + 1) % V             # position 3 disagrees
    target[0, 2, wrong] = 10.0
    target[0, 2, tok[0, 2]] = 9.0
    cu, ids, req, pos, padded = O.pack(None, anchor, tok, [], cap=gamma + 1)
    packed = I.gather_packed_target(target, req, pos, padded)
    out, acc, ceil, _ = O.verify(packed, cu, None, O.STATIC, anchor, tok, lx, lse, U, W1, W2t,
                                 0.0, 0, 0, dtype="f32")
    assert acc[0] == 2 and list(out[0, :3]) == [tok[0, 0], tok[0, 1], wrong] and out[0, 3] == -1
    # everything agrees -> bonus = argmax of the row after the block
    for k in range(gamma):
        target[0, k, tok[0, k]] = 20.0
    packed = I.gather_packed_target(target, req, pos, padded)
    out, acc, _, _ = O.verify(packed, cu, None, O.STATIC, anchor, tok, lx, lse, U, W1, W2t,
                              0.0, 0, 0, dtype="f32")
    assert acc[0] == gamma and out[0, gamma] == int(np.argmax(target[0, gamma]))


def test_verify_rejects_mismatched_packing():
    U, W1, W2t, target, anchor = _setup(V=16, gamma=3, reps=2)
    tok, lx, lse, _ = O.draft_block(U, W1, W2t, anchor, 1.0, 0, 0, dtype="f32")
    cu, ids, req, pos, padded = O.pack(np.array([1, 2]), anchor, tok, [], cap=8)
    packed = I.gather_packed_target(target, req, pos, padded)
    with pytest.raises(ValueError):
        O.verify(packed, cu, np.array([2, 2]), O.COMPACT, anchor, tok, lx, lse, U, W1, W2t,
                 1.0, 0, 0, dtype="f32")


def test_explicit_draft_logits_equal_recomputed_ones():
    """Given the draft's own logits (fp32 of U + W1[x] W2), verify decides as when it recomputes
    them, except where a decision margin is below the fp32 rounding of the logits."""
    U, W1, W2t, target, anchor = _setup(V=40, reps=60, seed=3, noise=1.2)
    bs, gamma, V = U.shape
    for step in range(4):
        tok, lx, lse, _ = O.draft_block(U, W1, W2t, anchor, 1.0, 5, step, dtype="f32")
        f = lambda a: a.astype(np.float64)
        prev = np.concatenate([anchor[:, None], tok[:, :-1]], axis=1)
        D = (f(U) + np.einsum("bkr,vr->bkv", f(W1)[prev], f(W2t))).astype(np.float32)
        window = I.random_windows(bs, gamma, 70 + step)
        cu, ids, req, pos, padded = O.pack(window, anchor, tok, [], cap=bs * (gamma + 1))
        packed = I.gather_packed_target(target, req, pos, padded)
        a = O.verify(packed, cu, window, O.COMPACT, anchor, tok, lx, lse, U, W1, W2t, 1.0, 5, step, dtype="f32")
        b = O.verify(packed, cu, window, O.COMPACT, anchor, tok, lx, lse, None, None, None, 1.0, 5, step,
                     dtype="f32", draft_logits=D)
        sure = np.minimum(a[3], b[3]) > 1e-5
        assert sure.mean() > 0.95
        np.testing.assert_array_equal(a[0][sure], b[0][sure])
        np.testing.assert_array_equal(a[1][sure], b[1][sure])


def test_explicit_draft_equal_to_target_accepts_everything():
    """p_d = p_t (the draft's logits are the target's): every tested token is accepted and the
    extra token is the bonus draw of the next row."""
    rng = np.random.default_rng(9)
    bs, gamma, V = 30, 3, 24
    target = rng.normal(0, 1.5, size=(bs, gamma + 1, V)).astype(np.float32)
    D = target[:, :gamma].copy()
    tok = rng.integers(0, V, size=(bs, gamma)).astype(np.int32)
    anchor = rng.integers(0, V, size=bs).astype(np.int32)
    f = target[:, :gamma].astype(np.float64)
    lse = (np.log(np.exp(f - f.max(-1, keepdims=True)).sum(-1)) + f.max(-1)).astype(np.float32)
    lx = np.take_along_axis(f, tok[..., None].astype(np.int64), -1)[..., 0].astype(np.float32)
    cu, ids, req, pos, padded = O.pack(None, anchor, tok, [], cap=bs * (gamma + 1), gamma=gamma)
    packed = I.gather_packed_target(target, req, pos, padded)
    out, acc, _, _ = O.verify(packed, cu, None, O.STATIC, anchor, tok, lx, lse, None, None, None, 1.0, 2, 0,
                              dtype="f32", draft_logits=D)
    assert (acc == gamma).all()
    np.testing.assert_array_equal(out[:, :gamma], tok)


@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_explicit_draft_logits_first_committed_token_is_target_distributed(tau):
    """Losslessness with an arbitrary draft distribution given as logits (not a Markov head), at
    temperature tau: the draft draws from softmax(D / tau), reports the tempered logit of its
    token and the tempered log-sum-exp, and the first committed token follows softmax(t / tau)
    -- so the residual's p_d must be tempered too."""
    rng = np.random.default_rng(11)
    V, gamma, bs = 12, 1, 400
    t_row = rng.normal(0, 1.3, size=V)
    d_row = rng.normal(0, 1.3, size=V)
    target = np.broadcast_to(np.stack([t_row, rng.normal(0, 1.3, size=V)]).astype(np.float32),
                             (bs, gamma + 1, V)).copy()
    D = np.broadcast_to(d_row.astype(np.float32), (bs, gamma, V)).copy()
    p_d = softmax(d_row / tau)
    dt = d_row / tau
    lse_d = np.float32(np.log(np.exp(dt - dt.max()).sum()) + dt.max())
    counts = np.zeros(V)
    for step in range(40):
        tok = rng.choice(V, size=(bs, gamma), p=p_d).astype(np.int32)
        lx = (D[np.arange(bs)[:, None], np.arange(gamma)[None, :], tok].astype(np.float64) / tau).astype(np.float32)
        lse = np.full((bs, gamma), lse_d, dtype=np.float32)
        anchor = np.zeros(bs, dtype=np.int32)
        cu, ids, req, pos, padded = O.pack(None, anchor, tok, [], cap=bs * (gamma + 1), gamma=gamma)
        packed = I.gather_packed_target(target, req, pos, padded)
        out, _, _, _ = O.verify(packed, cu, None, O.STATIC, anchor, tok, lx, lse, None, None, None, tau, 4, step,
                                dtype="f32", draft_logits=D)
        np.add.at(counts, out[:, 0], 1)
    assert stats.chisquare(counts, softmax(t_row.astype(np.float32).astype(np.float64) / tau) * counts.sum()).pvalue > 1e-4
