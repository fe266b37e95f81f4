"""Pins of the oracle's RNN sequential head (rnn_state_step, rnn_draft_block, verify with the
draft's states).

- bf16 rounding of the state: the oracle's frexp-based round-half-even equals the input
  module's bit-level float32 -> bf16 conversion on float32 values, ties included;
- the gated update against a scalar-loop recurrence written from its definition;
- special cases: a closed gate (g = 0) is the Markov head bit for bit (s_k = W1[x_{k-1}]); an
  open gate (g = 1) keeps s_k = 0, i.e. softmax(U_k) alone;
- the joint law of (x_1, x_2, x_3) equals the exact law from enumerating every prefix with the
  recurrence (chi-square), and position 3's law depends on x_1 as well as x_2 (the state sees
  the whole prefix, unlike the Markov head);
- verify recomputes p_d from the states: a closed gate matches the Markov recompute exactly,
  and the first committed token follows the target (lossless) under the RNN draft."""
import itertools

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import inputs as I


def test_round_bf16_equals_bit_level_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 2000), rng.normal(0, 300, 2000)])
    x = x.astype(np.float32)
    # exact ties of bf16: the low 16 bits of the float32 are 0x8000 (both parities of bit 16)
    ties = (np.arange(1, 2001, dtype=np.uint32) << 16 | np.uint32(0x8000) | np.uint32(0x3F000000)).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, 1.0, -2.5, 65280.0])])
    got = O.round_bf16(x.astype(np.float64))
    ref = I.bf16_bits_to_f32(I.f32_to_bf16_bits(x)).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def _scalar_step(e, s_prev, Wg, bg):
    """The gated update written element by element from its definition."""
    n, r = e.shape
    out = np.zeros((n, r))
    for b in range(n):
        for i in range(r):
            z = bg[i]
            for j in range(r):
                z += e[b, j] * Wg[j, i]
            for j in range(r):
                z += s_prev[b, j] * Wg[r + j, i]
            g = 1.0 / (1.0 + np.exp(-z))
            out[b, i] = g * s_prev[b, i] + (1.0 - g) * e[b, i]
    return out


def test_state_step_equals_scalar_recurrence():
    rng = np.random.default_rng(1)
    n, r = 5, 6
    e, s = rng.normal(0, 0.3, (n, r)), rng.normal(0, 0.3, (n, r))
    Wg, bg = rng.normal(0, 1.0, (2 * r, r)), rng.normal(0, 1.0, r)
    ref = _scalar_step(e, s, Wg, bg)
    np.testing.assert_allclose(O.rnn_state_step(e, s, Wg, bg, "f32"), ref, rtol=1e-12, atol=1e-15)
    # bf16 state: the same values rounded to bf16 (ties aside, which random data does not hit)
    np.testing.assert_array_equal(O.rnn_state_step(e, s, Wg, bg, "bf16"), O.round_bf16(ref))


def _tiny(dtype, seed=2, bs=6, gamma=4, V=300, r=8):
    wl = I.WORKLOADS["qwen3_4b"].with_(bs=bs, gamma=gamma, V=V, r=r, d=16, dtype=dtype, seed=seed)
    return wl, I.make_host_inputs(wl, with_target=False, with_hidden=False, with_rnn=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tau", [1.0, 0.0])
def test_closed_gate_is_the_markov_head(dtype, tau):
    wl, h = _tiny(dtype)
    bg = np.full(wl.r, -np.inf, dtype=np.float32)
    a = O.draft_block(h["U"], h["W1"], h["W2t"], h["anchor"], tau, 3, 5, dtype=dtype)
    b = O.rnn_draft_block(h["U"], h["W1"], h["W2t"], h["Wg"], bg, h["anchor"], tau, 3, 5, dtype=dtype)
    for x, y in zip(a, b[:4]):
        np.testing.assert_array_equal(x, y)
    prev = np.concatenate([h["anchor"][:, None], a[0][:, :-1]], axis=1)
    np.testing.assert_array_equal(b[4], O.to_f64(h["W1"], dtype)[prev])


def test_open_gate_keeps_the_state_at_zero():
    wl, h = _tiny("f32")
    bg = np.full(wl.r, np.inf, dtype=np.float32)
    b = O.rnn_draft_block(h["U"], h["W1"], h["W2t"], h["Wg"], bg, h["anchor"], 1.0, 3, 5, dtype="f32")
    assert not b[4].any()
    zero = np.zeros_like(h["W2t"])
    a = O.draft_block(h["U"], h["W1"], zero, h["anchor"], 1.0, 3, 5, dtype="f32")
    for x, y in zip(a, b[:4]):
        np.testing.assert_array_equal(x, y)


def _exact_joint(U, W1, W2t, Wg, bg, x0, gamma):
    """Probability of every (x_1 .. x_gamma) by enumerating prefixes with the scalar recurrence."""
    V, r = W1.shape
    probs = {}
    for seq in itertools.product(range(V), repeat=gamma):
        s = np.zeros((1, r))
        p = 1.0
        prev = x0
        for k in range(gamma):
            s = _scalar_step(W1[prev][None, :], s, Wg, bg)
            p *= softmax(U[k] + s[0] @ W2t.T)[seq[k]]
            prev = seq[k]
        probs[seq] = p
    return probs


def test_joint_law_of_the_first_three_tokens():
    rng = np.random.default_rng(5)
    V, r, gamma, n = 5, 3, 3, 12000
    U1 = rng.normal(0, 0.8, (gamma, V))
    W1 = rng.normal(0, 1.2, (V, r))
    W2t = rng.normal(0, 1.2, (V, r))
    Wg = rng.normal(0, 1.5, (2 * r, r))
    bg = rng.normal(0, 1.0, r)
    x0 = 2
    exact = _exact_joint(U1, W1, W2t, Wg, bg, x0, gamma)
    # the state carries x_1 into position 3: its law given (x_1, x_2 = 0) differs across x_1
    cond = [np.array([exact[(a, 0, c)] for c in range(V)]) for a in range(V)]
    cond = [c / c.sum() for c in cond]
    assert max(np.abs(cond[a] - cond[0]).max() for a in range(V)) > 0.02
    U = np.repeat(U1[None], n, 0).astype(np.float32)
    tok, _, _, _, _ = O.rnn_draft_block(U, W1.astype(np.float32), W2t.astype(np.float32), Wg.astype(np.float32),
                                        bg.astype(np.float32), np.full(n, x0, np.int32), 1.0, 11, 0, dtype="f32")
    # the float32 inputs are what the draft saw: recompute the exact law from them
    exact = _exact_joint(U1.astype(np.float32).astype(np.float64), W1.astype(np.float32).astype(np.float64),
                         W2t.astype(np.float32).astype(np.float64), Wg.astype(np.float32).astype(np.float64),
                         bg.astype(np.float32).astype(np.float64), x0, gamma)
    keys = list(exact)
    idx = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for row in tok:
        counts[idx[tuple(int(v) for v in row)]] += 1
    expect = np.array([exact[k] for k in keys]) * n
    ok = expect > 5  # pool the rare cells
    obs = np.append(counts[ok], counts[~ok].sum())
    exp = np.append(expect[ok], expect[~ok].sum())
    assert stats.chisquare(obs, exp).pvalue > 1e-4
    # (x_1, x_2) marginal as well
    c12 = np.zeros((V, V))
    e12 = np.zeros((V, V))
    for k, i in idx.items():
        c12[k[0], k[1]] += counts[i]
        e12[k[0], k[1]] += exact[k] * n
    assert stats.chisquare(c12.ravel(), e12.ravel()).pvalue > 1e-4


def test_verify_with_closed_gate_states_equals_markov_recompute():
    wl, h = _tiny("f32", seed=7, bs=40, gamma=4, V=200)
    t = I.make_host_inputs(wl, with_hidden=False)["target"]
    bg = np.full(wl.r, -np.inf, dtype=np.float32)
    tok, lx, lse, _, st = O.rnn_draft_block(h["U"], h["W1"], h["W2t"], h["Wg"], bg, h["anchor"], 1.0, 3, 1,
                                            dtype="f32")
    win = I.random_windows(wl.bs, wl.gamma, 9)
    cu, ids, req, pos, padded = O.pack(win, h["anchor"], tok, [], wl.bs * (wl.gamma + 1))
    packed = I.gather_packed_target(t, req, pos, padded)
    a = O.verify(packed, cu, win, O.COMPACT, h["anchor"], tok, lx, lse, h["U"], h["W1"], h["W2t"], 1.0, 3, 1,
                 dtype="f32")
    b = O.verify(packed, cu, win, O.COMPACT, h["anchor"], tok, lx, lse, h["U"], h["W1"], h["W2t"], 1.0, 3, 1,
                 dtype="f32", draft_states=st)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_rnn_draft_first_committed_token_is_target_distributed(tau):
    """Lossless with the RNN head: residuals drawn against the RNN draft's p_d (recomputed from
    its states) leave the first committed token distributed as softmax(t / tau)."""
    rng = np.random.default_rng(12)
    V, r, gamma, bs = 12, 4, 2, 300
    U1 = rng.normal(0, 1.2, (1, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.9, (V, r)).astype(np.float32)
    W2t = rng.normal(0, 0.9, (V, r)).astype(np.float32)
    Wg = rng.normal(0, 1.0, (2 * r, r)).astype(np.float32)
    bg = rng.normal(0, 1.0, r).astype(np.float32)
    target1 = rng.normal(0, 1.5, (1, gamma + 1, V)).astype(np.float32)
    U, target = np.repeat(U1, bs, 0), np.repeat(target1, bs, 0)
    anchor = np.full(bs, 3, np.int32)
    pt1 = softmax(target1[0, 0].astype(np.float64) / tau)
    counts = np.zeros(V)
    for step in range(20):
        tok, lx, lse, _, st = O.rnn_draft_block(U, W1, W2t, Wg, bg, anchor, tau, 4, step, dtype="f32")
        win = I.random_windows(bs, gamma, 300 + step)
        cu, ids, req, pos, padded = O.pack(win, anchor, tok, [], bs * (gamma + 1))
        packed = I.gather_packed_target(target, req, pos, padded)
        out, _, _, _ = O.verify(packed, cu, win, O.COMPACT, anchor, tok, lx, lse, U, W1, W2t, tau, 4, step,
                                dtype="f32", draft_states=st)
        np.add.at(counts, out[:, 0], 1)
    assert stats.chisquare(counts, pt1 * counts.sum()).pvalue > 1e-4
