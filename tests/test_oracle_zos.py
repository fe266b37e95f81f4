"""Pins of the oracle's asynchronous (zero-overhead) scheduler: the verify budget of step t is
the global-search budget of step t - 2's survival, the windows are the top-K slots of step t's
own survival.

- zos_select equals exhaustive search over every prefix-length assignment with sum K
  (exact rational arithmetic), and follows the scheduler's tie order (hand-computed);
- the budget of step t does not depend on the survival of steps t - 1 and t (causal barrier);
- the first two steps, with nothing recorded, reduce to the synchronous global search;
- with a stationary survival the windows equal the synchronous global search's at every step;
- the stale budget is clamped to the current batch and table."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import inputs as I


def _table(m_max, seed, tier_step=1):
    rng = np.random.default_rng(seed)
    T = 1.0 + rng.random() * 3.0 + 0.05 * np.arange(m_max + 1)
    tiers = list(range(tier_step, m_max, tier_step)) + [m_max]
    return O.build_sps(T, tiers)


def _best_prefix_assignment(a: np.ndarray, K: int):
    """Every prefix-length assignment with sum K; the one(s) of largest exact survival sum."""
    bs, gamma = a.shape
    af = [[Fraction(float(a[r, j])) for j in range(gamma)] for r in range(bs)]
    best, arg = None, []
    for ls in itertools.product(range(gamma + 1), repeat=bs):
        if sum(ls) != K:
            continue
        s = sum((sum(af[r][:ls[r]], Fraction(0)) for r in range(bs)), Fraction(0))
        if best is None or s > best:
            best, arg = s, [ls]
        elif s == best:
            arg.append(ls)
    return best, arg


@pytest.mark.parametrize("seed", range(6))
def test_select_equals_exhaustive_top_k(seed):
    bs, gamma = (3, 3) if seed % 2 else (2, 4)
    a = I.random_survival(bs, gamma, 300 + seed)
    assert len(np.unique(a)) == a.size   # distinct values: a unique optimum for every K
    for K in range(bs * gamma + 1):
        win = O.zos_select(a, K)
        best, arg = _best_prefix_assignment(a, K)
        assert len(arg) == 1 and tuple(int(v) for v in win) == arg[0]
        assert win.sum() == K


def test_select_tie_order_by_hand():
    a = np.array([[0.5, 0.5, 0.25], [0.5, 0.25, 0.25]], dtype=np.float32)
    # rank order: (0,0) (0,1) (1,0) [0.5, lower request first] then (0,2) (1,1) (1,2) [0.25]
    expect = {0: [0, 0], 1: [1, 0], 2: [2, 0], 3: [2, 1], 4: [3, 1], 5: [3, 2], 6: [3, 3]}
    for K, w in expect.items():
        assert list(O.zos_select(a, K)) == w
    assert list(O.zos_select(a, 99)) == [3, 3] and list(O.zos_select(a, -1)) == [0, 0]


def test_budget_comes_from_two_steps_back_only():
    bs, gamma = 6, 5
    sps = _table(bs * (gamma + 1), 1, tier_step=4)
    seq = [I.random_survival(bs, gamma, 40 + t) for t in range(6)]
    ring = [-1, -1]
    got = [O.zos_step(s, sps, ring, t) for t, s in enumerate(seq)]
    for t in range(2, 6):
        K_expect = min(O.zos_budget(seq[t - 2], sps), bs * gamma)
        assert got[t][1] == K_expect
        np.testing.assert_array_equal(got[t][0], O.zos_select(seq[t], K_expect))
    # change the survival of steps t - 1 and t: the budget of step t stays
    alt = list(seq)
    alt[2] = I.random_survival(bs, gamma, 999)
    alt[3] = np.full((bs, gamma), 0.01, dtype=np.float32)
    ring2 = [-1, -1]
    got2 = [O.zos_step(s, sps, ring2, t) for t, s in enumerate(alt)]
    assert got2[3][1] == got[3][1]          # K_3 comes from step 1, unchanged
    assert got2[4][1] == O.zos_budget(alt[2], sps)


def test_first_two_steps_are_the_synchronous_global_search():
    bs, gamma = 5, 4
    sps = _table(bs * (gamma + 1), 2, tier_step=3)
    ring = [-1, -1]
    for t in range(2):
        s = I.random_survival(bs, gamma, 70 + t)
        win, K = O.zos_step(s, sps, ring, t)
        w_sync, K_sync, _, _ = O.schedule(s, sps, O.GLOBAL_ARGMAX)
        assert K == K_sync and np.array_equal(win, w_sync)
    assert ring[0] >= 0 and ring[1] >= 0


def test_stationary_survival_equals_synchronous_schedule():
    bs, gamma = 4, 4
    sps = _table(bs * (gamma + 1), 3, tier_step=2)
    s = I.random_survival(bs, gamma, 5)
    w_sync, K_sync, _, _ = O.schedule(s, sps, O.GLOBAL_ARGMAX)
    ring = [-1, -1]
    for t in range(5):
        win, K = O.zos_step(s, sps, ring, t)
        assert K == K_sync and np.array_equal(win, w_sync)


def test_stale_budget_is_clamped_to_the_current_batch():
    sps = np.ones(40)                     # flat table: the global search admits every slot
    big = np.full((4, 6), 0.9, dtype=np.float32)
    ring = [-1, -1]
    win, K = O.zos_step(big, sps, ring, 0)
    assert K == 24 and ring[0] == 24
    small = np.full((2, 3), 0.5, dtype=np.float32)   # two steps later: a smaller batch
    win, K = O.zos_step(small, sps, ring, 2)
    assert K == 6 and list(win) == [3, 3]
    short = np.ones(9)                    # m_max = 8: at most 8 - bs slots for a batch of 2
    ring = [7, -1]
    win, K = O.zos_step(small, short, ring, 0)
    assert K == 6
    ring = [7, -1]
    win, K = O.zos_step(np.full((3, 3), 0.5, dtype=np.float32), short, ring, 0)
    assert K == 5 and list(win) == [3, 2, 0]   # equal keys: lower request first
