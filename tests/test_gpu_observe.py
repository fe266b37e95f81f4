"""GPU parity of observability and calibration through the C ABI: the confidence head's
pre-STS logits, the per-step observability records (compact, cap-accept and static runs;
integer fields bit-exact, fixed-point score sums within their quantum) and the sequential
temperature scaling fit (chosen temperatures and ECE against the oracle; recovery of a known
law at full size)."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from tests.parity import TOL, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

INT_FIELDS = ["steps", "requests", "sum_window", "sum_accepted", "ceiling_requests", "sum_ceiling",
              "sum_accepted_ceiling"]


def test_confidence_logits_output():
    wl = I.WORKLOADS["qwen3_4b"].with_(V=4096, bs=16)
    inp = I.make_device_inputs(wl, torch.device("cuda"), with_target=False)
    bs, gamma = wl.bs, wl.gamma
    tokens = torch.as_tensor(I.random_tokens(bs, gamma, wl.V, 3), device="cuda")
    conf, surv, z = (torch.zeros((bs, gamma), dtype=torch.float32, device="cuda") for _ in range(3))
    conf2, surv2 = torch.zeros_like(conf), torch.zeros_like(conf)
    B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], tokens, inp["w"], inp["b"], inp["sts_T"], conf, surv,
                        z_logit=z)
    B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], tokens, inp["w"], inp["b"], inp["sts_T"], conf2, surv2)
    assert torch.equal(conf, conf2) and torch.equal(surv, surv2)   # the extra output changes nothing
    _, _, z_o = O.confidence(to_np(inp["h"]), to_np(inp["W1"]), to_np(inp["anchor"]), to_np(tokens),
                             to_np(inp["w"]), inp["b"], to_np(inp["sts_T"]))
    np.testing.assert_allclose(z.cpu().numpy(), z_o, rtol=TOL["bf16"], atol=1e-4)
    # STS divides exactly this logit
    c = 1.0 / (1.0 + np.exp(-z.cpu().numpy().astype(np.float64) / to_np(inp["sts_T"])[None, :]))
    np.testing.assert_allclose(conf.cpu().numpy(), c, rtol=1e-5)


def _check_stats(st, ref, n_bins, gamma):
    for k in INT_FIELDS:
        assert getattr(st, k) == int(ref[k]), k
    for k in ("window_hist", "accepted_hist", "ceiling_hist"):
        assert list(getattr(st, k)) == [int(v) for v in ref[k]], k
    assert list(st.bin_count[:n_bins]) == [int(v) for v in ref["bin_count"]]
    assert list(st.bin_label[:n_bins]) == [int(v) for v in ref["bin_label"]]
    assert all(v == 0 for v in st.bin_count[n_bins:])
    # fixed-point sums: sum of floor(a 2^32) is within `count` quanta below the exact sum
    for fx, sc, cnt in ((st.bin_score_fx[:n_bins], ref["bin_score"], ref["bin_count"]),
                        (st.pos_score_fx[:gamma], ref["pos_score"], ref["pos_count"])):
        for g, s, c in zip(fx, sc, cnt):
            assert -int(c) - 1 <= g - s * 2.0 ** 32 <= 1, (g, s * 2.0 ** 32, c)
    assert list(st.pos_count[:gamma]) == [int(v) for v in ref["pos_count"]]
    assert list(st.pos_label[:gamma]) == [int(v) for v in ref["pos_label"]]


@pytest.mark.parametrize("bs,gamma,n_bins,run", [(256, 7, 10, "compact"), (256, 7, 15, "cap_accept"),
                                                 (1, 16, 64, "static"), (100, 3, 1, "compact"),
                                                 (37, 5, 20, "cap_accept")])
def test_observe_records_bit_exact(bs, gamma, n_bins, run):
    rng = np.random.default_rng(bs + gamma)
    stats = B.alloc_obs_stats()
    ws = B.alloc_workspace(bs, gamma, 1024)
    recs = []
    for t in range(4):
        surv = I.random_survival(bs, gamma, 900 + t, ties=(t == 2))
        if t == 3:
            surv[:, -1] = 1.0          # the edge of the last bin
            surv[0, :] = 0.0
        ceiling = rng.integers(0, gamma + 1, bs).astype(np.int32)
        window = rng.integers(0, gamma + 1, bs).astype(np.int32)
        if run == "static":
            window_arg, acc, ceil_arg = None, ceiling, ceiling
        else:
            acc = np.minimum(ceiling, window).astype(np.int32)
            window_arg, ceil_arg = window, (ceiling if run == "cap_accept" else None)
        d = lambda x: None if x is None else torch.as_tensor(x, device="cuda")
        B.dspark_observe(d(surv), d(window_arg), d(acc), d(ceil_arg), n_bins, stats, ws)
        recs.append(O.observe(surv, window_arg, acc, ceil_arg, n_bins))
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK
    ref = {k: sum(r[k] for r in recs) for k in recs[0]}
    st = B.obs_stats_from(stats)
    _check_stats(st, ref, n_bins, gamma)
    rep, rep_o = B.dspark_obs_report(st, n_bins), O.obs_report(ref)
    for k in ("mean_window", "mean_accepted", "ece"):
        assert rep[k] == pytest.approx(rep_o[k], rel=1e-9, abs=1e-9)
    if run != "compact":
        assert rep["utilisation"] == pytest.approx(rep_o["utilisation"], rel=1e-12)


def test_observe_rejects_inconsistent_records():
    bs, gamma = 8, 4
    stats = B.alloc_obs_stats()
    ws = B.alloc_workspace(bs, gamma, 1024)
    surv = torch.as_tensor(I.random_survival(bs, gamma, 1), device="cuda")
    win = torch.full((bs,), 2, dtype=torch.int32, device="cuda")
    acc = torch.full((bs,), 3, dtype=torch.int32, device="cuda")       # more accepted than verified
    B.dspark_observe(surv, win, acc, None, 10, stats, ws)
    assert B.dspark_read_device_status(ws) == B.DSPARK_EINVAL
    assert int(stats.abs().sum().item()) == 0                         # nothing recorded
    acc.fill_(1)
    B.dspark_observe(surv, win, acc, None, 10, stats, ws)
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK
    assert B.obs_stats_from(stats).steps == 1


def _fit_gpu(z, ceiling, grid, n_bins):
    N, gamma = z.shape
    T = torch.zeros(gamma, dtype=torch.float32, device="cuda")
    e = torch.zeros(gamma, dtype=torch.float64, device="cuda")
    B.dspark_sts_fit(torch.as_tensor(z, device="cuda"), torch.as_tensor(ceiling, device="cuda"),
                     torch.as_tensor(grid, dtype=torch.float32, device="cuda"), n_bins, T, e)
    return T.cpu().numpy(), e.cpu().numpy()


@pytest.mark.parametrize("N,gamma,n_bins", [(12000, 5, 10), (3001, 3, 15), (1, 2, 4)])
def test_sts_fit_matches_oracle(N, gamma, n_bins):
    T_true = [1.6, 1.9, 1.3, 2.2, 1.0][:gamma]
    z, ceiling = I.calibration_steps(N, gamma, T_true, seed=N)
    grid = np.float32(np.round(np.arange(0.5, 3.01, 0.1), 6))
    T_g, e_g = _fit_gpu(z, ceiling, grid, n_bins)
    T_o, e_o, table = O.sts_fit(z, ceiling, grid.astype(np.float64), n_bins)
    tol = 5.0 / N + 1e-9   # a few scores on the other side of a bin edge (fp32 vs fp64 chains)
    for k in range(gamma):
        g = int(np.argmin(np.abs(grid - T_g[k])))
        assert grid[g] == T_g[k]
        assert table[k, g] <= table[k].min() + tol, (k, T_g[k], T_o[k])   # the GPU's choice is a minimum
        assert abs(e_g[k] - table[k, g]) <= tol, (k, e_g[k], table[k, g])
        if T_g[k] != np.float32(T_o[k]):
            break   # a near-tie took another temperature: later positions condition on it


def test_sts_fit_full_size_recovers_the_law():
    """2^20 labelled prefixes, 7 positions, 64 grid values: the fit recovers the temperatures of
    the law that drew the labels, and the reported ECE is the oracle's ECE at those values."""
    N, gamma = 1 << 20, 7
    T_true = [1.5, 1.8, 1.2, 2.0, 1.4, 1.1, 1.7]
    z, ceiling = I.calibration_steps(N, gamma, T_true, seed=77, mu0=3.0, mu_slope=-0.1)
    grid = np.float32(np.round(np.linspace(0.5, 3.65, 64), 6))
    T_g, e_g = _fit_gpu(z, ceiling, grid, 15)
    step = float(grid[1] - grid[0])
    assert np.all(np.abs(T_g[:5] - T_true[:5]) <= 2 * step + 1e-6), (T_g, T_true)
    # the reported ECE at the chosen temperatures, recomputed by the oracle on 2^17 of the prefixes
    sub = slice(0, 1 << 17)
    prev = np.ones(1 << 17)
    for k in range(gamma):
        prev = prev / (1.0 + np.exp(-z[sub, k].astype(np.float64) / float(T_g[k])))
    e_sub = O.ece(prev.astype(np.float32), (ceiling[sub] >= gamma).astype(np.int64), 15)[0]
    assert e_g[-1] == pytest.approx(e_sub, abs=0.01)   # a subsample: sampling noise only
    assert np.all(e_g < 0.02)
