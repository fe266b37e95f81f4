"""Planted mistakes: each one, put into a copy of the oracle, must make one of its pins fail.

Opt-in (DSPARK_MUTATION=1; each case runs a pytest subprocess on a copy of oracle/, tests/ and
the package, a few minutes in all).  A mistake that no pin catches would mean the oracle could
be wrong in that way unnoticed; every case here is caught.  The mutations are planted in the
oracle only, on the CPU."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# name -> (text in oracle/dspark_oracle.py, its replacement, the pins that must catch it)
MUTS = {
 "ratio_inverted": ("ratio = math.exp(lp_t - lp_d)", "ratio = math.exp(lp_d - lp_t)", "tests/test_oracle_verify.py::test_monte_carlo_acceptance_equals_one_minus_tv"),
 "verify_accept_untempered": ("                t = trow(k) / temperature\n                lp_t = t[x[k]] - logsumexp(t)",
                              "                t = trow(k)\n                lp_t = t[x[k]] - logsumexp(t)",
                              "tests/test_oracle_verify.py::test_monte_carlo_acceptance_equals_one_minus_tv"),
 "verify_residual_untempered": ("                t = trow(k) / temperature\n                p_t = np.exp(t - logsumexp(t))",
                                "                t = trow(k)\n                p_t = np.exp(t - logsumexp(t))",
                                "tests/test_oracle_verify.py::test_first_committed_token_is_target_distributed"),
 "verify_bonus_untempered": ("                t = trow(k) / temperature\n                x_new, m2 = two_level_gumbel(t,",
                             "                t = trow(k)\n                x_new, m2 = two_level_gumbel(t,",
                             "tests/test_oracle_verify.py::test_first_committed_token_is_target_distributed"),
 "verify_explicit_pd_untempered": ("d = Df[r, k - 1] / temperature", "d = Df[r, k - 1]",
                                   "tests/test_oracle_verify.py::test_explicit_draft_logits_first_committed_token_is_target_distributed"),
 "residual_flipped": ("res = np.maximum(0.0, p_t - p_d)", "res = np.maximum(0.0, p_d - p_t)", "tests/test_oracle_verify.py::test_first_committed_token_is_target_distributed"),
 "bias_wrong_token": ("x_prev = tokens[:, k - 1].astype(np.int64)", "x_prev = x_prev", "tests/test_oracle_sampling.py::test_draft_joint_distribution_of_first_two_tokens"),
 "conf_x_index": ("np.asarray(tokens, dtype=np.int64)[:, :gamma - 1]], axis=1)", "np.asarray(tokens, dtype=np.int64)[:, 1:gamma]], axis=1)", "tests/test_oracle_schedule_pack.py::test_confidence_feature_indexing"),
 "philox_round": ("c = [hi1 ^ c[1] ^ np.uint64(ka), lo1, hi0 ^ c[3] ^ np.uint64(kb), lo0]", "c = [hi0 ^ c[1] ^ np.uint64(ka), lo1, hi1 ^ c[3] ^ np.uint64(kb), lo0]", "tests/test_oracle_philox.py::test_philox_matches_triton_library_implementation"),
 "sched_nonstrict": ("if not theta[K + 1] > theta[K]:", "if theta[K + 1] < theta[K]:", "tests/test_oracle_schedule_pack.py"),
 "chunk_mass_max": ("safe_m + np.log(np.exp(blocks - safe_m[:, None]).sum(axis=1))", "safe_m", "tests/test_oracle_sampling.py::test_two_level_sampler_chunk_marginal_is_chunk_mass"),
 "zos_wrong_slot": ("    slot = step % 2\n", "    slot = (step + 1) % 2\n", "tests/test_oracle_zos.py"),
 "zos_budget_early_stop": ("return int(schedule(surv_f32, sps, GLOBAL_ARGMAX)[1])", "return int(schedule(surv_f32, sps, EARLY_STOP)[1])", "tests/test_oracle_zos.py"),
 "zos_tie_order": ("slots = sorted(((float(a[r, j]), r, j) for r in range(bs) for j in range(gamma)),\n                   key=lambda s: (-s[0], s[1], s[2]))", "slots = sorted(((float(a[r, j]), r, j) for r in range(bs) for j in range(gamma)),\n                   key=lambda s: (-s[0], -s[1], s[2]))", "tests/test_oracle_zos.py"),
 "zos_no_clamp": ("    K = min(K, bs * gamma, m_max - bs)\n", "    K = min(K, bs * gamma)\n", "tests/test_oracle_zos.py"),
 "ece_per_bin_norm": ("    e = float(np.sum(np.abs(lab - sc)) / N) if N else 0.0", "    e = float(np.sum(np.abs(lab - sc)) / max(int(cnt.max()), 1)) if N else 0.0", "tests/test_oracle_observe.py"),
 "ece_round_bins": ("    b = np.floor(a * np.float32(n_bins)).astype(np.int64)", "    b = np.round(a * np.float32(n_bins)).astype(np.int64)", "tests/test_oracle_observe.py"),
 "labels_strict": ("        return (c >= k).astype(np.int64), np.ones((bs, gamma), dtype=bool)", "        return (c > k).astype(np.int64), np.ones((bs, gamma), dtype=bool)", "tests/test_oracle_observe.py"),
 "labels_known_window_only": ("    known = (k <= w[:, None]) | (acc[:, None] < w[:, None])", "    known = (k <= w[:, None])", "tests/test_oracle_observe.py"),
 "util_inverted": ('st["sum_accepted_ceiling"] / st["sum_ceiling"] if st["sum_ceiling"]', 'st["sum_ceiling"] / st["sum_accepted_ceiling"] if st["sum_ceiling"]', "tests/test_oracle_observe.py"),
 "sts_label_offby1": ("        y = (c >= k + 1).astype(np.int64)", "        y = (c >= k).astype(np.int64)", "tests/test_oracle_observe.py"),
 "sts_no_carry": ("        prev = prev / (1.0 + np.exp(-z[:, k] / T[k]))", "        prev = prev", "tests/test_oracle_observe.py"),
 "sts_argmax": ("        g_star = int(np.argmin(table[k]))  # first minimum", "        g_star = int(np.argmax(table[k]))", "tests/test_oracle_observe.py"),
 "rnn_gate_swapped": ("    s = g * s_prev + (1.0 - g) * e\n", "    s = (1.0 - g) * s_prev + g * e\n",
                      "tests/test_oracle_rnn.py::test_closed_gate_is_the_markov_head"),
 "rnn_state_not_carried": ("        s = rnn_state_step(W1[x_prev], s, Wg, bg, dtype)",
                           "        s = rnn_state_step(W1[x_prev], np.zeros_like(s), Wg, bg, dtype)",
                           "tests/test_oracle_rnn.py::test_joint_law_of_the_first_three_tokens"),
 "rnn_verify_markov_row": ("a_row = W1f[x[k - 1]] if draft_states is None else np.asarray(draft_states[r][k - 1], np.float64)",
                           "a_row = W1f[x[k - 1]]",
                           "tests/test_oracle_rnn.py::test_rnn_draft_first_committed_token_is_target_distributed"),
 "cdf_nonstrict": ("    j = int(np.argmax(C > t))", "    j = int(np.argmax(C >= t))", "tests/test_oracle_sampling.py::test_inverse_cdf_by_hand"),
 "cdf_reversed_sums": ("    C = np.cumsum(w)\n", "    C = np.cumsum(w[::-1])\n", "tests/test_oracle_sampling.py::test_inverse_cdf_by_hand"),
 "cdf_wrong_uniform": ("    u = float(uniform(seed, step, purpose_elem, req, pos, np.array([0]))[0])",
                       "    u = float(uniform(seed, step, purpose_elem, req, pos, np.array([1]))[0])",
                       "tests/test_oracle_sampling.py::test_chunk_cdf_sampler_levels"),
 "cdf_chunk_offset_dropped": ("    return lo + j, min(_top2_gap(Kc), m2)", "    return j, min(_top2_gap(Kc), m2)",
                              "tests/test_oracle_sampling.py::test_chunk_cdf_sampler_matches_softmax_with_ragged_chunks"),
 "resid_u_row": ("d = (Uf[r, k - 1] + a_row @ W2f.T) / temperature", "d = (Uf[r, min(k, gamma - 1)] + a_row @ W2f.T) / temperature", "tests/test_oracle_verify.py"),
 "resid_cond_token": ("a_row = W1f[x[k - 1]] if", "a_row = W1f[x[k]] if", "tests/test_oracle_verify.py"),
 "resid_pd_untempered": ("d = (Uf[r, k - 1] + a_row @ W2f.T) / temperature", "d = (Uf[r, k - 1] + a_row @ W2f.T)", "tests/test_oracle_verify.py"),
 "draft_logit_x_raw": ("return v, t[v], logsumexp(t), mg", "return v, ell_row[v], logsumexp(t), mg", "tests/test_oracle_verify.py tests/test_oracle_sampling.py"),
 "ceiling_offby1": ("ceiling[r] = (first_reject - 1) if", "ceiling[r] = first_reject if", "tests/test_oracle_verify.py"),
 "captests_window": ("L_test = lr if mode == COMPACT else gamma", "L_test = lr if mode != STATIC else gamma", "tests/test_oracle_verify.py"),
 "explicit_row_offby1": ("d = Df[r, k - 1] / temperature", "d = Df[r, min(k, gamma - 1)] / temperature", "tests/test_oracle_verify.py"),
 "sched_tau_no_bs": ("tau = bs + math.ldexp(float(S), -FIX_SHIFT)", "tau = math.ldexp(float(S), -FIX_SHIFT)", "tests/test_oracle_schedule_pack.py"),
 "sched_sps_index": ("theta[K] = tau * float(sps[bs + K])", "theta[K] = tau * float(sps[min(K + bs + 1, m_max)])", "tests/test_oracle_schedule_pack.py"),
 "sched_fixed_ceil": ("S += int(math.floor(max(slots[K - 1][0], 0.0) * 2.0 ** FIX_SHIFT))", "S += int(math.ceil(max(slots[K - 1][0], 0.0) * 2.0 ** FIX_SHIFT))", "tests/test_oracle_schedule_pack.py"),
 'rnn_no_round': ('return round_bf16(s) if dtype == "bf16" else s', 'return s', 'tests/test_oracle_rnn.py'),
 "gumbel_level2_uniform": ("ke = logw[lo:hi] + gumbel(", "ke = 0.0 * logw[lo:hi] + gumbel(", "tests/test_oracle_sampling.py tests/test_oracle_verify.py"),
 "greedy_correction_next_row": ("                x_new = _first_argmax(trow(k))\n", "                x_new = _first_argmax(trow(min(k + 1, L_test + 1)))\n", "tests/test_oracle_verify.py"),
 "conf_T_reversed": ("conf = 1.0 / (1.0 + np.exp(-z / T[None, :]))", "conf = 1.0 / (1.0 + np.exp(-z / T[None, ::-1]))", "tests/test_oracle_schedule_pack.py"),
 "sps_no_tier": ("            sps[M] = 1.0 / T_mono[t]", "            sps[M] = 1.0 / T_mono[M]", "tests/test_oracle_schedule_pack.py"),
 "pack_pos_offby1": ("            pos[p] = j\n", "            pos[p] = j + 1\n", "tests/test_oracle_schedule_pack.py"),
 "lse_d_dropped": ("lp_d = float(logit_x[r, k - 1]) - float(lse[r, k - 1])", "lp_d = float(logit_x[r, k - 1])", "tests/test_oracle_verify.py"),
 "draft_lse_untempered": ("return v, t[v], logsumexp(t), mg", "return v, t[v], logsumexp(ell_row), mg", "tests/test_oracle_verify.py tests/test_oracle_sampling.py"),
 "tier_strict": ("        if t >= M:\n            return int(t)", "        if t > M:\n            return int(t)", "tests/test_oracle_schedule_pack.py"),
 "uniform_shift8": ("return ((b >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23", "return ((b >> np.uint32(8)).astype(np.float64) + 0.5) * 2.0 ** -23", "tests/test_oracle_philox.py"),
 "chunk_pad_zero": ("    padded = np.full(nc * chunk, -np.inf)\n", "    padded = np.zeros(nc * chunk)\n", "tests/test_oracle_sampling.py"),
 "icdf_unscaled": ("    t = u * S\n", "    t = u\n", "tests/test_oracle_sampling.py"),
 "early_stop_plus1": ("                K_star = K\n                break", "                K_star = K + 1\n                break", "tests/test_oracle_schedule_pack.py"),
 "sched_ascending": ("    slots.sort(key=lambda s: (-s[0], s[1], s[2]))", "    slots.sort(key=lambda s: (s[0], s[1], s[2]))", "tests/test_oracle_schedule_pack.py"),
 "verify_acc_k": ("            acc = k - 1\n", "            acc = k\n", "tests/test_oracle_verify.py"),
 "verify_out_anchor": ("        out[r, :acc] = x[1:acc + 1]", "        out[r, :acc] = x[0:acc]", "tests/test_oracle_verify.py"),
 "rnn_no_bias": ("    z = np.concatenate([e, s_prev], axis=1) @ Wg + bg[None, :]", "    z = np.concatenate([e, s_prev], axis=1) @ Wg", "tests/test_oracle_rnn.py"),
 "rnn_s0_anchor": ("    s = np.zeros((bs, r))\n    x_prev", "    s = W1[np.asarray(anchor, dtype=np.int64)]\n    x_prev", "tests/test_oracle_rnn.py"),
 "sps_min_accumulate": ("    T_mono = np.maximum.accumulate(T_raw)", "    T_mono = np.minimum.accumulate(T_raw)", "tests/test_oracle_schedule_pack.py"),
 "conf_surv_shift": ("    surv = np.cumprod(conf, axis=1)", "    surv = np.cumprod(np.concatenate([np.ones((bs, 1)), conf[:, :-1]], axis=1), axis=1)", "tests/test_oracle_schedule_pack.py"),
 "markov_no_U": ("    return U_k + W1[x_prev] @ W2t.T", "    return W1[x_prev] @ W2t.T", "tests/test_oracle_sampling.py"),
 "draft_greedy_last_max": ("        v = _first_argmax(ell_row)\n", "        v = int(len(ell_row) - 1 - np.argmax(ell_row[::-1]))\n", "tests/test_oracle_sampling.py"),
 "ece_no_abs": ("    e = float(np.sum(np.abs(lab - sc)) / N) if N else 0.0", "    e = float(abs(np.sum(lab - sc)) / N) if N else 0.0", "tests/test_oracle_observe.py"),
}


@pytest.mark.skipif(os.environ.get("DSPARK_MUTATION") != "1", reason="opt-in: DSPARK_MUTATION=1")
@pytest.mark.parametrize("name", list(MUTS))
def test_planted_mistake_is_caught(name, tmp_path):
    a, b, pins = MUTS[name]
    src = open(os.path.join(ROOT, "oracle", "dspark_oracle.py")).read()
    assert a in src, "the mutated text is no longer in the oracle"
    for d in ("oracle", "tests", "speculative_decoding_draft_markov_gb300"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d, ignore=shutil.ignore_patterns("lib", "*.so", "__pycache__"))
    (tmp_path / "oracle" / "dspark_oracle.py").write_text(src.replace(a, b))
    env = dict(os.environ, DSPARK_MUTATION="0")
    p = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *pins.split()],
                       capture_output=True, text=True, cwd=tmp_path, env=env, timeout=900)
    assert p.returncode == 1, (f"planted mistake {name!r} passed every pin in {pins}" if p.returncode == 0
                               else f"the pins of {name!r} did not run (exit {p.returncode}): {p.stdout[-400:]}")
