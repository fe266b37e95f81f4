"""The near-margin divergence rate at full size: every request of the mixed-difficulty batch
(bs 256, gamma 7, V 151936, bf16), over ten steps of the orchestrated path (draft, confidence,
the global scheduler and the pack, the stand-in target forward, compact verification), against
the oracle run on all 256 requests of every step.

Decisions are the draft draws (one per position compared; a request's positions after a
divergence depend on the diverged token and are not counted) and the verification's accept
tests plus its one residual or bonus draw per request (fed forward: the oracle verifies the
GPU's drafted tokens, windows and draft statistics).  A decision may differ from the oracle
only where the oracle's own margin is below 1e-4; such divergences must stay below 0.01 % of
all decisions (the stated tolerance).  The rate is printed."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from oracle import pool as OP
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from tests.parity import NEAR, TOL, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

STEPS = 10


def _draft_decisions(tg, lg, sg, to, lo, so, mo):
    """(decisions, divergences) of the draft, checking every compared position's probabilities."""
    dec = div = 0
    bs, gamma = to.shape
    for r in range(bs):
        for k in range(gamma):
            dec += 1
            if tg[r, k] != to[r, k]:
                assert mo[r, k] < NEAR, (r, k, mo[r, k])
                div += 1
                break
            assert abs(np.expm1((lg[r, k] - sg[r, k]) - (lo[r, k] - so[r, k]))) <= TOL["bf16"], (r, k)
    return dec, div


def test_near_margin_divergence_rate_full_batch():
    wl = I.WORKLOADS["mixed_bs256"]
    dev = torch.device("cuda")
    inp = I.make_device_inputs(wl, dev)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    cap = int(I.tiers_for(wl)[-1])
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype, dev)
    sps = S.sps_table(inp["T_raw"], inp["tiers"], dev)
    tiers = torch.as_tensor(inp["tiers"], device=dev)
    fwd = S.gather_target_forward(inp["target"])
    U_h, anchor, target_h = to_np(inp["U"]), to_np(inp["anchor"]), to_np(inp["target"])
    dec = div = vdec = vdiv = 0
    with OP.pool(to_np(inp["W1"]), to_np(inp["W2t"]), "bf16") as p:
        for step in range(STEPS):
            S.run_step(inp, buf, sps, fwd, wl.temperature, wl.seed, 100 + step, B.DSPARK_COMPACT,
                       B.DSPARK_SCHED_GLOBAL_ARGMAX, tiers=tiers)
            assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
            tg, lg, sg = to_np(buf.tokens), to_np(buf.logit_x), to_np(buf.lse)
            (to, lo, so, mo), _ = OP.draft_all(p, U_h, anchor, wl.temperature, wl.seed, 100 + step)
            d, v = _draft_decisions(tg, lg, sg, to, lo, so, mo)
            dec, div = dec + d, div + v
            win = to_np(buf.window)
            (out_o, acc_o, _, mv_o), _ = OP.verify_all(p, target_h, U_h, win, O.COMPACT, anchor, tg, lg, sg,
                                                       wl.temperature, wl.seed, 100 + step)
            out_g, acc_g = to_np(buf.out_tokens), to_np(buf.acc_len)
            for r in range(bs):
                vdec += min(int(acc_o[r]) + 1, int(win[r])) + 1  # accept tests + the one draw
                if acc_g[r] != acc_o[r] or not np.array_equal(out_g[r], out_o[r]):
                    assert mv_o[r] < NEAR, (step, r, out_g[r], out_o[r], mv_o[r])
                    vdiv += 1
    rate = (div + vdiv) / (dec + vdec)
    print(f"\nnear-margin divergences: draft {div} of {dec} decisions, verify {vdiv} of {vdec}; "
          f"rate {rate:.2e} over {STEPS} steps x {bs} requests")
    assert dec >= STEPS * bs * gamma * 0.99 and vdec >= STEPS * bs
    assert rate < 1e-4
