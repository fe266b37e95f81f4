"""Full-size parity for every benchmark workload, on sampled requests.

The GPU runs the whole workload through the C ABI (every request, full vocabulary); the
oracle recomputes a sample of requests one by one from the same input bytes (copied from
the device) with the same random streams (req_ids), and decisions must agree except at
near-margin decisions (< 1e-4).  Verify windows come from the seeded generator (the
scheduler is checked bit-exactly on full-size generator survival in test_gpu_parity)."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from tests.parity import NEAR, TOL, compare_draft, compare_verify, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [
    ("qwen3_4b", I.WORKLOADS["qwen3_4b"], [O.COMPACT], 1.0),
    ("mixed_bs256", I.WORKLOADS["mixed_bs256"], [O.COMPACT, O.CAP_ACCEPT], 1.0),
    ("long_block_t1", I.WORKLOADS["long_block"], [O.COMPACT], 1.0),
    ("long_block_greedy", I.WORKLOADS["long_block"], [O.STATIC, O.COMPACT], 0.0),
] + [(f"dsv4_bs{b}", I.dsv4(b), [O.STATIC, O.COMPACT], 1.0) for b in I.DSV4_BATCHES]


def _sample(bs):
    idx = sorted({0, bs // 3, (2 * bs) // 3, bs - 1})
    return np.array(idx)


@pytest.mark.parametrize("name,wl,modes,temperature", CASES, ids=[c[0] for c in CASES])
def test_workload_full_size(name, wl, modes, temperature):
    dev = torch.device("cuda")
    inp = I.make_device_inputs(wl, dev)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    rows = _sample(bs)
    t_rows = torch.as_tensor(rows, device=dev)
    step = 5
    cap = bs * (gamma + 1)
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype, dev)

    # S1 draft: every request on the GPU, sampled requests in the oracle
    B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], temperature, wl.seed, step,
                         buf.tokens, buf.logit_x, buf.lse, buf.ws)
    assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
    W1, W2t = to_np(inp["W1"]), to_np(inp["W2t"])
    U_s = to_np(inp["U"][t_rows])
    anchor = to_np(inp["anchor"])
    to, lo, so, mo = O.draft_block(U_s, W1, W2t, anchor[rows], temperature, wl.seed, step, dtype="bf16",
                                   req_ids=rows)
    tg, lg, sg = (to_np(t)[rows] for t in (buf.tokens, buf.logit_x, buf.lse))
    compare_draft(tg, lg, sg, to, lo, so, mo, "bf16", greedy=temperature == 0.0)
    same = np.array([np.array_equal(tg[i], to[i]) for i in range(len(rows))])

    # S2 confidence on the GPU's tokens, checked for the sampled requests
    B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], buf.tokens, inp["w"], inp["b"], inp["sts_T"],
                        buf.conf, buf.surv)
    c_o, a_o, _ = O.confidence(to_np(inp["h"][t_rows]), W1, anchor[rows], to_np(buf.tokens)[rows],
                               to_np(inp["w"]), inp["b"], to_np(inp["sts_T"]))
    np.testing.assert_allclose(to_np(buf.conf)[rows], c_o, rtol=TOL["bf16"], atol=0)
    np.testing.assert_allclose(to_np(buf.surv)[rows], a_o, rtol=TOL["bf16"], atol=0)

    # S4 + S5 with generator windows, every mode of the workload
    win = I.random_windows(bs, gamma, wl.seed + 7)
    buf.window.copy_(torch.as_tensor(win, device=dev))
    target_s = to_np(inp["target"][t_rows])
    for mode in modes:
        B.dspark_pack(buf.window if mode == O.COMPACT else None, inp["anchor"], buf.tokens, None, buf.cu,
                      buf.ids, buf.req, buf.pos, buf.padded, buf.ws)
        S.gather_target_forward(inp["target"])(buf)
        S.verify(inp, buf, temperature, wl.seed, step, mode)
        assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
        keep = np.nonzero(same)[0]
        if keep.size == 0:
            continue
        ks = rows[keep]
        # the oracle's own packing of the sampled requests
        cu_o, _, req_o, pos_o, _ = O.pack(win[ks] if mode == O.COMPACT else None, anchor[ks], to[keep], [],
                                         len(ks) * (gamma + 1), gamma=gamma)
        packed = I.gather_packed_target(target_s[keep], req_o, pos_o, len(ks) * (gamma + 1))
        out_o, acc_o, ceil_o, mv_o = O.verify(packed, cu_o, win[ks], mode, anchor[ks], to[keep], lo[keep],
                                              so[keep], U_s[keep], W1, W2t, temperature, wl.seed, step,
                                              dtype="bf16", req_ids=ks)
        ceil_g = to_np(buf.ceiling)[ks] if mode == O.CAP_ACCEPT else None
        compare_verify(to_np(buf.out_tokens)[ks], to_np(buf.acc_len)[ks], out_o, acc_o, mv_o,
                       ceil_g, ceil_o if ceil_g is not None else None)
