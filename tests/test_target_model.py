"""The workloads' synthetic target model, "target = U + W1[x_{k-1}] W2 + noise" (the drafter's
logits at the drafted prefix plus noise): with zero noise in fp32 it equals the draft's own
logits, so the oracle's verification accepts every drafted token; a Markov term taken at the
wrong prefix token would not (the weights are scaled up so that the term dominates U).  The GPU
test checks that the device forward and the host one compute the same rows."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from oracle import dspark_oracle as O  # noqa: E402
from speculative_decoding_draft_markov_gb300 import inputs as I  # noqa: E402


def test_markov_target_at_zero_noise_accepts_every_draft_token():
    wl = I.WORKLOADS["tiny_fp32"].with_(sigmas=(0.0,), w_std=0.5)
    h = I.make_host_inputs(wl)
    bs, gamma = wl.bs, wl.gamma
    n = acc_sum = 0
    for step in range(8):
        tok, lx, lse, _ = O.draft_block(h["U"], h["W1"], h["W2t"], h["anchor"], 1.0, wl.seed, step, dtype="f32")
        target = bench._host_target(h, tok, "f32")
        window = np.full(bs, gamma, dtype=np.int32)
        cu, ids, req, pos, padded = O.pack(window, h["anchor"], tok, [], cap=bs * (gamma + 1))
        packed = I.gather_packed_target(target, req, pos, padded)
        _, acc, _, _ = O.verify(packed, cu, window, O.COMPACT, h["anchor"], tok, lx, lse, h["U"], h["W1"],
                                h["W2t"], 1.0, wl.seed, step, dtype="f32")
        n += bs * gamma
        acc_sum += int(acc.sum())
    assert acc_sum == n


def test_markov_target_with_noise_is_base_plus_term():
    """bf16: each row is the base row plus the rounded Markov term of its prefix, rounded once
    more; row 0 takes the anchor's term."""
    wl = I.WORKLOADS["tiny_fp32"].with_(dtype="bf16")
    h = I.make_host_inputs(wl)
    rng = np.random.default_rng(3)
    tok = rng.integers(0, wl.V, size=(wl.bs, wl.gamma)).astype(np.int32)
    t = bench._host_target(h, tok, "bf16")
    f = I.bf16_bits_to_f32
    W1, W2t = f(h["W1"]).astype(np.float64), f(h["W2t"]).astype(np.float64)
    for b in range(wl.bs):
        for j in range(wl.gamma + 1):
            x = h["anchor"][b] if j == 0 else tok[b, j - 1]
            want = f(h["target"][b, j]).astype(np.float64) + W1[x] @ W2t.T
            # two bf16 roundings: half an ulp of the row and half an ulp of the term
            err = np.abs(f(t[b, j]) - want)
            assert np.all(err <= 2 ** -8 * np.abs(want) + 2 ** -8 * np.abs(W1[x] @ W2t.T) + 1e-6), (b, j, err.max())


@pytest.mark.gpu
def test_device_target_forward_equals_the_host_one():
    import torch
    from speculative_decoding_draft_markov_gb300 import binding as B
    from speculative_decoding_draft_markov_gb300 import step as S
    wl = I.WORKLOADS["qwen3_4b"].with_(bs=8, V=4096)
    dev = torch.device("cuda")
    inp = I.make_device_inputs(wl, dev)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    buf = S.StepBuffers.allocate(bs, gamma, V, bs * (gamma + 1), inp["U"].dtype, dev)
    B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, wl.seed, 0, buf.tokens, buf.logit_x,
                         buf.lse, buf.ws)
    buf.window.fill_(gamma)
    B.dspark_pack(buf.window, inp["anchor"], buf.tokens, None, buf.cu, buf.ids, buf.req, buf.pos, buf.padded, buf.ws)
    S.markov_target_forward(S.gather_target_forward(inp["target"]), inp["W1"], inp["W2t"])(buf)
    h = {"anchor": inp["anchor"].cpu().numpy(), "W1": inp["W1"].cpu().view(torch.int16).numpy().view(np.uint16),
         "W2t": inp["W2t"].cpu().view(torch.int16).numpy().view(np.uint16),
         "target": inp["target"].cpu().view(torch.int16).numpy().view(np.uint16)}
    want = bench._host_target(h, buf.tokens.cpu().numpy(), "bf16")
    got = buf.packed.cpu().view(torch.int16).numpy().view(np.uint16)
    req, pos = buf.req.cpu().numpy(), buf.pos.cpu().numpy()
    f = I.bf16_bits_to_f32
    for p in range(int(buf.cu[bs])):
        # the two GEMMs accumulate in different orders: a term one ulp apart moves the row by at
        # most that ulp plus one of its own
        np.testing.assert_allclose(f(got[p]), f(want[req[p], pos[p]]), rtol=2 ** -7, atol=2 ** -6 * 0.25)
