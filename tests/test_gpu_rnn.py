"""GPU parity of the RNN sequential head through the C ABI (dspark_draft_block_rnn, and
dspark_verify with the draft's states) against the oracle (rnn_draft_block, verify with
draft_states) on the same seeded inputs.

States: fp32 within 1e-5 relative; bf16 states are rounded to nearest even after every update
on both sides (the GPU from its fp32 update, the oracle from fp64), so a value that sits within
the fp32 error of a rounding boundary may land one bf16 step apart, and the recurrence carries
that step on: at most 2 % of the elements may differ, each within 2^-6 of its row's largest
magnitude, everything else equal.  Tokens and accepted lengths: bit-exact except at
near-margin decisions (< 1e-4), as for the Markov head."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from tests.parity import NEAR, compare_draft, compare_verify, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = {
    "tiny_fp32": I.WORKLOADS["tiny_fp32"].with_(bs=9),
    "bf16_tc_ragged": I.WORKLOADS["qwen3_4b"].with_(name="rnn_bf16", bs=20, gamma=5, V=3000, d=64, seed=51),
    "bf16_r32_simt": I.WORKLOADS["qwen3_4b"].with_(name="rnn_r32", bs=11, gamma=4, V=1000, r=32, d=64, seed=52),
    "bf16_two_mtiles": I.WORKLOADS["qwen3_4b"].with_(name="rnn_2mt", bs=150, gamma=3, V=2000, r=128, d=64,
                                                    seed=53),
}


def _rnn_gpu(inp, temperature, seed, step, bg=None):
    U = inp["U"]
    bs, gamma, V = U.shape
    r = inp["W1"].shape[1]
    tok = torch.zeros((bs, gamma), dtype=torch.int32, device="cuda")
    lx = torch.zeros((bs, gamma), dtype=torch.float32, device="cuda")
    lse = torch.zeros_like(lx)
    st = torch.full((bs, gamma, r), 7.0, dtype=U.dtype, device="cuda")
    ws = B.alloc_workspace(bs, gamma, V)
    B.dspark_draft_block_rnn(U, inp["W1"], inp["W2t"], inp["Wg"], inp["bg"] if bg is None else bg, inp["anchor"],
                             temperature, seed, step, tok, lx, lse, st, ws)
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK
    return tok, lx, lse, st


def _check_states(st_g, st_o, tok_g, tok_o, dtype):
    """States of the positions whose prefix agrees (s_k depends on x_0 .. x_{k-1})."""
    bs, gamma = tok_o.shape
    g = to_np(st_g)
    g = O.to_f64(g, dtype)
    n = off = 0
    for b in range(bs):
        for k in range(gamma):
            if k > 0 and tok_g[b, k - 1] != tok_o[b, k - 1]:
                break
            a, o = g[b, k], st_o[b, k]
            if dtype == "f32":
                np.testing.assert_allclose(a, o, rtol=1e-5, atol=1e-7)
            else:
                # A value rounded to the other side of a bf16 boundary differs by one step; the
                # recurrence carries such a step into later states (through g s_{k-1}, and into
                # every gate through Wg), where it can be several steps of a smaller value.  So
                # the bound is on the row's scale: 2^-6 of its largest magnitude -- a wrong gate,
                # row or position is off by the state's own size.
                tol = 2.0 ** -6 * np.abs(o).max()
                i = int(np.argmax(np.abs(a - o)))
                assert np.abs(a - o).max() <= tol, (b, k, i, a[i], o[i])
                off += int(np.sum(a != o))
            n += a.size
    assert n > 0 and off <= max(2, n // 50), (off, n)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
def test_rnn_draft_parity(name, temperature):
    wl = CASES[name]
    host = I.make_host_inputs(wl, with_target=False, with_hidden=False, with_rnn=True)
    inp = S.device_inputs_from_host(host)
    for step in (0, 3):
        tok, lx, lse, st = _rnn_gpu(inp, temperature, wl.seed, step)
        to, lo, so, mo, st_o = O.rnn_draft_block(host["U"], host["W1"], host["W2t"], host["Wg"], host["bg"],
                                                 host["anchor"], temperature, wl.seed, step, dtype=wl.dtype)
        tg = tok.cpu().numpy()
        checked, near = compare_draft(tg, lx.cpu().numpy(), lse.cpu().numpy(), to, lo, so, mo, wl.dtype,
                                      greedy=temperature == 0.0)
        assert near <= 1 and checked >= wl.bs * wl.gamma - near * wl.gamma
        _check_states(st, st_o, tg, to, wl.dtype)


@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_tc_ragged"])
def test_rnn_closed_gate_equals_markov_draft(name):
    """With every gate closed (b_g = -inf) the RNN head is the Markov head: the same tokens and
    statistics as dspark_draft_block, bit for bit, and s_k = W1[x_{k-1}]."""
    wl = CASES[name]
    host = I.make_host_inputs(wl, with_target=False, with_hidden=False, with_rnn=True)
    inp = S.device_inputs_from_host(host)
    bg = torch.full((wl.r,), float("-inf"), dtype=torch.float32, device="cuda")
    tok, lx, lse, st = _rnn_gpu(inp, 1.0, wl.seed, 2, bg=bg)
    t2, l2, s2 = (torch.zeros_like(x) for x in (tok, lx, lse))
    ws = B.alloc_workspace(wl.bs, wl.gamma, wl.V)
    B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, wl.seed, 2, t2, l2, s2, ws)
    assert torch.equal(tok, t2) and torch.equal(lx, l2) and torch.equal(lse, s2)
    prev = torch.cat([inp["anchor"][:, None], tok[:, :-1]], dim=1).long()
    assert torch.equal(st, inp["W1"][prev])


@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_tc_ragged", "bf16_two_mtiles"])
@pytest.mark.parametrize("mode", [O.STATIC, O.COMPACT])
@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_rnn_verify_chain_parity(name, mode, temperature):
    """RNN draft -> pack -> target rows -> verify with the draft's states; the oracle verifies the
    GPU's draft (fed forward: tokens, statistics and states), its p_d rows from those states."""
    wl = CASES[name].with_(sigmas=(0.3, 1.0, 3.0))
    host = I.make_host_inputs(wl, with_hidden=False, with_rnn=True)
    inp = S.device_inputs_from_host(host)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    cap = bs * (gamma + 1)
    checked = near = 0
    for step in range(3):
        tok, lx, lse, st = _rnn_gpu(inp, temperature, wl.seed, step)
        win = I.random_windows(bs, gamma, 40 + step)
        buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype)
        buf.tokens.copy_(tok)
        buf.logit_x.copy_(lx)
        buf.lse.copy_(lse)
        buf.window.copy_(torch.as_tensor(win, device="cuda"))
        B.dspark_pack(buf.window if mode == O.COMPACT else None, inp["anchor"], buf.tokens, None, buf.cu, buf.ids,
                      buf.req, buf.pos, buf.padded, buf.ws)
        S.gather_target_forward(inp["target"])(buf)
        S.verify(inp, buf, temperature, wl.seed, step, mode, states=st)
        assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
        tg = tok.cpu().numpy()
        cu, ids, req, pos, padded = O.pack(win if mode == O.COMPACT else None, host["anchor"], tg, [], cap)
        packed = I.gather_packed_target(host["target"], req, pos, cap)
        out_o, acc_o, _, mv_o = O.verify(packed, cu, win, mode, host["anchor"], tg, lx.cpu().numpy(),
                                         lse.cpu().numpy(), host["U"], host["W1"], host["W2t"], temperature,
                                         wl.seed, step, dtype=wl.dtype, draft_states=O.to_f64(to_np(st), wl.dtype))
        c, n = compare_verify(buf.out_tokens.cpu().numpy(), buf.acc_len.cpu().numpy(), out_o, acc_o, mv_o)
        checked += c
        near += n
    assert near <= 1 and checked >= 3 * bs - 1


def test_rnn_full_size_sampled_rows():
    """The mixed-difficulty batch's shapes (bs 256, gamma 7, V 151936, r 256) on the tensor
    cores, sampled requests against the oracle."""
    wl = I.WORKLOADS["mixed_bs256"]
    inp = I.make_device_inputs(wl, "cuda", with_target=False, with_hidden=False, with_rnn=True)
    rows = np.array([0, 100, 129, 255])
    for temperature in (1.0, 0.0):
        tok, lx, lse, st = _rnn_gpu(inp, temperature, wl.seed, 4)
        U = to_np(inp["U"][torch.as_tensor(rows, device="cuda")])
        to, lo, so, mo, st_o = O.rnn_draft_block(U, to_np(inp["W1"]), to_np(inp["W2t"]), to_np(inp["Wg"]),
                                                 to_np(inp["bg"]), to_np(inp["anchor"])[rows], temperature, wl.seed,
                                                 4, dtype="bf16", req_ids=rows)
        tg = to_np(tok)[rows]
        checked, near = compare_draft(tg, to_np(lx)[rows], to_np(lse)[rows], to, lo, so, mo, "bf16",
                                      greedy=temperature == 0.0)
        assert near <= 1
        _check_states(st[torch.as_tensor(rows, device="cuda")], st_o, tg, to, "bf16")
