"""Device-side failure detection without a GPU fault: the bounded waits of the tensor-core
kernels (the draft's vocabulary pass, verify's decision pass) are made to run out (a 1 ns
deadline); the kernel records DSPARK_ETIMEOUT, drains its own copies and MMAs, frees its tensor
memory and returns; the context stays usable and the next call with the normal deadline is
correct again."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from tests.parity import compare_draft, compare_verify

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_recovers():
    wl = I.WORKLOADS["qwen3_4b"].with_(name="timeout", bs=40, gamma=3, V=20000, d=64, seed=41)
    host = I.make_host_inputs(wl, with_target=False, with_hidden=False)
    inp = S.device_inputs_from_host(host)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    tok = torch.zeros((bs, gamma), dtype=torch.int32, device="cuda")
    lx = torch.zeros((bs, gamma), dtype=torch.float32, device="cuda")
    lse = torch.zeros_like(lx)
    ws = B.alloc_workspace(bs, gamma, V)
    old = B.dspark_set_wait_timeout_ns(1)
    try:
        B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, wl.seed, 0, tok, lx, lse, ws)
        st = B.dspark_read_device_status(ws)
    finally:
        B.dspark_set_wait_timeout_ns(old)
    assert st == B.DSPARK_ETIMEOUT, B.dspark_status_string(st)
    # the context is usable and the status word was cleared by the read
    B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, wl.seed, 0, tok, lx, lse, ws)
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK
    to, lo, so, mo = O.draft_block(host["U"], host["W1"], host["W2t"], host["anchor"], 1.0, wl.seed, 0)
    compare_draft(tok.cpu().numpy(), lx.cpu().numpy(), lse.cpu().numpy(), to, lo, so, mo, "bf16")


def test_decide_wait_timeout_is_reported_and_recovers():
    """verify's tensor-core decision pass (bf16, r = 256): several vocabulary tiles per CTA so
    that its pipelines are deep when the waits give up."""
    wl = I.WORKLOADS["qwen3_4b"].with_(name="timeout_decide", bs=40, gamma=3, V=60000, d=64, seed=42,
                                       sigmas=(2.0,))
    host = I.make_host_inputs(wl, with_hidden=False)
    inp = S.device_inputs_from_host(host)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    cap = bs * (gamma + 1)
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype)
    B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, wl.seed, 0, buf.tokens, buf.logit_x,
                         buf.lse, buf.ws)
    B.dspark_pack(None, inp["anchor"], buf.tokens, None, buf.cu, buf.ids, buf.req, buf.pos, buf.padded, buf.ws)
    S.gather_target_forward(inp["target"])(buf)
    assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
    old = B.dspark_set_wait_timeout_ns(1)
    try:
        S.verify(inp, buf, 1.0, wl.seed, 0, B.DSPARK_STATIC)
        st = B.dspark_read_device_status(buf.ws)
    finally:
        B.dspark_set_wait_timeout_ns(old)
    assert st == B.DSPARK_ETIMEOUT, B.dspark_status_string(st)
    # usable again: the same verification with the normal deadline equals the oracle's
    S.verify(inp, buf, 1.0, wl.seed, 0, B.DSPARK_STATIC)
    assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
    tok, lx, lse = (buf.tokens.cpu().numpy(), buf.logit_x.cpu().numpy(), buf.lse.cpu().numpy())
    cu, ids, req, pos, padded = O.pack(None, host["anchor"], tok, [], cap)
    packed = I.gather_packed_target(host["target"], req, pos, cap)
    out_o, acc_o, _, mv_o = O.verify(packed, cu, None, O.STATIC, host["anchor"], tok, lx, lse, host["U"], host["W1"],
                                     host["W2t"], 1.0, wl.seed, 0)
    checked, near = compare_verify(buf.out_tokens.cpu().numpy(), buf.acc_len.cpu().numpy(), out_o, acc_o, mv_o)
    assert near <= 1 and checked >= bs - 1
    assert (acc_o < gamma).sum() > bs // 4  # the decision pass had residual rows to work on
