"""Device-side failure detection without a GPU fault: the tensor-core draft kernel's bounded
waits are made to run out (a 1 ns deadline), the kernel records DSPARK_ETIMEOUT, drains its own
copies and MMAs, frees its tensor memory and returns; the context stays usable and the next call
with the normal deadline is correct again."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from tests.parity import compare_draft

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
