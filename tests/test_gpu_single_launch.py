"""The single-launch draft (all positions in one cooperative kernel with grid barriers) against
the stage-by-stage draft (one vocabulary pass and one select launch per position).

The two run the same arithmetic in the same order, so the drawn tokens are identical and
logit_x / lse agree to the last bits; dspark_draft_block_noalloc always runs stage by stage,
which makes it the comparison.  Shapes: the full mixed batch, a ragged long vocabulary (more
tiles per CTA than the Gumbels drawn up front), one M-tile, greedy and sampled."""
import ctypes

import numpy as np
import pytest

from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = {
    "mixed_bs256": I.WORKLOADS["mixed_bs256"],
    "long_vocab_bs136": I.WORKLOADS["mixed_bs256"].with_(name="lv", bs=136, gamma=3, V=213000, seed=41),
    "one_mtile_bs40": I.WORKLOADS["qwen3_4b"].with_(name="one", bs=40, gamma=4, V=20000, seed=42),
}


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("name", list(CASES))
def test_single_launch_equals_stage_by_stage(name):
    wl = CASES[name]
    inp = I.make_device_inputs(wl, "cuda", with_target=False, with_hidden=False)
    U, W1, W2t, anchor = inp["U"], inp["W1"], inp["W2t"], inp["anchor"]
    bs, gamma, V = U.shape
    r = W1.shape[1]
    assert B.dspark_draft_single_launch(B.DSPARK_BF16, bs, gamma, V, r)
    ws = B.alloc_workspace(bs, gamma, V)
    L = B.lib()
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for temperature, step in [(1.0, 3), (0.0, 4), (0.7, 5)]:
        one = [torch.zeros((bs, gamma), dtype=t, device="cuda") for t in (torch.int32, torch.float32, torch.float32)]
        stg = [torch.full((bs, gamma), -5, dtype=t, device="cuda") for t in (torch.int32, torch.float32, torch.float32)]
        B.dspark_draft_block(U, W1, W2t, anchor, temperature, wl.seed, step, *one, ws)
        rc = L.dspark_draft_block_noalloc(_ptr(U), _ptr(W1), _ptr(W2t), B.DSPARK_BF16, _ptr(anchor), bs, gamma, V, r,
                                          ctypes.c_float(temperature), wl.seed, step, _ptr(stg[0]), _ptr(stg[1]),
                                          _ptr(stg[2]), _ptr(status), ctypes.c_void_p(stream))
        assert rc == B.DSPARK_OK
        torch.cuda.synchronize()
        assert B.dspark_read_device_status(ws) == B.DSPARK_OK and int(status.item()) == 0
        np.testing.assert_array_equal(one[0].cpu().numpy(), stg[0].cpu().numpy())
        for a, b in zip(one[1:], stg[1:]):
            np.testing.assert_allclose(a.cpu().numpy(), b.cpu().numpy(), rtol=1e-6, atol=1e-6)
