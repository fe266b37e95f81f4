"""The host-to-device packed-row copy helper reproduces, byte for byte, the rows a packed
verify batch reads (the device gather of the same rows), and a step fed by it verifies the
same tokens as a step fed by the gather."""
import numpy as np
import pytest

from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_copied_rows_equal_the_gather():
    wl = I.WORKLOADS["qwen3_4b"].with_(name="copy_rows", bs=37, gamma=5, V=3000, d=64, seed=31)
    dev = torch.device("cuda")
    inp = I.make_device_inputs(wl, dev)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    cap = int(I.tiers_for(wl)[-1])
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype, dev)
    sps = S.sps_table(inp["T_raw"], inp["tiers"], dev)
    S.draft_and_schedule(inp, buf, sps, wl.temperature, wl.seed, 0, B.DSPARK_SCHED_GLOBAL_ARGMAX)
    S.gather_target_forward(inp["target"])(buf)
    want = buf.packed.clone()
    cu = buf.cu.cpu()
    M = int(cu[bs])
    assert 0 < M <= cap
    buf.packed.zero_()
    host = inp["target"].cpu().pin_memory()
    B.dspark_copy_packed_rows_async(buf.packed, host, cu)
    torch.cuda.synchronize()
    assert torch.equal(buf.packed[:M], want[:M])
