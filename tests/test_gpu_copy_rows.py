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


def test_runs_of_equal_row_counts():
    """Hand-made packings with runs of equal row counts (strided copies), lone requests and
    empty ones: every packed row holds its request's row."""
    bs, rpr, V = 12, 6, 200
    host = torch.randn(bs, rpr, V).to(torch.bfloat16).pin_memory()
    for counts in ([1, 1, 1, 3, 3, 0, 0, 2, 1, 1, 6, 6], [2] * 12, [0, 4, 1, 4, 1, 0, 5, 5, 5, 1, 0, 3]):
        n = torch.tensor(counts, dtype=torch.int32)
        cu = torch.zeros(bs + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(n, 0)
        M = int(cu[-1])
        packed = torch.zeros((M + 3, V), dtype=torch.bfloat16, device="cuda")
        B.dspark_copy_packed_rows_async(packed, host, cu)
        torch.cuda.synchronize()
        want = torch.cat([host[r, :counts[r]] for r in range(bs)]) if M else host[:0, 0]
        assert torch.equal(packed[:M].cpu(), want)
        assert not packed[M:].any()
