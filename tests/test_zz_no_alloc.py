"""dspark_draft_block_noalloc: the draft for callers that cannot allocate device memory.

Such callers (a plugin living inside another framework's device-memory pool, or a service
whose device footprint is fixed at start-up) have no workspace to hand over, so this entry
point takes its scratch from a fixed array inside the library.  These tests call it through
the C ABI and check it against dspark_draft_block (same kernels, caller-owned workspace) on
two calls in a row -- the second call finds the first call's contents still in the shared
array -- and check that sizes beyond the array are refused.  This file is collected last."""
import ctypes

import numpy as np
import pytest

from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import build as BUILD
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from tests.parity import TOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = {
    "bf16": I.WORKLOADS["qwen3_4b"].with_(name="noalloc_bf16", bs=24, gamma=5, V=4104, d=64, seed=31),
    "f32": I.WORKLOADS["tiny_fp32"].with_(name="noalloc_f32", bs=6, seed=32),
}


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_draft_matches_workspace_draft_on_two_calls(name):
    BUILD.build()
    L = B.lib()
    wl = CASES[name]
    inp = S.device_inputs_from_host(I.make_host_inputs(wl, with_target=False, with_hidden=False))
    U, W1, W2t, anchor = inp["U"], inp["W1"], inp["W2t"], inp["anchor"]
    bs, gamma, V = U.shape
    r = W1.shape[1]
    dt = B.DSPARK_F32 if U.dtype == torch.float32 else B.DSPARK_BF16
    stream = torch.cuda.current_stream().cuda_stream
    ws = B.alloc_workspace(bs, gamma, V)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tol = TOL[wl.dtype]
    for call, (temperature, step) in enumerate([(1.0, 3), (0.8, 4)]):  # two calls in a row
        ref = [torch.zeros((bs, gamma), dtype=t, device="cuda") for t in (torch.int32, torch.float32, torch.float32)]
        got = [torch.full((bs, gamma), -5, dtype=t, device="cuda") for t in (torch.int32, torch.float32, torch.float32)]
        B.dspark_draft_block(U, W1, W2t, anchor, temperature, wl.seed, step, *ref, ws)
        rc = L.dspark_draft_block_noalloc(_ptr(U), _ptr(W1), _ptr(W2t), dt, _ptr(anchor), bs, gamma, V, r,
                                          ctypes.c_float(temperature), wl.seed, step, _ptr(got[0]), _ptr(got[1]),
                                          _ptr(got[2]), _ptr(status), ctypes.c_void_p(stream))
        assert rc == B.DSPARK_OK, B.dspark_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
        for g, rf in zip(got[1:], ref[1:]):
            np.testing.assert_allclose(g.cpu().numpy(), rf.cpu().numpy(), rtol=tol, atol=tol)
    # the library's own status word path (device_status = NULL) also works
    rc = L.dspark_draft_block_noalloc(_ptr(U), _ptr(W1), _ptr(W2t), dt, _ptr(anchor), bs, gamma, V, r,
                                      ctypes.c_float(1.0), wl.seed, 5, _ptr(got[0]), _ptr(got[1]), _ptr(got[2]),
                                      None, ctypes.c_void_p(stream))
    assert rc == B.DSPARK_OK
    torch.cuda.synchronize()
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    BUILD.build()
    L = B.lib()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    # bs = 256 and V = 2^23 need 256 * 65536 * 8 bytes of statistics, far beyond the array
    rc = L.dspark_draft_block_noalloc(fake, fake, fake, B.DSPARK_BF16, fake, 256, 7, 1 << 23, 256,
                                      ctypes.c_float(1.0), 0, 0, fake, fake, fake, None, None)
    assert rc == B.DSPARK_EUNSUPPORTED
