"""dspark_draft_block_noalloc: the draft for callers that cannot allocate device memory.

Such callers (a plugin living inside another framework's device-memory pool, or a service
whose device footprint is fixed at start-up) have no workspace to hand over, so this entry
point takes its scratch from a fixed array inside the library.  These tests call it through
the C ABI and check it against dspark_draft_block (same kernels, caller-owned workspace) on
two calls in a row -- the second call finds the first call's contents still in the shared
array -- at the mixed-difficulty batch's shape (bs 256, V 151936, also against the oracle)
and at large vocabularies, and check that sizes beyond the scratch are refused.
This file is collected last."""
import ctypes

import numpy as np
import pytest

from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import build as BUILD
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S
from oracle import dspark_oracle as O
from tests.parity import TOL, compare_draft, to_np

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
    # the library's own status word path (device_status = NULL): same outputs as the workspace draft
    _compare_with_workspace_draft(L, U, W1, W2t, anchor, 1.0, wl.seed, 5, ws, None, tol)


def _compare_with_workspace_draft(L, U, W1, W2t, anchor, temperature, seed, step, ws, status, tol):
    """One allocation-free call against dspark_draft_block on the same inputs."""
    bs, gamma, V = U.shape
    r = W1.shape[1]
    dt = B.DSPARK_F32 if U.dtype == torch.float32 else B.DSPARK_BF16
    stream = torch.cuda.current_stream().cuda_stream
    ref = [torch.zeros((bs, gamma), dtype=t, device="cuda") for t in (torch.int32, torch.float32, torch.float32)]
    got = [torch.full((bs, gamma), -5, dtype=t, device="cuda") for t in (torch.int32, torch.float32, torch.float32)]
    B.dspark_draft_block(U, W1, W2t, anchor, temperature, seed, step, *ref, ws)
    rc = L.dspark_draft_block_noalloc(_ptr(U), _ptr(W1), _ptr(W2t), dt, _ptr(anchor), bs, gamma, V, r,
                                      ctypes.c_float(temperature), seed, step, _ptr(got[0]), _ptr(got[1]),
                                      _ptr(got[2]), _ptr(status), ctypes.c_void_p(stream))
    assert rc == B.DSPARK_OK, B.dspark_status_string(rc)
    torch.cuda.synchronize()
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK
    if status is not None:
        assert int(status.item()) == 0
    np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
    for g, rf in zip(got[1:], ref[1:]):
        np.testing.assert_allclose(g.cpu().numpy(), rf.cpu().numpy(), rtol=tol, atol=tol)
    return got


# Largest vocabulary the CUDA-core pass accepts at bs = 256: 256 B + 256 * ceil(V / 64) * 16 B
# <= 8 MiB gives ceil(V / 64) <= 2047.  The tensor-core pass writes one slot per CTA (at most one
# per SM), so at bs = 256 it needs 256 * 152 * 16 B whatever V: it has no such limit, and a large
# vocabulary there is checked to run.
V_LARGE_TC, V_MAX_SIMT = 2047 * 128, 2047 * 64


def test_noalloc_headline_shape_against_oracle_rows():
    """bs = 256, V = 151936 in bf16 (the mixed-difficulty batch) is accepted, equals the workspace
    draft, and its sampled requests equal the oracle's draws."""
    BUILD.build()
    L = B.lib()
    wl = I.WORKLOADS["mixed_bs256"].with_(name="noalloc_full", gamma=2, seed=33)
    inp = I.make_device_inputs(wl, "cuda", with_target=False, with_hidden=False)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    ws = B.alloc_workspace(bs, gamma, V)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _compare_with_workspace_draft(L, inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, wl.seed, 2, ws,
                                        status, TOL["bf16"])
    rows = np.array([0, 100, 255])
    U = to_np(inp["U"][torch.as_tensor(rows, device="cuda")])
    to, lo, so, mo = O.draft_block(U, to_np(inp["W1"]), to_np(inp["W2t"]), to_np(inp["anchor"])[rows], 1.0,
                                   wl.seed, 2, dtype="bf16", req_ids=rows)
    g = [to_np(x)[rows] for x in got]
    checked, near = compare_draft(g[0], g[1], g[2], to, lo, so, mo, "bf16")
    assert near <= 1 and checked >= (len(rows) - near) * gamma


@pytest.mark.parametrize("dtype,V", [("bf16", V_LARGE_TC), ("f32", V_MAX_SIMT)])
def test_noalloc_at_large_vocabularies(dtype, V):
    """bs = 256 at the largest vocabulary the CUDA-core pass accepts (f32), and at a vocabulary
    beyond it on the tensor-core pass (bf16), runs and equals the workspace draft."""
    BUILD.build()
    L = B.lib()
    bs, gamma, r = 256, 1, 256 if dtype == "bf16" else 32
    g = torch.Generator(device="cuda")
    g.manual_seed(34)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    U = (torch.randn((bs, gamma, V), device="cuda", generator=g) * 3.0).to(tdt)
    W1 = (torch.randn((V, r), device="cuda", generator=g) * 0.05).to(tdt)
    W2t = (torch.randn((V, r), device="cuda", generator=g) * 0.05).to(tdt)
    anchor = torch.randint(0, V, (bs,), device="cuda", generator=g, dtype=torch.int64).to(torch.int32)
    ws = B.alloc_workspace(bs, gamma, V)
    _compare_with_workspace_draft(L, U, W1, W2t, anchor, 1.0, 34, 0, ws, None, TOL[dtype])


@pytest.mark.parametrize("dtype,V,r", [("f32", V_MAX_SIMT + 8, 32), ("bf16", V_MAX_SIMT + 8, 32),
                                       ("f32", 1 << 23, 256)])
def test_noalloc_rejects_sizes_beyond_its_scratch(dtype, V, r):
    """One vocabulary step past the CUDA-core pass's limit at bs = 256 (fp32, or bf16 with r = 32,
    which takes that pass) is refused before anything runs, and so is a far larger one."""
    BUILD.build()
    L = B.lib()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    dt = B.DSPARK_BF16 if dtype == "bf16" else B.DSPARK_F32
    rc = L.dspark_draft_block_noalloc(fake, fake, fake, dt, fake, 256, 7, V, r,
                                      ctypes.c_float(1.0), 0, 0, fake, fake, fake, None, None)
    assert rc == B.DSPARK_EUNSUPPORTED
