"""Out-of-bounds write checks without a sanitizer: every output buffer of every entry point, and
the workspace, sit inside a larger allocation whose guard regions (256 bytes before and after)
hold a sentinel pattern; after each call the guards must be intact.  Run at small ragged shapes
and at the benchmark's shapes (bs 256, gamma 7, V 151936)."""
import numpy as np
import pytest

from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I
from speculative_decoding_draft_markov_gb300 import step as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 256  # bytes on each side; keeps 256-byte alignment of the guarded view


class Guarded:
    """A tensor view of `shape` inside an allocation with sentinel-filled guards."""

    def __init__(self, shape, dtype, device="cuda"):
        es = torch.empty(0, dtype=dtype).element_size()
        self.g = GUARD // es
        self.n = int(np.prod(shape)) if len(shape) else 1
        self.big = torch.empty(self.n + 2 * self.g, dtype=dtype, device=device)
        self.big.view(torch.uint8).fill_(0xA5)
        self.t = self.big[self.g:self.g + self.n].view(shape)

    def intact(self) -> bool:
        u8 = self.big.view(torch.uint8)
        gb = self.g * self.big.element_size()
        return bool((u8[:gb] == 0xA5).all()) and bool((u8[u8.numel() - gb:] == 0xA5).all())


def _ws(bs, gamma, V):
    w = Guarded((B.dspark_workspace_bytes(bs, gamma, V),), torch.uint8)
    w.t.zero_()
    return w


def _check(*gs):
    torch.cuda.synchronize()
    for g in gs:
        assert g.intact(), "a guard region was written"


@pytest.mark.parametrize("shape", ["small", "bench"])
def test_step_entry_points_keep_their_bounds(shape):
    wl = (I.WORKLOADS["qwen3_4b"].with_(name="canary", bs=5, gamma=3, V=2000, d=64, seed=21) if shape == "small"
          else I.WORKLOADS["mixed_bs256"])
    dev = torch.device("cuda")
    inp = I.make_device_inputs(wl, dev)
    bs, gamma, V, r = wl.bs, wl.gamma, wl.V, wl.r
    ws = _ws(bs, gamma, V)
    tok, lx, lse = Guarded((bs, gamma), torch.int32), Guarded((bs, gamma), torch.float32), \
        Guarded((bs, gamma), torch.float32)
    B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, 3, 4, tok.t, lx.t, lse.t, ws.t)
    _check(ws, tok, lx, lse)
    assert B.dspark_read_device_status(ws.t) == B.DSPARK_OK
    conf, surv, z = (Guarded((bs, gamma), torch.float32) for _ in range(3))
    B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], tok.t, inp["w"], inp["b"], inp["sts_T"], conf.t, surv.t,
                        z_logit=z.t)
    _check(conf, surv, z)
    # the fused draft + confidence call, into fresh guarded outputs
    f_out = [Guarded((bs, gamma), t) for t in (torch.int32, torch.float32, torch.float32, torch.float32,
                                                 torch.float32, torch.float32)]
    B.dspark_draft_confidence_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], 1.0, 3, 4, f_out[0].t, f_out[1].t,
                                    f_out[2].t, inp["h"], inp["w"], inp["b"], inp["sts_T"], f_out[3].t, f_out[4].t,
                                    ws.t, z_logit=f_out[5].t)
    _check(ws, *f_out)
    assert B.dspark_read_device_status(ws.t) == B.DSPARK_OK
    sps = S.sps_table(inp["T_raw"], inp["tiers"], dev)
    win, K, th = Guarded((bs,), torch.int32), Guarded((1,), torch.int32), Guarded((1,), torch.float64)
    B.dspark_schedule(surv.t, sps, B.DSPARK_SCHED_GLOBAL_ARGMAX, win.t, K.t, th.t, ws.t)
    _check(win, K, th)
    ring = Guarded((2,), torch.int32)
    ring.t.fill_(-1)
    win2, K2 = Guarded((bs,), torch.int32), Guarded((1,), torch.int32)
    for step in range(3):
        B.dspark_schedule_zos_select(surv.t, sps, ring.t, step, win2.t, K2.t, ws.t)
        B.dspark_schedule_zos_budget(surv.t, sps, ring.t, step, ws.t)
    _check(ring, win2, K2)
    cap = bs * (gamma + 1)
    tiers = torch.as_tensor(inp["tiers"], device=dev) if len(inp["tiers"]) else None
    cap = max(cap, int(inp["tiers"][-1])) if len(inp["tiers"]) else cap
    cu, padded = Guarded((bs + 1,), torch.int32), Guarded((1,), torch.int32)
    ids, req, pos = (Guarded((cap,), torch.int32) for _ in range(3))
    for mode in (B.DSPARK_STATIC, B.DSPARK_CAP_ACCEPT, B.DSPARK_COMPACT):
        B.dspark_pack(None if mode != B.DSPARK_COMPACT else win.t, inp["anchor"], tok.t, tiers, cu.t, ids.t, req.t,
                      pos.t, padded.t, ws.t)
        _check(cu, ids, req, pos, padded, ws)
        g1, V_ = gamma + 1, V
        flat = inp["target"].view(bs * g1, V_)
        idx = torch.where(req.t >= 0, req.t * g1 + pos.t, torch.zeros_like(req.t)).long()
        packed = torch.index_select(flat, 0, idx)
        out, acc, ceil = Guarded((bs, gamma + 1), torch.int32), Guarded((bs,), torch.int32), \
            Guarded((bs,), torch.int32)
        for temperature in (1.0, 0.0):
            B.dspark_verify(packed, cu.t, win.t, mode, inp["anchor"], tok.t, lx.t, lse.t, inp["U"], inp["W1"],
                            inp["W2t"], temperature, 5, 6, out.t, acc.t,
                            ceil.t if mode == B.DSPARK_CAP_ACCEPT else None, ws.t)
            _check(out, acc, ceil, ws)
            assert B.dspark_read_device_status(ws.t) == B.DSPARK_OK
        if mode == B.DSPARK_CAP_ACCEPT:
            stats = Guarded((B.alloc_obs_stats().numel(),), torch.int64)
            stats.t.zero_()
            B.dspark_observe(surv.t, win.t, acc.t, ceil.t, 15, stats.t, ws.t)
            _check(stats, ws)
            assert B.dspark_read_device_status(ws.t) == B.DSPARK_OK


def test_temperature_fit_keeps_its_bounds():
    N, gamma, n_grid, n_bins = 5000, 5, 37, 11
    z, c = I.calibration_steps(N, gamma, [1.5] * gamma, seed=3)
    T, e = Guarded((gamma,), torch.float32), Guarded((gamma,), torch.float64)
    ws = Guarded((B.dspark_sts_fit_workspace_bytes(n_grid, n_bins),), torch.uint8)
    grid = torch.linspace(0.5, 3.0, n_grid, device="cuda")
    B.dspark_sts_fit(torch.as_tensor(z, device="cuda"), torch.as_tensor(c, device="cuda"), grid, n_bins, T.t, e.t,
                     ws=ws.t)
    _check(T, e, ws)


@pytest.mark.parametrize("shape", ["small", "bench"])
def test_rnn_head_keeps_its_bounds(shape):
    """The RNN head's draft (states written position by position) and verify reading them."""
    wl = (I.WORKLOADS["qwen3_4b"].with_(name="canary_rnn", bs=5, gamma=3, V=2000, d=64, seed=22) if shape == "small"
          else I.WORKLOADS["mixed_bs256"])
    dev = torch.device("cuda")
    inp = I.make_device_inputs(wl, dev, with_hidden=False, with_rnn=True)
    bs, gamma, V, r = wl.bs, wl.gamma, wl.V, wl.r
    ws = _ws(bs, gamma, V)
    tok, lx, lse = Guarded((bs, gamma), torch.int32), Guarded((bs, gamma), torch.float32), \
        Guarded((bs, gamma), torch.float32)
    st = Guarded((bs, gamma, r), inp["U"].dtype)
    B.dspark_draft_block_rnn(inp["U"], inp["W1"], inp["W2t"], inp["Wg"], inp["bg"], inp["anchor"], 1.0, 3, 4, tok.t,
                             lx.t, lse.t, st.t, ws.t)
    _check(ws, tok, lx, lse, st)
    assert B.dspark_read_device_status(ws.t) == B.DSPARK_OK
    cap = bs * (gamma + 1)
    cu, padded = Guarded((bs + 1,), torch.int32), Guarded((1,), torch.int32)
    ids, req, pos = (Guarded((cap,), torch.int32) for _ in range(3))
    B.dspark_pack(None, inp["anchor"], tok.t, None, cu.t, ids.t, req.t, pos.t, padded.t, ws.t)
    g1 = gamma + 1
    idx = torch.where(req.t >= 0, req.t * g1 + pos.t, torch.zeros_like(req.t)).long()
    packed = torch.index_select(inp["target"].view(bs * g1, V), 0, idx)
    out, acc = Guarded((bs, gamma + 1), torch.int32), Guarded((bs,), torch.int32)
    B.dspark_verify(packed, cu.t, None, B.DSPARK_STATIC, inp["anchor"], tok.t, lx.t, lse.t, inp["U"], inp["W1"],
                    inp["W2t"], 1.0, 5, 6, out.t, acc.t, None, ws.t, draft_states=st.t)
    _check(out, acc, ws, st)
    assert B.dspark_read_device_status(ws.t) == B.DSPARK_OK
