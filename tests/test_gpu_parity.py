"""GPU parity: every stage through the C ABI against the oracle on the same seeded inputs.

Small cases span several 128-id vocabulary tiles (two 64-id draft chunks each) with a ragged
tail, including tails that end in either half of a tile; the full-size case uses the
bs=256, gamma=7, V=151936 workload and checks sampled requests one by one."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import inputs as I
from tests.parity import NEAR, TOL, compare_draft, compare_verify, to_np

from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import step as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _dev(host):
    return S.device_inputs_from_host(host)


def _draft_gpu(inp, temperature, seed, step):
    U = inp["U"]
    bs, gamma, V = U.shape
    tok = torch.zeros((bs, gamma), dtype=torch.int32, device="cuda")
    lx = torch.zeros((bs, gamma), dtype=torch.float32, device="cuda")
    lse = torch.zeros_like(lx)
    ws = B.alloc_workspace(bs, gamma, V)
    B.dspark_draft_block(U, inp["W1"], inp["W2t"], inp["anchor"], temperature, seed, step, tok, lx, lse, ws)
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK
    return tok.cpu().numpy(), lx.cpu().numpy(), lse.cpu().numpy()


SMALL = {
    "tiny_fp32": I.WORKLOADS["tiny_fp32"],
    "bf16_ragged": I.WORKLOADS["qwen3_4b"].with_(name="bf16_ragged", bs=5, gamma=3, V=2000, d=64, seed=11),
    "bf16_r64": I.WORKLOADS["qwen3_4b"].with_(name="bf16_r64", bs=9, gamma=4, V=1032, r=64, d=64, seed=12),
    # r = 32 takes the CUDA-core statistics pass in bf16; V = 1000 ends 40 ids into a draft chunk
    "bf16_r32_simt": I.WORKLOADS["qwen3_4b"].with_(name="bf16_r32_simt", bs=7, gamma=3, V=1000, r=32, d=64,
                                                   seed=14),
    "bf16_two_mtiles": I.WORKLOADS["qwen3_4b"].with_(name="bf16_two_mtiles", bs=200, gamma=2, V=3000, r=128,
                                                     d=64, seed=13),
    # the tensor-core pass runs all positions in one persistent launch: the longest block the
    # ABI allows (16 positions, 31 grid barriers) and a single position (no barrier between)
    "bf16_gamma16": I.WORKLOADS["qwen3_4b"].with_(name="bf16_gamma16", bs=150, gamma=16, V=2600, d=64, seed=15),
    "bf16_gamma1": I.WORKLOADS["qwen3_4b"].with_(name="bf16_gamma1", bs=33, gamma=1, V=1800, d=64, seed=16),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
def test_draft_parity_small(name, temperature):
    wl = SMALL[name]
    host = I.make_host_inputs(wl, with_target=False, with_hidden=False)
    inp = _dev(host)
    for step in (0, 5):
        tg, lg, sg = _draft_gpu(inp, temperature, wl.seed, step)
        to, lo, so, mo = O.draft_block(host["U"], host["W1"], host["W2t"], host["anchor"], temperature,
                                       wl.seed, step, dtype=wl.dtype)
        checked, near = compare_draft(tg, lg, sg, to, lo, so, mo, wl.dtype, greedy=temperature == 0.0)
        assert checked >= wl.bs * wl.gamma - near * wl.gamma and near <= 1


@pytest.mark.parametrize("name", ["bf16_ragged", "bf16_r32_simt", "bf16_two_mtiles"])
@pytest.mark.parametrize("temperature", [0.2, 3.0])
def test_draft_parity_far_temperatures(name, temperature):
    """A sharply peaked (tau 0.2: tempered logits up to ~60 in magnitude) and a flat (tau 3.0)
    draft distribution, on both statistics passes; bf16 (at tau 0.2 the fp32 rounding of the
    logits, amplified five times, stays far inside the bf16 tolerance)."""
    wl = SMALL[name]
    host = I.make_host_inputs(wl, with_target=False, with_hidden=False)
    inp = _dev(host)
    for step in (0, 3):
        tg, lg, sg = _draft_gpu(inp, temperature, wl.seed, step)
        to, lo, so, mo = O.draft_block(host["U"], host["W1"], host["W2t"], host["anchor"], temperature,
                                       wl.seed, step, dtype=wl.dtype)
        checked, near = compare_draft(tg, lg, sg, to, lo, so, mo, wl.dtype)
        assert checked >= wl.bs * wl.gamma - near * wl.gamma and near <= 1


@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_ragged", "bf16_r32_simt", "bf16_two_mtiles", "bf16_gamma16",
                                  "mixed_bs256", "dsv4_bs256"])
@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_draft_confidence_block_equals_the_two_calls(name, temperature):
    """dspark_draft_confidence_block = dspark_draft_block then dspark_confidence, bit for bit: on the
    tensor-core pass the confidence head runs inside the draft's launch (a warp of each CTA, in the
    confidence kernel's summation order), on the CUDA-core pass as its own launch."""
    # full shapes: d 4096 (two h parts of 8 groups a lane) and d 7168, gamma 5 (14 groups a part)
    wl = {"mixed_bs256": I.WORKLOADS["mixed_bs256"],
          "dsv4_bs256": I.WORKLOADS["dsv4_sweep"].with_(bs=256)}.get(name) or SMALL[name]
    inp = I.make_device_inputs(wl, "cuda", with_target=False)
    bs, gamma, V = wl.bs, wl.gamma, wl.V

    def outs():
        return ([torch.zeros((bs, gamma), dtype=torch.int32, device="cuda")] +
                [torch.zeros((bs, gamma), dtype=torch.float32, device="cuda") for _ in range(5)])

    ws = B.alloc_workspace(bs, gamma, V)
    a = outs()
    B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], temperature, wl.seed, 6, a[0], a[1], a[2], ws)
    B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], a[0], inp["w"], inp["b"], inp["sts_T"], a[3], a[4],
                        z_logit=a[5])
    f = outs()
    B.dspark_draft_confidence_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], temperature, wl.seed, 6, f[0], f[1],
                                    f[2], inp["h"], inp["w"], inp["b"], inp["sts_T"], f[3], f[4], ws, z_logit=f[5])
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK
    for x, y, what in zip(a, f, ["tokens", "logit_x", "lse", "conf", "surv", "z"]):
        assert torch.equal(x, y), what


def test_draft_parity_full_size_sampled_rows():
    wl = I.WORKLOADS["mixed_bs256"]
    inp = I.make_device_inputs(wl, "cuda", with_target=False, with_hidden=False)
    rows = np.array([0, 84, 85, 200, 255])
    for temperature in (1.0, 0.0):
        tg, lg, sg = _draft_gpu(inp, temperature, wl.seed, 3)
        U = to_np(inp["U"][torch.as_tensor(rows, device="cuda")])
        to, lo, so, mo = O.draft_block(U, to_np(inp["W1"]), to_np(inp["W2t"]), to_np(inp["anchor"])[rows],
                                       temperature, wl.seed, 3, dtype="bf16", req_ids=rows)
        compare_draft(tg[rows], lg[rows], sg[rows], to, lo, so, mo, "bf16", greedy=temperature == 0.0)


def test_draft_parity_long_vocabulary_sampled_rows():
    """V = 213000 (1665 vocabulary tiles, ragged last tile) at bs = 136: a tensor-core CTA
    takes 22 tiles, more than its warp sets draw Gumbels for up front, and the second
    128-request M-tile is ragged."""
    wl = I.WORKLOADS["mixed_bs256"].with_(name="long_vocab", bs=136, gamma=2, V=213000, seed=21)
    inp = I.make_device_inputs(wl, "cuda", with_target=False, with_hidden=False)
    rows = np.array([0, 67, 127, 128, 135])
    for temperature in (1.0, 0.0):
        tg, lg, sg = _draft_gpu(inp, temperature, wl.seed, 9)
        U = to_np(inp["U"][torch.as_tensor(rows, device="cuda")])
        to, lo, so, mo = O.draft_block(U, to_np(inp["W1"]), to_np(inp["W2t"]), to_np(inp["anchor"])[rows],
                                       temperature, wl.seed, 9, dtype="bf16", req_ids=rows)
        compare_draft(tg[rows], lg[rows], sg[rows], to, lo, so, mo, "bf16", greedy=temperature == 0.0)


# d 4096 and 7168 (the benchmark's and DSV4's hidden sizes; two h parts at gamma <= 8) and
# gamma 16 (one part)
@pytest.mark.parametrize("name,d", [("tiny_fp32", 64), ("bf16_ragged", 4096), ("bf16_ragged", 7168),
                                    ("bf16_gamma16", 4096)])
def test_confidence_parity(name, d):
    wl = SMALL[name].with_(d=d, bs=24)
    host = I.make_host_inputs(wl, with_target=False)
    tokens = I.random_tokens(wl.bs, wl.gamma, wl.V, 5)
    inp = _dev(host)
    conf = torch.zeros((wl.bs, wl.gamma), dtype=torch.float32, device="cuda")
    surv = torch.zeros_like(conf)
    B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], torch.as_tensor(tokens, device="cuda"),
                        inp["w"], 0.25, inp["sts_T"], conf, surv)
    c_o, a_o, _ = O.confidence(host["h"], host["W1"], host["anchor"], tokens, host["w"], 0.25,
                               host["sts_T"], dtype=wl.dtype)
    tol = TOL[wl.dtype]
    np.testing.assert_allclose(conf.cpu().numpy(), c_o, rtol=tol, atol=0)
    # survival: a product of gamma confidences, held to the same relative tolerance as each one
    np.testing.assert_allclose(surv.cpu().numpy(), a_o, rtol=tol, atol=0)


def _sched_cases():
    cases = []
    for (bs, gamma, seed, ties, kind) in [(4, 7, 0, False, "tiny"), (256, 7, 1, False, "mixed"),
                                          (256, 7, 2, True, "mixed"), (256, 16, 3, False, "wide"),
                                          (1, 1, 4, False, "one"), (33, 5, 5, True, "steep"),
                                          (128, 15, 6, False, "long"), (64, 7, 7, False, "short"),
                                          (200, 3, 8, False, "unsorted"),
                                          # each sort size: up to 1024, 2048 (merge sort) and 4096
                                          # (bitonic) slots, with and without ties
                                          (205, 5, 9, True, "tiers16"), (256, 5, 10, False, "flat"),
                                          (256, 8, 11, False, "const"), (129, 8, 12, False, "mixed"),
                                          (256, 4, 13, False, "unsorted")]:
        a = I.random_survival(bs, gamma, seed, ties=ties)
        if kind == "unsorted":  # rows not non-increasing: the per-request runs need sorting
            a = np.random.default_rng(seed).random((bs, gamma)).astype(np.float32)
        if kind == "const":     # every key equal: the slot order decides
            a = np.full((bs, gamma), 0.5, dtype=np.float32)
        if kind == "tiny":
            sps = O.build_sps(1.0 + 0.002 * np.arange(65), [])
        elif kind == "steep":
            sps = O.build_sps(1.0 + 0.5 * np.arange(bs * (gamma + 1) + 1), [])
        elif kind == "short":   # table shorter than bs + bs*gamma: K is capped by m_max
            sps = O.build_sps(5.0 + 0.01 * np.arange(200), list(range(16, 200, 16)) + [199])
        elif kind == "flat":    # constant step time: the global search admits every slot
            sps = O.build_sps(np.full(bs * (gamma + 1) + 1, 5.0), [])
        else:
            m = bs * (gamma + 1)
            step = 64 if kind in ("mixed", "const") else 16
            sps = O.build_sps(5.0 + 0.01 * np.arange(m + 1), list(range(step, m, step)) + [m])
        cases.append((a, sps))
    return cases


@pytest.mark.parametrize("mode", [O.EARLY_STOP, O.GLOBAL_ARGMAX])
def test_schedule_bit_exact(mode):
    for a, sps in _sched_cases():
        bs, gamma = a.shape
        win = torch.zeros(bs, dtype=torch.int32, device="cuda")
        K = torch.zeros(1, dtype=torch.int32, device="cuda")
        th = torch.zeros(1, dtype=torch.float64, device="cuda")
        ws = B.alloc_workspace(bs, gamma, 1024)
        B.dspark_schedule(torch.as_tensor(a, device="cuda"), torch.as_tensor(sps, device="cuda"), mode, win, K, th,
                          ws)
        assert B.dspark_read_device_status(ws) == B.DSPARK_OK
        w_o, K_o, th_o, _ = O.schedule(a, sps, mode)
        np.testing.assert_array_equal(win.cpu().numpy(), w_o)
        assert int(K.item()) == K_o
        assert th.item() == th_o  # bit-exact fp64


@pytest.mark.parametrize("static", [False, True])
def test_pack_bit_exact(static):
    for bs, gamma, tier_step, seed in [(4, 7, 0, 0), (256, 7, 64, 1), (20, 7, 16, 2), (128, 15, 128, 3), (1, 5, 16, 4)]:
        win = None if static else I.random_windows(bs, gamma, seed)
        tokens = I.random_tokens(bs, gamma, 1000, seed)
        anchor = I.random_tokens(bs, 1, 1000, seed + 50)[:, 0].copy()
        cap = bs * (gamma + 1) + 64
        tiers = (list(range(tier_step, bs * (gamma + 1), tier_step)) + [bs * (gamma + 1)]) if tier_step else []
        cu_o, ids_o, req_o, pos_o, pad_o = O.pack(win, anchor, tokens, tiers, cap, gamma=gamma)
        t = lambda x: torch.as_tensor(np.asarray(x, dtype=np.int32), device="cuda")
        cu, ids, req, pos = (torch.full((n,), -7, dtype=torch.int32, device="cuda") for n in (bs + 1, cap, cap, cap))
        padded = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = B.alloc_workspace(bs, gamma, 1000)
        B.dspark_pack(None if static else t(win), t(anchor), t(tokens), t(tiers) if tiers else None,
                      cu, ids, req, pos, padded, ws)
        assert B.dspark_read_device_status(ws) == B.DSPARK_OK
        assert int(padded.item()) == pad_o
        np.testing.assert_array_equal(cu.cpu().numpy(), cu_o)
        for g, o in ((ids, ids_o), (req, req_o), (pos, pos_o)):
            np.testing.assert_array_equal(g.cpu().numpy()[:pad_o], o[:pad_o])


def test_pack_device_errors_and_recovery():
    bs, gamma = 6, 4
    t = lambda x: torch.as_tensor(np.asarray(x, dtype=np.int32), device="cuda")
    anchor, tokens = t(np.arange(bs)), t(np.zeros((bs, gamma)))
    cu, ids, req, pos = (torch.zeros(n, dtype=torch.int32, device="cuda") for n in (bs + 1, 64, 64, 64))
    padded = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = B.alloc_workspace(bs, gamma, 64)
    B.dspark_pack(t([1, 2, 9, 0, 0, 0]), anchor, tokens, None, cu, ids, req, pos, padded, ws)   # window > gamma
    assert B.dspark_read_device_status(ws) == B.DSPARK_EINVAL and padded.item() == -1
    B.dspark_pack(t([4] * bs), anchor, tokens, t([8, 16]), cu, ids, req, pos, padded, ws)      # M = 30 > 16
    assert B.dspark_read_device_status(ws) == B.DSPARK_EINVAL
    B.dspark_pack(t([1] * bs), anchor, tokens, t([8, 16]), cu, ids, req, pos, padded, ws)      # fine again
    assert B.dspark_read_device_status(ws) == B.DSPARK_OK and padded.item() == 16
    # tiers not strictly increasing (a repeat, a decrease) or not positive
    for bad in ([8, 8, 16], [16, 8, 32], [0, 16], [-4, 16]):
        padded.fill_(7)
        B.dspark_pack(t([1] * bs), anchor, tokens, t(bad), cu, ids, req, pos, padded, ws)
        assert B.dspark_read_device_status(ws) == B.DSPARK_EINVAL, bad
        assert padded.item() == -1


def test_schedule_rejects_a_table_that_increases():
    """A cost table whose entries rise with M (or are negative / not finite) is reported by every
    scheduler entry point that searches it; a table from dspark_build_sps never is."""
    bs, gamma = 16, 4
    a = I.random_survival(bs, gamma, 3)
    surv = torch.as_tensor(a, device="cuda")
    m = bs * (gamma + 1)
    good = O.build_sps(5.0 + 0.01 * np.arange(m + 1), [])
    t = lambda x: torch.as_tensor(np.asarray(x, dtype=np.int32), device="cuda")
    win = torch.zeros(bs, dtype=torch.int32, device="cuda")
    K = torch.zeros(1, dtype=torch.int32, device="cuda")
    th = torch.zeros(1, dtype=torch.float64, device="cuda")
    cu = torch.zeros(bs + 1, dtype=torch.int32, device="cuda")
    ids, req, pos = (torch.zeros(m, dtype=torch.int32, device="cuda") for _ in range(3))
    padded = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = B.alloc_workspace(bs, gamma, 1024)
    anchor, tokens = t(np.arange(bs)), t(np.zeros((bs, gamma)))
    bads = []
    for where, val in ((bs + 3, 1.0), (bs, -1.0), (bs + 7, np.inf), (bs + 1, np.nan)):
        b = good.copy()
        b[where] = val if val != 1.0 else b[where - 1] * 1.001  # one entry above the one before
        bads.append(b)
    for sps_h, expect in [(good, B.DSPARK_OK)] + [(b, B.DSPARK_EINVAL) for b in bads]:
        sps = torch.as_tensor(sps_h, device="cuda")
        B.dspark_schedule(surv, sps, B.DSPARK_SCHED_GLOBAL_ARGMAX, win, K, th, ws)
        assert B.dspark_read_device_status(ws) == expect
        B.dspark_schedule_pack(surv, sps, B.DSPARK_SCHED_EARLY_STOP, win, K, th, anchor, tokens, None, cu, ids, req,
                               pos, padded, ws)
        assert B.dspark_read_device_status(ws) == expect
        ring = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        B.dspark_schedule_zos_select(surv, sps, ring, 0, win, K, ws)   # empty ring: the global search
        assert B.dspark_read_device_status(ws) == expect
        B.dspark_schedule_zos_budget(surv, sps, ring, 0, ws)
        assert B.dspark_read_device_status(ws) == expect


def _verify_chain(wl, temperature, mode, windows_seed, step=0, windows=None):
    """GPU: draft -> pack(generator windows, or the given ones) -> gather target -> verify;
    oracle: the same chain."""
    host = I.make_host_inputs(wl, with_hidden=False)
    inp = _dev(host)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    tg, lg, sg = _draft_gpu(inp, temperature, wl.seed, step)
    to, lo, so, mo = O.draft_block(host["U"], host["W1"], host["W2t"], host["anchor"], temperature, wl.seed,
                                   step, dtype=wl.dtype)
    win = I.random_windows(bs, gamma, windows_seed) if windows is None else np.asarray(windows, np.int32)
    pack_win = win if mode == O.COMPACT else None
    cap = bs * (gamma + 1)
    # oracle chain
    cu_o, ids_o, req_o, pos_o, pad_o = O.pack(pack_win, host["anchor"], to, [], cap)
    packed_o = I.gather_packed_target(host["target"], req_o, pos_o, cap)
    out_o, acc_o, ceil_o, mv_o = O.verify(packed_o, cu_o, win, mode, host["anchor"], to, lo, so, host["U"],
                                          host["W1"], host["W2t"], temperature, wl.seed, step, dtype=wl.dtype)
    # GPU chain
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype)
    buf.tokens.copy_(torch.as_tensor(tg, device="cuda"))
    buf.logit_x.copy_(torch.as_tensor(lg, device="cuda"))
    buf.lse.copy_(torch.as_tensor(sg, device="cuda"))
    buf.window.copy_(torch.as_tensor(win, device="cuda"))
    B.dspark_pack(buf.window if mode == O.COMPACT else None, inp["anchor"], buf.tokens, None, buf.cu, buf.ids,
                  buf.req, buf.pos, buf.padded, buf.ws)
    S.gather_target_forward(inp["target"])(buf)
    S.verify(inp, buf, temperature, wl.seed, step, mode)
    assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
    # requests whose draft diverged at a near-margin decision are excluded from the verify check
    div = np.array([not np.array_equal(tg[r], to[r]) for r in range(bs)])
    for r in np.nonzero(div)[0]:
        assert mo[r].min() < NEAR
    keep = ~div
    ceil_g = buf.ceiling.cpu().numpy() if mode == O.CAP_ACCEPT else None
    checked, near = compare_verify(buf.out_tokens.cpu().numpy()[keep], buf.acc_len.cpu().numpy()[keep],
                                   out_o[keep], acc_o[keep], mv_o[keep],
                                   ceil_g[keep] if ceil_g is not None else None,
                                   ceil_o[keep] if ceil_g is not None else None)
    return checked, near, acc_o


VERIFY_WL = {
    "tiny_fp32": I.WORKLOADS["tiny_fp32"].with_(bs=12),
    "bf16_ragged": SMALL["bf16_ragged"].with_(bs=16, gamma=5, sigmas=(0.3, 1.0, 3.0)),
    # two request tiles (the second ragged), the longest block, a ragged last vocabulary chunk
    "bf16_two_mtiles_g16": SMALL["bf16_two_mtiles"].with_(name="bf16_two_mtiles_g16", bs=200, gamma=16,
                                                          sigmas=(0.3, 1.0, 3.0)),
}


@pytest.mark.parametrize("name", list(VERIFY_WL))
@pytest.mark.parametrize("mode", [O.STATIC, O.COMPACT, O.CAP_ACCEPT])
@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
def test_verify_chain_parity(name, mode, temperature):
    wl = VERIFY_WL[name]
    total_checked = 0
    for step, ws in ((0, 1), (1, 2), (2, 3)):
        checked, near, acc_o = _verify_chain(wl, temperature, mode, ws, step)
        assert near <= 1
        total_checked += checked
    assert total_checked >= 3 * wl.bs - 3


@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_ragged"])
@pytest.mark.parametrize("mode", [O.COMPACT, O.CAP_ACCEPT])
@pytest.mark.parametrize("fill", ["none", "all"])
@pytest.mark.parametrize("temperature", [1.0, 0.7, 0.0])
def test_verify_degenerate_windows(name, mode, fill, temperature):
    """The scheduler's two extremes: no slot admitted (every request packs its anchor row alone
    and commits the bonus draw of row 0; cap-accept still tests the whole block for its ceiling)
    and every slot admitted (the compact layout is then the static one)."""
    wl = VERIFY_WL[name]
    win = np.full(wl.bs, 0 if fill == "none" else wl.gamma, dtype=np.int32)
    checked = 0
    for step in (0, 1):
        c, near, acc_o = _verify_chain(wl, temperature, mode, None, step, windows=win)
        assert near <= 1
        checked += c
        if fill == "none":
            assert (acc_o == 0).all()
    assert checked >= 2 * wl.bs - 2


@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_ragged"])
@pytest.mark.parametrize("mode", [O.STATIC, O.COMPACT])
@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_verify_draft_equal_to_target_accepts_everything(name, mode, temperature):
    """The degenerate draft p_d = p_t: the caller's draft logits are the target rows themselves, so
    every tested token passes (u < p_t / p_d = 1) and the extra token is the bonus draw of the
    row after the window -- on the GPU as in the oracle, except where |u - p_t / p_d| < 1e-4 (the
    two sides round the row statistics differently)."""
    wl = VERIFY_WL[name]
    host = I.make_host_inputs(wl, with_hidden=False)
    inp = _dev(host)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    D_host = np.ascontiguousarray(host["target"][:, :gamma])  # row k - 1 scores position k
    Df = O.to_f64(D_host, wl.dtype)
    D_dev = inp["target"][:, :gamma].contiguous()
    rng = np.random.default_rng(78)
    Dt = Df / temperature
    m = Dt.max(-1, keepdims=True)
    lse = np.log(np.exp(Dt - m).sum(-1)) + m[..., 0]
    p = np.exp(Dt - lse[..., None])
    tok = np.array([[rng.choice(V, p=p[b, k] / p[b, k].sum()) for k in range(gamma)] for b in range(bs)], np.int32)
    lx = np.take_along_axis(Dt, tok[..., None].astype(np.int64), -1)[..., 0].astype(np.float32)
    lse = lse.astype(np.float32)
    win = I.random_windows(bs, gamma, 124)
    pack_win = win if mode == O.COMPACT else None
    cap = bs * (gamma + 1)
    cu_o, ids_o, req_o, pos_o, pad_o = O.pack(pack_win, host["anchor"], tok, [], cap)
    packed_o = I.gather_packed_target(host["target"], req_o, pos_o, cap)
    commit = win if mode == O.COMPACT else np.full(bs, gamma, dtype=np.int32)
    checked = near = 0
    for step in range(2):
        out_o, acc_o, _, mv_o = O.verify(packed_o, cu_o, win, mode, host["anchor"], tok, lx, lse, None, None, None,
                                         temperature, wl.seed, step, dtype=wl.dtype, draft_logits=D_host)
        sure = mv_o >= NEAR
        np.testing.assert_array_equal(acc_o[sure], commit[sure])
        buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype)
        buf.tokens.copy_(torch.as_tensor(tok, device="cuda"))
        buf.logit_x.copy_(torch.as_tensor(lx, device="cuda"))
        buf.lse.copy_(torch.as_tensor(lse, device="cuda"))
        buf.window.copy_(torch.as_tensor(win, device="cuda"))
        B.dspark_pack(buf.window if mode == O.COMPACT else None, inp["anchor"], buf.tokens, None, buf.cu, buf.ids,
                      buf.req, buf.pos, buf.padded, buf.ws)
        S.gather_target_forward(inp["target"])(buf)
        B.dspark_verify(buf.packed, buf.cu, buf.window, mode, inp["anchor"], buf.tokens, buf.logit_x, buf.lse,
                        None, None, None, temperature, wl.seed, step, buf.out_tokens, buf.acc_len, buf.ceiling,
                        buf.ws, draft_logits=D_dev)
        assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
        c, n = compare_verify(buf.out_tokens.cpu().numpy(), buf.acc_len.cpu().numpy(), out_o, acc_o, mv_o)
        checked += c
        near += n
    assert near <= 1 and checked >= 2 * bs - 1


@pytest.mark.parametrize("name", list(VERIFY_WL))
@pytest.mark.parametrize("mode", [O.STATIC, O.COMPACT])
@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_verify_with_explicit_draft_logits(name, mode, temperature):
    """dspark_verify given the draft's logits (no U / W1 / W2t): the residual's p_d comes from
    them.  The logits here are a fresh draw (not a Markov head), with logit_x / lse taken from
    them, so the test covers a drafter whose distribution the library never computes."""
    wl = VERIFY_WL[name]
    host = I.make_host_inputs(wl, with_hidden=False)
    inp = _dev(host)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    rng = np.random.default_rng(77)
    D64 = rng.normal(0.0, 3.0, size=(bs, gamma, V))
    if wl.dtype == "bf16":
        D_host = I.f32_to_bf16_bits(D64.astype(np.float32))
        Df = O.to_f64(D_host, "bf16")
        D_dev = torch.as_tensor(D_host.view(np.int16), device="cuda").view(torch.bfloat16)
    else:
        D_host = D64.astype(np.float32)
        Df = D_host.astype(np.float64)
        D_dev = torch.as_tensor(D_host, device="cuda")
    # draft tokens drawn from softmax(D / T); logit_x / lse consistent with D at temperature T
    Dt = Df / temperature
    m = Dt.max(-1, keepdims=True)
    lse = (np.log(np.exp(Dt - m).sum(-1)) + m[..., 0])
    p = np.exp(Dt - lse[..., None])
    tok = np.array([[rng.choice(V, p=p[b, k] / p[b, k].sum()) for k in range(gamma)] for b in range(bs)], np.int32)
    lx = np.take_along_axis(Dt, tok[..., None].astype(np.int64), -1)[..., 0]
    lx, lse = lx.astype(np.float32), lse.astype(np.float32)
    win = I.random_windows(bs, gamma, 123)
    pack_win = win if mode == O.COMPACT else None
    cap = bs * (gamma + 1)
    cu_o, ids_o, req_o, pos_o, pad_o = O.pack(pack_win, host["anchor"], tok, [], cap)
    packed_o = I.gather_packed_target(host["target"], req_o, pos_o, cap)
    checked = near = 0
    for step in range(3):
        out_o, acc_o, _, mv_o = O.verify(packed_o, cu_o, win, mode, host["anchor"], tok, lx, lse, None, None, None,
                                         temperature, wl.seed, step, dtype=wl.dtype, draft_logits=D_host)
        buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype)
        buf.tokens.copy_(torch.as_tensor(tok, device="cuda"))
        buf.logit_x.copy_(torch.as_tensor(lx, device="cuda"))
        buf.lse.copy_(torch.as_tensor(lse, device="cuda"))
        buf.window.copy_(torch.as_tensor(win, device="cuda"))
        B.dspark_pack(buf.window if mode == O.COMPACT else None, inp["anchor"], buf.tokens, None, buf.cu, buf.ids,
                      buf.req, buf.pos, buf.padded, buf.ws)
        S.gather_target_forward(inp["target"])(buf)
        B.dspark_verify(buf.packed, buf.cu, buf.window, mode, inp["anchor"], buf.tokens, buf.logit_x, buf.lse,
                        None, None, None, temperature, wl.seed, step, buf.out_tokens, buf.acc_len, buf.ceiling,
                        buf.ws, draft_logits=D_dev)
        assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
        c, n = compare_verify(buf.out_tokens.cpu().numpy(), buf.acc_len.cpu().numpy(), out_o, acc_o, mv_o)
        checked += c
        near += n
    assert near <= 1 and checked >= 3 * bs - 1
