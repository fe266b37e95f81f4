"""GPU parity of the asynchronous (zero-overhead) scheduler through the C ABI: the budget ring,
the radix top-K select and the first-steps fallback, bit-exact against the oracle over
sequences of steps, at the benchmark's sizes and at the edges (one slot, 4096 slots, ties,
K = 0, K beyond the batch, a table shorter than the batch)."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import inputs as I

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _WS():
    """A status-word workspace for the scheduler calls (they use only its first word)."""
    return torch.zeros(256, dtype=torch.uint8, device="cuda")


def _table(bs, gamma, kind):
    m = bs * (gamma + 1)
    if kind == "tiny":
        return O.build_sps(1.0 + 0.002 * np.arange(65), [])
    if kind == "short":    # K capped by m_max - bs
        return O.build_sps(5.0 + 0.01 * np.arange(200), list(range(16, 200, 16)) + [199])
    if kind == "flat":     # the global search admits every slot
        return np.ones(m + 1)
    step = 64 if kind == "sawtooth" else 16
    return O.build_sps(5.0 + 0.01 * np.arange(m + 1), list(range(step, m, step)) + [m])


CASES = [(4, 7, "tiny", False), (256, 7, "sawtooth", False), (256, 7, "sawtooth", True),
         (256, 16, "tiers16", False), (1, 1, "tiers16", False), (33, 5, "tiers16", True),
         (128, 15, "tiers16", False), (64, 7, "short", False), (200, 3, "flat", True)]


def _survival(bs, gamma, seed, ties, t):
    a = I.random_survival(bs, gamma, 1000 * seed + t, ties=ties)
    if t == 3:   # all-equal keys and zeros in one step
        a = np.where(np.arange(gamma)[None, :] < gamma // 2, np.float32(1.0), np.float32(0.0)).repeat(bs, 0)
        a = a.astype(np.float32)
    return a


@pytest.mark.parametrize("case", range(len(CASES)))
def test_zos_sequence_bit_exact(case):
    bs, gamma, kind, ties = CASES[case]
    sps_h = _table(bs, gamma, kind)
    sps = torch.as_tensor(sps_h, device="cuda")
    ring = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    ring_o = [-1, -1]
    win = torch.zeros(bs, dtype=torch.int32, device="cuda")
    K = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(6):
        a = _survival(bs, gamma, case, ties, t)
        surv = torch.as_tensor(a, device="cuda")
        B.dspark_schedule_zos_select(surv, sps, ring, t, win, K, _WS())
        B.dspark_schedule_zos_budget(surv, sps, ring, t, _WS())
        w_o, K_o = O.zos_step(a, sps_h, ring_o, t)
        np.testing.assert_array_equal(win.cpu().numpy(), w_o)
        assert int(K.item()) == K_o, (t, int(K.item()), K_o)
        assert ring.cpu().tolist() == ring_o, (t, ring.cpu().tolist(), ring_o)


@pytest.mark.parametrize("shape", [(256, 7), (256, 16), (1, 1), (37, 5), (128, 15)])
def test_zos_select_every_budget(shape):
    """Budgets planted in the ring: the radix select equals the oracle's top-K for each."""
    bs, gamma = shape
    n = bs * gamma
    m_max = bs + n
    sps = torch.ones(m_max + 1, dtype=torch.float64, device="cuda")
    win = torch.zeros(bs, dtype=torch.int32, device="cuda")
    K = torch.zeros(1, dtype=torch.int32, device="cuda")
    for ties in (False, True):
        a = I.random_survival(bs, gamma, n + ties, ties=ties)
        surv = torch.as_tensor(a, device="cuda")
        for Kp in sorted({0, 1, 2, n // 3, n // 2, n - 1, n, n + 5}):
            if Kp < 0:
                continue
            ring = torch.tensor([Kp, -1], dtype=torch.int32, device="cuda")
            B.dspark_schedule_zos_select(surv, sps, ring, 0, win, K, _WS())
            Ke = min(Kp, n)
            assert int(K.item()) == Ke
            np.testing.assert_array_equal(win.cpu().numpy(), O.zos_select(a, Ke), err_msg=f"K={Kp}")


def test_zos_select_tie_and_sign_edge_cases():
    bs, gamma = 64, 8
    sps = torch.ones(bs * (gamma + 1) + 1, dtype=torch.float64, device="cuda")
    win = torch.zeros(bs, dtype=torch.int32, device="cuda")
    K = torch.zeros(1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(5)
    variants = [np.ones((bs, gamma), np.float32),                     # every key equal
                np.zeros((bs, gamma), np.float32),
                np.full((bs, gamma), -0.0, np.float32),                # ranks as 0
                -np.sort(-rng.choice(np.float32([1.0, 0.5, 2.0 ** -30, 1e-38, 0.0]),
                                     size=(bs, gamma)), axis=1).astype(np.float32)]
    for a in variants:
        surv = torch.as_tensor(a, device="cuda")
        for Kp in (0, 1, 63, 64, 65, 300, 511, 512):
            ring = torch.tensor([-1, Kp], dtype=torch.int32, device="cuda")
            B.dspark_schedule_zos_select(surv, sps, ring, 1, win, K, _WS())
            Ke = min(Kp, bs * gamma)
            expect = O.zos_select(np.maximum(a, 0) + np.float32(0), Ke)
            np.testing.assert_array_equal(win.cpu().numpy(), expect)


def test_zos_inside_the_step_with_a_second_stream():
    """The orchestrated step (step.run_step with a ring and a side stream for the budget): over
    five steps of the mixed workload the windows of each step equal the oracle's asynchronous
    scheduler applied to the survival the GPU produced, with the oracle's own ring."""
    from speculative_decoding_draft_markov_gb300 import step as S
    dev = torch.device("cuda")
    wl = I.WORKLOADS["mixed_bs256"]
    inp = I.make_device_inputs(wl, dev)
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    cap = int(I.tiers_for(wl)[-1])
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype, dev)
    sps = S.sps_table(inp["T_raw"], inp["tiers"], dev)
    sps_h = sps.cpu().numpy()
    tiers = torch.as_tensor(inp["tiers"], device=dev)
    fwd = S.gather_target_forward(inp["target"])
    ring, ring_o = S.zos_ring(dev), [-1, -1]
    side = torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)
    for t in range(5):
        S.run_step(inp, buf, sps, fwd, wl.temperature, wl.seed, t, B.DSPARK_COMPACT, tiers=tiers,
                   stream=main, ring=ring, side_stream=side)
        torch.cuda.synchronize(dev)
        assert B.dspark_read_device_status(buf.ws) == B.DSPARK_OK
        w_o, K_o = O.zos_step(buf.surv.cpu().numpy(), sps_h, ring_o, t)
        np.testing.assert_array_equal(buf.window.cpu().numpy(), w_o)
        assert int(buf.K.item()) == K_o
        assert ring.cpu().tolist() == ring_o
        # the packed layout and the verify used those windows
        assert int(buf.cu[-1].item()) == bs + K_o
        assert np.all(buf.acc_len.cpu().numpy() <= w_o)


@pytest.mark.parametrize("sched_mode", [0, 1])
def test_fused_schedule_pack_equals_the_two_calls(sched_mode):
    """dspark_schedule_pack writes exactly what dspark_schedule followed by dspark_pack write."""
    wl = I.WORKLOADS["qwen3_4b"].with_(name="fused_sched", bs=77, gamma=6, V=2048, d=64, seed=41)
    dev = torch.device("cuda")
    bs, gamma = wl.bs, wl.gamma
    surv = torch.as_tensor(I.random_survival(bs, gamma, 9), device=dev)
    tokens = torch.as_tensor(I.random_tokens(bs, gamma, wl.V, 3), device=dev)
    anchor = torch.arange(bs, dtype=torch.int32, device=dev)
    tiers = torch.as_tensor(np.arange(32, bs * (gamma + 1) + 32, 32, dtype=np.int32), device=dev)
    T = 1.0 + 0.01 * np.arange(bs * (gamma + 1) + 1)
    sps = torch.as_tensor(O.build_sps(T, list(range(32, bs * (gamma + 1) + 32, 32))), device=dev)
    cap = int(tiers[-1])
    outs = []
    for fused in (False, True):
        ws = B.alloc_workspace(bs, gamma, wl.V)
        win = torch.zeros(bs, dtype=torch.int32, device=dev)
        K = torch.zeros(1, dtype=torch.int32, device=dev)
        th = torch.zeros(1, dtype=torch.float64, device=dev)
        cu = torch.zeros(bs + 1, dtype=torch.int32, device=dev)
        ids, req, pos = (torch.full((cap,), -7, dtype=torch.int32, device=dev) for _ in range(3))
        pad = torch.zeros(1, dtype=torch.int32, device=dev)
        if fused:
            B.dspark_schedule_pack(surv, sps, sched_mode, win, K, th, anchor, tokens, tiers, cu, ids, req, pos, pad, ws)
        else:
            B.dspark_schedule(surv, sps, sched_mode, win, K, th, ws)
            B.dspark_pack(win, anchor, tokens, tiers, cu, ids, req, pos, pad, ws)
        assert B.dspark_read_device_status(ws) == B.DSPARK_OK
        outs.append([t.cpu() for t in (win, K, th, cu, ids, req, pos, pad)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
