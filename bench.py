"""Benchmark: DSpark step tokens/s at bs=256, V=151936, gamma=7 (the mixed-difficulty batch),
then the pages' other workloads.

One step = draft_block -> confidence -> schedule -> pack -> [target forward] -> verify, all
through the C ABI on one stream; the timed steps replay CUDA graphs captured from those calls
(one graph per stage and step, each with its own step counter), the e2e steps call the API
directly with host buffers.  The target forward is the caller's model and is not part of this
path: in the timed steps it is a device row gather outside the timed segments; in the e2e steps
it copies the step's packed rows from host memory, inside the timing.  Everything else is timed
with CUDA events on the launching stream.  The L2 is flushed (256 MB write) before every timed
step.  tokens/step = sum over requests of (accepted + 1); `value` = tokens of all K timed steps /
their summed time, `value_median` the same at the median step.  Rooflines per stage: the
draft against HBM (U, W2 once, the gathered W1 rows) and the tensor pipe (2 bs gamma r V flops),
the verification against HBM (the packed target rows, and at temperature > 0 one U row per
request and W2 for the recompute of p_d).  The same steps are timed again under the
asynchronous scheduler ("zos"), and every further configuration gets its own result under
"configs" (Qwen3-4B-shaped bs 64; the DeepSeek-V4-shaped sweep bs 1..256 with static and compact
budgets; the long block at temperature 1 and greedy).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload all|none|NAME]

--gpus N > 1 runs under torchrun: one independent replica per GPU (the path has no
cross-request exchange that needs a collective), barrier + max-over-ranks timing; value is
the tokens of all ranks / that time ("scaling": "weak").
--impl reference times the CPU oracle (plain numpy, fp64; draft and verify over the host cores
in worker processes) on bounded samples of the same workload."""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "mixed_bs256"
# The workload's cost table is a sawtooth (graph tiers every 64 tokens, and bs = 256 sits on a
# tier boundary), so Theta(K) is not unimodal: the first admitted slot crosses into the next
# tier and an early stop would admit nothing.  The DSpark technical summary ("Infra") runs
# the global search over a sawtooth SPS curve; the benchmark does the same.
SCHED = 1  # DSPARK_SCHED_GLOBAL_ARGMAX
METRIC = "DSpark step tokens/s at bs=256,V=151936,γ=7; % of HBM/tensor roofline"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and clock-event reasons of the benchmark's GPU, sampled every ~2 ms by a thread
    during the timed region: NVML read-only queries through ctypes (the device is matched by
    PCI bus id), else `nvidia-smi -lms 200`.  Nothing is set."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.samples = []  # (sm_mhz, max_mhz, reasons bitmask)
        self.lines = []
        self.proc = None
        self.stop = threading.Event()
        self.nvml = None

    def _nvml_handle(self):
        import ctypes
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None
        props = torch.cuda.get_device_properties(self.device)
        h = ctypes.c_void_p()
        bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
        if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByUUID(("GPU-" + str(props.uuid)).encode(), ctypes.byref(h)) != 0:
                return None
        self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return nv, h

    def _poll(self):
        import ctypes
        nv, h = self.nvml
        mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and
                    nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    self.reason_fn(h, ctypes.byref(rs)) == 0):
                self.samples.append((mhz.value, mx.value, rs.value))
            time.sleep(0.002)

    def __enter__(self):
        try:
            self.nvml = self._nvml_handle()
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.nvml is not None:
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        for s_mhz, m_mhz, bits in self.samples:
            sm.append(float(s_mhz))
            mx.append(float(m_mhz))
            reasons.update(n for b, n in self.REASONS.items() if bits & b)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvml" if self.samples else "nvidia-smi"}

# ------------------------------------------------------------------------------- CPU oracle
def _host_target(h, tok, dtype: str):
    """The workloads' target model on the host, as step.markov_target_forward computes it on the
    device: every (request, position) row j of the drawn base target (U + noise) plus W1[x_j] W2,
    x_0 the anchor and x_j the drafted tokens; the term is accumulated in fp32 and rounded to the
    logits' dtype, then added to the row with one more rounding."""
    from speculative_decoding_draft_markov_gb300 import inputs as I
    x = np.concatenate([np.asarray(h["anchor"])[:, None], np.asarray(tok)], axis=1)  # [n, gamma + 1]
    if dtype == "f32":
        W1, W2t = h["W1"], h["W2t"]
        return np.ascontiguousarray(h["target"] + np.stack([W1[x[:, j]] @ W2t.T for j in range(x.shape[1])], 1))
    W1, W2t = I.bf16_bits_to_f32(h["W1"]), I.bf16_bits_to_f32(h["W2t"])
    out = np.empty_like(h["target"])
    for j in range(x.shape[1]):  # a position at a time keeps the fp32 temporaries at [n, V]
        term = I.bf16_bits_to_f32(I.f32_to_bf16_bits(W1[x[:, j]] @ W2t.T))
        out[:, j] = I.f32_to_bf16_bits(I.bf16_bits_to_f32(h["target"][:, j]) + term)
    return out


def _oracle_steps(wl_name: str, n_req: int, steps, mode_name: str = "compact", sched: int = SCHED):
    """The oracle's full step (draft, confidence, schedule, pack, verify) on the first n_req
    requests of a workload, on every host core (oracle.pool: one worker per core, requests in
    slices).  Host inputs are generated and the pool started before the clock; each step's
    (tokens, seconds) is returned."""
    from oracle import dspark_oracle as O
    from oracle import pool as OP
    from speculative_decoding_draft_markov_gb300 import inputs as I
    wl = I.WORKLOADS[wl_name].with_(bs=n_req)
    h = I.make_host_inputs(wl)
    sps = O.build_sps(h["T_raw"], h["tiers"])
    mode = {"compact": O.COMPACT, "static": O.STATIC}[mode_name]
    per = max(1, -(-n_req // OP.workers()))
    out = []
    with OP.pool(h["W1"], h["W2t"], wl.dtype) as p:
        for s in steps:
            t0 = time.perf_counter()
            (tok, lx, lse, _), _ = OP.draft_all(p, h["U"], h["anchor"], wl.temperature, wl.seed, s, per=per)
            t1 = time.perf_counter()
            target = _host_target(h, tok, wl.dtype)  # the target model's forward: not the oracle's time
            t_fwd = time.perf_counter() - t1
            if mode == O.COMPACT:
                _, surv, _ = O.confidence(h["h"], h["W1"], h["anchor"], tok, h["w"], h["b"], h["sts_T"],
                                          dtype=wl.dtype)
                win, _, _, _ = O.schedule(surv.astype(np.float32), sps, sched)
                cu, _, _, _, _ = O.pack(win, h["anchor"], tok, h["tiers"], max(n_req * (wl.gamma + 1),
                                                                                 int(h["tiers"][-1])))
            else:
                win = np.full(n_req, wl.gamma, dtype=np.int32)
            (_, acc, _, _), _ = OP.verify_all(p, target, h["U"], win, mode, h["anchor"], tok,
                                              lx.astype(np.float32), lse.astype(np.float32), wl.temperature,
                                              wl.seed, s, per=per)
            out.append((O.step_tokens(acc), time.perf_counter() - t0 - t_fwd))
    return out, OP.workers()


def cpu_baseline(n_req: int = 128, steps: int = 3):
    """The oracle, as it stands, on every host core: a bounded sample of the workload."""
    try:
        res, cores = _oracle_steps(WORKLOAD, n_req, range(steps))
    except Exception as e:  # reported, never fatal for the GPU line
        return {"value": None, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                "error": repr(e)[-300:]}
    tok = sum(r[0] for r in res)
    sec = sum(r[1] for r in res)
    return {"value": tok / sec, "unit": "tokens/s", "cores": cores, "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"first {n_req} of the 256 requests of mixed_bs256 (full V=151936, gamma=7), all five "
                      f"stages (oracle draft and verify in {cores} worker processes, one BLAS thread each), "
                      f"{steps} steps: {tok} tokens in {sec:.1f} s"}


# ------------------------------------------------------------------------------- rooflines
# Algorithmic bytes and flops per call, as the hot-path scope table counts them.

def draft_bytes(bs: int, gamma: int, V: int, r: int, esize: int = 2) -> int:
    """One dspark_draft_block call: U [bs, gamma, V] read once, W2 [r, V] read once, and the
    gamma x bs gathered W1 rows.  Any re-read of W2 from DRAM by a later position (it stays in
    L2 inside the persistent draft kernel, mostly) is traffic, reported beside this, not
    algorithmic bytes."""
    return bs * gamma * V * esize + V * r * esize + bs * gamma * r * esize


def draft_flops(bs: int, gamma: int, V: int, r: int) -> int:
    return 2 * bs * gamma * r * V


def verify_bytes(rows: float, bs: int, V: int, r: int, greedy: bool, esize: int = 2) -> float:
    """One dspark_verify call: every packed target row once; at temperature > 0 the decision
    pass's recompute of p_d adds one U row per request and W2 once (the deciding target rows are
    counted as L2 re-reads)."""
    b = rows * V * esize
    if not greedy:
        b += bs * V * esize + V * r * esize
    return b


def _sources_sha(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "speculative_decoding_draft_markov_gb300", "csrc", f), "rb").read())
    # of the header, the constants (the kernels' sizes and chunk widths), not its documentation
    for line in open(os.path.join(ROOT, "include", "dspark.h"), "rb"):
        if line.startswith(b"#define"):
            h.update(line)
    return h.hexdigest()


def _profiled_traffic(name: str):
    """DRAM bytes per call of a stage from its committed ncu summary (profiles/<name>.json), or
    None when the kernels' sources changed after that capture (the summary records their
    SHA-256)."""
    path = os.path.join(ROOT, "profiles", name + ".json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("sources_sha256") != _sources_sha(d.get("sources", [])):
        return None
    return d.get("dram_bytes_per_call")


DRAFT_SOURCES = ["draft_tc.cu", "draft.cu", "draft_select.cuh", "confidence.cuh", "common.cuh", "tc_ptx.cuh", "tc_host.h"]
VERIFY_SOURCES = ["verify.cu", "decide_tc.cu", "f32x2.cuh", "common.cuh", "tc_ptx.cuh", "tc_host.h"]


def rooflines(wl, stage_ms, rows, tau, profile_key=None, conf_in_draft=False):
    hbm, bf16, peak_kind = _peaks()
    bs, gamma, V, r = wl.bs, wl.gamma, wl.V, wl.r
    # with the confidence head inside the draft's launch its h rows count with the draft's bytes
    db = draft_bytes(bs, gamma, V, r) + (bs * gamma * wl.d * 2 if conf_in_draft else 0)
    dflop = draft_flops(bs, gamma, V, r)
    dsec = stage_ms["draft"] * 1e-3
    traffic = (_profiled_traffic(f"{'draft_confidence_block' if conf_in_draft else 'draft_block'}_{profile_key}_dram")
               if profile_key else None)
    vb = verify_bytes(rows, bs, V, r, tau == 0.0)
    vsec = stage_ms["verify"] * 1e-3
    vtraffic = _profiled_traffic(f"verify_{profile_key}_dram") if profile_key else None
    return {
        "bound": "hbm", "achieved": db / dsec / 1e9, "peak": hbm, "unit": "GB/s", "frac": db / dsec / 1e9 / hbm,
        "traffic": traffic, "traffic_over_algorithmic": (traffic / db) if traffic else None,
        "kernel": ("dspark_draft_confidence_block" if conf_in_draft else "dspark_draft_block")
                  + ": one persistent cooperative draft_tc_kernel launch over all gamma positions (vocabulary "
                  "passes + in-kernel selects" + (" + the confidence head" if conf_in_draft else "") +
                  "); one C-ABI call, CUDA events around it in the timed steps",
        "algorithmic_bytes": db, "peak_kind": peak_kind,
        "tensor": {"achieved": dflop / dsec / 1e12, "peak": bf16, "unit": "TFLOP/s",
                   "frac": dflop / dsec / 1e12 / bf16, "flops": dflop},
        "verify": {"bound": "hbm", "achieved": vb / vsec / 1e9, "peak": hbm, "unit": "GB/s",
                   "frac": vb / vsec / 1e9 / hbm, "algorithmic_bytes": vb, "packed_rows": rows,
                   "traffic": vtraffic,
                   "kernel": "dspark_verify (row statistics over the packed target rows, accept scan, and at "
                             "temperature > 0 the tensor-core decision pass and its select), events around it"},
    }


def aggregate_over_ranks(times_ms, counts, device):
    """Replica aggregation of the timed region: the slowest rank's durations (MAX) and the work
    of all ranks (SUM), over the default process group when one with more than one rank is up;
    the inputs unchanged otherwise."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in times_ms], [float(x) for x in counts]
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    n = torch.tensor([float(x) for x in counts], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], [float(x) for x in n.tolist()]


# ------------------------------------------------------------------------------- GPU arm
class Path:
    """One workload's device inputs, buffers and the three stages of its step through the API.

    mode: "compact" (confidence, global scheduler + pack, compact verify) or "static" (pack of
    the whole block, static verify); tau: sampling temperature (0 = greedy)."""

    def __init__(self, wl, dev, mode="compact", tau=None, sched=SCHED, rnn=False):
        import torch

        from speculative_decoding_draft_markov_gb300 import binding as B
        from speculative_decoding_draft_markov_gb300 import inputs as I
        from speculative_decoding_draft_markov_gb300 import step as S
        self.B, self.S = B, S
        self.wl, self.dev, self.mode, self.sched = wl, dev, mode, sched
        self.tau = wl.temperature if tau is None else tau
        self.inp = I.make_device_inputs(wl, dev, with_rnn=rnn)
        self.states = (torch.empty((wl.bs, wl.gamma, wl.r), dtype=self.inp["U"].dtype, device=dev)
                       if rnn else None)
        self.cap = int(I.tiers_for(wl)[-1]) if len(I.tiers_for(wl)) else wl.bs * (wl.gamma + 1)
        self.cap = max(self.cap, wl.bs * (wl.gamma + 1))
        self.buf = S.StepBuffers.allocate(wl.bs, wl.gamma, wl.V, self.cap, self.inp["U"].dtype, dev)
        self.sps = S.sps_table(self.inp["T_raw"], self.inp["tiers"], dev)
        self.tiers = torch.as_tensor(self.inp["tiers"], device=dev) if len(self.inp["tiers"]) else None
        self.fwd = S.markov_target_forward(S.gather_target_forward(self.inp["target"]), self.inp["W1"],
                                           self.inp["W2t"])
        self.ring = S.zos_ring(dev)
        self.vmode = B.DSPARK_COMPACT if mode == "compact" else B.DSPARK_STATIC
        # the Markov head's compact step computes the confidence inside the draft's launch
        # (dspark_draft_confidence_block); the RNN head's step runs it as its own launch
        self.fused = mode == "compact" and not rnn
        tc = self.inp["U"].dtype == torch.bfloat16 and wl.r in (64, 128, 256)
        draft_l = 1 if tc else (3 if rnn else 2) * wl.gamma
        conf_l = 0 if (mode != "compact" or self.fused) else 1
        # launches of one synchronous-scheduler step (the asynchronous one adds two: its
        # select + pack in place of the fused schedule+pack, and the budget search)
        self.launches = draft_l + conf_l + 1 + (4 if self.tau > 0 else 2)

    def draft(self, it):
        inp, buf = self.inp, self.buf
        if self.states is not None:  # the RNN sequential head
            self.B.dspark_draft_block_rnn(inp["U"], inp["W1"], inp["W2t"], inp["Wg"], inp["bg"], inp["anchor"],
                                          self.tau, self.wl.seed, it, buf.tokens, buf.logit_x, buf.lse, self.states,
                                          buf.ws)
            return
        if self.fused:
            self.B.dspark_draft_confidence_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], self.tau,
                                                 self.wl.seed, it, buf.tokens, buf.logit_x, buf.lse, inp["h"],
                                                 inp["w"], inp["b"], inp["sts_T"], buf.conf, buf.surv, buf.ws)
            return
        self.B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], self.tau, self.wl.seed, it,
                                  buf.tokens, buf.logit_x, buf.lse, buf.ws)

    def sched_pack(self, it, zos=False):
        B, inp, buf = self.B, self.inp, self.buf
        if self.mode == "static":
            B.dspark_pack(None, inp["anchor"], buf.tokens, self.tiers, buf.cu, buf.ids, buf.req, buf.pos, buf.padded,
                          buf.ws)
            return
        if not self.fused:
            B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], buf.tokens, inp["w"], inp["b"], inp["sts_T"],
                                buf.conf, buf.surv)
        if zos:
            B.dspark_schedule_zos_select(buf.surv, self.sps, self.ring, it, buf.window, buf.K, buf.ws)
            B.dspark_pack(buf.window, inp["anchor"], buf.tokens, self.tiers, buf.cu, buf.ids, buf.req, buf.pos,
                          buf.padded, buf.ws)
        else:  # the synchronous scheduler and the pack of its windows in one launch
            B.dspark_schedule_pack(buf.surv, self.sps, self.sched, buf.window, buf.K, buf.theta, inp["anchor"],
                                   buf.tokens, self.tiers, buf.cu, buf.ids, buf.req, buf.pos, buf.padded, buf.ws)

    def verify(self, it, zos=False, stream=None, side=None):
        # asynchronous scheduler: the budget for step it + 2 forks onto a second stream and
        # runs beside the verify, joined at the end of the stage
        if zos:
            self.S.schedule_budget(self.buf, self.sps, self.ring, it, stream, side)
        self.S.verify(self.inp, self.buf, self.tau, self.wl.seed, it, self.vmode, states=self.states)
        if zos:
            self.S.join_budget(stream, side)


def time_steps(path, steps, warmup, zos=False, world=1):
    """Warm-up, graph capture and the timed steps of one path.  The timed steps replay CUDA
    graphs of the API calls (one per stage and step, each with its own step counter); the L2 is
    flushed (256 MB write) before every step, outside the timed segments, and the stand-in target
    forward runs outside them too.  Returns per-step segment times [steps, 3] (draft + sched/pack,
    verify, draft alone) in ms, tokens, packed rows and admitted slots summed over the steps, the
    host enqueue time and the clock record."""
    import torch
    import torch.distributed as dist
    B, buf, dev = path.B, path.buf, path.dev
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev) if zos else None
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    acc = torch.zeros(3, dtype=torch.int64, device=dev)  # tokens, packed rows, admitted slots

    def count():
        acc[0].add_((buf.acc_len.to(torch.int64) + 1).sum())
        acc[1].add_(buf.cu[-1].to(torch.int64))
        acc[2].add_(buf.K[0].to(torch.int64))

    if zos:
        path.ring.fill_(-1)
    for w in range(warmup):  # eager, through the API: every op of the timed loop runs once before it
        path.draft(10_000 + w)
        path.sched_pack(10_000 + w, zos)
        path.fwd(buf)
        path.verify(10_000 + w, zos, stream, side)
        count()
    graphs = []
    for it in range(steps):
        gs = [torch.cuda.CUDAGraph() for _ in range(3)]
        with torch.cuda.graph(gs[0]):
            path.draft(it)
        with torch.cuda.graph(gs[1]):
            path.sched_pack(it, zos)
        with torch.cuda.graph(gs[2]):
            path.verify(it, zos, torch.cuda.current_stream(dev), side)
        graphs.append(gs)
    for gs in graphs:  # once untimed, so that the timed replays find the graphs resident
        gs[0].replay()
        gs[1].replay()
        path.fwd(buf)
        gs[2].replay()
    torch.cuda.synchronize(dev)
    st = B.dspark_read_device_status(buf.ws)
    if st != 0:
        raise RuntimeError(f"{path.wl.name}: device status after warm-up: " + B.dspark_status_string(st))
    acc.zero_()
    buf.K.zero_()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk:
        t_host = time.perf_counter()
        for it in range(steps):
            flush.fill_(it & 0xFF)  # L2 flush, outside the timed segments
            e, gs = evs[it], graphs[it]
            e[0].record(stream)
            gs[0].replay()
            e[1].record(stream)
            gs[1].replay()
            e[2].record(stream)
            path.fwd(buf)  # the caller's target forward: outside the timed segments
            e[3].record(stream)
            gs[2].replay()
            e[4].record(stream)
            count()
        t_host = time.perf_counter() - t_host  # host time to enqueue (the device may still run)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    seg = np.array([[e[0].elapsed_time(e[2]), e[3].elapsed_time(e[4]), e[0].elapsed_time(e[1])] for e in evs])
    st = B.dspark_read_device_status(buf.ws)
    if st != 0:
        raise RuntimeError(f"{path.wl.name}: device status after the timed steps: " + B.dspark_status_string(st))
    tokens, rows, slots = (int(x) for x in acc.tolist())
    del graphs
    return seg, tokens, rows, slots, t_host, clk.summary()


def time_e2e(path, steps):
    """The same step end to end through the public API with host buffers (pinned), every copy
    inside the timing: U, h and the anchors of each step copied host -> device on a second stream
    one step ahead (double-buffered); the base target logits (U + noise) of every (request,
    position) stay in pinned host memory and each step's target forward reads the packed layout
    back (cu_seqlens, after the pack), copies exactly the rows that step verifies
    (dspark_copy_packed_rows_async) and adds their Markov term on the device
    (step.markov_target_forward); out_tokens and acc_len come back every step.  Returns
    (tokens/s, h2d bytes per step, d2h bytes per step, steps)."""
    import torch
    B, S, buf, inp, wl, dev = path.B, path.S, path.buf, path.inp, path.wl, path.dev
    bs, gamma = wl.bs, wl.gamma
    stream = torch.cuda.current_stream(dev)
    keys = ("U", "h", "anchor") if path.mode == "compact" else ("U", "anchor")
    host = {k: inp[k].cpu().pin_memory() for k in keys}
    host_target = inp["target"].cpu().pin_memory()
    cu_host = torch.empty(bs + 1, dtype=torch.int32).pin_memory()
    target_rows = []

    def host_rows(b):
        cu_host.copy_(b.cu, non_blocking=True)
        stream.synchronize()  # the packed layout is known once the pack has run
        B.dspark_copy_packed_rows_async(b.packed, host_target, cu_host, stream)
        target_rows.append(int(cu_host[bs]))

    # the Markov term over the step's rows rounded up to a multiple of 256: a handful of GEMM
    # shapes, each run once here before the timing (so that cuBLAS has picked its kernel for
    # each), instead of a new shape at every step's packed total
    cap = buf.packed.shape[0]
    rounded = lambda: min(cap, -(-target_rows[-1] // 256) * 256)
    host_target_forward = S.markov_target_forward(host_rows, inp["W1"], inp["W2t"], rounded)
    for n in range(256, cap + 256, 256):
        n = min(n, cap)
        torch.matmul(inp["W1"][:n], inp["W2t"].t())

    inps = [inp, dict(inp)]
    for k in host:
        inps[1][k] = torch.empty_like(inp[k])
    outs = [torch.empty((bs, gamma + 1), dtype=torch.int32).pin_memory() for _ in range(steps)]
    accs = [torch.empty(bs, dtype=torch.int32).pin_memory() for _ in range(steps)]
    bo = outs[0].numel() * 4 + accs[0].numel() * 4 + cu_host.numel() * 4
    cstream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    released = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(it):
        d = inps[it % 2]
        cstream.wait_event(released[it % 2])  # the step that last read this buffer is done
        with torch.cuda.stream(cstream):
            for k, h in host.items():
                d[k].copy_(h, non_blocking=True)
        copied[it % 2].record(cstream)

    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cstream.wait_stream(stream)
    issue_copy(0)
    for it in range(steps):
        if it + 1 < steps:
            issue_copy(it + 1)
        stream.wait_event(copied[it % 2])
        S.run_step(inps[it % 2], buf, path.sps, host_target_forward, path.tau, wl.seed, 20_000 + it, path.vmode,
                   path.sched, tiers=path.tiers)
        released[it % 2].record(stream)
        outs[it].copy_(buf.out_tokens, non_blocking=True)
        accs[it].copy_(buf.acc_len, non_blocking=True)
    e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    tokens = sum(int((a.to(torch.int64) + 1).sum()) for a in accs)
    row_bytes = host_target[0, 0].numel() * host_target.element_size()
    bi = sum(t.numel() * t.element_size() for t in host.values()) + int(np.mean(target_rows)) * row_bytes
    st = B.dspark_read_device_status(buf.ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after the end-to-end steps: " + B.dspark_status_string(st))
    del host, host_target
    return tokens / (ms * 1e-3), bi, bo, steps, ms


def measure(path, steps, warmup, e2e_steps, profile_key=None, world=1):
    """Device-timed steps, end-to-end steps and the rooflines of one path, as a result dict."""
    seg, tokens, rows, slots, t_host, clocks = time_steps(path, steps, warmup, world=world)
    step_ms = seg[:, 0] + seg[:, 1]
    (total_ms,), (tokens_all,) = aggregate_over_ranks([float(step_ms.sum())], [tokens], path.dev)
    stage_ms = {"draft": float(seg[:, 2].mean()), "sched_pack": float((seg[:, 0] - seg[:, 2]).mean()),
                "verify": float(seg[:, 1].mean())}
    e2e_v, bi, bo, e_steps, e_ms = time_e2e(path, e2e_steps)
    (e_ms_all,), (e2e_tok,) = aggregate_over_ranks([e_ms], [e2e_v * e_ms * 1e-3], path.dev)
    wl = path.wl
    return {
        "value": tokens_all / (total_ms * 1e-3), "unit": "tokens/s", "steps": steps, "ms_per_step": total_ms / steps,
        "median_ms_per_step": float(np.median(step_ms)),
        "value_median": tokens / steps / (float(np.median(step_ms)) * 1e-3),
        "tokens_per_step": tokens / steps, "packed_rows_per_step": rows / steps,
        "admitted_slots_per_step": slots / steps if path.mode == "compact" else wl.bs * wl.gamma,
        "stage_ms": stage_ms, "host_enqueue_ms_per_step": t_host * 1e3 / steps,
        "roofline": rooflines(wl, stage_ms, rows / steps, path.tau, profile_key, conf_in_draft=path.fused),
        "e2e": {"value": e2e_tok / (e_ms_all * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "steps": e_steps},
        "gpu_launches": path.launches * steps, "clocks": clocks,
    }


def config_lines(args, dev):
    """Every other configuration of the pages' workloads, one result each: Qwen3-4B-shaped (bs 64,
    compact), the DeepSeek-V4-shaped sweep (bs 1..256, static and compact budgets) and the long
    block (bs 128, gamma 15, temperature 1 and greedy)."""
    import gc

    import torch

    from speculative_decoding_draft_markov_gb300 import inputs as I
    runs = [("qwen3_4b", I.WORKLOADS["qwen3_4b"], "compact", None)]
    for b in I.DSV4_BATCHES:
        for mode in ("static", "compact"):
            runs.append((f"dsv4_bs{b}_{mode}", I.dsv4(b), mode, None))
    runs += [("long_block_t1", I.WORKLOADS["long_block"], "compact", 1.0),
             ("long_block_greedy", I.WORKLOADS["long_block"], "compact", 0.0)]
    out = []
    for name, wl, mode, tau in runs:
        if args.workload not in ("all", name, wl.name):
            continue
        path = Path(wl, dev, mode, tau)
        r = measure(path, args.config_steps, args.warmup, 4)
        r = {"workload": name, "bs": wl.bs, "gamma": wl.gamma, "V": wl.V, "r": wl.r, "d": wl.d, "mode": mode,
             "temperature": path.tau, "scheduler": "global-argmax" if mode == "compact" else "none (whole block)",
             **r}
        out.append(r)
        del path
        gc.collect()
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank: int, world: int):
    import torch

    from speculative_decoding_draft_markov_gb300 import inputs as I

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[WORKLOAD].with_(seed=I.WORKLOADS[WORKLOAD].seed + 1000 * rank)
    path = Path(wl, dev, "compact")
    head = measure(path, args.steps, args.warmup, max(2, min(args.steps, 10)), profile_key=WORKLOAD, world=world)
    # the same steps under the asynchronous scheduler (budget from two steps back, computed on a
    # second stream beside the verify; the select alone on the step's path)
    zseg, ztokens, _, _, _, zclocks = time_steps(path, args.steps, args.warmup, zos=True, world=world)
    (ztotal_ms,), (ztokens,) = aggregate_over_ranks([float((zseg[:, 0] + zseg[:, 1]).sum())], [ztokens], dev)
    obs = measure_observability(args, path.inp, path.buf, path.tau, wl, dev, torch.cuda.current_stream(dev),
                                path.tiers, path.fwd)
    res = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "median_ms_per_step": head["median_ms_per_step"],
        "value_median": head["value_median"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; U~N(0,3^2), W~N(0,0.05^2), target = U + W1[x_{k-1}]W2 + N(0,sigma^2) at the "
                "drafted prefix, sigma 0.5/1/2 by thirds)",
        "config": {"workload": "mixed_bs256: bs=256, gamma=7, V=151936, r=256, d=4096, compact verify, "
                               "temperature 1, sawtooth cost table with tiers every 64 to 2048, global-argmax scheduler",
                   "global_batch": wl.bs * world, "l2": "flushed between steps (256 MB write)",
                   "timed": "draft+confidence+schedule+pack and verify segments; target forward excluded; "
                            "each stage of each timed step a captured CUDA graph of its API calls",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_step": head["tokens_per_step"] / world,
        "packed_rows_per_step": head["packed_rows_per_step"],
        "admitted_slots_per_step": head["admitted_slots_per_step"],
        "host_enqueue_ms_per_step": head["host_enqueue_ms_per_step"],
        "stage_ms": head["stage_ms"],
        "roofline": head["roofline"],
        "e2e": dict(head["e2e"], note="U, h, anchors copied from pinned host memory every step on a second stream, "
                                      "one step ahead (double-buffered); the target forward copies the step's "
                                      "packed base target rows (U + noise) from pinned host memory after the pack "
                                      "(cu_seqlens read back) and adds their Markov term W1[x_j]W2 on the device"),
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "observability": obs,
        "zos": {"value": ztokens / (ztotal_ms * 1e-3), "unit": "tokens/s", "ms_per_step": ztotal_ms / args.steps,
                "tokens_per_step": ztokens / args.steps / world,
                "stage_ms": {"draft": float(zseg[:, 2].mean()),
                             "sched_pack": float((zseg[:, 0] - zseg[:, 2]).mean()),
                             "verify_with_budget": float(zseg[:, 1].mean())},
                "scheduler": "asynchronous: budget from the survival two steps back (global search, second "
                             "stream beside the verify), radix top-K select on the step's path",
                "gpu_launches": (path.launches + 2) * args.steps, "clocks": zclocks},
    }
    del path
    # the same step with the RNN sequential head (device-timed; the draft adds one state-update
    # launch per position and verify recomputes p_d from the states)
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    rpath = Path(wl, dev, "compact", rnn=True)
    rseg, rtokens, rrows, _, _, rclocks = time_steps(rpath, args.steps, args.warmup, world=world)
    (rtotal_ms,), (rtokens,) = aggregate_over_ranks([float((rseg[:, 0] + rseg[:, 1]).sum())], [rtokens], dev)
    rstage = {"draft": float(rseg[:, 2].mean()), "conf_sched_pack": float((rseg[:, 0] - rseg[:, 2]).mean()),
              "verify": float(rseg[:, 1].mean())}
    rroof = rooflines(wl, rstage, rrows / args.steps, rpath.tau)
    res["rnn"] = {"value": rtokens / (rtotal_ms * 1e-3), "unit": "tokens/s", "ms_per_step": rtotal_ms / args.steps,
                  "tokens_per_step": rtokens / args.steps / world, "stage_ms": rstage,
                  "draft_frac_hbm": rroof["frac"], "verify_frac_hbm": rroof["verify"]["frac"],
                  "head": "RNN sequential head: gated recurrent state s_k (bf16), bias s_k W2; the same single "
                          "persistent draft launch, which computes s_1 in its prologue and each request's "
                          "next state right after its select; the confidence head in its own launch",
                  "gpu_launches": rpath.launches * args.steps, "clocks": rclocks}
    del rpath
    if not args.no_configs:
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        res["configs"] = config_lines(args, dev)
    return res


def measure_observability(args, inp, buf, tau, wl, dev, stream, tiers_dev, fwd):
    """Observability and calibration beside the step: one cap-accept verification of the last
    drafted block exposes the ceiling; dspark_observe records it (timed per call with events);
    the temperature fit runs on 2^20 synthetic labelled prefixes drawn from a known law
    (7 positions, 64 grid temperatures, 15 bins), timed after one untimed fit."""
    import torch

    from speculative_decoding_draft_markov_gb300 import binding as B
    from speculative_decoding_draft_markov_gb300 import inputs as I
    from speculative_decoding_draft_markov_gb300 import step as S
    n_bins = 15
    gamma = wl.gamma
    # cap-accept verifies the whole block: static packing of the last drafted block, the
    # stand-in target forward, then the verification with the scheduler's windows
    B.dspark_pack(None, inp["anchor"], buf.tokens, tiers_dev, buf.cu, buf.ids, buf.req, buf.pos, buf.padded,
                  buf.ws)
    fwd(buf)
    S.verify(inp, buf, tau, wl.seed, 30_000, B.DSPARK_CAP_ACCEPT)
    stats = B.alloc_obs_stats(dev)
    B.dspark_observe(buf.surv, buf.window, buf.acc_len, buf.ceiling, n_bins, stats, buf.ws)
    torch.cuda.synchronize(dev)
    # device time per call: a CUDA graph of `reps` back-to-back calls, replayed once untimed
    # (eager calls from Python would time the host's launch rate instead)
    reps = 20
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            B.dspark_observe(buf.surv, buf.window, buf.acc_len, buf.ceiling, n_bins, stats, buf.ws)
    g.replay()
    torch.cuda.synchronize(dev)
    stats.zero_()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    observe_us = e0.elapsed_time(e1) * 1e3 / reps
    st = B.dspark_read_device_status(buf.ws)
    if st != 0:
        raise RuntimeError("device status after dspark_observe: " + B.dspark_status_string(st))
    rep = B.dspark_obs_report(stats, n_bins)

    N = 1 << 20
    T_true = [1.5, 1.8, 1.2, 2.0, 1.4, 1.1, 1.7]
    z_h, c_h = I.calibration_steps(N, gamma, T_true[:gamma], seed=77, mu0=3.0, mu_slope=-0.1)
    z, c = torch.as_tensor(z_h, device=dev), torch.as_tensor(c_h, device=dev)
    grid = torch.linspace(0.5, 3.65, 64, device=dev, dtype=torch.float32)
    T = torch.zeros(gamma, dtype=torch.float32, device=dev)
    ece = torch.zeros(gamma, dtype=torch.float64, device=dev)
    ws = torch.empty(B.dspark_sts_fit_workspace_bytes(64, n_bins), dtype=torch.uint8, device=dev)
    B.dspark_sts_fit(z, c, grid, n_bins, T, ece, ws)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    B.dspark_sts_fit(z, c, grid, n_bins, T, ece, ws)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return {"observe_us_per_step": observe_us,
            "record": {"calls": reps, "verify": "cap-accept (ceiling exposed, commits as compact)",
                       "mean_window": rep["mean_window"], "mean_accepted": rep["mean_accepted"],
                       "mean_ceiling": rep["mean_ceiling"], "utilisation": rep["utilisation"],
                       "ece": rep["ece"], "bins": n_bins},
            "sts_fit": {"ms": e0.elapsed_time(e1), "prefixes": N, "positions": gamma, "grid": 64,
                        "bins": n_bins, "T_true": T_true[:gamma],
                        "T_fit": [round(float(x), 4) for x in T.tolist()],
                        "ece": [round(float(x), 5) for x in ece.tolist()]}}


def run_reference(args):
    """The CPU oracle as the reference arm, on every host core: each step is a bounded sample of
    the workload (its first 32 requests, full vocabulary, all five stages)."""
    n_req = 32
    res, cores = _oracle_steps(WORKLOAD, n_req, range(args.warmup + args.steps))
    res = res[args.warmup:]
    toks = sum(r[0] for r in res)
    secs = sum(r[1] for r in res)
    v = toks / secs
    return {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "median_ms_per_step": float(np.median([r[1] for r in res])) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": f"mixed_bs256 sample: first {n_req} of the 256 requests, full V=151936, gamma=7"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "nproc": os.cpu_count(), "kind": "oracle",
                             "sample": f"{n_req} requests per step (oracle draft and verify in {cores} worker "
                                       f"processes), {args.steps} timed steps after {args.warmup} warm-up steps"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """A small, self-contained case for ncu captures: one stage of the mixed_bs256 workload
    (bs 256, V 151936) with gamma = args.gamma, repeated args.steps times.  Prints the mean time."""
    import torch

    from speculative_decoding_draft_markov_gb300 import binding as B
    from speculative_decoding_draft_markov_gb300 import build
    from speculative_decoding_draft_markov_gb300 import inputs as I
    from speculative_decoding_draft_markov_gb300 import step as S
    build.build()
    dev = torch.device("cuda", 0)
    wl = I.WORKLOADS[WORKLOAD].with_(gamma=args.gamma)
    if args.profile_case == "observe":
        run_observe_case(args, dev)
        return
    if args.profile_case == "schedule":
        wl = I.WORKLOADS[WORKLOAD]
    inp = I.make_device_inputs(wl, dev, with_target=args.profile_case not in ("draft", "schedule"))
    bs, gamma, V = wl.bs, wl.gamma, wl.V
    cap = bs * (gamma + 1)
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype, dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    if args.profile_case == "schedule":
        # the benchmark's scheduler input: one drafted block's survival, its sawtooth table
        sps = S.sps_table(inp["T_raw"], inp["tiers"], dev)
        B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], wl.temperature, wl.seed, 0,
                             buf.tokens, buf.logit_x, buf.lse, buf.ws)
        B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], buf.tokens, inp["w"], inp["b"], inp["sts_T"],
                            buf.conf, buf.surv)
        ring = S.zos_ring(dev)
        ring.fill_(200)
        tiers = torch.as_tensor(inp["tiers"], device=dev)

        def run(it):
            B.dspark_schedule(buf.surv, sps, SCHED, buf.window, buf.K, buf.theta, buf.ws)
            B.dspark_schedule_zos_select(buf.surv, sps, ring, it, buf.window, buf.K, buf.ws)
            # the benchmark's own call: the scheduler and the pack in one launch
            B.dspark_schedule_pack(buf.surv, sps, SCHED, buf.window, buf.K, buf.theta, inp["anchor"], buf.tokens,
                                   tiers, buf.cu, buf.ids, buf.req, buf.pos, buf.padded, buf.ws)
    elif args.profile_case == "draft":
        # the benchmark's draft stage: the draft and the confidence head in one call
        def run(it):
            B.dspark_draft_confidence_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], wl.temperature, wl.seed,
                                            it, buf.tokens, buf.logit_x, buf.lse, inp["h"], inp["w"], inp["b"],
                                            inp["sts_T"], buf.conf, buf.surv, buf.ws)
    else:
        # the benchmark's own packing: its cost table and graph tiers, the global scheduler
        cap = max(cap, int(inp["tiers"][-1]))
        buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype, dev)
        sps = S.sps_table(inp["T_raw"], inp["tiers"], dev)
        S.draft_and_schedule(inp, buf, sps, wl.temperature, wl.seed, 0, SCHED,
                             tiers=torch.as_tensor(inp["tiers"], device=dev))
        S.markov_target_forward(S.gather_target_forward(inp["target"]), inp["W1"], inp["W2t"])(buf)

        def run(it):
            S.verify(inp, buf, wl.temperature, wl.seed, it)
    for it in range(2):
        run(it)
    torch.cuda.synchronize()
    ev[0].record()
    for it in range(args.steps):
        run(it)
    ev[1].record()
    torch.cuda.synchronize()
    st = B.dspark_read_device_status(buf.ws)
    print(json.dumps({"case": args.profile_case, "gamma": gamma, "ms_per_call": ev[0].elapsed_time(ev[1]) / args.steps,
                      "packed_rows": int(buf.cu[-1].item()), "status": B.dspark_status_string(st)}))
    if st != 0:
        sys.exit(1)


def run_observe_case(args, dev):
    """Observability and calibration kernels on their own: 3 + 20 dspark_observe calls of a
    bs 256, gamma 7 record (cap-accept, 15 bins; the 20 as one CUDA graph) and one
    dspark_sts_fit on 2^18 labelled prefixes (7 positions, 64 grid values, 15 bins)."""
    import torch

    from speculative_decoding_draft_markov_gb300 import binding as B
    from speculative_decoding_draft_markov_gb300 import inputs as I
    bs, gamma, n_bins = 256, 7, 15
    surv = torch.as_tensor(I.random_survival(bs, gamma, 1), device=dev)
    rng = np.random.default_rng(0)
    ceil = torch.as_tensor(rng.integers(0, gamma + 1, bs).astype(np.int32), device=dev)
    win = torch.as_tensor(rng.integers(0, gamma + 1, bs).astype(np.int32), device=dev)
    acc = torch.minimum(ceil, win).contiguous()
    stats = B.alloc_obs_stats(dev)
    ws = B.alloc_workspace(bs, gamma, 1024, dev)
    for _ in range(3):
        B.dspark_observe(surv, win, acc, ceil, n_bins, stats, ws)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(20):
            B.dspark_observe(surv, win, acc, ceil, n_bins, stats, ws)
    N = 1 << 18
    z, c = I.calibration_steps(N, gamma, [1.5] * gamma, seed=1)
    z, c = torch.as_tensor(z, device=dev), torch.as_tensor(c, device=dev)
    grid = torch.linspace(0.5, 3.65, 64, device=dev)
    T = torch.zeros(gamma, device=dev)
    e = torch.zeros(gamma, dtype=torch.float64, device=dev)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev[0].record()
    g.replay()
    ev[1].record()
    B.dspark_sts_fit(z, c, grid, n_bins, T, e)
    ev[2].record()
    torch.cuda.synchronize()
    st = B.dspark_read_device_status(ws)
    print(json.dumps({"case": "observe", "observe_us_per_call": ev[0].elapsed_time(ev[1]) * 1e3 / 20,
                      "sts_fit_ms_2e18": ev[1].elapsed_time(ev[2]), "status": B.dspark_status_string(st)}))
    if st != 0:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="all",
                    help="the configurations measured after the headline one: all (default), none, or one name "
                         "(qwen3_4b, dsv4_bs<b>_<static|compact>, long_block_t1, long_block_greedy)")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps of each further configuration")
    ap.add_argument("--profile-case", choices=["draft", "verify", "observe", "schedule"], default=None,
                    help="run one stage of the workload (small gamma) for an ncu capture; no JSON contract")
    ap.add_argument("--gamma", type=int, default=2, help="block length of --profile-case")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    args.warmup = max(args.warmup, 3)
    args.no_configs = args.workload == "none"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from speculative_decoding_draft_markov_gb300 import build
    build.build()
    res = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
