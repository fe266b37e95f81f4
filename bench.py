"""Benchmark: DSpark step tokens/s at bs=256, V=151936, gamma=7 (the mixed-difficulty batch).

One step = draft_block -> confidence -> schedule -> pack -> [target forward] -> verify, all
through the C ABI on one stream; the timed steps replay CUDA graphs captured from those calls
(one graph per stage and step, each with its own step counter), the e2e steps call the API
directly.  The target forward is the caller's model and is not part of this path: in the timed
steps it is a device row gather outside the timed segments; in the e2e steps it copies the
step's packed rows from host memory, inside the timing.  Everything else is timed with CUDA
events on the launching stream.  The L2 is flushed (256 MB write) between timed steps.
tokens/step = sum over requests of (accepted + 1).  The same steps are timed again under the
asynchronous scheduler (budget from two steps back on a second stream) and reported under "zos".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--gpus N > 1 runs under torchrun: one independent replica per GPU (the path has no
cross-request exchange that needs a collective), barrier + max-over-ranks timing; value is
the tokens of all ranks / that time ("scaling": "weak").
--impl reference times the CPU oracle (plain numpy, fp64) on bounded samples of the same
workload."""
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
_SAMPLE_CACHE = {}


def _oracle_sample(n_req: int, step: int, wl_name: str = WORKLOAD):
    """Run the oracle's full step on the first n_req requests of the workload (host inputs).
    Returns (tokens, seconds).  Inputs are generated (once per sample size) before the clock starts."""
    from oracle import dspark_oracle as O
    from speculative_decoding_draft_markov_gb300 import inputs as I
    wl = I.WORKLOADS[wl_name].with_(bs=n_req)
    if n_req not in _SAMPLE_CACHE:
        h = I.make_host_inputs(wl)
        _SAMPLE_CACHE[n_req] = (h, O.build_sps(h["T_raw"], h["tiers"]))
    host, sps = _SAMPLE_CACHE[n_req]
    t0 = time.perf_counter()
    tok, lx, lse, _ = O.draft_block(host["U"], host["W1"], host["W2t"], host["anchor"], wl.temperature, wl.seed, step)
    _, surv, _ = O.confidence(host["h"], host["W1"], host["anchor"], tok, host["w"], host["b"], host["sts_T"])
    win, K, _, _ = O.schedule(surv.astype(np.float32), sps, SCHED)
    cap = wl.bs * (wl.gamma + 1)
    cu, ids, req, pos, padded = O.pack(win, host["anchor"], tok, host["tiers"], max(cap, int(host["tiers"][-1])))
    packed = I.gather_packed_target(host["target"], req, pos, int(cu[-1]))
    _, acc, _, _ = O.verify(packed, cu, win, O.COMPACT, host["anchor"], tok, lx, lse, host["U"], host["W1"],
                            host["W2t"], wl.temperature, wl.seed, step)
    dt = time.perf_counter() - t0
    return O.step_tokens(acc), dt


def cpu_baseline(n_req: int = 64, reps: int = 4):
    """Time the oracle in a child process limited to one BLAS/OpenMP thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, json; sys.path.insert(0, %r); import bench; "
            "r = [bench._oracle_sample(%d, s) for s in range(%d)]; print(json.dumps(r))" % (ROOT, n_req, reps))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if out.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "error": out.stderr[-300:]}
    res = json.loads(out.stdout.strip().splitlines()[-1])
    tok = sum(r[0] for r in res)
    sec = sum(r[1] for r in res)
    return {"value": tok / sec, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_req} of the 256 requests, full V=151936, gamma=7, all five stages, {reps} step(s); "
                      f"{tok} tokens in {sec:.1f} s"}


# ------------------------------------------------------------------------------- GPU arm
def draft_block_bytes(bs: int, gamma: int, V: int, r: int, n_sm: int) -> int:
    """Compulsory HBM bytes of one dspark_draft_block call (bf16), position by position.
    Vocabulary pass: U_k [bs, V] and W2t [V, r] read once (a GEMM [bs, r] x [r, V] whose
    operands are consumed as they stream; W2t is re-read by every position because the positions
    are serially dependent), the gathered A rows W1[x] [bs, r], and the partial-draw entries
    written (16 bytes per request and CTA column).  Select: the entries read back, the W1 row,
    the 64 W2t rows and U_k values of the drawn draft chunk, and the three outputs."""
    n_mt = (bs + 127) // 128
    n_slots = (n_sm // n_mt)
    vocab = bs * V * 2 + V * r * 2 + bs * r * 2 + bs * n_slots * 16
    chunk = 64  # ids per draft chunk
    select = bs * (n_slots * 16 + r * 2 + chunk * r * 2 + chunk * 2 + 12)
    return gamma * (vocab + select)


def _profiled_traffic():
    """DRAM bytes of one draft block from the committed ncu summary, or None when the draft
    kernels' sources changed after that capture (the summary records their SHA-256)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "draft_block_mixed_bs256_dram.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    h = hashlib.sha256()
    for f in ("draft_tc.cu", "draft.cu", "common.cuh", "tc_ptx.cuh", "tc_host.h"):
        h.update(open(os.path.join(ROOT, "speculative_decoding_draft_markov_gb300", "csrc", f), "rb").read())
    # of the header, the constants (the kernels' sizes and chunk widths), not its documentation
    for line in open(os.path.join(ROOT, "include", "dspark.h"), "rb"):
        if line.startswith(b"#define"):
            h.update(line)
    if fields.get("sources_sha256") != h.hexdigest() or "dram_bytes_per_draft_block_gamma7" not in fields:
        return None
    return int(fields["dram_bytes_per_draft_block_gamma7"])


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


def run_ours(args, rank: int, world: int):
    import torch
    import torch.distributed as dist

    from speculative_decoding_draft_markov_gb300 import binding as B
    from speculative_decoding_draft_markov_gb300 import inputs as I
    from speculative_decoding_draft_markov_gb300 import step as S

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = I.WORKLOADS[WORKLOAD].with_(seed=I.WORKLOADS[WORKLOAD].seed + 1000 * rank)
    bs, gamma, V, r = wl.bs, wl.gamma, wl.V, wl.r
    inp = I.make_device_inputs(wl, dev)
    cap = int(I.tiers_for(wl)[-1])
    buf = S.StepBuffers.allocate(bs, gamma, V, cap, inp["U"].dtype, dev)
    sps = S.sps_table(inp["T_raw"], inp["tiers"], dev)
    tiers_dev = torch.as_tensor(inp["tiers"], device=dev)
    fwd = S.gather_target_forward(inp["target"])
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    tokens_acc = torch.zeros(1, dtype=torch.int64, device=dev)
    tau = wl.temperature

    side = torch.cuda.Stream(dev)
    ring = S.zos_ring(dev)

    def draft_stage(it):
        B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], tau, wl.seed, it, buf.tokens,
                             buf.logit_x, buf.lse, buf.ws)

    def conf_sched_pack_stage(it, zos):
        B.dspark_confidence(inp["h"], inp["W1"], inp["anchor"], buf.tokens, inp["w"], inp["b"], inp["sts_T"],
                            buf.conf, buf.surv)
        if zos:
            B.dspark_schedule_zos_select(buf.surv, sps, ring, it, buf.window, buf.K)
            B.dspark_pack(buf.window, inp["anchor"], buf.tokens, tiers_dev, buf.cu, buf.ids, buf.req, buf.pos,
                          buf.padded, buf.ws)
        else:  # the synchronous scheduler and the pack of its windows in one launch
            B.dspark_schedule_pack(buf.surv, sps, SCHED, buf.window, buf.K, buf.theta, inp["anchor"], buf.tokens,
                                   tiers_dev, buf.cu, buf.ids, buf.req, buf.pos, buf.padded, buf.ws)

    def verify_stage(it, zos):
        # asynchronous scheduler: the budget for step it + 2 forks onto a second stream and
        # runs beside the verify, joined at the end of the stage
        if zos:
            S.schedule_budget(buf, sps, ring, it, stream, side)
        S.verify(inp, buf, tau, wl.seed, it, B.DSPARK_COMPACT)
        if zos:
            S.join_budget(stream, side)

    def count_tokens():
        tokens_acc.add_((buf.acc_len.to(torch.int64) + 1).sum())

    def measure(zos):
        """Warm-up, graph capture and the timed steps of one scheduler variant."""
        for w in range(args.warmup):  # eager, through the API
            draft_stage(10_000 + w)
            conf_sched_pack_stage(10_000 + w, zos)
            fwd(buf)
            verify_stage(10_000 + w, zos)
            count_tokens()  # every op of the timed loop runs once before it (first-use set-up)
        tokens_acc.zero_()

        # The timed steps replay CUDA graphs of the same API calls, one per stage and step,
        # captured here with each step's own counter (the draws differ step to step), then
        # replayed once untimed so that the timed replays find them resident.
        graphs = []
        for it in range(args.steps):
            gs = [torch.cuda.CUDAGraph() for _ in range(3)]
            with torch.cuda.graph(gs[0]):
                draft_stage(it)
            with torch.cuda.graph(gs[1]):
                conf_sched_pack_stage(it, zos)
            with torch.cuda.graph(gs[2]):
                verify_stage(it, zos)
            graphs.append(gs)
        for gs in graphs:
            gs[0].replay()
            gs[1].replay()
            fwd(buf)
            gs[2].replay()
        torch.cuda.synchronize(dev)
        st = B.dspark_read_device_status(buf.ws)
        if st != 0:
            raise RuntimeError("device status after warm-up: " + B.dspark_status_string(st))
        tokens_acc.zero_()

        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(dev) as clk:
            t_host = time.perf_counter()
            for it in range(args.steps):
                flush.fill_(it & 0xFF)  # L2 flush, outside the timed segments
                e, gs = evs[it], graphs[it]
                e[0].record(stream)
                gs[0].replay()
                e[1].record(stream)
                gs[1].replay()
                e[2].record(stream)
                fwd(buf)  # the caller's target forward: outside the timed segments
                e[3].record(stream)
                gs[2].replay()
                e[4].record(stream)
                count_tokens()
            t_host = time.perf_counter() - t_host  # host time to enqueue (the device may still run)
            torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        seg = np.array([[e[0].elapsed_time(e[2]), e[3].elapsed_time(e[4]), e[0].elapsed_time(e[1])] for e in evs])
        st = B.dspark_read_device_status(buf.ws)
        if st != 0:
            raise RuntimeError("device status after the timed steps: " + B.dspark_status_string(st))
        tokens = int(tokens_acc.item())
        del graphs
        return seg, tokens, t_host, clk.summary()

    seg, tokens, t_host, clocks = measure(False)
    step_ms = seg[:, 0] + seg[:, 1]
    total_ms = float(step_ms.sum())
    # the same steps under the asynchronous scheduler (budget from two steps back, computed on
    # a second stream beside the verify; the select alone on the step's path)
    zseg, ztokens, _, zclocks = measure(True)
    ztotal_ms = float((zseg[:, 0] + zseg[:, 1]).sum())

    # ---- end to end through the public API with host buffers (pinned), copies inside the timing.
    # Every step copies its own inputs host -> device and reads its result back.  U, h and the
    # anchors are double-buffered, so that the copy of step t + 1 (a second stream) runs while
    # step t computes.  The target logits stay in host memory as the target model's output for
    # every (request, position); each step's target forward reads back the packed layout
    # (cu_seqlens) and copies exactly the rows that step verifies (dspark_copy_packed_rows_async).
    # The timed region holds every copy and every step; each step's inputs exceed L2.
    host = {k: inp[k].cpu().pin_memory() for k in ("U", "h", "anchor")}
    host_target = inp["target"].cpu().pin_memory()
    cu_host = torch.empty(bs + 1, dtype=torch.int32).pin_memory()
    target_rows = []

    def host_target_forward(b):
        cu_host.copy_(b.cu, non_blocking=True)
        stream.synchronize()  # the packed layout is known once the pack has run
        B.dspark_copy_packed_rows_async(b.packed, host_target, cu_host, stream)
        target_rows.append(int(cu_host[bs]))

    inps = [inp, dict(inp)]
    for k in host:
        inps[1][k] = torch.empty_like(inp[k])
    fwds = [host_target_forward, host_target_forward]
    e2e_steps = max(2, min(args.steps, 10))
    outs = [torch.empty((bs, gamma + 1), dtype=torch.int32).pin_memory() for _ in range(e2e_steps)]
    accs = [torch.empty(bs, dtype=torch.int32).pin_memory() for _ in range(e2e_steps)]
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
    for it in range(e2e_steps):
        if it + 1 < e2e_steps:
            issue_copy(it + 1)
        stream.wait_event(copied[it % 2])
        S.run_step(inps[it % 2], buf, sps, fwds[it % 2], tau, wl.seed, 20_000 + it, B.DSPARK_COMPACT, SCHED,
                   tiers=tiers_dev)
        released[it % 2].record(stream)
        outs[it].copy_(buf.out_tokens, non_blocking=True)
        accs[it].copy_(buf.acc_len, non_blocking=True)
    e1.record(stream)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_tokens = sum(int((a.to(torch.int64) + 1).sum()) for a in accs)
    row_bytes = host_target[0, 0].numel() * host_target.element_size()
    bi = sum(t.numel() * t.element_size() for t in host.values()) + int(np.mean(target_rows)) * row_bytes

    # aggregate over ranks: max time, summed tokens
    (total_ms, e2e_ms, ztotal_ms), (tokens, e2e_tokens, ztokens) = aggregate_over_ranks(
        [total_ms, e2e_ms, ztotal_ms], [tokens, e2e_tokens, ztokens], dev)
    tokens, e2e_tokens, ztokens = int(tokens), int(e2e_tokens), int(ztokens)

    obs = measure_observability(args, inp, buf, tau, wl, dev, stream, tiers_dev, fwd)

    hbm, bf16, peak_kind = _peaks()
    draft_bytes = draft_block_bytes(bs, gamma, V, r, torch.cuda.get_device_properties(dev).multi_processor_count)
    draft_ms = float(seg[:, 2].mean())
    achieved = draft_bytes / (draft_ms * 1e-3) / 1e9
    traffic = _profiled_traffic()
    # per step: gamma vocabulary passes + gamma selects, confidence, schedule+pack (one launch),
    # verify rows, decide, and at temperature > 0 the decision statistics and select
    launches_per_step = 2 * gamma + 2 + (4 if tau > 0 else 2)
    return {
        "metric": METRIC,
        "value": tokens / (total_ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; U~N(0,3^2), W~N(0,0.05^2), target = base logits + N(0,sigma^2), "
                "sigma 0.5/1/2 by thirds)",
        "config": {"workload": "mixed_bs256: bs=256, gamma=7, V=151936, r=256, d=4096, compact verify, "
                               "temperature 1, sawtooth cost table with tiers every 64 to 2048, global-argmax scheduler",
                   "global_batch": bs * world, "l2": "flushed between steps (256 MB write)",
                   "timed": "draft+confidence+schedule+pack and verify segments; target forward excluded; "
                            "each stage of each timed step a captured CUDA graph of its API calls",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_step": tokens / args.steps / world,
        "host_enqueue_ms_per_step": t_host * 1e3 / args.steps,
        "stage_ms": {"draft": draft_ms, "conf_sched_pack": float((seg[:, 0] - seg[:, 2]).mean()),
                     "verify": float(seg[:, 1].mean())},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": "dspark_draft_block: gamma tensor-core vocabulary passes (draft_tc_kernel, "
                               "the dominant kernel) + gamma selects, one C-ABI call, events around it",
                     "algorithmic_bytes": draft_bytes, "peak_kind": peak_kind},
        "e2e": {"value": e2e_tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "steps": e2e_steps,
                "note": "U, h, anchors copied from pinned host memory every step on a second stream, one step "
                        "ahead (double-buffered); the target forward copies the step's packed target rows "
                        "from pinned host memory after the pack (cu_seqlens read back); host-to-device "
                        "copies run at ~210 GB/s on this box"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "observability": obs,
        "zos": {"value": ztokens / (ztotal_ms * 1e-3), "unit": "tokens/s", "ms_per_step": ztotal_ms / args.steps,
                "tokens_per_step": ztokens / args.steps / world,
                "stage_ms": {"draft": float(zseg[:, 2].mean()),
                             "conf_sched_pack": float((zseg[:, 0] - zseg[:, 2]).mean()),
                             "verify_with_budget": float(zseg[:, 1].mean())},
                "scheduler": "asynchronous: budget from the survival two steps back (global search, second "
                             "stream beside the verify), radix top-K select on the step's path",
                "gpu_launches": (launches_per_step + 2) * args.steps, "clocks": zclocks},
    }


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
    """The CPU oracle as the reference arm: each step is a bounded sample of the workload."""
    n_req = 4
    toks, secs = 0, 0.0
    for s in range(args.warmup + args.steps):
        t, dt = _oracle_sample(n_req, s)
        if s >= args.warmup:
            toks += t
            secs += dt
    v = toks / secs
    return {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "mixed_bs256 sample: first 4 of the 256 requests, full V=151936, gamma=7"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n_req} requests per step, {args.steps} timed steps"},
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
    inp = I.make_device_inputs(wl, dev, with_hidden=args.profile_case != "draft",
                               with_target=args.profile_case not in ("draft", "schedule"))
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

        def run(it):
            B.dspark_schedule(buf.surv, sps, SCHED, buf.window, buf.K, buf.theta)
            B.dspark_schedule_zos_select(buf.surv, sps, ring, it, buf.window, buf.K)
    elif args.profile_case == "draft":
        def run(it):
            B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], wl.temperature, wl.seed, it,
                                 buf.tokens, buf.logit_x, buf.lse, buf.ws)
    else:
        sps = S.sps_table(I.cost_curve_ms(wl.with_(tier_max=cap)), np.zeros(0, np.int32), dev)
        S.draft_and_schedule(inp, buf, sps, wl.temperature, wl.seed, 0, SCHED)
        S.gather_target_forward(inp["target"])(buf)

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
                      "status": B.dspark_status_string(st)}))
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["draft", "verify", "observe", "schedule"], default=None,
                    help="run one stage of the workload (small gamma) for an ncu capture; no JSON contract")
    ap.add_argument("--gamma", type=int, default=2, help="block length of --profile-case")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    args.warmup = max(args.warmup, 3)
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
