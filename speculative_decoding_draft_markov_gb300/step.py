"""One DSpark decoding step through the C ABI, on one CUDA stream, with no host readback.

    draft_block -> confidence -> schedule -> pack -> target_forward(packed ids) -> verify

or, with the asynchronous scheduler, schedule_zos_select in place of schedule and
schedule_zos_budget beside the target forward and the verify (a second stream).

`target_forward` is the caller's model: it receives the packed batch (ids / req / pos /
cu_seqlens / padded total, all on the device) and fills the packed target-logit rows.
Buffers are allocated once by PyTorch; the library itself allocates nothing."""
from __future__ import annotations

import contextlib
import dataclasses
import os
from typing import Callable, Optional

import numpy as np

from . import binding as B

# NVTX ranges around the stages (for a timeline profiler) when DSPARK_NVTX=1; off by default
_NVTX = os.environ.get("DSPARK_NVTX", "0") == "1"


@contextlib.contextmanager
def stage(name: str):
    if not _NVTX:
        yield
        return
    import torch
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


@dataclasses.dataclass
class StepBuffers:
    bs: int
    gamma: int
    V: int
    cap: int
    tokens: "object" = None
    logit_x: "object" = None
    lse: "object" = None
    conf: "object" = None
    surv: "object" = None
    window: "object" = None
    K: "object" = None
    theta: "object" = None
    cu: "object" = None
    ids: "object" = None
    req: "object" = None
    pos: "object" = None
    padded: "object" = None
    packed: "object" = None
    out_tokens: "object" = None
    acc_len: "object" = None
    ceiling: "object" = None
    ws: "object" = None

    @staticmethod
    def allocate(bs: int, gamma: int, V: int, cap: int, dtype, device="cuda") -> "StepBuffers":
        import torch
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        b = StepBuffers(bs, gamma, V, cap)
        b.tokens = torch.zeros((bs, gamma), **i32)
        b.logit_x = torch.zeros((bs, gamma), **f32)
        b.lse = torch.zeros((bs, gamma), **f32)
        b.conf = torch.zeros((bs, gamma), **f32)
        b.surv = torch.zeros((bs, gamma), **f32)
        b.window = torch.zeros(bs, **i32)
        b.K = torch.zeros(1, **i32)
        b.theta = torch.zeros(1, dtype=torch.float64, device=device)
        b.cu = torch.zeros(bs + 1, **i32)
        b.ids = torch.full((cap,), -1, **i32)
        b.req = torch.full((cap,), -1, **i32)
        b.pos = torch.full((cap,), -1, **i32)
        b.padded = torch.zeros(1, **i32)
        b.packed = torch.zeros((cap, V), dtype=dtype, device=device)
        b.out_tokens = torch.full((bs, gamma + 1), -1, **i32)
        b.acc_len = torch.zeros(bs, **i32)
        b.ceiling = torch.zeros(bs, **i32)
        b.ws = B.alloc_workspace(bs, gamma, V, device)
        return b


def sps_table(T_raw, tiers, device="cuda"):
    import torch
    return torch.tensor(B.dspark_build_sps(T_raw, tiers), dtype=torch.float64, device=device)


def gather_target_forward(target_full):
    """A stand-in target model for tests and benchmarks: the packed row p gets the precomputed
    row target_full[req[p], pos[p]] (pad rows get row 0 of request 0; verify never reads them)."""
    import torch
    bs, g1, V = target_full.shape
    flat = target_full.view(bs * g1, V)

    def fwd(buf: StepBuffers) -> None:
        idx = torch.where(buf.req >= 0, buf.req * g1 + buf.pos, torch.zeros_like(buf.req)).long()
        torch.index_select(flat, 0, idx, out=buf.packed)

    return fwd


def markov_target_forward(base_forward, W1, W2t, n_rows=None):
    """The workloads' target model, "target = U + W1[x_{k-1}] W2 + noise": the drafter's own
    logits at the drafted prefix plus noise.  base_forward fills each packed row with its base
    part (U + noise, drawn per (request, position) in advance); this adds the Markov term of the
    row's prefix.  Packed row p scores the token after ids[p] (the pack's input token of the row:
    the anchor, then the drafted tokens), so it gets W1[ids[p]] W2 -- a cuBLAS GEMM with fp32
    accumulation, standing in for the target model's own compute, rounded to the rows' dtype and
    then added to the row with one more rounding.  n_rows: a callable giving the packed total when the
    caller knows it on the host; else every row of the buffer is computed (pad rows, whose ids
    are -1, take W1[0]; verify never reads them)."""
    import torch

    def fwd(buf: StepBuffers) -> None:
        base_forward(buf)
        n = buf.packed.shape[0] if n_rows is None else int(n_rows())
        if n > 0:
            buf.packed[:n].add_(torch.matmul(W1.index_select(0, buf.ids[:n].clamp(min=0).long()), W2t.t()))

    return fwd


def zos_ring(device="cuda"):
    """The two-entry budget ring of the asynchronous scheduler, empty (-1) before the first step."""
    import torch
    return torch.full((2,), -1, dtype=torch.int32, device=device)


def draft_and_schedule(inp: dict, buf: StepBuffers, sps, temperature: float, seed: int, step: int,
                       sched_mode: int = B.DSPARK_SCHED_EARLY_STOP, mode: int = B.DSPARK_COMPACT,
                       tiers=None, stream=None, ring=None) -> None:
    """Stages S1-S4 (everything before the target forward).  With a budget ring the scheduler
    is the asynchronous one: the windows take the budget recorded two steps back
    (schedule_budget records this step's).  STATIC verification tests the whole block, so it
    needs no windows: the draft is packed as it is, without confidence or scheduler."""
    if mode == B.DSPARK_STATIC and ring is None:
        B.dspark_draft_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], temperature, seed, step,
                             buf.tokens, buf.logit_x, buf.lse, buf.ws, stream)
        B.dspark_pack(None, inp["anchor"], buf.tokens, tiers, buf.cu, buf.ids, buf.req, buf.pos, buf.padded,
                      buf.ws, stream)
        return
    # the draft and the confidence head in one call (one launch on the tensor-core pass)
    B.dspark_draft_confidence_block(inp["U"], inp["W1"], inp["W2t"], inp["anchor"], temperature, seed, step,
                                    buf.tokens, buf.logit_x, buf.lse, inp["h"], inp["w"], inp["b"], inp["sts_T"],
                                    buf.conf, buf.surv, buf.ws, stream)
    if ring is None and mode == B.DSPARK_COMPACT:  # the windows are the packing: one launch for both
        B.dspark_schedule_pack(buf.surv, sps, sched_mode, buf.window, buf.K, buf.theta, inp["anchor"], buf.tokens,
                               tiers, buf.cu, buf.ids, buf.req, buf.pos, buf.padded, buf.ws, stream)
        return
    if ring is not None:
        B.dspark_schedule_zos_select(buf.surv, sps, ring, step, buf.window, buf.K, buf.ws, stream)
    else:
        B.dspark_schedule(buf.surv, sps, sched_mode, buf.window, buf.K, buf.theta, buf.ws, stream)
    B.dspark_pack(buf.window if mode == B.DSPARK_COMPACT else None, inp["anchor"], buf.tokens, tiers,
                  buf.cu, buf.ids, buf.req, buf.pos, buf.padded, buf.ws, stream)


def verify(inp: dict, buf: StepBuffers, temperature: float, seed: int, step: int,
           mode: int = B.DSPARK_COMPACT, stream=None, states=None) -> None:
    """Stage S5 on the packed target rows in buf.packed (states: the RNN head's, if it drafted)."""
    B.dspark_verify(buf.packed, buf.cu, buf.window, mode, inp["anchor"], buf.tokens, buf.logit_x, buf.lse,
                    inp["U"], inp["W1"], inp["W2t"], temperature, seed, step, buf.out_tokens, buf.acc_len,
                    buf.ceiling, buf.ws, stream, draft_states=states)


def schedule_budget(buf: StepBuffers, sps, ring, step: int, main=None, side=None) -> None:
    """Record the budget this step's survival predicts for step + 2.  With a side stream the
    call forks off `main` (after this step's select) and `join_budget` merges it back, so it
    overlaps the target forward and the verify instead of sitting on the step's path."""
    import torch
    if side is None:
        B.dspark_schedule_zos_budget(buf.surv, sps, ring, step, buf.ws, main)
        return
    main = main if main is not None else torch.cuda.current_stream()
    side.wait_stream(main)
    B.dspark_schedule_zos_budget(buf.surv, sps, ring, step, buf.ws, side)


def join_budget(main=None, side=None) -> None:
    import torch
    if side is not None:
        (main if main is not None else torch.cuda.current_stream()).wait_stream(side)


def run_step(inp: dict, buf: StepBuffers, sps, target_forward: Callable[[StepBuffers], None],
             temperature: float, seed: int, step: int, mode: int = B.DSPARK_COMPACT,
             sched_mode: int = B.DSPARK_SCHED_EARLY_STOP, tiers=None, stream=None, ring=None,
             side_stream=None) -> None:
    with stage("dspark.draft_confidence_schedule_pack"):
        draft_and_schedule(inp, buf, sps, temperature, seed, step, sched_mode, mode, tiers, stream, ring)
    if ring is not None:
        with stage("dspark.schedule_budget"):
            schedule_budget(buf, sps, ring, step, stream, side_stream)
    with stage("dspark.target_forward"):
        target_forward(buf)
    with stage("dspark.verify"):
        verify(inp, buf, temperature, seed, step, mode, stream)
    if ring is not None:
        join_budget(stream, side_stream)


def device_inputs_from_host(host: dict, device="cuda") -> dict:
    """Copy numpy inputs (bf16 as uint16 bit patterns) to device tensors of the right dtype."""
    import torch
    out = {}
    for k, v in host.items():
        if isinstance(v, np.ndarray) and k not in ("T_raw",):
            t = torch.from_numpy(np.ascontiguousarray(v))
            if v.dtype == np.uint16:
                t = t.view(torch.int16).view(torch.bfloat16)
            out[k] = t.to(device)
        else:
            out[k] = v
    return out
