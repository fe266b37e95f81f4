"""The oracle over many requests at once: a process pool (spawn start, one BLAS thread per
worker) that runs dspark_oracle's draft and verification on slices of a batch.

TEST INFRASTRUCTURE ONLY, like dspark_oracle itself: only tests/ and bench.py's CPU-baseline and
reference legs use it.  It adds no arithmetic: each worker receives the weights once (bf16 bit
patterns), widens them to fp64 once (exact), and calls the oracle's own functions on slices of
requests; every request keeps its own random streams (req_ids), so a slice computes exactly
what the whole batch would for those requests.  Arrays already widened are passed to the oracle
with dtype "f64" (its conversion then only copies)."""
from __future__ import annotations

import concurrent.futures as cf
import contextlib
import multiprocessing as mp
import os
import time

import numpy as np

_W = {}


def _init(W1, W2t, dtype):
    from oracle import dspark_oracle as O
    _W["W1"] = O.to_f64(W1, dtype)
    _W["W2t"] = O.to_f64(W2t, dtype)
    _W["dtype"] = dtype


def _draft(args):
    from oracle import dspark_oracle as O
    U, anchor, req_ids, temperature, seed, step = args
    t0 = time.perf_counter()
    out = O.draft_block(O.to_f64(U, _W["dtype"]), _W["W1"], _W["W2t"], anchor, temperature, seed, step,
                        dtype="f64", req_ids=req_ids)
    return out, time.perf_counter() - t0


def _verify(args):
    from oracle import dspark_oracle as O
    (packed, cu, window, mode, anchor, tokens, lx, lse, U, req_ids, temperature, seed, step) = args
    t0 = time.perf_counter()
    out = O.verify(O.to_f64(packed, _W["dtype"]), cu, window, mode, anchor, tokens, lx, lse,
                   O.to_f64(U, _W["dtype"]), _W["W1"], _W["W2t"], temperature, seed, step, dtype="f64",
                   req_ids=req_ids)
    return out, time.perf_counter() - t0


def workers() -> int:
    return max(1, min(os.cpu_count() or 1, 16))


@contextlib.contextmanager
def pool(W1, W2t, dtype: str, n: int | None = None):
    """A spawn pool whose workers hold W1, W2t (numpy; bf16 as uint16 bit patterns)."""
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        # an executor, not a Pool: a worker that dies raises BrokenProcessPool instead of hanging
        p = cf.ProcessPoolExecutor(n or workers(), mp_context=mp.get_context("spawn"), initializer=_init,
                                   initargs=(W1, W2t, dtype))
        p.submit(int, 0).result()  # start the workers while the environment says one thread each
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield p
    finally:
        p.shutdown(wait=True, cancel_futures=True)


def slices(bs: int, per: int):
    return [np.arange(i, min(bs, i + per)) for i in range(0, bs, per)]


def draft_all(p, U, anchor, temperature, seed, step, per: int = 16):
    """The oracle's draft of every request of U [bs, gamma, V]: (tokens, logit_x, lse, margin)
    and the summed worker seconds."""
    bs = U.shape[0]
    jobs = [(U[s], anchor[s], s, temperature, seed, step) for s in slices(bs, per)]
    res = list(p.map(_draft, jobs))
    parts = [r[0] for r in res]
    return tuple(np.concatenate([q[i] for q in parts]) for i in range(4)), sum(r[1] for r in res)


def verify_all(p, target, U, window, mode, anchor, tokens, lx, lse, temperature, seed, step, per: int = 16,
               static_mode: int = 0, compact_mode: int = 1):
    """The oracle's verification of every request with the given windows and draft outputs:
    each slice packs its own requests' target rows ([x_0, x_1 .. x_n] scoring rows 0 .. n, with
    n the tested window), then verifies.  Returns (out_tokens, acc_len, ceiling, margin) and the
    summed worker seconds."""
    bs, gamma = tokens.shape
    jobs = []
    for s in slices(bs, per):
        n_test = window[s] if mode == compact_mode else np.full(len(s), gamma)
        cu = np.concatenate([[0], np.cumsum(n_test + 1)]).astype(np.int32)
        packed = np.concatenate([target[r, :n + 1] for r, n in zip(s, n_test)], axis=0)
        jobs.append((packed, cu, window[s], mode, anchor[s], tokens[s], lx[s], lse[s], U[s], s, temperature,
                     seed, step))
    res = list(p.map(_verify, jobs))
    parts = [r[0] for r in res]
    return tuple(np.concatenate([q[i] for q in parts]) for i in range(4)), sum(r[1] for r in res)
