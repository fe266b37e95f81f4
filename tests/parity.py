"""Helpers for GPU-vs-oracle parity tests.

Decision rule (the stated parity tolerances): integer decisions (tokens, accepted lengths,
windows, cu_seqlens) must match exactly unless the oracle's own decision margin -- the
top-two key gap of a Gumbel-max draw or argmax, or |u - p_t/p_d| of an accept test -- is
below NEAR (1e-4); such near-margin decisions are counted and must stay rare.
Probabilities / confidences: relative 2e-3 for bf16 inputs, 1e-5 for fp32 inputs."""
import numpy as np

NEAR = 1e-4
TOL = {"bf16": 2e-3, "f32": 1e-5}


def to_np(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def compare_draft(tok_g, lx_g, lse_g, tok_o, lx_o, lse_o, margin_o, dtype, greedy=False):
    """Return (checked positions, near-margin divergences).  Rows are compared position by
    position until the first divergence; a divergence must be near-margin."""
    tol = TOL[dtype]
    bs, gamma = tok_o.shape
    checked = near = 0
    for r in range(bs):
        for k in range(gamma):
            if tok_g[r, k] != tok_o[r, k]:
                assert margin_o[r, k] < NEAR, (
                    f"draft token mismatch at row {r} pos {k + 1}: gpu {tok_g[r, k]} oracle {tok_o[r, k]} "
                    f"margin {margin_o[r, k]:.3g}")
                near += 1
                break
            checked += 1
            if greedy:
                assert abs(lx_g[r, k] - lx_o[r, k]) <= tol * max(1.0, abs(lx_o[r, k])), (r, k)
            else:
                # log p_d of the drawn token and the row log-sum-exp
                dg = lx_g[r, k] - lse_g[r, k]
                do = lx_o[r, k] - lse_o[r, k]
                assert abs(np.expm1(dg - do)) <= tol, (r, k, dg, do)
                assert abs(lse_g[r, k] - lse_o[r, k]) <= tol * max(1.0, abs(lse_o[r, k])), (r, k)
    return checked, near


def compare_verify(out_g, acc_g, out_o, acc_o, margin_o, ceil_g=None, ceil_o=None):
    checked = near = 0
    for r in range(out_o.shape[0]):
        same = (acc_g[r] == acc_o[r]) and np.array_equal(out_g[r], out_o[r])
        if ceil_g is not None:
            same = same and ceil_g[r] == ceil_o[r]
        if not same:
            assert margin_o[r] < NEAR, (f"verify mismatch at request {r}: gpu {out_g[r]} / {acc_g[r]} "
                                        f"oracle {out_o[r]} / {acc_o[r]} margin {margin_o[r]:.3g}")
            near += 1
        else:
            checked += 1
    return checked, near
