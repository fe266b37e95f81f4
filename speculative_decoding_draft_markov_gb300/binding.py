"""Thin ctypes binding over libdspark.so (include/dspark.h).

Same names as the C ABI; the only work here is argument marshalling: sizes are read from
tensor shapes, pointers from data_ptr(), the stream from torch's current stream.  Every
step of the path runs in the library's CUDA kernels.  If the library is missing the
calls raise -- there is no fallback."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

DSPARK_OK, DSPARK_EINVAL, DSPARK_EUNSUPPORTED, DSPARK_ECUDA, DSPARK_ETIMEOUT, DSPARK_EWORKSPACE = range(6)
DSPARK_F32, DSPARK_BF16 = 0, 1
DSPARK_STATIC, DSPARK_COMPACT, DSPARK_CAP_ACCEPT = 0, 1, 2
DSPARK_SCHED_EARLY_STOP, DSPARK_SCHED_GLOBAL_ARGMAX = 0, 1
DSPARK_MAX_BS, DSPARK_MAX_GAMMA, DSPARK_CHUNK, DSPARK_DRAFT_CHUNK = 256, 16, 128, 64

_vp, _i, _f, _u64, _sz, _d = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_double

_SIGS = {
    "dspark_status_string": (ctypes.c_char_p, [_i]),
    "dspark_workspace_bytes": (_sz, [_i, _i, _i]),
    "dspark_workspace_init": (_i, [_vp, _sz, _vp]),
    "dspark_read_device_status": (_i, [_vp, _vp]),
    "dspark_build_sps": (_i, [_vp, _i, _vp, _i, _vp]),
    "dspark_copy_packed_rows_async": (_i, [_vp, _vp, _sz, _i, _i, _vp, _vp]),
    "dspark_set_wait_timeout_ns": (_u64, [_u64]),
    "dspark_draft_block": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _f, _u64, _u64,
                                _vp, _vp, _vp, _vp, _sz, _vp]),
    "dspark_draft_confidence_block": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _f, _u64, _u64,
                                           _vp, _vp, _vp, _vp, _i, _vp, _f, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dspark_draft_block_noalloc": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _f, _u64, _u64,
                                        _vp, _vp, _vp, _vp, _vp]),
    "dspark_draft_block_rnn": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _f, _u64, _u64,
                                    _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dspark_confidence": (_i, [_vp, _vp, _i, _vp, _vp, _vp, _f, _vp, _i, _i, _i, _i, _i,
                               _vp, _vp, _vp, _vp]),
    "dspark_schedule": (_i, [_vp, _i, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dspark_schedule_zos_select": (_i, [_vp, _i, _i, _vp, _i, _vp, _u64, _vp, _vp, _vp, _sz, _vp]),
    "dspark_schedule_zos_budget": (_i, [_vp, _i, _i, _vp, _i, _vp, _u64, _vp, _sz, _vp]),
    "dspark_pack": (_i, [_vp, _vp, _vp, _i, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dspark_schedule_pack": (_i, [_vp, _i, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _sz, _vp]),
    "dspark_observe": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "dspark_obs_report": (_i, [_vp, _i, _vp]),
    "dspark_sts_fit_workspace_bytes": (_sz, [_i, _i]),
    "dspark_sts_fit": (_i, [_vp, _vp, _i, _i, _vp, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "dspark_verify": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                           _i, _f, _u64, _u64, _vp, _vp, _vp, _vp, _sz, _vp]),
}

_LIB: Optional[ctypes.CDLL] = None


class DSparkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dspark_status_string(status) if _LIB else status}")


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libdspark.so (built by __graft_entry__.build()); raise if it is not there."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libdspark.so is not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _LIB = L
    return _LIB


def _check(rc: int, where: str) -> None:
    if rc != DSPARK_OK:
        raise DSparkError(rc, where)


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdspark must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DSPARK_F32
    if t.dtype == torch.bfloat16:
        return DSPARK_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------------------- utilities

def dspark_status_string(status: int) -> str:
    return lib().dspark_status_string(int(status)).decode()


def dspark_workspace_bytes(bs: int, gamma: int, V: int) -> int:
    return int(lib().dspark_workspace_bytes(bs, gamma, V))


def dspark_workspace_init(ws, stream=None) -> None:
    _check(lib().dspark_workspace_init(_p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "dspark_workspace_init")


def dspark_read_device_status(ws, stream=None) -> int:
    return int(lib().dspark_read_device_status(_p(ws), _stream(stream)))


def dspark_set_wait_timeout_ns(ns: int) -> int:
    """Deadline of device-side waits in the tensor-core kernels; returns the previous value."""
    return int(lib().dspark_set_wait_timeout_ns(int(ns)))


def alloc_workspace(bs: int, gamma: int, V: int, device="cuda"):
    """A zero-initialised workspace tensor (allocated by PyTorch) for one step."""
    import torch
    n = dspark_workspace_bytes(bs, gamma, V)
    if n == 0:
        raise ValueError("invalid sizes for a workspace")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    dspark_workspace_init(ws)
    return ws


def dspark_build_sps(T_raw, tiers) -> np.ndarray:
    """Host cost-table builder: sps[M] = 1 / T_mono(tier(M))."""
    T = np.ascontiguousarray(T_raw, dtype=np.float64)
    t = np.ascontiguousarray(tiers, dtype=np.int32)
    out = np.empty_like(T)
    _check(lib().dspark_build_sps(T.ctypes.data, T.size - 1, t.ctypes.data if t.size else None,
                                  t.size, out.ctypes.data), "dspark_build_sps")
    return out


def dspark_copy_packed_rows_async(packed, rows_host, cu_host, stream=None) -> None:
    """Enqueue the host-to-device copies of the rows a packed batch reads: request r's rows
    0 .. n_r - 1 of rows_host [bs, rows_per_req, ...] (pinned CPU tensor) into packed rows
    cu[r] .. cu[r+1] - 1 of `packed` (device); cu_host is the batch's cu_seqlens on the host."""
    import torch
    if rows_host.is_cuda or cu_host.device.type != "cpu":
        raise ValueError("rows_host and cu_host must be host tensors")
    if cu_host.dtype != torch.int32 or cu_host.numel() != rows_host.shape[0] + 1:
        raise ValueError("cu_host must be int32 with one entry per request plus one")
    cu = cu_host.contiguous()
    bs, rpr = rows_host.shape[0], rows_host.shape[1]
    row_bytes = rows_host[0, 0].numel() * rows_host.element_size()
    _check(lib().dspark_copy_packed_rows_async(_p(packed), _p(rows_host), row_bytes, bs, rpr, cu.data_ptr(),
                                               _stream(stream)), "dspark_copy_packed_rows_async")


# ----------------------------------------------------------------------------- the path

def dspark_draft_block(U, W1, W2t, anchor, temperature, seed, step, tokens, logit_x, lse, ws, stream=None):
    bs, gamma, V = U.shape
    r = W1.shape[1]
    _check(lib().dspark_draft_block(_p(U), _p(W1), _p(W2t), _dtype(U), _p(anchor), bs, gamma, V, r,
                                    float(temperature), int(seed), int(step), _p(tokens), _p(logit_x),
                                    _p(lse), _p(ws), ws.numel(), _stream(stream)), "dspark_draft_block")


def dspark_draft_confidence_block(U, W1, W2t, anchor, temperature, seed, step, tokens, logit_x, lse, h, w, b, sts_T,
                                  conf, surv, ws, stream=None, z_logit=None):
    """dspark_draft_block then dspark_confidence on the drafted tokens, as one call (the confidence
    computed inside the draft's launch on the tensor-core pass)."""
    bs, gamma, V = U.shape
    r = W1.shape[1]
    d = h.shape[2]
    _check(lib().dspark_draft_confidence_block(_p(U), _p(W1), _p(W2t), _dtype(U), _p(anchor), bs, gamma, V, r,
                                               float(temperature), int(seed), int(step), _p(tokens), _p(logit_x),
                                               _p(lse), _p(h), d, _p(w), float(b), _p(sts_T), _p(conf), _p(surv),
                                               _p(z_logit), _p(ws), ws.numel(), _stream(stream)),
           "dspark_draft_confidence_block")


def dspark_draft_block_noalloc(U, W1, W2t, anchor, temperature, seed, step, tokens, logit_x, lse,
                               device_status=None, stream=None):
    """The draft without a workspace, for callers that cannot allocate device memory: the
    library's own fixed scratch array is used (see include/dspark.h for its limit and rules)."""
    bs, gamma, V = U.shape
    r = W1.shape[1]
    _check(lib().dspark_draft_block_noalloc(_p(U), _p(W1), _p(W2t), _dtype(U), _p(anchor), bs, gamma, V, r,
                                            float(temperature), int(seed), int(step), _p(tokens), _p(logit_x),
                                            _p(lse), _p(device_status), _stream(stream)),
           "dspark_draft_block_noalloc")


def dspark_draft_block_rnn(U, W1, W2t, Wg, bg, anchor, temperature, seed, step, tokens, logit_x, lse, states, ws,
                           stream=None):
    """The block draft with the RNN head: Wg [2r, r] (U's dtype), bg [r] fp32; writes the
    recurrent states s_1..s_gamma into states [bs, gamma, r] (U's dtype)."""
    bs, gamma, V = U.shape
    r = W1.shape[1]
    _check(lib().dspark_draft_block_rnn(_p(U), _p(W1), _p(W2t), _p(Wg), _p(bg), _dtype(U), _p(anchor), bs, gamma, V,
                                        r, float(temperature), int(seed), int(step), _p(tokens), _p(logit_x), _p(lse),
                                        _p(states), _p(ws), ws.numel(), _stream(stream)), "dspark_draft_block_rnn")


def dspark_confidence(h, W1, anchor, tokens, w, b, sts_T, conf, surv, stream=None, z_logit=None):
    bs, gamma, d = h.shape
    V, r = W1.shape
    _check(lib().dspark_confidence(_p(h), _p(W1), _dtype(h), _p(anchor), _p(tokens), _p(w), float(b),
                                   _p(sts_T), bs, gamma, d, r, V, _p(conf), _p(surv), _p(z_logit),
                                   _stream(stream)), "dspark_confidence")


def dspark_schedule(surv, sps, mode, window, K_out, theta_out, ws, stream=None):
    bs, gamma = surv.shape
    _check(lib().dspark_schedule(_p(surv), bs, gamma, _p(sps), sps.numel() - 1, int(mode), _p(window),
                                 _p(K_out), _p(theta_out), _p(ws), ws.numel(), _stream(stream)), "dspark_schedule")


def dspark_schedule_zos_select(surv, sps, budget_ring, step, window, K_out, ws, stream=None):
    bs, gamma = surv.shape
    _check(lib().dspark_schedule_zos_select(_p(surv), bs, gamma, _p(sps), sps.numel() - 1, _p(budget_ring),
                                            int(step), _p(window), _p(K_out), _p(ws), ws.numel(), _stream(stream)),
           "dspark_schedule_zos_select")


def dspark_schedule_zos_budget(surv, sps, budget_ring, step, ws, stream=None):
    bs, gamma = surv.shape
    _check(lib().dspark_schedule_zos_budget(_p(surv), bs, gamma, _p(sps), sps.numel() - 1, _p(budget_ring),
                                            int(step), _p(ws), ws.numel(), _stream(stream)),
           "dspark_schedule_zos_budget")


def dspark_pack(window, anchor, tokens, tiers, cu_seqlens, ids, req, pos, padded_total, ws, stream=None):
    bs, gamma = tokens.shape
    n_t = 0 if tiers is None else tiers.numel()
    _check(lib().dspark_pack(_p(window), _p(anchor), _p(tokens), bs, gamma, _p(tiers) if n_t else None, n_t,
                             ids.numel(), _p(cu_seqlens), _p(ids), _p(req), _p(pos), _p(padded_total),
                             _p(ws), ws.numel(), _stream(stream)), "dspark_pack")


def dspark_schedule_pack(surv, sps, mode, window, K_out, theta_out, anchor, tokens, tiers, cu_seqlens, ids, req,
                         pos, padded_total, ws, stream=None):
    """dspark_schedule then dspark_pack of its windows, in one launch."""
    bs, gamma = surv.shape
    n_t = 0 if tiers is None else tiers.numel()
    _check(lib().dspark_schedule_pack(_p(surv), bs, gamma, _p(sps), sps.numel() - 1, mode, _p(window), _p(K_out),
                                      _p(theta_out), _p(anchor), _p(tokens), _p(tiers) if n_t else None, n_t,
                                      ids.numel(), _p(cu_seqlens), _p(ids), _p(req), _p(pos), _p(padded_total),
                                      _p(ws), ws.numel(), _stream(stream)), "dspark_schedule_pack")


def dspark_verify(target, cu_seqlens, window, mode, anchor, tokens, logit_x, lse, U, W1, W2t,
                  temperature, seed, step, out_tokens, acc_len, ceiling, ws, stream=None, draft_logits=None,
                  draft_states=None):
    """draft_logits [bs, gamma, V] (optional): the draft's logits; then U, W1, W2t may be None.
    draft_states [bs, gamma, r] (optional): the RNN head's states (dspark_draft_block_rnn)."""
    bs, gamma = tokens.shape
    V = target.shape[1]
    r = W1.shape[1] if W1 is not None else 0
    _check(lib().dspark_verify(_p(target), _dtype(target), _p(cu_seqlens), _p(window), int(mode), bs, gamma,
                               V, _p(anchor), _p(tokens), _p(logit_x), _p(lse), _p(draft_logits),
                               _p(draft_states), _p(U), _p(W1),
                               _p(W2t), r,
                               float(temperature), int(seed), int(step), _p(out_tokens), _p(acc_len),
                               _p(ceiling), _p(ws), ws.numel(), _stream(stream)), "dspark_verify")


# ----------------------------------------------------------------------------- observability

DSPARK_OBS_MAX_BINS = 64
_H = DSPARK_MAX_GAMMA + 1


class ObsStats(ctypes.Structure):
    """dspark_obs_stats (include/dspark.h), field for field."""
    _fields_ = [(n, ctypes.c_int64) for n in ("steps", "requests", "sum_window", "sum_accepted",
                                               "ceiling_requests", "sum_ceiling", "sum_accepted_ceiling",
                                               "reserved")] + \
               [("window_hist", ctypes.c_int64 * _H), ("accepted_hist", ctypes.c_int64 * _H),
                ("ceiling_hist", ctypes.c_int64 * _H),
                ("bin_count", ctypes.c_int64 * DSPARK_OBS_MAX_BINS), ("bin_label", ctypes.c_int64 * DSPARK_OBS_MAX_BINS),
                ("bin_score_fx", ctypes.c_int64 * DSPARK_OBS_MAX_BINS),
                ("pos_count", ctypes.c_int64 * DSPARK_MAX_GAMMA), ("pos_label", ctypes.c_int64 * DSPARK_MAX_GAMMA),
                ("pos_score_fx", ctypes.c_int64 * DSPARK_MAX_GAMMA)]


class ObsSummary(ctypes.Structure):
    """dspark_obs_summary (include/dspark.h)."""
    _fields_ = [(n, ctypes.c_double) for n in ("mean_window", "mean_accepted", "mean_ceiling", "utilisation",
                                                "ece")] + \
               [("pos_mean_survival", ctypes.c_double * DSPARK_MAX_GAMMA),
                ("pos_pass_rate", ctypes.c_double * DSPARK_MAX_GAMMA), ("scored", ctypes.c_int64)]


def alloc_obs_stats(device="cuda"):
    """Zeroed device records (an int64 tensor laid out as dspark_obs_stats)."""
    import torch
    return torch.zeros(ctypes.sizeof(ObsStats) // 8, dtype=torch.int64, device=device)


def obs_stats_from(stats) -> ObsStats:
    """Host copy of device records as the C structure."""
    host = stats.detach().cpu().numpy().astype(np.int64)
    out = ObsStats()
    ctypes.memmove(ctypes.addressof(out), host.ctypes.data, ctypes.sizeof(ObsStats))
    return out


def dspark_observe(surv, window, acc_len, ceiling, n_bins, stats, ws, stream=None):
    bs, gamma = surv.shape
    _check(lib().dspark_observe(_p(surv), _p(window), _p(acc_len), _p(ceiling), bs, gamma, int(n_bins), _p(stats),
                                _p(ws), ws.numel() * ws.element_size(), _stream(stream)), "dspark_observe")


def dspark_obs_report(stats, n_bins) -> dict:
    """The host summary of device (or host ObsStats) records, as a dict."""
    st = stats if isinstance(stats, ObsStats) else obs_stats_from(stats)
    out = ObsSummary()
    _check(lib().dspark_obs_report(ctypes.addressof(st), int(n_bins), ctypes.addressof(out)), "dspark_obs_report")
    return {"mean_window": out.mean_window, "mean_accepted": out.mean_accepted, "mean_ceiling": out.mean_ceiling,
            "utilisation": out.utilisation, "ece": out.ece, "scored": out.scored,
            "pos_mean_survival": list(out.pos_mean_survival), "pos_pass_rate": list(out.pos_pass_rate)}


def dspark_sts_fit_workspace_bytes(n_grid: int, n_bins: int) -> int:
    return int(lib().dspark_sts_fit_workspace_bytes(int(n_grid), int(n_bins)))


def dspark_sts_fit(z, ceiling, grid, n_bins, T_out, ece_out, ws=None, stream=None):
    """Sequential temperature scaling fit on labelled steps (device tensors); allocates its
    scratch with PyTorch when `ws` is None."""
    import torch
    N, gamma = z.shape
    n_grid = grid.numel()
    nbytes = dspark_sts_fit_workspace_bytes(n_grid, n_bins)
    if ws is None:
        ws = torch.empty(max(nbytes, 8), dtype=torch.uint8, device=z.device)
    _check(lib().dspark_sts_fit(_p(z), _p(ceiling), N, gamma, _p(grid), n_grid, int(n_bins), _p(T_out), _p(ece_out),
                                _p(ws), ws.numel() * ws.element_size(), _stream(stream)), "dspark_sts_fit")
