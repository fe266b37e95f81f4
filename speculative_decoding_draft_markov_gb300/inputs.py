"""Seeded synthetic inputs for the DSpark per-step token path.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It holds none of the method's arithmetic: only random draws with
the shapes and value distributions of the workloads, round-to-nearest-even
conversion to bf16, the cost curve T(M) of each workload (an input table),
and the row gather that stands in for the target model's forward pass over
the packed verify batch.

Workloads (shapes of the models and batches the pages evaluate on; the value laws
are seeded synthetic stand-ins for their data):

  tiny_fp32    bs=4,   gamma=7,  V=1024,   r=32,  d=64,   fp32
  qwen3_4b     bs=64,  gamma=7,  V=151936, r=256, d=2560, bf16
  mixed_bs256  bs=256, gamma=7,  V=151936, r=256, d=4096, bf16   (timed workload)
  dsv4_sweep   bs in {1,8,32,128,256}, gamma=5, V=129280, r=256, d=7168, bf16
  long_block   bs=128, gamma=15, V=151936, r=256, d=4096, bf16

Tensors produced (layouts are the library's):
  U       [bs, gamma, V]      draft base logits U_1..U_gamma
  W1      [V, r]              Markov factor, looked up by the previous token
  W2t     [V, r]              Markov projection stored transposed (W2 = W2t^T)
  anchor  [bs] int32          last committed token x_0
  target  [bs, gamma+1, V]    base target logits U_{j+1} + noise; row j scores the token at
                              j+1 (the workloads' target adds the Markov term W1[x_j] W2 of the
                              drafted prefix: step.markov_target_forward, after the draft)
  h       [bs, gamma, d]      backbone hidden states
  w       [d + r] f32         confidence-head weight over [h_k ; W1[x_{k-1}]]
  b       float               confidence-head bias (0)
  sts_T   [gamma] f32         per-position STS temperatures T_k = 1 + 0.1 k
  T_raw   [m_max + 1] f64     profiled step time in ms for M verify tokens
  tiers   [n] int32           captured graph totals (strictly increasing)
  Wg, bg  [2r, r], [r]        RNN head gate weights and bias (with_rnn only)
"""
from __future__ import annotations

import dataclasses
import math
from typing import Sequence

import numpy as np



# ---------------------------------------------------------------------------
# bf16 helpers (bit patterns stored as uint16 in numpy)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bit patterns.

    bits + 0x7FFF + (bit 16), then the high 16 bits, taken through a little-endian uint16 view
    (numpy's integer shifts are slow on some builds)."""
    b = np.ascontiguousarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    half = b.view(np.uint16)
    if half.size and not np.little_endian:
        raise RuntimeError("big-endian hosts are not supported")
    lsb = (half[1::2] & np.uint16(1)).astype(np.uint32)
    rounded = b + np.uint32(0x7FFF) + lsb  # wraps only for negative NaN patterns
    return np.ascontiguousarray(rounded.view(np.uint16)[1::2]).reshape(np.shape(x))


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Workload descriptions
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    bs: int
    gamma: int
    V: int
    r: int
    d: int
    dtype: str                     # "f32" or "bf16"
    u_std: float                   # std of U
    w_std: float                   # std of W1 and W2
    sigmas: Sequence[float]        # target noise std per contiguous group of requests
    temperature: float
    seed: int
    mode: str                      # verify mode of the workload
    tier_step: int                 # graph tiers every tier_step tokens (0: every M is a tier)
    tier_max: int                  # largest tier / table length m_max
    cost: str                      # "sps_direct" (tiny) or "linear_ms" (T = 5 + 0.01 * tier)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 4, 7, 1024, 32, 64, "f32", math.sqrt(2.0), 0.1,
                          (0.5, 1.0, 1.5, 2.0), 1.0, 0, "compact", 0, 64, "sps_direct"),
    "qwen3_4b": Workload("qwen3_4b", 64, 7, 151936, 256, 2560, "bf16", 3.0, 0.05,
                         (1.0,), 1.0, 1, "compact", 16, 512, "linear_ms"),
    "mixed_bs256": Workload("mixed_bs256", 256, 7, 151936, 256, 4096, "bf16", 3.0, 0.05,
                            (0.5, 1.0, 2.0), 1.0, 2, "compact", 64, 2048, "linear_ms"),
    "dsv4_sweep": Workload("dsv4_sweep", 256, 5, 129280, 256, 7168, "bf16", 3.0, 0.05,
                           (1.0,), 1.0, 3, "compact", 16, 6 * 256, "linear_ms"),
    "long_block": Workload("long_block", 128, 15, 151936, 256, 4096, "bf16", 3.0, 0.05,
                           (1.25,), 1.0, 4, "compact", 128, 2048, "linear_ms"),
}

DSV4_BATCHES = (1, 8, 32, 128, 256)


def dsv4(bs: int) -> Workload:
    """The DeepSeek-V4-shaped sweep point at batch bs: tiers every 16 up to (gamma+1)*bs."""
    g = WORKLOADS["dsv4_sweep"]
    return g.with_(name=f"dsv4_bs{bs}", bs=bs, tier_max=(g.gamma + 1) * bs)


def sigma_per_request(bs: int, sigmas: Sequence[float]) -> np.ndarray:
    """Split the batch into len(sigmas) contiguous groups (floor boundaries) with one noise std each."""
    g = len(sigmas)
    out = np.empty(bs, dtype=np.float64)
    for i in range(g):
        lo, hi = (i * bs) // g, ((i + 1) * bs) // g
        out[lo:hi] = sigmas[i]
    return out


def tiers_for(wl: Workload) -> np.ndarray:
    """Captured graph totals: every tier_step up to tier_max, tier_max itself always included.

    tier_step == 0 means every total is its own tier (no padding): an empty list."""
    if wl.tier_step == 0:
        return np.zeros(0, dtype=np.int32)
    t = list(range(wl.tier_step, wl.tier_max, wl.tier_step)) + [wl.tier_max]
    return np.asarray(sorted(set(t)), dtype=np.int32)


def cost_curve_ms(wl: Workload) -> np.ndarray:
    """Profiled step time T_raw[M] for M = 0..m_max (an input table, like a start-up profile).

    tiny: SPS(M) = 1 / (1 + 0.002 M) is given, i.e. T = 1 + 0.002 M.
    others: T = 5 ms + 0.01 ms per verify token (graph padding applied by the table builder)."""
    M = np.arange(wl.tier_max + 1, dtype=np.float64)
    if wl.cost == "sps_direct":
        return 1.0 + 0.002 * M
    return 5.0 + 0.01 * M


# ---------------------------------------------------------------------------
# Host (numpy) generator
# ---------------------------------------------------------------------------

_TAGS = {"U": 1, "Ux": 2, "W1": 3, "W2t": 4, "anchor": 5, "noise": 6, "h": 7, "w": 8, "Wg": 9, "bg": 10}


def _rng(seed: int, tag: str, extra: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), _TAGS[tag], int(extra)]))


def _as_dtype(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    return f32_to_bf16_bits(x32)


def rnn_gate_std(wl: Workload) -> float:
    """Std of the RNN head's gate weights Wg [2r, r]: the gate pre-activation [e ; s] Wg has
    unit variance when e and s have the weights' std (w_std)."""
    return 1.0 / (wl.w_std * math.sqrt(2 * wl.r))


def make_host_inputs(wl: Workload, with_target: bool = True, with_hidden: bool = True,
                     with_rnn: bool = False) -> dict:
    """All inputs of one step as numpy arrays (bf16 tensors as uint16 bit patterns).
    with_rnn adds the RNN head's gate weights: Wg [2r, r] ~ N(0, rnn_gate_std^2) in the
    workload's dtype and bg [r] ~ N(0, 1) float32."""
    bs, g, V, r, d = wl.bs, wl.gamma, wl.V, wl.r, wl.d
    s = wl.seed
    U32 = (_rng(s, "U").standard_normal((bs, g, V), dtype=np.float32) * np.float32(wl.u_std))
    out = {
        "U": _as_dtype(U32, wl.dtype),
        "W1": _as_dtype(_rng(s, "W1").standard_normal((V, r), dtype=np.float32) * np.float32(wl.w_std), wl.dtype),
        "W2t": _as_dtype(_rng(s, "W2t").standard_normal((V, r), dtype=np.float32) * np.float32(wl.w_std), wl.dtype),
        "anchor": _rng(s, "anchor").integers(0, V, size=bs, dtype=np.int64).astype(np.int32),
        "b": 0.0,
        "sts_T": (1.0 + 0.1 * np.arange(1, g + 1)).astype(np.float32),
        "T_raw": cost_curve_ms(wl),
        "tiers": tiers_for(wl),
        "dtype": wl.dtype,
    }
    if with_hidden:
        out["h"] = _as_dtype(_rng(s, "h").standard_normal((bs, g, d), dtype=np.float32), wl.dtype)
        out["w"] = (_rng(s, "w").standard_normal(d + r) / math.sqrt(d + r)).astype(np.float32)
    if with_rnn:
        out["Wg"] = _as_dtype(_rng(s, "Wg").standard_normal((2 * r, r), dtype=np.float32)
                              * np.float32(rnn_gate_std(wl)), wl.dtype)
        out["bg"] = _rng(s, "bg").standard_normal(r).astype(np.float32)
    if with_target:
        # target row j (scoring the token at j+1) = base logits of that position + noise;
        # row gamma (the bonus row) takes an extra independent base-logit draw.
        Ux = _rng(s, "Ux").standard_normal((bs, 1, V), dtype=np.float32) * np.float32(wl.u_std)
        Ubase = U32 if wl.dtype == "f32" else bf16_bits_to_f32(out["U"])
        Uxb = Ux if wl.dtype == "f32" else bf16_bits_to_f32(f32_to_bf16_bits(Ux))
        sig = sigma_per_request(bs, wl.sigmas).astype(np.float32)[:, None, None]
        noise = _rng(s, "noise").standard_normal((bs, g + 1, V), dtype=np.float32) * sig
        out["target"] = _as_dtype(np.concatenate([Ubase, Uxb], axis=1) + noise, wl.dtype)
    return out


def random_survival(bs: int, gamma: int, seed: int, ties: bool = False) -> np.ndarray:
    """A [bs, gamma] float32 array, non-increasing along each row, in (0, 1].

    With ties=True values are drawn from a coarse grid so that equal keys occur."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 101]))
    if ties:
        v = rng.integers(1, 9, size=(bs, gamma)).astype(np.float32) / np.float32(8)
    else:
        v = rng.random((bs, gamma), dtype=np.float32)
        v = np.maximum(v, np.float32(1e-7))
    return -np.sort(-v, axis=1)


def calibration_steps(N: int, gamma: int, T_true, seed: int, mu0: float = 2.5, mu_slope: float = -0.25,
                      z_std: float = 1.5):
    """Synthetic labelled steps for the temperature fit (no real drafter: a known law).

    Confidence logits z[i, k] ~ N(mu0 + mu_slope k, z_std^2) (float32).  Position k + 1 passes,
    given that its prefix passed, with probability 1 / (1 + exp(-z[i, k] / T_true[k])); the
    label is the accepted prefix length (the ceiling of a full-block verification).
    Returns (z [N, gamma] float32, ceiling [N] int32)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 104]))
    z = (mu0 + mu_slope * np.arange(gamma)[None, :]
         + z_std * rng.standard_normal((N, gamma))).astype(np.float32)
    T = np.asarray(T_true, dtype=np.float64)[None, :]
    p_pass = 1.0 / (1.0 + np.exp(-z.astype(np.float64) / T))
    passes = rng.random((N, gamma)) < p_pass
    ceiling = np.where(passes.all(axis=1), gamma, np.argmin(passes, axis=1)).astype(np.int32)
    return z, ceiling


def random_windows(bs: int, gamma: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed, 102]))
    return rng.integers(0, gamma + 1, size=bs).astype(np.int32)


def random_tokens(bs: int, gamma: int, V: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed, 103]))
    return rng.integers(0, V, size=(bs, gamma)).astype(np.int32)


def gather_packed_target(target: np.ndarray, req: np.ndarray, pos: np.ndarray, rows: int) -> np.ndarray:
    """Stand-in for the target forward on the packed batch: row p = target[req[p], pos[p]].

    Pad rows (req == -1) are zero.  The result has `rows` rows (>= the packed total)."""
    V = target.shape[2]
    out = np.zeros((rows, V), dtype=target.dtype)
    n = min(rows, len(req))
    sel = np.nonzero(req[:n] >= 0)[0]
    out[sel] = target[req[sel], pos[sel]]
    return out


# ---------------------------------------------------------------------------
# Device (torch) generator for full-size workloads
# ---------------------------------------------------------------------------

def make_device_inputs(wl: Workload, device, with_target: bool = True, with_hidden: bool = True,
                       with_rnn: bool = False) -> dict:
    """Same recipe as make_host_inputs, drawn on the device with torch's seeded generator.

    The draws differ bit-wise from the numpy ones (another generator) but follow the same
    laws; tests that compare with the oracle copy these exact tensors to the host."""
    import torch

    bs, g, V, r, d = wl.bs, wl.gamma, wl.V, wl.r, wl.d
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16

    def gen(tag: str) -> "torch.Generator":
        gg = torch.Generator(device=device)
        gg.manual_seed(int(wl.seed) * 1000003 + _TAGS[tag])
        return gg

    def normal(shape, std, tag):
        x = torch.empty(shape, device=device, dtype=torch.float32)
        x.normal_(0.0, float(std), generator=gen(tag))
        return x

    U32 = normal((bs, g, V), wl.u_std, "U")
    out = {
        "U": U32.to(tdt),
        "W1": normal((V, r), wl.w_std, "W1").to(tdt),
        "W2t": normal((V, r), wl.w_std, "W2t").to(tdt),
        "anchor": torch.randint(0, V, (bs,), generator=gen("anchor"), device=device, dtype=torch.int64).to(torch.int32),
        "b": 0.0,
        "sts_T": torch.tensor(1.0 + 0.1 * np.arange(1, g + 1), dtype=torch.float32, device=device),
        "T_raw": cost_curve_ms(wl),
        "tiers": tiers_for(wl),
        "dtype": wl.dtype,
    }
    del U32
    if with_hidden:
        out["h"] = normal((bs, g, d), 1.0, "h").to(tdt)
        out["w"] = normal((d + r,), 1.0 / math.sqrt(d + r), "w")
    if with_rnn:
        out["Wg"] = normal((2 * r, r), rnn_gate_std(wl), "Wg").to(tdt)
        out["bg"] = normal((r,), 1.0, "bg")
    if with_target:
        sig = torch.tensor(sigma_per_request(bs, wl.sigmas), dtype=torch.float32, device=device)
        target = torch.empty((bs, g + 1, V), device=device, dtype=tdt)
        noise_gen = gen("noise")
        for j in range(g + 1):  # row by row keeps the fp32 temporaries small
            base = out["U"][:, j].float() if j < g else normal((bs, V), wl.u_std, "Ux").to(tdt).float()
            nz = torch.empty((bs, V), device=device, dtype=torch.float32)
            nz.normal_(0.0, 1.0, generator=noise_gen)
            target[:, j] = (base + nz * sig[:, None]).to(tdt)
        out["target"] = target
    return out
