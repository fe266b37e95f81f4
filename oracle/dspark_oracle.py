"""CPU reference oracle for the DSpark per-step token path (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import this module.  It shares no code with the
CUDA library: the only common module is the seeded input generator, which holds
none of the method's arithmetic.

It computes, plainly and slowly, in IEEE double:
  S1 draft_block   -- Markov sequential head, left-to-right sampling
     rnn_draft_block -- the same with the RNN sequential head (gated recurrent state)
  S2 confidence    -- confidence head + sequential temperature scaling + prefix survival
  S3 schedule      -- hardware-aware global top-B prefix scheduler
  S4 pack          -- ragged cu_seqlens packing rounded up to a captured graph tier
  S5 verify        -- rejection-sampling verification (static / compact / cap-accept, greedy)
  zos_*            -- the asynchronous scheduler (budget predicted two steps back)
  observe, sts_fit -- observability records (ceiling, utilisation, ECE) and the sequential
                      temperature scaling fit
plus the host cost-table preparation (build_sps) and the shared random-number
contract (Philox4x32-10 uniforms, Gumbel keys, the two-level samplers: Gumbel-max over
chunks, then inverse CDF (draft) or Gumbel-max (verification) inside the drawn chunk).

Sources, cited by page and section:
  [SUMMARY]  "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
             Generation" -- technical summary page (AI Research survey), sections
             "Architecture (drafter)", "Verification scheduling (system side)", "Infra".
  [SGLANG]   "DSpark in SGLang" blog post (Vietnamese and Chinese translations), sections
             "Verify modes", "Ragged verify under full CUDA graphs" (Fig. 2),
             "Observability", "Per-request differentiation under mixed traffic" (Fig. 4),
             "ZOS", "Cost-table profiling" (Fig. 6).
  [VLLM]     "vLLM adaptive verification with DSpark", sections "DSpark confidence
             scheduling mechanism", "Technical implementation and CUDA Graphs".
  [PHILOX]   Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
             SC'11 -- the Philox4x32 round function, multipliers and Weyl key schedule.

Where the pages are silent the reading taken is stated at the function.  Every
function here is pinned by tests under tests/
(test_oracle_*.py) against closed forms, brute force, distributional tests and an
independent library Philox.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

CHUNK = 128        # ids per chunk of verify's draws (residual and bonus)
DRAFT_CHUNK = 64   # ids per chunk of the draft's draws

# Philox purposes (counter word 3, bits 24..31)
P_DRAFT_CHUNK = 1
P_DRAFT_ELEM = 2
P_ACCEPT = 3
P_DECIDE_CHUNK = 4
P_DECIDE_ELEM = 5

STATIC, COMPACT, CAP_ACCEPT = 0, 1, 2
EARLY_STOP, GLOBAL_ARGMAX = 0, 1

_MASK32 = np.uint64(0xFFFFFFFF)


# ---------------------------------------------------------------------------
# Input conversion
# ---------------------------------------------------------------------------

def to_f64(x, dtype: str) -> np.ndarray:
    """bf16 bit patterns (uint16) or float32 -> float64 (exact)."""
    x = np.asarray(x)
    if dtype == "bf16":
        return (x.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


# ---------------------------------------------------------------------------
# Random numbers [PHILOX]
# ---------------------------------------------------------------------------

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds [PHILOX, Sec. 3: the Philox S-box and key schedule].

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
        (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))
    and the key is bumped by the Weyl constants (W0, W1) between rounds."""
    c = [np.asarray(x).astype(np.uint64) & _MASK32 for x in (c0, c1, c2, c3)]
    shape = np.broadcast(*c).shape
    c = [np.broadcast_to(x, shape).copy() for x in c]
    ka, kb = int(k0) & 0xFFFFFFFF, int(k1) & 0xFFFFFFFF
    for _ in range(10):
        p0 = c[0] * np.uint64(PHILOX_M0)
        p1 = c[2] * np.uint64(PHILOX_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ np.uint64(ka), lo1, hi0 ^ c[3] ^ np.uint64(kb), lo0]
        ka = (ka + PHILOX_W0) & 0xFFFFFFFF
        kb = (kb + PHILOX_W1) & 0xFFFFFFFF
    return [x.astype(np.uint32) for x in c]


def random_bits(seed: int, step: int, purpose: int, req: int, pos: int, idx) -> np.ndarray:
    """The 32-bit word drawn for (purpose, request, position, index) at (seed, step).

    Counter = (idx >> 2, req, step_lo32, purpose << 24 | pos << 16 | step_hi16), key = seed
    (lo, hi); the word is lane idx & 3 of the Philox output.  (The pages name no generator;
    the counter layout is this library's contract.)"""
    idx = np.asarray(idx, dtype=np.uint64)
    step = int(step)
    seed = int(seed)
    c3 = ((purpose & 0xFF) << 24) | ((pos & 0xFF) << 16) | ((step >> 32) & 0xFFFF)
    out = philox4x32_10(idx >> np.uint64(2), np.uint64(req & 0xFFFFFFFF),
                        np.uint64(step & 0xFFFFFFFF), np.uint64(c3),
                        seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    lane = (idx & np.uint64(3)).astype(np.int64)
    stacked = np.stack(out, axis=-1)
    return np.take_along_axis(stacked, lane[..., None], axis=-1)[..., 0]


def bits_to_uniform(bits) -> np.ndarray:
    """u = ((bits >> 9) + 1/2) * 2^-23, strictly inside (0, 1) and exact in fp32 and fp64."""
    b = np.asarray(bits, dtype=np.uint32)
    return ((b >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def uniform(seed, step, purpose, req, pos, idx) -> np.ndarray:
    return bits_to_uniform(random_bits(seed, step, purpose, req, pos, idx))


def gumbel(u) -> np.ndarray:
    """Standard Gumbel variate from a uniform: -ln(-ln u)."""
    return -np.log(-np.log(np.asarray(u, dtype=np.float64)))


# ---------------------------------------------------------------------------
# Samplers
# ---------------------------------------------------------------------------

def _top2_gap(keys: np.ndarray) -> float:
    k = keys[np.isfinite(keys)]
    if k.size < 2:
        return math.inf
    part = np.partition(k, -2)[-2:]
    return float(part[1] - part[0])


def _first_argmax(keys: np.ndarray) -> int:
    """Index of the largest key, the lowest index among equal maxima."""
    return int(np.argmax(keys))  # numpy returns the first occurrence


def logsumexp(x: np.ndarray) -> float:
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x)
    if not np.isfinite(m):
        return float(m)
    return float(m + np.log(np.sum(np.exp(x - m))))


def chunk_log_mass(logw: np.ndarray, chunk: int = CHUNK) -> np.ndarray:
    """L_c = log sum_{v in chunk c} exp(logw[v]) over consecutive chunks (-inf if empty)."""
    logw = np.asarray(logw, dtype=np.float64)
    n = logw.size
    nc = (n + chunk - 1) // chunk
    padded = np.full(nc * chunk, -np.inf)
    padded[:n] = logw
    blocks = padded.reshape(nc, chunk)
    with np.errstate(divide="ignore", invalid="ignore"):
        m = blocks.max(axis=1)
        safe_m = np.where(np.isfinite(m), m, 0.0)
        return np.where(np.isfinite(m), safe_m + np.log(np.exp(blocks - safe_m[:, None]).sum(axis=1)), -np.inf)


def two_level_gumbel(logw: np.ndarray, seed: int, step: int, req: int, pos: int,
                     purpose_chunk: int, purpose_elem: int, chunk: int = CHUNK):
    """Exact draw of v with probability proportional to exp(logw[v]).

    Level 1: the vocabulary is cut into consecutive chunks of `chunk` entries; chunk c gets
    the key L_c + G_c with L_c = log sum_{v in c} exp(logw[v]) and G_c a Gumbel variate
    (purpose_chunk, index c).  The largest key picks the chunk -- by the Gumbel-max property
    this chooses c with probability equal to its share of the total mass.
    Level 2: inside the chosen chunk, entry v gets logw[v] + G'_v (purpose_elem, index =
    offset of v in the chunk); the largest key is the draw.  Given the chunk, the entry is
    then drawn in proportion to exp(logw[v]), so the product is exact.

    Entries with logw = -inf never win.  Ties go to the lowest index at both levels.
    Returns (v, margin) where margin is the smaller of the two levels' top-two key gaps."""
    logw = np.asarray(logw, dtype=np.float64)
    n = logw.size
    L = chunk_log_mass(logw, chunk)
    nc = L.size
    Kc = L + gumbel(uniform(seed, step, purpose_chunk, req, pos, np.arange(nc)))
    if not np.any(np.isfinite(Kc)):
        raise ValueError("two_level_gumbel: no entry with positive weight")
    c = _first_argmax(Kc)
    lo, hi = c * chunk, min(n, (c + 1) * chunk)
    ke = logw[lo:hi] + gumbel(uniform(seed, step, purpose_elem, req, pos, np.arange(hi - lo)))
    j = _first_argmax(ke)
    return lo + j, min(_top2_gap(Kc), _top2_gap(ke))


def inverse_cdf(w: np.ndarray, u: float):
    """Inverse-CDF draw from non-negative weights w (not all zero) with one uniform u in (0, 1):
    with partial sums C_j = w_0 + ... + w_j and S = C_last, the first j with C_j > u S, so that
    j is drawn with probability w_j / S (zero weights are never drawn).  Returns (j, margin),
    margin = the distance of u S to the partial sums on either side of the decision, over S."""
    w = np.asarray(w, dtype=np.float64)
    C = np.cumsum(w)
    S = C[-1]
    t = u * S
    j = int(np.argmax(C > t))
    lo = C[j - 1] if j > 0 else 0.0
    return j, float(min(t - lo, C[j] - t) / S)


def two_level_cdf(logw: np.ndarray, seed: int, step: int, req: int, pos: int,
                  purpose_chunk: int, purpose_elem: int, chunk: int = DRAFT_CHUNK):
    """Exact draw of v with probability proportional to exp(logw[v]): a chunk by Gumbel-max over
    the chunks' log-masses, then an id inside the chunk by inverse CDF.

    Level 1 as in two_level_gumbel (chunk key L_c + G_c, purpose_chunk, index c).  Level 2: one
    uniform u (purpose_elem, index 0) and the chunk's weights w_i = exp(logw[v_i] - m), m the
    chunk's largest log-weight; the id is inverse_cdf(w, u).  Given the chunk, an id is drawn in
    proportion to exp(logw), so the product is exact.  Returns (v, margin), margin = the smaller
    of the level-1 top-two key gap and the level-2 distance to a partial-sum boundary."""
    logw = np.asarray(logw, dtype=np.float64)
    n = logw.size
    L = chunk_log_mass(logw, chunk)
    nc = L.size
    Kc = L + gumbel(uniform(seed, step, purpose_chunk, req, pos, np.arange(nc)))
    if not np.any(np.isfinite(Kc)):
        raise ValueError("two_level_cdf: no entry with positive weight")
    c = _first_argmax(Kc)
    lo, hi = c * chunk, min(n, (c + 1) * chunk)
    seg = logw[lo:hi]
    u = float(uniform(seed, step, purpose_elem, req, pos, np.array([0]))[0])
    j, m2 = inverse_cdf(np.exp(seg - np.max(seg)), u)
    return lo + j, min(_top2_gap(Kc), m2)


# ---------------------------------------------------------------------------
# S1 -- Markov-head block draft
# ---------------------------------------------------------------------------

def markov_logits(U_k: np.ndarray, W1: np.ndarray, W2t: np.ndarray, x_prev: np.ndarray) -> np.ndarray:
    """l_k = U_k + W1[x_{k-1}] . W2 for every request, [bs, V] in fp64.

    [SUMMARY, "Architecture (drafter)", Markov head]: the transition bias depends only on the
    previous token and factors through rank r as W1 (V x r, a lookup table) times W2 (r x V).
    W2 is stored transposed (W2t = W2^T, V x r)."""
    return U_k + W1[x_prev] @ W2t.T


def draft_block(U, W1, W2t, anchor, temperature: float, seed: int, step: int,
                dtype: str = "bf16", chunk: int = DRAFT_CHUNK, req_ids=None):
    """S1: draw x_1..x_gamma left to right from p_k(v) = softmax(U_k(v) + B_k(v)).

    [SUMMARY, "Architecture (drafter)"]: the parallel backbone yields U_1..U_gamma in one pass
    with the anchor as the first predicted position, and the sequential head samples from
    the causal per-position distributions left to right; per-token probabilities stay exact
    softmax values, which rejection sampling needs.
    Readings: x_0 = anchor feeds B_1; the sampling temperature divides the logits; at
    temperature 0 the draw is the argmax (lowest index on ties); the draw is two_level_cdf
    over chunks of DRAFT_CHUNK = 64 ids: a chunk by Gumbel-max over chunk masses, then an id by
    inverse CDF inside it (the law is exactly softmax for any chunk width).

    Returns tokens [bs, gamma] int32, logit_x [bs, gamma] (tempered logit of the drawn
    token; raw logit at temperature 0), lse [bs, gamma] (log-sum-exp of the tempered
    logits; 0 at temperature 0) and margin [bs, gamma] (decision margin).
    req_ids (optional) gives each row's request index in the random streams (default: row)."""
    U = to_f64(U, dtype)
    W1 = to_f64(W1, dtype)
    W2t = to_f64(W2t, dtype)
    bs, gamma, V = U.shape
    tokens = np.zeros((bs, gamma), dtype=np.int32)
    logit_x = np.zeros((bs, gamma))
    lse = np.zeros((bs, gamma))
    margin = np.zeros((bs, gamma))
    x_prev = np.asarray(anchor, dtype=np.int64).copy()
    for k in range(1, gamma + 1):
        ell = markov_logits(U[:, k - 1], W1, W2t, x_prev)
        for r in range(bs):
            rid = r if req_ids is None else int(req_ids[r])
            tokens[r, k - 1], logit_x[r, k - 1], lse[r, k - 1], margin[r, k - 1] = \
                _draw_position(ell[r], temperature, seed, step, rid, k, chunk)
        x_prev = tokens[:, k - 1].astype(np.int64)
    return tokens, logit_x, lse, margin


def _draw_position(ell_row, temperature: float, seed: int, step: int, rid: int, k: int, chunk: int):
    """The draw of one request at position k from its logits l_k (the draft's sampling rule):
    temperature 0 -> the argmax (lowest index); else two_level_cdf of l_k / temperature.
    Returns (token, logit_x, lse, margin) as draft_block reports them."""
    if temperature == 0.0:
        v = _first_argmax(ell_row)
        return v, ell_row[v], 0.0, _top2_gap(ell_row)
    t = ell_row / temperature
    v, mg = two_level_cdf(t, seed, step, rid, k, P_DRAFT_CHUNK, P_DRAFT_ELEM, chunk)
    return v, t[v], logsumexp(t), mg


# ---------------------------------------------------------------------------
# S1 with the RNN sequential head
# ---------------------------------------------------------------------------

def round_bf16(x) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even, returned in float64: with x = m 2^e and
    0.5 <= |m| < 1, keep 8 significant bits of m (bf16 has a 7-bit stored mantissa)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.round(m * 256.0) / 256.0, e)  # np.round: half to even


def rnn_state_step(e, s_prev, Wg, bg, dtype: str = "bf16"):
    """One update of the RNN head's gated recurrent state.

    [SUMMARY, "Architecture (drafter)", RNN head]: the head keeps a gated recurrent state s_k
    across the whole block, so position k sees the full prefix history.  The pages give no
    equations; reading (the plainest gated recurrence over the Markov head's inputs):
        g_k = sigmoid([e_k ; s_{k-1}] Wg + b_g)        (Wg: [2r, r], b_g: [r])
        s_k = g_k * s_{k-1} + (1 - g_k) * e_k           (s_0 = 0, e_k = W1[x_{k-1}])
    and the state is held in the head's parameter precision: rounded to bf16 after every
    update when the head is bf16 (the tensor cores read it as an operand).  A closed gate
    (g = 0) gives s_k = e_k, the Markov head; an open gate (g = 1) keeps s_k = 0.
    Inputs are float64 arrays ([n, r] e and s_prev); returns s_k [n, r]."""
    z = np.concatenate([e, s_prev], axis=1) @ Wg + bg[None, :]
    with np.errstate(over="ignore"):
        g = 1.0 / (1.0 + np.exp(-z))
    s = g * s_prev + (1.0 - g) * e
    return round_bf16(s) if dtype == "bf16" else s


def rnn_draft_block(U, W1, W2t, Wg, bg, anchor, temperature: float, seed: int, step: int,
                    dtype: str = "bf16", chunk: int = DRAFT_CHUNK, req_ids=None):
    """S1 with the RNN head: p_k(v) = softmax(U_k(v) + B_k(v)), B_k = s_k W2 with the gated
    recurrent state s_k of rnn_state_step (W2 = W2t^T, the Markov head's projection), drawn
    left to right with the draft's sampling rule and random streams (as draft_block).
    Wg, W1, W2t, U in `dtype`; bg float32 [r].  Returns tokens, logit_x, lse, margin (as
    draft_block) and states [bs, gamma, r] (float64 values of the bf16 / fp32 state s_k)."""
    U = to_f64(U, dtype)
    W1 = to_f64(W1, dtype)
    W2t = to_f64(W2t, dtype)
    Wg = to_f64(Wg, dtype)
    bg = np.asarray(bg, dtype=np.float64)
    bs, gamma, V = U.shape
    r = W1.shape[1]
    tokens = np.zeros((bs, gamma), dtype=np.int32)
    logit_x = np.zeros((bs, gamma))
    lse = np.zeros((bs, gamma))
    margin = np.zeros((bs, gamma))
    states = np.zeros((bs, gamma, r))
    s = np.zeros((bs, r))
    x_prev = np.asarray(anchor, dtype=np.int64).copy()
    for k in range(1, gamma + 1):
        s = rnn_state_step(W1[x_prev], s, Wg, bg, dtype)
        states[:, k - 1] = s
        ell = U[:, k - 1] + s @ W2t.T
        for r_ in range(bs):
            rid = r_ if req_ids is None else int(req_ids[r_])
            tokens[r_, k - 1], logit_x[r_, k - 1], lse[r_, k - 1], margin[r_, k - 1] = \
                _draw_position(ell[r_], temperature, seed, step, rid, k, chunk)
        x_prev = tokens[:, k - 1].astype(np.int64)
    return tokens, logit_x, lse, margin, states


# ---------------------------------------------------------------------------
# S2 -- confidence head, STS, prefix survival
# ---------------------------------------------------------------------------

def confidence(h, W1, anchor, tokens, w, b: float, sts_T, dtype: str = "bf16"):
    """S2: c_{r,k} = sigmoid(z_{r,k} / T_k), a_{r,j} = prod_{i<=j} c_{r,i}.

    [SUMMARY, "Verification scheduling", confidence head]: a linear projection of the
    concatenation [h_k ; W1[x_{k-1}]] followed by a sigmoid gives c_k, the probability that
    draft token k passes given that its prefix passed.
    [SUMMARY, same section, STS]: a per-position temperature calibrates the score; read as
    dividing the confidence logit by T_k (order preserving at each position).
    [SUMMARY, same section, scheduler]: prefix survival a_{r,j} is the running product of c.
    Readings: bias b = 0 unless given; x_0 = anchor; T_k indexed from k = 1.
    Returns conf [bs, gamma], surv [bs, gamma], z [bs, gamma] (all fp64)."""
    h = to_f64(h, dtype)
    W1 = to_f64(W1, dtype)
    w = np.asarray(w, dtype=np.float64)
    T = np.asarray(sts_T, dtype=np.float64)
    bs, gamma, d = h.shape
    x_prev = np.concatenate([np.asarray(anchor, dtype=np.int64)[:, None],
                             np.asarray(tokens, dtype=np.int64)[:, :gamma - 1]], axis=1)
    feats = np.concatenate([h, W1[x_prev]], axis=2)          # [bs, gamma, d + r]
    z = feats @ w + float(b)
    conf = 1.0 / (1.0 + np.exp(-z / T[None, :]))
    surv = np.cumprod(conf, axis=1)
    return conf, surv, z


# ---------------------------------------------------------------------------
# Cost table (host preparation)
# ---------------------------------------------------------------------------

def tier_of(M: int, tiers) -> Optional[int]:
    """Smallest captured total >= M ([VLLM, "CUDA Graph Padding"]: a 121-token batch runs
    the 128-token graph).  With no tiers every total is its own graph.  None if M exceeds
    the largest tier."""
    tiers = list(tiers)
    if not tiers:
        return M
    for t in tiers:
        if t >= M:
            return int(t)
    return None


def build_sps(T_raw, tiers) -> np.ndarray:
    """SPS table from a profiled step-time curve: sps[M] = 1 / T_mono(tier(M)).

    [VLLM, "Cost Modeling"]: the profiled curve is forced monotone increasing (running
    maximum here).  [VLLM, "CUDA Graph Padding"] and [SGLANG, "Ragged verify"]: the step
    runs the graph of the next captured tier, so the cost of M tokens is the cost of tier(M).
    Totals beyond the largest tier or the profiled range get sps = 0 (never admitted)."""
    T_raw = np.asarray(T_raw, dtype=np.float64)
    m_max = T_raw.size - 1
    T_mono = np.maximum.accumulate(T_raw)
    sps = np.zeros(m_max + 1)
    for M in range(m_max + 1):
        t = tier_of(M, tiers)
        if t is None or t > m_max:
            sps[M] = 0.0
        else:
            sps[M] = 1.0 / T_mono[t]
    return sps


# ---------------------------------------------------------------------------
# S3 -- hardware-aware global top-B prefix scheduler
# ---------------------------------------------------------------------------

FIX_SHIFT = 40


def schedule(surv_f32, sps, mode: int = EARLY_STOP):
    """S3: admit draft slots in descending survival, maximising Theta = tau * SPS(bs + K).

    [SUMMARY, "Verification scheduling", Hardware-Aware Prefix Scheduler (Algorithm 1)]:
    verify-length choice is a global throughput maximisation; because a_{r,j} does not grow
    with j the greedy admits slots globally in descending a_{r,j}, updates Theta in O(1) per
    admit from the table, and stops as soon as Theta drops.
    [VLLM, "DSpark confidence scheduling mechanism"]: expected tokens = one extra token per
    request plus the survival of the admitted slots; the admitted slots of a request form a
    contiguous prefix.
    [SUMMARY, "Infra"]: without the early stop, a global search over the table (GLOBAL_ARGMAX).

    Readings: keys are the fp32 survival values; ties go to the lower request, then the lower
    position.  Survival sums are exact fixed point, S_K = sum floor(a * 2^40), and
    tau(K) = bs + S_K * 2^-40 (exact in fp64); Theta(K) = tau(K) * sps[bs + K] with one
    rounding.  A slot is admitted only if Theta strictly increases (positive expected gain).
    K ranges over 0..min(bs*gamma, m_max - bs).

    Returns (window [bs] int32, K, Theta(K), Theta array over K)."""
    a = np.asarray(surv_f32, dtype=np.float32)
    bs, gamma = a.shape
    sps = np.asarray(sps, dtype=np.float64)
    m_max = sps.size - 1
    if m_max < bs:
        raise ValueError("sps table shorter than the batch")
    slots = [(float(a[r, j]), r, j) for r in range(bs) for j in range(gamma)]
    slots.sort(key=lambda s: (-s[0], s[1], s[2]))
    n = bs * gamma
    kmax = min(n, m_max - bs)
    theta = np.zeros(kmax + 1)
    S = 0
    for K in range(kmax + 1):
        if K > 0:
            S += int(math.floor(max(slots[K - 1][0], 0.0) * 2.0 ** FIX_SHIFT))
        tau = bs + math.ldexp(float(S), -FIX_SHIFT)
        theta[K] = tau * float(sps[bs + K])
    if mode == EARLY_STOP:
        K_star = kmax
        for K in range(kmax):
            if not theta[K + 1] > theta[K]:
                K_star = K
                break
    else:
        K_star = int(np.argmax(theta))  # first maximum
    window = np.zeros(bs, dtype=np.int32)
    for i in range(K_star):
        window[slots[i][1]] += 1
    return window, K_star, float(theta[K_star]), theta


# ---------------------------------------------------------------------------
# S3 under zero-overhead scheduling -- the budget is predicted two steps back
# ---------------------------------------------------------------------------

def zos_budget(surv_f32, sps) -> int:
    """The verify budget that step t's survival predicts for step t + 2.

    [SUMMARY, "Infra"], scheduler bullet: to run under CUDA graph replay and the
    zero-overhead (overlap) scheduler, the top-K truncation length of the current step is
    predicted from the confidence of two steps earlier; that stale information is a causal
    barrier, so the early-stop break is dropped and the search over the (sawtooth) SPS table
    is global.  [SGLANG, "ZOS"]: the confidence relay reads back two steps.
    Reading: the budget is K* of the global search (GLOBAL_ARGMAX) over that step's own
    survival, batch size and table, exactly as `schedule` computes it."""
    return int(schedule(surv_f32, sps, GLOBAL_ARGMAX)[1])


def zos_select(surv_f32, K: int) -> np.ndarray:
    """The K top-ranked slots of the current survival, as per-request window lengths.

    [SUMMARY, "Infra"]: the candidates of the current step are still ranked by the latest
    cumulative confidence.  Ranking as `schedule`: descending fp32 survival, ties to the lower
    request, then the lower position.  K is clamped to [0, bs * gamma]."""
    a = np.asarray(surv_f32, dtype=np.float32)
    bs, gamma = a.shape
    slots = sorted(((float(a[r, j]), r, j) for r in range(bs) for j in range(gamma)),
                   key=lambda s: (-s[0], s[1], s[2]))
    window = np.zeros(bs, dtype=np.int32)
    for i in range(max(0, min(int(K), bs * gamma))):
        window[slots[i][1]] += 1
    return window


def zos_step(surv_f32, sps, ring: list, step: int):
    """One step of the asynchronous scheduler with a two-slot budget ring.

    K_t = ring[t mod 2], the budget step t - 2 recorded; when no step recorded one (the first
    two steps; ring entries start at -1) it is the budget of the current survival itself.
    K_t is clamped to min(bs * gamma, m_max - bs) of the current batch, the windows are the
    K_t top-ranked current slots, and ring[t mod 2] then receives the budget the current
    survival predicts for step t + 2.  Returns (window, K_t); `ring` is updated in place."""
    a = np.asarray(surv_f32, dtype=np.float32)
    bs, gamma = a.shape
    m_max = np.asarray(sps).size - 1
    slot = step % 2
    K = ring[slot] if ring[slot] >= 0 else zos_budget(a, sps)
    K = min(K, bs * gamma, m_max - bs)
    window = zos_select(a, K)
    ring[slot] = zos_budget(a, sps)
    return window, K


# ---------------------------------------------------------------------------
# S4 -- ragged packing
# ---------------------------------------------------------------------------

def pack(window, anchor, tokens, tiers, cap: int, gamma: Optional[int] = None):
    """S4: pack the verify windows front to back into a cu_seqlens batch.

    [SGLANG, "Ragged verify under full CUDA graphs", Fig. 2]: the variable-length requests
    are packed into one compact buffer keyed by the total token count, rounded up to the
    nearest captured tier.  [VLLM, "Graph Capture"]: a request verifies 1..gamma+1 tokens.
    Request r contributes n_r = l_r + 1 query tokens [x_0, x_1..x_{l_r}].  window=None is the
    static layout (l_r = gamma).  Pad rows carry -1 in ids, req and pos.

    Returns (cu_seqlens [bs+1], ids, req, pos [cap] int32, padded_total)."""
    tokens = np.asarray(tokens, dtype=np.int32)
    bs = tokens.shape[0]
    g = tokens.shape[1] if gamma is None else gamma
    l = np.full(bs, g, dtype=np.int64) if window is None else np.asarray(window, dtype=np.int64)
    cu = np.zeros(bs + 1, dtype=np.int64)
    for r in range(bs):
        cu[r + 1] = cu[r] + l[r] + 1
    M = int(cu[bs])
    padded = tier_of(M, tiers)
    if padded is None:
        raise ValueError("packed total exceeds the largest tier")
    if padded > cap:
        raise ValueError("packed total exceeds the buffer capacity")
    ids = np.full(cap, -1, dtype=np.int32)
    req = np.full(cap, -1, dtype=np.int32)
    pos = np.full(cap, -1, dtype=np.int32)
    for r in range(bs):
        for j in range(int(l[r]) + 1):
            p = int(cu[r]) + j
            ids[p] = anchor[r] if j == 0 else tokens[r, j - 1]
            req[p] = r
            pos[p] = j
    return cu.astype(np.int32), ids, req, pos, padded


# ---------------------------------------------------------------------------
# S5 -- rejection-sampling verification
# ---------------------------------------------------------------------------

def verify(target_packed, cu_seqlens, window, mode: int, anchor, tokens, logit_x, lse,
           U, W1, W2t, temperature: float, seed: int, step: int, dtype: str = "bf16",
           chunk: int = CHUNK, req_ids=None, draft_logits=None, draft_states=None):
    """S5: accept the longest valid prefix of each request's window, then one more token.

    [SUMMARY, "Abstract" and "Architecture (drafter)"]: lossless speculative decoding accepts
    the longest prefix under rejection sampling with exact per-token probabilities: draft
    token x_k is accepted with probability min(1, p_t(x_k) / p_d(x_k)); on the first rejection
    a replacement is drawn from normalise(max(0, p_t - p_d)); if every tested token passes, a
    bonus token is drawn from the target distribution of the next position.
    [SGLANG, "Verify modes"]: static verifies the whole block; compact verifies only the
    scheduler's window; cap-accept verifies the whole block but commits only up to the
    window, committing exactly what compact commits while exposing the full-block ceiling.

    Readings: accept iff u < p_t/p_d (strict); the residual and bonus draws use the
    two-level Gumbel sampler (P_DECIDE_* streams at the position being drawn); if the
    residual has no mass the draw falls back to p_t; greedy (temperature 0) accepts iff
    x_k is the target argmax (lowest index) and the extra token is the target argmax.
    Draft probabilities come from logit_x - lse (the draft's outputs); the residual's draft
    distribution p_d is recomputed from U, W1, W2 at the rejected position, or, when the
    caller holds the draft's logits, taken from draft_logits [bs, gamma, V] (same dtype).
    With the RNN head the low-rank factor of position k is the state s_k, not W1[x_{k-1}]:
    draft_states [bs, gamma, r] (the states rnn_draft_block returns) then replaces the lookup.

    target_packed row cu[r] + k - 1 holds the target logits that score position k
    (k = 1..n_r).  Returns out_tokens [bs, gamma+1] (-1 padded), acc_len [bs],
    ceiling [bs] (tested-window accepted count; the full-block ceiling in cap-accept) and
    margin [bs] (smallest decision margin among the decisions that shaped the output).
    req_ids (optional) gives each row's request index in the random streams (default: row)."""
    tgt = to_f64(target_packed, dtype)
    if draft_logits is None:
        Uf = to_f64(U, dtype)
        W1f = to_f64(W1, dtype)
        W2f = to_f64(W2t, dtype)
    else:
        Df = to_f64(draft_logits, dtype)
    tokens = np.asarray(tokens, dtype=np.int64)
    bs, gamma = tokens.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.full((bs, gamma + 1), -1, dtype=np.int32)
    acc_len = np.zeros(bs, dtype=np.int32)
    ceiling = np.zeros(bs, dtype=np.int32)
    margin = np.full(bs, math.inf)
    for r in range(bs):
        rid = r if req_ids is None else int(req_ids[r])
        lr = int(window[r]) if window is not None else gamma
        L_test = lr if mode == COMPACT else gamma
        L_commit = gamma if mode == STATIC else lr
        n_r = int(cu[r + 1] - cu[r])
        if n_r != L_test + 1:
            raise ValueError(f"request {r}: packed rows {n_r} != tested window + 1 = {L_test + 1}")

        def trow(k):  # target logits scoring position k
            return tgt[cu[r] + k - 1]

        x = [int(anchor[r])] + [int(v) for v in tokens[r]]
        first_reject = None
        mg = math.inf
        for k in range(1, L_test + 1):
            if temperature == 0.0:
                row = trow(k)
                ok = (_first_argmax(row) == x[k])
                mg = min(mg, _top2_gap(row))
            else:
                t = trow(k) / temperature
                lp_t = t[x[k]] - logsumexp(t)
                lp_d = float(logit_x[r, k - 1]) - float(lse[r, k - 1])
                ratio = math.exp(lp_t - lp_d)
                u = float(uniform(seed, step, P_ACCEPT, rid, k, 0))
                ok = u < ratio
                mg = min(mg, abs(u - ratio))
            if not ok:
                first_reject = k
                break
        ceiling[r] = (first_reject - 1) if first_reject is not None else L_test
        if first_reject is not None and first_reject <= L_commit:
            k = first_reject
            acc = k - 1
            if temperature == 0.0:
                x_new = _first_argmax(trow(k))
            else:
                t = trow(k) / temperature
                p_t = np.exp(t - logsumexp(t))
                if draft_logits is None:
                    a_row = W1f[x[k - 1]] if draft_states is None else np.asarray(draft_states[r][k - 1], np.float64)
                    d = (Uf[r, k - 1] + a_row @ W2f.T) / temperature
                else:
                    d = Df[r, k - 1] / temperature
                p_d = np.exp(d - logsumexp(d))
                res = np.maximum(0.0, p_t - p_d)
                with np.errstate(divide="ignore"):
                    logw = np.log(res) if res.sum() > 0.0 else t
                x_new, m2 = two_level_gumbel(logw, seed, step, rid, k, P_DECIDE_CHUNK, P_DECIDE_ELEM, chunk)
                mg = min(mg, m2)
        else:
            acc = L_commit
            k = L_commit + 1
            if temperature == 0.0:
                row = trow(k)
                x_new = _first_argmax(row)
                mg = min(mg, _top2_gap(row))
            else:
                t = trow(k) / temperature
                x_new, m2 = two_level_gumbel(t, seed, step, rid, k, P_DECIDE_CHUNK, P_DECIDE_ELEM, chunk)
                mg = min(mg, m2)
        out[r, :acc] = x[1:acc + 1]
        out[r, acc] = x_new
        acc_len[r] = acc
        margin[r] = mg
    return out, acc_len, ceiling, margin


def step_tokens(acc_len) -> int:
    """Tokens committed by one step: accepted drafts plus the one extra token per request."""
    return int(np.sum(np.asarray(acc_len, dtype=np.int64) + 1))


# ---------------------------------------------------------------------------
# Observability and calibration
# ---------------------------------------------------------------------------

def ece_bin(conf_f32, n_bins: int) -> np.ndarray:
    """Equal-width bin of a score in [0, 1]: floor(a * M) in fp32 arithmetic (the decision
    both sides take in the same precision), the last bin closed at 1, negatives in bin 0."""
    a = np.asarray(conf_f32, dtype=np.float32)
    b = np.floor(a * np.float32(n_bins)).astype(np.int64)
    return np.clip(b, 0, n_bins - 1)


def ece(conf_f32, label, n_bins: int = 10):
    """Expected calibration error of scores against 0/1 outcomes.

    [SUMMARY, "Verification scheduling", STS] and [SGLANG, "Observability"] report ECE
    without defining it.  Reading: the textbook definition -- M equal-width bins over [0, 1];
    ECE = sum_b (n_b / N) |mean outcome_b - mean score_b| = sum_b |sum outcome_b - sum score_b| / N.
    Returns (ece, count[M], sum outcome[M], sum score[M]); ece = 0 when N = 0."""
    a = np.asarray(conf_f32, dtype=np.float32).ravel()
    y = np.asarray(label, dtype=np.int64).ravel()
    b = ece_bin(a, n_bins)
    cnt = np.zeros(n_bins, dtype=np.int64)
    lab = np.zeros(n_bins, dtype=np.int64)
    sc = np.zeros(n_bins, dtype=np.float64)
    for i in range(a.size):
        cnt[b[i]] += 1
        lab[b[i]] += y[i]
        sc[b[i]] += float(a[i])
    N = a.size
    e = float(np.sum(np.abs(lab - sc)) / N) if N else 0.0
    return e, cnt, lab, sc


def prefix_labels(window, acc_len, ceiling, gamma: int):
    """Realised outcome of each prefix survival a_{r,k}: did positions 1..k all pass?

    With a ceiling (the accepted length over the whole block: cap-accept, or static's own
    accepted length) the outcome is [ceiling >= k] at every k.  Without one (compact) it is
    known only where the run decided it ([SGLANG, "Observability"]: pruning hides the
    ceiling): [acc >= k] for k <= l_r, and 0 beyond l_r when the window was rejected inside;
    unknown beyond l_r when the whole window passed.
    Returns (label [bs, gamma] int64, known [bs, gamma] bool)."""
    acc = np.asarray(acc_len, dtype=np.int64)
    bs = acc.size
    k = np.arange(1, gamma + 1)[None, :]
    if ceiling is not None:
        c = np.asarray(ceiling, dtype=np.int64)[:, None]
        return (c >= k).astype(np.int64), np.ones((bs, gamma), dtype=bool)
    w = np.full(bs, gamma, dtype=np.int64) if window is None else np.asarray(window, dtype=np.int64)
    label = (acc[:, None] >= k).astype(np.int64)
    known = (k <= w[:, None]) | (acc[:, None] < w[:, None])
    return label, known


MAX_GAMMA = 16  # histogram length - 1 (the block-length limit of the library's interface)


def observe(surv_f32, window, acc_len, ceiling, n_bins: int = 10) -> dict:
    """One step's observability record ([SGLANG, "Observability"]; "Per-request
    differentiation under mixed traffic", Fig. 4):
      - window and accepted-length sums and histograms, and with a ceiling (cap-accept) the
        ceiling sum / histogram and the accepted sum over those requests (utilisation);
      - calibration: ECE bins of the prefix survival against the realised prefix outcome,
        over the (r, k) whose outcome is known, and the same per position k.
    window None means gamma (static)."""
    a = np.asarray(surv_f32, dtype=np.float32)
    bs, gamma = a.shape
    w = np.full(bs, gamma, dtype=np.int64) if window is None else np.asarray(window, dtype=np.int64)
    acc = np.asarray(acc_len, dtype=np.int64)
    H = MAX_GAMMA + 1
    st = {"steps": 1, "requests": bs, "sum_window": int(w.sum()), "sum_accepted": int(acc.sum()),
          "window_hist": np.bincount(w, minlength=H)[:H], "accepted_hist": np.bincount(acc, minlength=H)[:H],
          "ceiling_requests": 0, "sum_ceiling": 0, "sum_accepted_ceiling": 0,
          "ceiling_hist": np.zeros(H, dtype=np.int64)}
    if ceiling is not None:
        c = np.asarray(ceiling, dtype=np.int64)
        st.update(ceiling_requests=bs, sum_ceiling=int(c.sum()), sum_accepted_ceiling=int(acc.sum()),
                  ceiling_hist=np.bincount(c, minlength=H)[:H])
    label, known = prefix_labels(w, acc, ceiling, gamma)
    _, cnt, lab, sc = ece(a[known], label[known], n_bins)
    st.update(bin_count=cnt, bin_label=lab, bin_score=sc)
    st["pos_count"] = known.sum(axis=0).astype(np.int64)
    st["pos_label"] = (label * known).sum(axis=0).astype(np.int64)
    st["pos_score"] = np.array([float(np.sum(a[known[:, k], k].astype(np.float64))) for k in range(gamma)])
    return st


def obs_report(st: dict) -> dict:
    """Summary of accumulated observability records: mean window, mean accepted length, mean
    ceiling, utilisation = accepted / ceiling (ratio of sums over the requests that carry a
    ceiling; Fig. 4's "utilisation against the ceiling"), ECE of the survival, and per
    position the mean survival next to the realised pass rate."""
    n = max(st["requests"], 1)
    nc = st["ceiling_requests"]
    N = int(np.sum(st["bin_count"]))
    return {"mean_window": st["sum_window"] / n, "mean_accepted": st["sum_accepted"] / n,
            "mean_ceiling": st["sum_ceiling"] / nc if nc else float("nan"),
            "utilisation": st["sum_accepted_ceiling"] / st["sum_ceiling"] if st["sum_ceiling"] else float("nan"),
            "ece": float(np.sum(np.abs(st["bin_label"] - st["bin_score"])) / N) if N else 0.0,
            "pos_mean_survival": np.where(st["pos_count"] > 0, st["pos_score"] / np.maximum(st["pos_count"], 1), np.nan),
            "pos_pass_rate": np.where(st["pos_count"] > 0, st["pos_label"] / np.maximum(st["pos_count"], 1), np.nan)}


def sts_fit(z, ceiling, grid, n_bins: int = 10):
    """Sequential temperature scaling fit ([SUMMARY, "Verification scheduling", STS]): left to
    right over the positions, a one-dimensional grid search of T_k minimising the ECE of the
    cumulative survival prod_{i<=k} sigmoid(z_i / T_i) (earlier T fixed), against the prefix
    outcome [ceiling >= k]; dividing a logit by T > 0 keeps each position's order.
    Ties: the lowest grid index.  Returns (T [gamma], ece of the chosen T [gamma], ece of
    every grid value [gamma, n_grid])."""
    z = np.asarray(z, dtype=np.float64)
    N, gamma = z.shape
    grid = np.asarray(grid, dtype=np.float64)
    c = np.asarray(ceiling, dtype=np.int64)
    prev = np.ones(N)
    T = np.zeros(gamma)
    best = np.zeros(gamma)
    table = np.zeros((gamma, grid.size))
    for k in range(gamma):
        y = (c >= k + 1).astype(np.int64)
        for g in range(grid.size):
            a = prev / (1.0 + np.exp(-z[:, k] / grid[g]))
            table[k, g] = ece(a.astype(np.float32), y, n_bins)[0]
        g_star = int(np.argmin(table[k]))  # first minimum
        T[k] = grid[g_star]
        best[k] = table[k, g_star]
        prev = prev / (1.0 + np.exp(-z[:, k] / T[k]))
    return T, best, table
