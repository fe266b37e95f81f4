// S5 -- rejection-sampling verification of the packed windows.
//
// DSpark technical summary, "Abstract" and "Architecture (drafter)": a draft token is
// accepted with probability min(1, p_t / p_d) using exact per-token probabilities; the
// first rejected position is redrawn from normalise(max(0, p_t - p_d)); if every tested
// token passes, one bonus token comes from the target distribution of the next position.
// DSpark in SGLang, "Verify modes": static / compact / cap-accept.
//
// Launch sequence (one stream):
//   verify_rows     one block per packed row: row log-sum-exp (or argmax) and the tempered
//                   target logit of the draft token it tests -- the HBM stream over target
//   verify_decide   one thread per request: accept tests, first rejection, commit, ceiling
//   decision_stats  (temperature > 0) per (request, 128-id chunk): residual mass and target
//                   mass of the deciding row, p_d recomputed from U, W1, W2 (or read from the
//                   caller's draft logits)
//   decision_select (temperature > 0) one block per request: two-level Gumbel-max draw
#include <climits>

#include "common.cuh"
#include "f32x2.cuh"
#include "internal.h"
#include "pdl.h"

namespace dspark {

// ---------------------------------------------------------------------------------------
// Row statistics.  16-byte vector loads, per-thread online (max, sum-exp), fixed-order
// block merge.
// ---------------------------------------------------------------------------------------
constexpr int kRowThreads = 256;

// Hardware base-2 exponential (relative error near 2^-22; subnormal results flush to zero: the
// sum's leading term is 1).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One 16-byte group of a row as raw bits (loaded ahead of use) and its values.
template <typename T>
__device__ __forceinline__ void unpack_group(const uint4& q, float* x);
template <>
__device__ __forceinline__ void unpack_group<__nv_bfloat16>(const uint4& q, float* x) {
  x[0] = bf16lo(q.x); x[1] = bf16hi(q.x); x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
  x[4] = bf16lo(q.z); x[5] = bf16hi(q.z); x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
}
template <>
__device__ __forceinline__ void unpack_group<float>(const uint4& q, float* x) {
  x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y); x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
}

// One batch of the online row sum: groups cur[u] = row groups e0 + u 256 (kFull: all of them
// inside the row, so no per-group test).  The batch maximum is taken on the raw bf16 pairs
// (max.bf16x2: exact, a quarter of the instructions of unpacking first); then m2 and s2 are
// rescaled if it raised the maximum, and s2 gains sum 2^(x c2 - m2) in the fixed order
// (four partial sums by element index mod 4).
template <typename T, bool kFull, int kBatch>
__device__ __forceinline__ void lse_batch(const uint4 (&cur)[kBatch], int e0, int ng, float c2, float& m2,
                                          float& s2) {
  constexpr int G = sizeof(T) == 2 ? 8 : 4;
  float bm;
  if constexpr (sizeof(T) == 2) {
    __nv_bfloat162 mv = __float2bfloat162_rn(-INFINITY);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (kFull || e0 + u * kRowThreads < ng) {
        const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&cur[u]);
        mv = __hmax2(mv, __hmax2(__hmax2(v[0], v[1]), __hmax2(v[2], v[3])));
      }
    }
    bm = fmaxf(__low2float(mv), __high2float(mv));
  } else {
    bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (kFull || e0 + u * kRowThreads < ng) {
        float x[8];
        unpack_group<T>(cur[u], x);
#pragma unroll
        for (int q = 0; q < G; ++q) bm = fmaxf(bm, x[q]);
      }
    }
  }
  const float bm2 = bm * c2;
  if (bm2 > m2) {
    s2 = (s2 == 0.f) ? 0.f : s2 * ex2_approx(m2 - bm2);
    m2 = bm2;
  }
  // the four partial sums as two pairs (s4[0], s4[1]) and (s4[2], s4[3]): element q of a group
  // goes to s4[q & 3] as before, with the scale-and-shift and the adds done two lanes at a time
  // (fma.rn.f32x2 / add.rn.f32x2: each lane rounds exactly as fmaf / + do)
  unsigned long long s01 = pack_f32x2(0.f, 0.f), s23 = pack_f32x2(0.f, 0.f);
  const unsigned long long cc = pack_f32x2(c2, c2), mm = pack_f32x2(-m2, -m2);
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    if (kFull || e0 + u * kRowThreads < ng) {
      float x[8];
      unpack_group<T>(cur[u], x);
#pragma unroll
      for (int q = 0; q < G; q += 2) {
        float a0, a1;
        unpack_f32x2(fma_f32x2(pack_f32x2(x[q], x[q + 1]), cc, mm), a0, a1);
        const unsigned long long e = pack_f32x2(ex2_approx(a0), ex2_approx(a1));
        if ((q & 3) == 0) s01 = add_f32x2(s01, e);
        else s23 = add_f32x2(s23, e);
      }
    }
  }
  float s0, s1, s2p, s3;
  unpack_f32x2(s01, s0, s1);
  unpack_f32x2(s23, s2p, s3);
  s2 += (s0 + s1) + (s2p + s3);
}

// greedy (temperature 0: the row's argmax) is a template parameter, so that each variant's
// registers are allocated for its own loop
template <typename T, bool greedy>
__global__ void __launch_bounds__(kRowThreads, 3) verify_rows_kernel(
    const T* __restrict__ target, const int32_t* __restrict__ cu, const int32_t* __restrict__ tokens,
    int bs, int gamma, int V, float inv_tau, RowStat* __restrict__ rs, uint32_t* status) {
  __shared__ float sv[kRowThreads / 32], ss[kRowThreads / 32];
  __shared__ int si[kRowThreads / 32];
  __shared__ int s_cu[DSPARK_MAX_BS + 1];
  pdl_enter();
  const int p = blockIdx.x, tid = threadIdx.x;
  // cu_seqlens in one coalesced read, then the row's request by binary search in shared memory
  for (int i = tid; i <= bs; i += kRowThreads) s_cu[i] = cu[i];
  __syncthreads();
  const int M = s_cu[bs];
  if (p >= M) return;
  int lo = 0, hi = bs;  // cu[lo] <= p < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_cu[mid] <= p) lo = mid; else hi = mid;
  }
  const int r = lo, j = p - s_cu[r], n_r = s_cu[r + 1] - s_cu[r];
  const T* row = target + size_t(p) * V;
  constexpr int G = sizeof(T) == 2 ? 8 : 4;
  const int ng = V / G;
  // Each thread reads groups tid, tid + 256, ... in batches of kBatch; the next batch's loads
  // are issued before the current batch is reduced, so two batches (64 KB a block) are in
  // flight.  The arithmetic and its order do not depend on the prefetch.
  constexpr int kBatch = 8;
  constexpr int kStride = kBatch * kRowThreads;
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  uint4 cur[kBatch], nxt[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int e = tid + u * kRowThreads;
    if (e < ng) cur[u] = rv[e];
  }
  if constexpr (greedy) {
    ArgMax best{-INFINITY, INT_MAX};
    for (int e0 = tid; e0 < ng; e0 += kStride) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + kStride + u * kRowThreads;
        if (e < ng) nxt[u] = rv[e];
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kRowThreads;
        if (e >= ng) break;
        float x[8];
        unpack_group<T>(cur[u], x);
#pragma unroll
        for (int q = 0; q < G; ++q)
          if (x[q] > best.v) best = ArgMax{x[q], e * G + q};
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) cur[u] = nxt[u];
    }
    best = block_argmax<kRowThreads>(best, sv, si);
    if (tid == 0) {
      RowStat o{0.f, 0.f, best.i, 0};
      if (j < n_r - 1 && j < gamma) {
        const int xt = tokens[size_t(r) * gamma + j];
        if (xt < 0 || xt >= V) set_status(status, DSPARK_EINVAL);
        else o.tx = ld_f32(row, xt);
      }
      rs[p] = o;
    }
    return;
  }
  // online sum in base 2: m2 = running max of x c2 (c2 = log2(e) / T), s = sum of 2^(x c2 - m2),
  // rescaled only when a batch of kBatch * G values raises the max
  const float c2 = inv_tau * 1.4426950408889634f;
  float m2 = -INFINITY, s2 = 0.f;
  for (int e0 = tid; e0 < ng; e0 += kStride) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = e0 + kStride + u * kRowThreads;
      if (e < ng) nxt[u] = rv[e];
    }
    if (e0 + (kBatch - 1) * kRowThreads < ng) lse_batch<T, true>(cur, e0, ng, c2, m2, s2);
    else lse_batch<T, false>(cur, e0, ng, c2, m2, s2);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) cur[u] = nxt[u];
  }
  LsePair acc{m2 * 0.69314718055994531f, s2};  // natural units for the block merge
  acc = block_lse<kRowThreads>(acc, sv, ss);
  if (tid == 0) {
    RowStat o{acc.m + logf(acc.s), -INFINITY, -1, 0};
    if (j < n_r - 1 && j < gamma) {
      const int xt = tokens[size_t(r) * gamma + j];
      if (xt < 0 || xt >= V) set_status(status, DSPARK_EINVAL);
      else o.tx = ld_f32(row, xt) * inv_tau;
    }
    rs[p] = o;
  }
}

// ---------------------------------------------------------------------------------------
// Decide: accept tests in order, first rejection, committed prefix, ceiling.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) verify_decide_kernel(
    const int32_t* __restrict__ cu, const int32_t* __restrict__ window, int mode, int bs, int gamma,
    const int32_t* __restrict__ tokens, const float* __restrict__ logit_x,
    const float* __restrict__ lse, const RowStat* __restrict__ rs, int greedy, uint64_t seed,
    uint64_t step, int32_t* __restrict__ out_tokens, int32_t* __restrict__ acc_len,
    int32_t* __restrict__ ceiling, Decision* __restrict__ dec, uint32_t* status) {
  pdl_enter();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= bs) return;
  int32_t* out = out_tokens + size_t(r) * (gamma + 1);
  const int l = (mode == DSPARK_STATIC) ? gamma : window[r];
  const int n_r = cu[r + 1] - cu[r];
  const int L_test = (mode == DSPARK_COMPACT) ? l : gamma;
  const int L_commit = (mode == DSPARK_STATIC) ? gamma : l;
  if (l < 0 || l > gamma || n_r != L_test + 1) {
    set_status(status, DSPARK_EINVAL);
    for (int i = 0; i <= gamma; ++i) out[i] = -1;
    acc_len[r] = 0;
    if (ceiling) ceiling[r] = 0;
    dec[r] = Decision{0, 0, kDecNone, 0};
    return;
  }
  // every tested position's facts are read before the first test (one round trip, not one per
  // position), then the tests run in order up to the first rejection
  const int c0 = cu[r];
  RowStat st[DSPARK_MAX_GAMMA];
  int xk[DSPARK_MAX_GAMMA];
  float lpd[DSPARK_MAX_GAMMA];
#pragma unroll
  for (int k = 0; k < DSPARK_MAX_GAMMA; ++k) {
    if (k < L_test) {
      st[k] = rs[c0 + k];
      xk[k] = tokens[size_t(r) * gamma + k];
      lpd[k] = greedy ? 0.f : logit_x[size_t(r) * gamma + k] - lse[size_t(r) * gamma + k];
    }
  }
  int first = 0;
#pragma unroll
  for (int k = 1; k <= DSPARK_MAX_GAMMA; ++k) {
    if (k > L_test) break;
    bool ok;
    if (greedy) {
      ok = (st[k - 1].argmax == xk[k - 1]);
    } else {
      const float lp_t = st[k - 1].tx - st[k - 1].lse;
      const float ratio = expf(lp_t - lpd[k - 1]);
      const float u = bits_to_uniform(philox_group(seed, step, kAccept, r, k, 0).x);
      ok = u < ratio;
    }
    if (!ok) {
      first = k;
      break;
    }
  }
  const int ceil_r = first ? first - 1 : L_test;
  int acc, kdec, kind;
  if (first && first <= L_commit) {
    acc = first - 1;
    kdec = first;
    kind = kDecResidual;
  } else {
    acc = L_commit;
    kdec = L_commit + 1;
    kind = kDecBonus;
  }
  const int pdec = cu[r] + kdec - 1;
  for (int i = 0; i <= gamma; ++i) out[i] = (i < acc) ? tokens[size_t(r) * gamma + i] : -1;
  if (greedy) out[acc] = rs[pdec].argmax;
  acc_len[r] = acc;
  if (ceiling) ceiling[r] = ceil_r;
  dec[r] = Decision{kdec, pdec, greedy ? kDecNone : kind, acc};
}

// ---------------------------------------------------------------------------------------
// Decision chunk masses (temperature > 0).  Block = 128 ids of one chunk, RB requests.
// Residual rows: w = max(0, p_t - p_d) with p_d recomputed (fp32 FMA, fixed order);
// bonus rows: w = p_t.  Stores (sum w, sum p_t) per (request, chunk).
// ---------------------------------------------------------------------------------------
template <typename T, int RB>
__global__ void __launch_bounds__(128) decision_stats_simt_kernel(
    const T* __restrict__ target, const T* __restrict__ U, const T* __restrict__ W1,
    const T* __restrict__ W2t, const T* __restrict__ states, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const float* __restrict__ lse_d, const RowStat* __restrict__ rs,
    const Decision* __restrict__ dec, int bs, int gamma, int V, int r, float inv_tau, uint64_t seed, uint64_t step,
    DecideEntry* __restrict__ entries, int n_chunks) {
  __shared__ float sA[RB][64];
  __shared__ float sW[kChunk][65];
  __shared__ float red[4];
  const int c = blockIdx.x, rb = blockIdx.y * RB, tid = threadIdx.x;
  const int v = c * kChunk + tid;
  float acc[RB];
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) acc[rr] = 0.f;
  for (int i0 = 0; i0 < r; i0 += 64) {
    const int sl = min(64, r - i0);
    for (int e = tid; e < RB * sl; e += kChunk) {
      const int rr = e / sl, ii = e % sl, row = rb + rr;
      float val = 0.f;
      if (row < bs) {
        const Decision d = dec[row];
        if (d.kind == kDecResidual)
          val = ld_f32(factor_row(W1, states, anchor, tokens, row, d.kdec, gamma, V, r), i0 + ii);
      }
      sA[rr][ii] = val;
    }
    for (int e = tid; e < kChunk * sl; e += kChunk) {
      const int vv = e / sl, ii = e % sl, vg = c * kChunk + vv;
      sW[vv][ii] = (vg < V) ? ld_f32(W2t, size_t(vg) * r + i0 + ii) : 0.f;
    }
    __syncthreads();
    for (int ii = 0; ii < sl; ++ii) {
      const float w = sW[tid][ii];
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) acc[rr] = fmaf(sA[rr][ii], w, acc[rr]);
    }
    __syncthreads();
  }
  const bool valid = v < V;
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    const int row = rb + rr;
    if (row >= bs) break;
    const Decision d = dec[row];
    if (d.kind == kDecNone) continue;  // uniform over the block
    float pt = 0.f, w = 0.f;
    if (valid) {
      const float t = ld_f32(target, size_t(d.pdec) * V + v) * inv_tau;
      pt = expf(t - rs[d.pdec].lse);
      w = pt;
      if (d.kind == kDecResidual) {
        const float dl = (acc[rr] + ld_f32(U, (size_t(row) * gamma + d.kdec - 1) * V + v)) * inv_tau;
        const float pd = expf(dl - lse_d[size_t(row) * gamma + d.kdec - 1]);
        w = fmaxf(0.f, pt - pd);
      }
    }
    const float R = block_sum<kChunk>(w, red);
    const float P = block_sum<kChunk>(pt, red);
    if (tid == 0) {  // the chunk's entry: masses and keys log(mass) + G_c (purpose 4, index c)
      const uint4 gw = philox_group(seed, step, kDecideChunk, uint32_t(row), d.kdec, uint32_t(c) >> 2);
      const float g = gumbel_from_bits(pick_word(gw, c & 3));
      DecideEntry e{R, P, -INFINITY, -INFINITY, INT_MAX, INT_MAX, 0, 0};
      if (R > 0.f) { e.kR = logf(R) + g; e.cR = c; }
      if (P > 0.f) { e.kP = logf(P) + g; e.cP = c; }
      entries[size_t(row) * n_chunks + c] = e;
    }
  }
}

// ---------------------------------------------------------------------------------------
// Decision draw: one 256-thread block per request (temperature > 0).
// ---------------------------------------------------------------------------------------
// ---------------------------------------------------------------------------------------
// Decision masses from the caller's draft logits (no recompute): block = one 128-id chunk x RB
// rows; p_d = exp(logits / T - lse_d) of the row at the decision's position.  One DecideEntry
// per (request, chunk).
// ---------------------------------------------------------------------------------------
template <typename T, int RB>
__global__ void __launch_bounds__(128) decision_stats_logits_kernel(
    const T* __restrict__ target, const T* __restrict__ draft_logits, const float* __restrict__ lse_d,
    const RowStat* __restrict__ rs, const Decision* __restrict__ dec, int bs, int gamma, int V, float inv_tau,
    uint64_t seed, uint64_t step, DecideEntry* __restrict__ entries, int n_chunks) {
  __shared__ float red[4];
  const int c = blockIdx.x, rb = blockIdx.y * RB, tid = threadIdx.x;
  const int v = c * kChunk + tid;
  const bool valid = v < V;
  for (int rr = 0; rr < RB; ++rr) {
    const int row = rb + rr;
    if (row >= bs) break;
    const Decision d = dec[row];
    if (d.kind == kDecNone) continue;  // uniform over the block
    float pt = 0.f, w = 0.f;
    if (valid) {
      pt = expf(ld_f32(target, size_t(d.pdec) * V + v) * inv_tau - rs[d.pdec].lse);
      w = pt;
      if (d.kind == kDecResidual) {
        const size_t drow = size_t(row) * gamma + d.kdec - 1;
        const float pd = expf(ld_f32(draft_logits, drow * V + v) * inv_tau - lse_d[drow]);
        w = fmaxf(0.f, pt - pd);
      }
    }
    const float R = block_sum<kChunk>(w, red);
    const float P = block_sum<kChunk>(pt, red);
    if (tid == 0) {
      const uint4 gw = philox_group(seed, step, kDecideChunk, uint32_t(row), d.kdec, uint32_t(c) >> 2);
      const float g = gumbel_from_bits(pick_word(gw, c & 3));
      DecideEntry e{R, P, -INFINITY, -INFINITY, INT_MAX, INT_MAX, 0, 0};
      if (R > 0.f) { e.kR = logf(R) + g; e.cR = c; }
      if (P > 0.f) { e.kP = logf(P) + g; e.cP = c; }
      entries[size_t(row) * n_chunks + c] = e;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256, 1) decision_select_kernel(
    const T* __restrict__ target, const T* __restrict__ U, const T* __restrict__ W1,
    const T* __restrict__ W2t, const T* __restrict__ states, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const float* __restrict__ lse_d, const RowStat* __restrict__ rs,
    const Decision* __restrict__ dec, const T* __restrict__ draft_logits, const DecideEntry* __restrict__ entries,
    int n_slots, int bs, int gamma,
    int V, int r, float inv_tau, uint64_t seed, uint64_t step, int32_t* __restrict__ out_tokens,
    uint32_t* status) {
  __shared__ float sA[256];
  __shared__ float tw[kChunk], tp[kChunk];
  __shared__ float rv[8];
  __shared__ int ri[8];
  __shared__ int s_use_res, s_win;
  pdl_enter();
  const int b = blockIdx.x, tid = threadIdx.x;
  const Decision d = dec[b];
  if (d.kind == kDecNone) return;
  // a residual decision's factor row (needed unless the residual has no mass) does not depend on
  // the merge: warps 1.. fetch it while warp 0 merges
  const bool maybe_recompute = d.kind == kDecResidual && draft_logits == nullptr;
  if (maybe_recompute && tid >= 32) {
    const T* arow = factor_row(W1, states, anchor, tokens, b, d.kdec, gamma, V, r);
    for (int i = tid - 32; i < r; i += 256 - 32) sA[i] = ld_f32(arow, i);
  }
  // merge the request's partial draws: total residual mass (does the residual have mass?) and
  // the winning chunk of the residual or, without residual mass, of the target draw
  if (tid < 32) {
    const DecideEntry* en = entries + size_t(b) * n_slots;
    float R = 0.f;
    ArgMax bR{-INFINITY, INT_MAX}, bP{-INFINITY, INT_MAX};
    for (int i = tid; i < n_slots; i += 32) {
      const DecideEntry e = en[i];
      R += e.R;
      bR = better(bR, ArgMax{e.kR, e.cR});
      bP = better(bP, ArgMax{e.kP, e.cP});
    }
    R = warp_sum(R);
    bR = warp_argmax(bR);
    bP = warp_argmax(bP);
    if (tid == 0) {
      s_use_res = R > 0.f;
      s_win = (R > 0.f) ? bR.i : bP.i;
    }
  }
  __syncthreads();
  const bool use_res = s_use_res;
  // only non-finite statistics leave the winner unset; a winner outside the vocabulary means the
  // entries were not written by this call's statistics pass (it gave up): report, use 0
  int cstar = (s_win == INT_MAX) ? 0 : s_win;
  if (cstar < 0 || cstar >= (V + kChunk - 1) / kChunk) {
    if (tid == 0) set_status(status, DSPARK_EINVAL);
    cstar = 0;
  }
  const bool resid = (d.kind == kDecResidual) && use_res;
  const bool recompute = resid && draft_logits == nullptr;  // sA was filled before the merge
  const float lse_t = rs[d.pdec].lse;
  if (recompute) chunk_dots<T>(W2t, r, V, cstar * kChunk, sA, tw, threadIdx.x);
  __syncthreads();
  if (tid < kChunk) {
    const int v = cstar * kChunk + tid;
    float pt = 0.f, w = 0.f;
    if (v < V) {
      pt = expf(ld_f32(target, size_t(d.pdec) * V + v) * inv_tau - lse_t);
      w = pt;
      if (resid) {
        const size_t drow = size_t(b) * gamma + d.kdec - 1;
        const float dl = draft_logits ? ld_f32(draft_logits, drow * V + v) * inv_tau
                                      : (tw[tid] + ld_f32(U, drow * V + v)) * inv_tau;
        w = fmaxf(0.f, pt - expf(dl - lse_d[size_t(b) * gamma + d.kdec - 1]));
      }
    }
    tw[tid] = w;
    tp[tid] = pt;
  }
  __syncthreads();
  ArgMax ew{-INFINITY, INT_MAX}, ep{-INFINITY, INT_MAX};
  if (tid < kChunk) {
    const uint4 w = philox_group(seed, step, kDecideElem, b, d.kdec, tid >> 2);
    const float g = gumbel_from_bits(pick_word(w, tid & 3));
    if (tw[tid] > 0.f) ew = ArgMax{logf(tw[tid]) + g, tid};
    if (tp[tid] > 0.f) ep = ArgMax{logf(tp[tid]) + g, tid};
  }
  ew = block_argmax<256>(ew, rv, ri);
  ep = block_argmax<256>(ep, rv, ri);
  if (tid == 0) {
    // the recomputed chunk agrees with its mass except in degenerate rounding; fall back to p_t
    const int e = (ew.i != INT_MAX) ? ew.i : ep.i;
    out_tokens[size_t(b) * (gamma + 1) + d.acc] = (e != INT_MAX) ? cstar * kChunk + e : -1;
  }
}

template <typename T>
static cudaError_t verify_typed(const T* target, const int32_t* cu, const int32_t* window, int mode,
                               int bs, int gamma, int V, const int32_t* anchor,
                               const int32_t* tokens, const float* logit_x, const float* lse,
                               const T* draft_logits, const T* U, const T* W1, const T* W2t, const T* states,
                               int r,
                               float inv_tau, int greedy, uint64_t seed, uint64_t step,
                               int32_t* out_tokens, int32_t* acc_len, int32_t* ceiling, void* ws,
                               cudaStream_t s) {
  const WsLayout L = ws_layout(bs, gamma, V);
  char* w = static_cast<char*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(w + L.status);
  DecideEntry* entries = reinterpret_cast<DecideEntry*>(w + L.stats);
  RowStat* rs = reinterpret_cast<RowStat*>(w + L.rowstats);
  Decision* dec = reinterpret_cast<Decision*>(w + L.dec);
  cudaError_t le = greedy ? launch_pdl(verify_rows_kernel<T, true>, dim3(bs * (gamma + 1)), dim3(kRowThreads), 0, s,
                                       target, cu, tokens, bs, gamma, V, inv_tau, rs, status)
                          : launch_pdl(verify_rows_kernel<T, false>, dim3(bs * (gamma + 1)), dim3(kRowThreads), 0, s,
                                       target, cu, tokens, bs, gamma, V, inv_tau, rs, status);
  if (le != cudaSuccess) return le;
  le = launch_pdl(verify_decide_kernel, dim3((bs + 127) / 128), dim3(128), 0, s, cu, window, mode, bs, gamma, tokens,
                  logit_x, lse, static_cast<const RowStat*>(rs), greedy, seed, step, out_tokens, acc_len, ceiling, dec,
                  status);
  if (le != cudaSuccess) return le;
  if (!greedy) {
    constexpr int RB = 32;
    constexpr bool kBf16 = sizeof(T) == 2;
    int n_slots = L.n_chunks;
    if (draft_logits) {  // p_d from the caller's draft logits: a stream over two rows per request
      decision_stats_logits_kernel<T, RB><<<dim3(L.n_chunks, (bs + RB - 1) / RB), kChunk, 0, s>>>(
          target, draft_logits, lse, rs, dec, bs, gamma, V, inv_tau, seed, step, entries, L.n_chunks);
    } else if (kBf16 && draft_tc_supported(DSPARK_BF16, bs, V, r)) {
      const cudaError_t e = launch_decision_stats_tc(target, U, W1, W2t, states, anchor, tokens, lse, rs, dec, bs,
                                                     gamma, V,
                                                     r, inv_tau, seed, step, entries, L.n_chunks, &n_slots, status, s);
      if (e != cudaSuccess) return e;
    } else {
      decision_stats_simt_kernel<T, RB><<<dim3(L.n_chunks, (bs + RB - 1) / RB), kChunk, 0, s>>>(
          target, U, W1, W2t, states, anchor, tokens, lse, rs, dec, bs, gamma, V, r, inv_tau, seed, step, entries,
          L.n_chunks);
    }
    le = launch_pdl(decision_select_kernel<T>, dim3(bs), dim3(256), 0, s, target, U, W1, W2t, states, anchor, tokens,
                    lse,
                    static_cast<const RowStat*>(rs), static_cast<const Decision*>(dec), draft_logits,
                    static_cast<const DecideEntry*>(entries), n_slots, bs, gamma, V, r, inv_tau, seed, step,
                    out_tokens, status);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_verify(int dtype, const void* target, const int32_t* cu, const int32_t* window,
                          int mode, int bs, int gamma, int V, const int32_t* anchor,
                          const int32_t* tokens, const float* logit_x, const float* lse,
                          const void* draft_logits, const void* U, const void* W1, const void* W2t,
                          const void* states, int r, float inv_tau, int greedy, uint64_t seed, uint64_t step,
                          int32_t* out_tokens, int32_t* acc_len, int32_t* ceiling, void* ws,
                          cudaStream_t s) {
  if (dtype == DSPARK_F32)
    return verify_typed<float>((const float*)target, cu, window, mode, bs, gamma, V, anchor, tokens,
                               logit_x, lse, (const float*)draft_logits, (const float*)U, (const float*)W1,
                               (const float*)W2t, (const float*)states, r, inv_tau, greedy, seed, step, out_tokens, acc_len,
                               ceiling, ws, s);
  return verify_typed<__nv_bfloat16>((const __nv_bfloat16*)target, cu, window, mode, bs, gamma, V,
                                     anchor, tokens, logit_x, lse, (const __nv_bfloat16*)draft_logits,
                                     (const __nv_bfloat16*)U, (const __nv_bfloat16*)W1,
                                     (const __nv_bfloat16*)W2t, (const __nv_bfloat16*)states, r, inv_tau, greedy, seed, step, out_tokens,
                                     acc_len, ceiling, ws, s);
}

}  // namespace dspark
