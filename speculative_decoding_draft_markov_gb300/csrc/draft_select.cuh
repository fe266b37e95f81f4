// The draft's select step for one request at one position: merge the request's partial draws
// (DraftEntry, one per slot) and draw x_k.  Shared by the CUDA-core path's select kernel and the
// tensor-core pass, which runs it inside its persistent kernel between positions.
//
// DSpark technical summary, "Architecture (drafter)": x_k ~ softmax((U_k + B_k) / T), drawn in
// two levels -- a 64-id draft chunk c* by Gumbel-max over the chunks' log-masses (the entries
// carry each slot's best key), then the id inside c* by inverse CDF.
//   temperature > 0: the chunk's 64 logits are recomputed (fixed-order fp32 dot products of the
//   factor row with W2t) and an inverse-CDF draw over them with the row's uniform (Philox
//   purpose 2, index 0) picks x_k.  logit_x = the tempered logit of x_k, lse = the row LSE of
//   the tempered logits from the entries' (max, sum-exp) pairs.
//   temperature = 0: the winner is x_k itself (lowest-index argmax), logit_x its raw logit.
#pragma once

#include <climits>

#include "common.cuh"

namespace dspark {

// Scratch the select needs in shared memory: the factor row (r <= 256 floats), the chunk's 64
// dot products, and the merged (lse, best key, winner).
struct SelectScratch {
  float a[256];
  float tv[kDraftIds];
  float lse, best;
  int win;
};

// Pull row x of the factor table W1 into L2: the next position gathers it as its A row.
template <typename T>
__device__ __forceinline__ void prefetch_row_l2(const T* W1, int x, int r, int V) {
  const char* row = reinterpret_cast<const char*>(W1 + size_t(clamp_token(x, V)) * r);
  for (int off = 0; off < r * int(sizeof(T)); off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
}

// One request b at position k by a group of NG warps (gt = the thread's index in the group,
// 0 .. 32 NG - 1); group_sync() synchronises exactly the group's threads.  prefetch_next: the
// Markov head's next position reads W1[x_k] right after this select -- pull it into L2.
// The entries are read with plain (coherent) loads: inside the persistent tensor-core kernel
// they were written by other CTAs of the same launch.
template <typename T, int NG, typename GroupSync>
__device__ __forceinline__ void select_row(int b, int gt, const float4* entries, int n_slots,
                                           const T* __restrict__ U, const T* __restrict__ W1,
                                           const T* __restrict__ W2t, const T* __restrict__ states,
                                           const int32_t* __restrict__ anchor, int32_t* tokens, float* logit_x,
                                           float* lse, int gamma, int V, int r, int k, float inv_tau, int greedy,
                                           uint64_t seed, uint64_t step, uint32_t* status, SelectScratch* sm,
                                           GroupSync group_sync, bool prefetch_next = false) {
  static_assert(NG >= 2 && kDraftIds % NG == 0, "a group of at least two warps splits a draft chunk");
  const float4* en = entries + size_t(b) * n_slots;
  const size_t out = size_t(b) * gamma + (k - 1);
  // the factor row (W1[x_{k-1}], or the RNN state s_k) does not depend on the draw: warps
  // 1 .. NG - 1 fetch it while warp 0 merges the entries, so that neither waits for the other
  if (!greedy && gt >= 32) {
    const T* arow = factor_row(W1, states, anchor, tokens, b, k, gamma, V, r);
    for (int i = gt - 32; i < r; i += 32 * (NG - 1)) sm->a[i] = ld_f32(arow, i);
  }
  if (gt < 32) {
    LsePair lp{-INFINITY, 0.f};
    ArgMax best{-INFINITY, INT_MAX};
    for (int i = gt; i < n_slots; i += 32) {
      const float4 e = en[i];
      lp = lse_merge(lp, LsePair{e.x, e.y});
      best = better(best, ArgMax{e.z, __float_as_int(e.w)});
    }
    lp = warp_lse(lp);
    best = warp_argmax(best);
    if (gt == 0) {
      sm->lse = lp.m + logf(lp.s);
      sm->best = best.v;
      sm->win = best.i;
    }
  }
  group_sync();
  if (greedy) {
    if (gt == 0) {
      const int x = (sm->win == INT_MAX) ? 0 : sm->win;
      tokens[out] = x;
      logit_x[out] = sm->best;
      lse[out] = 0.f;
      if (prefetch_next) prefetch_row_l2(W1, x, r, V);
    }
    return;
  }
  // only non-finite statistics leave the winner unset; a winner outside the vocabulary means the
  // entries were not written by this position's statistics pass (it gave up): report, use 0
  int cstar = (sm->win == INT_MAX) ? 0 : sm->win;
  if (cstar < 0 || cstar >= n_draft_chunks(V)) {
    if (gt == 0) set_status(status, DSPARK_EINVAL);
    cstar = 0;
  }
  // the U values of the chosen chunk (warp 0: offsets lane and lane + 32) load together with its
  // W2t rows
  const int v0 = cstar * kDraftIds + gt, v1 = v0 + 32;
  const size_t urow = (size_t(b) * gamma + (k - 1)) * V;
  float u0 = 0.f, u1 = 0.f;
  if (gt < 32) {
    if (v0 < V) u0 = ld_f32(U, urow + v0);
    if (v1 < V) u1 = ld_f32(U, urow + v1);
  }
  chunk_dots<T, kDraftIds / NG>(W2t, r, V, cstar * kDraftIds, sm->a, sm->tv, gt);
  group_sync();
  // the id inside the chunk by inverse CDF (warp 0, two offsets a lane: lane and lane + 32): the
  // first offset whose partial sum of exp(t - max) exceeds u times the total, u the row's
  // uniform of Philox purpose 2, index 0; should rounding leave every partial sum at or below
  // it, the last id with a finite logit
  if (gt < 32) {
    const float a0 = v0 < V ? (sm->tv[gt] + u0) * inv_tau : -INFINITY;
    const float a1 = v1 < V ? (sm->tv[gt + 32] + u1) * inv_tau : -INFINITY;
    const float mc = warp_max(fmaxf(a0, a1));
    const float w0 = a0 > -INFINITY ? expf(a0 - mc) : 0.f, w1 = a1 > -INFINITY ? expf(a1 - mc) : 0.f;
    float c0 = w0, c1 = w1;  // inclusive scans over offsets 0..31 and 32..63
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_up_sync(0xFFFFFFFFu, c0, o), y1 = __shfl_up_sync(0xFFFFFFFFu, c1, o);
      if (gt >= o) { c0 += y0; c1 += y1; }
    }
    c1 += __shfl_sync(0xFFFFFFFFu, c0, 31);
    const float total = __shfl_sync(0xFFFFFFFFu, c1, 31);
    const float u = bits_to_uniform(philox_group(seed, step, kDraftElem, b, k, 0).x);
    const float tgt = u * total;
    const unsigned hit0 = __ballot_sync(0xFFFFFFFFu, w0 > 0.f && c0 > tgt);
    const unsigned hit1 = __ballot_sync(0xFFFFFFFFu, w1 > 0.f && c1 > tgt);
    const unsigned pos0 = __ballot_sync(0xFFFFFFFFu, w0 > 0.f), pos1 = __ballot_sync(0xFFFFFFFFu, w1 > 0.f);
    int ei;
    if (hit0) ei = __ffs(hit0) - 1;
    else if (hit1) ei = 32 + __ffs(hit1) - 1;
    else if (pos1) ei = 32 + 31 - __clz(pos1);
    else ei = pos0 ? 31 - __clz(pos0) : 0;
    const float te = __shfl_sync(0xFFFFFFFFu, (ei & 32) ? a1 : a0, ei & 31);  // tempered logit of x_k
    if (gt == 0) {
      const int x = min(cstar * kDraftIds + ei, V - 1);
      tokens[out] = x;
      logit_x[out] = te;
      lse[out] = sm->lse;
      if (prefetch_next) prefetch_row_l2(W1, x, r, V);
    }
  }
}

}  // namespace dspark
