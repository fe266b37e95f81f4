// S1 -- Markov-head block draft: per-position chunk statistics (CUDA-core path) and the
// per-row merge + two-level draw (a chunk by Gumbel-max, the id inside it by inverse CDF).
//
// DSpark technical summary, "Architecture (drafter)": the sequential Markov head adds the
// rank-r bias W1[x_{k-1}] W2 to the backbone's base logits U_k and samples left to right.
// One position k is two launches: draft_stats (partial draws: per row, one DraftEntry per
// slot of chunks) and draft_select (one block per row: merge the entries, draw x_k).
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace dspark {

// ---------------------------------------------------------------------------------------
// CUDA-core statistics pass.  Block = 128 threads = one 128-id vocabulary tile = two draft
// chunks (threads 0..63 and 64..127), each its own slot; RB rows per block.  Serves fp32
// inputs (exact fp32 FMA) and small problems; bf16 at scale uses the tensor-core pass in
// draft_tc.cu.
// ---------------------------------------------------------------------------------------

// Reductions over each 64-thread half of a 128-thread block (warps 2q, 2q + 1); every thread
// of half q returns its half's result.  Fixed order: warp tree, then warp 2q before 2q + 1.
__device__ __forceinline__ float half_max(float v, float* scratch) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[w] = v;
  __syncthreads();
  return fmaxf(scratch[w & ~1], scratch[w | 1]);
}
__device__ __forceinline__ float half_sum(float v, float* scratch) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[w] = v;
  __syncthreads();
  return scratch[w & ~1] + scratch[w | 1];
}
__device__ __forceinline__ ArgMax half_argmax(ArgMax a, float* sv, int* si) {
  a = warp_argmax(a);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) { sv[w] = a.v; si[w] = a.i; }
  __syncthreads();
  return better(ArgMax{sv[w & ~1], si[w & ~1]}, ArgMax{sv[w | 1], si[w | 1]});
}

template <typename T, int RB>
__global__ void __launch_bounds__(128) draft_stats_simt_kernel(
    const T* __restrict__ U, const T* __restrict__ W1, const T* __restrict__ W2t, const T* __restrict__ states,
    const int32_t* __restrict__ anchor, const int32_t* __restrict__ tokens, int bs, int gamma,
    int V, int r, int k, float inv_tau, int greedy, uint64_t seed, uint64_t step,
    float4* __restrict__ entries, int n_slots) {
  __shared__ float sA[RB][64];
  __shared__ float sW[kChunk][65];
  __shared__ float red[4];
  __shared__ int redi[4];
  const int c = blockIdx.x, rb = blockIdx.y * RB, tid = threadIdx.x;
  const int v = c * kChunk + tid;
  const int cc = 2 * c + (tid >> 6);  // this thread's draft chunk
  float acc[RB];
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) acc[rr] = 0.f;

  for (int i0 = 0; i0 < r; i0 += 64) {
    const int sl = min(64, r - i0);
    for (int e = tid; e < RB * sl; e += kChunk) {
      const int rr = e / sl, ii = e % sl, row = rb + rr;
      float val = 0.f;
      if (row < bs) val = ld_f32(factor_row(W1, states, anchor, tokens, row, k, gamma, V, r), i0 + ii);
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
  const bool writer = (tid & 63) == 0 && cc < n_slots;
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    const int row = rb + rr;
    if (row >= bs) break;  // uniform over the block
    const float l = valid ? acc[rr] + ld_f32(U, (size_t(row) * gamma + (k - 1)) * V + v) : 0.f;
    float4* out = entries + size_t(row) * n_slots + cc;
    if (greedy) {
      const ArgMax am = half_argmax(ArgMax{valid ? l : -INFINITY, valid ? v : INT_MAX}, red, redi);
      if (writer) *out = make_float4(-INFINITY, 0.f, am.v, __int_as_float(am.i));
    } else {
      const float t = valid ? l * inv_tau : -INFINITY;
      const float m = half_max(t, red);
      const float s = half_sum(valid ? expf(t - m) : 0.f, red);
      if (writer) {
        float4 e = make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(INT_MAX));
        if (m > -INFINITY) {  // chunk key: log-mass + Gumbel (purpose 1, index cc)
          const uint4 w = philox_group(seed, step, kDraftChunk, uint32_t(row), k, uint32_t(cc) >> 2);
          e = make_float4(m, s, m + logf(s) + gumbel_from_bits(pick_word(w, cc & 3)), __int_as_float(cc));
        }
        *out = e;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Select pass: one 256-thread block per row.  Warp 0 merges the row's entries: the row LSE
// from the (max, sum-exp) pairs, and the winner = argmax of the keys (lowest index on ties).
//   temperature > 0: the winner is the draft chunk c* of the first Gumbel level; its 64 logits
//   are recomputed (fixed-order fp32 dot products) and an inverse-CDF draw over them with the
//   row's uniform (purpose 2, index 0) picks x_k.
//   temperature = 0: the winner is x_k itself (lowest-index argmax).
// ---------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256, 1) draft_select_kernel(
    const float4* __restrict__ entries, int n_slots, const T* __restrict__ U,
    const T* __restrict__ W1, const T* __restrict__ W2t, const T* __restrict__ states,
    const int32_t* __restrict__ anchor, int32_t* __restrict__ tokens, float* __restrict__ logit_x,
    float* __restrict__ lse, int bs,
    int gamma, int V, int r, int k, float inv_tau, int greedy, uint64_t seed, uint64_t step,
    uint32_t* status) {
  __shared__ float sA[256];
  __shared__ float tv[kDraftIds];
  __shared__ float s_lse, s_best;
  __shared__ int s_win;
  const int b = blockIdx.x, tid = threadIdx.x;
  const float4* en = entries + size_t(b) * n_slots;
  // launched as a programmatic dependent of the statistics pass: wait for it to complete, then
  // let the next position's statistics kernel start its set-up
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t out = size_t(b) * gamma + (k - 1);

  // the factor row (W1[x_{k-1}], or the RNN state s_k) does not depend on the draw: warps 1..7
  // fetch it while warp 0 merges the entries, so that neither waits for the other's loads
  if (!greedy && tid >= 32) {
    const T* arow = factor_row(W1, states, anchor, tokens, b, k, gamma, V, r);
    for (int i = tid - 32; i < r; i += 224) sA[i] = ld_f32(arow, i);
  }
  if (tid < 32) {
    LsePair lp{-INFINITY, 0.f};
    ArgMax best{-INFINITY, INT_MAX};
    for (int i = tid; i < n_slots; i += 32) {
      const float4 e = en[i];
      lp = lse_merge(lp, LsePair{e.x, e.y});
      best = better(best, ArgMax{e.z, __float_as_int(e.w)});
    }
    lp = warp_lse(lp);
    best = warp_argmax(best);
    if (tid == 0) {
      s_lse = lp.m + logf(lp.s);
      s_best = best.v;
      s_win = best.i;
    }
  }
  __syncthreads();
  if (greedy) {
    if (tid == 0) {
      tokens[out] = (s_win == INT_MAX) ? 0 : s_win;
      logit_x[out] = s_best;
      lse[out] = 0.f;
    }
    return;
  }
  // only non-finite statistics leave the winner unset; a winner outside the vocabulary means the
  // entries were not written by this position's statistics pass (it gave up): report, use 0
  int cstar = (s_win == INT_MAX) ? 0 : s_win;
  if (cstar < 0 || cstar >= n_draft_chunks(V)) {
    if (tid == 0) set_status(status, DSPARK_EINVAL);
    cstar = 0;
  }
  // the U values of the chosen chunk (warp 0: offsets lane and lane + 32) load together with its
  // W2t rows
  const int v0 = cstar * kDraftIds + tid, v1 = v0 + 32;
  const size_t urow = (size_t(b) * gamma + (k - 1)) * V;
  float u0 = 0.f, u1 = 0.f;
  if (tid < 32) {
    if (v0 < V) u0 = ld_f32(U, urow + v0);
    if (v1 < V) u1 = ld_f32(U, urow + v1);
  }
  chunk_dots<T, kDraftIds / 8>(W2t, r, V, cstar * kDraftIds, sA, tv);
  __syncthreads();
  // the id inside the chunk by inverse CDF (warp 0, two offsets a lane: lane and lane + 32): the
  // first offset whose partial sum of exp(t - max) exceeds u times the total, u the row's
  // uniform of Philox purpose 2, index 0; should rounding leave every partial sum at or below
  // it, the last id with a finite logit
  if (tid < 32) {
    const float a0 = v0 < V ? (tv[tid] + u0) * inv_tau : -INFINITY;
    const float a1 = v1 < V ? (tv[tid + 32] + u1) * inv_tau : -INFINITY;
    const float mc = warp_max(fmaxf(a0, a1));
    const float w0 = a0 > -INFINITY ? expf(a0 - mc) : 0.f, w1 = a1 > -INFINITY ? expf(a1 - mc) : 0.f;
    float c0 = w0, c1 = w1;  // inclusive scans over offsets 0..31 and 32..63
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_up_sync(0xFFFFFFFFu, c0, o), y1 = __shfl_up_sync(0xFFFFFFFFu, c1, o);
      if (tid >= o) { c0 += y0; c1 += y1; }
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
    if (tid == 0) {
      tokens[out] = min(cstar * kDraftIds + ei, V - 1);
      logit_x[out] = te;
      lse[out] = s_lse;
    }
  }
}

cudaError_t launch_draft_stats_simt(int dtype, const void* U, const void* W1, const void* W2t, const void* states,
                                    const int32_t* anchor, const int32_t* tokens, int bs, int gamma,
                                    int V, int r, int k, float inv_tau, int greedy, uint64_t seed,
                                    uint64_t step, void* entries, int n_slots, cudaStream_t s) {
  constexpr int RB = 32;
  dim3 grid((V + kChunk - 1) / kChunk, (bs + RB - 1) / RB);
  if (dtype == DSPARK_F32)
    draft_stats_simt_kernel<float, RB><<<grid, kChunk, 0, s>>>(
        (const float*)U, (const float*)W1, (const float*)W2t, (const float*)states, anchor, tokens, bs, gamma, V, r, k,
        inv_tau, greedy, seed, step, (float4*)entries, n_slots);
  else
    draft_stats_simt_kernel<__nv_bfloat16, RB><<<grid, kChunk, 0, s>>>(
        (const __nv_bfloat16*)U, (const __nv_bfloat16*)W1, (const __nv_bfloat16*)W2t, (const __nv_bfloat16*)states,
        anchor,
        tokens, bs, gamma, V, r, k, inv_tau, greedy, seed, step, (float4*)entries, n_slots);
  return cudaGetLastError();
}

cudaError_t launch_draft_select(int dtype, const void* entries, int n_slots, const void* U,
                                const void* W1, const void* W2t, const void* states, const int32_t* anchor,
                                int32_t* tokens, float* logit_x, float* lse, int bs, int gamma,
                                int V, int r, int k, float inv_tau, int greedy, uint64_t seed,
                                uint64_t step, uint32_t* status, cudaStream_t s) {
  if (dtype == DSPARK_F32)
    draft_select_kernel<float><<<bs, 256, 0, s>>>(
        (const float4*)entries, n_slots, (const float*)U, (const float*)W1, (const float*)W2t, (const float*)states,
        anchor, tokens, logit_x, lse, bs, gamma, V, r, k, inv_tau, greedy, seed, step, status);
  else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(bs);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, draft_select_kernel<__nv_bfloat16>, (const float4*)entries, n_slots,
                              (const __nv_bfloat16*)U, (const __nv_bfloat16*)W1, (const __nv_bfloat16*)W2t,
                              (const __nv_bfloat16*)states, anchor, tokens, logit_x, lse, bs, gamma, V, r, k, inv_tau, greedy, seed, step,
                              status);
  }
  return cudaGetLastError();
}

}  // namespace dspark
