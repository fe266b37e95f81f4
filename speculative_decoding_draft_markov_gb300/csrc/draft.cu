// S1 -- Markov-head block draft: per-position chunk statistics (CUDA-core path) and the
// per-row merge + two-level draw (a chunk by Gumbel-max, the id inside it by inverse CDF).
//
// DSpark technical summary, "Architecture (drafter)": the sequential Markov head adds the
// rank-r bias W1[x_{k-1}] W2 to the backbone's base logits U_k and samples left to right.
// One position k is two launches: draft_stats (partial draws: per row, one DraftEntry per
// slot of chunks) and draft_select (one block per row: merge the entries, draw x_k).
#include <climits>

#include "common.cuh"
#include "draft_select.cuh"
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
// Select pass: one 256-thread block per row runs select_row (draft_select.cuh): warp 0 merges
// the row's entries -- the row LSE from the (max, sum-exp) pairs, the winner = argmax of the
// keys (lowest index on ties) -- and, at temperature > 0, draws x_k inside the winning chunk.
// ---------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256, 1) draft_select_kernel(
    const float4* __restrict__ entries, int n_slots, const T* __restrict__ U,
    const T* __restrict__ W1, const T* __restrict__ W2t, const T* __restrict__ states,
    const int32_t* __restrict__ anchor, int32_t* __restrict__ tokens, float* __restrict__ logit_x,
    float* __restrict__ lse, int bs,
    int gamma, int V, int r, int k, float inv_tau, int greedy, uint64_t seed, uint64_t step,
    uint32_t* status) {
  __shared__ SelectScratch sm;
  // launched as a programmatic dependent of the statistics pass: wait for it to complete, then
  // let the next position's statistics kernel start its set-up
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  select_row<T, 8>(blockIdx.x, threadIdx.x, entries, n_slots, U, W1, W2t, states, anchor, tokens, logit_x, lse,
                   gamma, V, r, k, inv_tau, greedy, seed, step, status, &sm, [] { __syncthreads(); });
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
