// S1 with the RNN sequential head: the gated recurrent state of each request, one position at a
// time.
//
// DSpark technical summary, "Architecture (drafter)", RNN head: a gated recurrent state s_k is
// carried across the whole block, so position k's transition bias sees the full prefix.  The
// pages give no equations; this library takes the plainest gated recurrence over the Markov
// head's inputs (the oracle's reading, stated there):
//     e_k = W1[x_{k-1}]                      (x_0 = anchor)
//     g_k = sigmoid([e_k ; s_{k-1}] Wg + b_g)  Wg [2r, r], b_g [r]      (s_0 = 0)
//     s_k = g_k * s_{k-1} + (1 - g_k) * e_k   held in the head's precision (bf16: rounded to
//                                             nearest even after every update)
// and the bias B_k = s_k W2, so the vocabulary pass and the select take s_k where the Markov
// head takes W1[x_{k-1}].  The state update is a small GEMM [bs, 2r] x [2r, r] (33 MFLOP at
// bs = 256, r = 256) on the CUDA cores, fp32 accumulate in a fixed order.
#include "common.cuh"
#include "internal.h"

namespace dspark {

namespace {

constexpr int kRnnRows = 8;    // requests per block
constexpr int kRnnGates = 64;  // gates (state dimensions) per block

// Block (request group, gate group): 256 threads = 64 gates x 4 request pairs.  The block's
// [e ; s_{k-1}] rows sit in shared memory as fp32; Wg is read once per block, coalesced along
// the gate dimension.
template <typename T>
__global__ void __launch_bounds__(256) rnn_state_kernel(const T* __restrict__ W1, const T* __restrict__ Wg,
                                                        const float* __restrict__ bg,
                                                        const int32_t* __restrict__ anchor,
                                                        const int32_t* __restrict__ tokens, T* __restrict__ states,
                                                        int bs, int gamma, int V, int r, int k) {
  extern __shared__ float xs[];  // [kRnnRows][2r]
  const int rb = blockIdx.x * kRnnRows, tid = threadIdx.x;
  const int twor = 2 * r;
  for (int e = tid; e < kRnnRows * twor; e += 256) {
    const int rr = e / twor, j = e - rr * twor, row = rb + rr;
    float v = 0.f;
    if (row < bs) {
      if (j < r) {
        const int xp = clamp_token((k == 1) ? anchor[row] : tokens[size_t(row) * gamma + k - 2], V);
        v = ld_f32(W1, size_t(xp) * r + j);
      } else if (k > 1) {
        v = ld_f32(states, (size_t(row) * gamma + (k - 2)) * r + (j - r));
      }
    }
    xs[e] = v;
  }
  __syncthreads();
  const int gi = blockIdx.y * kRnnGates + (tid & (kRnnGates - 1));
  const int q = tid / kRnnGates;  // rows 2q, 2q + 1 of the block
  if (gi >= r) return;
  const float* x0 = xs + (2 * q) * twor;
  const float* x1 = x0 + twor;
  float a0 = bg[gi], a1 = a0;
  for (int j = 0; j < twor; ++j) {
    const float w = ld_f32(Wg, size_t(j) * r + gi);
    a0 = fmaf(x0[j], w, a0);
    a1 = fmaf(x1[j], w, a1);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = rb + 2 * q + h;
    if (row >= bs) break;
    const float* x = h ? x1 : x0;
    const float g = 1.f / (1.f + expf(-(h ? a1 : a0)));
    const float s = g * x[r + gi] + (1.f - g) * x[gi];
    T* dst = states + (size_t(row) * gamma + (k - 1)) * r + gi;
    if constexpr (sizeof(T) == 2) {
      *dst = __float2bfloat16_rn(s);
    } else {
      *dst = s;
    }
  }
}

}  // namespace

cudaError_t launch_rnn_state(int dtype, const void* W1, const void* Wg, const float* bg, const int32_t* anchor,
                             const int32_t* tokens, void* states, int bs, int gamma, int V, int r, int k,
                             cudaStream_t s) {
  const dim3 grid((bs + kRnnRows - 1) / kRnnRows, (r + kRnnGates - 1) / kRnnGates);
  const size_t smem = size_t(kRnnRows) * 2 * r * sizeof(float);  // <= 16 KB at r = 256
  if (dtype == DSPARK_F32)
    rnn_state_kernel<float><<<grid, 256, smem, s>>>(static_cast<const float*>(W1), static_cast<const float*>(Wg), bg,
                                                   anchor, tokens, static_cast<float*>(states), bs, gamma, V, r, k);
  else
    rnn_state_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(
        static_cast<const __nv_bfloat16*>(W1), static_cast<const __nv_bfloat16*>(Wg), bg, anchor, tokens,
        static_cast<__nv_bfloat16*>(states), bs, gamma, V, r, k);
  return cudaGetLastError();
}

}  // namespace dspark
