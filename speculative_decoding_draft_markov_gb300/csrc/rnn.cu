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
// Requires r in {32, 64, 128, 256} (the library's ranks).
#include "common.cuh"
#include "internal.h"

namespace dspark {

namespace {

constexpr int kRnnRows = 8;    // requests per block
constexpr int kRnnGates = 64;  // gates (state dimensions) per block

// Block (request group, gate group): 256 threads = 64 gates x 4 request pairs.  The block first
// stages its [e ; s_{k-1}] rows (fp32) and its 64-column slice of Wg ([2r, 64], the input dtype)
// in shared memory with every load independent, then each thread runs two dot products of
// length 2r out of shared memory (eight partial sums each, added in a fixed order).
template <typename T>
__global__ void __launch_bounds__(256) rnn_state_kernel(const T* __restrict__ W1, const T* __restrict__ Wg,
                                                        const float* __restrict__ bg,
                                                        const int32_t* __restrict__ anchor,
                                                        const int32_t* __restrict__ tokens, T* __restrict__ states,
                                                        int bs, int gamma, int V, int r, int k) {
  extern __shared__ __align__(16) float smem[];
  const int twor = 2 * r;
  float* xs = smem;                                             // [kRnnRows][2r]
  T* wsl = reinterpret_cast<T*>(smem + kRnnRows * twor);        // [2r][kRnnGates]
  const int rb = blockIdx.x * kRnnRows, g0 = blockIdx.y * kRnnGates, tid = threadIdx.x;
  // Wg slice: rows j of columns g0 .. g0 + ncols - 1 (ncols = 64, or r when r = 32), 16-byte
  // pieces (r is a multiple of 32 and g0 of 64, so the pieces are aligned and inside the row)
  constexpr int kPer = 16 / sizeof(T);                           // elements per piece
  const int pieces = min(kRnnGates, r - g0) / kPer;              // pieces per row
  for (int e = tid; e < twor * pieces; e += 256) {
    const int j = e / pieces, c = e - j * pieces;
    *reinterpret_cast<uint4*>(wsl + j * kRnnGates + c * kPer) =
        *reinterpret_cast<const uint4*>(Wg + size_t(j) * r + g0 + c * kPer);
  }
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
  const int gl = tid & (kRnnGates - 1), gi = g0 + gl;
  const int q = tid / kRnnGates;  // rows 2q, 2q + 1 of the block
  if (gi >= r) return;
  const float* x0 = xs + (2 * q) * twor;
  const float* x1 = x0 + twor;
  float p0[8], p1[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) p0[u] = p1[u] = 0.f;
  for (int j = 0; j < twor; j += 8) {  // 2r is a multiple of 64
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float w = ld_f32(wsl, size_t(j + u) * kRnnGates + gl);
      p0[u] = fmaf(x0[j + u], w, p0[u]);
      p1[u] = fmaf(x1[j + u], w, p1[u]);
    }
  }
  const float a0 = bg[gi] + (((p0[0] + p0[1]) + (p0[2] + p0[3])) + ((p0[4] + p0[5]) + (p0[6] + p0[7])));
  const float a1 = bg[gi] + (((p1[0] + p1[1]) + (p1[2] + p1[3])) + ((p1[4] + p1[5]) + (p1[6] + p1[7])));
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
  // [e ; s] rows (fp32) + the Wg slice: at r = 256, 16 KB + 64 KB (bf16) or 128 KB (fp32)
  const size_t es = dtype == DSPARK_F32 ? 4 : 2;
  const size_t smem = size_t(kRnnRows) * 2 * r * sizeof(float) + size_t(2 * r) * kRnnGates * es;
  if (smem > 48 * 1024) {
    const cudaError_t e = dtype == DSPARK_F32
        ? cudaFuncSetAttribute(rnn_state_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))
        : cudaFuncSetAttribute(rnn_state_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(smem));
    if (e != cudaSuccess) return e;
  }
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
