// The confidence head's logit, shared by the confidence kernel (sched_pack.cu) and the
// persistent draft kernel (draft_tc.cu, which computes it while the draft runs), so that both
// produce the same bits.
//
// DSpark technical summary, "Verification scheduling (system side)": the confidence head is a
// linear projection of [h_k ; W1[x_{k-1}]] followed by a sigmoid; sequential temperature
// scaling divides the logit by T_k; prefix survival is the running product.
//
// Fixed order: z = ((H_0 + H_1 + ... + H_{parts-1}) + X) + b, where H_q is part q of the d-long
// h term (part q takes the 256-element groups q, q + parts, ...; lane l the 8 elements
// 8l .. 8l + 7 of each group, kConfLoads groups' loads in flight at once) and X the r-long
// W1[x_{k-1}] term (lane l: elements 8l .. 8l + 7), each reduced over its warp by the
// xor-shuffle tree.  The h terms do not depend on the drafted tokens, so the persistent draft
// kernel computes them ahead, while x_{k-1} is still being drawn.
#pragma once

#include "common.cuh"

namespace dspark {

constexpr int kConfLoads = 8;

// One 8-element group of a feature row: 16 bytes of bf16 (or two 16-byte halves of fp32).
template <typename T>
__device__ __forceinline__ void load_hgroup(const T* x, uint4* q) {
  if constexpr (sizeof(T) == 2) {
    q[0] = *reinterpret_cast<const uint4*>(x);
  } else {
    q[0] = *reinterpret_cast<const uint4*>(x);
    q[1] = *reinterpret_cast<const uint4*>(x + 4);
  }
}
// Its dot with w[0 .. 8), w read at the time of use.
template <typename T>
__device__ __forceinline__ float dot_hgroup(const uint4* q, const float* __restrict__ w) {
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(w));
  const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + 4));
  if constexpr (sizeof(T) == 2) {
    float a = bf16lo(q[0].x) * w0.x;
    a = fmaf(bf16hi(q[0].x), w0.y, a);
    a = fmaf(bf16lo(q[0].y), w0.z, a);
    a = fmaf(bf16hi(q[0].y), w0.w, a);
    a = fmaf(bf16lo(q[0].z), w1.x, a);
    a = fmaf(bf16hi(q[0].z), w1.y, a);
    a = fmaf(bf16lo(q[0].w), w1.z, a);
    a = fmaf(bf16hi(q[0].w), w1.w, a);
    return a;
  } else {
    float a = __uint_as_float(q[0].x) * w0.x;
    a = fmaf(__uint_as_float(q[0].y), w0.y, a);
    a = fmaf(__uint_as_float(q[0].z), w0.z, a);
    a = fmaf(__uint_as_float(q[0].w), w0.w, a);
    a = fmaf(__uint_as_float(q[1].x), w1.x, a);
    a = fmaf(__uint_as_float(q[1].y), w1.y, a);
    a = fmaf(__uint_as_float(q[1].z), w1.z, a);
    a = fmaf(__uint_as_float(q[1].w), w1.w, a);
    return a;
  }
}

// Warps per position of the confidence logit: at most 512 threads per block for gamma <= 8.
__host__ __device__ inline int conf_parts(int gamma) { return gamma <= 8 ? 2 : 1; }

// Lane `lane`'s share of part `part` of the h term of one (request, position): hr = the h row
// (d elements).  Not yet reduced over the warp.
template <typename T>
__device__ __forceinline__ float conf_hpart(const T* hr, const float* __restrict__ w, int d, int part, int parts,
                                            int lane) {
  const int stride = parts * 256;
  float acc = 0.f;
  for (int e0 = part * 256 + lane * 8; e0 < d; e0 += kConfLoads * stride) {
    uint4 q[kConfLoads][sizeof(T) == 4 ? 2 : 1];
#pragma unroll
    for (int u = 0; u < kConfLoads; ++u) {
      const int e = e0 + u * stride;
      if (e < d) load_hgroup<T>(hr + e, q[u]);
    }
#pragma unroll
    for (int u = 0; u < kConfLoads; ++u) {
      const int e = e0 + u * stride;
      if (e < d) acc += dot_hgroup<T>(q[u], w + e);
    }
  }
  return acc;
}

// Lane `lane`'s share of the W1[x_{k-1}] term from its 8-element group qa (loaded by the caller
// from w1row + 8 lane when 8 lane < r): the dot with w[d + 8 lane ..).  Not yet reduced.
template <typename T>
__device__ __forceinline__ float conf_xpart(const uint4* qa, const float* __restrict__ w, int d, int r, int lane) {
  return lane * 8 < r ? dot_hgroup<T>(qa, w + d + lane * 8) : 0.f;
}

}  // namespace dspark
