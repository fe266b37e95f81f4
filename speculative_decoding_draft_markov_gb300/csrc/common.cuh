// Shared device helpers of libdspark: status word, workspace layout, Philox4x32-10 uniforms,
// Gumbel keys, element loads and deterministic block reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

constexpr int kChunk = DSPARK_CHUNK;          // ids per chunk of verify's draws
constexpr int kDraftIds = DSPARK_DRAFT_CHUNK;  // ids per chunk of the draft's draws
static_assert(kChunk == 2 * kDraftIds, "a verify-width vocabulary tile holds two draft chunks");

// The draft's partial draw over a set of chunks ("slot") of one request, as a float4:
//   x, y : running (max t, sum exp(t - max)) of the tempered logits t = l / T over the slot's
//          chunks (-inf, 0 when empty; unused at temperature 0)
//   z    : best key -- temperature > 0: max over the slot's draft chunks (kDraftIds ids each)
//          of the chunk's log-mass plus its Gumbel (Philox purpose 1, index c); temperature 0:
//          the max logit
//   w    : int bits of the argmax of z -- the draft chunk index (T > 0) or the token id (T = 0);
//          INT_MAX when empty.  Ties go to the lowest index.
// The select merges a request's entries: LSE from (x, y), winner = argmax (z, lowest w).
// Slots never share a chunk, so the merged winner is the two-level draw's chunk.

// Philox purposes (counter word 3, bits 24..31).
enum Purpose : uint32_t {
  kDraftChunk = 1,
  kDraftElem = 2,
  kAccept = 3,
  kDecideChunk = 4,
  kDecideElem = 5,
};

// Decision kinds written by the verify decide pass.
enum DecisionKind : int { kDecNone = 0, kDecResidual = 1, kDecBonus = 2 };

// ----------------------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned)
//   status   : uint32 status word (first device-detected error wins)
//   stats    : 32 bytes per (row, chunk): the draft's entries (float4 [bs][n_slots]) or
//              verify's DecideEntry [bs][n_slots], n_slots <= n_chunks
//   rowstats : RowStat [bs * (gamma + 1)]  per packed target row
//   dec      : Decision [bs]               per-request verify decision
// ----------------------------------------------------------------------------------------
struct RowStat {
  float lse;     // log-sum-exp of the tempered target row (temperature > 0)
  float tx;      // tempered target logit of the tested draft token (or raw at T = 0)
  int argmax;    // lowest-index argmax of the row (temperature 0)
  int pad;
};

struct Decision {
  int kdec;      // position drawn by the decision (1 .. gamma + 1)
  int pdec;      // packed target row of that position
  int kind;      // DecisionKind
  int acc;       // accepted draft tokens
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Verify's partial draw of the deciding row over a set of chunks ("slot"), 32 bytes:
//   R, P   : sums over the slot's chunks of the residual mass max(0, p_t - p_d) and of p_t
//   kR, cR : best residual key log R_c + G_c (Philox purpose 4, index c) and its chunk
//   kP, cP : best target key log P_c + G_c and its chunk (the bonus draw, and the fallback of
//            a residual with no mass); -inf / INT_MAX when empty, ties to the lowest chunk
struct DecideEntry {
  float R, P, kR, kP;
  int cR, cP, pad0, pad1;
};

// The draft's scratch alone (16-byte entries, at most one per draft chunk).  The stats region
// of the workspace (32 bytes per verify chunk) holds it: n_draft_chunks <= 2 n_chunks.
__host__ __device__ inline int n_draft_chunks(int V) { return (V + kDraftIds - 1) / kDraftIds; }
__host__ __device__ inline size_t draft_stats_bytes(int bs, int n_slots) {
  return size_t(bs) * n_slots * sizeof(float4);
}
__host__ __device__ inline size_t stats_bytes(int bs, int n_chunks) {
  return size_t(bs) * n_chunks * sizeof(DecideEntry);
}

struct WsLayout {
  size_t status = 0, stats = 0, rowstats = 0, dec = 0, total = 0;
  int n_chunks = 0;
};

__host__ __device__ inline WsLayout ws_layout(int bs, int gamma, int V) {
  WsLayout L;
  L.n_chunks = (V + kChunk - 1) / kChunk;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.stats = off;
  off += align256(stats_bytes(bs, L.n_chunks));
  L.rowstats = off;
  off += align256(size_t(bs) * (gamma + 1) * sizeof(RowStat));
  L.dec = off;
  off += align256(size_t(bs) * sizeof(Decision));
  L.total = off;
  return L;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
  if (status) atomicCAS(status, 0u, code);
}

// A device-side wait that gave up: DSPARK_ETIMEOUT in the status word and, for the first one
// since the record was cleared, where (diag[0] = the wait's site code, diag[1] = the CTA,
// diag[2] = the site's progress counter: tile, position or barrier number).  diag may be null.
__device__ __forceinline__ void note_timeout(uint32_t* status, uint32_t* diag, uint32_t site, uint32_t info) {
  set_status(status, DSPARK_ETIMEOUT);
  if (diag && atomicCAS(diag, 0u, site) == 0u) {
    diag[1] = blockIdx.x;
    diag[2] = info;
  }
}

// Token ids read from device memory index weight rows: clamp into [0, V) so that bad data
// can never address outside W1 (the kernels that own a status word also report it).
__device__ __forceinline__ int clamp_token(int x, int V) { return x < 0 ? 0 : (x >= V ? V - 1 : x); }

// The row of the draft's low-rank factor that multiplies W2 at position k of request b: the
// Markov head's lookup W1[x_{k-1}] (x_0 = the anchor), or, with the RNN head, its recurrent
// state s_k, row (b, k - 1) of states [bs, gamma, r].
template <typename T>
__device__ __forceinline__ const T* factor_row(const T* W1, const T* states, const int32_t* anchor,
                                               const int32_t* tokens, int b, int k, int gamma, int V, int r) {
  if (states) return states + (size_t(b) * gamma + (k - 1)) * r;
  const int xp = clamp_token((k == 1) ? anchor[b] : tokens[size_t(b) * gamma + k - 2], V);
  return W1 + size_t(xp) * r;
}

// ----------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): per round
//   (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
// with the key advanced by the Weyl constants between rounds.
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// The four words of counter group `grp` (indices 4*grp .. 4*grp+3) of one stream.
__device__ __forceinline__ uint4 philox_group(uint64_t seed, uint64_t step, uint32_t purpose,
                                              uint32_t req, uint32_t pos, uint32_t grp) {
  const uint4 c = make_uint4(grp, req, uint32_t(step),
                             (purpose << 24) | ((pos & 0xFFu) << 16) | uint32_t((step >> 32) & 0xFFFFu));
  return philox10(c, uint32_t(seed), uint32_t(seed >> 32));
}

__device__ __forceinline__ uint32_t pick_word(uint4 w, int lane) {
  return lane == 0 ? w.x : lane == 1 ? w.y : lane == 2 ? w.z : w.w;
}

// u = ((bits >> 9) + 1/2) 2^-23, exactly: [1, 2) from the mantissa, minus (1 - 2^-24).
__device__ __forceinline__ float bits_to_uniform(uint32_t b) {
  return __uint_as_float(0x3F800000u | (b >> 9)) - __uint_as_float(0x3F7FFFFFu);
}

__device__ __forceinline__ float gumbel_from_bits(uint32_t b) {
  return -logf(-logf(bits_to_uniform(b)));
}

// ----------------------------------------------------------------------------------------
// Element loads
// ----------------------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float ld_f32(const T* p, size_t i);
template <> __device__ __forceinline__ float ld_f32<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ----------------------------------------------------------------------------------------
// Dot products W2t[v] . a for the NG NW ids v0 .. v0 + NG NW - 1 of one sampler chunk, by a
// group of NG warps (gt = the thread's index in the group): warp w takes ids v0 + NW w ..
// + NW - 1, lane l the K slice [8l, 8l + 8).  (8 warps x NW = 16: a verify chunk of 128 ids;
// 8 x 8 or 4 x 16: a draft chunk of 64.)  All NW rows' loads are issued before any arithmetic;
// fixed summation order.  out[i] (shared memory) receives the dot of id v0 + i, 0 for ids >= V.
// Requires r % 8 == 0 and r <= 256.
// ----------------------------------------------------------------------------------------
template <typename T, int NW = 16>
__device__ __forceinline__ void chunk_dots(const T* __restrict__ W2t, int r, int V, int v0,
                                           const float* __restrict__ a, float* out, int gt) {
  const int warp = gt >> 5, lane = gt & 31;
  const bool on = lane * 8 < r;
  float av[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) av[e] = on ? a[lane * 8 + e] : 0.f;
  float part[NW];
  if constexpr (sizeof(T) == 2) {
    uint4 q[NW];
#pragma unroll
    for (int j = 0; j < NW; ++j) {
      const int v = v0 + warp * NW + j;
      q[j] = (on && v < V) ? *reinterpret_cast<const uint4*>(W2t + size_t(v) * r + lane * 8)
                           : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < NW; ++j) {
      float acc = bf16lo(q[j].x) * av[0];
      acc = fmaf(bf16hi(q[j].x), av[1], acc);
      acc = fmaf(bf16lo(q[j].y), av[2], acc);
      acc = fmaf(bf16hi(q[j].y), av[3], acc);
      acc = fmaf(bf16lo(q[j].z), av[4], acc);
      acc = fmaf(bf16hi(q[j].z), av[5], acc);
      acc = fmaf(bf16lo(q[j].w), av[6], acc);
      acc = fmaf(bf16hi(q[j].w), av[7], acc);
      part[j] = acc;
    }
  } else {
#pragma unroll
    for (int j = 0; j < NW; ++j) {
      const int v = v0 + warp * NW + j;
      float acc = 0.f;
      if (on && v < V) {
        const float4 x0 = *reinterpret_cast<const float4*>(W2t + size_t(v) * r + lane * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(W2t + size_t(v) * r + lane * 8 + 4);
        acc = x0.x * av[0];
        acc = fmaf(x0.y, av[1], acc);
        acc = fmaf(x0.z, av[2], acc);
        acc = fmaf(x0.w, av[3], acc);
        acc = fmaf(x1.x, av[4], acc);
        acc = fmaf(x1.y, av[5], acc);
        acc = fmaf(x1.z, av[6], acc);
        acc = fmaf(x1.w, av[7], acc);
      }
      part[j] = acc;
    }
  }
#pragma unroll
  for (int j = 0; j < NW; ++j) {
    float t = part[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    if (lane == j) out[warp * NW + j] = t;
  }
}

// ----------------------------------------------------------------------------------------
// Deterministic reductions (fixed shuffle tree, fixed warp order)
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// (value, index) argmax; ties -> lower index.  Index INT_MAX marks "none".
struct ArgMax {
  float v;
  int i;
};
__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}
__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax b{__shfl_xor_sync(0xFFFFFFFFu, a.v, o), __shfl_xor_sync(0xFFFFFFFFu, a.i, o)};
    a = better(a, b);
  }
  return a;
}

// Online log-sum-exp pair: value = m + log(s).
struct LsePair {
  float m;
  float s;
};
__device__ __forceinline__ LsePair lse_merge(LsePair a, LsePair b) {
  if (b.s == 0.f) return a;
  if (a.s == 0.f) return b;
  const float m = fmaxf(a.m, b.m);
  return LsePair{m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}
__device__ __forceinline__ LsePair warp_lse(LsePair a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    LsePair b{__shfl_xor_sync(0xFFFFFFFFu, a.m, o), __shfl_xor_sync(0xFFFFFFFFu, a.s, o)};
    a = lse_merge(a, b);
  }
  return a;
}

// Block-wide reductions for blockDim.x = NT (multiple of 32).  `scratch` needs NT/32 slots.
// Every thread returns the result.  Order: warp tree, then warps 0..NT/32-1 in order.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t += scratch[i];
  return t;
}
template <int NT>
__device__ __forceinline__ float block_max(float v, float* scratch) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  float t = -INFINITY;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t = fmaxf(t, scratch[i]);
  return t;
}
template <int NT>
__device__ __forceinline__ ArgMax block_argmax(ArgMax a, float* sv, int* si) {
  a = warp_argmax(a);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) { sv[w] = a.v; si[w] = a.i; }
  __syncthreads();
  ArgMax t{sv[0], si[0]};
#pragma unroll
  for (int i = 1; i < NT / 32; ++i) t = better(t, ArgMax{sv[i], si[i]});
  return t;
}
template <int NT>
__device__ __forceinline__ LsePair block_lse(LsePair a, float* sm, float* ss) {
  a = warp_lse(a);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) { sm[w] = a.m; ss[w] = a.s; }
  __syncthreads();
  LsePair t{sm[0], ss[0]};
#pragma unroll
  for (int i = 1; i < NT / 32; ++i) t = lse_merge(t, LsePair{sm[i], ss[i]});
  return t;
}

}  // namespace dspark
