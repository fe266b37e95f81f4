// S1 draft statistics on the tensor cores: tcgen05.mma (bf16 in, fp32 accumulate in TMEM),
// operands staged by TMA, fused epilogue (+ U, temperature, per-chunk max / sum-exp or
// argmax).  No [bs, V] logit tensor ever reaches HBM.
//
// DSpark technical summary, "Architecture (drafter)": the Markov head's bias for position k
// is W1[x_{k-1}] W2 (rank r = 256), added to the backbone's base logits U_k over the full
// vocabulary.  Per position this is a GEMM [bs, r] x [r, V] whose output is consumed
// immediately by the sampler's chunk statistics.
//
// Work decomposition (one launch = one position k):
//   tile      = 128 requests (TMEM lanes) x 128 vocabulary ids (= one sampler chunk), K = r
//   CTA       = persistent; fixed 128-request M-tile, strided over vocabulary chunks;
//               the gathered A operand W1[x_{k-1}] (128 x r) stays resident in shared memory
//   warp 0    = TMA producer: U tile (3-D map over [bs, gamma, V], evict-first) and the W2t
//               tile in K-stages of 64 (evict-last: W2 is re-read by every position)
//   warp 1    = TMEM owner + single-thread tcgen05.mma issuer, commits to mbarriers
//   warps 2-5 = epilogue: tcgen05.ld of the 128 x 128 fp32 accumulator (one row per thread),
//               + U from the swizzled tile, chunk statistics to the workspace
//   2 TMEM accumulators (256 columns) and 2 U stages let MMA, loads and epilogue overlap.
// Every mbarrier wait is bounded (globaltimer deadline + shared abort flag); on give-up the
// kernel records DSPARK_ETIMEOUT, waits (bounded) for its own copies / MMAs in flight,
// frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 64;
constexpr int kBStages = 4;
constexpr int kUStages = 2;
constexpr int kAccBufs = 2;
constexpr int kThreads = 192;
constexpr uint32_t kAtomBytes = kBM * kBK * 2;   // 16 KB: 128 rows x 128 bytes
constexpr uint32_t kUHalf = kBM * 64 * 2;        // 16 KB: one 64-column box of U
constexpr uint32_t kTmemCols = kAccBufs * kBN;   // 256

struct Barriers {
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t u_full[kUStages], u_empty[kUStages];
  uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__host__ __device__ constexpr size_t smem_bytes(int r) {
  return 1024 /* alignment slack */ + size_t(r / kBK) * kAtomBytes + kBStages * kAtomBytes +
         kUStages * 2 * kUHalf + sizeof(Barriers);
}

__global__ void __launch_bounds__(kThreads, 1) draft_stats_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_u,
    const __nv_bfloat16* __restrict__ W1, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, int bs, int gamma, int V, int r, int k, float inv_tau,
    int greedy, float2* __restrict__ stats, int n_chunks, uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nk = r / kBK;
  uint8_t* sA = smem;                                   // nk atoms
  uint8_t* sB = sA + nk * kAtomBytes;                   // kBStages atoms
  uint8_t* sU = sB + kBStages * kAtomBytes;             // kUStages x 32 KB
  Barriers* bar = reinterpret_cast<Barriers*>(sU + kUStages * 2 * kUHalf);
  volatile int* abort_flag = &bar->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_mt = (bs + kBM - 1) / kBM;
  const int mt = blockIdx.x % n_mt;
  const int m0 = mt * kBM;
  const int cstride = gridDim.x / n_mt;
  const int c0 = blockIdx.x / n_mt;
  const int n_tiles = (c0 < n_chunks) ? (n_chunks - c0 + cstride - 1) / cstride : 0;

  if (tid == 0) {
    for (int s = 0; s < kBStages; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->b_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&bar->b_empty[s]), 1);
    }
    for (int s = 0; s < kUStages; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->u_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&bar->u_empty[s]), kBM);
    }
    for (int s = 0; s < kAccBufs; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->acc_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&bar->acc_empty[s]), kBM);
    }
    tc::mbar_init(tc::smem_u32(&bar->drain), 1);
    bar->abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w2);
    tc::prefetch_tensormap(&tmap_u);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&bar->tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  // A operand: rows m0..m0+127 of W1[x_{k-1}] in the 128-byte-swizzled K-major layout
  {
    const int cpr = r / 8;  // 16-byte chunks per row
    for (int idx = tid; idx < kBM * cpr; idx += kThreads) {
      const int row = idx / cpr, ch = idx % cpr;
      const int grow = m0 + row;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (grow < bs) {
        const int xp = clamp_token((k == 1) ? anchor[grow] : tokens[size_t(grow) * gamma + k - 2], V);
        v = *reinterpret_cast<const uint4*>(W1 + size_t(xp) * r + ch * 8);
      }
      const int kb = ch >> 3, j = ch & 7;
      *reinterpret_cast<uint4*>(sA + kb * kAtomBytes + row * 128 + ((j ^ (row & 7)) << 4)) = v;
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = bar->tmem_base;
  const uint64_t deadline = tc::globaltimer_ns() + timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last(), stream = tc::policy_evict_first();
      int bstage = 0, bph = 0, us = 0, uph = 0;
      int b_issued[kBStages], u_issued[kUStages];
      for (int s = 0; s < kBStages; ++s) b_issued[s] = -1;
      for (int s = 0; s < kUStages; ++s) u_issued[s] = -1;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int n0 = (c0 + t * cstride) * kBN;
        if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->u_empty[us]), uph ^ 1, deadline, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t ufull = tc::smem_u32(&bar->u_full[us]);
        tc::mbar_arrive_expect_tx(ufull, 2 * kUHalf);
        const uint32_t ud = tc::smem_u32(sU + us * 2 * kUHalf);
        tc::tma_load_3d(ud, &tmap_u, ufull, n0, k - 1, m0, stream);
        tc::tma_load_3d(ud + kUHalf, &tmap_u, ufull, n0 + 64, k - 1, m0, stream);
        u_issued[us] = uph;
        if (++us == kUStages) { us = 0; uph ^= 1; }
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->b_empty[bstage]), bph ^ 1, deadline, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bfull = tc::smem_u32(&bar->b_full[bstage]);
          tc::mbar_arrive_expect_tx(bfull, kAtomBytes);
          tc::tma_load_2d(tc::smem_u32(sB + bstage * kAtomBytes), &tmap_w2, bfull, kb * kBK, n0, keep);
          b_issued[bstage] = bph;
          if (++bstage == kBStages) { bstage = 0; bph ^= 1; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(status, DSPARK_ETIMEOUT);
        // wait (bounded) for every copy this thread put in flight before the CTA exits
        const uint64_t dl = tc::globaltimer_ns() + 200000000ull;
        const volatile int never = 0;
        for (int s = 0; s < kBStages; ++s)
          if (b_issued[s] >= 0) tc::mbar_wait_bounded(tc::smem_u32(&bar->b_full[s]), b_issued[s], dl, &never);
        for (int s = 0; s < kUStages; ++s)
          if (u_issued[s] >= 0) tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[s]), u_issued[s], dl, &never);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
      int bstage = 0, bph = 0, ab = 0, aph = 0;
      bool ok = true, issued = false;
      for (int t = 0; t < n_tiles && ok; ++t) {
        if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_empty[ab]), aph ^ 1, deadline, abort_flag)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + ab * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->b_full[bstage]), bph, deadline, abort_flag)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a_addr = tc::smem_u32(sA + kb * kAtomBytes);
          const uint32_t b_addr = tc::smem_u32(sB + bstage * kAtomBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc::mma_bf16(d, tc::sdesc_kmajor_sw128(a_addr + kk * 32), tc::sdesc_kmajor_sw128(b_addr + kk * 32),
                         idesc, (kb | kk) != 0);
          issued = true;
          tc::mma_commit(tc::smem_u32(&bar->b_empty[bstage]));
          if (++bstage == kBStages) { bstage = 0; bph ^= 1; }
        }
        if (!ok) break;
        tc::mma_commit(tc::smem_u32(&bar->acc_full[ab]));
        if (++ab == kAccBufs) { ab = 0; aph ^= 1; }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(status, DSPARK_ETIMEOUT);
        if (issued) {  // wait (bounded) for the MMAs already issued before TMEM is freed
          tc::mma_commit(tc::smem_u32(&bar->drain));
          const volatile int never = 0;
          tc::mbar_wait_bounded(tc::smem_u32(&bar->drain), 0, tc::globaltimer_ns() + 200000000ull, &never);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (128 threads)
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int m = wq * 32 + lane;     // tile row = TMEM lane
    const int grow = m0 + m;
    const float c2 = inv_tau * 1.4426950408889634f;
    int us = 0, uph = 0, ab = 0, aph = 0;
    for (int t = 0; t < n_tiles; ++t) {
      const int c = c0 + t * cstride;
      const int n0 = c * kBN;
      const int valid = min(kBN, V - n0);
      if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_full[ab]), aph, deadline, abort_flag) ||
          !tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[us]), uph, deadline, abort_flag)) {
        *abort_flag = 1;
        set_status(status, DSPARK_ETIMEOUT);
        break;
      }
      tc::tc_fence_after();
      float v[kBN];
      const uint32_t taddr = tmem_base + (uint32_t(wq * 32) << 16) + ab * kBN;
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) tc::tmem_ld32(taddr + q * 32, reinterpret_cast<uint32_t*>(v + q * 32));
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(tc::smem_u32(&bar->acc_empty[ab]));
      if (++ab == kAccBufs) { ab = 0; aph ^= 1; }

      const uint8_t* ub = sU + us * 2 * kUHalf + m * 128;
#pragma unroll
      for (int j16 = 0; j16 < kBN / 8; ++j16) {
        const int h = j16 >> 3, j = j16 & 7;
        const uint4 q = *reinterpret_cast<const uint4*>(ub + h * kUHalf + ((j ^ (m & 7)) << 4));
        v[8 * j16 + 0] += bf16lo(q.x);
        v[8 * j16 + 1] += bf16hi(q.x);
        v[8 * j16 + 2] += bf16lo(q.y);
        v[8 * j16 + 3] += bf16hi(q.y);
        v[8 * j16 + 4] += bf16lo(q.z);
        v[8 * j16 + 5] += bf16hi(q.z);
        v[8 * j16 + 6] += bf16lo(q.w);
        v[8 * j16 + 7] += bf16hi(q.w);
      }
      tc::mbar_arrive(tc::smem_u32(&bar->u_empty[us]));
      if (++us == kUStages) { us = 0; uph ^= 1; }

      float2 out;
      if (greedy) {
        float best = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i < valid && v[i] > best) { best = v[i]; bi = i; }
        out = make_float2(best, __int_as_float(bi == INT_MAX ? INT_MAX : n0 + bi));
      } else {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i < valid) mx = fmaxf(mx, v[i]);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i < valid) s += exp2f((v[i] - mx) * c2);
        out = make_float2(mx * inv_tau, s);
      }
      if (grow < bs) stats[size_t(grow) * n_chunks + c] = out;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

uint64_t g_wait_timeout_ns = 1000000000ull;  // 1 s; changed only through dspark_set_wait_timeout_ns

bool draft_tc_supported(int dtype, int bs, int V, int r) {
  return dtype == DSPARK_BF16 && bs >= 1 && bs <= 2 * kBM && r % kBK == 0 && r <= 256 && V % 8 == 0 &&
         encode_fn() != nullptr;
}

cudaError_t launch_draft_stats_tc(const void* U, const void* W1, const void* W2t,
                                  const int32_t* anchor, const int32_t* tokens, int bs, int gamma,
                                  int V, int r, int k, float inv_tau, int greedy, void* stats,
                                  int n_chunks, uint32_t* status, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map_w2, map_u;
  {
    const cuuint64_t dims[2] = {cuuint64_t(r), cuuint64_t(V)};
    const cuuint64_t strides[1] = {cuuint64_t(r) * 2};
    const cuuint32_t box[2] = {kBK, kBN};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&map_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2t), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {cuuint64_t(V), cuuint64_t(gamma), cuuint64_t(bs)};
    const cuuint64_t strides[2] = {cuuint64_t(V) * 2, cuuint64_t(gamma) * V * 2};
    const cuuint32_t box[3] = {64, 1, kBM};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&map_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const size_t smem = smem_bytes(r);
  const cudaError_t attr_err = cudaFuncSetAttribute(
      draft_stats_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_bytes(256)));
  if (attr_err != cudaSuccess) return attr_err;
  const int n_mt = (bs + kBM - 1) / kBM;
  int grid = (sm_count() / n_mt) * n_mt;
  grid = min(grid, n_mt * n_chunks);
  draft_stats_tc_kernel<<<grid, kThreads, smem, s>>>(map_w2, map_u, static_cast<const __nv_bfloat16*>(W1), anchor,
                                                     tokens, bs, gamma, V, r, k, inv_tau, greedy,
                                                     static_cast<float2*>(stats), n_chunks, status,
                                                     g_wait_timeout_ns);
  return cudaGetLastError();
}

}  // namespace dspark
