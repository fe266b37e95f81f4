// The draft's vocabulary pass on the tensor cores: tcgen05.mma (bf16 in, fp32 accumulate in
// TMEM), operands staged by TMA, fused epilogue.  No [bs, V] logit tensor ever reaches HBM.
//
// DSpark technical summary, "Architecture (drafter)": the Markov head's bias for position k
// is W1[x_{k-1}] W2 (rank r = 256), added to the backbone's base logits U_k over the full
// vocabulary.  Per position this is a GEMM [bs, r] x [r, V] consumed at once by a sampler:
// one launch per position k computes l = U_k + A_k W2 (A_k = W1[x_{k-1}], or the RNN head's
// state s_k) and reduces it to per-request partial draws (DraftEntry, common.cuh).
//
// What paces the pass on this part is the issue of tcgen05.mma instructions: measured, an
// issuing loop that also waits on its operand barriers sustains one MMA per ~180 SM cycles
// whatever N is, while an M = 128, N = 128, K = 16 MMA's arithmetic takes ~64.  So each
// instruction is made as wide as the tensor core allows, N = 256: a tile of 128 requests x
// 256 vocabulary ids is 16 MMAs (K = 256), half the instructions per logit of N = 128.
//
// Work decomposition:
//   tile      = 128 requests (TMEM lanes) x 256 vocabulary ids (= four 64-id draft chunks),
//               K = r; the accumulator is 256 TMEM columns, two of them (512 columns) let the
//               MMA of the next tile overlap the epilogue of this one
//   CTA       = persistent, one per SM; fixed 128-request M-tile, strided over vocabulary
//               tiles; the gathered A operand (W1[x_{k-1}], or s_k) stays in shared memory
//   warp 0    = TMA producer: W2t K-stages [256 ids x 64 K] (32 KB, a three-deep ring,
//               evict-last: every position re-reads W2t and it stays in L2), then the two
//               halves of the U_k tile (3-D map over [bs, gamma, V], evict-first)
//   warp 1    = TMEM owner + single-thread tcgen05.mma issuer, commits to mbarriers
//   warps 2-9 = epilogue, two warp sets of four (one warp per TMEM lane quarter, one request
//               row per thread).  Set h takes columns 128 h .. 128 h + 127 of every tile (the
//               tile's draft chunks 2h and 2h + 1) and U half h: it adds U_k to its 128
//               accumulator values (adding U_k on the tensor core through an identity operand
//               costs more tensor-pipe time than these adds cost issue slots), forms each
//               chunk's log-mass and Gumbel key and keeps, in registers, the row's running
//               (max, sum-exp) and best key.  The two sets merge through shared memory at the
//               end and write one entry per request, so the select merges one entry per CTA
//               column.
// Every mbarrier wait is bounded (SM cycle-counter deadline + shared abort flag); on give-up the
// kernel records DSPARK_ETIMEOUT, waits (bounded) for its own copies / MMAs in flight,
// frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;                          // ids per tile
constexpr int kHalfN = kBN / 2;                   // ids per epilogue set (two draft chunks)
static_assert(kHalfN == 2 * kDraftIds, "an epilogue set takes two draft chunks of a tile");
constexpr int kBK = 64;                           // K per stage: one 128-byte swizzle row
constexpr int kBStages = 3;                       // W2t ring of 32 KB stages
constexpr int kAccBufs = 2;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t kAAtom = kBM * kBK * 2;        // 16 KB: A rows [128 x 64 K]
constexpr uint32_t kBStage = kBN * kBK * 2;       // 32 KB: W2t rows [256 x 64 K]
constexpr uint32_t kUBox = kBM * 64 * 2;          // 16 KB: U [128 rows x 64 ids]
constexpr uint32_t kUHalfTile = 2 * kUBox;        // 32 KB: one epilogue set's 128 ids
constexpr uint32_t kTmemCols = kAccBufs * kBN;    // 512
constexpr float kLog2e = 1.4426950408889634f;

struct Barriers {
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t u_full[2], u_empty[2];  // U half h (one per epilogue set)
  uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  uint64_t drain;
  uint64_t a_ready;  // the A operand is in shared memory (one arrival per epilogue warp)
  uint32_t tmem_base;
  int abort;
  int mma_pending;   // the issuer's MMAs that nobody has waited for (set by the issuing thread)
  int xrow[kBM];     // row of the factor table for each A row (-1: zero row)
  float4 xch[kBM];   // warp set 1's entry of each row, merged by set 0 at the end
};

struct Params {
  const __nv_bfloat16* W1;
  const __nv_bfloat16* states;  // RNN head: the states s_k [bs, gamma, r] (A rows); else null
  const int32_t* anchor;
  const int32_t* tokens;
  int bs, gamma, V, r, k;
  float inv_tau;
  int greedy;
  int n_tiles;      // 256-id vocabulary tiles
  uint32_t* status;
  uint64_t timeout_ns;
  float4* entries;  // per (request, slot): DraftEntry
  int n_slots;
  uint64_t seed, step;
};

// Dynamic shared memory: A atoms | W2t ring | U halves | barriers.  The buffer is declared
// 1024-byte aligned (128-byte swizzle atoms).
constexpr size_t smem_bytes(int r) {
  return size_t(r / kBK) * kAAtom + kBStages * size_t(kBStage) + 2 * size_t(kUHalfTile) + sizeof(Barriers);
}
static_assert(smem_bytes(256) <= 232448, "dynamic shared memory beyond the 227 KB per-block limit");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The Gumbels of set h's two draft chunks 4c + 2h, 4c + 2h + 1 of vocabulary tile c, request
// `req`, position k (Philox purpose 1, indices = chunk ids): counter group c, words 2h, 2h + 1.
__device__ __forceinline__ float2 tile_gumbels(uint64_t seed, uint64_t step, int req, int k, int c, int h) {
  const uint4 w = philox_group(seed, step, kDraftChunk, uint32_t(req), k, uint32_t(c));
  return h ? make_float2(gumbel_from_bits(w.z), gumbel_from_bits(w.w))
           : make_float2(gumbel_from_bits(w.x), gumbel_from_bits(w.y));
}
// Kept out of line for the tile loop: inlined there its Philox rounds raise register pressure
// enough to spill, although the loop only calls it for tiles past the ones drawn up front.
__device__ __noinline__ float2 tile_gumbels_call(uint64_t seed, uint64_t step, int req, int k, int c, int h) {
  return tile_gumbels(seed, step, req, k, c, h);
}

// Max of the first `valid` of kDraftIds values (all of them when !kRagged), four chains.
template <bool kRagged>
__device__ __forceinline__ float row_max(const float* v, int valid) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < kDraftIds; ++i)
    if (!kRagged || i < valid) m4[i & 3] = fmaxf(m4[i & 3], v[i]);
  return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}
// sum over the first `valid` of kDraftIds values of 2^(v c2 - mc2), mc2 = max * c2 (each term
// <= 1), with the hardware base-2 exponential (relative error near 2^-22), eight chains.
template <bool kRagged>
__device__ __forceinline__ float row_sum_exp2(const float* v, int valid, float mc2, float c2) {
  float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kDraftIds; ++i) {
    const float e = tc::ex2_approx(fmaf(v[i], c2, -mc2));
    if (!kRagged || i < valid) s8[i & 7] += e;
  }
  return ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
}

// Warp 1 at the end of the kernel: free the tensor memory.  An epilogue that gave up has not
// waited for every accumulator, so then the MMAs still in flight are waited for (bounded) first.
// Out of line: it takes no registers from the kernel's loops.
__device__ __noinline__ void free_tmem(Barriers* bar, uint32_t tmem_base, int lane) {
  if (lane == 0 && bar->mma_pending && bar->abort) {
    tc::mma_commit(tc::smem_u32(&bar->drain));
    const volatile int never = 0;
    tc::mbar_wait_bounded(tc::smem_u32(&bar->drain), 0, tc::deadline_after_ns(200000000ull), &never);
  }
  __syncwarp();
  tc::tc_fence_after();
  tc::tmem_dealloc(tmem_base, kTmemCols);
}

__global__ void __launch_bounds__(kThreads, 1) draft_tc_kernel(const __grid_constant__ CUtensorMap tmap_w2,
                                                                const __grid_constant__ CUtensorMap tmap_u,
                                                                const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (tc::smem_u32(smem_raw) & 1023u) {  // the swizzled layouts need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, DSPARK_EUNSUPPORTED);
    return;
  }
  const int nk = p.r / kBK;
  uint8_t* sA = smem_raw;                    // nk atoms
  uint8_t* sB = sA + nk * kAAtom;            // kBStages x 32 KB
  uint8_t* sU = sB + kBStages * kBStage;     // 2 x 32 KB (U half of each epilogue set)
  Barriers* bar = reinterpret_cast<Barriers*>(sU + 2 * kUHalfTile);
  volatile int* abort_flag = &bar->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bs = p.bs, V = p.V, r = p.r;
  const int n_mt = (bs + kBM - 1) / kBM;
  const int m0 = (blockIdx.x % n_mt) * kBM;
  const int cstride = gridDim.x / n_mt;
  const int c0 = blockIdx.x / n_mt;
  const int n_tiles = (c0 < p.n_tiles) ? (p.n_tiles - c0 + cstride - 1) / cstride : 0;

  if (tid == 0) {
    for (int s = 0; s < kBStages; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->b_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&bar->b_empty[s]), 1);
    }
    for (int h = 0; h < 2; ++h) {
      tc::mbar_init(tc::smem_u32(&bar->u_full[h]), 1);
      tc::mbar_init(tc::smem_u32(&bar->u_empty[h]), kEpiWarps / 2);  // the warp set of the half
    }
    for (int s = 0; s < kAccBufs; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->acc_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&bar->acc_empty[s]), kEpiWarps);  // both sets read every tile
    }
    tc::mbar_init(tc::smem_u32(&bar->drain), 1);
    tc::mbar_init(tc::smem_u32(&bar->a_ready), kEpiWarps);
    bar->abort = 0;
    bar->mma_pending = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w2);
    tc::prefetch_tensormap(&tmap_u);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&bar->tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = bar->tmem_base;
  const long long deadline = tc::deadline_after_ns(p.timeout_ns);
  tc::grid_launch_dependents();  // the next kernel may start its own set-up now
  float4 xmine = make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(INT_MAX));  // epilogue entry

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // U_k and W2t do not depend on the previous kernel: the rings fill while it finishes.
    // Per tile: its W2t K-stages first (paced by the MMA), then the two U halves (paced by the
    // epilogue sets, one tile deep).
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last(), stream = tc::policy_evict_first();
      int bstage = 0, bph = 0;
      int b_issued[kBStages], u_issued[2] = {-1, -1};
      for (int s = 0; s < kBStages; ++s) b_issued[s] = -1;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int n0 = (c0 + t * cstride) * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->b_empty[bstage]), bph ^ 1, deadline, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bfull = tc::smem_u32(&bar->b_full[bstage]);
          tc::mbar_arrive_expect_tx(bfull, kBStage);
          tc::tma_load_2d(tc::smem_u32(sB + bstage * kBStage), &tmap_w2, bfull, kb * kBK, n0, keep);
          b_issued[bstage] = bph;
          if (++bstage == kBStages) { bstage = 0; bph ^= 1; }
        }
        for (int h = 0; h < 2 && ok; ++h) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->u_empty[h]), (t & 1) ^ 1, deadline, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t ufull = tc::smem_u32(&bar->u_full[h]);
          tc::mbar_arrive_expect_tx(ufull, kUHalfTile);
          const uint32_t ud = tc::smem_u32(sU + h * kUHalfTile);
          tc::tma_load_3d(ud, &tmap_u, ufull, n0 + h * kHalfN, p.k - 1, m0, stream);
          tc::tma_load_3d(ud + kUBox, &tmap_u, ufull, n0 + h * kHalfN + 64, p.k - 1, m0, stream);
          u_issued[h] = t & 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, DSPARK_ETIMEOUT);
        // wait (bounded) for every copy this thread put in flight before the CTA exits
        const long long dl = tc::deadline_after_ns(200000000ull);
        const volatile int never = 0;
        for (int s = 0; s < kBStages; ++s)
          if (b_issued[s] >= 0) tc::mbar_wait_bounded(tc::smem_u32(&bar->b_full[s]), b_issued[s], dl, &never);
        for (int h = 0; h < 2; ++h)
          if (u_issued[h] >= 0) tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[h]), u_issued[h], dl, &never);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
      int bstage = 0, bph = 0, ab = 0, aph = 0;
      bool ok = tc::mbar_wait_bounded(tc::smem_u32(&bar->a_ready), 0, deadline, abort_flag);
      bool issued = false;
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
          const uint32_t a_addr = tc::smem_u32(sA + kb * kAAtom);
          const uint32_t b_addr = tc::smem_u32(sB + bstage * kBStage);
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
        set_status(p.status, DSPARK_ETIMEOUT);
        if (issued) {  // wait (bounded) for the MMAs already issued before TMEM is freed
          tc::mma_commit(tc::smem_u32(&bar->drain));
          const volatile int never = 0;
          tc::mbar_wait_bounded(tc::smem_u32(&bar->drain), 0, tc::deadline_after_ns(200000000ull), &never);
        }
      } else {
        bar->mma_pending = issued;  // complete only once the epilogue has consumed every accumulator
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int m = wq * 32 + lane;     // tile row = TMEM lane
    const int half = (warp - 2) >> 2; // warp set: columns 128 half .. 128 half + 127 of each tile
    const int grow = m0 + m;
    const float inv_tau = p.inv_tau;
    const float c2 = inv_tau * kLog2e;
    // The chunk Gumbels (Philox purpose 1) of this row and of the first kGReg tiles do not
    // depend on any logit: draw them before waiting for the previous kernel, so that the Philox
    // rounds overlap its tail instead of the tile loop.  Later tiles draw theirs in the loop.
    constexpr int kGReg = 6;
    float2 gk[kGReg];
#pragma unroll
    for (int i = 0; i < kGReg; ++i) {
      gk[i] = make_float2(0.f, 0.f);
      if (!p.greedy && i < n_tiles) gk[i] = tile_gumbels(p.seed, p.step, grow, p.k, c0 + i * cstride, half);
    }
    // x_{k-1} comes from the previous kernel (the select of position k-1): everything above
    // -- barrier set-up, TMEM, the producer's U / W2 prefetch, the Gumbels -- overlapped with it
    tc::grid_dependency_wait();
    {
      // A operand: rows m0..m0+127 of the factor -- W1[x_{k-1}] (Markov head) or s_k (RNN head)
      // -- in the 128-byte-swizzled K-major layout.  Row indices first, then every 16-byte row
      // chunk as an independent cp.async.
      const __nv_bfloat16* base = p.states ? p.states : p.W1;
      const int et = tid - 64;
      for (int mm = et; mm < kBM; mm += kEpiThreads) {
        const int gr = m0 + mm;
        int idx = -1;
        if (gr < bs)
          idx = p.states ? gr * p.gamma + p.k - 1
                         : clamp_token((p.k == 1) ? p.anchor[gr] : p.tokens[size_t(gr) * p.gamma + p.k - 2], V);
        bar->xrow[mm] = idx;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      const int cpr = r / 8;  // 16-byte chunks per row
      for (int idx = et; idx < kBM * cpr; idx += kEpiThreads) {
        const int row = idx / cpr, ch = idx % cpr;
        const int xp = bar->xrow[row];
        const int kb = ch >> 3, j = ch & 7;
        const uint32_t dst = tc::smem_u32(sA + kb * kAAtom + row * 128 + ((j ^ (row & 7)) << 4));
        cp_async16(dst, xp >= 0 ? base + size_t(xp) * r + ch * 8 : base, xp >= 0 ? 16u : 0u);
      }
      cp_async_wait_all();
      tc::fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->a_ready));

    const uint32_t taddr = tmem_base + (uint32_t(wq * 32) << 16) + half * kHalfN;
    const uint8_t* ub = sU + half * kUHalfTile + m * 128;  // this row in U half `half`
    // running (max, sum-exp) in log2 units: run_m = max of l c2, run_s = sum of 2^(l c2 - run_m)
    float run_m = -INFINITY, run_s = 0.f, best_key = -INFINITY;
    int best_c = INT_MAX;
    for (int t = 0; t < n_tiles; ++t) {
      const int c = c0 + t * cstride;
      const int n0 = c * kBN + half * kHalfN;  // this set's first id
      const int valid = min(kHalfN, V - n0);   // <= 0: this set's half lies past the vocabulary
      const int ab = t & 1;
      bool ok = tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_full[ab]), (t >> 1) & 1, deadline, abort_flag) &&
                tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[half]), t & 1, deadline, abort_flag);
      // one decision per warp before the .sync.aligned TMEM loads; warps run independently
      // (no named barrier in this loop), so a warp that gives up can hold up no other
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, DSPARK_ETIMEOUT);
        break;
      }
      tc::tc_fence_after();
      float v[kHalfN];
#pragma unroll
      for (int q = 0; q < kHalfN / 32; ++q)
        tc::tmem_ld32(taddr + ab * kBN + q * 32, reinterpret_cast<uint32_t*>(v + q * 32));
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->acc_empty[ab]));
#pragma unroll
      for (int j = 0; j < kHalfN / 8; ++j) {  // + U_k: 16-byte groups of the half's two 64-id boxes
        const uint4 q = *reinterpret_cast<const uint4*>(ub + (j >> 3) * kUBox + (((j & 7) ^ (m & 7)) << 4));
        v[8 * j + 0] += bf16lo(q.x); v[8 * j + 1] += bf16hi(q.x);
        v[8 * j + 2] += bf16lo(q.y); v[8 * j + 3] += bf16hi(q.y);
        v[8 * j + 4] += bf16lo(q.z); v[8 * j + 5] += bf16hi(q.z);
        v[8 * j + 6] += bf16lo(q.w); v[8 * j + 7] += bf16hi(q.w);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->u_empty[half]));

      if (p.greedy) {
        float best = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int q = 0; q < kHalfN; ++q)
          if (q < valid && v[q] > best) { best = v[q]; bi = q; }
        // chunks arrive in increasing order: a strict > keeps the lowest index on ties
        if (best > best_key) { best_key = best; best_c = n0 + bi; }
      } else {
        float2 g;
        if (t < kGReg) {
          g = gk[0];
#pragma unroll
          for (int j = 0; j + 1 < kGReg; ++j) gk[j] = gk[j + 1];
        } else {
          g = tile_gumbels_call(p.seed, p.step, grow, p.k, c, half);
        }
        // the set's draft chunks 4c + 2h (ids 0..63 of its half) and 4c + 2h + 1, in that order;
        // only the last tile of a vocabulary that is not a multiple of 256 is ragged
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float* vq = v + q * kDraftIds;
          const int vl = valid - q * kDraftIds;
          const bool full = vl >= kDraftIds;
          const float mx = full ? row_max<false>(vq, vl) : row_max<true>(vq, vl);
          if (mx > -INFINITY) {
            const float sc = full ? row_sum_exp2<false>(vq, vl, mx * c2, c2)
                                  : row_sum_exp2<true>(vq, vl, mx * c2, c2);
            const float key = mx * inv_tau + logf(sc) + (q ? g.y : g.x);  // log-mass + Gumbel
            if (key > best_key) { best_key = key; best_c = 4 * c + 2 * half + q; }
            const float m2 = mx * c2;
            if (m2 > run_m) {
              run_s = run_s * exp2f(run_m - m2) + sc;
              run_m = m2;
            } else {
              run_s += sc * exp2f(m2 - run_m);
            }
          }
        }
      }
    }
    run_m *= 0.69314718055994531f;  // back to natural units: max of l / T
    // the two warp sets of a lane quarter meet in shared memory after the final barrier
    if (half == 1) bar->xch[m] = make_float4(run_m, run_s, best_key, __int_as_float(best_c));
    xmine = make_float4(run_m, run_s, best_key, __int_as_float(best_c));
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) free_tmem(bar, tmem_base, lane);
  if (warp >= 2 && warp < 6) {
    // warp set 0 merges the other set's entry of the same row and writes the CTA's entry
    // (request grow, slot c0); within a tile set 0's chunks come first, so on equal keys its
    // (lower) chunk wins, as the merge's lowest-index rule gives
    const int m = (warp & 3) * 32 + lane, grow = m0 + m;
    const float4 o = bar->xch[m];
    const LsePair l = lse_merge(LsePair{xmine.x, xmine.y}, LsePair{o.x, o.y});
    const ArgMax a = better(ArgMax{xmine.z, __float_as_int(xmine.w)}, ArgMax{o.z, __float_as_int(o.w)});
    if (grow < bs) p.entries[size_t(grow) * p.n_slots + c0] = make_float4(l.m, l.s, a.v, __int_as_float(a.i));
  }
}

}  // namespace

uint64_t g_wait_timeout_ns = 1000000000ull;  // 1 s; changed only through dspark_set_wait_timeout_ns

bool draft_tc_supported(int dtype, int bs, int V, int r) {
  return dtype == DSPARK_BF16 && bs >= 1 && bs <= 2 * kBM && r % kBK == 0 && r <= 256 && V % 8 == 0 &&
         tch::encode_fn() != nullptr;
}

int draft_tc_slots(int bs, int V) {
  const int n_mt = (bs + kBM - 1) / kBM;
  return tch::vocab_grid(bs, (V + kBN - 1) / kBN) / n_mt;
}

cudaError_t launch_draft_stats_tc(const void* U, const void* W1, const void* W2t, const void* states,
                                  const int32_t* anchor, const int32_t* tokens, int bs, int gamma,
                                  int V, int r, int k, float inv_tau, int greedy, uint64_t seed,
                                  uint64_t step, void* entries, int n_chunks, int* n_slots,
                                  uint32_t* status, cudaStream_t s) {
  (void)n_chunks;
  if (!tch::encode_fn()) return cudaErrorNotSupported;
  CUtensorMap map_w2, map_u;
  if (!tch::encode_bf16_2d(&map_w2, W2t, size_t(V), size_t(r), kBN)) return cudaErrorInvalidValue;
  {
    const cuuint64_t dims[3] = {cuuint64_t(V), cuuint64_t(gamma), cuuint64_t(bs)};
    const cuuint64_t strides[2] = {cuuint64_t(V) * 2, cuuint64_t(gamma) * V * 2};
    const cuuint32_t box[3] = {64, 1, kBM};
    const cuuint32_t es[3] = {1, 1, 1};
    if (tch::encode_fn()(&map_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static bool smem_set[tch::kMaxDevices] = {};
  static std::mutex smem_mu;
  if (cudaError_t e = tch::set_smem_once(draft_tc_kernel, int(smem_bytes(256)), smem_set, &smem_mu)) return e;
  const int n_tiles = (V + kBN - 1) / kBN;
  const int grid = tch::vocab_grid(bs, n_tiles);
  Params prm{};
  prm.W1 = static_cast<const __nv_bfloat16*>(W1);
  prm.states = static_cast<const __nv_bfloat16*>(states);
  prm.anchor = anchor;
  prm.tokens = tokens;
  prm.bs = bs; prm.gamma = gamma; prm.V = V; prm.r = r; prm.k = k;
  prm.inv_tau = inv_tau;
  prm.greedy = greedy;
  prm.n_tiles = n_tiles;
  prm.status = status;
  prm.timeout_ns = g_wait_timeout_ns;
  prm.entries = static_cast<float4*>(entries);
  prm.n_slots = grid / ((bs + kBM - 1) / kBM);
  prm.seed = seed;
  prm.step = step;
  *n_slots = prm.n_slots;
  // programmatic dependent launch: set-up and prefetch overlap the previous kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes(r);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, draft_tc_kernel, map_w2, map_u, prm);
}

}  // namespace dspark
