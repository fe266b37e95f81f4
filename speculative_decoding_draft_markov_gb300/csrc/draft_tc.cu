// Tensor-core vocabulary passes: tcgen05.mma (bf16 in, fp32 accumulate in TMEM), operands
// staged by TMA, fused epilogues.  No [bs, V] logit tensor ever reaches HBM.
//
// DSpark technical summary, "Architecture (drafter)": the Markov head's bias for position k
// is W1[x_{k-1}] W2 (rank r = 256), added to the backbone's base logits U_k over the full
// vocabulary.  Per position this is a GEMM [bs, r] x [r, V] consumed at once by a sampler.
// Two passes share the kernel:
//   DRAFT  (S1, one launch per position k): l = U_k + W1[x_{k-1}] W2; per (request, 128-id
//          chunk): (max l/tau, sum exp(l/tau - max)), or (max l, argmax) at temperature 0.
//   DECIDE (S5, after the accept scan): for each request's deciding row, p_t = softmax of the
//          target row, p_d = softmax of the draft logits recomputed at the rejected position;
//          per chunk: (sum max(0, p_t - p_d), sum p_t) -- the residual / bonus masses.
//
// Work decomposition:
//   tile      = 128 requests (TMEM lanes) x 128 vocabulary ids (= one sampler chunk), K = r
//   CTA       = persistent; fixed 128-request M-tile, strided over vocabulary chunks; the
//               gathered A operand W1[x] (128 x r) stays resident in shared memory
//   warp 0    = TMA producer: W2t tiles in K-stages of 64 (evict-last: W2 is re-read by every
//               position) and, in DRAFT, the U tile (3-D map over [bs, gamma, V], evict-first)
//   warp 1    = TMEM owner + single-thread tcgen05.mma issuer, commits to mbarriers
//   warps 2-9 = epilogue, two warps per TMEM lane quarter (one request row per thread).
//               DRAFT: the two warp sets take alternate tiles (full 128-id chunks) and keep
//               per-row running statistics and the best chunk key in registers; each CTA
//               writes one entry per request at the end (DraftEntry), so the select merges
//               one entry per CTA instead of one per chunk.  DECIDE: each warp reduces 64 of
//               a tile's 128 columns into a half-chunk entry.
//   warps 10-11 = (DECIDE) cp.async gather of each request's U row and target row, one warp
//               per 64-column half, so one half refills while the other is being reduced
//   2 TMEM accumulators (256 columns) let MMA, loads and epilogue overlap.
// Every mbarrier wait is bounded (SM cycle-counter deadline + shared abort flag); on give-up the
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
constexpr int kBStagesMax = 6;
constexpr int kUStages = 2;                      // DRAFT: U ring; DECIDE: one U + one target stage
constexpr int kAccBufs = 2;
constexpr uint32_t kAtomBytes = kBM * kBK * 2;   // 16 KB: 128 rows x 128 bytes
constexpr uint32_t kUHalf = kBM * 64 * 2;        // 16 KB: one 64-column half of a 128 x 128 bf16 tile
constexpr uint32_t kTmemCols = kAccBufs * kBN;   // 256
constexpr float kLog2e = 1.4426950408889634f;

// 8 epilogue warps, two per TMEM lane quarter.  DRAFT: W2t ring of 5 K-stages (leaving room
// for a select block to sit beside this one on an SM).  DECIDE: 4 K-stages and two gather
// warps, one per 64-column half of the U and target rows, each half with its own full / empty
// barrier pair.
template <bool kDecide>
__host__ __device__ constexpr int b_stages() { return kDecide ? 4 : 5; }
template <bool kDecide>
__host__ __device__ constexpr int epi_warps() { return 8; }
template <bool kDecide>
__host__ __device__ constexpr int threads() { return 32 * (2 + epi_warps<kDecide>() + (kDecide ? 2 : 0)); }

struct Barriers {
  uint64_t b_full[kBStagesMax], b_empty[kBStagesMax];
  uint64_t u_full[kUStages], u_empty[kUStages];
  uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  uint64_t drain;
  uint64_t a_ready;  // DRAFT: the A operand is in shared memory (one arrival per epilogue warp)
  uint32_t tmem_base;
  int abort;
  int xrow[kBM];  // W1 row of each A row (-1: zero row)
  float4 xch[kBM];  // DRAFT: warp set 1's entry of each row, merged by set 0 at the end
};

// Per-row facts of the DECIDE pass (one request per tile row).
struct RowMeta {
  long long u_off;  // element offset of U[b, kdec-1, 0] (residual rows)
  long long t_off;  // element offset of target[pdec, 0] (live rows)
  float a_t;        // lse_t * log2(e)
  float a_d;        // lse_d * log2(e)
  int resid;        // residual row (else bonus, or dead)
  int live;         // the request has a decision
};

struct Params {
  const __nv_bfloat16* W1;
  const int32_t* anchor;
  const int32_t* tokens;
  int bs, gamma, V, r, k;
  float inv_tau;
  int greedy;
  float2* stats;    // DECIDE: per (request, chunk) half-chunk masses
  int n_chunks;
  uint32_t* status;
  uint64_t timeout_ns;
  // DRAFT only
  float4* entries;  // per (request, slot): see DraftEntry
  int n_slots;
  uint64_t seed, step;
  // DECIDE only
  const __nv_bfloat16* U;
  const __nv_bfloat16* target;
  const float* lse_d;
  const RowStat* rs;
  const Decision* dec;
};

// Dynamic shared memory: A atoms | W2t ring | U stages | DECIDE row facts | barriers.  The
// buffer is declared 1024-byte aligned (128-byte swizzle atoms).
template <bool kDecide>
__host__ __device__ constexpr size_t extra_bytes() {
  return kDecide ? kBM * sizeof(RowMeta) : 0;
}
template <bool kDecide>
__host__ __device__ constexpr size_t smem_bytes(int r) {
  return size_t(r / kBK) * kAtomBytes + b_stages<kDecide>() * kAtomBytes + kUStages * 2 * kUHalf +
         extra_bytes<kDecide>() + sizeof(Barriers);
}

static_assert(smem_bytes<false>(256) <= 232448 && smem_bytes<true>(256) <= 232448,
              "dynamic shared memory beyond the 227 KB per-block limit");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The chunk Gumbel G_c of request `req` at position k (Philox purpose 1, index c).  Kept out of
// line: inlined into the DRAFT tile loop its Philox rounds raise register pressure there
// enough to spill, although the loop only calls it for tiles past the ones drawn up front.
__device__ __noinline__ float chunk_gumbel_call(uint64_t seed, uint64_t step, int req, int k, int c) {
  const uint4 w = philox_group(seed, step, kDraftChunk, uint32_t(req), k, uint32_t(c) >> 2);
  return gumbel_from_bits(pick_word(w, c & 3));
}

__device__ __forceinline__ void unpack8(const uint4 q, float* x) {
  x[0] = bf16lo(q.x); x[1] = bf16hi(q.x); x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
  x[4] = bf16lo(q.z); x[5] = bf16hi(q.z); x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
}

template <bool kDecide>
__global__ void __launch_bounds__(threads<kDecide>(), 1) stats_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_u, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int kBStages = b_stages<kDecide>();
  constexpr int kEpiThreads = 32 * epi_warps<kDecide>();
  if (tc::smem_u32(smem_raw) & 1023u) {  // the swizzled layouts need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, DSPARK_EUNSUPPORTED);
    return;
  }
  uint8_t* smem = smem_raw;
  const int nk = p.r / kBK;
  uint8_t* sA = smem;                                   // nk atoms
  uint8_t* sB = sA + nk * kAtomBytes;                   // kBStages atoms
  uint8_t* sU = sB + kBStages * kAtomBytes;             // kUStages x 32 KB
  uint8_t* sX = sU + kUStages * 2 * kUHalf;             // row facts (DECIDE)
  RowMeta* meta = reinterpret_cast<RowMeta*>(sX);
  Barriers* bar = reinterpret_cast<Barriers*>(sX + extra_bytes<kDecide>());
  volatile int* abort_flag = &bar->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bs = p.bs, V = p.V, r = p.r;
  const int n_mt = (bs + kBM - 1) / kBM;
  const int m0 = (blockIdx.x % n_mt) * kBM;
  const int cstride = gridDim.x / n_mt;
  const int c0 = blockIdx.x / n_mt;
  const int n_tiles = (c0 < p.n_chunks) ? (p.n_chunks - c0 + cstride - 1) / cstride : 0;

  if (tid == 0) {
    for (int s = 0; s < kBStages; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->b_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&bar->b_empty[s]), 1);
    }
    for (int s = 0; s < kUStages; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->u_full[s]), kDecide ? 32 : 1);  // DECIDE: one arrive per loader lane
      // one arrival per epilogue warp that reads the stage: DRAFT, the warp set of tiles with
      // this parity; DECIDE, the warps of the column half the stage holds
      tc::mbar_init(tc::smem_u32(&bar->u_empty[s]), kEpiThreads / 64);
    }
    for (int s = 0; s < kAccBufs; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->acc_full[s]), 1);
      // DRAFT: one warp set per accumulator buffer; DECIDE: every epilogue warp
      tc::mbar_init(tc::smem_u32(&bar->acc_empty[s]), kDecide ? kEpiThreads / 32 : kEpiThreads / 64);
    }
    tc::mbar_init(tc::smem_u32(&bar->drain), 1);
    tc::mbar_init(tc::smem_u32(&bar->a_ready), kEpiThreads / 32);
    bar->abort = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w2);
    if (!kDecide) tc::prefetch_tensormap(&tmap_u);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&bar->tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  if (kDecide) {
    tc::grid_dependency_wait();  // the decisions come from the previous kernel
    for (int m = tid; m < kBM; m += threads<kDecide>()) {
      RowMeta rm{0, 0, 0.f, 0.f, 0, 0};
      const int grow = m0 + m;
      if (grow < bs) {
        const Decision d = p.dec[grow];
        if (d.kind != kDecNone) {
          rm.live = 1;
          rm.t_off = (long long)d.pdec * V;
          rm.a_t = p.rs[d.pdec].lse * kLog2e;
          if (d.kind == kDecResidual) {
            rm.resid = 1;
            rm.u_off = ((long long)grow * p.gamma + d.kdec - 1) * V;
            rm.a_d = p.lse_d[(size_t)grow * p.gamma + d.kdec - 1] * kLog2e;
          }
        }
      }
      meta[m] = rm;
    }
  }
  // A operand: rows m0..m0+127 of W1[x] in the 128-byte-swizzled K-major layout, where x is
  // x_{k-1} (DRAFT) or the token before each residual row's rejected position (DECIDE).
  // Token ids first, then every 16-byte row chunk as an independent cp.async.  `first` and
  // `count` select the threads that take part, `sync` makes the token ids visible to them.
  auto gather_a = [&](int first, int count, auto sync) {
    for (int m = tid - first; m < kBM; m += count) {
      const int grow = m0 + m;
      int xp = -1;
      if (grow < bs) {
        int kx = p.k;  // position whose previous token selects the W1 row
        bool use = true;
        if (kDecide) {
          const Decision d = p.dec[grow];
          use = d.kind == kDecResidual;
          kx = d.kdec;
        }
        if (use) xp = clamp_token((kx == 1) ? p.anchor[grow] : p.tokens[size_t(grow) * p.gamma + kx - 2], V);
      }
      bar->xrow[m] = xp;
    }
    sync();
    const int cpr = r / 8;  // 16-byte chunks per row
    for (int idx = tid - first; idx < kBM * cpr; idx += count) {
      const int row = idx / cpr, ch = idx % cpr;
      const int xp = bar->xrow[row];
      const int kb = ch >> 3, j = ch & 7;
      const uint32_t dst = tc::smem_u32(sA + kb * kAtomBytes + row * 128 + ((j ^ (row & 7)) << 4));
      cp_async16(dst, xp >= 0 ? p.W1 + size_t(xp) * r + ch * 8 : p.W1, xp >= 0 ? 16u : 0u);
    }
    cp_async_wait_all();
    tc::fence_proxy_async_smem();
  };
  if (kDecide) gather_a(0, threads<kDecide>(), [] { __syncthreads(); });
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = bar->tmem_base;
  const long long deadline = tc::deadline_after_ns(p.timeout_ns);
  tc::grid_launch_dependents();  // the next kernel may start its own set-up now
  float4 xmine = make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(INT_MAX));  // DRAFT epilogue entry

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
        if (!kDecide) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->u_empty[us]), uph ^ 1, deadline, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t ufull = tc::smem_u32(&bar->u_full[us]);
          tc::mbar_arrive_expect_tx(ufull, 2 * kUHalf);
          const uint32_t ud = tc::smem_u32(sU + us * 2 * kUHalf);
          tc::tma_load_3d(ud, &tmap_u, ufull, n0, p.k - 1, m0, stream);
          tc::tma_load_3d(ud + kUHalf, &tmap_u, ufull, n0 + 64, p.k - 1, m0, stream);
          u_issued[us] = uph;
          if (++us == kUStages) { us = 0; uph ^= 1; }
        }
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
        set_status(p.status, DSPARK_ETIMEOUT);
        // wait (bounded) for every copy this thread put in flight before the CTA exits
        const long long dl = tc::deadline_after_ns(200000000ull);
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
      bool ok = kDecide || tc::mbar_wait_bounded(tc::smem_u32(&bar->a_ready), 0, deadline, abort_flag);
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
        set_status(p.status, DSPARK_ETIMEOUT);
        if (issued) {  // wait (bounded) for the MMAs already issued before TMEM is freed
          tc::mma_commit(tc::smem_u32(&bar->drain));
          const volatile int never = 0;
          tc::mbar_wait_bounded(tc::smem_u32(&bar->drain), 0, tc::deadline_after_ns(200000000ull), &never);
        }
      }
    }
  } else if (kDecide && warp >= 2 + epi_warps<kDecide>()) {
    // ------------------------------------------------------------------ row gather (DECIDE)
    // Gather warp h fills column half h of the U rows (first 32 KB) and target rows (second
    // 32 KB); barrier pair h (u_full / u_empty) guards that half.
    const int h = warp - (2 + epi_warps<kDecide>());
    int ph = 0;
    bool ok = true;
    const int j = lane & 7, rsub = lane >> 3;  // 16-byte chunk in the half row, row within a group of 4
    const uint32_t su = tc::smem_u32(sU + h * kUHalf), st = tc::smem_u32(sU + 2 * kUHalf + h * kUHalf);
    for (int t = 0; t < n_tiles; ++t) {
      const int n0 = (c0 + t * cstride) * kBN;
      if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->u_empty[h]), ph ^ 1, deadline, abort_flag)) {
        ok = false;
        break;
      }
      const int col = n0 + h * 64 + j * 8;
      const bool in_v = col < V;
#pragma unroll 4
      for (int it = 0; it < kBM / 4; ++it) {
        const int row = it * 4 + rsub;
        const RowMeta rm = meta[row];
        const uint32_t off = row * 128 + ((j ^ (row & 7)) << 4);
        const bool gu = rm.resid && in_v, gt = rm.live && in_v;
        cp_async16(su + off, gu ? p.U + rm.u_off + col : p.U, gu ? 16u : 0u);
        cp_async16(st + off, gt ? p.target + rm.t_off + col : p.target, gt ? 16u : 0u);
      }
      cp_async_arrive_noinc(tc::smem_u32(&bar->u_full[h]));
      ph ^= 1;
    }
    if (!ok) {
      *abort_flag = 1;
      set_status(p.status, DSPARK_ETIMEOUT);
    }
    cp_async_wait_all();  // no copy of this warp outlives the CTA
  } else if (!kDecide && warp >= 2 && warp < 2 + epi_warps<kDecide>()) {
    // ------------------------------------------------------------------ DRAFT epilogue
    // Warp set `half` (4 warps, one per TMEM lane quarter) takes the CTA's tiles t = half,
    // half + 2, ...: accumulator buffer `half` and U stage `half` always.  A thread owns one
    // request row and, per tile (= one 128-id chunk), reduces the chunk to its log-mass and the
    // chunk's Gumbel key, keeping in registers the running (max, sum-exp) over its chunks and
    // the best key seen (at temperature 0: the running max logit and its lowest index).
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int m = wq * 32 + lane;     // tile row = TMEM lane
    const int half = (warp - 2) >> 2; // warp set
    const int grow = m0 + m;
    const float inv_tau = p.inv_tau;
    const float c2 = inv_tau * kLog2e;
    // The chunk Gumbels (Philox purpose 1) of this row and of the set's first kGReg tiles do not
    // depend on any logit: draw them before waiting for the previous kernel, so that the Philox
    // rounds overlap its tail instead of the tile loop.  Later tiles draw theirs in the loop.
    constexpr int kGReg = 8;
    auto chunk_gumbel = [&](int c) {
      const uint4 w = philox_group(p.seed, p.step, kDraftChunk, uint32_t(grow), p.k, uint32_t(c) >> 2);
      return gumbel_from_bits(pick_word(w, c & 3));
    };
    float gk[kGReg];
#pragma unroll
    for (int i = 0; i < kGReg; ++i) {
      const int t = half + 2 * i;
      gk[i] = (!p.greedy && t < n_tiles) ? chunk_gumbel(c0 + t * cstride) : 0.f;
    }
    // x_{k-1} comes from the previous kernel (the select of position k-1): everything above
    // -- barrier set-up, TMEM, the producer's U / W2 prefetch, the Gumbels -- overlapped with it
    tc::grid_dependency_wait();
    gather_a(64, kEpiThreads, [] { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); });
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->a_ready));

    const uint32_t taddr = tmem_base + (uint32_t(wq * 32) << 16) + half * kBN;
    const uint8_t* ub = sU + half * 2 * kUHalf + m * 128;
    // running (max, sum-exp) in log2 units: run_m = max of l c2, run_s = sum of 2^(l c2 - run_m)
    float run_m = -INFINITY, run_s = 0.f, best_key = -INFINITY;
    int best_c = INT_MAX;
    int ph = 0;
    for (int t = half, i = 0; t < n_tiles; t += 2, ++i, ph ^= 1) {
      const int c = c0 + t * cstride;
      const int n0 = c * kBN;
      const int valid = min(kBN, V - n0);
      bool ok = tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_full[half]), ph, deadline, abort_flag) &&
                tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[half]), ph, deadline, abort_flag);
      // one decision per warp before the .sync.aligned TMEM loads; warps run independently
      // (no named barrier in this loop), so a warp that gives up can hold up no other
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, DSPARK_ETIMEOUT);
        break;
      }
      tc::tc_fence_after();
      float v[kBN];
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) tc::tmem_ld32(taddr + q * 32, reinterpret_cast<uint32_t*>(v + q * 32));
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->acc_empty[half]));
#pragma unroll
      for (int j = 0; j < kBN / 8; ++j) {  // + U_k: 16-byte groups of the two 64-column halves
        float x[8];
        unpack8(*reinterpret_cast<const uint4*>(ub + (j >> 3) * kUHalf + (((j & 7) ^ (m & 7)) << 4)), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * j + e] += x[e];
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->u_empty[half]));

      if (p.greedy) {
        float best = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i < valid && v[i] > best) { best = v[i]; bi = i; }
        // chunks arrive in increasing order: a strict > keeps the lowest index on ties
        if (best > best_key) { best_key = best; best_c = n0 + bi; }
      } else {
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i < valid) m4[i & 3] = fmaxf(m4[i & 3], v[i]);
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i < valid) s4[i & 3] += exp2f((v[i] - mx) * c2);
        const float sc = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        float g;
        if (i < kGReg) {
          g = gk[0];
#pragma unroll
          for (int j = 0; j + 1 < kGReg; ++j) gk[j] = gk[j + 1];
        } else {
          g = chunk_gumbel_call(p.seed, p.step, grow, p.k, c);
        }
        if (mx > -INFINITY) {
          const float key = mx * inv_tau + logf(sc) + g;  // chunk log-mass + Gumbel
          if (key > best_key) { best_key = key; best_c = c; }
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
    run_m *= 0.69314718055994531f;  // back to natural units: max of l / T
    // the two warp sets of a lane quarter meet in shared memory after the final barrier
    if (half == 1) bar->xch[m] = make_float4(run_m, run_s, best_key, __int_as_float(best_c));
    xmine = make_float4(run_m, run_s, best_key, __int_as_float(best_c));
  } else if (kDecide && warp >= 2 && warp < 2 + epi_warps<kDecide>()) {
    // ------------------------------------------------------------------ DECIDE epilogue
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int m = wq * 32 + lane;     // tile row = TMEM lane
    const int half = (warp - 2) >> 2; // which 64 of the 128 columns this warp takes
    const int grow = m0 + m;
    const float inv_tau = p.inv_tau;
    const float c2 = inv_tau * kLog2e;
    int uph = 0, ab = 0, aph = 0;
    for (int t = 0; t < n_tiles; ++t) {
      const int c = c0 + t * cstride;
      const int n0 = c * kBN;
      const int valid = min(kBN, V - n0);
      bool ok = tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_full[ab]), aph, deadline, abort_flag) &&
                tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[half]), uph, deadline, abort_flag);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, DSPARK_ETIMEOUT);
        break;
      }
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t(wq * 32) << 16) + ab * kBN;
      // residual / bonus masses of this half row, 32 columns at a time
      constexpr int kH = kBN / 2;
      const RowMeta rm = meta[m];
      const uint8_t* ub = sU + half * kUHalf + m * 128;              // U rows, this half
      const uint8_t* tb = sU + 2 * kUHalf + half * kUHalf + m * 128; // target rows, this half
      const int vh = valid - half * kH;
      float R = 0.f, P = 0.f;
#pragma unroll
      for (int q = 0; q < kH / 32; ++q) {
        float v[32];
        tc::tmem_ld32(taddr + half * kH + q * 32, reinterpret_cast<uint32_t*>(v));
        tc::tmem_ld_wait();
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const int j = q * 4 + j4;  // 16-byte chunk within the half row
          const uint32_t off = ((j ^ (m & 7)) << 4);
          float xu[8], xt[8];
          unpack8(*reinterpret_cast<const uint4*>(ub + off), xu);
          unpack8(*reinterpret_cast<const uint4*>(tb + off), xt);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = 8 * j + e;
            const float pt = exp2f(fmaf(xt[e], c2, -rm.a_t));
            const float pd = exp2f(fmaf(v[8 * j4 + e] + xu[e], c2, -rm.a_d));
            const float w = rm.resid ? fmaxf(0.f, pt - pd) : pt;
            if (i < vh && rm.live) {
              R += w;
              P += pt;
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(tc::smem_u32(&bar->acc_empty[ab]));
        tc::mbar_arrive(tc::smem_u32(&bar->u_empty[half]));
      }
      if (++ab == kAccBufs) { ab = 0; aph ^= 1; }
      uph ^= 1;  // each half's stage is refilled every tile
      if (grow < bs) p.stats[(size_t(grow) * p.n_chunks + c) * kStatsPerChunk + half] = make_float2(R, P);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
  if (!kDecide && warp >= 2 && warp < 6) {
    // DRAFT: warp set 0 merges the other set's entry of the same row and writes the CTA's
    // entry (request grow, slot c0) -- see DraftEntry
    const int m = (warp & 3) * 32 + lane, grow = m0 + m;
    const float4 o = bar->xch[m];
    const LsePair l = lse_merge(LsePair{xmine.x, xmine.y}, LsePair{o.x, o.y});
    const ArgMax a = better(ArgMax{xmine.z, __float_as_int(xmine.w)}, ArgMax{o.z, __float_as_int(o.w)});
    if (grow < bs) p.entries[size_t(grow) * p.n_slots + c0] = make_float4(l.m, l.s, a.v, __int_as_float(a.i));
  }
}

// ---------------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

constexpr int kMaxDevices = 64;

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

// Multiprocessor count of the current device (queried once per device).
int sm_count() {
  static int cache[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

bool encode_w2(CUtensorMap* map, const void* W2t, int V, int r) {
  const cuuint64_t dims[2] = {cuuint64_t(r), cuuint64_t(V)};
  const cuuint64_t strides[1] = {cuuint64_t(r) * 2};
  const cuuint32_t box[2] = {kBK, kBN};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2t), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Persistent grid: one CTA per SM, a whole number of CTAs per 128-request M-tile, at most one
// per (M-tile, chunk).  CTA b takes M-tile b % n_mt and chunks b / n_mt + j * (grid / n_mt).
int grid_size(int bs, int n_chunks) {
  const int n_mt = (bs + kBM - 1) / kBM;
  const int grid = (sm_count() / n_mt) * n_mt;
  return max(n_mt, min(grid, n_mt * n_chunks));
}

template <bool kDecide>
cudaError_t launch(const CUtensorMap& w2, const CUtensorMap& u, const Params& prm, cudaStream_t s) {
  const size_t smem = smem_bytes<kDecide>(prm.r);
  static bool attr_set[kMaxDevices] = {};  // the shared-memory opt-in, once per device
  static std::mutex attr_mutex;
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(attr_mutex);
    if (!attr_set[dev]) {
      const cudaError_t attr = cudaFuncSetAttribute(stats_tc_kernel<kDecide>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    int(smem_bytes<kDecide>(256)));
      if (attr != cudaSuccess) return attr;
      attr_set[dev] = true;
    }
  }
  const int grid = grid_size(prm.bs, prm.n_chunks);
  // programmatic dependent launch: set-up and prefetch overlap the previous kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads<kDecide>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stats_tc_kernel<kDecide>, w2, u, prm);
}

}  // namespace

uint64_t g_wait_timeout_ns = 1000000000ull;  // 1 s; changed only through dspark_set_wait_timeout_ns

bool draft_tc_supported(int dtype, int bs, int V, int r) {
  return dtype == DSPARK_BF16 && bs >= 1 && bs <= 2 * kBM && r % kBK == 0 && r <= 256 && V % 8 == 0 &&
         encode_fn() != nullptr;
}

cudaError_t launch_draft_stats_tc(const void* U, const void* W1, const void* W2t,
                                  const int32_t* anchor, const int32_t* tokens, int bs, int gamma,
                                  int V, int r, int k, float inv_tau, int greedy, uint64_t seed,
                                  uint64_t step, void* entries, int n_chunks, int* n_slots,
                                  uint32_t* status, cudaStream_t s) {
  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap map_w2, map_u;
  if (!encode_w2(&map_w2, W2t, V, r)) return cudaErrorInvalidValue;
  {
    const cuuint64_t dims[3] = {cuuint64_t(V), cuuint64_t(gamma), cuuint64_t(bs)};
    const cuuint64_t strides[2] = {cuuint64_t(V) * 2, cuuint64_t(gamma) * V * 2};
    const cuuint32_t box[3] = {64, 1, kBM};
    const cuuint32_t es[3] = {1, 1, 1};
    if (encode_fn()(&map_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  Params prm{};
  prm.W1 = static_cast<const __nv_bfloat16*>(W1);
  prm.anchor = anchor;
  prm.tokens = tokens;
  prm.bs = bs; prm.gamma = gamma; prm.V = V; prm.r = r; prm.k = k;
  prm.inv_tau = inv_tau;
  prm.greedy = greedy;
  prm.n_chunks = n_chunks;
  prm.status = status;
  prm.timeout_ns = g_wait_timeout_ns;
  prm.entries = static_cast<float4*>(entries);
  prm.n_slots = grid_size(bs, n_chunks) / ((bs + kBM - 1) / kBM);
  prm.seed = seed;
  prm.step = step;
  *n_slots = prm.n_slots;
  return launch<false>(map_w2, map_u, prm, s);
}

cudaError_t launch_decision_stats_tc(const void* target, const void* U, const void* W1, const void* W2t,
                                     const int32_t* anchor, const int32_t* tokens, const float* lse_d,
                                     const void* rs, const void* dec, int bs, int gamma, int V, int r,
                                     float inv_tau, void* stats, int n_chunks, uint32_t* status,
                                     cudaStream_t s) {
  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap map_w2;
  if (!encode_w2(&map_w2, W2t, V, r)) return cudaErrorInvalidValue;
  Params prm{};
  prm.W1 = static_cast<const __nv_bfloat16*>(W1);
  prm.anchor = anchor;
  prm.tokens = tokens;
  prm.bs = bs; prm.gamma = gamma; prm.V = V; prm.r = r; prm.k = 0;
  prm.inv_tau = inv_tau;
  prm.greedy = 0;
  prm.stats = static_cast<float2*>(stats);
  prm.n_chunks = n_chunks;
  prm.status = status;
  prm.timeout_ns = g_wait_timeout_ns;
  prm.U = static_cast<const __nv_bfloat16*>(U);
  prm.target = static_cast<const __nv_bfloat16*>(target);
  prm.lse_d = lse_d;
  prm.rs = static_cast<const RowStat*>(rs);
  prm.dec = static_cast<const Decision*>(dec);
  return launch<true>(map_w2, map_w2, prm, s);
}

}  // namespace dspark
