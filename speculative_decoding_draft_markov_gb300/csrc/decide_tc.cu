// Verify's decision masses on the tensor cores (bf16): for each request's deciding row, per
// 128-id chunk, the residual mass sum max(0, p_t - p_d) and the target mass sum p_t, reduced at
// once to per-CTA partial draws (DecideEntry, common.cuh): mass sums and the best chunk keys
// log(mass) + Gumbel for the first level of the residual / bonus draw.
//
// DSpark technical summary, "Verification": a rejected draft token is replaced by a sample of
// normalise(max(0, p_t - p_d)) at the rejected position, and a fully accepted block takes a
// bonus token from p_t.  p_d there is the draft distribution softmax((U_k + W1[x_{k-1}] W2)/T)
// at the rejected position k, so the pass recomputes those logits with one GEMM
// [bs, r] x [r, V] (rows of requests whose decision is a bonus or absent use a zero A row).
// No [bs, V] tensor reaches HBM: the masses are reduced in the epilogue.
//
// Work decomposition (one persistent CTA per SM, as in the draft pass):
//   tile      = 128 requests (TMEM lanes) x 128 vocabulary ids (one chunk), K = r
//   A operand = W1[x] of each residual request, held in tensor memory (tcgen05.st by the
//               first epilogue warp set; 128 columns), which leaves shared memory to two
//               (U, target) gather stages
//   warp 0    = TMA producer: W2t tiles [128 ids x 64 K] in a ring of K-stages (evict-last)
//   warp 1    = TMEM owner + single-thread tcgen05.mma issuer (A from TMEM, B from smem)
//   warps 2-9 = epilogue, two warp sets of four (one per TMEM lane quarter); set h takes the
//               tiles t = h, h + 2, ...: accumulator buffer h and gather stage h
//   warps 10-13 = cp.async gather of the U rows and target rows of each tile by half tile: a
//               ring of four half-tile slots (two per epilogue set), one warp per slot, each
//               slot refilled as soon as its half is reduced
// Every mbarrier wait is bounded (SM cycle-counter deadline + shared abort flag); on give-up the
// kernel records DSPARK_ETIMEOUT, waits (bounded) for its own copies / MMAs in flight, frees
// TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <type_traits>
#include <mutex>

#include "common.cuh"
#include "f32x2.cuh"
#include "internal.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;                            // ids per tile: one chunk
constexpr int kBK = 64;                             // K per stage: one 128-byte swizzle row
constexpr int kBStages = 5;                         // W2t K-stages (1.25 tiles of K = 256)
constexpr int kSlots = 4;                           // (U, target) half-tile gather slots
constexpr int kAccBufs = 2;
constexpr int kEpiWarps = 8;
constexpr int kGatherWarps = kSlots;                // one per slot
constexpr int kThreads = 32 * (2 + kEpiWarps + kGatherWarps);
constexpr uint32_t kBAtom = kBN * kBK * 2;          // 16 KB: W2t rows [128 x 64 K]
constexpr uint32_t kHalf = kBM * 64 * 2;            // 16 KB: [128 rows x 64 ids] bf16
constexpr uint32_t kSlotBytes = 2 * kHalf;          // U half tile | target half tile
constexpr uint32_t kTmemCols = 512;                 // 2 accumulators x 128 + A (128) -> 512
constexpr uint32_t kTmemA = kAccBufs * kBN;         // first column of A
constexpr float kLog2e = 1.4426950408889634f;

struct Bars {
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t s_full[kSlots], s_empty[kSlots];
  uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  uint64_t drain;
  uint64_t a_ready;  // A is in TMEM (one arrival per warp of epilogue set 0)
  uint32_t tmem_base;
  int abort;
  int mma_pending;   // the issuer's MMAs that nobody has waited for (set by the issuing thread)
  DecideEntry xch[kBM];  // warp set 1's partial draw of each row, merged by set 0 at the end
};

// Per-row facts (one request per tile row).
struct RowMeta {
  int u_row;        // row b * gamma + kdec - 1 of U viewed as [bs * gamma, V] (residual rows; else 0)
  int t_row;        // packed target row pdec (live rows; else 0)
  float a_t;        // lse_t * log2(e)
  float a_d;        // lse_d * log2(e)
  int resid;        // residual row (else bonus, or dead)
  int live;         // the request has a decision
  int kdec;         // position of the decision (Philox counter of its chunk Gumbels)
  int pad;
};

struct Params {
  const __nv_bfloat16* W1;
  const __nv_bfloat16* states;  // RNN head: the draft's states s_k [bs, gamma, r] (A rows); else null
  const __nv_bfloat16* U;
  const __nv_bfloat16* target;
  const int32_t* anchor;
  const int32_t* tokens;
  const float* lse_d;
  const RowStat* rs;
  const Decision* dec;
  int bs, gamma, V, r;
  float inv_tau;
  DecideEntry* entries;  // [bs][n_slots]: one partial draw per request and CTA column
  int n_slots;
  int n_chunks;
  uint64_t seed, step;
  uint32_t* status;
  uint32_t* diag;  // where a wait gave up (note_timeout)
  uint64_t timeout_ns;
};

// Dynamic shared memory: W2t ring | gather slots | row facts | barriers.
constexpr size_t kSmemBytes =
    kBStages * size_t(kBAtom) + kSlots * size_t(kSlotBytes) + kBM * sizeof(RowMeta) + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "dynamic shared memory beyond the 227 KB per-block limit");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// The chunk Gumbel of a decision (Philox purpose 4, index c).  Out of line: inlined into the
// tile loop its rounds raise register pressure there.
__device__ __noinline__ float decide_gumbel_call(uint64_t seed, uint64_t step, int req, int kdec, int c) {
  const uint4 w = philox_group(seed, step, kDecideChunk, uint32_t(req), kdec, uint32_t(c) >> 2);
  return gumbel_from_bits(pick_word(w, c & 3));
}

__device__ __forceinline__ void unpack8(const uint4 q, float* x) {
  x[0] = bf16lo(q.x); x[1] = bf16hi(q.x); x[2] = bf16lo(q.y); x[3] = bf16hi(q.y);
  x[4] = bf16lo(q.z); x[5] = bf16hi(q.z); x[6] = bf16lo(q.w); x[7] = bf16hi(q.w);
}

// Warp 1 at the end of the kernel: free the tensor memory.  An epilogue that gave up has not
// waited for every accumulator, so then the MMAs still in flight are waited for (bounded) first.
// Out of line: it takes no registers from the kernel's loops.
__device__ __noinline__ void free_tmem(Bars* bar, uint32_t tmem_base, int lane) {
  if (lane == 0 && bar->mma_pending && bar->abort) {
    tc::mma_commit(tc::smem_u32(&bar->drain));
    const volatile int never = 0;
    tc::mbar_wait_bounded(tc::smem_u32(&bar->drain), 0, tc::deadline_after_ns(200000000ull), &never);
  }
  __syncwarp();
  tc::tc_fence_after();
  tc::tmem_dealloc(tmem_base, kTmemCols);
}

__global__ void __launch_bounds__(kThreads, 1) decide_tc_kernel(const __grid_constant__ CUtensorMap tmap_w2,
                                                                 const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (tc::smem_u32(smem_raw) & 1023u) {  // the swizzled layouts need 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, DSPARK_EUNSUPPORTED);
    return;
  }
  const int nk = p.r / kBK;
  uint8_t* sB = smem_raw;                          // W2t ring
  uint8_t* sS = sB + kBStages * kBAtom;            // gather slots
  RowMeta* meta = reinterpret_cast<RowMeta*>(sS + kSlots * kSlotBytes);
  Bars* bar = reinterpret_cast<Bars*>(meta + kBM);
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
    for (int s = 0; s < kSlots; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->s_full[s]), 1);   // the slot's gather warp
      tc::mbar_init(tc::smem_u32(&bar->s_empty[s]), 4);  // the epilogue set of the slot
    }
    for (int s = 0; s < kAccBufs; ++s) {
      tc::mbar_init(tc::smem_u32(&bar->acc_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&bar->acc_empty[s]), 4);
    }
    tc::mbar_init(tc::smem_u32(&bar->drain), 1);
    tc::mbar_init(tc::smem_u32(&bar->a_ready), 4);
    bar->abort = 0;
    bar->mma_pending = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w2);
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
  DecideEntry xmine{0.f, 0.f, -INFINITY, -INFINITY, INT_MAX, INT_MAX, 0, 0};  // epilogue set 0's draw

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // W2t does not depend on the previous kernel: the ring fills while the others wait for it.
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last();
      int bstage = 0, bph = 0;
      int b_issued[kBStages];
      for (int s = 0; s < kBStages; ++s) b_issued[s] = -1;
      bool ok = true;
      uint32_t fail_info = 0;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int n0 = (c0 + t * cstride) * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->b_empty[bstage]), bph ^ 1, deadline, abort_flag)) {
            ok = false;
            fail_info = uint32_t(t);
            break;
          }
          const uint32_t bfull = tc::smem_u32(&bar->b_full[bstage]);
          tc::mbar_arrive_expect_tx(bfull, kBAtom);
          tc::tma_load_2d(tc::smem_u32(sB + bstage * kBAtom), &tmap_w2, bfull, kb * kBK, n0, keep);
          b_issued[bstage] = bph;
          if (++bstage == kBStages) { bstage = 0; bph ^= 1; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        note_timeout(p.status, p.diag, 11u, fail_info);
        // wait (bounded) for every copy this thread put in flight before the CTA exits
        const long long dl = tc::deadline_after_ns(200000000ull);
        const volatile int never = 0;
        for (int s = 0; s < kBStages; ++s)
          if (b_issued[s] >= 0) tc::mbar_wait_bounded(tc::smem_u32(&bar->b_full[s]), b_issued[s], dl, &never);
      }
    }
    return;  // takes no part in the named barriers below
  }

  // ---------------------------------------------------------------- everyone else: row facts
  tc::grid_dependency_wait();  // the decisions come from the previous kernel
  tc::grid_launch_dependents();  // the decision select may be scheduled (it waits for this grid)
  constexpr int kRest = kThreads - 32;
  for (int m = tid - 32; m < kBM; m += kRest) {
    RowMeta rm{0, 0, 0.f, 0.f, 0, 0, 0, 0};
    const int grow = m0 + m;
    if (grow < bs) {
      const Decision d = p.dec[grow];
      if (d.kind != kDecNone) {
        rm.live = 1;
        rm.kdec = d.kdec;
        rm.t_row = d.pdec;
        rm.a_t = p.rs[d.pdec].lse * kLog2e;
        if (d.kind == kDecResidual) {
          rm.resid = 1;
          rm.u_row = grow * p.gamma + d.kdec - 1;
          rm.a_d = p.lse_d[(size_t)grow * p.gamma + d.kdec - 1] * kLog2e;
        }
      }
    }
    meta[m] = rm;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kRest) : "memory");

  if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
      int bstage = 0, bph = 0;
      bool ok = tc::mbar_wait_bounded(tc::smem_u32(&bar->a_ready), 0, deadline, abort_flag);
      uint32_t fail_site = 12u, fail_info = 0;
      bool issued = false;
      tc::tc_fence_after();
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int ab = t & 1, ph = (t >> 1) & 1;  // accumulator buffer t % 2 and its phase
        if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_empty[ab]), ph ^ 1, deadline, abort_flag)) {
          ok = false;
          fail_site = 13u;
          fail_info = uint32_t(t);
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + ab * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->b_full[bstage]), bph, deadline, abort_flag)) {
            ok = false;
            fail_site = 14u;
            fail_info = uint32_t(t) | (uint32_t(kb) << 24);
            break;
          }
          tc::tc_fence_after();
          const uint32_t b_addr = tc::smem_u32(sB + bstage * kBAtom);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // A columns: 8 per 16 K values
            tc::mma_bf16_ts(d, tmem_base + kTmemA + kb * (kBK / 2) + kk * 8,
                            tc::sdesc_kmajor_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0);
          issued = true;
          tc::mma_commit(tc::smem_u32(&bar->b_empty[bstage]));
          if (++bstage == kBStages) { bstage = 0; bph ^= 1; }
        }
        if (!ok) break;
        tc::mma_commit(tc::smem_u32(&bar->acc_full[ab]));
      }
      if (!ok) {
        *abort_flag = 1;
        note_timeout(p.status, p.diag, fail_site, fail_info);
        if (issued) {  // wait (bounded) for the MMAs already issued before TMEM is freed
          tc::mma_commit(tc::smem_u32(&bar->drain));
          const volatile int never = 0;
          tc::mbar_wait_bounded(tc::smem_u32(&bar->drain), 0, tc::deadline_after_ns(200000000ull), &never);
        }
      } else {
        bar->mma_pending = issued;  // complete only once the epilogue has consumed every accumulator
      }
    }
  } else if (warp >= 2 + kEpiWarps) {
    // ------------------------------------------------------------------ row gather
    // Warp g fills slot g: half h = g & 1 of the tiles t with t & 1 == g >> 1 -- the U rows of
    // the residual requests and the target rows of the live ones (zero otherwise), 64 ids from
    // column (chunk) * 128 + 64 h.  Only CUDA-core loads read the slots, so the warp waits for
    // its own copies and arrives.
    const int sl = warp - (2 + kEpiWarps), h = sl & 1;
    const int j = lane & 7, rsub = lane >> 3;  // 16-byte group in a 128-byte row, row within 4
    const uint32_t su = tc::smem_u32(sS + sl * kSlotBytes), st = su + kHalf;
    bool ok = true;
    uint32_t fail_info = 0;
    for (int t = sl >> 1, i = 0; t < n_tiles; t += 2, ++i) {
      if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->s_empty[sl]), (i & 1) ^ 1, deadline, abort_flag)) {
        ok = false;
        fail_info = uint32_t(t) | (uint32_t(sl) << 24);
        break;
      }
      const int col = (c0 + t * cstride) * kBN + h * 64 + j * 8;
      const bool in_v = col < V;
#pragma unroll 4
      for (int it = 0; it < kBM / 4; ++it) {
        const int row = it * 4 + rsub;
        const RowMeta rm = meta[row];
        const uint32_t off = row * 128 + ((j ^ (row & 7)) << 4);
        const bool gu = rm.resid && in_v, gt = rm.live && in_v;
        cp_async16(su + off, gu ? p.U + (size_t)rm.u_row * V + col : p.U, gu ? 16u : 0u);
        cp_async16(st + off, gt ? p.target + (size_t)rm.t_row * V + col : p.target, gt ? 16u : 0u);
      }
      // the rows of this slot's next fill (tile t + 2) into L2 while this one completes: one
      // prefetch per 128-byte row segment, lane = row within a group of 32
      if (t + 2 < n_tiles) {
        const int ncol = (c0 + (t + 2) * cstride) * kBN + h * 64;
        if (ncol < V) {
#pragma unroll
          for (int q = 0; q < kBM / 32; ++q) {
            const RowMeta rm = meta[q * 32 + lane];
            if (rm.resid) prefetch_l2(p.U + (size_t)rm.u_row * V + ncol);
            if (rm.live) prefetch_l2(p.target + (size_t)rm.t_row * V + ncol);
          }
        }
      }
      cp_async_wait_all();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->s_full[sl]));
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) note_timeout(p.status, p.diag, 15u, fail_info);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int wq = warp & 3;           // TMEM lane quarter this warp may access
    const int m = wq * 32 + lane;      // tile row = TMEM lane
    const int set = (warp - 2) >> 2;   // tiles t = set, set + 2, ...
    const int grow = m0 + m;
    const float c2 = p.inv_tau * kLog2e;
    const RowMeta rm = meta[m];
    const uint32_t lane_base = tmem_base + (uint32_t(wq * 32) << 16);
    if (set == 0) {
      // A operand into TMEM: this row's factor at the deciding position -- W1[x] (Markov head)
      // or the state s_k (RNN head); zero unless the request's decision is a residual -- 64 K
      // values (32 columns) per store
      const int xp = rm.resid ? 0 : -1;  // -1: a zero row
      const uint4* src = reinterpret_cast<const uint4*>(
          rm.resid ? factor_row(p.W1, p.states, p.anchor, p.tokens, grow, rm.kdec, p.gamma, V, r) : p.W1);
      for (int kb = 0; kb < nk; ++kb) {
        uint32_t a32[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w = xp >= 0 ? src[kb * 8 + q] : make_uint4(0u, 0u, 0u, 0u);
          a32[4 * q + 0] = w.x; a32[4 * q + 1] = w.y; a32[4 * q + 2] = w.z; a32[4 * q + 3] = w.w;
        }
        tc::tmem_st32(lane_base + kTmemA + kb * 32, a32);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->a_ready));
    }
    const float neg_at = -rm.a_t, neg_ad = rm.resid ? -rm.a_d : -INFINITY;
    const uint32_t taddr = lane_base + set * kBN;
    const uint8_t* ub0 = sS + (2 * set) * kSlotBytes + m * 128;  // U row in slot 2 set + h (+ h slots)
    // the row's partial draw over this set's chunks; the chunk Gumbels of the first kGReg tiles
    // are drawn before the loop
    constexpr int kGReg = 8;
    float gk[kGReg];
#pragma unroll
    for (int q = 0; q < kGReg; ++q) {
      const int t = set + 2 * q;
      gk[q] = 0.f;
      if (rm.live && t < n_tiles) {
        const int c = c0 + t * cstride;
        const uint4 w = philox_group(p.seed, p.step, kDecideChunk, uint32_t(grow), rm.kdec, uint32_t(c) >> 2);
        gk[q] = gumbel_from_bits(pick_word(w, c & 3));
      }
    }
    DecideEntry pe{0.f, 0.f, -INFINITY, -INFINITY, INT_MAX, INT_MAX, 0, 0};
    for (int t = set, i = 0; t < n_tiles; t += 2, ++i) {
      const int c = c0 + t * cstride;
      const int valid = min(kBN, V - c * kBN);
      bool ok = tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_full[set]), i & 1, deadline, abort_flag);
      // one decision per warp before the .sync.aligned TMEM loads
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        *abort_flag = 1;
        if (lane == 0) note_timeout(p.status, p.diag, 16u, uint32_t(t) | (uint32_t(warp) << 24));
        break;
      }
      tc::tc_fence_after();
      float R4[4] = {0.f, 0.f, 0.f, 0.f}, P4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {  // 64 columns at a time (one copy of the code for both)
        const int sl = 2 * set + h;
        // one decision per warp before the .sync.aligned TMEM loads
        if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait_bounded(tc::smem_u32(&bar->s_full[sl]), i & 1, deadline,
                                                           abort_flag))) {
          *abort_flag = 1;
          if (lane == 0) note_timeout(p.status, p.diag, 17u, uint32_t(t) | (uint32_t(sl) << 24));
          ok = false;
          break;
        }
        const uint8_t* ub = ub0 + h * kSlotBytes;  // U row of this half
        const uint8_t* tb = ub + kHalf;            // target row of this half
        float l[64];  // W1[x] W2 part of the draft logits (residual rows)
        tc::tmem_ld32(taddr + h * 64, reinterpret_cast<uint32_t*>(l));
        tc::tmem_ld32(taddr + h * 64 + 32, reinterpret_cast<uint32_t*>(l + 32));
        tc::tmem_ld_wait();
        if (h == 1) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->acc_empty[set]));
        }
        if (rm.live) {
          // w = max(0, p_t - p_d); a bonus row's p_d offset is -inf, so p_d = 0 and w = p_t.
          // Full chunks take no per-element bound check (elements past V add +0 instead).  The
          // arithmetic runs two elements at a time (paired fp32 FMA / add, each lane rounded as
          // the scalar operation; element e still goes to sum e & 3, in the same order).
          auto half_sums = [&](auto full) {
            const unsigned long long cc = pack_f32x2(c2, c2), at2 = pack_f32x2(neg_at, neg_at),
                                     ad2 = pack_f32x2(neg_ad, neg_ad), neg1 = pack_f32x2(-1.f, -1.f);
            unsigned long long r01 = pack_f32x2(R4[0], R4[1]), r23 = pack_f32x2(R4[2], R4[3]);
            unsigned long long p01 = pack_f32x2(P4[0], P4[1]), p23 = pack_f32x2(P4[2], P4[3]);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const uint32_t off = (jj ^ (m & 7)) << 4;
              float xu[8], xt[8];
              unpack8(*reinterpret_cast<const uint4*>(ub + off), xu);
              unpack8(*reinterpret_cast<const uint4*>(tb + off), xt);
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                float t0, t1, d0, d1;
                unpack_f32x2(fma_f32x2(pack_f32x2(xt[e], xt[e + 1]), cc, at2), t0, t1);
                const unsigned long long dl =
                    add_f32x2(pack_f32x2(l[8 * jj + e], l[8 * jj + e + 1]), pack_f32x2(xu[e], xu[e + 1]));
                unpack_f32x2(fma_f32x2(dl, cc, ad2), d0, d1);
                const unsigned long long pt = pack_f32x2(tc::ex2_approx(t0), tc::ex2_approx(t1));
                const unsigned long long pd = pack_f32x2(tc::ex2_approx(d0), tc::ex2_approx(d1));
                float w0, w1, q0, q1;
                unpack_f32x2(fma_f32x2(pd, neg1, pt), w0, w1);  // p_t - p_d, one rounding
                unpack_f32x2(pt, q0, q1);
                w0 = fmaxf(0.f, w0);
                w1 = fmaxf(0.f, w1);
                if (!decltype(full)::value) {
                  const int v = h * 64 + 8 * jj + e;
                  if (v >= valid) w0 = q0 = 0.f;
                  if (v + 1 >= valid) w1 = q1 = 0.f;
                }
                if ((e & 3) == 0) {
                  r01 = add_f32x2(r01, pack_f32x2(w0, w1));
                  p01 = add_f32x2(p01, pack_f32x2(q0, q1));
                } else {
                  r23 = add_f32x2(r23, pack_f32x2(w0, w1));
                  p23 = add_f32x2(p23, pack_f32x2(q0, q1));
                }
              }
            }
            unpack_f32x2(r01, R4[0], R4[1]);
            unpack_f32x2(r23, R4[2], R4[3]);
            unpack_f32x2(p01, P4[0], P4[1]);
            unpack_f32x2(p23, P4[2], P4[3]);
          };
          if (valid == kBN) half_sums(std::true_type{});
          else half_sums(std::false_type{});
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->s_empty[sl]));
      }
      if (!ok) break;
      float g;
      if (i < kGReg) {
        g = gk[0];
#pragma unroll
        for (int q = 0; q + 1 < kGReg; ++q) gk[q] = gk[q + 1];
      } else {
        g = rm.live ? decide_gumbel_call(p.seed, p.step, grow, rm.kdec, c) : 0.f;
      }
      const float R = (R4[0] + R4[1]) + (R4[2] + R4[3]), P = (P4[0] + P4[1]) + (P4[2] + P4[3]);
      pe.R += R;
      pe.P += P;
      // chunks arrive in increasing order: a strict > keeps the lowest chunk on ties
      if (R > 0.f) {
        const float kr = logf(R) + g;
        if (kr > pe.kR) { pe.kR = kr; pe.cR = c; }
      }
      if (P > 0.f) {
        const float kp = logf(P) + g;
        if (kp > pe.kP) { pe.kP = kp; pe.cP = c; }
      }
    }
    if (set == 1) bar->xch[m] = pe;
    xmine = pe;
  }

  tc::tc_fence_before();
  asm volatile("bar.sync 1, %0;" ::"n"(kRest) : "memory");
  if (warp == 1) free_tmem(bar, tmem_base, lane);
  if (warp >= 2 && warp < 6) {
    // warp set 0 merges the other set's partial draw of the same row and writes the CTA's
    // entry (request grow, slot c0)
    const int m = (warp & 3) * 32 + lane, grow = m0 + m;
    const DecideEntry o = bar->xch[m];
    DecideEntry e = xmine;
    e.R += o.R;
    e.P += o.P;
    if (o.kR > e.kR || (o.kR == e.kR && o.cR < e.cR)) { e.kR = o.kR; e.cR = o.cR; }
    if (o.kP > e.kP || (o.kP == e.kP && o.cP < e.cP)) { e.kP = o.kP; e.cP = o.cP; }
    if (grow < bs) p.entries[size_t(grow) * p.n_slots + c0] = e;
  }
}

}  // namespace

cudaError_t launch_decision_stats_tc(const void* target, const void* U, const void* W1, const void* W2t,
                                     const void* states, const int32_t* anchor, const int32_t* tokens, const float* lse_d,
                                     const void* rs, const void* dec, int bs, int gamma, int V, int r,
                                     float inv_tau, uint64_t seed, uint64_t step, void* entries,
                                     int n_chunks, int* n_slots, uint32_t* status, cudaStream_t s) {
  if (!tch::encode_fn()) return cudaErrorNotSupported;
  if (r % kBK != 0 || r > 256) return cudaErrorInvalidValue;
  CUtensorMap map_w2;
  if (!tch::encode_bf16_2d(&map_w2, W2t, size_t(V), size_t(r), kBN)) return cudaErrorInvalidValue;
  static bool smem_set[tch::kMaxDevices] = {};
  static std::mutex smem_mu;
  if (cudaError_t e = tch::set_smem_once(decide_tc_kernel, int(kSmemBytes), smem_set, &smem_mu)) return e;
  Params prm{};
  prm.W1 = static_cast<const __nv_bfloat16*>(W1);
  prm.states = static_cast<const __nv_bfloat16*>(states);
  prm.U = static_cast<const __nv_bfloat16*>(U);
  prm.target = static_cast<const __nv_bfloat16*>(target);
  prm.anchor = anchor;
  prm.tokens = tokens;
  prm.lse_d = lse_d;
  prm.rs = static_cast<const RowStat*>(rs);
  prm.dec = static_cast<const Decision*>(dec);
  prm.bs = bs; prm.gamma = gamma; prm.V = V; prm.r = r;
  prm.inv_tau = inv_tau;
  prm.entries = static_cast<DecideEntry*>(entries);
  prm.n_chunks = n_chunks;
  prm.seed = seed;
  prm.step = step;
  prm.status = status;
  prm.diag = status ? status + 4 : nullptr;  // the workspace status block's words 4 .. 6
  prm.timeout_ns = g_wait_timeout_ns;
  const int grid = tch::vocab_grid(bs, n_chunks);
  prm.n_slots = grid / ((bs + kBM - 1) / kBM);
  *n_slots = prm.n_slots;
  // programmatic dependent launch: barrier set-up, TMEM and the W2t ring overlap the previous
  // kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decide_tc_kernel, map_w2, prm);
}

}  // namespace dspark
