// The draft's vocabulary pass on the tensor cores: tcgen05.mma (bf16 in, fp32 accumulate in
// TMEM), operands staged by TMA, fused epilogue.  No [bs, V] logit tensor ever reaches HBM.
//
// DSpark technical summary, "Architecture (drafter)": the Markov head's bias for position k
// is W1[x_{k-1}] W2 (rank r = 256), added to the backbone's base logits U_k over the full
// vocabulary.  Per position this is a GEMM [bs, r] x [r, V] consumed at once by a sampler:
// l = U_k + A_k W2 (A_k = W1[x_{k-1}], or the RNN head's state s_k), reduced to per-request
// partial draws (DraftEntry, common.cuh), which the select step (draft_select.cuh) merges into
// x_k.  x_k is the next position's A row, so the positions run strictly left to right.
//
// One persistent launch runs positions k_first .. k_last (all gamma of them).  With the RNN
// head, the epilogue first computes every request's first state s_1 (one more grid barrier), and
// the group that draws x_k updates that request's recurrent state to s_{k+1} before the next
// position.  Between positions
// the CTAs meet at a grid barrier (a cooperative launch, so that every CTA is resident), run the
// select of the requests assigned to them, and meet again before the next position's A gather.
// Compared with a launch per pass this removes two kernel boundaries per position, and the TMA
// producers run on into the next position's W2t / U tiles while the select runs.
//
// Instruction width: back to back, with operands resident, the tensor core retires an
// M = 128, K = 16 MMA in 64 SM cycles at N = 128 and 128 at N = 256 (its arithmetic rate; two
// issuing warps share it).  In this pass every 64-K stage adds a barrier wait and a commit, so
// wide N = 256 MMAs halve that per-stage overhead per logit: a tile of 128 requests x 256
// vocabulary ids is 16 MMAs (K = 256).
//
// What bounds the pass is how fast W2t reaches shared memory: every position streams all of W2t
// from L2 (where it stays), and a 32 KB stage takes about 2 us to arrive while the U stream loads
// the memory system, so a CTA needs as many bytes in flight as that round trip times the tensor
// core's consumption.  Hence the A operand lives in tensor memory, not shared memory, and the
// freed space holds a W2t ring of one whole tile (so the next tile's operands are in flight
// while this tile's MMAs run) beside a ring of U_k boxes 1.5 tiles deep.
//
// Work decomposition:
//   tile      = 128 requests (TMEM lanes) x 256 vocabulary ids (= four 64-id draft chunks),
//               K = r; the accumulator is TMEM columns 0-255, the A operand columns 256-383
//   CTA       = persistent, one per SM; fixed 128-request M-tile, strided over vocabulary
//               tiles; the gathered A operand (W1[x_{k-1}], or s_k) is written once into tensor
//               memory by the epilogue warps (tcgen05.st)
//   warp 0    = TMA producer of W2t K-stages [256 ids x 64 K] (32 KB, a four-deep ring,
//               evict-last: every position re-reads W2t and it stays in L2)
//   warp 18   = TMA producer of the U_k tile's four 64-id boxes (3-D map over [bs, gamma, V],
//               evict-first; a ring of six 16 KB boxes), on its own so that U never waits
//               behind a W2t stage
//   warp 1    = TMEM owner + single-thread tcgen05.mma issuer, commits to mbarriers; the next
//               tile's MMAs start once both epilogue sets have read the accumulator into
//               registers (a single accumulator: its readout is short next to the tile)
//   warps 2-17 = epilogue, four warp sets of four (one warp per TMEM lane quarter, one request
//               row per thread).  Set s takes columns 64 s .. 64 s + 63 of every tile -- the
//               tile's draft chunk 4c + s -- and the matching 64-id box of U: it adds U_k to its
//               64 accumulator values (adding U_k on the tensor core through an identity operand
//               costs more tensor-pipe time than these adds cost issue slots), forms the chunk's
//               log-mass and Gumbel key and keeps, in registers, the row's running (max,
//               sum-exp) and best key.  Four sets rather than two: the per-element work is a
//               chain of dependent ALU / MUFU operations, and with two warps per scheduler most
//               issue slots went unused.  After a position the sets merge through spare TMEM
//               columns (shared memory is full) and set 0 writes one entry per request, so the
//               select merges one entry per CTA column.
//   select    = the epilogue warps as two groups of eight, one request each (request
//               blockIdx + (2 j + group) * gridDim)
//   warp 19   = the confidence head when the call asks for it: the h terms of the requests
//               blockIdx + j gridDim ahead of time (they need no drafted token), then position
//               k's confidence and survival as soon as x_{k-1} is readable, so that it finishes
//               under the draft's own time
// Every mbarrier and grid-barrier wait is bounded (SM cycle-counter deadline + shared abort flag,
// and a grid-wide abort word); on give-up the kernel records DSPARK_ETIMEOUT, waits (bounded) for
// its own copies / MMAs in flight, frees TMEM and returns.  The grid barrier's words live in the
// workspace's status block; the last CTA to leave zeroes them for the next launch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "confidence.cuh"
#include "draft_select.cuh"
#include "internal.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace dspark {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;                          // ids per tile
static_assert(kBN == 4 * kDraftIds, "a tile is four draft chunks, one per epilogue set");
constexpr int kBK = 64;                           // K per stage: one 128-byte swizzle row
constexpr int kBStages = 4;                       // W2t ring of 32 KB stages: one whole tile
constexpr int kUSlots = 6;                        // U ring of 64-id boxes: 1.5 tiles
constexpr int kEpiSets = 4;                       // warp sets of four warps, one draft chunk each
constexpr int kEpiWarps = 4 * kEpiSets;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kUWarp = 2 + kEpiWarps;             // warp 18: the U producer
constexpr int kConfWarp = 3 + kEpiWarps;          // warp 19: the confidence head (when asked for)
constexpr int kThreads = 32 * (4 + kEpiWarps);
constexpr uint32_t kBStage = kBN * kBK * 2;       // 32 KB: W2t rows [256 x 64 K]
constexpr uint32_t kUBox = kBM * 64 * 2;          // 16 KB: U [128 rows x 64 ids]
constexpr uint32_t kTmemA = kBN;                  // A: columns 256 .. 256 + r / 2 - 1 (bf16 pairs)
constexpr uint32_t kTmemX = kTmemA + 128;         // 384 + 4 s: warp set s's entry, merged by set 0
constexpr uint32_t kTmemCols = 512;               // allocation: a power of two >= 256 + 128
constexpr float kLog2e = 1.4426950408889634f;

struct Barriers {
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t u_full[kUSlots], u_empty[kUSlots];  // U box q = 4 T + s (tile T, set s) in slot q % kUSlots
  uint64_t acc_full, acc_empty;
  uint64_t drain;
  uint64_t a_ready;  // the A operand is in tensor memory (one arrival per epilogue warp)
  uint32_t tmem_base;
  int abort;
  int mma_pending;   // the issuer's MMAs that nobody has waited for (set by the issuing thread)
  int bail;          // the epilogue's shared decision after a grid barrier (1: stop)
  uint32_t tok_pos;  // positions whose x_{k-1} every CTA can read (release / acquire; conf warp)
  SelectScratch sel[2];  // the two select groups' scratch
};

struct Params {
  const __nv_bfloat16* U;
  const __nv_bfloat16* W1;
  const __nv_bfloat16* W2t;
  const __nv_bfloat16* states;  // RNN head: the states s_k [bs, gamma, r] (A rows); else null
  const __nv_bfloat16* Wg;      // RNN head: gate weights [2r, r]; the kernel updates the states
  const float* bg;              // RNN head: gate bias [r]
  const __nv_bfloat16* h;       // confidence head: h [bs, gamma, d], or null (no confidence here)
  const float* wconf;           // [d + r]
  const float* sts_T;           // [gamma]
  float* conf;                  // [bs, gamma] out
  float* surv;                  // [bs, gamma] out
  float* z_logit;               // [bs, gamma] out or null
  float bconf;
  int d;
  const int32_t* anchor;
  int32_t* tokens;
  float* logit_x;
  float* lse;
  int bs, gamma, V, r, k_first, k_last;
  float inv_tau;
  int greedy;
  int n_tiles;      // 256-id vocabulary tiles
  uint32_t* status;
  uint32_t* diag;   // where a wait gave up (note_timeout)
  uint32_t* ctl;    // grid barrier: ctl[0] arrivals, ctl[kCtlAbort] abort, ctl[kCtlExit] exits
  uint64_t timeout_ns;
  float4* entries;  // per (request, slot): DraftEntry
  int n_slots;
  uint64_t seed, step;
};

constexpr int kCtlAbort = 16, kCtlExit = 32;  // words of the grid barrier block (64 bytes apart)

// Dynamic shared memory: W2t ring | U halves | barriers.  The buffer is declared 1024-byte
// aligned (128-byte swizzle atoms).
constexpr size_t kSmemBytes = kBStages * size_t(kBStage) + kUSlots * size_t(kUBox) + sizeof(Barriers);
static_assert(kSmemBytes <= 232448, "dynamic shared memory beyond the 227 KB per-block limit");

// The Gumbel of draft chunk 4c + s (warp set s's chunk of vocabulary tile c), request `req`,
// position k (Philox purpose 1, index = the chunk id): counter group c, word s.  Out of line:
// called in the tile loop before the accumulator wait (when few registers are live), its
// Philox rounds add nothing to the loop's register pressure.
__device__ __noinline__ float chunk_gumbel_call(uint64_t seed, uint64_t step, int req, int k, int c, int s) {
  return gumbel_from_bits(pick_word(philox_group(seed, step, kDraftChunk, uint32_t(req), k, uint32_t(c)), s));
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

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// The epilogue warps' named barrier (id 1, 256 threads); the producers and the MMA warp run on.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

// One thread per CTA: arrive at grid barrier number `idx` (0, 1, ...) of this launch and wait
// (bounded) until every CTA has arrived.  Release / acquire at GPU scope around the counter, so
// what the CTA wrote before the barrier (fenced by the caller's CTA barrier) is visible to the
// CTAs after it.  Returns false on give-up: the deadline, the CTA's own abort flag, or the
// grid-wide abort word (which it then sets, so that the other CTAs stop waiting too).
__device__ __noinline__ bool grid_arrive_wait(uint32_t* ctl, int idx, long long deadline, const volatile int* abort,
                                              uint32_t* status, uint32_t* diag) {
  volatile uint32_t* gabort = ctl + kCtlAbort;
  if (*abort) {
    *gabort = 1u;
    __threadfence();
    return false;
  }
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctl) : "memory");
  const uint32_t target = uint32_t(idx + 1) * gridDim.x;
  while (ld_acquire_gpu(ctl) < target) {
    if (*gabort) return false;
    if (clock64() > deadline) {
      note_timeout(status, diag, 8u, uint32_t(idx) | (ld_acquire_gpu(ctl) << 8));
      *gabort = 1u;
      __threadfence();
      return false;
    }
  }
  return true;
}

// The epilogue's grid barrier: CTA barrier, one thread arrives and waits, CTA barrier.  Returns
// the shared decision to stop (uniform across the epilogue warps: bar->bail is written only
// between the two CTA barriers and read right after the second).
__device__ __forceinline__ bool epi_grid_barrier(Barriers* bar, uint32_t* ctl, int idx, int et, long long deadline,
                                                 uint32_t* status, uint32_t* diag) {
  epi_sync();
  if (et == 0) bar->bail = grid_arrive_wait(ctl, idx, deadline, &bar->abort, status, diag) ? 0 : 1;
  epi_sync();
  return bar->bail != 0;
}

// Release / acquire on a shared-memory word of this CTA (the confidence warp's position count).
__device__ __forceinline__ void st_release_cta(uint32_t* a, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(tc::smem_u32(a)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* a) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(tc::smem_u32(a)) : "memory");
  return v;
}

// The h term of one (request, position), reduced over the warp: its parts in order.
__device__ __noinline__ float conf_h_term(const __nv_bfloat16* hr, const float* w, int d, int parts, int lane) {
  float z = warp_sum(conf_hpart<__nv_bfloat16>(hr, w, d, 0, parts, lane));
  for (int q = 1; q < parts; ++q) z += warp_sum(conf_hpart<__nv_bfloat16>(hr, w, d, q, parts, lane));
  return z;
}

// The confidence head, computed by one warp of each CTA while the draft runs, for the requests
// blockIdx + j gridDim: the logit z = w [h_k ; W1[x_{k-1}]] + b in the confidence kernel's order
// (confidence.cuh), then c = sigmoid(z / T_k) and the survival a_k = a_{k-1} c -- the same bits
// as dspark_confidence.  The h terms need no drafted token: they are computed ahead, position by
// position, whenever the next position to finish is still waiting for its x_{k-1}, so that
// finishing a position is one W1-row term per request.  tok_pos (set by the epilogue after each
// position's tokens are visible grid-wide) counts the positions whose x_{k-1} is readable.
// Returns false if a wait gave up.
template <typename P>
__device__ __noinline__ bool confidence_warp(const P& p, const uint32_t* tok_pos, int npos, long long deadline,
                                             const volatile int* abort, int lane) {
  constexpr int kAhead = 2;  // requests per CTA whose h terms are kept (more are computed in place)
  const int parts = conf_parts(p.gamma);
  float hsum[kAhead][DSPARK_MAX_GAMMA];
  auto h_term = [&](int b, int k) {
    return conf_h_term(p.h + (size_t(b) * p.gamma + k - 1) * p.d, p.wconf, p.d, parts, lane);
  };
  int ahead = 0;  // positions (from the first) whose h terms are in hsum
  for (int pi = 0; pi < npos; ++pi) {
    const int k = p.k_first + pi;
    for (;;) {
      const bool ready = ld_acquire_cta(tok_pos) > uint32_t(pi);
      if (ready && ahead > pi) break;
      if (ahead < npos && (ahead <= pi || !ready)) {  // the h terms of the next position
        const int ka = p.k_first + ahead;
        for (int j = 0, b = blockIdx.x; j < kAhead && b < p.bs; ++j, b += gridDim.x) hsum[j][ahead] = h_term(b, ka);
        ++ahead;
        continue;
      }
      if (*abort) return false;
      if (clock64() > deadline) {
        if (lane == 0) note_timeout(p.status, p.diag, 9u, uint32_t(k));
        return false;
      }
      __nanosleep(256);
    }
    int j = 0;
    for (int b = blockIdx.x; b < p.bs; b += gridDim.x, ++j) {
      const int xp = clamp_token(k == 1 ? p.anchor[b] : p.tokens[size_t(b) * p.gamma + k - 2], p.V);
      uint4 qa[1];
      if (lane * 8 < p.r) load_hgroup<__nv_bfloat16>(p.W1 + size_t(xp) * p.r + lane * 8, qa);
      float z = j < kAhead ? hsum[j][pi] : h_term(b, k);
      z += warp_sum(conf_xpart<__nv_bfloat16>(qa, p.wconf, p.d, p.r, lane));
      z += p.bconf;
      if (lane == 0) {
        const size_t o = size_t(b) * p.gamma + k - 1;
        if (p.z_logit) p.z_logit[o] = z;
        const float c = 1.f / (1.f + expf(-z / p.sts_T[k - 1]));
        const float a = (k == 1 ? 1.f : p.surv[o - 1]) * c;
        p.conf[o] = c;
        p.surv[o] = a;
      }
      __syncwarp();
    }
  }
  return true;
}

// RNN head, the state of position k + 1 of request b from the x_k just drawn, by the 256 threads
// of a select group (gt = thread):
//   g = sigmoid([e ; s_k] Wg + b_g),  e = W1[x_k],  s_{k+1} = g s_k + (1 - g) e,
// in fp32, rounded to bf16 (nearest even).  Warp w of the group takes input rows
// [w 2r / 8, (w + 1) 2r / 8) -- all of e (w < 4) or all of s_k -- and lane l the output columns
// 8l .. 8l + 7 (16-byte loads of each Wg row), sixteen rows in flight at a time; the warps'
// partial sums meet in the group's scratch in warp order, so the summation order is fixed.  s_k
// comes from this kernel (or, for the first position, from the update kernel before it): plain
// loads.
template <typename P, typename GroupSync>
__device__ __forceinline__ void rnn_next_state(const P& p, int b, int k, int gt, float* red, GroupSync group_sync) {
  const int r = p.r, rows = r / 4;  // 2r / 8 input rows per warp
  const int w = gt >> 5, lane = gt & 31;
  // k = 0: the first state, from the anchor and s_0 = 0
  const int x = clamp_token(k == 0 ? p.anchor[b] : p.tokens[size_t(b) * p.gamma + k - 1], p.V);
  const __nv_bfloat16* sk = k == 0 ? nullptr : p.states + (size_t(b) * p.gamma + k - 1) * r;
  const int j0 = w * rows;  // first input row of this warp
  const __nv_bfloat16* in = j0 < r ? p.W1 + size_t(x) * r + j0 : sk + (j0 - r);
  const bool on = lane * 8 < r;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int jb = 0; jb < rows && in != nullptr && !(k == 0 && j0 >= r); jb += 16) {  // rows: a multiple of 16
    uint4 wq[16];
#pragma unroll
    for (int u = 0; u < 16; ++u)
      wq[u] = on ? __ldg(reinterpret_cast<const uint4*>(p.Wg + size_t(j0 + jb + u) * r) + lane)
                 : make_uint4(0u, 0u, 0u, 0u);
    const uint4 iq0 = *reinterpret_cast<const uint4*>(in + jb), iq1 = *reinterpret_cast<const uint4*>(in + jb + 8);
    const float xin[16] = {bf16lo(iq0.x), bf16hi(iq0.x), bf16lo(iq0.y), bf16hi(iq0.y),
                           bf16lo(iq0.z), bf16hi(iq0.z), bf16lo(iq0.w), bf16hi(iq0.w),
                           bf16lo(iq1.x), bf16hi(iq1.x), bf16lo(iq1.y), bf16hi(iq1.y),
                           bf16lo(iq1.z), bf16hi(iq1.z), bf16lo(iq1.w), bf16hi(iq1.w)};
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      acc[0] = fmaf(xin[u], bf16lo(wq[u].x), acc[0]); acc[1] = fmaf(xin[u], bf16hi(wq[u].x), acc[1]);
      acc[2] = fmaf(xin[u], bf16lo(wq[u].y), acc[2]); acc[3] = fmaf(xin[u], bf16hi(wq[u].y), acc[3]);
      acc[4] = fmaf(xin[u], bf16lo(wq[u].z), acc[4]); acc[5] = fmaf(xin[u], bf16hi(wq[u].z), acc[5]);
      acc[6] = fmaf(xin[u], bf16lo(wq[u].w), acc[6]); acc[7] = fmaf(xin[u], bf16hi(wq[u].w), acc[7]);
    }
  }
  for (int ww = 0; ww < 8; ++ww) {  // red[c] = sum over warps 0 .. 7 in order
    if (w == ww && on) {
#pragma unroll
      for (int c = 0; c < 8; ++c) red[lane * 8 + c] = (ww == 0 ? 0.f : red[lane * 8 + c]) + acc[c];
    }
    group_sync();
  }
  if (gt < r) {
    const float g = 1.f / (1.f + expf(-(p.bg[gt] + red[gt])));
    const float ei = __bfloat162float(p.W1[size_t(x) * r + gt]);
    const float si = k == 0 ? 0.f : __bfloat162float(sk[gt]);
    const_cast<__nv_bfloat16*>(p.states)[(size_t(b) * p.gamma + k) * r + gt] =
        __float2bfloat16_rn(g * si + (1.f - g) * ei);
  }
}

// RNN head: the first state s_1 of this CTA's requests (blockIdx + (2 j + group) gridDim), before
// the first position.  Out of line, like the select.
template <typename P>
__device__ __noinline__ void rnn_first_states(const P& p, int et, SelectScratch* sm) {
  const int grp = et >> 8, gt = et & 255;
  auto group_sync = [grp] { asm volatile("bar.sync %0, 256;" ::"r"(2 + grp) : "memory"); };
  for (int b = blockIdx.x + grp * int(gridDim.x); b < p.bs; b += 2 * int(gridDim.x))
    rnn_next_state(p, b, 0, gt, sm->a, group_sync);
}

// The select of position k for this CTA's requests: the epilogue's 512 threads (et) as two
// groups of eight warps, group g taking requests blockIdx + (2 j + g) gridDim.  Out of line: its
// registers are not added to the tile loop's.
template <typename P>
__device__ __noinline__ void select_requests(const P& p, int k, int et, SelectScratch* sm) {
  const int grp = et >> 8, gt = et & 255;
  auto group_sync = [grp] { asm volatile("bar.sync %0, 256;" ::"r"(2 + grp) : "memory"); };
  for (int b = blockIdx.x + grp * int(gridDim.x); b < p.bs; b += 2 * int(gridDim.x)) {
    select_row<__nv_bfloat16, 8>(b, gt, p.entries, p.n_slots, p.U, p.W1, p.W2t, p.states, p.anchor, p.tokens,
                                 p.logit_x, p.lse, p.gamma, p.V, p.r, k, p.inv_tau, p.greedy, p.seed, p.step,
                                 p.status, sm, group_sync, p.states == nullptr && k < p.k_last);
    if (p.Wg && k < p.k_last) {  // the RNN head's next state, from the token just drawn
      group_sync();              // x_k (written by the group's thread 0) is visible to the group
      rnn_next_state(p, b, k, gt, sm->a, group_sync);
    }
  }
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
  uint8_t* sB = smem_raw;                    // kBStages x 32 KB
  uint8_t* sU = sB + kBStages * kBStage;     // kUSlots x 16 KB
  Barriers* bar = reinterpret_cast<Barriers*>(sU + kUSlots * kUBox);
  volatile int* abort_flag = &bar->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bs = p.bs, V = p.V, r = p.r;
  const int npos = p.k_last - p.k_first + 1;
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
    for (int j = 0; j < kUSlots; ++j) {
      tc::mbar_init(tc::smem_u32(&bar->u_full[j]), 1);
      tc::mbar_init(tc::smem_u32(&bar->u_empty[j]), 4);  // the four warps of the box's set
    }
    tc::mbar_init(tc::smem_u32(&bar->acc_full), 1);
    tc::mbar_init(tc::smem_u32(&bar->acc_empty), kEpiWarps);  // every set reads every tile
    tc::mbar_init(tc::smem_u32(&bar->drain), 1);
    tc::mbar_init(tc::smem_u32(&bar->a_ready), kEpiWarps);
    bar->abort = 0;
    bar->mma_pending = 0;
    bar->bail = 0;
    bar->tok_pos = 0u;
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

  if (warp == 0) {
    // ------------------------------------------------------------------ W2t producer
    // W2t does not depend on the previous kernel: the ring fills while it finishes.
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last();
      int bstage = 0, bph = 0;
      int b_issued[kBStages];
      for (int s = 0; s < kBStages; ++s) b_issued[s] = -1;
      bool ok = true;
      uint32_t fail_info = 0;
      for (int T = 0; T < npos * n_tiles && ok; ++T) {  // the same tiles at every position
        const int n0 = (c0 + (T % n_tiles) * cstride) * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->b_empty[bstage]), bph ^ 1, deadline, abort_flag)) {
            ok = false;
            fail_info = uint32_t(T);
            break;
          }
          const uint32_t bfull = tc::smem_u32(&bar->b_full[bstage]);
          tc::mbar_arrive_expect_tx(bfull, kBStage);
          tc::tma_load_2d(tc::smem_u32(sB + bstage * kBStage), &tmap_w2, bfull, kb * kBK, n0, keep);
          b_issued[bstage] = bph;
          if (++bstage == kBStages) { bstage = 0; bph ^= 1; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        note_timeout(p.status, p.diag, 1u, fail_info);
        // wait (bounded) for every copy this thread put in flight before the CTA exits
        const long long dl = tc::deadline_after_ns(200000000ull);
        const volatile int never = 0;
        for (int s = 0; s < kBStages; ++s)
          if (b_issued[s] >= 0) tc::mbar_wait_bounded(tc::smem_u32(&bar->b_full[s]), b_issued[s], dl, &never);
      }
    }
  } else if (warp == kUWarp) {
    // ------------------------------------------------------------------ U producer
    // U_k does not depend on the previous kernel either.  Per tile its four 64-id boxes, box s
    // paced by epilogue set s, through a ring of kUSlots boxes.
    if (lane == 0) {
      const uint64_t stream = tc::policy_evict_first();
      int u_issued[kUSlots];
      for (int j = 0; j < kUSlots; ++j) u_issued[j] = -1;
      bool ok = true;
      uint32_t fail_info = 0;
      for (int T = 0; T < npos * n_tiles && ok; ++T) {  // tile T % n_tiles of position T / n_tiles
        const int n0 = (c0 + (T % n_tiles) * cstride) * kBN;
        const int k = p.k_first + T / n_tiles;
        for (int sb = 0; sb < kEpiSets; ++sb) {
          const int q = kEpiSets * T + sb, j = q % kUSlots, ph = (q / kUSlots) & 1;
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->u_empty[j]), ph ^ 1, deadline, abort_flag)) {
            ok = false;
            fail_info = uint32_t(q);
            break;
          }
          const uint32_t ufull = tc::smem_u32(&bar->u_full[j]);
          tc::mbar_arrive_expect_tx(ufull, kUBox);
          tc::tma_load_3d(tc::smem_u32(sU + j * kUBox), &tmap_u, ufull, n0 + sb * kDraftIds, k - 1, m0, stream);
          u_issued[j] = ph;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        note_timeout(p.status, p.diag, 2u, fail_info);
        const long long dl = tc::deadline_after_ns(200000000ull);
        const volatile int never = 0;
        for (int j = 0; j < kUSlots; ++j)
          if (u_issued[j] >= 0) tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[j]), u_issued[j], dl, &never);
      }
    }
  } else if (warp == kConfWarp) {
    // ------------------------------------------------------------------ confidence head
    if (p.h && !confidence_warp(p, &bar->tok_pos, npos, deadline, abort_flag, lane)) *abort_flag = 1;
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
      int bstage = 0, bph = 0;
      bool ok = true;
      bool issued = false;
      uint32_t fail_site = 0, fail_info = 0;
      for (int T = 0; T < npos * n_tiles && ok; ++T) {
        // each position's A operand is written by the epilogue once it has read the previous
        // position's last accumulator (so every MMA that read the old A has completed)
        if (T % n_tiles == 0 &&
            !tc::mbar_wait_bounded(tc::smem_u32(&bar->a_ready), (T / n_tiles) & 1, deadline, abort_flag)) {
          ok = false;
          fail_site = 3u;
          fail_info = uint32_t(T);
          break;
        }
        if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_empty), (T & 1) ^ 1, deadline, abort_flag)) {
          ok = false;
          fail_site = 4u;
          fail_info = uint32_t(T);
          break;
        }
        tc::tc_fence_after();
        for (int kb = 0; kb < nk; ++kb) {
          if (!tc::mbar_wait_bounded(tc::smem_u32(&bar->b_full[bstage]), bph, deadline, abort_flag)) {
            ok = false;
            fail_site = 5u;
            fail_info = uint32_t(T) | (uint32_t(kb) << 24);
            break;
          }
          tc::tc_fence_after();
          const uint32_t b_addr = tc::smem_u32(sB + bstage * kBStage);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // A: 8 TMEM columns (16 bf16) per K step
            tc::mma_bf16_ts(tmem_base, tmem_base + kTmemA + kb * (kBK / 2) + kk * 8,
                            tc::sdesc_kmajor_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0);
          issued = true;
          tc::mma_commit(tc::smem_u32(&bar->b_empty[bstage]));
          if (++bstage == kBStages) { bstage = 0; bph ^= 1; }
        }
        if (!ok) break;
        tc::mma_commit(tc::smem_u32(&bar->acc_full));
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
  } else {
    // ------------------------------------------------------------------ epilogue
    const int et = tid - 64;          // 0 .. 511
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int m = wq * 32 + lane;     // tile row = TMEM lane
    const int set = (warp - 2) >> 2;  // warp set: columns 64 set .. 64 set + 63 of each tile
    const int grow = m0 + m;
    const float inv_tau = p.inv_tau;
    const float c2 = inv_tau * kLog2e;
    const uint32_t lane_base = tmem_base + (uint32_t(wq * 32) << 16);
    const uint32_t taddr = lane_base + set * kDraftIds;
    const uint8_t* urow = sU + m * 128;  // this row in U slot 0
    // x_0 (the anchors) and the first position's inputs come from earlier kernels: everything
    // above -- barrier set-up, TMEM, the producers' U / W2 prefetch -- overlapped with them
    tc::grid_dependency_wait();
    if (et == 0) st_release_cta(&bar->tok_pos, 1u);  // x_0 (the anchors) are readable
    int T = 0;     // tiles consumed so far, over all positions (accumulator / U ring phases)
    int nbar = 0;  // grid barriers passed so far
    bool stop = false;
    if (p.Wg && p.k_first == 1) {  // RNN head: every request's first state before position 1
      rnn_first_states(p, et, &bar->sel[et >> 8]);
      if (epi_grid_barrier(bar, p.ctl, nbar++, et, deadline, p.status, p.diag)) {
        *abort_flag = 1;
        stop = true;
      }
    }
    for (int pi = 0; pi < npos && !stop; ++pi) {
      const int k = p.k_first + pi;
      {
        // A operand into tensor memory: this row's W1[x_{k-1}] (Markov head) or s_k (RNN head)
        // (a zero row past the batch).  The four warp sets of a lane quarter share the row, set s
        // its K values [s r / 4, (s + 1) r / 4) (r / 8 columns of bf16 pairs), all of its loads
        // issued before its stores (one round trip for the gather).  Every MMA that read the
        // previous position's A has completed: this thread has waited for the accumulator of
        // that position's last tile.
        const bool live = grow < bs;
        const uint4* src = reinterpret_cast<const uint4*>(
            live ? factor_row(p.W1, p.states, p.anchor, p.tokens, grow, k, p.gamma, V, r) : p.W1);
        const int nq = r / 32;  // 16-byte pieces of the set's K range: 2, 4 or 8
        uint4 w[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          w[q] = (live && q < nq) ? src[set * nq + q] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
          if (q < nq) {
            const uint32_t a8[8] = {w[q].x, w[q].y, w[q].z, w[q].w, w[q + 1].x, w[q + 1].y, w[q + 1].z, w[q + 1].w};
            tc::tmem_st8(lane_base + kTmemA + set * (r / 8) + q * 4, a8);
          }
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->a_ready));
      }

      // running (max, sum-exp) in log2 units: run_m = max of l c2, run_s = sum of 2^(l c2 - run_m)
      float run_m = -INFINITY, run_s = 0.f, best_key = -INFINITY;
      int best_c = INT_MAX;
      for (int t = 0; t < n_tiles; ++t, ++T) {
        const int c = c0 + t * cstride;
        const int n0 = c * kBN + set * kDraftIds;  // this set's first id: draft chunk 4c + set
        const int valid = min(kDraftIds, V - n0);  // <= 0: the chunk lies past the vocabulary
        // the chunk's Gumbel (Philox purpose 1) depends on no logit: drawn before the wait for
        // the accumulator, while the tile's MMAs run
        const float g = p.greedy ? 0.f : chunk_gumbel_call(p.seed, p.step, grow, k, c, set);
        bool ok = tc::mbar_wait_bounded(tc::smem_u32(&bar->acc_full), T & 1, deadline, abort_flag);
        // one decision per warp before the .sync.aligned TMEM loads; warps run independently
        // (no named barrier in this loop), so a warp that gives up can hold up no other
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
          *abort_flag = 1;
          if (lane == 0) note_timeout(p.status, p.diag, 6u, uint32_t(T) | (uint32_t(warp) << 24));
          break;
        }
        tc::tc_fence_after();
        float v[kDraftIds];
        tc::tmem_ld32(taddr, reinterpret_cast<uint32_t*>(v));
        tc::tmem_ld32(taddr + 32, reinterpret_cast<uint32_t*>(v + 32));
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->acc_empty));  // the next tile's MMAs may start
        // This set's U box of the tile: box uq, the un-th use of slot uj.  The slot's previous box
        // (uq - kUSlots) belongs to another set, which may still be waiting for it or reading it:
        // a parity wait on u_full alone could then see that older phase's parity and pass early.
        // So first wait until the previous box has been consumed (u_empty, phase un - 1): u_full
        // is then at most one phase behind, and its parity wait is unambiguous.  (The slot's box
        // before that, uq - 2 kUSlots, is this set's own of three tiles back, long consumed.)
        const int uq = kEpiSets * T + set, uj = uq % kUSlots, un = uq / kUSlots;
        ok = (un == 0 || tc::mbar_wait_bounded(tc::smem_u32(&bar->u_empty[uj]), (un - 1) & 1, deadline,
                                               abort_flag)) &&
             tc::mbar_wait_bounded(tc::smem_u32(&bar->u_full[uj]), un & 1, deadline, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
          *abort_flag = 1;
          if (lane == 0) note_timeout(p.status, p.diag, 7u, uint32_t(T) | (uint32_t(warp) << 24));
          break;
        }
        const uint8_t* ub = urow + uj * kUBox;
#pragma unroll
        for (int j = 0; j < kDraftIds / 8; ++j) {  // + U_k: the box's 16-byte groups of this row
          const uint4 q = *reinterpret_cast<const uint4*>(ub + ((j ^ (m & 7)) << 4));
          v[8 * j + 0] += bf16lo(q.x); v[8 * j + 1] += bf16hi(q.x);
          v[8 * j + 2] += bf16lo(q.y); v[8 * j + 3] += bf16hi(q.y);
          v[8 * j + 4] += bf16lo(q.z); v[8 * j + 5] += bf16hi(q.z);
          v[8 * j + 6] += bf16lo(q.w); v[8 * j + 7] += bf16hi(q.w);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bar->u_empty[uj]));

        if (p.greedy) {
          // eight independent (max, first index) chains over offsets q = j (mod 8), merged with
          // the lowest offset on ties; a strict > inside a chain keeps its lowest offset
          float b8[8];
          int i8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) { b8[j] = -INFINITY; i8[j] = INT_MAX; }
#pragma unroll
          for (int q = 0; q < kDraftIds; ++q)
            if (q < valid && v[q] > b8[q & 7]) { b8[q & 7] = v[q]; i8[q & 7] = q; }
          float best = b8[0];
          int bi = i8[0];
#pragma unroll
          for (int j = 1; j < 8; ++j)
            if (b8[j] > best || (b8[j] == best && i8[j] < bi)) { best = b8[j]; bi = i8[j]; }
          // chunks arrive in increasing order: a strict > keeps the lowest index on ties
          if (best > best_key) { best_key = best; best_c = n0 + bi; }
        } else {
          // only the last tile of a vocabulary that is not a multiple of 256 is ragged
          const bool full = valid >= kDraftIds;
          const float mx = full ? row_max<false>(v, valid) : row_max<true>(v, valid);
          if (mx > -INFINITY) {
            const float sc = full ? row_sum_exp2<false>(v, valid, mx * c2, c2)
                                  : row_sum_exp2<true>(v, valid, mx * c2, c2);
            const float key = mx * inv_tau + logf(sc) + g;  // log-mass + Gumbel
            if (key > best_key) { best_key = key; best_c = 4 * c + set; }
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
      // The four sets' entries of a row meet in TMEM columns 384 + 4 s; set 0 merges them in set
      // order and writes the CTA's entry (request grow, slot c0).  Within a tile a lower set's
      // chunk comes first, so on equal keys the lower chunk wins, as the merge's lowest-index
      // rule gives.  (A warp that gave up above still passes every barrier below; the grid
      // barrier then stops the whole epilogue.)
      {
        const uint32_t e4[4] = {__float_as_uint(run_m), __float_as_uint(run_s), __float_as_uint(best_key),
                                uint32_t(best_c)};
        tc::tmem_st4(lane_base + kTmemX + 4 * set, e4);
        tc::tmem_st_wait();
      }
      tc::tc_fence_before();
      epi_sync();
      tc::tc_fence_after();
      if (set == 0) {
        uint32_t x[16];
        tc::tmem_ld16(lane_base + kTmemX, x);
        tc::tmem_ld_wait();
        LsePair l{__uint_as_float(x[0]), __uint_as_float(x[1])};
        ArgMax a{__uint_as_float(x[2]), int(x[3])};
#pragma unroll
        for (int q = 1; q < kEpiSets; ++q) {
          l = lse_merge(l, LsePair{__uint_as_float(x[4 * q]), __uint_as_float(x[4 * q + 1])});
          a = better(a, ArgMax{__uint_as_float(x[4 * q + 2]), int(x[4 * q + 3])});
        }
        if (grow < bs) p.entries[size_t(grow) * p.n_slots + c0] = make_float4(l.m, l.s, a.v, __int_as_float(a.i));
      }
      // every CTA's entries of position k are written: the select of k, two requests at a time
      if (epi_grid_barrier(bar, p.ctl, nbar++, et, deadline, p.status, p.diag)) {
        *abort_flag = 1;
        break;
      }
      select_requests(p, k, et, &bar->sel[et >> 8]);
      // x_k of every request is written before any CTA gathers the next position's A rows
      if (pi + 1 < npos && epi_grid_barrier(bar, p.ctl, nbar++, et, deadline, p.status, p.diag)) {
        *abort_flag = 1;
        break;
      }
      if (et == 0) st_release_cta(&bar->tok_pos, uint32_t(pi + 2));  // x_k is readable grid-wide
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) free_tmem(bar, tmem_base, lane);
  if (tid == 0) {
    // the last CTA out zeroes the grid barrier's words for the next launch (which touches them
    // only after its grid-dependency wait, i.e. after this grid has completed)
    __threadfence();
    if (atomicAdd(p.ctl + kCtlExit, 1u) == gridDim.x - 1) {
      p.ctl[0] = 0u;
      p.ctl[kCtlAbort] = 0u;
      __threadfence();
      p.ctl[kCtlExit] = 0u;
    }
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

cudaError_t launch_draft_tc(const void* U, const void* W1, const void* W2t, const void* states, const void* Wg,
                            const float* bg, const ConfArgs* cf, const int32_t* anchor,
                            int32_t* tokens, float* logit_x, float* lse, int bs, int gamma, int V, int r, int k_first,
                            int k_last, float inv_tau, int greedy, uint64_t seed, uint64_t step, void* entries,
                            uint32_t* ctl, uint32_t* status, uint32_t* diag, cudaStream_t s) {
  if (!tch::encode_fn()) return cudaErrorNotSupported;
  if (k_first < 1 || k_last < k_first || k_last > gamma) return cudaErrorInvalidValue;
  if ((Wg != nullptr) != (states != nullptr && bg != nullptr)) return cudaErrorInvalidValue;
  if (cf && (k_first != 1 || k_last != gamma || !cf->h)) return cudaErrorInvalidValue;
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
  if (cudaError_t e = tch::set_smem_once(draft_tc_kernel, int(kSmemBytes), smem_set, &smem_mu)) return e;
  const int n_tiles = (V + kBN - 1) / kBN;
  const int grid = tch::vocab_grid(bs, n_tiles);  // at most one CTA per SM: all resident together
  Params prm{};
  prm.U = static_cast<const __nv_bfloat16*>(U);
  prm.W1 = static_cast<const __nv_bfloat16*>(W1);
  prm.W2t = static_cast<const __nv_bfloat16*>(W2t);
  prm.states = static_cast<const __nv_bfloat16*>(states);
  prm.Wg = static_cast<const __nv_bfloat16*>(Wg);
  prm.bg = bg;
  if (cf) {
    prm.h = static_cast<const __nv_bfloat16*>(cf->h);
    prm.wconf = cf->w;
    prm.sts_T = cf->sts_T;
    prm.conf = cf->conf;
    prm.surv = cf->surv;
    prm.z_logit = cf->z_logit;
    prm.bconf = cf->b;
    prm.d = cf->d;
  }
  prm.anchor = anchor;
  prm.tokens = tokens;
  prm.logit_x = logit_x;
  prm.lse = lse;
  prm.bs = bs; prm.gamma = gamma; prm.V = V; prm.r = r;
  prm.k_first = k_first; prm.k_last = k_last;
  prm.inv_tau = inv_tau;
  prm.greedy = greedy;
  prm.n_tiles = n_tiles;
  prm.status = status;
  prm.diag = diag;
  prm.ctl = ctl;
  prm.timeout_ns = g_wait_timeout_ns;
  prm.entries = static_cast<float4*>(entries);
  prm.n_slots = grid / ((bs + kBM - 1) / kBM);
  prm.seed = seed;
  prm.step = step;
  // cooperative: the CTAs wait on one another at the grid barriers, so the launch must make them
  // all resident; programmatic dependent launch: set-up and prefetch overlap the previous
  // kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, draft_tc_kernel, map_w2, map_u, prm);
}

}  // namespace dspark
