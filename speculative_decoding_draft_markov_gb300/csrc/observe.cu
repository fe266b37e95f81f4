// Observability and calibration.
//
// DSpark in SGLang, "Observability": compact verification hides the ceiling (what a full-block
// verification would accept); a cap-accept run exposes it while committing what compact
// commits; per-request confidence and calibration metrics (ECE) are reported for analysis.
// "Per-request differentiation under mixed traffic" (Fig. 4): windows per workload, their
// utilisation against the ceiling, the per-step distribution of window lengths.
// DSpark technical summary, "Verification scheduling", STS: the temperatures are fitted left
// to right, one position at a time, by a one-dimensional grid search minimising the ECE of the
// cumulative survival.
//
// observe_kernel: one block adds one step's record (sums, histograms, ECE bins of the
// survival against the prefix outcomes) to a device dspark_obs_stats with integer atomics
// (exact, so the records do not depend on the order of the additions).
// STS fit, per position k: sts_bins_kernel (sample slices x grid chunks) accumulates the ECE
// bins of every grid temperature, sts_pick_kernel takes the grid value of least ECE.
#include "common.cuh"
#include "internal.h"
#include "tc_host.h"

namespace dspark {

constexpr int kObsThreads = 1024;
constexpr int kStsThreads = 256;
constexpr int kHist = DSPARK_MAX_GAMMA + 1;

// floor(a * 2^32) of a score from its bits: a = (m | 2^23) 2^(e - 150), so a 2^32 =
// (m | 2^23) 2^(e - 118).  Exact for 0 <= a <= 1; negatives and subnormals give 0.
__device__ __forceinline__ unsigned long long fix32(float a) {
  const uint32_t bits = __float_as_uint(a);
  if (bits & 0x80000000u) return 0ull;
  const int e = int(bits >> 23);
  if (e == 0) return 0ull;
  const unsigned long long mm = (bits & 0x7FFFFFu) | 0x800000u;
  const int sh = e - 118;
  if (sh >= 0) return mm << (sh < 40 ? sh : 40);
  return sh <= -24 ? 0ull : (mm >> (-sh));
}

// Equal-width bin of a score: floor(a * M) in fp32, clamped to [0, M - 1] (1.0 lands in the
// last bin).
__device__ __forceinline__ int score_bin(float a, int M) {
  const float x = floorf(a * static_cast<float>(M));
  if (!(x >= 0.f)) return 0;
  return x >= static_cast<float>(M - 1) ? M - 1 : static_cast<int>(x);
}

__device__ __forceinline__ void add64(int64_t* dst, unsigned long long v) {
  if (v) atomicAdd(reinterpret_cast<unsigned long long*>(dst), v);
}

// ---------------------------------------------------------------------------------------
// One step's record.  Outcome of a_{r,k}: with a ceiling [c_r >= k] everywhere; without, known
// for k <= l_r ([acc_r >= k]) and, when the window was rejected inside (acc_r < l_r), 0 beyond.
// Every warp owns a private slice of shared sums (slots 0 .. n_bins-1: score bins;
// DSPARK_OBS_MAX_BINS + k - 1: positions) filled with plain 32-bit shared atomics; the score
// is split in 16-bit halves so that the 32-bit sums stay exact (<= 4096 scores per call).  The
// slices are added up in a fixed order at the end.
// ---------------------------------------------------------------------------------------
constexpr int kObsWarps = kObsThreads / 32;
constexpr int kObsSlots = DSPARK_OBS_MAX_BINS + DSPARK_MAX_GAMMA;

__global__ void __launch_bounds__(kObsThreads) observe_kernel(
    const float* __restrict__ surv, const int32_t* __restrict__ window,
    const int32_t* __restrict__ acc_len, const int32_t* __restrict__ ceiling, int bs, int gamma,
    int n_bins, dspark_obs_stats* __restrict__ st, uint32_t* __restrict__ status) {
  __shared__ unsigned s_part[kObsWarps][4][kObsSlots];  // count, passed, score lo, score hi
  __shared__ unsigned s_hist[3][kHist];
  __shared__ unsigned s_sum[3];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = bs * gamma;

  // every global read first (elements tid + j * 1024, j < 4, then this thread's request), so
  // that their latencies overlap each other and the shared-memory set-up
  float a[4];
  int wk[4], acck[4], ck[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + j * kObsThreads;
    a[j] = 0.f;
    wk[j] = acck[j] = ck[j] = 0;
    if (e < n) {
      const int r = e / gamma;
      a[j] = surv[e];
      wk[j] = window ? window[r] : gamma;
      acck[j] = acc_len[r];
      ck[j] = ceiling ? ceiling[r] : 0;
    }
  }
  int w = 0, acc = 0, c = 0;
  if (tid < bs) {
    w = window ? window[tid] : gamma;
    acc = acc_len[tid];
    c = ceiling ? ceiling[tid] : 0;
  }
  for (int i = tid; i < kObsWarps * 4 * kObsSlots; i += kObsThreads) (&s_part[0][0][0])[i] = 0u;
  if (tid < 3 * kHist) (&s_hist[0][0])[tid] = 0u;
  if (tid < 3) s_sum[tid] = 0u;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // per request: checks, sums and histograms (bs <= 256: warps 0..7)
  if (tid < ((bs + 31) & ~31)) {
    bool ok = false;
    if (tid < bs) {
      const bool bad = w < 0 || w > gamma || acc < 0 || acc > w ||
                       (ceiling && (c < 0 || c > gamma || acc > c));
      if (bad) s_bad = 1;
      ok = !bad;
    }
    const unsigned sw = __reduce_add_sync(0xFFFFFFFFu, ok ? unsigned(w) : 0u);
    const unsigned sa = __reduce_add_sync(0xFFFFFFFFu, ok ? unsigned(acc) : 0u);
    const unsigned sc = __reduce_add_sync(0xFFFFFFFFu, ok ? unsigned(c) : 0u);
    if (lane == 0) {
      atomicAdd(&s_sum[0], sw);
      atomicAdd(&s_sum[1], sa);
      atomicAdd(&s_sum[2], sc);
    }
    if (ok) {
      atomicAdd(&s_hist[0][w], 1u);
      atomicAdd(&s_hist[1][acc], 1u);
      if (ceiling) atomicAdd(&s_hist[2][c], 1u);
    }
  }
  __syncthreads();
  if (s_bad) {  // uniform: nothing of this step is recorded
    if (tid == 0) set_status(status, DSPARK_EINVAL);
    return;
  }

  unsigned* cnt = s_part[warp][0];
  unsigned* lab = s_part[warp][1];
  unsigned* lo = s_part[warp][2];
  unsigned* hi = s_part[warp][3];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid + j * kObsThreads;
    if (e >= n) break;
    const int k = e - (e / gamma) * gamma + 1;
    unsigned passed;
    if (ceiling) {
      passed = ck[j] >= k;
    } else {
      passed = acck[j] >= k;
      if (!(k <= wk[j] || acck[j] < wk[j])) continue;  // outcome unknown: the whole window passed
    }
    const unsigned long long fx = fix32(a[j]);
    const unsigned flo = static_cast<unsigned>(fx & 0xFFFFu), fhi = static_cast<unsigned>(fx >> 16);
    const int b = score_bin(a[j], n_bins), p = DSPARK_OBS_MAX_BINS + k - 1;
    atomicAdd(&cnt[b], 1u);
    atomicAdd(&cnt[p], 1u);
    if (passed) {
      atomicAdd(&lab[b], 1u);
      atomicAdd(&lab[p], 1u);
    }
    atomicAdd(&lo[b], flo);
    atomicAdd(&lo[p], flo);
    atomicAdd(&hi[b], fhi);
    atomicAdd(&hi[p], fhi);
  }
  __syncthreads();

  // each (array, slot) summed over the warps in a fixed order by its own thread, the halves of
  // the score recombined through shared memory, then the 64-bit accumulators
  unsigned long long* s_tot = reinterpret_cast<unsigned long long*>(&s_part[0][0][0]);  // reuses warp 0..
  unsigned long long tot = 0;
  const int q = tid / kObsSlots, i = tid - q * kObsSlots;  // array q < 4, slot i
  const bool used = q < 4 && (i < n_bins || (i >= DSPARK_OBS_MAX_BINS && i < DSPARK_OBS_MAX_BINS + gamma));
  if (used)
    for (int wv = 0; wv < kObsWarps; ++wv) tot += s_part[wv][q][i];
  __syncthreads();
  if (used) s_tot[q * kObsSlots + i] = tot;
  __syncthreads();
  if (used && q < 3) {
    unsigned long long v = tot;
    if (q == 2) v = (s_tot[3 * kObsSlots + i] << 16) + tot;  // hi 2^16 + lo
    if (i < n_bins) {
      add64(q == 0 ? &st->bin_count[i] : (q == 1 ? &st->bin_label[i] : &st->bin_score_fx[i]), v);
    } else {
      const int k = i - DSPARK_OBS_MAX_BINS;
      add64(q == 0 ? &st->pos_count[k] : (q == 1 ? &st->pos_label[k] : &st->pos_score_fx[k]), v);
    }
  } else if (tid >= 512 && tid < 512 + 3 * kHist) {
    const int h = (tid - 512) / kHist, hi_i = (tid - 512) % kHist;
    int64_t* dst = h == 0 ? st->window_hist : (h == 1 ? st->accepted_hist : st->ceiling_hist);
    add64(&dst[hi_i], s_hist[h][hi_i]);
  } else if (tid == 600) {
    add64(&st->steps, 1ull);
    add64(&st->requests, static_cast<unsigned long long>(bs));
    add64(&st->sum_window, s_sum[0]);
    add64(&st->sum_accepted, s_sum[1]);
    if (ceiling) {
      add64(&st->ceiling_requests, static_cast<unsigned long long>(bs));
      add64(&st->sum_ceiling, s_sum[2]);
      add64(&st->sum_accepted_ceiling, s_sum[1]);
    }
  }
}

cudaError_t launch_observe(const float* surv, const int32_t* window, const int32_t* acc_len,
                           const int32_t* ceiling, int bs, int gamma, int n_bins, void* stats,
                           uint32_t* status, cudaStream_t s) {
  observe_kernel<<<1, kObsThreads, 0, s>>>(surv, window, acc_len, ceiling, bs, gamma, n_bins,
                                           static_cast<dspark_obs_stats*>(stats), status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// STS fit.  Accumulators per grid value g: [g][0][b] scored count, [g][1][b] passed prefixes,
// [g][2][b] sum of floor(a 2^24) (the fit's internal quantum; the ECE it gives is within
// 2^-24 of the exact one).  Block (x, y) takes samples [x S, x S + S) (S <= 2^15) and the grid
// values of chunk y.  A warp loads 32 samples at a time (prefix product a_{k-1} with the fixed
// temperatures, logit z_k, outcome) and then walks them one by one: the sample is broadcast
// and lane l bins it for grid values l, l + 32, ...; so the lanes of an atomic never share a
// slot.  Shared sums are 32-bit (score in 12-bit halves), flushed to 64-bit at the end.
// ---------------------------------------------------------------------------------------
constexpr int kStsChunkBins = 2048;      // grid values x bins held in shared memory per block
constexpr int kStsMaxSamples = 1 << 15;  // samples per block: the 32-bit shared sums stay exact

// sigmoid(x) with the fast exponential and division intrinsics (relative error ~1e-6: the fit
// only bins the scores)
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

__global__ void __launch_bounds__(kStsThreads) sts_bins_kernel(
    const float* __restrict__ z, const int32_t* __restrict__ ceiling, int N, int gamma, int k,
    const float* __restrict__ grid, int n_grid, const float* __restrict__ T_fixed, int n_bins,
    int per_block, unsigned long long* __restrict__ acc) {
  __shared__ unsigned s_cnt[kStsChunkBins], s_lab[kStsChunkBins], s_lo[kStsChunkBins], s_hi[kStsChunkBins];
  __shared__ float s_invT[DSPARK_MAX_GAMMA];
  __shared__ float s_inv[kStsChunkBins];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_chunk = kStsChunkBins / n_bins;
  const int g0 = blockIdx.y * per_chunk;
  const int ng = min(per_chunk, n_grid - g0);
  for (int i = tid; i < ng * n_bins; i += kStsThreads) s_cnt[i] = s_lab[i] = s_lo[i] = s_hi[i] = 0u;
  for (int i = tid; i < ng; i += kStsThreads) s_inv[i] = 1.f / grid[g0 + i];
  if (tid < k) s_invT[tid] = 1.f / T_fixed[tid];
  __syncthreads();
  const float fM = static_cast<float>(n_bins);
  const int i0 = blockIdx.x * per_block, i1 = min(N, i0 + per_block);
  for (int base = i0 + warp * 32; base < i1; base += kStsThreads) {
    const int i = base + lane;
    float prev = 0.f, zk = 0.f;
    unsigned passed = 0u;
    if (i < i1) {
      const float* zi = z + size_t(i) * gamma;
      prev = 1.f;
      for (int j = 0; j < k; ++j) prev *= sigmoid_fast(zi[j] * s_invT[j]);
      zk = zi[k];
      passed = ceiling[i] >= k + 1 ? 1u : 0u;
    }
    const int cnt_s = min(32, i1 - base);
    for (int s = 0; s < cnt_s; ++s) {  // uniform per warp
      const float p = __shfl_sync(0xFFFFFFFFu, prev, s);
      const float zz = __shfl_sync(0xFFFFFFFFu, zk, s);
      const unsigned ps = __shfl_sync(0xFFFFFFFFu, passed, s);
      for (int g = lane; g < ng; g += 32) {
        const float a = p * sigmoid_fast(zz * s_inv[g]);
        const float xb = floorf(a * fM);
        const int b = xb >= fM - 1.f ? n_bins - 1 : (xb >= 0.f ? static_cast<int>(xb) : 0);
        const unsigned fx = static_cast<unsigned>(a * 16777216.f);  // floor(a 2^24), a in [0, 1]
        const int slot = g * n_bins + b;
        atomicAdd(&s_cnt[slot], 1u);
        if (ps) atomicAdd(&s_lab[slot], 1u);
        atomicAdd(&s_lo[slot], fx & 0xFFFu);
        atomicAdd(&s_hi[slot], fx >> 12);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < ng * n_bins; i += kStsThreads) {
    const int g = g0 + i / n_bins, b = i % n_bins;
    unsigned long long* row = acc + size_t(g) * 3 * n_bins;
    if (s_cnt[i]) atomicAdd(&row[b], static_cast<unsigned long long>(s_cnt[i]));
    if (s_lab[i]) atomicAdd(&row[n_bins + b], static_cast<unsigned long long>(s_lab[i]));
    const unsigned long long sc = (static_cast<unsigned long long>(s_hi[i]) << 12) + s_lo[i];
    if (sc) atomicAdd(&row[2 * n_bins + b], sc);
  }
}

// ECE of every grid value from the integer sums (|passed 2^24 - score sum| exact in int64,
// then fp64 in bin order), and the least one (lowest grid index on ties).
__global__ void __launch_bounds__(kStsThreads) sts_pick_kernel(
    const unsigned long long* __restrict__ acc, int n_grid, int n_bins, int N, int k,
    const float* __restrict__ grid, float* __restrict__ T_out, double* __restrict__ ece_out) {
  __shared__ double s_e[1024];
  for (int g = threadIdx.x; g < n_grid; g += kStsThreads) {
    const unsigned long long* row = acc + size_t(g) * 3 * n_bins;
    double num = 0.0;
    for (int b = 0; b < n_bins; ++b) {
      const long long d = static_cast<long long>(row[n_bins + b] << 24) - static_cast<long long>(row[2 * n_bins + b]);
      num += static_cast<double>(d < 0 ? -d : d);
    }
    s_e[g] = num * 0x1p-24 / static_cast<double>(N);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = 0;
    for (int g = 1; g < n_grid; ++g)
      if (s_e[g] < s_e[best]) best = g;
    T_out[k] = grid[best];
    ece_out[k] = s_e[best];
  }
}

size_t sts_fit_ws_bytes(int n_grid, int n_bins) { return size_t(n_grid) * 3 * n_bins * 8; }

cudaError_t launch_sts_fit(const float* z, const int32_t* ceiling, int N, int gamma, const float* grid,
                           int n_grid, int n_bins, float* T_out, double* ece_out, void* ws,
                           cudaStream_t s) {
  unsigned long long* acc = static_cast<unsigned long long*>(ws);
  const int per_chunk = kStsChunkBins / n_bins;
  const int chunks = (n_grid + per_chunk - 1) / per_chunk;
  // about four blocks per SM in all, at most 2^15 samples per block, whole warps of samples
  const int want = 4 * tch::sm_count();
  long long per = (static_cast<long long>(N) * chunks + want - 1) / want;
  per = ((per + kStsThreads - 1) / kStsThreads) * kStsThreads;
  if (per < kStsThreads) per = kStsThreads;
  if (per > kStsMaxSamples) per = kStsMaxSamples;
  const int slices = static_cast<int>((N + per - 1) / per);
  for (int k = 0; k < gamma; ++k) {
    cudaError_t e = cudaMemsetAsync(acc, 0, sts_fit_ws_bytes(n_grid, n_bins), s);
    if (e != cudaSuccess) return e;
    sts_bins_kernel<<<dim3(slices, chunks), kStsThreads, 0, s>>>(z, ceiling, N, gamma, k, grid, n_grid, T_out,
                                                                 n_bins, static_cast<int>(per), acc);
    sts_pick_kernel<<<1, kStsThreads, 0, s>>>(acc, n_grid, n_bins, N, k, grid, T_out, ece_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
