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
// survival against the prefix outcomes) to a device dspark_obs_stats with integer atomics.
// STS fit, per position k: sts_bins_kernel (grid values x sample slices) accumulates the ECE
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
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kObsThreads) observe_kernel(
    const float* __restrict__ surv, const int32_t* __restrict__ window,
    const int32_t* __restrict__ acc_len, const int32_t* __restrict__ ceiling, int bs, int gamma,
    int n_bins, dspark_obs_stats* __restrict__ st, uint32_t* __restrict__ status) {
  __shared__ unsigned int s_cnt[DSPARK_OBS_MAX_BINS + DSPARK_MAX_GAMMA];
  __shared__ unsigned int s_lab[DSPARK_OBS_MAX_BINS + DSPARK_MAX_GAMMA];
  __shared__ unsigned long long s_sc[DSPARK_OBS_MAX_BINS + DSPARK_MAX_GAMMA];
  __shared__ unsigned int s_hist[3][kHist];
  __shared__ unsigned int s_sum[3];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  constexpr int kSlots = DSPARK_OBS_MAX_BINS + DSPARK_MAX_GAMMA;
  for (int i = tid; i < kSlots; i += kObsThreads) {
    s_cnt[i] = 0u;
    s_lab[i] = 0u;
    s_sc[i] = 0ull;
  }
  if (tid < 3 * kHist) (&s_hist[0][0])[tid] = 0u;
  if (tid < 3) s_sum[tid] = 0u;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  for (int r = tid; r < bs; r += kObsThreads) {
    const int w = window ? window[r] : gamma, acc = acc_len[r], c = ceiling ? ceiling[r] : 0;
    const bool bad = w < 0 || w > gamma || acc < 0 || acc > w ||
                     (ceiling && (c < 0 || c > gamma || acc > c));
    if (bad) {
      s_bad = 1;
      continue;
    }
    atomicAdd(&s_sum[0], unsigned(w));
    atomicAdd(&s_sum[1], unsigned(acc));
    atomicAdd(&s_hist[0][w], 1u);
    atomicAdd(&s_hist[1][acc], 1u);
    if (ceiling) {
      atomicAdd(&s_sum[2], unsigned(c));
      atomicAdd(&s_hist[2][c], 1u);
    }
  }
  __syncthreads();
  if (s_bad) {  // uniform: nothing of this step is recorded
    if (tid == 0) set_status(status, DSPARK_EINVAL);
    return;
  }

  const int n = bs * gamma;
  for (int e = tid; e < n; e += kObsThreads) {
    const int r = e / gamma, k = e - r * gamma + 1;
    const int w = window ? window[r] : gamma, acc = acc_len[r];
    int label;
    bool known = true;
    if (ceiling) {
      label = ceiling[r] >= k;
    } else {
      label = acc >= k;
      known = k <= w || acc < w;
    }
    if (!known) continue;
    const float a = surv[e];
    const unsigned long long fx = fix32(a);
    const int b = score_bin(a, n_bins), p = DSPARK_OBS_MAX_BINS + (k - 1);
    atomicAdd(&s_cnt[b], 1u);
    atomicAdd(&s_cnt[p], 1u);
    if (label) {
      atomicAdd(&s_lab[b], 1u);
      atomicAdd(&s_lab[p], 1u);
    }
    atomicAdd(&s_sc[b], fx);
    atomicAdd(&s_sc[p], fx);
  }
  __syncthreads();

  if (tid < n_bins) {
    add64(&st->bin_count[tid], s_cnt[tid]);
    add64(&st->bin_label[tid], s_lab[tid]);
    add64(&st->bin_score_fx[tid], s_sc[tid]);
  } else if (tid >= DSPARK_OBS_MAX_BINS && tid < DSPARK_OBS_MAX_BINS + gamma) {
    const int k = tid - DSPARK_OBS_MAX_BINS;
    add64(&st->pos_count[k], s_cnt[tid]);
    add64(&st->pos_label[k], s_lab[tid]);
    add64(&st->pos_score_fx[k], s_sc[tid]);
  } else if (tid >= 128 && tid < 128 + 3 * kHist) {
    const int h = (tid - 128) / kHist, i = (tid - 128) % kHist;
    int64_t* dst = h == 0 ? st->window_hist : (h == 1 ? st->accepted_hist : st->ceiling_hist);
    add64(&dst[i], s_hist[h][i]);
  } else if (tid == 256) {
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
// [g][2][b] sum of floor(a 2^32).  Warp-aggregated: lanes of one bin add once through the lane
// with the lowest index (the score split in 16-bit halves so that the warp sums stay exact).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

__global__ void __launch_bounds__(kStsThreads) sts_bins_kernel(
    const float* __restrict__ z, const int32_t* __restrict__ ceiling, int N, int gamma, int k,
    const float* __restrict__ grid, const float* __restrict__ T_fixed, int n_bins,
    unsigned long long* __restrict__ acc) {
  __shared__ unsigned int s_cnt[DSPARK_OBS_MAX_BINS], s_lab[DSPARK_OBS_MAX_BINS];
  __shared__ unsigned long long s_sc[DSPARK_OBS_MAX_BINS];
  __shared__ float s_T[DSPARK_MAX_GAMMA];
  const int tid = threadIdx.x, lane = tid & 31, g = blockIdx.x;
  if (tid < DSPARK_OBS_MAX_BINS) {
    s_cnt[tid] = 0u;
    s_lab[tid] = 0u;
    s_sc[tid] = 0ull;
  }
  if (tid < k) s_T[tid] = T_fixed[tid];
  __syncthreads();
  const float Tg = grid[g];
  const int stride = gridDim.y * kStsThreads;
  for (int base = blockIdx.y * kStsThreads; base < N; base += stride) {  // uniform per warp
    const int i = base + tid;
    const bool live = i < N;
    unsigned int b = 0xFFFFFFFFu, lab = 0u, lo = 0u, hi = 0u;
    if (live) {
      const float* zi = z + size_t(i) * gamma;
      float a = 1.f;
      for (int j = 0; j < k; ++j) a *= sigmoid_f(zi[j] / s_T[j]);
      a *= sigmoid_f(zi[k] / Tg);
      b = static_cast<unsigned int>(score_bin(a, n_bins));
      lab = ceiling[i] >= k + 1 ? 1u : 0u;
      const unsigned long long fx = fix32(a);  // <= 2^32
      lo = static_cast<unsigned int>(fx & 0xFFFFu);
      hi = static_cast<unsigned int>(fx >> 16);
    }
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, b);
    const unsigned n_peer = __popc(peers);
    const unsigned sum_lab = __reduce_add_sync(peers, lab);
    const unsigned sum_lo = __reduce_add_sync(peers, lo);
    const unsigned sum_hi = __reduce_add_sync(peers, hi);
    if (live && lane == __ffs(peers) - 1) {
      atomicAdd(&s_cnt[b], n_peer);
      if (sum_lab) atomicAdd(&s_lab[b], sum_lab);
      atomicAdd(&s_sc[b], (static_cast<unsigned long long>(sum_hi) << 16) + sum_lo);
    }
  }
  __syncthreads();
  if (tid < n_bins) {
    unsigned long long* row = acc + size_t(g) * 3 * n_bins;
    if (s_cnt[tid]) atomicAdd(&row[tid], static_cast<unsigned long long>(s_cnt[tid]));
    if (s_lab[tid]) atomicAdd(&row[n_bins + tid], static_cast<unsigned long long>(s_lab[tid]));
    if (s_sc[tid]) atomicAdd(&row[2 * n_bins + tid], s_sc[tid]);
  }
}

// ECE of every grid value from the integer sums (|passed 2^32 - score sum| exact in int64,
// then fp64 in bin order), and the least one (lowest grid index on ties).
__global__ void __launch_bounds__(kStsThreads) sts_pick_kernel(
    const unsigned long long* __restrict__ acc, int n_grid, int n_bins, int N, int k,
    const float* __restrict__ grid, float* __restrict__ T_out, double* __restrict__ ece_out) {
  __shared__ double s_e[1024];
  for (int g = threadIdx.x; g < n_grid; g += kStsThreads) {
    const unsigned long long* row = acc + size_t(g) * 3 * n_bins;
    double num = 0.0;
    for (int b = 0; b < n_bins; ++b) {
      const long long d = static_cast<long long>(row[n_bins + b] << 32) - static_cast<long long>(row[2 * n_bins + b]);
      num += static_cast<double>(d < 0 ? -d : d);
    }
    s_e[g] = num * 0x1p-32 / static_cast<double>(N);
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
  const int want = 8 * tch::sm_count();  // blocks in flight across the grid values
  int slices = (want + n_grid - 1) / n_grid;
  const int max_slices = (N + kStsThreads - 1) / kStsThreads;
  slices = slices < 1 ? 1 : (slices > max_slices ? max_slices : slices);
  if (slices > 65535) slices = 65535;
  for (int k = 0; k < gamma; ++k) {
    cudaError_t e = cudaMemsetAsync(acc, 0, sts_fit_ws_bytes(n_grid, n_bins), s);
    if (e != cudaSuccess) return e;
    sts_bins_kernel<<<dim3(n_grid, slices), kStsThreads, 0, s>>>(z, ceiling, N, gamma, k, grid, T_out,
                                                                 n_bins, acc);
    sts_pick_kernel<<<1, kStsThreads, 0, s>>>(acc, n_grid, n_bins, N, k, grid, T_out, ece_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
