// C ABI of libdspark: host-side argument checks, workspace handling and kernel launches.
// Every entry point validates before launching anything; nothing here allocates memory.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "internal.h"

using namespace dspark;

namespace {

inline bool al(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ECUDA; }

inline bool valid_dtype(int dt) { return dt == DSPARK_F32 || dt == DSPARK_BF16; }

// Sizes shared by the draft, confidence and verify calls.
int check_core(int bs, int gamma, int V, int r) {
  if (bs < 1 || gamma < 1 || V < 8 || r < 1) return DSPARK_EINVAL;
  if (V % 8 != 0) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA || V >= (1 << 24)) return DSPARK_EUNSUPPORTED;
  if (!(r == 32 || r == 64 || r == 128 || r == 256)) return DSPARK_EUNSUPPORTED;
  return DSPARK_OK;
}

int check_ws(const void* ws, size_t ws_bytes, int bs, int gamma, int V) {
  if (!ws || !al(ws, 256)) return DSPARK_EWORKSPACE;
  if (ws_bytes < ws_layout(bs, gamma, V).total) return DSPARK_EWORKSPACE;
  return DSPARK_OK;
}

}  // namespace

extern "C" {

const char* dspark_status_string(int status) {
  switch (status) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_EINVAL: return "DSPARK_EINVAL: invalid argument or data";
    case DSPARK_EUNSUPPORTED: return "DSPARK_EUNSUPPORTED: outside the supported sizes or types";
    case DSPARK_ECUDA: return "DSPARK_ECUDA: CUDA runtime or launch failure";
    case DSPARK_ETIMEOUT: return "DSPARK_ETIMEOUT: a device-side wait timed out";
    case DSPARK_EWORKSPACE: return "DSPARK_EWORKSPACE: workspace missing, misaligned or too small";
    default: return "DSPARK_UNKNOWN";
  }
}

size_t dspark_workspace_bytes(int bs, int gamma, int V) {
  if (bs < 1 || gamma < 1 || V < 8 || bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA || V >= (1 << 24))
    return 0;
  return ws_layout(bs, gamma, V).total;
}

int dspark_workspace_init(void* ws, size_t ws_bytes, dspark_stream_t stream) {
  if (!ws || ws_bytes < 256 || !al(ws, 256)) return DSPARK_EWORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_read_device_status(void* ws, dspark_stream_t stream) {
  if (!ws || !al(ws, 256)) return DSPARK_EWORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ECUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DSPARK_ECUDA;
  if (word != 0 && cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return DSPARK_ECUDA;
  return static_cast<int>(word);
}

uint64_t dspark_set_wait_timeout_ns(uint64_t ns) {
  const uint64_t old = g_wait_timeout_ns;
  g_wait_timeout_ns = ns;
  return old;
}

int dspark_copy_packed_rows_async(void* packed, const void* rows, size_t row_bytes, int bs, int rows_per_req,
                                  const int32_t* cu, dspark_stream_t stream) {
  if (!packed || !rows || !cu || row_bytes < 1 || rows_per_req < 1 || bs < 1) return DSPARK_EINVAL;
  for (int r = 0; r < bs; ++r) {  // validate everything before the first copy is enqueued
    const int n = cu[r + 1] - cu[r];
    if (cu[r] < 0 || n < 0 || n > rows_per_req) return DSPARK_EINVAL;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* dst = static_cast<char*>(packed);
  const char* src = static_cast<const char*>(rows);
  const size_t spitch = size_t(rows_per_req) * row_bytes;
  // consecutive requests with the same row count n are one strided copy: their packed rows are
  // contiguous (n rows each), their host rows sit rows_per_req rows apart
  for (int r = 0; r < bs;) {
    const int n = cu[r + 1] - cu[r];
    int e = r + 1;
    while (e < bs && cu[e + 1] - cu[e] == n) ++e;
    if (n > 0) {
      const size_t width = size_t(n) * row_bytes;
      const cudaError_t ce =
          (e - r == 1) ? cudaMemcpyAsync(dst + size_t(cu[r]) * row_bytes, src + size_t(r) * spitch, width,
                                         cudaMemcpyHostToDevice, s)
                       : cudaMemcpy2DAsync(dst + size_t(cu[r]) * row_bytes, width, src + size_t(r) * spitch, spitch,
                                           width, size_t(e - r), cudaMemcpyHostToDevice, s);
      if (ce != cudaSuccess) return DSPARK_ECUDA;
    }
    r = e;
  }
  return DSPARK_OK;
}

int dspark_build_sps(const double* T_raw, int m_max, const int32_t* tiers, int n_tiers,
                     double* sps_out) {
  if (!T_raw || !sps_out || m_max < 0 || n_tiers < 0 || (n_tiers > 0 && !tiers)) return DSPARK_EINVAL;
  for (int i = 0; i < n_tiers; ++i)
    if (tiers[i] <= 0 || (i > 0 && tiers[i] <= tiers[i - 1])) return DSPARK_EINVAL;
  for (int M = 0; M <= m_max; ++M)
    if (!(T_raw[M] > 0.0) || !std::isfinite(T_raw[M])) return DSPARK_EINVAL;
  // running maximum of the profiled curve, then the tier staircase
  double run = 0.0;
  int ti = 0;
  for (int M = 0; M <= m_max; ++M) {
    run = (M == 0 || T_raw[M] > run) ? T_raw[M] : run;
    sps_out[M] = run;  // T_mono[M] (replaced below)
  }
  for (int M = 0; M <= m_max; ++M) {
    int tier = M;
    if (n_tiers > 0) {
      while (ti < n_tiers && tiers[ti] < M) ++ti;
      tier = (ti < n_tiers) ? tiers[ti] : -1;
    }
    // sps_out[t] still holds T_mono for t >= M: tier >= M
    sps_out[M] = (tier < 0 || tier > m_max) ? 0.0 : 1.0 / sps_out[tier];
  }
  return DSPARK_OK;
}

}  // extern "C"

namespace {

// The gamma positions of a block draft, left to right: per position the RNN head's state update
// (states non-null), the vocabulary pass (tensor cores or CUDA cores) and the select.  The
// tensor-core pass runs every position in one launch, with the selects and, for the RNN head,
// the state updates after the first inside it.
int draft_positions(int dtype, const void* U, const void* W1, const void* W2t, const void* Wg, const float* bg,
                    void* states, const int32_t* anchor, int bs, int gamma, int V, int r, float temperature,
                    uint64_t seed, uint64_t step, int32_t* tokens, float* logit_x, float* lse, void* ws,
                    cudaStream_t s, const ConfArgs* cf = nullptr) {
  const WsLayout L = ws_layout(bs, gamma, V);
  char* w = static_cast<char*>(ws);
  void* stats = w + L.stats;
  uint32_t* status = reinterpret_cast<uint32_t*>(w + L.status);
  const int greedy = temperature == 0.f;
  const float inv_tau = greedy ? 1.f : static_cast<float>(1.0 / static_cast<double>(temperature));
  const bool tc = draft_tc_supported(dtype, bs, V, r);
  uint32_t* ctl = reinterpret_cast<uint32_t*>(w + L.status + 64);
  uint32_t* diag = reinterpret_cast<uint32_t*>(w + L.status + 16);
  if (tc)  // every position in one persistent launch, the RNN head's state updates inside it
    return launch_draft_tc(U, W1, W2t, states, states ? Wg : nullptr, states ? bg : nullptr, cf, anchor, tokens, logit_x,
                           lse, bs, gamma, V, r, 1, gamma, inv_tau, greedy, seed, step, stats, ctl, status, diag,
                           s) == cudaSuccess
               ? DSPARK_OK
               : DSPARK_ECUDA;
  for (int k = 1; k <= gamma; ++k) {
    if (states && launch_rnn_state(dtype, W1, Wg, bg, anchor, tokens, states, bs, gamma, V, r, k, s) != cudaSuccess)
      return DSPARK_ECUDA;
    const int n_slots = n_draft_chunks(V);  // the CUDA-core pass: one slot per draft chunk
    cudaError_t e = launch_draft_stats_simt(dtype, U, W1, W2t, states, anchor, tokens, bs, gamma, V, r, k, inv_tau,
                                            greedy, seed, step, stats, n_slots, s);
    if (e == cudaSuccess)
      e = launch_draft_select(dtype, stats, n_slots, U, W1, W2t, states, anchor, tokens, logit_x, lse, bs, gamma, V,
                              r, k, inv_tau, greedy, seed, step, status, s);
    if (e != cudaSuccess) return DSPARK_ECUDA;
  }
  if (cf && launch_confidence(dtype, cf->h, W1, anchor, tokens, cf->w, cf->b, cf->sts_T, bs, gamma, cf->d, r, V,
                              cf->conf, cf->surv, cf->z_logit, s) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

int check_draft_args(const void* U, const void* W1, const void* W2t, int dtype, const int32_t* anchor, int bs,
                     int gamma, int V, int r, float temperature, const int32_t* tokens, const float* logit_x,
                     const float* lse) {
  if (!U || !W1 || !W2t || !anchor || !tokens || !logit_x || !lse) return DSPARK_EINVAL;
  if (!valid_dtype(dtype) || !std::isfinite(temperature) || temperature < 0.f) return DSPARK_EINVAL;
  if (int e = check_core(bs, gamma, V, r)) return e;
  if (!al(U, 16) || !al(W1, 16) || !al(W2t, 16) || !al(anchor, 4) || !al(tokens, 4) ||
      !al(logit_x, 4) || !al(lse, 4))
    return DSPARK_EINVAL;
  return DSPARK_OK;
}

}  // namespace

extern "C" {

int dspark_draft_block(const void* U, const void* W1, const void* W2t, int dtype,
                       const int32_t* anchor, int bs, int gamma, int V, int r, float temperature,
                       uint64_t seed, uint64_t step, int32_t* tokens, float* logit_x, float* lse,
                       void* ws, size_t ws_bytes, dspark_stream_t stream) {
  if (int e = check_draft_args(U, W1, W2t, dtype, anchor, bs, gamma, V, r, temperature, tokens, logit_x, lse))
    return e;
  if (int e = check_ws(ws, ws_bytes, bs, gamma, V)) return e;
  return draft_positions(dtype, U, W1, W2t, nullptr, nullptr, nullptr, anchor, bs, gamma, V, r, temperature, seed,
                         step, tokens, logit_x, lse, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dspark_draft_confidence_block(const void* U, const void* W1, const void* W2t, int dtype, const int32_t* anchor,
                                  int bs, int gamma, int V, int r, float temperature, uint64_t seed, uint64_t step,
                                  int32_t* tokens, float* logit_x, float* lse, const void* h, int d, const float* w,
                                  float b, const float* sts_T, float* conf, float* surv, float* z_logit, void* ws,
                                  size_t ws_bytes, dspark_stream_t stream) {
  if (int e = check_draft_args(U, W1, W2t, dtype, anchor, bs, gamma, V, r, temperature, tokens, logit_x, lse))
    return e;
  if (!h || !w || !sts_T || !conf || !surv || !std::isfinite(b)) return DSPARK_EINVAL;
  if (d < 8 || d % 8 != 0) return DSPARK_EINVAL;
  if (d > 65536) return DSPARK_EUNSUPPORTED;
  if (!al(h, 16) || !al(w, 16) || !al(sts_T, 4) || !al(conf, 4) || !al(surv, 4) || !al(z_logit, 4))
    return DSPARK_EINVAL;
  if (int e = check_ws(ws, ws_bytes, bs, gamma, V)) return e;
  const ConfArgs cf{h, w, b, sts_T, d, conf, surv, z_logit};
  return draft_positions(dtype, U, W1, W2t, nullptr, nullptr, nullptr, anchor, bs, gamma, V, r, temperature, seed,
                         step, tokens, logit_x, lse, ws, reinterpret_cast<cudaStream_t>(stream), &cf);
}

int dspark_draft_block_rnn(const void* U, const void* W1, const void* W2t, const void* Wg, const float* bg,
                           int dtype, const int32_t* anchor, int bs, int gamma, int V, int r, float temperature,
                           uint64_t seed, uint64_t step, int32_t* tokens, float* logit_x, float* lse,
                           void* states, void* ws, size_t ws_bytes, dspark_stream_t stream) {
  if (int e = check_draft_args(U, W1, W2t, dtype, anchor, bs, gamma, V, r, temperature, tokens, logit_x, lse))
    return e;
  if (!Wg || !bg || !states || !al(Wg, 16) || !al(bg, 16) || !al(states, 16)) return DSPARK_EINVAL;
  if (int e = check_ws(ws, ws_bytes, bs, gamma, V)) return e;
  return draft_positions(dtype, U, W1, W2t, Wg, bg, states, anchor, bs, gamma, V, r, temperature, seed, step,
                         tokens, logit_x, lse, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dspark_confidence(const void* h, const void* W1, int dtype, const int32_t* anchor,
                      const int32_t* tokens, const float* w, float b, const float* sts_T, int bs,
                      int gamma, int d, int r, int V, float* conf, float* surv, float* z_logit,
                      dspark_stream_t stream) {
  if (!h || !W1 || !anchor || !tokens || !w || !sts_T || !conf || !surv) return DSPARK_EINVAL;
  if (!valid_dtype(dtype) || !std::isfinite(b)) return DSPARK_EINVAL;
  if (int e = check_core(bs, gamma, V, r)) return e;
  if (d < 8 || d % 8 != 0) return DSPARK_EINVAL;
  if (d > 65536) return DSPARK_EUNSUPPORTED;
  if (!al(h, 16) || !al(W1, 16) || !al(w, 16) || !al(anchor, 4) || !al(tokens, 4) ||
      !al(sts_T, 4) || !al(conf, 4) || !al(surv, 4) || !al(z_logit, 4))
    return DSPARK_EINVAL;
  return cuda_status(launch_confidence(dtype, h, W1, anchor, tokens, w, b, sts_T, bs, gamma, d, r, V,
                                       conf, surv, z_logit, reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_schedule(const float* surv, int bs, int gamma, const double* sps, int m_max, int mode,
                    int32_t* window, int32_t* K_out, double* theta_out, void* ws, size_t ws_bytes,
                    dspark_stream_t stream) {
  if (!surv || !sps || !window || !K_out || !theta_out) return DSPARK_EINVAL;
  if (bs < 1 || gamma < 1 || m_max < bs) return DSPARK_EINVAL;
  if (mode != DSPARK_SCHED_EARLY_STOP && mode != DSPARK_SCHED_GLOBAL_ARGMAX) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA || bs * gamma > 4096) return DSPARK_EUNSUPPORTED;
  if (!al(surv, 4) || !al(sps, 8) || !al(window, 4) || !al(K_out, 4) || !al(theta_out, 8))
    return DSPARK_EINVAL;
  if (!ws || !al(ws, 256) || ws_bytes < 256) return DSPARK_EWORKSPACE;
  return cuda_status(launch_schedule(surv, bs, gamma, sps, m_max, mode, window, K_out, theta_out,
                                     static_cast<uint32_t*>(ws), reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_schedule_zos_select(const float* surv, int bs, int gamma, const double* sps, int m_max,
                               const int32_t* budget_ring, uint64_t step, int32_t* window,
                               int32_t* K_out, void* ws, size_t ws_bytes, dspark_stream_t stream) {
  if (!surv || !sps || !budget_ring || !window || !K_out) return DSPARK_EINVAL;
  if (bs < 1 || gamma < 1 || m_max < bs) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA || bs * gamma > 4096) return DSPARK_EUNSUPPORTED;
  if (!al(surv, 4) || !al(sps, 8) || !al(budget_ring, 4) || !al(window, 4) || !al(K_out, 4))
    return DSPARK_EINVAL;
  if (!ws || !al(ws, 256) || ws_bytes < 256) return DSPARK_EWORKSPACE;
  return cuda_status(launch_zos_select(surv, bs, gamma, sps, m_max, budget_ring, step, window, K_out,
                                       static_cast<uint32_t*>(ws), reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_schedule_zos_budget(const float* surv, int bs, int gamma, const double* sps, int m_max,
                               int32_t* budget_ring, uint64_t step, void* ws, size_t ws_bytes,
                               dspark_stream_t stream) {
  if (!surv || !sps || !budget_ring) return DSPARK_EINVAL;
  if (bs < 1 || gamma < 1 || m_max < bs) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA || bs * gamma > 4096) return DSPARK_EUNSUPPORTED;
  if (!al(surv, 4) || !al(sps, 8) || !al(budget_ring, 4)) return DSPARK_EINVAL;
  if (!ws || !al(ws, 256) || ws_bytes < 256) return DSPARK_EWORKSPACE;
  return cuda_status(launch_zos_budget(surv, bs, gamma, sps, m_max, budget_ring, step,
                                       static_cast<uint32_t*>(ws), reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_pack(const int32_t* window, const int32_t* anchor, const int32_t* tokens, int bs,
                int gamma, const int32_t* tiers, int n_tiers, int cap, int32_t* cu_seqlens,
                int32_t* ids, int32_t* req, int32_t* pos, int32_t* padded_total, void* ws,
                size_t ws_bytes, dspark_stream_t stream) {
  if (!anchor || !tokens || !cu_seqlens || !ids || !req || !pos || !padded_total) return DSPARK_EINVAL;
  if (n_tiers < 0 || (n_tiers > 0 && !tiers) || cap < 1) return DSPARK_EINVAL;
  if (bs < 1 || gamma < 1) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA) return DSPARK_EUNSUPPORTED;
  if (!ws || !al(ws, 256) || ws_bytes < 256) return DSPARK_EWORKSPACE;
  return cuda_status(launch_pack(window, anchor, tokens, bs, gamma, tiers, n_tiers, cap, cu_seqlens,
                                 ids, req, pos, padded_total, static_cast<uint32_t*>(ws),
                                 reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_schedule_pack(const float* surv, int bs, int gamma, const double* sps, int m_max, int mode,
                         int32_t* window, int32_t* K_out, double* theta_out, const int32_t* anchor,
                         const int32_t* tokens, const int32_t* tiers, int n_tiers, int cap, int32_t* cu_seqlens,
                         int32_t* ids, int32_t* req, int32_t* pos, int32_t* padded_total, void* ws,
                         size_t ws_bytes, dspark_stream_t stream) {
  // the argument checks of dspark_schedule and of dspark_pack
  if (!surv || !sps || !window || !K_out || !theta_out) return DSPARK_EINVAL;
  if (bs < 1 || gamma < 1 || m_max < bs) return DSPARK_EINVAL;
  if (mode != DSPARK_SCHED_EARLY_STOP && mode != DSPARK_SCHED_GLOBAL_ARGMAX) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA || bs * gamma > 4096) return DSPARK_EUNSUPPORTED;
  if (!al(surv, 4) || !al(sps, 8) || !al(window, 4) || !al(K_out, 4) || !al(theta_out, 8))
    return DSPARK_EINVAL;
  if (!anchor || !tokens || !cu_seqlens || !ids || !req || !pos || !padded_total) return DSPARK_EINVAL;
  if (n_tiers < 0 || (n_tiers > 0 && !tiers) || cap < 1) return DSPARK_EINVAL;
  if (!ws || !al(ws, 256) || ws_bytes < 256) return DSPARK_EWORKSPACE;
  return cuda_status(launch_schedule_pack(surv, bs, gamma, sps, m_max, mode, window, K_out, theta_out, anchor,
                                          tokens, tiers, n_tiers, cap, cu_seqlens, ids, req, pos, padded_total,
                                          static_cast<uint32_t*>(ws), reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_verify(const void* target, int dtype, const int32_t* cu_seqlens, const int32_t* window,
                  int mode, int bs, int gamma, int V, const int32_t* anchor, const int32_t* tokens,
                  const float* logit_x, const float* lse, const void* draft_logits, const void* draft_states,
                  const void* U, const void* W1, const void* W2t, int r, float temperature, uint64_t seed,
                  uint64_t step, int32_t* out_tokens, int32_t* acc_len, int32_t* ceiling, void* ws,
                  size_t ws_bytes, dspark_stream_t stream) {
  if (!target || !cu_seqlens || !anchor || !tokens || !logit_x || !lse || !out_tokens || !acc_len)
    return DSPARK_EINVAL;
  if (!draft_logits && (!U || !W1 || !W2t)) return DSPARK_EINVAL;  // p_d needs one source
  if (draft_logits) {  // U, W1, W2t, draft_states and r unused
    if (!al(draft_logits, 16)) return DSPARK_EINVAL;
    U = W1 = W2t = draft_states = nullptr;
    r = 32;
  }
  if (draft_states && !al(draft_states, 16)) return DSPARK_EINVAL;
  if (mode != DSPARK_STATIC && mode != DSPARK_COMPACT && mode != DSPARK_CAP_ACCEPT) return DSPARK_EINVAL;
  if (mode != DSPARK_STATIC && !window) return DSPARK_EINVAL;
  if (mode == DSPARK_CAP_ACCEPT && !ceiling) return DSPARK_EINVAL;
  if (!valid_dtype(dtype) || !std::isfinite(temperature) || temperature < 0.f) return DSPARK_EINVAL;
  if (int e = check_core(bs, gamma, V, r)) return e;
  if (!al(target, 16) || (U && !al(U, 16)) || (W1 && !al(W1, 16)) || (W2t && !al(W2t, 16))) return DSPARK_EINVAL;
  if (int e = check_ws(ws, ws_bytes, bs, gamma, V)) return e;
  const int greedy = temperature == 0.f;
  const float inv_tau = greedy ? 1.f : static_cast<float>(1.0 / static_cast<double>(temperature));
  return cuda_status(launch_verify(dtype, target, cu_seqlens, window, mode, bs, gamma, V, anchor,
                                   tokens, logit_x, lse, draft_logits, U, W1, W2t, draft_states, r, inv_tau, greedy,
                                   seed, step, out_tokens, acc_len, ceiling, ws,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_observe(const float* surv, const int32_t* window, const int32_t* acc_len,
                   const int32_t* ceiling, int bs, int gamma, int n_bins, dspark_obs_stats* stats,
                   void* ws, size_t ws_bytes, dspark_stream_t stream) {
  if (!surv || !acc_len || !stats) return DSPARK_EINVAL;
  if (bs < 1 || gamma < 1 || n_bins < 1 || n_bins > DSPARK_OBS_MAX_BINS) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA) return DSPARK_EUNSUPPORTED;
  if (!al(surv, 4) || !al(window, 4) || !al(acc_len, 4) || !al(ceiling, 4) || !al(stats, 8))
    return DSPARK_EINVAL;
  if (!ws || !al(ws, 256) || ws_bytes < 256) return DSPARK_EWORKSPACE;
  return cuda_status(launch_observe(surv, window, acc_len, ceiling, bs, gamma, n_bins, stats,
                                    static_cast<uint32_t*>(ws), reinterpret_cast<cudaStream_t>(stream)));
}

int dspark_obs_report(const dspark_obs_stats* st, int n_bins, dspark_obs_summary* out) {
  if (!st || !out || n_bins < 1 || n_bins > DSPARK_OBS_MAX_BINS) return DSPARK_EINVAL;
  const double nan = std::nan("");
  std::memset(out, 0, sizeof(*out));
  const double n = st->requests > 0 ? static_cast<double>(st->requests) : 1.0;
  out->mean_window = static_cast<double>(st->sum_window) / n;
  out->mean_accepted = static_cast<double>(st->sum_accepted) / n;
  out->mean_ceiling = st->ceiling_requests > 0
                          ? static_cast<double>(st->sum_ceiling) / static_cast<double>(st->ceiling_requests)
                          : nan;
  out->utilisation = st->sum_ceiling > 0
                         ? static_cast<double>(st->sum_accepted_ceiling) / static_cast<double>(st->sum_ceiling)
                         : nan;
  int64_t scored = 0;
  double num = 0.0;
  for (int b = 0; b < n_bins; ++b) {
    scored += st->bin_count[b];
    // |passed 2^32 - score sum| exact in integers, then scaled
    const int64_t d = static_cast<int64_t>(static_cast<uint64_t>(st->bin_label[b]) << 32) - st->bin_score_fx[b];
    num += static_cast<double>(d < 0 ? -d : d);
  }
  out->scored = scored;
  out->ece = scored > 0 ? std::ldexp(num, -32) / static_cast<double>(scored) : 0.0;
  for (int k = 0; k < DSPARK_MAX_GAMMA; ++k) {
    const int64_t c = st->pos_count[k];
    out->pos_mean_survival[k] = c > 0 ? std::ldexp(static_cast<double>(st->pos_score_fx[k]), -32) / c : nan;
    out->pos_pass_rate[k] = c > 0 ? static_cast<double>(st->pos_label[k]) / c : nan;
  }
  return DSPARK_OK;
}

size_t dspark_sts_fit_workspace_bytes(int n_grid, int n_bins) {
  if (n_grid < 1 || n_grid > 1024 || n_bins < 1 || n_bins > DSPARK_OBS_MAX_BINS) return 0;
  return sts_fit_ws_bytes(n_grid, n_bins);
}

int dspark_sts_fit(const float* z, const int32_t* ceiling, int N, int gamma, const float* grid,
                   int n_grid, int n_bins, float* T_out, double* ece_out, void* ws, size_t ws_bytes,
                   dspark_stream_t stream) {
  if (!z || !ceiling || !grid || !T_out || !ece_out) return DSPARK_EINVAL;
  if (N < 1 || N > (1 << 30) || gamma < 1 || n_grid < 1 || n_bins < 1 || n_bins > DSPARK_OBS_MAX_BINS)
    return DSPARK_EINVAL;
  if (gamma > DSPARK_MAX_GAMMA || n_grid > 1024) return DSPARK_EUNSUPPORTED;
  if (!al(z, 4) || !al(ceiling, 4) || !al(grid, 4) || !al(T_out, 4) || !al(ece_out, 8)) return DSPARK_EINVAL;
  if (!ws || !al(ws, 8) || ws_bytes < sts_fit_ws_bytes(n_grid, n_bins)) return DSPARK_EWORKSPACE;
  return cuda_status(launch_sts_fit(z, ceiling, N, gamma, grid, n_grid, n_bins, T_out, ece_out, ws,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
