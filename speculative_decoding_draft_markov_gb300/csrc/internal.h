// Internal launchers of libdspark (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dspark {

// ---- S1 draft ---------------------------------------------------------------------------
// Partial draws of l_k = U_k + A_k W2 for one position k, A_k = W1[x_{k-1}] (Markov head) or
// the RNN head's state s_k (`states` non-null, [bs, gamma, r]): per (row, slot) a
// DraftEntry (common.cuh) over the slot's draft chunks.  The CUDA-core pass has one slot per
// draft chunk (n_slots = n_draft_chunks(V)).
cudaError_t launch_draft_stats_simt(int dtype, const void* U, const void* W1, const void* W2t,
                                    const void* states, const int32_t* anchor, const int32_t* tokens, int bs, int gamma,
                                    int V, int r, int k, float inv_tau, int greedy, uint64_t seed,
                                    uint64_t step, void* entries, int n_slots, cudaStream_t s);
// The tensor-core pass (tcgen05 + TMEM + TMA), bf16 only, positions k_first .. k_last in one
// persistent cooperative launch that also runs each position's select (tokens, logit_x, lse
// written): one entry slot per CTA column (draft_tc_slots(bs, V) of them).  ctl: the grid
// barrier's words (the workspace status block + 64 bytes; 192 bytes, zero between calls);
// diag: three words recording the first wait that gave up (note_timeout), or null.  RNN head:
// states, Wg, bg non-null; the kernel writes s_1 .. s_{k_last} when k_first = 1 (else
// states[:, k_first - 1] must already hold s_{k_first}, and it writes the states after it).
// cf: the confidence head to compute while drafting (bf16, k_first = 1), or null.
struct ConfArgs {  // the confidence head's inputs and outputs, as dspark_confidence takes them
  const void* h;
  const float* w;
  float b;
  const float* sts_T;
  int d;
  float* conf;
  float* surv;
  float* z_logit;
};
cudaError_t launch_draft_tc(const void* U, const void* W1, const void* W2t, const void* states, const void* Wg,
                            const float* bg, const ConfArgs* cf, const int32_t* anchor,
                            int32_t* tokens, float* logit_x, float* lse, int bs, int gamma, int V, int r, int k_first,
                            int k_last, float inv_tau, int greedy, uint64_t seed, uint64_t step, void* entries,
                            uint32_t* ctl, uint32_t* status, uint32_t* diag, cudaStream_t s);
bool draft_tc_supported(int dtype, int bs, int V, int r);
// Slots (entries per request) the tensor-core pass writes: one per CTA column (at most one per
// SM, and per 256-id vocabulary tile).
int draft_tc_slots(int bs, int V);
// Verify's decision masses on the tensor cores (bf16): per request and CTA column a
// DecideEntry (common.cuh) over the column's chunks of the request's deciding row (residual
// mass sum max(0, p_t - p_d), target mass sum p_t, best chunk keys); n_slots returned.
cudaError_t launch_decision_stats_tc(const void* target, const void* U, const void* W1, const void* W2t,
                                     const void* states, const int32_t* anchor, const int32_t* tokens, const float* lse_d,
                                     const void* rs, const void* dec, int bs, int gamma, int V, int r,
                                     float inv_tau, uint64_t seed, uint64_t step, void* entries,
                                     int n_chunks, int* n_slots, uint32_t* status, cudaStream_t s);
extern uint64_t g_wait_timeout_ns;  // deadline of device-side waits (dspark_set_wait_timeout_ns)
// Merge the n_slots entries of each row of one position and draw x_k.
cudaError_t launch_draft_select(int dtype, const void* entries, int n_slots, const void* U,
                                const void* W1, const void* W2t, const void* states, const int32_t* anchor,
                                int32_t* tokens, float* logit_x, float* lse, int bs, int gamma,
                                int V, int r, int k, float inv_tau, int greedy, uint64_t seed,
                                uint64_t step, uint32_t* status, cudaStream_t s);

// RNN head: the recurrent states s_k of position k for every request (states [bs, gamma, r]),
// from s_{k-1} and W1[x_{k-1}] (x_0 = anchor, s_0 = 0).
cudaError_t launch_rnn_state(int dtype, const void* W1, const void* Wg, const float* bg, const int32_t* anchor,
                             const int32_t* tokens, void* states, int bs, int gamma, int V, int r, int k,
                             cudaStream_t s);

// ---- S2 / S3 / S4 -----------------------------------------------------------------------
cudaError_t launch_confidence(int dtype, const void* h, const void* W1, const int32_t* anchor,
                              const int32_t* tokens, const float* w, float b, const float* sts_T,
                              int bs, int gamma, int d, int r, int V, float* conf, float* surv,
                              float* z_out, cudaStream_t s);
cudaError_t launch_schedule(const float* surv, int bs, int gamma, const double* sps, int m_max,
                            int mode, int32_t* window, int32_t* K_out, double* theta_out,
                            uint32_t* status, cudaStream_t s);
cudaError_t launch_zos_select(const float* surv, int bs, int gamma, const double* sps, int m_max,
                              const int32_t* ring, uint64_t step, int32_t* window, int32_t* K_out,
                              uint32_t* status, cudaStream_t s);
cudaError_t launch_observe(const float* surv, const int32_t* window, const int32_t* acc_len,
                           const int32_t* ceiling, int bs, int gamma, int n_bins, void* stats,
                           uint32_t* status, cudaStream_t s);
size_t sts_fit_ws_bytes(int n_grid, int n_bins);
cudaError_t launch_sts_fit(const float* z, const int32_t* ceiling, int N, int gamma, const float* grid,
                           int n_grid, int n_bins, float* T_out, double* ece_out, void* ws, cudaStream_t s);
cudaError_t launch_zos_budget(const float* surv, int bs, int gamma, const double* sps, int m_max,
                              int32_t* ring, uint64_t step, uint32_t* status, cudaStream_t s);
cudaError_t launch_pack(const int32_t* window, const int32_t* anchor, const int32_t* tokens,
                        int bs, int gamma, const int32_t* tiers, int n_tiers, int cap,
                        int32_t* cu, int32_t* ids, int32_t* req, int32_t* pos, int32_t* padded,
                        uint32_t* status, cudaStream_t s);
// S3 and S4 in one launch (the scheduler's block packs the windows it writes).
cudaError_t launch_schedule_pack(const float* surv, int bs, int gamma, const double* sps, int m_max, int mode,
                                 int32_t* window, int32_t* K_out, double* theta_out, const int32_t* anchor,
                                 const int32_t* tokens, const int32_t* tiers, int n_tiers, int cap, int32_t* cu,
                                 int32_t* ids, int32_t* req, int32_t* pos, int32_t* padded, uint32_t* status,
                                 cudaStream_t s);

// ---- S5 verify --------------------------------------------------------------------------
cudaError_t launch_verify(int dtype, const void* target, const int32_t* cu, const int32_t* window,
                          int mode, int bs, int gamma, int V, const int32_t* anchor,
                          const int32_t* tokens, const float* logit_x, const float* lse,
                          const void* draft_logits, const void* U, const void* W1, const void* W2t,
                          const void* states, int r, float inv_tau, int greedy, uint64_t seed, uint64_t step,
                          int32_t* out_tokens, int32_t* acc_len, int32_t* ceiling, void* ws,
                          cudaStream_t s);

}  // namespace dspark
