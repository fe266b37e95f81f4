/*
 * dspark.h -- C ABI of the DSpark per-step speculative-decoding token path on GB300 (sm_103a).
 *
 * One decoding step of confidence-scheduled speculative decoding runs as five calls on one
 * CUDA stream, all asynchronous, none reading anything back to the host:
 *
 *   dspark_draft_block -> dspark_confidence -> dspark_schedule -> dspark_pack
 *       -> [the caller's target forward over the packed batch] -> dspark_verify
 * (dspark_draft_confidence_block does the first two in one call).
 *
 * Sources, cited by page and section:
 *   [SUMMARY] "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
 *             Generation" (technical summary page): "Architecture (drafter)",
 *             "Verification scheduling (system side)", "Infra".
 *   [SGLANG]  "DSpark in SGLang" blog: "Verify modes", "Ragged verify under full CUDA graphs".
 *   [VLLM]    "vLLM adaptive verification with DSpark": "DSpark confidence scheduling
 *             mechanism", "Technical implementation and CUDA Graphs".
 *
 * Conventions for every entry point
 *   - Pointers named as device pointers must point to device memory (or managed memory) of the
 *     current device; host pointers are plain host memory.  All tensors are dense, row-major,
 *     and every tensor pointer must be 16-byte aligned.
 *   - The caller owns every buffer.  The library allocates nothing and keeps no per-call
 *     state; scratch lives in the caller's workspace `ws` (size: dspark_workspace_bytes,
 *     zeroed once with dspark_workspace_init before first use).
 *   - Calls are enqueued on `stream` and return immediately.  The return value reports host-
 *     side argument checks (DSPARK_EINVAL / DSPARK_EUNSUPPORTED, nothing is launched) and
 *     launch failures (DSPARK_ECUDA).  Conditions only the device can see (a window larger
 *     than gamma, a packed total beyond the largest tier, a wait that timed out) are recorded
 *     in the workspace status word; dspark_read_device_status returns and clears it.
 *   - No exception or abort crosses the ABI.
 *   - Random numbers: Philox4x32-10 keyed by `seed`, counter (index >> 2, request, step low
 *     32 bits, purpose << 24 | position << 16 | step bits 32..47).  Purposes: 1 draft chunk
 *     key, 2 draft in-chunk uniform (index 0), 3 accept uniform, 4 decision chunk key,
 *     5 decision entry key.
 *     A uniform is ((word >> 9) + 0.5) * 2^-23.  A step is reproducible from (seed, step).
 *   - Sampling: a categorical draw over the vocabulary is two-level: chunks of consecutive ids
 *     get key log(mass) + Gumbel and the best chunk is drawn; then the id inside it.  The draft
 *     (chunks of DSPARK_DRAFT_CHUNK ids) takes the id by inverse CDF: the first id whose
 *     partial sum of the chunk's weights exceeds u times their total, u its in-chunk uniform.
 *     The verification (chunks of DSPARK_CHUNK ids) takes it by Gumbel-max over the chunk's
 *     log-weights.  Ties: lowest index.  Both laws are exactly the softmax for any chunk
 *     width; the width fixes which random words are used.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* dspark_stream_t; /* identical to cudaStream_t; NULL = default stream */

typedef enum {
    DSPARK_OK = 0,
    DSPARK_EINVAL = 1,       /* bad argument (host check) or bad data (device check)        */
    DSPARK_EUNSUPPORTED = 2, /* valid but outside what this build supports (sizes, dtypes)   */
    DSPARK_ECUDA = 3,        /* a CUDA runtime call or kernel launch failed                  */
    DSPARK_ETIMEOUT = 4,     /* a device-side wait gave up (status word only)                */
    DSPARK_EWORKSPACE = 5    /* workspace missing or smaller than dspark_workspace_bytes     */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

typedef enum { DSPARK_STATIC = 0, DSPARK_COMPACT = 1, DSPARK_CAP_ACCEPT = 2 } dspark_verify_mode;

typedef enum { DSPARK_SCHED_EARLY_STOP = 0, DSPARK_SCHED_GLOBAL_ARGMAX = 1 } dspark_sched_mode;

#define DSPARK_MAX_BS 256     /* requests per step                                   */
#define DSPARK_MAX_GAMMA 16   /* draft block length                                  */
#define DSPARK_CHUNK 128      /* chunk width of the verification's two-level draws   */
#define DSPARK_DRAFT_CHUNK 64 /* chunk width of the draft's two-level draws          */

/* Human-readable name of a status code (static string, never NULL). */
DSPARK_API const char* dspark_status_string(int status);

/* Bytes of workspace the calls of one step need for (bs, gamma, V); 0 on invalid sizes.
 * One workspace serves every call of a step; calls on the same stream may share it, calls
 * that can overlap on the device (different streams) must not. */
DSPARK_API size_t dspark_workspace_bytes(int bs, int gamma, int V);

/* Zero the whole workspace (asynchronous memset on `stream`); required once before first use:
 * besides the status word it holds counters that the kernels keep at zero between calls. */
DSPARK_API int dspark_workspace_init(void* ws, size_t ws_bytes, dspark_stream_t stream);

/* Synchronise `stream`, return the status recorded by device-side checks since the last
 * read (DSPARK_OK if none) and clear it.  The only call that waits for the device.
 * Diagnostics: when a device-side wait of a tensor-core kernel gives up (DSPARK_ETIMEOUT),
 * the first such wait since dspark_workspace_init is recorded in the workspace's 32-bit words
 * 4, 5, 6: the wait's site code, the CTA index and the site's progress counter (tile, box,
 * position or barrier number).  They are not cleared by this call. */
DSPARK_API int dspark_read_device_status(void* ws, dspark_stream_t stream);

/* Diagnostics: deadline, in nanoseconds from a kernel's start, of every device-side wait in
 * the tensor-core kernels (default 1 s).  A wait that runs out records DSPARK_ETIMEOUT in the
 * workspace status word; the kernel then waits (bounded) for its own copies in flight, frees
 * its tensor memory and returns, leaving the context usable.  Process-wide; returns the
 * previous value.  Tests use a tiny value to exercise that path. */
DSPARK_API uint64_t dspark_set_wait_timeout_ns(uint64_t ns);

/* Host: steps-per-second table from a profiled step-time curve ([VLLM] "Cost Modeling",
 * "CUDA Graph Padding"; [SGLANG] "Ragged verify"; [SUMMARY] "Verification scheduling").
 *   T_raw[M]   host, m_max+1 doubles: profiled step time (any unit) for M verify tokens.
 *   tiers      host, n_tiers strictly increasing totals of the captured graphs; n_tiers = 0
 *              means every total has its own graph.
 *   sps_out[M] host, m_max+1 doubles: 1 / max_{M' <= tier(M)} T_raw[M'], where tier(M) is the
 *              smallest tier >= M; 0 when tier(M) does not exist or exceeds m_max.
 * Returns DSPARK_EINVAL on null pointers, m_max < 0, non-positive or non-finite times, or
 * tiers that are not strictly increasing and positive. */
DSPARK_API int dspark_build_sps(const double* T_raw, int m_max, const int32_t* tiers, int n_tiers,
                     double* sps_out);

/* Host helper for a caller whose target-model logits sit in host memory (a host-side target
 * model, a replay of recorded logits): enqueue the host-to-device copies of exactly the rows a
 * packed verify batch reads ([SGLANG] "Ragged verify under full CUDA graphs": request r's
 * tested positions 0 .. n_r - 1 occupy packed rows cu[r] .. cu[r+1] - 1).
 *   packed     device [>= cu[bs], row_bytes]   destination rows (dspark_verify's `target`)
 *   rows       host   [bs, rows_per_req, row_bytes]  request r's candidate rows 0 .. rows_per_req-1
 *              (pinned memory for asynchronous copies)
 *   cu         host   [bs + 1] int32, the cu_seqlens that dspark_pack wrote (read back by the
 *              caller); request r contributes n_r = cu[r+1] - cu[r] rows.  Consecutive requests
 *              with the same n_r > 0 are one strided copy (cudaMemcpy2DAsync), a lone one a
 *              cudaMemcpyAsync.
 * Returns DSPARK_EINVAL on null pointers, row_bytes or rows_per_req < 1, decreasing cu or
 * n_r > rows_per_req (nothing is enqueued then), DSPARK_ECUDA when a copy fails to enqueue. */
DSPARK_API int dspark_copy_packed_rows_async(void* packed, const void* rows, size_t row_bytes, int bs,
                                             int rows_per_req, const int32_t* cu, dspark_stream_t stream);

/* S1. Markov-head block draft ([SUMMARY] "Architecture (drafter)", Markov head and
 * left-to-right sampling).  For k = 1..gamma, per request:
 *     l_k = U[:, k-1] + W1[x_{k-1}] . W2,   W2 = W2t^T,  x_0 = anchor
 *     temperature > 0:  x_k ~ softmax(l_k / temperature)  (chunk by Gumbel-max, id by inverse
 *                       CDF; purposes 1, 2)
 *                       logit_x = l_k[x_k] / temperature,  lse = logsumexp(l_k / temperature)
 *     temperature = 0:  x_k = argmax l_k (lowest index),  logit_x = l_k[x_k],  lse = 0
 *   U        device [bs, gamma, V]  base logits U_1..U_gamma of the parallel backbone
 *   W1       device [V, r]          Markov factor (row lookup by previous token)
 *   W2t      device [V, r]          Markov projection, stored transposed (a Linear(r, V) weight)
 *   dtype    element type of U, W1, W2t (fp32 or bf16); accumulation is fp32
 *   anchor   device [bs] int32      x_0, in [0, V)
 *   tokens   device [bs, gamma] int32 out;  logit_x, lse: device [bs, gamma] fp32 out
 * Limits: 1 <= bs <= 256, 1 <= gamma <= 16, V % 8 == 0, 8 <= V < 2^24, r in {32, 64, 128, 256}.
 * Errors: EINVAL (null, sizes, temperature < 0 or not finite, misaligned), EWORKSPACE. */
DSPARK_API int dspark_draft_block(const void* U, const void* W1, const void* W2t, int dtype,
                       const int32_t* anchor, int bs, int gamma, int V, int r,
                       float temperature, uint64_t seed, uint64_t step,
                       int32_t* tokens, float* logit_x, float* lse,
                       void* ws, size_t ws_bytes, dspark_stream_t stream);

/* S1 and S2 in one call: the outputs of dspark_draft_block followed by dspark_confidence on the
 * drafted tokens, bit for bit.  On the tensor-core pass (bf16, r = 64, 128 or 256) the confidence
 * of position k is computed inside the draft's launch as soon as x_{k-1} is drawn, so it finishes
 * under the draft's own time; otherwise the two run as their own launches.
 *   draft arguments   as dspark_draft_block
 *   h, d, w, b, sts_T, conf, surv, z_logit   as dspark_confidence (h in `dtype`)
 * Limits and errors: those of both calls. */
DSPARK_API int dspark_draft_confidence_block(const void* U, const void* W1, const void* W2t, int dtype,
                       const int32_t* anchor, int bs, int gamma, int V, int r,
                       float temperature, uint64_t seed, uint64_t step,
                       int32_t* tokens, float* logit_x, float* lse,
                       const void* h, int d, const float* w, float b, const float* sts_T,
                       float* conf, float* surv, float* z_logit,
                       void* ws, size_t ws_bytes, dspark_stream_t stream);

/* S1 with the RNN sequential head ([SUMMARY] "Architecture (drafter)", RNN head: a gated
 * recurrent state s_k carried across the block, so each position sees the whole prefix).  The
 * pages give no equations; this library's reading, per request:
 *     e_k = W1[x_{k-1}]  (x_0 = anchor),   s_0 = 0
 *     g_k = sigmoid([e_k ; s_{k-1}] Wg + bg)                 Wg [2r, r], bg [r]
 *     s_k = g_k * s_{k-1} + (1 - g_k) * e_k                  held in `dtype` (bf16: rounded to
 *                                                             nearest even after each update)
 *     l_k = U[:, k-1] + s_k . W2,  then the draw exactly as dspark_draft_block (same random
 *     streams, outputs and temperature rule).  A closed gate (g = 0) is the Markov head.
 *   Wg       device [2r, r] (dtype), row j < r multiplies e_k[j], row r + j multiplies s_{k-1}[j]
 *   bg       device [r] fp32
 *   states   device [bs, gamma, r] (dtype) out: s_1 .. s_gamma (dspark_verify's draft_states)
 *   other arguments, limits and errors as dspark_draft_block.
 * bf16 with r = 64, 128 or 256: the state updates run inside the draft's one launch; otherwise one
 * extra small launch per position (the state update: a [bs, 2r] x [2r, r] GEMM). */
DSPARK_API int dspark_draft_block_rnn(const void* U, const void* W1, const void* W2t, const void* Wg,
                                      const float* bg, int dtype, const int32_t* anchor, int bs, int gamma,
                                      int V, int r, float temperature, uint64_t seed, uint64_t step,
                                      int32_t* tokens, float* logit_x, float* lse, void* states, void* ws,
                                      size_t ws_bytes, dspark_stream_t stream);

/* S2. Confidence head, sequential temperature scaling and prefix survival ([SUMMARY]
 * "Verification scheduling": confidence head, STS, prefix survival):
 *     z_{r,k} = w[0:d] . h[r, k-1] + w[d:d+r] . W1[x_{r,k-1}] + b      (x_0 = anchor)
 *     conf_{r,k} = 1 / (1 + exp(-z_{r,k} / sts_T[k-1]))
 *     surv_{r,k} = conf_{r,1} * ... * conf_{r,k}        (fp32, left to right)
 *   h        device [bs, gamma, d] (dtype);  W1 device [V, r] (dtype)
 *   tokens   device [bs, gamma] int32 (x_1..x_gamma);  anchor device [bs] int32
 *   w        device [d + r] fp32;  sts_T device [gamma] fp32, each > 0
 *   conf, surv  device [bs, gamma] fp32 out
 *   z_logit  device [bs, gamma] fp32 out or NULL: z before STS (the input of dspark_sts_fit)
 * Limits: as dspark_draft_block, and d % 8 == 0, 8 <= d <= 65536. */
DSPARK_API int dspark_confidence(const void* h, const void* W1, int dtype, const int32_t* anchor,
                      const int32_t* tokens, const float* w, float b, const float* sts_T,
                      int bs, int gamma, int d, int r, int V,
                      float* conf, float* surv, float* z_logit, dspark_stream_t stream);

/* S3. Hardware-aware global top-B prefix scheduler ([SUMMARY] "Verification scheduling",
 * Algorithm 1; [VLLM] "DSpark confidence scheduling mechanism"; [SUMMARY] "Infra").
 * Slots (r, j) are ranked by descending fp32 surv[r, j] (ties: lower r, then lower j).
 * With S_K = sum over the first K slots of floor(surv * 2^40) (exact int64),
 *     Theta(K) = (bs + S_K * 2^-40) * sps[bs + K],   K = 0 .. min(bs*gamma, m_max - bs)
 * EARLY_STOP: K* = first K with Theta(K+1) <= Theta(K) (else the last K);
 * GLOBAL_ARGMAX: K* = smallest K maximising Theta.  window[r] = admitted slots of r.
 *   surv     device [bs, gamma] fp32, non-increasing along each row, in [0, 1]
 *   sps      device [m_max + 1] fp64 (dspark_build_sps), m_max >= bs; the entries the search
 *            reads, sps[bs .. bs + Kmax], must be finite, >= 0 and non-increasing in M
 *   window   device [bs] int32 out;  K_out device int32 out;  theta_out device fp64 out
 *   ws       the step's workspace (>= 256 bytes); only its status word is used, updated
 *            atomically, so a call on another stream may share it.
 * Device error (status word, EINVAL): a table entry the search reads that is negative, not
 * finite, or above the entry before it (the outputs are still written, from the table as given).
 * Limits: bs * gamma <= 4096.  One thread block; no host readback. */
DSPARK_API int dspark_schedule(const float* surv, int bs, int gamma, const double* sps, int m_max,
                    int mode, int32_t* window, int32_t* K_out, double* theta_out,
                    void* ws, size_t ws_bytes, dspark_stream_t stream);

/* S3 under zero-overhead (asynchronous) scheduling ([SUMMARY] "Infra", scheduler bullet;
 * [SGLANG] "ZOS"): the verify budget of step t is predicted from the survival of step t - 2,
 * the windows still take the top slots of step t's own survival.  Two calls per step, on a
 * two-entry device ring of budgets (int32, set to -1 before the first step):
 *   dspark_schedule_zos_select: K = budget_ring[step & 1]; K < 0 (nothing recorded two
 *     steps back) means K = the GLOBAL_ARGMAX K* of surv itself.  K is clamped to
 *     min(bs*gamma, m_max - bs); window[r] = how many of the K top-ranked slots of surv
 *     (ranking as dspark_schedule) belong to r;  K_out = K.  budget_ring is only read.
 *   dspark_schedule_zos_budget: budget_ring[step & 1] = the GLOBAL_ARGMAX K* of surv (as
 *     dspark_schedule), the budget of step + 2.
 * Ordering, the caller's: select(step) before budget(step) (both touch slot step & 1), and
 * budget(step) before select(step + 2).  On one stream in that order this holds; the budget
 * call may run on a second stream, off the step's critical path, joined by events.
 *   surv, sps, m_max, window, K_out, ws as dspark_schedule (the table check applies whenever
 *   the global search runs);  budget_ring device [2] int32
 * Limits: bs * gamma <= 4096.  One thread block each; no host readback. */
DSPARK_API int dspark_schedule_zos_select(const float* surv, int bs, int gamma, const double* sps,
                               int m_max, const int32_t* budget_ring, uint64_t step,
                               int32_t* window, int32_t* K_out, void* ws, size_t ws_bytes,
                               dspark_stream_t stream);
DSPARK_API int dspark_schedule_zos_budget(const float* surv, int bs, int gamma, const double* sps,
                               int m_max, int32_t* budget_ring, uint64_t step, void* ws,
                               size_t ws_bytes, dspark_stream_t stream);

/* S4. Ragged cu_seqlens packing rounded up to a captured graph tier ([SGLANG] "Ragged verify
 * under full CUDA graphs", Fig. 2; [VLLM] "Graph Capture", "CUDA Graph Padding").
 * Request r contributes n_r = l_r + 1 rows [x_0, x_1 .. x_{l_r}] where l_r = window[r]
 * (window == NULL: l_r = gamma, the static layout).  cu[0] = 0, cu[r+1] = cu[r] + n_r,
 * M = cu[bs]; padded = smallest tier >= M (n_tiers = 0: padded = M).  Row p < M holds
 * ids = token, req = request, pos = j; rows M .. padded-1 hold -1 in all three.
 *   window   device [bs] int32 or NULL;  anchor device [bs];  tokens device [bs, gamma]
 *   tiers    device [n_tiers] int32 strictly increasing;  cap = rows of ids/req/pos
 *   cu_seqlens device [bs+1] int32 out;  ids, req, pos device [cap] int32 out
 *   padded_total device [1] int32 out (-1 on a device-side error)
 * Device errors (status word, EINVAL; padded_total = -1, no rows written): l_r outside
 * [0, gamma], tiers not positive and strictly increasing, M beyond the largest tier, padded > cap. */
DSPARK_API int dspark_pack(const int32_t* window, const int32_t* anchor, const int32_t* tokens,
                int bs, int gamma, const int32_t* tiers, int n_tiers, int cap,
                int32_t* cu_seqlens, int32_t* ids, int32_t* req, int32_t* pos,
                int32_t* padded_total, void* ws, size_t ws_bytes, dspark_stream_t stream);

/* S3 then S4 in one launch: exactly dspark_schedule (window required) followed by dspark_pack
 * of the windows it wrote, with the arguments, outputs and errors of both (device checks of the
 * table and of the tiers included); one kernel boundary fewer on the step's path. */
DSPARK_API int dspark_schedule_pack(const float* surv, int bs, int gamma, const double* sps, int m_max,
                                    int mode, int32_t* window, int32_t* K_out, double* theta_out,
                                    const int32_t* anchor, const int32_t* tokens, const int32_t* tiers,
                                    int n_tiers, int cap, int32_t* cu_seqlens, int32_t* ids, int32_t* req,
                                    int32_t* pos, int32_t* padded_total, void* ws, size_t ws_bytes,
                                    dspark_stream_t stream);

/* S5. Rejection-sampling verification ([SUMMARY] "Abstract", "Architecture (drafter)";
 * [SGLANG] "Verify modes").  Per request r, with l_r = window[r]:
 *   tested positions  L_test   = l_r (COMPACT) or gamma (STATIC, CAP_ACCEPT)
 *   committed window  L_commit = l_r (COMPACT, CAP_ACCEPT) or gamma (STATIC)
 *   target row scoring position k: cu_seqlens[r] + k - 1 (k = 1 .. L_test + 1); the packed
 *   layout must give n_r = L_test + 1 (device check, EINVAL).
 *   temperature > 0: x_k is accepted iff u_k < p_t(x_k) / p_d(x_k) with
 *     log p_t = target_row/temperature at x_k minus its log-sum-exp, log p_d = logit_x - lse,
 *     u_k the accept uniform (purpose 3, position k, index 0).  At the first rejection
 *     k* <= L_commit the token is redrawn from normalise(max(0, p_t - p_d)) (p_t if that is
 *     empty), p_d recomputed from U, W1, W2t at position k* -- or, when draft_logits is given,
 *     p_d = exp(draft_logits[r, k*-1] / temperature - lse[r, k*-1]); if no tested position up to
 *     L_commit is rejected, a bonus token is drawn from p_t of row L_commit + 1
 *     (decision draws: purposes 4, 5 at the drawn position).
 *   temperature = 0: x_k is accepted iff it is the target argmax; the extra token is the
 *     argmax of the deciding row.
 *   out_tokens  device [bs, gamma+1] int32 out: x_1..x_acc, the extra token, then -1
 *   acc_len     device [bs] int32 out: accepted draft tokens
 *   ceiling     device [bs] int32 out or NULL: accepted count over the tested positions
 *               (the full-block ceiling in CAP_ACCEPT mode)
 *   target      device [rows, V] (dtype), rows >= cu_seqlens[bs]
 *   window      device [bs] int32 (ignored in STATIC mode, may be NULL there)
 *   tokens, logit_x, lse, anchor: the draft's outputs / inputs;  U, W1, W2t, r as in S1.
 *   draft_logits device [bs, gamma, V] (dtype) or NULL: the draft's logits l_k of every
 *               position, for callers that hold them (another drafter, or a caller that kept
 *               them); lse must be their log-sum-exp at temperature (as dspark_draft_block
 *               writes it).  Given, U, W1, W2t (may be NULL), draft_states and r are not used;
 *               NULL, U, W1, W2t are required and p_d is recomputed.
 *   draft_states device [bs, gamma, r] (dtype) or NULL: the RNN head's states s_k
 *               (dspark_draft_block_rnn); the recompute of p_d at position k* then takes
 *               U[:, k*-1] + s_k* . W2 instead of the Markov head's U + W1[x_{k*-1}] . W2.
 * Limits: as dspark_draft_block. */
DSPARK_API int dspark_verify(const void* target, int dtype, const int32_t* cu_seqlens,
                  const int32_t* window, int mode, int bs, int gamma, int V,
                  const int32_t* anchor, const int32_t* tokens, const float* logit_x,
                  const float* lse, const void* draft_logits, const void* draft_states,
                  const void* U, const void* W1, const void* W2t, int r, float temperature,
                  uint64_t seed, uint64_t step,
                  int32_t* out_tokens, int32_t* acc_len, int32_t* ceiling,
                  void* ws, size_t ws_bytes, dspark_stream_t stream);

/* Allocation-free variant of dspark_draft_block.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory and so have no workspace to
 * pass -- for example a plugin running inside another framework's device-memory pool (a
 * cudaMalloc would bypass that framework's allocator and its accounting), or a service that
 * fixes its device footprint at start-up and forbids later allocation.  Same computation,
 * arguments and limits as dspark_draft_block, without ws / ws_bytes; it allocates nothing.
 *   Scratch: a fixed 8 MiB array inside the library (every GPU that loads the library holds it
 *   until exit).  A call needs 256 B + bs * n * 16 B of it, n = the CTA columns of the
 *   tensor-core pass (bf16 with r = 64, 128 or 256; at most the SM count, fewer when bs > 128
 *   or when V has fewer 256-id tiles) and n = ceil(V / 64) on the CUDA-core pass (fp32, or
 *   r = 32); sizes needing more are rejected with DSPARK_EUNSUPPORTED.  Every V the library
 *   accepts fits the tensor-core pass (at most 128 x 152 or 256 x 76 slots of 16 B, 0.3 MB, on
 *   a 152-SM GB300); at bs = 256 the CUDA-core pass allows V <= 131,008.
 *   The first call on a device looks up the array's device address (once per device, with that
 *   device current); make that first call before any stream capture.  The address is kept for
 *   the life of the process: cudaDeviceReset between calls is not supported.
 *   All calls share the array and it keeps the last call's contents: calls whose work can
 *   overlap on the GPU (other streams, other host threads) race and must be serialised.
 *   device_status: device uint32 or NULL.  If given, device-side errors (a wait timeout) are
 *   recorded there (first error wins; the caller zeroes it); if NULL, they go to a status word
 *   in the array that each call clears and that the caller cannot read. */
DSPARK_API int dspark_draft_block_noalloc(const void* U, const void* W1, const void* W2t, int dtype,
                                          const int32_t* anchor, int bs, int gamma, int V, int r,
                                          float temperature, uint64_t seed, uint64_t step,
                                          int32_t* tokens, float* logit_x, float* lse,
                                          uint32_t* device_status, dspark_stream_t stream);

/* Observability and calibration ([SGLANG] "Observability", "Per-request differentiation under
 * mixed traffic" Fig. 4; [SUMMARY] "Verification scheduling", STS).
 *
 * The outcome of a prefix survival a_{r,k}: did positions 1..k all pass?  With a ceiling (the
 * accepted length over the whole block: a cap-accept run's `ceiling`, or a static run's
 * acc_len) it is [ceiling_r >= k] at every k.  Without one (compact) it is known where the run
 * decided it: [acc_r >= k] for k <= l_r, and 0 beyond l_r when the window was rejected inside;
 * unknown beyond l_r when the whole window passed (pruning hides the ceiling).
 * ECE over M equal-width bins of [0, 1] (bin = floor(a * M) in fp32, clamped to [0, M-1]):
 *     ECE = sum_b |sum of outcomes in b - sum of scores in b| / (scored pairs). */
#define DSPARK_OBS_MAX_BINS 64

/* Accumulated records (device memory, zeroed by the caller before the first record).  Score
 * sums are fixed point: sum of floor(a * 2^32) (a in [0, 1]; exact integer sums, so records
 * are order-independent and reproducible). */
typedef struct {
  int64_t steps, requests, sum_window, sum_accepted;
  int64_t ceiling_requests, sum_ceiling, sum_accepted_ceiling, reserved;
  int64_t window_hist[DSPARK_MAX_GAMMA + 1];    /* requests by window length l_r           */
  int64_t accepted_hist[DSPARK_MAX_GAMMA + 1];  /* requests by accepted length             */
  int64_t ceiling_hist[DSPARK_MAX_GAMMA + 1];   /* requests by ceiling (ceiling runs only) */
  int64_t bin_count[DSPARK_OBS_MAX_BINS];       /* scored (r, k) pairs per bin              */
  int64_t bin_label[DSPARK_OBS_MAX_BINS];       /* passed prefixes per bin                  */
  int64_t bin_score_fx[DSPARK_OBS_MAX_BINS];    /* sum of floor(a * 2^32) per bin           */
  int64_t pos_count[DSPARK_MAX_GAMMA];          /* the same three per position k            */
  int64_t pos_label[DSPARK_MAX_GAMMA];
  int64_t pos_score_fx[DSPARK_MAX_GAMMA];
} dspark_obs_stats;

typedef struct {
  double mean_window, mean_accepted, mean_ceiling; /* per request; mean_ceiling NaN if none */
  double utilisation;      /* sum accepted / sum ceiling over ceiling runs (NaN if none)     */
  double ece;              /* of the survival against the prefix outcomes                    */
  double pos_mean_survival[DSPARK_MAX_GAMMA], pos_pass_rate[DSPARK_MAX_GAMMA]; /* NaN if none */
  int64_t scored;          /* (r, k) pairs with a known outcome                              */
} dspark_obs_summary;

/* Add one step's record to `stats` (device).  surv device [bs, gamma] fp32 in [0, 1];
 * window device [bs] int32 or NULL (= gamma, static); acc_len device [bs] int32;
 * ceiling device [bs] int32 or NULL;  1 <= n_bins <= DSPARK_OBS_MAX_BINS.
 * Device check (status word via ws, EINVAL): window, acc_len or ceiling outside [0, gamma],
 * acc_len > window, or acc_len > ceiling; the step is then not recorded.  One thread block. */
DSPARK_API int dspark_observe(const float* surv, const int32_t* window, const int32_t* acc_len,
                   const int32_t* ceiling, int bs, int gamma, int n_bins,
                   dspark_obs_stats* stats, void* ws, size_t ws_bytes, dspark_stream_t stream);

/* Host: the summary of a host copy of accumulated records.  EINVAL on NULL or bad n_bins. */
DSPARK_API int dspark_obs_report(const dspark_obs_stats* stats, int n_bins, dspark_obs_summary* out);

/* Sequential temperature scaling fit ([SUMMARY] "Verification scheduling", STS): for
 * k = 1..gamma in order, T_k = the grid value minimising the ECE of
 *     a_{i,k} = prod_{j<k} sigmoid(z[i, j] / T_j) * sigmoid(z[i, k] / T)      (fp32)
 * against [ceiling_i >= k] over the N labelled prefixes (earlier T_j fixed; ties: the lowest
 * grid index).  The scores use the fast exponential (relative error ~1e-6: they are only
 * binned); the ECE of each grid value comes from exact integer sums of floor(a 2^24), in fp64.
 *   z        device [N, gamma] fp32: confidence logits before STS (dspark_confidence z_logit)
 *   ceiling  device [N] int32 in [0, gamma]: accepted prefix length over the whole block
 *   grid     device [n_grid] fp32 temperatures, each > 0 (1 <= n_grid <= 1024)
 *   T_out    device [gamma] fp32 out;  ece_out device [gamma] fp64 out (ECE at the chosen T)
 *   ws       device scratch of dspark_sts_fit_workspace_bytes(n_grid, n_bins) bytes
 * Limits: 1 <= N <= 2^30, 1 <= gamma <= DSPARK_MAX_GAMMA, 1 <= n_bins <= DSPARK_OBS_MAX_BINS.
 * 3 gamma launches, all asynchronous. */
DSPARK_API size_t dspark_sts_fit_workspace_bytes(int n_grid, int n_bins);
DSPARK_API int dspark_sts_fit(const float* z, const int32_t* ceiling, int N, int gamma,
                   const float* grid, int n_grid, int n_bins, float* T_out, double* ece_out,
                   void* ws, size_t ws_bytes, dspark_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
