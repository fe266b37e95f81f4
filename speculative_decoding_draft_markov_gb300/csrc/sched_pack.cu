// S2 confidence head + STS + prefix survival, S3 global top-B prefix scheduler, S4 ragged
// packing.  All three are small, latency-bound kernels that keep the step on the device.
#include <climits>

#include "common.cuh"
#include "confidence.cuh"
#include "internal.h"
#include "pdl.h"

namespace dspark {

// ---------------------------------------------------------------------------------------
// S2.  DSpark technical summary, "Verification scheduling (system side)": the confidence
// head is a linear projection of [h_k ; W1[x_{k-1}]] followed by a sigmoid; sequential
// temperature scaling divides the logit by T_k; prefix survival is the running product.
// fp32 dot products in a fixed order.
// ---------------------------------------------------------------------------------------
// One block per request; conf_parts(gamma) warps per position split the h term, the first of
// them also reduces the W1[x_{k-1}] term (confidence.cuh: the order shared with the persistent
// draft kernel).  Thread 0 then adds the terms in order and runs the sigmoid / STS / product
// chain.
template <typename T>
__global__ void __launch_bounds__(512) confidence_kernel(
    const T* __restrict__ h, const T* __restrict__ W1, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, const float* __restrict__ w, float b,
    const float* __restrict__ sts_T, int gamma, int d, int r, int V, int parts, float* __restrict__ conf,
    float* __restrict__ surv, float* __restrict__ z_out) {
  __shared__ float zp[DSPARK_MAX_GAMMA * 4], zx[DSPARK_MAX_GAMMA];
  pdl_enter();
  const int req = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pos = warp / parts, part = warp - pos * parts;
  if (pos < gamma) {
    const int k = pos + 1;
    // the W1[x_{k-1}] group is loaded first, so that its latency overlaps the h loads
    uint4 qa[sizeof(T) == 4 ? 2 : 1];
    if (part == 0 && lane * 8 < r)
      load_hgroup<T>(W1 + size_t(clamp_token((k == 1) ? anchor[req] : tokens[size_t(req) * gamma + k - 2], V)) * r +
                         lane * 8, qa);
    const float hq = warp_sum(conf_hpart<T>(h + (size_t(req) * gamma + pos) * d, w, d, part, parts, lane));
    if (lane == 0) zp[pos * 4 + part] = hq;
    if (part == 0) {
      const float xq = warp_sum(conf_xpart<T>(qa, w, d, r, lane));
      if (lane == 0) zx[pos] = xq;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 1.f;
    for (int k = 0; k < gamma; ++k) {
      float z = zp[k * 4];
      for (int q = 1; q < parts; ++q) z += zp[k * 4 + q];
      z += zx[k];
      z += b;
      if (z_out) z_out[size_t(req) * gamma + k] = z;  // the logit before STS (calibration input)
      const float c = 1.f / (1.f + expf(-z / sts_T[k]));
      a *= c;
      conf[size_t(req) * gamma + k] = c;
      surv[size_t(req) * gamma + k] = a;
    }
  }
}

cudaError_t launch_confidence(int dtype, const void* h, const void* W1, const int32_t* anchor,
                              const int32_t* tokens, const float* w, float b, const float* sts_T,
                              int bs, int gamma, int d, int r, int V, float* conf, float* surv,
                              float* z_out, cudaStream_t s) {
  const int parts = conf_parts(gamma);  // warps per position: at most 512 threads, two blocks per SM
  const int threads = 32 * parts * gamma;
  if (dtype == DSPARK_F32)
    return launch_pdl(confidence_kernel<float>, dim3(bs), dim3(threads), 0, s, (const float*)h, (const float*)W1,
                      anchor, tokens, w, b, sts_T, gamma, d, r, V, parts, conf, surv, z_out);
  return launch_pdl(confidence_kernel<__nv_bfloat16>, dim3(bs), dim3(threads), 0, s, (const __nv_bfloat16*)h,
                    (const __nv_bfloat16*)W1, anchor, tokens, w, b, sts_T, gamma, d, r, V, parts, conf, surv, z_out);
}

// ---------------------------------------------------------------------------------------
// S3.  DSpark technical summary, "Verification scheduling", Hardware-Aware Prefix Scheduler
// (Algorithm 1): admit slots globally by descending survival, Theta = tau * SPS(bs + K),
// stop when Theta stops growing ("Infra": or take the global maximum).  vLLM adaptive
// verification, "DSpark confidence scheduling mechanism": tau counts one extra token per
// request plus the survival of the admitted slots.
// One block of 1024 threads.  64-bit keys (descending fp32 survival bits, then slot index
// r * gamma + j) are sorted by a bitonic network held in registers (shuffles for the short
// distances, shared memory for the long ones).  Then exact int64 fixed-point prefix sums of floor(a * 2^40),
// Theta in fp64 with one rounding per product, block reductions for the stop / argmax.
// ---------------------------------------------------------------------------------------
constexpr int kSchedThreads = 1024;
constexpr int kSchedMaxSlots = 4096;

// floor(a * 2^40) of a non-negative fp32 value from its bits, in integer arithmetic (the fp64
// pipe of this part is narrow): a = (m | 2^23) 2^(e - 150), so a 2^40 = (m | 2^23) 2^(e - 110).
// Exact for a < 2^23; zero for subnormal a (a 2^40 < 1).
__device__ __forceinline__ long long fix40(uint32_t bits) {
  const int e = int((bits >> 23) & 0xFFu);
  if (e == 0) return 0;
  const unsigned long long mm = (bits & 0x7FFFFFu) | 0x800000u;
  const int sh = e - 110;
  if (sh >= 0) return static_cast<long long>(mm << (sh < 22 ? sh : 22));
  return sh <= -24 ? 0ll : static_cast<long long>(mm >> (-sh));
}

// T 2^-40 as a double for an integer 2^40 <= T < 2^53: exact, built from the bits (T has at most
// 53 significant bits, and the scale only lowers the exponent).
__device__ __forceinline__ double scaled_fixed(long long T) {
  const int e = 63 - __clzll(T);  // floor(log2 T), 40 .. 52
  const unsigned long long mant = (static_cast<unsigned long long>(T) << (52 - e)) & ((1ull << 52) - 1);
  return __longlong_as_double(static_cast<long long>((static_cast<unsigned long long>(e + 1023 - 40) << 52) | mant));
}

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Order-preserving 64-bit integer of a non-NaN double (-0 maps with +0).
__device__ __forceinline__ long long dkey(double x) {
  long long b = __double_as_longlong(x);
  if (b == static_cast<long long>(0x8000000000000000ull)) b = 0;
  return b >= 0 ? b : (b ^ 0x7FFFFFFFFFFFFFFFll);
}
__device__ __forceinline__ bool dnan(double x) {
  return (static_cast<unsigned long long>(__double_as_longlong(x)) & 0x7FFFFFFFFFFFFFFFull) > 0x7FF0000000000000ull;
}

// Sort key of slot e (survival bits descending, then slot index), or a sentinel for e >= n.
__device__ __forceinline__ unsigned long long sched_key(const float* __restrict__ surv, int e, int n) {
  if (e >= n) return (0xFFFFFFFFull << 32) | static_cast<unsigned>(kSchedMaxSlots + e);
  uint32_t bits = __float_as_uint(surv[e]);
  if (bits & 0x80000000u) bits = 0u;  // -0 and negatives rank as 0
  return (static_cast<unsigned long long>(0xFFFFFFFFu - bits) << 32) | static_cast<unsigned>(e);
}

// Ascending bitonic sort of the keys of slots 0 .. 1024 E - 1 by the 1024 threads of the block
// into out[0 .. 1024 E).  `out` also serves as the exchange buffer of the long distances; when
// it holds two such buffers (2 N <= kSchedMaxSlots) consecutive exchanges alternate between
// them, so that an exchange needs one barrier instead of two (a thread writes one buffer only
// after every thread has passed the barrier of the exchange that used the other).
template <int E>
__device__ void bitonic_sort(const float* __restrict__ surv, int n, unsigned long long* out, int tid) {
  constexpr int N = 1024 * E;
  constexpr bool kTwoBuffers = 2 * N <= kSchedMaxSlots;
  int ex = 0;  // exchanges through shared memory so far
  const int lane = tid & 31;
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = sched_key(surv, tid * E + e, n);
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int f = e ^ j;
          if (f > e) {
            const bool up = ((tid * E + e) & k) == 0;
            const unsigned long long lo = v[e] < v[f] ? v[e] : v[f], hi = v[e] < v[f] ? v[f] : v[e];
            v[e] = up ? lo : hi;
            v[f] = up ? hi : lo;
          }
        }
      } else if (j < 32 * E) {
        const int lm = j / E;  // partner lane distance
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = tid * E + e;
          const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, v[e], lm);
          const bool keep_min = ((i & k) == 0) == ((lane & lm) == 0);
          v[e] = keep_min ? (v[e] < o ? v[e] : o) : (v[e] < o ? o : v[e]);
        }
      } else {
        unsigned long long* xb = (kTwoBuffers && (ex & 1)) ? out + N : out;
        if (!kTwoBuffers) __syncthreads();  // earlier readers of `out` are done
#pragma unroll
        for (int e = 0; e < E; ++e) xb[tid * E + e] = v[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = tid * E + e;
          const unsigned long long o = xb[i ^ j];
          const bool keep_min = ((i & k) == 0) == ((i & j) == 0);
          v[e] = keep_min ? (v[e] < o ? v[e] : o) : (v[e] < o ? o : v[e]);
        }
        ++ex;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e) out[tid * E + e] = v[e];
}

// Ascending bitonic sort of each warp's 32 E keys (thread t holds keys t E .. t E + E - 1) in
// registers: exchanges at distance j < E inside the thread, longer ones by warp shuffles.  The
// last stage sorts every warp's run ascending (instead of alternating the directions).
template <int E>
__device__ __forceinline__ void warp_bitonic(unsigned long long (&v)[E], int tid) {
  constexpr int R = 32 * E;
  const int lane = tid & 31;
#pragma unroll
  for (int k = 2; k <= R; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int f = e ^ j;
          if (f > e) {
            const bool up = (k == R) || (((tid * E + e) & k) == 0);
            const unsigned long long lo = v[e] < v[f] ? v[e] : v[f], hi = v[e] < v[f] ? v[f] : v[e];
            v[e] = up ? lo : hi;
            v[f] = up ? hi : lo;
          }
        }
      } else {
        const int lm = j / E;  // partner lane distance
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, v[e], lm);
          const bool up = (k == R) || (((tid * E + e) & k) == 0);
          const bool keep_min = up == ((lane & lm) == 0);
          v[e] = keep_min ? (v[e] < o ? v[e] : o) : (v[e] < o ? o : v[e]);
        }
      }
    }
  }
}

// Ascending sort of the keys of slots 0 .. 1024 E - 1 by the 1024 threads of the block, for
// 2 N <= kSchedMaxSlots (N = 1024 E): each warp sorts its 32 E keys in registers, then merge
// rounds double the sorted runs up to N.  In a round a key's place in the merged run is its
// place in its own run plus the number of keys of the partner run below it (a branch-free
// binary search in shared memory: keys are distinct, the slot index being part of each), so the
// result is the unique ascending order, and a round is one barrier.  The sorted keys end in
// buf[0 .. N).
template <int E>
__device__ void merge_sort(const float* __restrict__ surv, int n, unsigned long long* buf, int tid) {
  constexpr int N = 1024 * E;
  static_assert(2 * N <= kSchedMaxSlots && (E == 1 || E == 2), "the merge sort ping-pongs between two halves of the buffer");
  unsigned long long* src = buf;
  unsigned long long* dst = buf + N;
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = sched_key(surv, tid * E + e, n);
  warp_bitonic<E>(v, tid);
#pragma unroll
  for (int e = 0; e < E; ++e) src[tid * E + e] = v[e];
  constexpr int LG = E == 1 ? 10 : 11;  // log2 N
  constexpr int S0 = E == 1 ? 5 : 6;    // log2 of the warp runs
#pragma unroll
  for (int s = S0; s < LG; ++s) {  // unrolled: each round's search length is a constant
    const int L = 1 << s;
    __syncthreads();  // src is complete (and dst no longer read by the previous round)
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int idx = tid * E + e;
      const unsigned long long key = src[idx];
      const int run = idx >> s;
      const unsigned long long* pr = src + ((run ^ 1) << s);  // the partner run
      int c = 0;  // keys of the partner run below key
#pragma unroll
      for (int h = L >> 1; h > 0; h >>= 1)
        if (pr[c + h - 1] < key) c += h;
      if (pr[c] < key) ++c;
      dst[((run >> 1) << (s + 1)) + (idx & (L - 1)) + c] = key;
    }
    unsigned long long* t = src;
    src = dst;
    dst = t;
  }
  __syncthreads();
  if (src != buf) {  // an odd number of rounds: copy the result down
#pragma unroll
    for (int e = 0; e < E; ++e) buf[tid * E + e] = src[tid * E + e];
    __syncthreads();
  }
}

// Shared state of one scheduler block.
struct SchedShared {
  unsigned long long buf[kSchedMaxSlots];  // sorted keys, then prefix sums (radix histogram)
  unsigned short slot[kSchedMaxSlots];     // slot index r * gamma + j of rank i
  long long wsum[32];
  long long red_v[32];
  int red_k[32];
  int win[DSPARK_MAX_BS];
  int kstar;
};

// The synchronous search: ranks the slots (sh.slot), forms the fixed-point prefix sums and
// returns K* of `mode` (also in sh.kstar); Theta(K*) goes to theta_out unless it is null.
// Zeroes sh.win.
__device__ int sched_search(const float* __restrict__ surv, int bs, int gamma,
                            const double* __restrict__ sps, int m_max, int mode, SchedShared& sh,
                            double* __restrict__ theta_out, uint32_t* status) {
  const int tid = threadIdx.x;
  const int n = bs * gamma;
  unsigned long long* src = sh.buf;
  unsigned short* slot = sh.slot;
  long long* wsum = sh.wsum;
  int* red_k = sh.red_k;
  long long* red_v = sh.red_v;
  int* win = sh.win;

  // Sort of the n keys padded with sentinels (above every real key: survival 0 has high word
  // 0xFFFFFFFF, real slot indices are below 4096) to N = max(1024, 2^ceil(log2 n)) <= 4096: the
  // merge sort up to N = 2048, the bitonic network (registers, warp shuffles, one shared buffer)
  // for N = 4096.  Both give the unique ascending order of the distinct keys.
  // the table is read after the sort: pulled into L2 now (16 doubles per 128-byte line)
  for (int i = tid * 16; i <= m_max; i += kSchedThreads * 16) prefetch_l2(sps + i);
  int lg_n = 10;
  while ((1 << lg_n) < n) ++lg_n;
  const int N = 1 << lg_n;
  for (int e = tid; e < DSPARK_MAX_BS; e += kSchedThreads) win[e] = 0;
  if (N == 1024) merge_sort<1>(surv, n, src, tid);
  else if (N == 2048) merge_sort<2>(surv, n, src, tid);
  else bitonic_sort<4>(surv, n, src, tid);
  __syncthreads();
  unsigned long long* key = src;  // sorted keys, then inclusive prefix sums
  // fixed-point values in sorted order, 4 consecutive per thread, then an exclusive block scan
  long long v[4];
  long long run = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = tid * 4 + q;
    long long x = 0;
    if (i < n) {
      const unsigned long long kv = key[i];
      slot[i] = static_cast<unsigned short>(kv & 0xFFFFFFFFu);
      x = fix40(0xFFFFFFFFu - static_cast<uint32_t>(kv >> 32));  // floor(a * 2^40), a >= 0
    }
    run += x;
    v[q] = run;  // inclusive within the thread
  }
  const int lane = tid & 31, warp = tid >> 5;
  long long incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long t = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    wsum[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const long long base = (incl - run) + (warp > 0 ? wsum[warp - 1] : 0ll);
  // each thread overwrites only the keys it read itself: no barrier needed before
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = tid * 4 + q;
    if (i < n) key[i] = static_cast<unsigned long long>(base + v[q]);  // S_{i+1}
  }
  __syncthreads();

  const int kmax = min(n, m_max - bs);
  // Theta(K) = tau(K) sps[bs + K], tau(K) = (bs 2^40 + S_K) 2^-40 formed exactly from the bits
  // (the integer stays below 2^53), so the one fp64 operation is the rounded product.
  // Candidates compare as order-preserving integers of the doubles; a NaN Theta never wins
  // and stops the early-stop scan (the host-built tables are finite and non-negative).
  auto theta = [&](int K) -> double {
    const long long T = static_cast<long long>(bs) * (1ll << 40) + ((K == 0) ? 0ll : static_cast<long long>(key[K - 1]));
    return __dmul_rn(scaled_fixed(T), sps[bs + K]);
  };
  int cand = INT_MAX;
  long long best_v = LLONG_MIN;
  int best_k = INT_MAX;
  bool bad_table = false;
  for (int K = tid; K <= kmax; K += kSchedThreads) {
    // the table entries the search reads must be finite, non-negative and non-increasing in M
    // (dspark_build_sps makes them so); a table that is not is reported, the search still runs
    // (integer tests on the bits: this part's fp64 pipe is narrow) s0 finite and >= 0 (or -0),
    // and the next entry not NaN and not above it
    const double s0 = sps[bs + K];
    const long long b0 = __double_as_longlong(s0);
    bool ok = (b0 >= 0 && b0 < 0x7FF0000000000000ll) || b0 == static_cast<long long>(0x8000000000000000ull);
    if (K < kmax) {
      const double s1 = sps[bs + K + 1];
      ok = ok && !dnan(s1) && dkey(s1) <= dkey(s0);
    }
    if (!ok) bad_table = true;
    const double t0 = theta(K);
    if (mode == DSPARK_SCHED_EARLY_STOP) {
      if (K < kmax) {
        const double t1 = theta(K + 1);
        if (dnan(t0) || dnan(t1) || !(dkey(t1) > dkey(t0))) cand = min(cand, K);
      }
    } else if (!dnan(t0)) {
      const long long v0 = dkey(t0);
      if (v0 > best_v || (v0 == best_v && K < best_k)) {
        best_v = v0;
        best_k = K;
      }
    }
  }
  // block reductions (min for early stop; argmax with lowest K for the global search)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cand = min(cand, __shfl_xor_sync(0xFFFFFFFFu, cand, o));
    const long long ov = __shfl_xor_sync(0xFFFFFFFFu, best_v, o);
    const int ok = __shfl_xor_sync(0xFFFFFFFFu, best_k, o);
    if (ov > best_v || (ov == best_v && ok < best_k)) {
      best_v = ov;
      best_k = ok;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad_table) && lane == 0) set_status(status, DSPARK_EINVAL);
  if (lane == 0) {
    red_k[warp] = (mode == DSPARK_SCHED_EARLY_STOP) ? cand : best_k;
    red_v[warp] = best_v;
  }
  __syncthreads();
  if (tid == 0) {
    int ks;
    if (mode == DSPARK_SCHED_EARLY_STOP) {
      ks = INT_MAX;
      for (int i = 0; i < 32; ++i) ks = min(ks, red_k[i]);
      if (ks == INT_MAX) ks = kmax;
    } else {
      long long bv = red_v[0];
      ks = red_k[0];
      for (int i = 1; i < 32; ++i)
        if (red_v[i] > bv || (red_v[i] == bv && red_k[i] < ks)) {
          bv = red_v[i];
          ks = red_k[i];
        }
      if (ks == INT_MAX) ks = 0;  // every Theta NaN
    }
    sh.kstar = ks;
    if (theta_out) *theta_out = theta(ks);
  }
  __syncthreads();
  return sh.kstar;
}

// window[r] = how many of the first K ranked slots (sh.slot) belong to request r.
__device__ void sched_windows(SchedShared& sh, int K, int bs, int gamma, int32_t* __restrict__ window) {
  const int tid = threadIdx.x;
  for (int i = tid; i < K; i += kSchedThreads) atomicAdd(&sh.win[sh.slot[i] / gamma], 1);
  __syncthreads();
  for (int r = tid; r < bs; r += kSchedThreads) window[r] = sh.win[r];
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(
    const float* __restrict__ surv, int bs, int gamma, const double* __restrict__ sps, int m_max,
    int mode, int32_t* __restrict__ window, int32_t* __restrict__ K_out,
    double* __restrict__ theta_out, uint32_t* status) {
  __shared__ SchedShared sh;
  pdl_enter();
  const int ks = sched_search(surv, bs, gamma, sps, m_max, mode, sh, theta_out, status);
  if (threadIdx.x == 0) *K_out = ks;
  if (window) sched_windows(sh, ks, bs, gamma, window);
}

cudaError_t launch_schedule(const float* surv, int bs, int gamma, const double* sps, int m_max,
                            int mode, int32_t* window, int32_t* K_out, double* theta_out,
                            uint32_t* status, cudaStream_t s) {
  return launch_pdl(schedule_kernel, dim3(1), dim3(kSchedThreads), 0, s, surv, bs, gamma, sps, m_max, mode, window,
                    K_out, theta_out, status);
}

// ---------------------------------------------------------------------------------------
// S3 under zero-overhead scheduling.  DSpark technical summary, "Infra" (scheduler bullet);
// DSpark in SGLang, "ZOS": the verify budget of step t is predicted from the confidence of
// step t - 2, while the current candidates are still ranked by the current survival; with the
// stale budget the search over the table is global (no early stop).
// The budget of a step is the global search above (schedule_kernel without windows), written
// to slot step & 1 of a two-entry device ring; the select of step t reads slot t & 1 before
// the budget of step t overwrites it.  The select needs no prefix sums and no full order: a
// three-pass radix selection (11, 11, 10 bits of the descending-survival key) finds the K
// smallest keys, equal keys going to the lower slot index, as in the full ranking.
// ---------------------------------------------------------------------------------------
constexpr int kRadixBins = 2048;

// Exclusive block-wide prefix sum of one int per thread over the 1024 threads; the block
// total goes to *total.  `wtot` holds 32 ints of shared memory.
__device__ __forceinline__ int block_excl_scan(int x, int* wtot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = wtot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    wtot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int res = incl - x + (warp > 0 ? wtot[warp - 1] : 0);
  *total = wtot[31];
  __syncthreads();  // wtot may be reused
  return res;
}

__global__ void __launch_bounds__(kSchedThreads) zos_select_kernel(
    const float* __restrict__ surv, int bs, int gamma, const double* __restrict__ sps, int m_max,
    const int32_t* __restrict__ ring, uint64_t step, int32_t* __restrict__ window,
    int32_t* __restrict__ K_out, uint32_t* status) {
  __shared__ SchedShared sh;
  __shared__ int s_K, s_bin, s_before;
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = bs * gamma;
  const int kmax = min(n, m_max - bs);
  if (tid == 0) s_K = ring[step & 1];
  for (int e = tid; e < DSPARK_MAX_BS; e += kSchedThreads) sh.win[e] = 0;
  __syncthreads();
  if (s_K < 0) {  // no budget recorded two steps back: the global search over this survival
    const int ks = sched_search(surv, bs, gamma, sps, m_max, DSPARK_SCHED_GLOBAL_ARGMAX, sh, nullptr, status);
    if (tid == 0) *K_out = ks;
    sched_windows(sh, ks, bs, gamma, window);
    return;
  }
  const int K = min(s_K, kmax);

  // Thread t holds slots t E .. t E + E - 1 (E <= 4): key = ~bits of the survival (negatives
  // rank as 0), state 0 undecided, 1 admitted, 2 not admitted.
  const int E = (n + kSchedThreads - 1) / kSchedThreads;
  uint32_t key[4];
  int st[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int i = tid * E + e;
    key[e] = 0u;
    st[e] = 2;
    if (e < E && i < n) {
      uint32_t bits = __float_as_uint(surv[i]);
      if (bits & 0x80000000u) bits = 0u;
      key[e] = 0xFFFFFFFFu - bits;
      st[e] = 0;
    }
  }
  int* hist = reinterpret_cast<int*>(sh.buf);  // kRadixBins ints
  int* wtot = sh.red_k;
  int need = K;  // undecided slots still to admit; the undecided ones number at least `need`
  for (int pass = 0; pass < 3 && need > 0; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t mask = pass == 2 ? 0x3FFu : 0x7FFu;
    hist[tid] = 0;
    hist[tid + kSchedThreads] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 4; ++e) {  // warp-aggregated histogram of the undecided keys' digits
      const bool live = st[e] == 0;
      const uint32_t d = live ? ((key[e] >> shift) & mask) : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, d);
      if (live && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
    }
    __syncthreads();
    const int h0 = hist[2 * tid], h1 = hist[2 * tid + 1];
    int total;
    const int ex = block_excl_scan(h0 + h1, wtot, &total);
    // the digit holding the need-th smallest undecided key
    if (ex < need && need <= ex + h0) {
      s_bin = 2 * tid;
      s_before = ex;
    } else if (ex + h0 < need && need <= ex + h0 + h1) {
      s_bin = 2 * tid + 1;
      s_before = ex + h0;
    }
    __syncthreads();
    const uint32_t bin = static_cast<uint32_t>(s_bin);
    need -= s_before;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (st[e] != 0) continue;
      const uint32_t d = (key[e] >> shift) & mask;
      st[e] = d < bin ? 1 : (d > bin ? 2 : 0);
    }
  }
  // The undecided slots share one key: the first `need` of them in slot order are admitted.
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) cnt += st[e] == 0;
  int total;
  int rank = block_excl_scan(cnt, wtot, &total);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (st[e] != 0) continue;
    st[e] = rank < need ? 1 : 2;
    ++rank;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (st[e] == 1) atomicAdd(&sh.win[(tid * E + e) / gamma], 1);
  __syncthreads();
  for (int r = tid; r < bs; r += kSchedThreads) window[r] = sh.win[r];
  if (tid == 0) *K_out = K;
}

cudaError_t launch_zos_select(const float* surv, int bs, int gamma, const double* sps, int m_max,
                              const int32_t* ring, uint64_t step, int32_t* window, int32_t* K_out,
                              uint32_t* status, cudaStream_t s) {
  return launch_pdl(zos_select_kernel, dim3(1), dim3(kSchedThreads), 0, s, surv, bs, gamma, sps, m_max, ring, step,
                    window, K_out, status);
}

cudaError_t launch_zos_budget(const float* surv, int bs, int gamma, const double* sps, int m_max,
                              int32_t* ring, uint64_t step, uint32_t* status, cudaStream_t s) {
  return launch_pdl(schedule_kernel, dim3(1), dim3(kSchedThreads), 0, s, surv, bs, gamma, sps, m_max,
                    int(DSPARK_SCHED_GLOBAL_ARGMAX), static_cast<int32_t*>(nullptr), ring + (step & 1),
                    static_cast<double*>(nullptr), status);
}

// ---------------------------------------------------------------------------------------
// S4.  DSpark in SGLang, "Ragged verify under full CUDA graphs" (Fig. 2): requests are
// packed front to back into a cu_seqlens buffer and the total is rounded up to the nearest
// captured tier.  One block; thread r owns request r.
// ---------------------------------------------------------------------------------------
// The pack of one block of any size (a multiple of 32, at least bs threads; every thread takes
// part in the barriers): request r is thread r.
__device__ void pack_block(const int32_t* window, const int32_t* __restrict__ anchor,
                           const int32_t* __restrict__ tokens, int bs, int gamma, const int32_t* __restrict__ tiers,
                           int n_tiers, int cap, int32_t* __restrict__ cu, int32_t* __restrict__ ids,
                           int32_t* __restrict__ req, int32_t* __restrict__ pos, int32_t* __restrict__ padded_out,
                           uint32_t* status) {
  __shared__ int wsum[32];
  __shared__ int s_padded, s_M, s_bad;
  __shared__ unsigned long long s_first;  // (index << 32) | value of the first tier >= M
  const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
  if (r == 0) {
    s_bad = 0;
    s_first = ~0ull;
  }
  __syncthreads();
  // the tiers must be positive and strictly increasing (the search below takes the first >= M)
  for (int i = r; i < n_tiers; i += blockDim.x)
    if (tiers[i] <= (i > 0 ? tiers[i - 1] : 0)) atomicExch(&s_bad, 1);
  int l = 0;
  if (r < bs) {
    l = window ? window[r] : gamma;
    if (l < 0 || l > gamma) {
      atomicExch(&s_bad, 1);
      l = 0;
    }
  }
  const int n = (r < bs) ? l + 1 : 0;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int i = 0; i < warp; ++i) base += wsum[i];
  const int start = base + incl - n;
  if (r < bs) cu[r] = start;
  if (r == bs - 1) {
    cu[bs] = start + n;
    s_M = start + n;
  }
  __syncthreads();
  // the first tier >= M, found by all threads at once (a serial scan would be one dependent load
  // per tier)
  for (int i = r; i < n_tiers; i += blockDim.x) {
    const int t = tiers[i];
    if (t >= s_M) atomicMin(&s_first, (static_cast<unsigned long long>(i) << 32) | static_cast<uint32_t>(t));
  }
  __syncthreads();
  if (r == 0) {
    const int M = s_M;
    int padded = M;
    if (n_tiers > 0) padded = (s_first == ~0ull) ? -1 : static_cast<int>(static_cast<uint32_t>(s_first));
    if (s_bad || padded < 0 || padded > cap) {
      set_status(status, DSPARK_EINVAL);
      padded = -1;
    }
    s_padded = padded;
    *padded_out = padded;
  }
  __syncthreads();
  const int padded = s_padded;
  if (padded < 0) return;
  if (r < bs) {
    for (int j = 0; j <= l; ++j) {
      const int p = start + j;
      ids[p] = (j == 0) ? anchor[r] : tokens[size_t(r) * gamma + j - 1];
      req[p] = r;
      pos[p] = j;
    }
  }
  for (int p = s_M + r; p < padded; p += blockDim.x) {
    ids[p] = -1;
    req[p] = -1;
    pos[p] = -1;
  }
}

__global__ void __launch_bounds__(DSPARK_MAX_BS) pack_kernel(
    const int32_t* __restrict__ window, const int32_t* __restrict__ anchor,
    const int32_t* __restrict__ tokens, int bs, int gamma, const int32_t* __restrict__ tiers,
    int n_tiers, int cap, int32_t* __restrict__ cu, int32_t* __restrict__ ids,
    int32_t* __restrict__ req, int32_t* __restrict__ pos, int32_t* __restrict__ padded_out,
    uint32_t* status) {
  pdl_enter();
  pack_block(window, anchor, tokens, bs, gamma, tiers, n_tiers, cap, cu, ids, req, pos, padded_out, status);
}

// S3 then S4 in one block: the windows the search writes are packed by the same block (one launch
// and one kernel boundary fewer per step than schedule_kernel + pack_kernel).
__global__ void __launch_bounds__(kSchedThreads) schedule_pack_kernel(
    const float* __restrict__ surv, int bs, int gamma, const double* __restrict__ sps, int m_max, int mode,
    int32_t* __restrict__ window, int32_t* __restrict__ K_out, double* __restrict__ theta_out,
    const int32_t* __restrict__ anchor, const int32_t* __restrict__ tokens, const int32_t* __restrict__ tiers,
    int n_tiers, int cap, int32_t* __restrict__ cu, int32_t* __restrict__ ids, int32_t* __restrict__ req,
    int32_t* __restrict__ pos, int32_t* __restrict__ padded_out, uint32_t* status) {
  __shared__ SchedShared sh;
  pdl_enter();
  // the pack's inputs are pulled into L2 while the search runs
  for (int i = threadIdx.x * 32; i < n_tiers; i += kSchedThreads * 32) prefetch_l2(tiers + i);
  for (int i = threadIdx.x * 32; i < bs; i += kSchedThreads * 32) prefetch_l2(anchor + i);
  for (int i = threadIdx.x * 32; i < bs * gamma; i += kSchedThreads * 32) prefetch_l2(tokens + i);
  const int ks = sched_search(surv, bs, gamma, sps, m_max, mode, sh, theta_out, status);
  if (threadIdx.x == 0) *K_out = ks;
  sched_windows(sh, ks, bs, gamma, window);
  __syncthreads();
  // the pack reads the windows from shared memory (sh.win, complete after the barrier in
  // sched_windows), not back from the global copy this block has just written
  pack_block(sh.win, anchor, tokens, bs, gamma, tiers, n_tiers, cap, cu, ids, req, pos, padded_out, status);
}

cudaError_t launch_pack(const int32_t* window, const int32_t* anchor, const int32_t* tokens,
                        int bs, int gamma, const int32_t* tiers, int n_tiers, int cap,
                        int32_t* cu, int32_t* ids, int32_t* req, int32_t* pos, int32_t* padded,
                        uint32_t* status, cudaStream_t s) {
  return launch_pdl(pack_kernel, dim3(1), dim3(DSPARK_MAX_BS), 0, s, window, anchor, tokens, bs, gamma, tiers,
                    n_tiers, cap, cu, ids, req, pos, padded, status);
}

cudaError_t launch_schedule_pack(const float* surv, int bs, int gamma, const double* sps, int m_max, int mode,
                                 int32_t* window, int32_t* K_out, double* theta_out, const int32_t* anchor,
                                 const int32_t* tokens, const int32_t* tiers, int n_tiers, int cap, int32_t* cu,
                                 int32_t* ids, int32_t* req, int32_t* pos, int32_t* padded, uint32_t* status,
                                 cudaStream_t s) {
  return launch_pdl(schedule_pack_kernel, dim3(1), dim3(kSchedThreads), 0, s, surv, bs, gamma, sps, m_max, mode,
                    window, K_out, theta_out, anchor, tokens, tiers, n_tiers, cap, cu, ids, req, pos, padded, status);
}

}  // namespace dspark
