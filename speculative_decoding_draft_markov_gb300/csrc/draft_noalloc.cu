// dspark_draft_block_noalloc: the Markov block draft for callers that cannot allocate device
// memory, so cannot hand the library a workspace.  Typical cases: a plugin that runs inside
// another framework's device-memory pool (a cudaMalloc there would bypass the host
// framework's allocator and its accounting), or a service that fixes its device footprint at
// start-up and forbids any later allocation.  Such a caller still passes every input and
// output buffer; only the draft's scratch (one status word and the per-(request, slot)
// statistics of one position) comes from a fixed array that is part of the library image.
//
// The array below is a file-scope __device__ variable: every GPU on which the library is
// loaded holds kNoAllocScratchBytes for it until the process exits.  In host code its name is
// only a host-side stand-in, not a device address: a kernel handed that name would fault or,
// where the GPU can reach host memory, silently use the wrong memory.  The device address is
// therefore looked up with cudaGetSymbolAddress, once per device, with that device current;
// the first call of this entry point on a device performs that lookup, so that first call
// should come before any stream capture.
//
// The device address is cached per device for the life of the process: a cudaDeviceReset
// between calls destroys the context the address belongs to, and is not supported.
//
// Every call shares the one array and the last call's contents stay in it.  The status word
// is cleared at the start of each call (when the caller does not pass its own); the chunk
// statistics need no clearing (each position writes all of them before reading any); the
// tensor-core pass's grid-barrier words (64 bytes after the status word) start at zero, as the
// array does, and every launch leaves them at zero.  Calls
// whose work can overlap on the GPU -- on different streams, or from several host threads --
// race on the array and must be serialised by the caller.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

using namespace dspark;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSPARK_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DSPARK_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DSPARK_OK;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" DSPARK_API int dspark_draft_block_noalloc(
    const void* U, const void* W1, const void* W2t, int dtype, const int32_t* anchor, int bs, int gamma,
    int V, int r, float temperature, uint64_t seed, uint64_t step, int32_t* tokens, float* logit_x,
    float* lse, uint32_t* device_status, dspark_stream_t stream) {
  // the same argument checks as dspark_draft_block
  if (!U || !W1 || !W2t || !anchor || !tokens || !logit_x || !lse) return DSPARK_EINVAL;
  if ((dtype != DSPARK_F32 && dtype != DSPARK_BF16) || !std::isfinite(temperature) || temperature < 0.f)
    return DSPARK_EINVAL;
  if (bs < 1 || gamma < 1 || V < 8 || r < 1 || V % 8 != 0) return DSPARK_EINVAL;
  if (bs > DSPARK_MAX_BS || gamma > DSPARK_MAX_GAMMA || V >= (1 << 24)) return DSPARK_EUNSUPPORTED;
  if (!(r == 32 || r == 64 || r == 128 || r == 256)) return DSPARK_EUNSUPPORTED;
  if (!aligned(U, 16) || !aligned(W1, 16) || !aligned(W2t, 16) || !aligned(anchor, 4) ||
      !aligned(tokens, 4) || !aligned(logit_x, 4) || !aligned(lse, 4) || !aligned(device_status, 4))
    return DSPARK_EINVAL;

  // The scratch this call needs: the status word, then 16 bytes per (request, slot) of the
  // pass that will run.  The tensor-core pass (bf16, r a multiple of 64) writes one slot per
  // CTA column (at most one per SM and per 256-id tile); the CUDA-core pass one per 64-id draft
  // chunk.
  const WsLayout L = ws_layout(bs, gamma, V);
  const bool tc = draft_tc_supported(dtype, bs, V, r);
  const size_t need = L.stats + draft_stats_bytes(bs, tc ? draft_tc_slots(bs, V) : n_draft_chunks(V));
  if (need > kNoAllocScratchBytes) return DSPARK_EUNSUPPORTED;

  void* scratch = nullptr;
  if (int e = noalloc_scratch(&scratch)) return e;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(scratch);
  uint32_t* status = device_status ? device_status : reinterpret_cast<uint32_t*>(w + L.status);
  if (!device_status && cudaMemsetAsync(w + L.status, 0, sizeof(uint32_t), s) != cudaSuccess)
    return DSPARK_ECUDA;
  void* stats = w + L.stats;

  const int greedy = temperature == 0.f;
  const float inv_tau = greedy ? 1.f : static_cast<float>(1.0 / static_cast<double>(temperature));
  if (tc)  // every position in one persistent launch (grid barrier words beside the status word)
    return launch_draft_tc(U, W1, W2t, nullptr, nullptr, nullptr, nullptr, anchor, tokens, logit_x, lse, bs, gamma, V,
                           r, 1, gamma, inv_tau, greedy, seed, step, stats,
                           reinterpret_cast<uint32_t*>(w + L.status + 64), status,
                           reinterpret_cast<uint32_t*>(w + L.status + 16), s) ==
                   cudaSuccess
               ? DSPARK_OK
               : DSPARK_ECUDA;
  const int n_slots = n_draft_chunks(V);  // the CUDA-core pass: one slot per draft chunk
  for (int k = 1; k <= gamma; ++k) {
    cudaError_t e = launch_draft_stats_simt(dtype, U, W1, W2t, nullptr, anchor, tokens, bs, gamma, V, r, k, inv_tau,
                                            greedy, seed, step, stats, n_slots, s);
    if (e == cudaSuccess)
      e = launch_draft_select(dtype, stats, n_slots, U, W1, W2t, nullptr, anchor, tokens, logit_x, lse, bs, gamma, V,
                              r, k, inv_tau, greedy, seed, step, status, s);
    if (e != cudaSuccess) return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}
