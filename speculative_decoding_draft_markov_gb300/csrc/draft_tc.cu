// S1 draft statistics on the tensor cores (tcgen05 + TMEM + TMA).  Not enabled yet: the
// CUDA-core pass in draft.cu serves every dtype until this kernel passes parity.
#include "common.cuh"
#include "internal.h"

namespace dspark {

uint64_t g_wait_timeout_ns = 1000000000ull;  // 1 s; changed only through dspark_set_wait_timeout_ns

bool draft_tc_supported(int, int, int, int) { return false; }

cudaError_t launch_draft_stats_tc(const void*, const void*, const void*, const int32_t*,
                                  const int32_t*, int, int, int, int, int, float, int, void*, int,
                                  uint32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace dspark
