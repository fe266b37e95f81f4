// Host-side helpers of the tensor-core passes: the driver's tensor-map encoder (looked up once),
// per-device caches, and 2-D bf16 tensor maps with the 128-byte swizzle.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace dspark {
namespace tch {

constexpr int kMaxDevices = 64;

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

inline int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

// Multiprocessor count of the current device (queried once per device).
inline int sm_count() {
  static int cache[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

// Row-major bf16 matrix [rows, cols] as a 2-D tensor map whose box is `box_rows` rows of 64
// columns (128 bytes, the swizzle span).  Out-of-range elements of a box read as zero.
inline bool encode_bf16_2d(CUtensorMap* map, const void* base, size_t rows, size_t cols, int box_rows) {
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  const cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opt a kernel into `bytes` of dynamic shared memory, once per device.
template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, bool* done, std::mutex* mu) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(*mu);
  if (!done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

// Persistent grid of the vocabulary passes: one CTA per SM, a whole number of CTAs per
// 128-request M-tile, at most one per (M-tile, chunk).  CTA b takes M-tile b % n_mt and chunks
// b / n_mt + j * (grid / n_mt).
inline int vocab_grid(int bs, int n_chunks) {
  const int n_mt = (bs + 127) / 128;
  const int grid = (sm_count() / n_mt) * n_mt;
  const int lim = n_mt * n_chunks;
  return grid < n_mt ? n_mt : (grid > lim ? lim : grid);
}

}  // namespace tch
}  // namespace dspark
