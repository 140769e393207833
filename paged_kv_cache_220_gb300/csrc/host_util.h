// Host-side argument checks shared by the C entry points.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

#include "../../include/pagedkv.h"

namespace pkv {

// Device error word registered with pkv_set_device_check (may be null).
int* device_error_ptr();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int elem_bytes(int dtype) { return dtype == PKV_DTYPE_FP8_E4M3 ? 1 : 2; }

// Shape checks common to every call that touches a pool.
inline int check_cache_desc(const pkv_cache_desc& c) {
  if (c.num_blocks <= 0 || c.num_kv_heads <= 0 || c.block_size <= 0 || c.head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (c.dtype != PKV_DTYPE_BF16 && c.dtype != PKV_DTYPE_FP8_E4M3) return PKV_ERR_INVALID_ARG;
  if (c.block_size != 16 && c.block_size != 32) return PKV_ERR_UNSUPPORTED;
  if (c.head_dim != 128 && c.head_dim != 256) return PKV_ERR_UNSUPPORTED;
  if (c.num_kv_heads > 32) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Launch as a programmatic dependent of the kernel before it on the stream:
// the CTAs may be scheduled before that kernel completes, and the kernel must
// call wait_prerequisite() before reading anything that kernel wrote.
template <typename... Params, typename... Args>
inline int launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) != cudaSuccess)
    return PKV_ERR_CUDA;
  return launch_status();
}

// Per-device flags of one-time set-up steps, safe to read and set from
// several host threads (two first calls may both do the set-up; every step
// guarded this way is idempotent).
using DeviceFlags = std::atomic<bool>[64];
constexpr int kMaxFlagDevices = 64;

// Raise a kernel's dynamic shared-memory limit once per device.
template <typename Kernel>
inline int ensure_smem(Kernel k, size_t bytes, DeviceFlags& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 0 && dev < kMaxFlagDevices && done[dev].load(std::memory_order_acquire))
    return PKV_OK;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (dev >= 0 && dev < kMaxFlagDevices) done[dev].store(true, std::memory_order_release);
  return PKV_OK;
}

}  // namespace pkv
