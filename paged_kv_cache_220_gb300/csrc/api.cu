// Library-wide C entry points: error word registration, status strings, the
// bounded-wait self-test.
#include <atomic>

#include "common.cuh"
#include "host_util.h"

namespace pkv {
static std::atomic<int*> g_dev_err{nullptr};
int* device_error_ptr() { return g_dev_err.load(std::memory_order_relaxed); }
}  // namespace pkv

extern "C" int pkv_set_device_check(int* dev_error_flag) {
  pkv::g_dev_err.store(dev_error_flag, std::memory_order_relaxed);
  return PKV_OK;
}

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_OUT_OF_BLOCKS: return "out of KV blocks";
    case PKV_ERR_NOT_FOUND: return "unknown sequence";
    case PKV_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

extern "C" int pkv_version(void) { return 100; }

namespace pkv {

// An mbarrier that expects one arrival nobody makes: the bounded wait gives up
// after limit_ns, records PKV_DEVERR_WAIT_TIMEOUT and the kernel returns.
__global__ void wait_timeout_selftest_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, err, limit_ns);
}

}  // namespace pkv

extern "C" int pkv_selftest_wait_timeout(int* dev_error_flag, int limit_us, void* stream) {
  if (!dev_error_flag || limit_us <= 0 || limit_us > 2000000) return PKV_ERR_INVALID_ARG;
  pkv::wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      dev_error_flag, static_cast<unsigned long long>(limit_us) * 1000ull);
  return pkv::launch_status();
}
