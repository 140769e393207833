// Library-wide C entry points: error word registration, status strings.
#include <atomic>

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
