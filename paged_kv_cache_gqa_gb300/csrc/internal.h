// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/mtkv.h"

namespace mtkv {

// Record `msg` as the calling thread's last error and return `st`.
mt_status fail(mt_status st, const std::string &msg);
// Clear the calling thread's last error and return MT_OK.
mt_status ok();
// Map a CUDA error to MT_ERR_CUDA with context (MT_OK for cudaSuccess).
mt_status cuda_check(cudaError_t e, const char *what);

// Cached device properties of the current device.
struct DeviceInfo {
  int device;
  int n_sm;
  int smem_optin;  // max dynamic shared memory per block (opt-in)
};
mt_status device_info(DeviceInfo *out);

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device (a per-device setting): cached per (device, kernel) behind a
// mutex, the return code checked. With max_carveout the kernel also prefers
// the largest shared-memory carveout.
mt_status kernel_smem(const void *kern, int bytes, const char *what, bool max_carveout = false);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace mtkv
