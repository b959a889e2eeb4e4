// Owner-local Muon step for callers that cannot allocate device memory.
//
// The regular entry point takes its scratch space (the Newton-Schulz iterates,
// the Gram and polynomial matrices, the norm partials) as a caller-provided
// workspace.  Some callers have no way to provide one: code that runs inside a
// host framework which owns every device allocation through its own pool and
// gives plug-ins no allocator, a callback that is not allowed to allocate (an
// allocation there could synchronise the device or fail under memory
// pressure), or a C program that links only this library.  This file gives
// them one entry point whose scratch is a fixed, file-scope device array, so
// the call allocates nothing.
//
// The array is MFSDP_STATIC_SCRATCH_BYTES (64 MiB) on every GPU that loads the
// library, held until the process exits.  Its host-side name is only a
// stand-in for the device array: host code must not hand it to a kernel.  The
// device address is looked up once per device with cudaGetSymbolAddress, with
// that device current, and cached.
#include <mutex>

#include "mfsdp.h"
#include "mfsdp_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MFSDP_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array (set-up on first use).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MFSDP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MFSDP_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MFSDP_OK;
}

}  // namespace

extern "C" int mfsdp_muon_owner_step_static_scratch(const mfsdp_matrix_shard* shards, int32_t n_shards,
                                                    const void* grad, int32_t grad_dtype, float* momentum,
                                                    void* update, int32_t update_dtype, int64_t numel, double beta,
                                                    int32_t nesterov, int32_t ns_steps, double a, double b, double c,
                                                    double eps, void* stream) {
  // The arguments are checked on the host before the scratch array's address
  // is looked up, so they fail with the regular entry point's statuses.
  size_t need = 0;
  const int checked = mfsdp::check_step_args(shards, n_shards, grad, grad_dtype, momentum, update, update_dtype,
                                             numel, beta, nesterov, ns_steps, a, b, c, eps, &need);
  if (checked != MFSDP_OK || n_shards == 0) return checked;
  if (need > (size_t)MFSDP_STATIC_SCRATCH_BYTES) return MFSDP_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != MFSDP_OK) return st;
  return mfsdp_muon_owner_step(shards, n_shards, grad, grad_dtype, momentum, update, update_dtype, numel, beta,
                               nesterov, ns_steps, a, b, c, eps, scratch, (size_t)MFSDP_STATIC_SCRATCH_BYTES, stream);
}
