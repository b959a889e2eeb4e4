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
// the call allocates nothing, and a query that reads the status word the
// step's kernels leave at the start of that array.
//
// The array is MFSDP_STATIC_SCRATCH_BYTES (64 MiB) on every GPU that loads the
// library, held until the process exits.  Its host-side name is only a
// stand-in for the device array: host code must not hand it to a kernel.  The
// device address is looked up with cudaGetSymbolAddress, with the device
// current, once per device and CUDA context: module globals belong to a
// context, so the cache is keyed by the context's unique id and a new context
// on the device (after cudaDeviceReset, or a context the caller made current)
// gets its own lookup instead of a stale address.
#include <cuda.h>

#include <mutex>

#include "mfsdp.h"
#include "mfsdp_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MFSDP_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct ScratchCache {
  unsigned long long ctx_id = 0;   // the context the address belongs to (0: none cached)
  void* addr = nullptr;
};

std::mutex g_scratch_mutex;
ScratchCache g_scratch[kMaxDevices];

// The CUDA driver API's context queries, looked up once through the runtime (the
// library links no driver library).  Null when the driver lacks them; the
// address is then looked up on every call.
struct CtxQueries {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxQueries& ctx_queries() {
  static const CtxQueries q = [] {
    CtxQueries r;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &res) == cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      r.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &res) == cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      r.get_id = reinterpret_cast<CtxGetIdFn>(f);
    return r;
  }();
  return q;
}

// Unique id of the calling thread's current context, 0 when there is none
// (or it cannot be queried).
unsigned long long current_ctx_id() {
  const CtxQueries& q = ctx_queries();
  if (!q.get_current || !q.get_id) return 0;
  CUcontext ctx = nullptr;
  if (q.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (q.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's current
// context (set-up on the first use in that context).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MFSDP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchCache& c = g_scratch[dev];
  const unsigned long long id = current_ctx_id();
  if (!c.addr || id == 0 || id != c.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MFSDP_ERR_CUDA;
    // the lookup makes the device's context current if none was: key the
    // cache by that context
    c.addr = p;
    c.ctx_id = id != 0 ? id : current_ctx_id();
  }
  *out = c.addr;
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

extern "C" int mfsdp_muon_static_scratch_status(void* stream, int32_t* detail) {
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != MFSDP_OK) return st;
  // The status word is the first word of the scratch array, exactly as it is
  // the first word of a caller's workspace.
  return mfsdp_muon_device_status(scratch, stream, detail);
}
