// A variant of the extended step (per-block step counters, locked blocks,
// per-block sum of g^2) for callers that cannot allocate device memory.
//
// The extended step needs device scratch for its sum-of-squares reduction.
// Normally the caller allocates it (lst_workspace_bytes) and passes it in.
// Some callers cannot: a plugin running inside a host application whose
// device memory is owned by another allocator, a training loop that has
// handed all device memory to a framework's caching pool, or code that must
// not allocate once it is running. For them this file keeps the scratch in a
// file-scope device array, created when the library's device code is loaded
// on a GPU and held there until the process exits.
#include <mutex>

#include "lst_internal.h"

namespace lst {

// Scratch of the sum-of-squares reduction: a reserved 256-byte header and
// one 8-byte partial sum per (CTA, block) of one launch (1024 CTAs x 128 blocks):
// 1 MiB + 256 bytes per device.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kWorkspaceBytes];

constexpr int kMaxDevicesNoAlloc = 64;
static void* g_noalloc_ptr[kMaxDevicesNoAlloc];
static std::mutex g_noalloc_mu;

// Device address of the array on the current device. The name
// g_noalloc_workspace is only a host-side handle: passing it to a kernel
// would hand the device a host address. So, once per device and with that
// device current, ask the runtime for the array's device address. The address
// is kept for the life of the process: it belongs to the device's primary
// context (the one the CUDA runtime uses), and stays valid as long as that
// context does, i.e. until cudaDeviceReset.
static cudaError_t noalloc_workspace(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevicesNoAlloc) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (err != cudaSuccess) return err;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace lst

using namespace lst;

extern "C" lst_status lst_adamw_step_ex_noalloc(const lst_layout* L, void* const* dev_blocks,
                                                const lst_adamw_hparams* hp, const int64_t* block_steps,
                                                const uint8_t* skip, double* grad_sq, void* cuda_stream) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_adamw_step_ex_noalloc: null layout");
  if (!hp) return fail(LST_ERR_INVALID_ARG, "lst_adamw_step_ex_noalloc: null hparams");
  Scalars s;
  if (!make_scalars(*hp, &s))
    return fail(LST_ERR_INVALID_ARG,
                "lst_adamw_step_ex_noalloc: hyperparameters outside their domain (step >= 1, 0 <= beta < 1, finite)");
  void* ws = nullptr;
  if (grad_sq) {
    // The array holds the partial sums of one launch (up to 128 blocks). A
    // step over more blocks runs as several launches on the one stream, each
    // update launch after the first starting only once the previous launch's
    // reduce has finished reading the array, so any number of blocks share it.
    cudaError_t err = noalloc_workspace(&ws);
    if (err != cudaSuccess) return cuda_fail(err, "lst_adamw_step_ex_noalloc: scratch address");
  }
  lst_step_options o;
  o.block_steps = block_steps;
  o.skip = skip;
  o.grad_sq = grad_sq;
  o.workspace = ws;
  return lst_adamw_step_ex(L, dev_blocks, hp, &o, cuda_stream);
}
