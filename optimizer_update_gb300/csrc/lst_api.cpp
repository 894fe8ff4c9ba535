// C ABI entry points of liblst: validation, step scalars, the device-resident
// step, host pinned allocation, status text and the host-side test hook.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include <sys/mman.h>
#include <unistd.h>

#include "lst_internal.h"

namespace lst {

static std::unordered_map<void*, size_t>& host_allocs() {
  static std::unordered_map<void*, size_t> m;
  return m;
}
static std::mutex& host_allocs_mu() {
  static std::mutex m;
  return m;
}

static thread_local char g_err[512] = "";

void clear_error() { g_err[0] = '\0'; }

lst_status fail(lst_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

lst_status cuda_fail(cudaError_t err, const char* what) {
  return fail(LST_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
}

Inject& inject() {
  static Inject s;
  return s;
}

bool valid_hparams(const lst_adamw_hparams* hp) {
  if (!hp) return false;
  if (hp->step < 1) return false;
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f)) return false;
  if (!(hp->beta2 >= 0.0f && hp->beta2 < 1.0f)) return false;
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->eps) || !std::isfinite(hp->weight_decay)) return false;
  return true;
}

// Step scalars: formed in double, rounded once to fp32 ("The Math": bias
// corrections 1 - beta^t with the global step t).
bool make_scalars(const lst_adamw_hparams& hp, Scalars* s) {
  if (!valid_hparams(&hp)) return false;
  const double b1 = hp.beta1, b2 = hp.beta2, t = (double)hp.step;
  s->beta1 = hp.beta1;
  s->beta2 = hp.beta2;
  s->one_minus_beta1 = (float)(1.0 - b1);
  s->one_minus_beta2 = (float)(1.0 - b2);
  s->bias_correction1 = (float)(1.0 - std::pow(b1, t));
  s->bias_correction2 = (float)(1.0 - std::pow(b2, t));
  s->eps = hp.eps;
  s->lr = hp.lr;
  s->decay = (float)(1.0 - (double)hp.lr * (double)hp.weight_decay);
  return true;
}

}  // namespace lst

using namespace lst;

static lst_status device_step(const lst_layout* L, void* const* dev_blocks, const Scalars& s, bool sgd,
                              void* cuda_stream, const char* who) {
  const int64_t n = (int64_t)L->blocks.size();
  if (n == 0) return LST_OK;
  if (!dev_blocks) return fail(LST_ERR_INVALID_ARG, "%s: dev_blocks is null", who);
  for (int64_t i = 0; i < n; ++i) {
    const Block& b = L->blocks[(size_t)i];
    if (b.bytes == 0) continue;
    if (!dev_blocks[i]) return fail(LST_ERR_INVALID_ARG, "%s: block %lld pointer is null", who, (long long)i);
    if (reinterpret_cast<uintptr_t>(dev_blocks[i]) % 16 != 0)
      return fail(LST_ERR_ALIGNMENT, "%s: block %lld pointer not 16-byte aligned", who, (long long)i);
  }
  std::vector<Run> runs;
  try {
    runs.reserve((size_t)n);
  } catch (...) {
    return fail(LST_ERR_OOM, "%s: out of host memory", who);
  }
  for (int64_t i = 0; i < n; ++i) {
    const Block& b = L->blocks[(size_t)i];
    if (b.padded == 0) continue;
    runs.push_back(block_run(*L, b, static_cast<char*>(dev_blocks[i]), 0, b.padded));
  }
  cudaError_t err = launch_update(L->fmt, sgd, runs.data(), (int)runs.size(), s,
                                  static_cast<cudaStream_t>(cuda_stream));
  if (err != cudaSuccess) return cuda_fail(err, who);
  return LST_OK;
}

extern "C" lst_status lst_adamw_step(const lst_layout* L, void* const* dev_blocks,
                                     const lst_adamw_hparams* hp, void* cuda_stream) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_adamw_step: null layout");
  if (!hp) return fail(LST_ERR_INVALID_ARG, "lst_adamw_step: null hparams");
  Scalars s;
  if (!make_scalars(*hp, &s))
    return fail(LST_ERR_INVALID_ARG,
                "lst_adamw_step: hyperparameters outside their domain (step >= 1, 0 <= beta < 1, finite)");
  return device_step(L, dev_blocks, s, false, cuda_stream, "lst_adamw_step");
}

extern "C" lst_status lst_sgd_step(const lst_layout* L, void* const* dev_blocks, float lr,
                                   void* cuda_stream) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_sgd_step: null layout");
  if (!std::isfinite(lr)) return fail(LST_ERR_INVALID_ARG, "lst_sgd_step: lr not finite");
  Scalars s;
  std::memset(&s, 0, sizeof(s));
  s.lr = lr;
  return device_step(L, dev_blocks, s, true, cuda_stream, "lst_sgd_step");
}

// Pinned host memory for blocks: page-aligned anonymous memory registered with
// CUDA (mapped and portable), so every block starts on a page boundary
// whatever its size (small cudaHostAlloc allocations need not be page aligned).
extern "C" int64_t lst_workspace_bytes(void) { return kWorkspaceBytes; }

namespace lst {

// Validates the options against the layout and builds, for every block that
// is not skipped, its bias corrections. Returns LST_OK or an error status.
lst_status prepare_options(const lst_layout* L, const lst_adamw_hparams& hp, const lst_step_options* o,
                           std::vector<float>* bc1, std::vector<float>* bc2, const char* who) {
  const int64_t n = (int64_t)L->blocks.size();
  bc1->assign((size_t)n, 0.0f);
  bc2->assign((size_t)n, 0.0f);
  if (o && o->grad_sq) {
    if (!o->workspace) return fail(LST_ERR_INVALID_ARG, "%s: grad_sq needs a workspace", who);
    if (reinterpret_cast<uintptr_t>(o->workspace) % 256)
      return fail(LST_ERR_ALIGNMENT, "%s: workspace not 256-byte aligned", who);
    if (reinterpret_cast<uintptr_t>(o->grad_sq) % 8)
      return fail(LST_ERR_ALIGNMENT, "%s: grad_sq not 8-byte aligned", who);
  }
  for (int64_t i = 0; i < n; ++i) {
    if (o && o->skip && o->skip[i]) continue;
    lst_adamw_hparams h = hp;
    if (o && o->block_steps) h.step = o->block_steps[i];
    Scalars s;
    if (!make_scalars(h, &s))
      return fail(LST_ERR_INVALID_ARG, "%s: block %lld: step must be >= 1", who, (long long)i);
    (*bc1)[(size_t)i] = s.bias_correction1;
    (*bc2)[(size_t)i] = s.bias_correction2;
  }
  return LST_OK;
}

}  // namespace lst

extern "C" lst_status lst_adamw_step_ex(const lst_layout* L, void* const* dev_blocks, const lst_adamw_hparams* hp,
                                        const lst_step_options* opts, void* cuda_stream) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_adamw_step_ex: null layout");
  if (!hp) return fail(LST_ERR_INVALID_ARG, "lst_adamw_step_ex: null hparams");
  Scalars s;
  if (!make_scalars(*hp, &s))
    return fail(LST_ERR_INVALID_ARG,
                "lst_adamw_step_ex: hyperparameters outside their domain (step >= 1, 0 <= beta < 1, finite)");
  std::vector<float> bc1, bc2;
  lst_status st = prepare_options(L, *hp, opts, &bc1, &bc2, "lst_adamw_step_ex");
  if (st != LST_OK) return st;
  const int64_t n = (int64_t)L->blocks.size();
  if (n == 0) return LST_OK;
  if (!dev_blocks) return fail(LST_ERR_INVALID_ARG, "lst_adamw_step_ex: dev_blocks is null");
  const bool want_sq = opts && opts->grad_sq;
  std::vector<RunEx> runs;
  for (int64_t i = 0; i < n; ++i) {
    if (opts && opts->skip && opts->skip[i]) continue;
    const Block& b = L->blocks[(size_t)i];
    if (b.bytes > 0) {
      if (!dev_blocks[i])
        return fail(LST_ERR_INVALID_ARG, "lst_adamw_step_ex: block %lld pointer is null", (long long)i);
      if (reinterpret_cast<uintptr_t>(dev_blocks[i]) % 16 != 0)
        return fail(LST_ERR_ALIGNMENT, "lst_adamw_step_ex: block %lld pointer not 16-byte aligned", (long long)i);
    }
    RunEx r;
    r.run = block_run(*L, b, static_cast<char*>(dev_blocks[i]), 0, b.padded);
    r.bias_correction1 = bc1[(size_t)i];
    r.bias_correction2 = bc2[(size_t)i];
    r.out_index = want_sq ? (int32_t)i : -1;
    r.accumulate = 0;
    if (r.run.elems == 0 && !want_sq) continue;
    runs.push_back(r);
  }
  if (runs.empty()) return LST_OK;
  cudaError_t err = launch_update_ex(L->fmt, runs.data(), (int)runs.size(), s, want_sq ? opts->workspace : nullptr,
                                     want_sq ? opts->grad_sq : nullptr, static_cast<cudaStream_t>(cuda_stream));
  if (err != cudaSuccess) return cuda_fail(err, "lst_adamw_step_ex");
  return LST_OK;
}

// Zero-copy step: the update kernel addresses the pinned, mapped host blocks
// directly, so every byte crosses the host link exactly once in each needed
// direction and neither device buffers nor copy engines are involved.
extern "C" lst_status lst_zero_copy_step(const lst_layout* L, void* const* host_blocks,
                                         const lst_adamw_hparams* hp, void* cuda_stream) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_zero_copy_step: null layout");
  if (!hp) return fail(LST_ERR_INVALID_ARG, "lst_zero_copy_step: null hparams");
  Scalars s;
  if (!make_scalars(*hp, &s))
    return fail(LST_ERR_INVALID_ARG,
                "lst_zero_copy_step: hyperparameters outside their domain (step >= 1, 0 <= beta < 1, finite)");
  const int64_t n = (int64_t)L->blocks.size();
  if (n == 0) return LST_OK;
  if (!host_blocks) return fail(LST_ERR_INVALID_ARG, "lst_zero_copy_step: host_blocks is null");
  std::vector<void*> dptr((size_t)n, nullptr);
  for (int64_t i = 0; i < n; ++i) {
    if (L->blocks[(size_t)i].bytes == 0) continue;
    if (!host_blocks[i])
      return fail(LST_ERR_INVALID_ARG, "lst_zero_copy_step: host block %lld is null", (long long)i);
    if (reinterpret_cast<uintptr_t>(host_blocks[i]) % 4096)
      return fail(LST_ERR_ALIGNMENT, "lst_zero_copy_step: host block %lld not 4096-byte aligned", (long long)i);
    cudaPointerAttributes a;
    cudaError_t err = cudaPointerGetAttributes(&a, host_blocks[i]);
    if (err != cudaSuccess) {
      cudaGetLastError();
      return fail(LST_ERR_NOT_PINNED, "lst_zero_copy_step: host block %lld is not pinned", (long long)i);
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr)
      return fail(LST_ERR_NOT_PINNED, "lst_zero_copy_step: host block %lld is not pinned, mapped host memory",
                  (long long)i);
    dptr[(size_t)i] = a.devicePointer;
  }
  return device_step(L, dptr.data(), s, false, cuda_stream, "lst_zero_copy_step");
}

extern "C" lst_status lst_host_alloc(int64_t bytes, void** out) {
  clear_error();
  if (!out) return fail(LST_ERR_INVALID_ARG, "lst_host_alloc: out is null");
  *out = nullptr;
  if (bytes <= 0) return fail(LST_ERR_INVALID_ARG, "lst_host_alloc: bytes must be > 0");
  long page = sysconf(_SC_PAGESIZE);
  if (page < 4096) page = 4096;
  const size_t size = ((size_t)bytes + (size_t)page - 1) / (size_t)page * (size_t)page;
  void* p = mmap(nullptr, size, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (p == MAP_FAILED) return fail(LST_ERR_OOM, "lst_host_alloc: %lld bytes: out of host memory", (long long)bytes);
  cudaError_t err = cudaHostRegister(p, size, cudaHostRegisterMapped | cudaHostRegisterPortable);
  if (err != cudaSuccess) {
    munmap(p, size);
    if (err == cudaErrorMemoryAllocation) {
      cudaGetLastError();
      return fail(LST_ERR_OOM, "lst_host_alloc: %lld bytes: cannot pin", (long long)bytes);
    }
    return cuda_fail(err, "lst_host_alloc");
  }
  {
    std::lock_guard<std::mutex> g(host_allocs_mu());
    host_allocs()[p] = size;
  }
  *out = p;
  return LST_OK;
}

extern "C" lst_status lst_host_free(void* p) {
  clear_error();
  if (!p) return LST_OK;
  size_t size = 0;
  {
    std::lock_guard<std::mutex> g(host_allocs_mu());
    auto it = host_allocs().find(p);
    if (it == host_allocs().end())
      return fail(LST_ERR_INVALID_ARG, "lst_host_free: pointer not from lst_host_alloc");
    size = it->second;
    host_allocs().erase(it);
  }
  cudaError_t err = cudaHostUnregister(p);
  munmap(p, size);
  if (err != cudaSuccess) return cuda_fail(err, "lst_host_free");
  return LST_OK;
}

extern "C" const char* lst_status_string(lst_status st) {
  switch (st) {
    case LST_OK: return "ok";
    case LST_ERR_INVALID_ARG: return "invalid argument";
    case LST_ERR_ALIGNMENT: return "misaligned pointer";
    case LST_ERR_NOT_PINNED: return "host memory not pinned";
    case LST_ERR_CUDA: return "CUDA error";
    case LST_ERR_OOM: return "out of memory";
    case LST_ERR_TIMEOUT: return "timed out";
    case LST_ERR_IO: return "file I/O error";
  }
  return "unknown status";
}

extern "C" const char* lst_last_error(void) { return g_err; }

extern "C" lst_status lst_test_inject(int32_t kind, int64_t k) {
  clear_error();
  if (kind < 0 || kind > 4) return fail(LST_ERR_INVALID_ARG, "lst_test_inject: unknown kind %d", kind);
  if ((kind == 1 || kind == 3 || kind == 4) && k < 1)
    return fail(LST_ERR_INVALID_ARG, "lst_test_inject: k must be >= 1");
  inject().k.store(k);
  inject().kind.store(kind);
  return LST_OK;
}
