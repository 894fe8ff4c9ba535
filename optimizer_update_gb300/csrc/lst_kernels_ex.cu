// Extended update kernel: per-block step counters and per-block sum of g^2,
// for progressive layer locking. Shares the element arithmetic and the
// coalesced accesses of the main kernel (lst_device.cuh).
#include <mutex>

#include "lst_device.cuh"

namespace lst {

// ---- the extended kernel: per-block step counters and per-block sum of g^2 ----
//
// Progressive layer locking ("Training 70B Models on Consumer Hardware",
// section "Progressive Layer Locking") freezes a layer once its gradient
// magnitude falls below a threshold; per-layer step counters keep Adam's bias
// correction exact for the layers that keep training (same page, note under
// "The Math"). This variant takes the bias corrections per run, and with
// GSQ=true also returns sum(g^2) over every run as a by-product of the same
// pass: per task each lane adds its 8 squares in fp32 (exact products for bf16
// g), accumulates tasks in fp64, the warp and the CTA reduce in a fixed order,
// each CTA writes one partial per run to the workspace, and the last CTA to
// finish adds the partials in CTA order. The result is deterministic for a
// given grid.

struct RunTableEx {
  int32_t n;
  int32_t pad_;
  struct Entry {
    const void* g;
    void* w;
    float* m;
    float* v;
    void* w16;
    long long tasks;
    long long first_task;
    float bias_correction1, bias_correction2;
    int32_t out_index;   // slot in grad_sq, -1 for none
    int32_t accumulate;  // 1: add to grad_sq[out_index]; 0: overwrite
  } r[kMaxRunsPerLaunch];
};
static_assert(sizeof(RunTableEx) < 30000, "kernel parameter space");

template <int FMT>
__device__ __forceinline__ void load_quad_ex(const RunTableEx::Entry& R, long long e, Quad<FMT, false>& q) {
  RunTable::Entry P{R.g, R.w, R.m, R.v, R.w16, R.tasks, R.first_task};
  load_quad<FMT, false>(P, e, q);
}

template <int FMT>
__device__ __forceinline__ void store_quad_ex(const RunTableEx::Entry& R, long long e, Quad<FMT, false>& q,
                                              const Scalars& s) {
  RunTable::Entry P{R.g, R.w, R.m, R.v, R.w16, R.tasks, R.first_task};
  update_store_quad<FMT, false>(P, e, q, s);
}

__device__ __forceinline__ float sum_sq8(const float4& a, const float4& b) {
  const float x = __fadd_rn(__fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y)),
                            __fadd_rn(__fmul_rn(a.z, a.z), __fmul_rn(a.w, a.w)));
  const float y = __fadd_rn(__fadd_rn(__fmul_rn(b.x, b.x), __fmul_rn(b.y, b.y)),
                            __fadd_rn(__fmul_rn(b.z, b.z), __fmul_rn(b.w, b.w)));
  return __fadd_rn(x, y);
}

template <int FMT, bool GSQ>
__global__ void __launch_bounds__(kThreads) lst_update_ex_kernel(const __grid_constant__ RunTableEx tab,
                                                                 const Scalars s0, double* partials,
                                                                 unsigned int* counter, double* grad_sq) {
  __shared__ double warp_sum[kThreads / 32];
  __shared__ int is_last;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const long long n_warps = (long long)gridDim.x * (kThreads / 32);
  const long long warp = (long long)blockIdx.x * (kThreads / 32) + wid;
  for (int r = 0; r < tab.n; ++r) {
    const RunTableEx::Entry& R = tab.r[r];
    Scalars s = s0;
    s.bias_correction1 = R.bias_correction1;
    s.bias_correction2 = R.bias_correction2;
    double acc = 0.0;
    long long j = (warp - R.first_task) % n_warps;
    if (j < 0) j += n_warps;
    for (; j < R.tasks; j += n_warps) {
      const long long e = j * 256 + lane * 4;
      Quad<FMT, false> a, b;
      load_quad_ex<FMT>(R, e, a);
      load_quad_ex<FMT>(R, e + 128, b);
      if (GSQ) acc += (double)sum_sq8(a.g, b.g);
      store_quad_ex<FMT>(R, e, a, s);
      store_quad_ex<FMT>(R, e + 128, b, s);
    }
    if (GSQ) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) warp_sum[wid] = acc;
      __syncthreads();
      if (threadIdx.x == 0) {
        double c = 0.0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) c += warp_sum[w];
        partials[(size_t)r * gridDim.x + blockIdx.x] = c;
      }
      __syncthreads();
    }
  }
  if (GSQ) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(counter, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (is_last) {
      __threadfence();
      for (int r = threadIdx.x; r < tab.n; r += kThreads) {
        const RunTableEx::Entry& R = tab.r[r];
        if (R.out_index < 0) continue;
        double sum = 0.0;
        for (unsigned c = 0; c < gridDim.x; ++c) sum += __ldcg(&partials[(size_t)r * gridDim.x + c]);
        grad_sq[R.out_index] = R.accumulate ? grad_sq[R.out_index] + sum : sum;
      }
      if (threadIdx.x == 0) *counter = 0u;
    }
  }
}

// Resident CTAs per SM for each instantiation, and SM count, per device.
struct DeviceInfoEx {
  int sms = 0;
  int ctas_per_sm[6] = {0, 0, 0, 0, 0, 0};
};
constexpr int kMaxDevicesEx = 64;
static DeviceInfoEx g_dev_ex[kMaxDevicesEx];
static std::mutex g_dev_ex_mu;

typedef void (*KernelExFn)(const RunTableEx, const Scalars, double*, unsigned int*, double*);

static KernelExFn kernel_ex_for(lst_format fmt, bool gsq) {
  switch (fmt) {
    case LST_L12_BF16: return gsq ? lst_update_ex_kernel<F_L12, true> : lst_update_ex_kernel<F_L12, false>;
    case LST_L16_MIXED: return gsq ? lst_update_ex_kernel<F_L16M, true> : lst_update_ex_kernel<F_L16M, false>;
    default: return gsq ? lst_update_ex_kernel<F_L16F, true> : lst_update_ex_kernel<F_L16F, false>;
  }
}

static cudaError_t resident_ctas_ex(lst_format fmt, bool gsq, int* total) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevicesEx) return cudaErrorInvalidDevice;
  const int slot = (int)fmt * 2 + (gsq ? 1 : 0);
  std::lock_guard<std::mutex> g(g_dev_ex_mu);
  DeviceInfoEx& d = g_dev_ex[dev];
  if (d.sms == 0) {
    err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
  }
  if (d.ctas_per_sm[slot] == 0) {
    int n = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel_ex_for(fmt, gsq), kThreads, 0);
    if (err != cudaSuccess) return err;
    d.ctas_per_sm[slot] = n > 0 ? n : 1;
  }
  *total = d.sms * d.ctas_per_sm[slot];
  if (*total > kMaxGridEx) *total = kMaxGridEx;
  return cudaSuccess;
}

cudaError_t launch_update_ex(lst_format fmt, const RunEx* runs, int n_runs, const Scalars& s, void* workspace,
                             double* grad_sq, cudaStream_t stream) {
  const bool gsq = grad_sq != nullptr;
  int max_ctas = 0;
  cudaError_t err = resident_ctas_ex(fmt, gsq, &max_ctas);
  if (err != cudaSuccess) return err;
  KernelExFn fn = kernel_ex_for(fmt, gsq);
  unsigned int* counter = gsq ? static_cast<unsigned int*>(workspace) : nullptr;
  double* partials = gsq ? reinterpret_cast<double*>(static_cast<char*>(workspace) + kWorkspaceHeader) : nullptr;
  int i = 0;
  while (i < n_runs) {
    RunTableEx tab;
    tab.n = 0;
    tab.pad_ = 0;
    long long tasks = 0;
    for (; i < n_runs && tab.n < kMaxRunsPerLaunch; ++i) {
      const RunEx& r = runs[i];
      if (r.run.elems <= 0 && r.out_index < 0) continue;
      RunTableEx::Entry& e = tab.r[tab.n++];
      e.g = r.run.g;
      e.w = r.run.w;
      e.m = r.run.m;
      e.v = r.run.v;
      e.w16 = r.run.w16;
      e.tasks = r.run.elems / kWarpSpan;
      e.first_task = tasks;
      e.bias_correction1 = r.bias_correction1;
      e.bias_correction2 = r.bias_correction2;
      e.out_index = r.out_index;
      e.accumulate = r.accumulate;
      tasks += e.tasks;
    }
    if (tab.n == 0) continue;
    long long grid = (tasks + kThreads / 32 - 1) / (kThreads / 32);
    if (grid < 1) grid = 1;
    if (grid > max_ctas) grid = max_ctas;
    if (gsq) {
      err = cudaMemsetAsync(counter, 0, sizeof(unsigned int), stream);
      if (err != cudaSuccess) return err;
    }
    fn<<<(unsigned)grid, kThreads, 0, stream>>>(tab, s, partials, counter, grad_sq);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace lst
