// Extended update kernel: per-block step counters and per-block sum of g^2,
// for progressive layer locking. Shares the element arithmetic and the
// coalesced accesses of the main kernel (lst_device.cuh).
#include <mutex>

#include "lst_device.cuh"

namespace lst {

// ---- the extended kernels: per-block step counters and per-block sum of g^2 ----
//
// Progressive layer locking ("Training 70B Models on Consumer Hardware",
// section "Progressive Layer Locking") freezes a layer once its gradient
// magnitude falls below a threshold; per-layer step counters keep Adam's bias
// correction exact for the layers that keep training (same page, note under
// "The Math"). These variants take the bias corrections per run, and with
// GSQ=true also return sum(g^2) over every run as a by-product of the same
// pass: per task each lane adds its 8 squares in fp32 (exact products for bf16
// g) and accumulates tasks in an fp32 pair with exact error recovery (below);
// a warp reduces its lanes' pairs in a fixed shuffle order, a CTA adds its
// warps' pairs per run in warp order and writes one partial pair per run to
// the workspace, and a second small launch adds each run's partials in a fixed
// order and forms the fp64 result. The result is deterministic for a given
// grid.
// Large launches walk run by run with the main kernel's prefetch schedule;
// small ones (many short runs, e.g. LoRA adapters) walk their global tasks
// across runs with a cursor, as the main small-launch kernel.

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

// The running sum of a lane's task sums is kept as an unevaluated pair of
// fp32 values hi + lo: each addition's rounding error is recovered exactly
// (Knuth's TwoSum) and collected in lo, so the pair carries about twice
// fp32's precision using fp32 adds only (this GPU has little fp64
// throughput). It becomes one fp64 value when the lane leaves a run; a
// non-finite hi is kept as it is (TwoSum would turn +inf into NaN).
struct SumPair {
  float hi, lo;
};

__device__ __forceinline__ void sum_pair_add(SumPair& p, float x) {
  const float s = __fadd_rn(p.hi, x);
  const float xb = __fsub_rn(s, p.hi);
  const float hb = __fsub_rn(s, xb);
  const float e = __fadd_rn(__fsub_rn(p.hi, hb), __fsub_rn(x, xb));
  p.hi = s;
  p.lo = __fadd_rn(p.lo, e);
}

__device__ __forceinline__ double sum_pair_value(const SumPair& p) {
  return isfinite(p.hi) ? (double)p.hi + (double)p.lo : (double)p.hi;
}

// The sum of two pairs as a pair: the high parts are added with their exact
// rounding error (TwoSum), the low parts and that error in fp32, and the
// result renormalised (the larger part first). About 2^-44 relative error for
// nonnegative terms, fp32 operations only: this GPU's fp64 rate is a small
// fraction of its fp32 rate, and a warp-wide fp64 reduction per run and warp
// cost several microseconds of a 27 us small launch. Commutative bit for bit
// (TwoSum's error term does not depend on the operand order), so a butterfly
// leaves the same value in every lane. An infinite or NaN sum is kept as is.
__device__ __forceinline__ SumPair pair_add(const SumPair& a, const SumPair& b) {
  const float s = __fadd_rn(a.hi, b.hi);
  if (!isfinite(s)) return SumPair{s, 0.0f};
  const float bb = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  const float t = __fadd_rn(__fadd_rn(a.lo, b.lo), e);
  const float hi = __fadd_rn(s, t);
  return SumPair{hi, __fsub_rn(t, __fsub_rn(hi, s))};
}

// Sum of the warp's lanes' pairs in a fixed butterfly order (every lane gets it).
__device__ __forceinline__ SumPair warp_sum_pair(SumPair p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const SumPair q{__shfl_xor_sync(0xffffffffu, p.hi, o), __shfl_xor_sync(0xffffffffu, p.lo, o)};
    p = pair_add(p, q);
  }
  return p;
}


// Programmatic dependent launch (PTX griddepcontrol): the update grid's CTAs
// signal once their partial sums are written, so the reduce grid that follows
// on the stream may be scheduled before the update grid has fully retired;
// the reduce grid waits (in hardware) until the update grid has completed and
// its memory is visible before it reads a partial. The wait ends when the
// update grid ends, so nothing here can hang. (Signalling as each update CTA
// starts instead was measured slower on GB300: 33.3 against 31.5 us per LoRA
// step with sums; without the dependent launch 33.7 us.)
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_prerequisite_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Second launch of a step with sums: one CTA per run adds the partial pairs
// of the CTAs that worked on that run (cta_lo[r] .. cta_hi[r]; thread k takes
// partials lo + k, lo + k + 256, ... in that order), then its threads' pairs
// in a fixed order (a butterfly per warp, then the warps in order; with at
// most 32 partials, as in small launches, warp 0 alone), all as fp32 pairs;
// only the final value is formed in fp64 (fp64 operations are slow on this
// GPU). A separate launch needs no ticket counter, fence or workspace
// initialisation. (Tickets taken by the update CTAs, with the last CTA adding
// the partials, measured slower: each CTA's fence waits for its own streaming
// stores; LoRA adapters with sums, L2 flushed, 33.9 against 30.4 us per step.
// The programmatic dependent launch saves about 2.4 us there.)
struct GradSqTable {
  int32_t n;                  // runs of the update launch
  int32_t partials_per_run;   // stride of the partials: CTAs of the update launch
  int32_t out_index[kMaxRunsPerLaunch];
  int32_t accumulate[kMaxRunsPerLaunch];
  int32_t cta_lo[kMaxRunsPerLaunch];  // first CTA holding a partial of the run
  int32_t cta_hi[kMaxRunsPerLaunch];  // one past the last (cta_lo == cta_hi: the run has no elements)
};

__global__ void __launch_bounds__(kThreads) lst_grad_sq_reduce_kernel(const __grid_constant__ GradSqTable t,
                                                                     const SumPair* partials, double* grad_sq) {
  __shared__ SumPair warp_total[kThreads / 32];
  wait_for_prerequisite_grid();
  const int r = blockIdx.x;
  const int out = t.out_index[r];
  if (out < 0) return;  // the whole CTA
  const int lo = t.cta_lo[r], hi = t.cta_hi[r];
  const bool one_warp = hi - lo <= 32;  // uniform over the CTA
  if (one_warp && threadIdx.x >= 32) return;
  const float2* p = reinterpret_cast<const float2*>(partials) + (size_t)r * t.partials_per_run;
  SumPair a{0.0f, 0.0f};
  for (int c = lo + threadIdx.x; c < hi; c += kThreads) {
    const float2 x = __ldcg(p + c);  // from L2: written by the other grid
    a = pair_add(a, SumPair{x.x, x.y});
  }
  SumPair sum = warp_sum_pair(a);
  if (!one_warp) {
    if ((threadIdx.x & 31) == 0) warp_total[threadIdx.x >> 5] = sum;
    __syncthreads();
    sum = warp_total[0];
#pragma unroll
    for (int k = 1; k < kThreads / 32; ++k) sum = pair_add(sum, warp_total[k]);
  }
  if (threadIdx.x == 0) {
    const double v = sum_pair_value(sum);
    grad_sq[out] = t.accumulate[r] ? grad_sq[out] + v : v;
  }
}

// Large launches: warps issue the next task's loads before computing the
// current one (register double-buffering), as the main kernel's prefetch
// schedule. Register budgets, measured on GB300 with the sum of squares on
// (fraction of the measured copy bandwidth, 1.1 G elements): the 12 B layout
// is held to 3 resident CTAs of 256 threads per SM (0.957, against 0.832
// uncapped and 0.888 with one task at a time); the 16 B layouts ask for no
// minimum (0: about 90-98 registers, 2 CTAs per SM, 0.963; a minimum of one
// CTA per SM let the compiler take 112 and measured 0.922).
template <int FMT, bool GSQ>
__global__ void __launch_bounds__(kThreads, (FMT == F_L12 ? 3 : 0))
    lst_update_ex_kernel(const __grid_constant__ RunTableEx tab, const Scalars s0, SumPair* partials) {
  __shared__ SumPair warp_sum[kThreads / 32];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const long long n_warps = (long long)gridDim.x * (kThreads / 32);
  const long long warp = (long long)blockIdx.x * (kThreads / 32) + wid;
  for (int r = 0; r < tab.n; ++r) {
    const RunTableEx::Entry& R = tab.r[r];
    Scalars s = s0;
    s.bias_correction1 = R.bias_correction1;
    s.bias_correction2 = R.bias_correction2;
    SumPair acc{0.0f, 0.0f};
    long long j = (warp - R.first_task) % n_warps;
    if (j < 0) j += n_warps;
    if (j < R.tasks) {
      long long e = j * 256 + lane * 4;
      Quad<FMT, false> a, b;
      load_quad_ex<FMT>(R, e, a);
      load_quad_ex<FMT>(R, e + 128, b);
      for (;;) {
        const long long jn = j + n_warps;
        const long long en = jn * 256 + lane * 4;
        Quad<FMT, false> na, nb;
        if (jn < R.tasks) {
          load_quad_ex<FMT>(R, en, na);
          load_quad_ex<FMT>(R, en + 128, nb);
        }
        if (GSQ) sum_pair_add(acc, sum_sq8(a.g, b.g));
        store_quad_ex<FMT>(R, e, a, s);
        store_quad_ex<FMT>(R, e + 128, b, s);
        if (jn >= R.tasks) break;
        a = na;
        b = nb;
        e = en;
        j = jn;
      }
    }
    if (GSQ) {
      const SumPair ws = warp_sum_pair(acc);
      if (lane == 0) warp_sum[wid] = ws;
      __syncthreads();
      if (threadIdx.x == 0) {
        SumPair c = warp_sum[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) c = pair_add(c, warp_sum[w]);
        partials[(size_t)r * gridDim.x + blockIdx.x] = c;
      }
      __syncthreads();
    }
  }
  if (GSQ) allow_dependent_launch();
}

// Small launches (many short runs, e.g. LoRA adapters): one task at a time
// at 4 CTAs of 256 threads per SM, a register cursor moving forward through
// the run table. Without sums, warp w takes global tasks w, w + n_warps, ...
// (round-robin). With sums, warp w takes the contiguous tasks [w k, (w + 1) k)
// (k = per_warp), so a CTA's 8 warps cover one contiguous range of 8 k tasks
// and a warp meets one or two runs; round-robin made nearly every task of a
// LoRA step start a new run, with a lane reduction each time. A warp meets
// each run in one unbroken stretch of its tasks, so its sum for that run is
// final when the cursor leaves the run: the warp stores it in shared memory
// (one slot per warp and run), and at the end the CTA adds its warps' slots
// per run in warp order and writes a partial pair for each run its range
// meets. Measured on GB300 (LoRA adapters, 6.3 M fp32 parameters in 22
// blocks, L2 flushed, mean of 200 steps): with sums 30.4-30.6 us contiguous
// against 31.5-31.7 round-robin (and 33.4 round-robin with each lane
// reduction moved under the next task's loads, which spilled); without sums
// round-robin 25.8-26.1 against 26.9 contiguous; contiguous ranges over two
// waves of CTAs, or longer ranges over fewer CTAs, were slower (34.2; 32-38).
template <int FMT, bool GSQ>
__global__ void __launch_bounds__(kThreads, 4)
    lst_update_ex_small_kernel(const __grid_constant__ RunTableEx tab, const Scalars s0, SumPair* partials,
                               const long long total_tasks, const long long per_warp) {
  __shared__ SumPair run_sum[GSQ ? kThreads / 32 : 1][GSQ ? kMaxRunsPerLaunch : 1];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  if (GSQ) {  // a warp's slot of a run it does not meet counts as zero
    for (int i = threadIdx.x; i < (kThreads / 32) * kMaxRunsPerLaunch; i += kThreads)
      (&run_sum[0][0])[i] = SumPair{0.0f, 0.0f};
    __syncthreads();
  }
  const long long n_warps = (long long)gridDim.x * (kThreads / 32);
  const long long warp = (long long)blockIdx.x * (kThreads / 32) + wid;
  // with sums: tasks [warp k, (warp + 1) k) (k = per_warp); without: warp,
  // warp + n_warps, ... (round-robin)
  long long g = GSQ ? warp * per_warp : warp;
  long long g_end = GSQ ? g + per_warp : total_tasks;
  if (g_end > total_tasks) g_end = total_tasks;
  const long long g_step = GSQ ? 1 : n_warps;
  int r = -1;
  long long first = 0, end = 0;
  Scalars s = s0;
  SumPair acc{0.0f, 0.0f};
  for (; g < g_end; g += g_step) {
    if (g >= end) {  // warp-uniform: g is the same in every lane
      if (GSQ && r >= 0) {
        const SumPair warp_total = warp_sum_pair(acc);
        if (lane == 0) run_sum[wid][r] = warp_total;
        acc = SumPair{0.0f, 0.0f};
      }
      do {
        ++r;
        first = tab.r[r].first_task;
        end = first + tab.r[r].tasks;
      } while (g >= end);
      s.bias_correction1 = tab.r[r].bias_correction1;
      s.bias_correction2 = tab.r[r].bias_correction2;
    }
    const RunTableEx::Entry& R = tab.r[r];
    const long long e = (g - first) * 256 + lane * 4;
    Quad<FMT, false> a, b;
    load_quad_ex<FMT>(R, e, a);
    load_quad_ex<FMT>(R, e + 128, b);
    if (GSQ) sum_pair_add(acc, sum_sq8(a.g, b.g));
    store_quad_ex<FMT>(R, e, a, s);
    store_quad_ex<FMT>(R, e + 128, b, s);
  }
  if (GSQ) {
    if (r >= 0) {
      const SumPair warp_total = warp_sum_pair(acc);
      if (lane == 0) run_sum[wid][r] = warp_total;
    }
    __syncthreads();
    // a partial for every run that meets the CTA's task range (the launch
    // computes the same CTA ranges per run for the reduce launch)
    const long long c_first = (long long)blockIdx.x * (kThreads / 32) * per_warp;
    const long long c_end = c_first + (kThreads / 32) * per_warp;
    for (int q = threadIdx.x; q < tab.n; q += kThreads) {
      const long long f = tab.r[q].first_task;
      if (tab.r[q].tasks > 0 && f < c_end && f + tab.r[q].tasks > c_first) {
        SumPair c = run_sum[0][q];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) c = pair_add(c, run_sum[w][q]);
        partials[(size_t)q * gridDim.x + blockIdx.x] = c;
      }
    }
    allow_dependent_launch();
  }
}

// Resident CTAs per SM for each instantiation, and SM count, per device.
struct DeviceInfoEx {
  int sms = 0;
  int ctas_per_sm[12] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
};
constexpr int kMaxDevicesEx = 64;
static DeviceInfoEx g_dev_ex[kMaxDevicesEx];
static std::mutex g_dev_ex_mu;

// Below this many algorithmic bytes a launch uses the small-launch kernel (as
// the main path: about twice the L2).
constexpr long long kSmallLaunchBytesEx = 256ll << 20;

typedef void (*KernelExFn)(const RunTableEx, const Scalars, SumPair*);
typedef void (*KernelExSmallFn)(const RunTableEx, const Scalars, SumPair*, const long long, const long long);

static KernelExFn kernel_ex_for(lst_format fmt, bool gsq) {
  switch (fmt) {
    case LST_L12_BF16: return gsq ? lst_update_ex_kernel<F_L12, true> : lst_update_ex_kernel<F_L12, false>;
    case LST_L16_MIXED: return gsq ? lst_update_ex_kernel<F_L16M, true> : lst_update_ex_kernel<F_L16M, false>;
    default: return gsq ? lst_update_ex_kernel<F_L16F, true> : lst_update_ex_kernel<F_L16F, false>;
  }
}

static KernelExSmallFn kernel_ex_small_for(lst_format fmt, bool gsq) {
  switch (fmt) {
    case LST_L12_BF16:
      return gsq ? lst_update_ex_small_kernel<F_L12, true> : lst_update_ex_small_kernel<F_L12, false>;
    case LST_L16_MIXED:
      return gsq ? lst_update_ex_small_kernel<F_L16M, true> : lst_update_ex_small_kernel<F_L16M, false>;
    default: return gsq ? lst_update_ex_small_kernel<F_L16F, true> : lst_update_ex_small_kernel<F_L16F, false>;
  }
}

static cudaError_t resident_ctas_ex(lst_format fmt, bool gsq, bool small, int* total) {  // per wave
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevicesEx) return cudaErrorInvalidDevice;
  const int slot = (int)fmt * 4 + (gsq ? 2 : 0) + (small ? 1 : 0);
  std::lock_guard<std::mutex> g(g_dev_ex_mu);
  DeviceInfoEx& d = g_dev_ex[dev];
  if (d.sms == 0) {
    err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
  }
  if (d.ctas_per_sm[slot] == 0) {
    int n = 0;
    err = small ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel_ex_small_for(fmt, gsq), kThreads, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel_ex_for(fmt, gsq), kThreads, 0);
    if (err != cudaSuccess) return err;
    d.ctas_per_sm[slot] = n > 0 ? n : 1;
  }
  *total = d.sms * d.ctas_per_sm[slot];  // one wave
  return cudaSuccess;
}

cudaError_t launch_update_ex(lst_format fmt, const RunEx* runs, int n_runs, const Scalars& s, void* workspace,
                             double* grad_sq, cudaStream_t stream) {
  const bool gsq = grad_sq != nullptr;
  const FormatInfo& fi = format_info(fmt);
  SumPair* partials = gsq ? reinterpret_cast<SumPair*>(static_cast<char*>(workspace) + kWorkspaceHeader) : nullptr;
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
    // algorithmic bytes of the launch: reads and writes of every element
    const long long bytes = tasks * kWarpSpan * (long long)(fi.bytes_per_param + (fmt == LST_L12_BF16 ? 10 : 12));
    const bool small = bytes < kSmallLaunchBytesEx;
    int per_wave = 0;
    cudaError_t err = resident_ctas_ex(fmt, gsq, small, &per_wave);
    if (err != cudaSuccess) return err;
    // large launches: waves as the main kernel; small ones: one wave of
    // warps with contiguous task ranges. At most kMaxGridEx: the workspace
    // holds one partial sum per CTA and run.
    long long max_ctas = (long long)per_wave * (small ? 1 : launch_waves(fmt, bytes));
    if (max_ctas > kMaxGridEx) max_ctas = kMaxGridEx;
    constexpr long long warps_per_cta = kThreads / 32;
    long long grid = (tasks + warps_per_cta - 1) / warps_per_cta;
    if (grid < 1) grid = 1;
    if (grid > max_ctas) grid = max_ctas;
    long long per_warp = 1;  // small launches with sums: tasks per warp
    if (small && gsq && tasks > 0) {
      per_warp = (tasks + grid * warps_per_cta - 1) / (grid * warps_per_cta);
      grid = (tasks + per_warp * warps_per_cta - 1) / (per_warp * warps_per_cta);  // no idle CTA
    }
    if (small)
      kernel_ex_small_for(fmt, gsq)<<<(unsigned)grid, kThreads, 0, stream>>>(tab, s, partials, tasks, per_warp);
    else
      kernel_ex_for(fmt, gsq)<<<(unsigned)grid, kThreads, 0, stream>>>(tab, s, partials);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (gsq) {
      GradSqTable t;
      t.n = tab.n;
      t.partials_per_run = (int32_t)grid;
      const long long cta_tasks = per_warp * warps_per_cta;
      for (int k = 0; k < tab.n; ++k) {
        t.out_index[k] = tab.r[k].out_index;
        t.accumulate[k] = tab.r[k].accumulate;
        if (!small) {  // every CTA walks every run
          t.cta_lo[k] = 0;
          t.cta_hi[k] = (int32_t)grid;
        } else if (tab.r[k].tasks > 0) {  // the CTAs whose task range meets the run's
          t.cta_lo[k] = (int32_t)(tab.r[k].first_task / cta_tasks);
          t.cta_hi[k] = (int32_t)((tab.r[k].first_task + tab.r[k].tasks - 1) / cta_tasks + 1);
        } else {  // no elements: the sum is zero
          t.cta_lo[k] = 0;
          t.cta_hi[k] = 0;
        }
      }
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)tab.n);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = 0;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      err = cudaLaunchKernelEx(&cfg, lst_grad_sq_reduce_kernel, t, static_cast<const SumPair*>(partials), grad_sq);
      if (err != cudaSuccess) return err;
    }
  }
  return cudaSuccess;
}

}  // namespace lst
