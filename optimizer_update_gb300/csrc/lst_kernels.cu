// Fused per-parameter AdamW / SGD update over packed per-layer state blocks.
//
// The arithmetic is the Adam rule written as an additive delta on the stored
// weight ("Training 70B Models on Consumer Hardware (If You're Willing to
// Wait)", section "The Math"), with decoupled weight decay applied to the
// pre-step weight, and the SGD form W += (-lr*g) (same page, section "The
// Assumption Everyone Makes"). Every step is one IEEE fp32 operation with
// round-to-nearest (explicit _rn intrinsics, so no multiply-add contraction),
// in the order stated in include/lst.h.
//
// Design (GB300, sm_103a). The update is elementwise and moves 22-28 bytes per
// parameter for ~15 flops, so it is bound by HBM bandwidth, not by tensor
// cores or ALUs. The kernel therefore:
//   * walks every segment with fully coalesced vector accesses: a warp covers
//     256 consecutive elements per task; lane k owns elements 4k..4k+3 and
//     128+4k..128+4k+3, so each warp-wide access is one contiguous 256 B
//     (bf16) or 512 B (fp32) range;
//   * is persistent and grid-strided: the grid is sized to fill every SM at
//     the occupancy the compiler allows, and tasks of all runs (blocks or
//     sub-chunks of blocks) are dealt round-robin over all warps from one
//     global task index, so many small runs (e.g. 308 LoRA tensors in 22
//     blocks) load-balance like one large one;
//   * keeps both quads of a task in flight before computing, and uses
//     streaming (evict-first) loads and stores: every byte is touched once.
// The run table travels in the kernel's parameter space (__grid_constant__),
// so a step needs no device-side scratch memory and no host-to-device copy of
// metadata.
#include <cstdio>
#include <mutex>

#include "lst_device.cuh"

namespace lst {

// ---- the kernel -------------------------------------------------------------

// How a warp keeps memory busy while it works through the division and
// square-root chain of its elements (chosen per format by measurement, see
// launch below):
//   SCHED_ONE       one task (2 quads per lane) loaded, computed, stored;
//   SCHED_TWO       two tasks loaded together, then computed and stored;
//   SCHED_PREFETCH  the next task's loads are issued before the current task
//                   is computed and stored (register double-buffering).
enum { SCHED_ONE = 0, SCHED_TWO = 1, SCHED_PREFETCH = 2 };

// Large launches: each warp walks its tasks run by run (task j of a run is
// global task first_task + j, owned by warp (first_task + j) mod n_warps).
// Every run spans many tasks per warp, so the schedule overlaps tasks inside
// a run and the run's entry stays in registers for the whole loop.
// Resident CTAs per SM the compiler must allow for: the 12 B layout's prefetch
// schedule is held to 80 registers (3 CTAs of 256 threads per SM), where it
// measured 0.977-0.980 of the copy bandwidth against 0.845 at 2 CTAs; the
// 16 B layouts measured best uncapped (a cap of 80 spilled and lost 7-9 %).
template <int FMT, int SCHED>
struct MinCtas {
  static constexpr int value = (FMT == F_L12 && SCHED == SCHED_PREFETCH) ? 3 : 1;
};

template <int FMT, bool SGD, int SCHED>
__global__ void __launch_bounds__(kThreads, (MinCtas<FMT, SCHED>::value))
    lst_update_kernel(const __grid_constant__ RunTable tab, const Scalars s, const long long total_tasks) {
  (void)total_tasks;
  const int lane = threadIdx.x & 31;
  const long long n_warps = (long long)gridDim.x * (kThreads / 32);
  const long long warp = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  for (int r = 0; r < tab.n; ++r) {
    const RunTable::Entry& R = tab.r[r];
    long long j = (warp - R.first_task) % n_warps;
    if (j < 0) j += n_warps;
    if (SCHED == SCHED_PREFETCH) {
      if (j >= R.tasks) continue;
      Quad<FMT, SGD> a, b;
      long long e = j * 256 + lane * 4;
      load_quad<FMT, SGD>(R, e, a);
      load_quad<FMT, SGD>(R, e + 128, b);
      for (;;) {
        const long long jn = j + n_warps;
        const long long en = jn * 256 + lane * 4;
        Quad<FMT, SGD> na, nb;
        if (jn < R.tasks) {
          load_quad<FMT, SGD>(R, en, na);
          load_quad<FMT, SGD>(R, en + 128, nb);
        }
        update_store_quad<FMT, SGD>(R, e, a, s);
        update_store_quad<FMT, SGD>(R, e + 128, b, s);
        if (jn >= R.tasks) break;
        a = na;
        b = nb;
        e = en;
        j = jn;
      }
    } else {
      constexpr int T = (SCHED == SCHED_TWO) ? 2 : 1;
      for (; j < R.tasks; j += T * n_warps) {
        Quad<FMT, SGD> q[2 * T];
#pragma unroll
        for (int k = 0; k < T; ++k) {
          const long long jj = j + k * n_warps;
          if (jj < R.tasks) {
            const long long e = jj * 256 + lane * 4;
            load_quad<FMT, SGD>(R, e, q[2 * k]);
            load_quad<FMT, SGD>(R, e + 128, q[2 * k + 1]);
          }
        }
#pragma unroll
        for (int k = 0; k < T; ++k) {
          const long long jj = j + k * n_warps;
          if (jj < R.tasks) {
            const long long e = jj * 256 + lane * 4;
            update_store_quad<FMT, SGD>(R, e, q[2 * k], s);
            update_store_quad<FMT, SGD>(R, e + 128, q[2 * k + 1], s);
          }
        }
      }
    }
  }
}

// A warp's position in the run table, held in registers: the run holding
// the current task and a copy of its entry. Tasks of a warp only increase,
// so the cursor only moves forward, and it reads the table only when a task
// falls past the end of the run it holds.
struct Cursor {
  int r;
  long long end;  // first global task after run r
  RunTable::Entry R;
};

__device__ __forceinline__ void cursor_seek(const RunTable& tab, long long g, Cursor& c) {
  if (g < c.end) return;
  int r = c.r;
  while (r < tab.n && g >= tab.r[r].first_task + tab.r[r].tasks) ++r;
  c.r = r;
  if (r < tab.n) {
    c.R = tab.r[r];
    c.end = c.R.first_task + c.R.tasks;
  }
}

// Small launches (many small runs, few tasks per warp, e.g. 22 LoRA blocks):
// each warp walks its global tasks g = warp, warp + n_warps, ... across run
// boundaries with a cursor, one task at a time, with as many resident warps as
// 64 registers allow (4 CTAs of 256 threads per SM): at this size the writes
// stay in L2 and the latency of the division chains, not HBM, sets the pace.
template <int FMT, bool SGD>
__global__ void __launch_bounds__(kThreads, 4) lst_update_small_kernel(const __grid_constant__ RunTable tab,
                                                                      const Scalars s, const long long total_tasks) {
  const int lane = threadIdx.x & 31;
  const long long n_warps = (long long)gridDim.x * (kThreads / 32);
  long long g = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (g >= total_tasks) return;
  Cursor cur;
  cur.r = 0;
  cur.end = 0;
  for (; g < total_tasks; g += n_warps) {
    cursor_seek(tab, g, cur);
    const long long e = (g - cur.R.first_task) * 256 + lane * 4;
    Quad<FMT, SGD> a, b;
    load_quad<FMT, SGD>(cur.R, e, a);
    load_quad<FMT, SGD>(cur.R, e + 128, b);
    update_store_quad<FMT, SGD>(cur.R, e, a, s);
    update_store_quad<FMT, SGD>(cur.R, e + 128, b, s);
  }
}

// ---- launch -----------------------------------------------------------------

typedef void (*KernelFn)(const RunTable, const Scalars, const long long);

// Per format, the schedule and grid that measured fastest on GB300 (1.1 G
// elements, median of 10 launches, fraction of the measured HBM copy
// bandwidth, several boxes): L16M prefetch 0.979-0.987 (one task
// 0.936-0.940); L16F two tasks 0.964-0.987 (one task 0.940); L12 prefetch at
// 3 CTAs per SM 0.968-0.980 (one task 0.917-0.943; two tasks 0.81), with
// grids of two waves of resident CTAs (the number of waves per launch size is
// set by waves_for below).
static KernelFn kernel_for(lst_format fmt, bool sgd, bool small) {
  if (small) {
    switch (fmt) {
      case LST_L12_BF16: return sgd ? lst_update_small_kernel<F_L12, true> : lst_update_small_kernel<F_L12, false>;
      case LST_L16_MIXED: return sgd ? lst_update_small_kernel<F_L16M, true> : lst_update_small_kernel<F_L16M, false>;
      default: return sgd ? lst_update_small_kernel<F_L16F, true> : lst_update_small_kernel<F_L16F, false>;
    }
  }
  // SGD (W += -lr*g: little arithmetic per byte), same measurement with the
  // launch-size waves: 12 B one task 0.996-0.998 (prefetch 0.972-0.978, two
  // tasks 0.915-0.922); 16 B mixed prefetch 0.958-0.961 (one task
  // 0.953-0.954, two tasks 0.953-0.954; one task in one wave 0.939-0.940).
  switch (fmt) {
    case LST_L12_BF16:
      return sgd ? lst_update_kernel<F_L12, true, SCHED_ONE> : lst_update_kernel<F_L12, false, SCHED_PREFETCH>;
    case LST_L16_MIXED:
      return sgd ? lst_update_kernel<F_L16M, true, SCHED_PREFETCH> : lst_update_kernel<F_L16M, false, SCHED_PREFETCH>;
    default:
      return sgd ? lst_update_kernel<F_L16F, true, SCHED_PREFETCH> : lst_update_kernel<F_L16F, false, SCHED_TWO>;
  }
}
// A launch moving less than this many algorithmic bytes is not HBM-bound: its
// writes stay in L2 and its reads take a few microseconds, so the latency of
// the fp32 division chains dominates; it uses lst_update_small_kernel.
constexpr long long kSmallLaunchBytes = 256ll << 20;  // about twice the L2


// Resident CTAs per SM for each kernel instantiation, and SM count, per device.
struct DeviceInfo {
  int sms = 0;
  int ctas_per_sm[12] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
};
constexpr int kMaxDevices = 64;
static DeviceInfo g_dev[kMaxDevices];
static std::mutex g_dev_mu;

static cudaError_t resident_ctas(lst_format fmt, bool sgd, bool small, int* total) {  // per wave
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const int slot = (int)fmt * 4 + (sgd ? 2 : 0) + (small ? 1 : 0);
  std::lock_guard<std::mutex> g(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.sms == 0) {
    err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
  }
  if (d.ctas_per_sm[slot] == 0) {
    int n = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel_for(fmt, sgd, small), kThreads, 0);
    if (err != cudaSuccess) return err;
    d.ctas_per_sm[slot] = n > 0 ? n : 1;
  }
  *total = d.sms * d.ctas_per_sm[slot];
  return cudaSuccess;
}

cudaError_t launch_update(lst_format fmt, bool sgd, const Run* runs, int n_runs, const Scalars& s,
                          cudaStream_t stream) {
  const FormatInfo& fi = format_info(fmt);
  int i = 0;
  while (i < n_runs) {
    RunTable tab;
    tab.n = 0;
    tab.pad_ = 0;
    long long tasks = 0;
    for (; i < n_runs && tab.n < kMaxRunsPerLaunch; ++i) {
      const Run& r = runs[i];
      if (r.elems <= 0) continue;
      RunTable::Entry& e = tab.r[tab.n++];
      e.g = r.g;
      e.w = r.w;
      e.m = r.m;
      e.v = r.v;
      e.w16 = r.w16;
      e.tasks = r.elems / kWarpSpan;
      e.first_task = tasks;
      tasks += e.tasks;
    }
    if (tab.n == 0) continue;
    // algorithmic bytes of the launch: reads and writes of every element
    const long long bytes = tasks * kWarpSpan * (long long)(fi.bytes_per_param + (fmt == LST_L12_BF16 ? 10 : 12));
    const bool small = bytes < kSmallLaunchBytes;
    int per_wave = 0;
    cudaError_t err = resident_ctas(fmt, sgd, small, &per_wave);
    if (err != cudaSuccess) return err;
    // small launches: two waves of the 4-CTA-per-SM kernel
    const long long max_ctas = (long long)per_wave * (small ? 2 : launch_waves(fmt, bytes));
    const long long warps_per_cta = kThreads / 32;
    long long grid = (tasks + warps_per_cta - 1) / warps_per_cta;
    if (grid > max_ctas) grid = max_ctas;
    kernel_for(fmt, sgd, small)<<<(unsigned)grid, kThreads, 0, stream>>>(tab, s, tasks);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace lst
