// Internal declarations shared by liblst's translation units (not installed).
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/lst.h"

namespace lst {

constexpr int kMaxFields = 5;
constexpr int64_t kTensorAlign = 8;     // elements: 16 B in a bf16 segment
constexpr int64_t kBlockAlign = 2048;   // elements: every segment a whole number of 4 KB pages
constexpr int64_t kWarpSpan = 256;      // elements one warp covers per task (kernel tiling)
constexpr int64_t kMaxBlockElems = int64_t(1) << 40;
constexpr int64_t kDefaultStreamChunk = int64_t(1) << 24;
constexpr int kMaxRunsPerLaunch = 128;

// Segment order and element size of each format.
struct FormatInfo {
  int n_segments;
  int field[kMaxFields];      // field id of segment k
  int elem_bytes[kMaxFields]; // element size of segment k
  int n_inputs;               // segments [0, n_inputs) are read by the update
  int first_output;           // segments [first_output, n_segments) are written
  int bytes_per_param;
};
const FormatInfo& format_info(lst_format fmt);

struct Block {
  int64_t params = 0;    // sum of tensor sizes
  int64_t padded = 0;    // elements per segment
  int64_t bytes = 0;
  int64_t seg_off[kMaxFields];    // by field id, -1 if absent
  int64_t h2d_off = 0, h2d_bytes = 0, d2h_off = 0, d2h_bytes = 0;
};

struct Tensor {
  int64_t layer = 0;
  int64_t elem_off = 0;
  int64_t numel = 0;
};

struct Engine;  // streamed-step resources (streams, events), per device

// What LST_COPY_AUTO learned about one block's host memory: the sub-chunk
// boundaries of the step that timed it, which sub-chunks the copy engines
// moved at under 0.4 of the best sub-chunk rate seen (those go through the
// copy kernel from then on), and the range of copy-engine rates timed. Valid
// while the block's host pointer, size and sub-chunk boundaries stay the same.
struct LinkChoice {
  const void* host = nullptr;
  int64_t bytes = 0;
  std::vector<int64_t> cuts;
  std::vector<uint8_t> slow_in, slow_out;
  bool measured = false;
  double engine_h2d_min = 0, engine_h2d_max = 0, engine_d2h_min = 0, engine_d2h_max = 0;  // GB/s
};

}  // namespace lst

struct lst_layout {
  lst_format fmt;
  int64_t n_params = 0;
  int64_t max_block_bytes = 0;
  int64_t stream_chunk = lst::kDefaultStreamChunk;
  int stream_copy_h2d = LST_COPY_AUTO;  // how the streamed steps move sub-chunks in
  int stream_copy_d2h = LST_COPY_AUTO;  // ... and out (lst_layout_set_stream_copy)
  std::vector<lst::LinkChoice> link;    // per block, for LST_COPY_AUTO
  lst_stream_stats last_step{};         // the last streamed step that completed
  std::vector<lst::Block> blocks;
  std::vector<lst::Tensor> tensors;
  std::mutex stream_mu;           // serialises lst_stream_step on this layout
  lst::Engine* engine = nullptr;  // created on first lst_stream_step
};

namespace lst {

// One contiguous run of elements the update kernel walks: pointers to the
// first element of the run in every segment it touches. `w` is the weight the
// update reads and writes (bf16 W for L12, fp32 master for L16M, fp32 W for
// L16F); `w16` is the bf16 W written from the master (L16M only).
struct Run {
  const void* g;
  void* w;
  float* m;
  float* v;
  void* w16;
  int64_t elems;  // multiple of kWarpSpan
};

// fp32 step scalars, formed in double on the host and rounded once.
struct Scalars {
  float beta1, beta2, one_minus_beta1, one_minus_beta2;
  float bias_correction1, bias_correction2;
  float eps, lr, decay;
};

bool make_scalars(const lst_adamw_hparams& hp, Scalars* s);
bool valid_hparams(const lst_adamw_hparams* hp);

// Build the run of block `b` whose base address is `base`, covering elements
// [e0, e1) of every segment.
Run block_run(const lst_layout& L, const Block& b, char* base, int64_t e0, int64_t e1);

// Enqueue the update over `runs` on `stream` (one launch per kMaxRunsPerLaunch
// runs). Returns the first CUDA error, cudaSuccess otherwise.
// SM copy of rows x row_bytes at the same pitch on both sides (lst_copy.cu).
cudaError_t launch_stream_copy(const void* src, void* dst, size_t row_bytes, size_t pitch, int rows,
                               cudaStream_t stream);

cudaError_t launch_update(lst_format fmt, bool sgd, const Run* runs, int n_runs, const Scalars& s,
                          cudaStream_t stream);

// A run of the extended update: per-run bias corrections and, optionally,
// the slot of grad_sq that receives the run's sum of g^2.
struct RunEx {
  Run run;
  float bias_correction1, bias_correction2;
  int32_t out_index;   // -1: no sum
  int32_t accumulate;  // 1: add to the slot, 0: overwrite it
};

// Waves of resident CTAs per launch of the large-launch update kernels (grid
// = waves x resident CTAs; each CTA walks its tasks, so the work per CTA is
// the same). A second wave starts
// mid-launch with a fresh ramp (first loads in flight), which a launch of a
// few hundred microseconds notices; over a long launch, extra waves let the
// SMs that finish early take more CTAs. Measured on GB300 (fraction of the
// copy bandwidth, 1, 2, 3, 4 waves): one 44 M-element 12 B layer (969 MB)
// 0.946 / 0.933 / 0.933 / 0.921; 1.1 G elements 12 B 0.961 / 0.962 / 0.961 /
// 0.960; 1.1 G elements 16 B mixed 0.964 / 0.970 / 0.973 / 0.973; and, 2
// against 1 or 3 waves: a 44 M-element 16 B mixed layer (1.2 GB) 0.928-0.932
// against 0.934-0.937 with one; 154 M elements 16 B mixed (4.3 GB) 0.965
// against 0.962-0.964 with three; 1.1 G elements fp32 0.970-0.973 against
// 0.976-0.978 with three.
constexpr long long kOneWaveBytes = 2ll << 30;
constexpr long long kThreeWaveBytes = 8ll << 30;
inline int launch_waves(lst_format fmt, long long bytes) {
  if (bytes < kOneWaveBytes) return 1;
  if (fmt == LST_L12_BF16 || bytes < kThreeWaveBytes) return 2;
  return 3;
}

// Workspace of the sum-of-squares reduction: a reserved 256-byte header, then
// one partial sum (a pair of fp32 values, 8 bytes) per (run, CTA) of a launch.
constexpr int kMaxGridEx = 1024;
constexpr int64_t kWorkspaceHeader = 256;
constexpr int64_t kWorkspaceBytes = kWorkspaceHeader + int64_t(8) * kMaxGridEx * kMaxRunsPerLaunch;

cudaError_t launch_update_ex(lst_format fmt, const RunEx* runs, int n_runs, const Scalars& s, void* workspace,
                             double* grad_sq, cudaStream_t stream);

// Error reporting (thread-local text).
lst_status fail(lst_status st, const char* fmt, ...);
lst_status cuda_fail(cudaError_t err, const char* what);
void clear_error();

// Fault-injection hook state (test only).
struct Inject {
  std::atomic<int> kind{0};
  std::atomic<int64_t> k{0};
};
Inject& inject();

void destroy_engine(Engine* e);

lst_status prepare_options(const lst_layout* L, const lst_adamw_hparams& hp, const lst_step_options* o,
                           std::vector<float>* bc1, std::vector<float>* bc2, const char* who);

}  // namespace lst
