// Streamed step: StreamIn -> update -> StreamOut over host-pinned blocks.
//
// "MegaTrain" summary page, sections on the double-buffered pipeline and on
// three-stream execution: host memory holds the authoritative state; two
// device buffers ping-pong; a weight-transfer stream copies host -> device, a
// compute stream runs the layer, a third stream copies device -> host; the
// streams are ordered only by events (weights ready, done, buffer free), with
// no host-side barrier and no CUDA Graph. Here the compute is the optimizer
// update itself, so the event that releases the outbound copy is
// "update done".
//
// GB300 specifics. The host link (NVLink-C2C on Grace systems) is duplex, so
// the inbound and outbound copies of different sub-chunks overlap. Each block
// is moved in sub-chunks (the layout's stream chunk, default 16 Mi elements):
// chunk c's update starts as soon as chunk c has arrived and its outbound copy
// as soon as its update is done, so the pipeline fills and drains in one
// sub-chunk rather than one whole block. The k-th block transferred is staged
// in buffer k & 1 at the block's own offsets; the (k+2)-th block's inbound
// copies wait for the event that the k-th block's last outbound copy recorded.
// Blocks go in index order, or in a caller's order (a backward pass finishes
// its layers last to first), and a block's update can wait for an event that
// marks its gradient complete ("MegaTrain" page, three-stream execution: the
// Backward-Done event). Events are re-recorded per chunk: a
// stream wait binds to the most recent record enqueued before it, and all
// enqueues come from this one host thread in order.
#include <chrono>
#include <new>
#include <thread>
#include <vector>

#include "lst_internal.h"

namespace lst {

struct Engine {
  int device = -1;
  cudaStream_t h2d = nullptr, compute = nullptr, d2h = nullptr;
  cudaEvent_t weights_ready[2] = {nullptr, nullptr};
  cudaEvent_t update_done[2] = {nullptr, nullptr};
  cudaEvent_t buffer_free[2] = {nullptr, nullptr};
  cudaEvent_t done = nullptr;
  size_t max_pitch = 0;  // the device's largest pitch for 2D copies
  // LST_COPY_AUTO: timing events around the copy-engine sub-chunk copies
  // (grown as needed, reused by every step), and the best sub-chunk rate
  // seen each way (GB/s: 0 inbound, 1 outbound)
  std::vector<cudaEvent_t> timers;
  double best_gbs[2] = {0.0, 0.0};
};

static void release(Engine* e) {
  for (int b = 0; b < 2; ++b) {
    if (e->weights_ready[b]) cudaEventDestroy(e->weights_ready[b]);
    if (e->update_done[b]) cudaEventDestroy(e->update_done[b]);
    if (e->buffer_free[b]) cudaEventDestroy(e->buffer_free[b]);
  }
  if (e->done) cudaEventDestroy(e->done);
  for (cudaEvent_t t : e->timers) cudaEventDestroy(t);
  e->timers.clear();
  if (e->h2d) cudaStreamDestroy(e->h2d);
  if (e->compute) cudaStreamDestroy(e->compute);
  if (e->d2h) cudaStreamDestroy(e->d2h);
  *e = Engine();
}

void destroy_engine(Engine* e) {
  if (!e) return;
  int prev = -1;
  if (e->device >= 0 && cudaGetDevice(&prev) == cudaSuccess) {
    cudaSetDevice(e->device);
    release(e);
    cudaSetDevice(prev);
  }
  delete e;
}

static cudaError_t create(Engine* e, int device) {
  e->device = device;
  cudaError_t err;
  int pitch = 0;
  if ((err = cudaDeviceGetAttribute(&pitch, cudaDevAttrMaxPitch, device)) != cudaSuccess) return err;
  e->max_pitch = pitch > 0 ? (size_t)pitch : 0;
  const unsigned f = cudaStreamNonBlocking;
  if ((err = cudaStreamCreateWithFlags(&e->h2d, f)) != cudaSuccess) return err;
  if ((err = cudaStreamCreateWithFlags(&e->compute, f)) != cudaSuccess) return err;
  if ((err = cudaStreamCreateWithFlags(&e->d2h, f)) != cudaSuccess) return err;
  const unsigned ef = cudaEventDisableTiming;
  for (int b = 0; b < 2; ++b) {
    if ((err = cudaEventCreateWithFlags(&e->weights_ready[b], ef)) != cudaSuccess) return err;
    if ((err = cudaEventCreateWithFlags(&e->update_done[b], ef)) != cudaSuccess) return err;
    if ((err = cudaEventCreateWithFlags(&e->buffer_free[b], ef)) != cudaSuccess) return err;
  }
  return cudaEventCreateWithFlags(&e->done, ef);
}

// Counts asynchronous enqueues so the test hook can fail the k-th one.
struct Enqueuer {
  int kind;
  int64_t k;
  int64_t count = 0;
  bool injected = false;
  cudaError_t operator()(cudaError_t (*issue)(void*), void* ctx) {
    ++count;
    if (kind == 1 && count == k) {
      injected = true;
      return cudaErrorUnknown;
    }
    return issue(ctx);
  }
};

struct CopyOp {
  void* dst;
  const void* src;
  size_t bytes;
  cudaMemcpyKind dir;
  cudaStream_t st;
};
static cudaError_t do_copy(void* p) {
  CopyOp* c = static_cast<CopyOp*>(p);
  return cudaMemcpyAsync(c->dst, c->src, c->bytes, c->dir, c->st);
}
// Rows of equal length at the same stride on both sides: the chunk ranges of
// consecutive segments with the same element size (segments are contiguous,
// each padded * element-size bytes long).
struct Copy2DOp {
  void* dst;
  const void* src;
  size_t pitch, width, rows;
  cudaMemcpyKind dir;
  cudaStream_t st;
};
static cudaError_t do_copy2d(void* p) {
  Copy2DOp* c = static_cast<Copy2DOp*>(p);
  return cudaMemcpy2DAsync(c->dst, c->pitch, c->src, c->pitch, c->width, c->rows, c->dir, c->st);
}
struct SmCopyOp {  // the same rows moved by the SMs (lst_copy.cu)
  void* dst;
  const void* src;
  size_t pitch, width, rows;
  cudaStream_t st;
};
static cudaError_t do_sm_copy(void* p) {
  SmCopyOp* c = static_cast<SmCopyOp*>(p);
  return launch_stream_copy(c->src, c->dst, c->width, c->pitch, (int)c->rows, c->st);
}
struct RecordOp {
  cudaEvent_t ev;
  cudaStream_t st;
};
static cudaError_t do_record(void* p) {
  RecordOp* r = static_cast<RecordOp*>(p);
  return cudaEventRecord(r->ev, r->st);
}
static cudaError_t do_wait(void* p) {
  RecordOp* r = static_cast<RecordOp*>(p);
  return cudaStreamWaitEvent(r->st, r->ev, 0);
}
struct LaunchOp {
  lst_format fmt;
  Run run;
  const Scalars* s;
  cudaStream_t st;
  bool ex;          // per-block options in use: the extended kernel
  RunEx run_ex;
  void* workspace;
  double* grad_sq;
};
static cudaError_t do_launch(void* p) {
  LaunchOp* l = static_cast<LaunchOp*>(p);
  if (l->ex) return launch_update_ex(l->fmt, &l->run_ex, 1, *l->s, l->workspace, l->grad_sq, l->st);
  return launch_update(l->fmt, false, &l->run, 1, *l->s, l->st);
}

// Chunk boundaries of one block: chunks of C elements, except that the
// step's first block starts with chunks of C/8, C/4, C/2 and its last block
// ends with C/2, C/4, C/8, so that the pipeline fills (first inbound copy
// before any update) and drains (last outbound copy after the last update) in
// a small chunk rather than a full one. Every boundary stays a multiple of
// 2048 elements.
static std::vector<int64_t> chunk_cuts(int64_t padded, int64_t C, bool first_block, bool last_block) {
  std::vector<int64_t> sizes;
  if (C >= padded) {
    sizes.push_back(padded);
  } else {
    int64_t left = padded;
    std::vector<int64_t> head, tail;
    for (int64_t k = 8; k >= 2; k /= 2) {  // C/8, C/4, C/2
      const int64_t c = (C / k) / kBlockAlign * kBlockAlign;
      if (first_block && c > 0 && left > C + c) {
        head.push_back(c);
        left -= c;
      }
      if (last_block && c > 0 && left > C + c) {
        tail.push_back(c);
        left -= c;
      }
    }
    sizes = head;
    while (left > 0) {
      const int64_t c = left < C ? left : C;
      sizes.push_back(c);
      left -= c;
    }
    sizes.insert(sizes.end(), tail.rbegin(), tail.rend());
  }
  std::vector<int64_t> cuts(1, 0);
  for (int64_t c : sizes) cuts.push_back(cuts.back() + c);
  return cuts;
}

// Enqueues the copies of elements [e0, e1) of segments [k0, k1) of a block
// between `from` and `to` (same layout on both sides). Consecutive segments
// with the same element size go as one 2D copy (one row per segment, the
// segment's byte length as the pitch), so a sub-chunk of the mixed layout is
// two copies per direction instead of four: fewer, larger copy-engine
// operations. Falls back to one copy per segment where the pitch exceeds the
// device's limit.
static cudaError_t enqueue_range(Enqueuer& enq, const Engine* E, const FormatInfo& fi, const Block& b, int k0, int k1,
                                 int64_t e0, int64_t e1, char* to, const char* from, cudaMemcpyKind dir,
                                 cudaStream_t st, bool sm) {
  int k = k0;
  while (k < k1) {
    const int64_t eb = fi.elem_bytes[k];
    const size_t pitch = (size_t)(b.padded * eb);
    int k2 = k + 1;
    while (k2 < k1 && fi.elem_bytes[k2] == eb &&
           b.seg_off[fi.field[k2]] == b.seg_off[fi.field[k2 - 1]] + (int64_t)pitch)
      ++k2;
    const int64_t off = b.seg_off[fi.field[k]] + e0 * eb;
    const size_t width = (size_t)((e1 - e0) * eb);
    if (sm) {  // one launch for the group, any pitch
      SmCopyOp c{to + off, from + off, pitch, width, (size_t)(k2 - k), st};
      cudaError_t err = enq(do_sm_copy, &c);
      if (err != cudaSuccess) return err;
    } else if (k2 - k > 1 && pitch <= E->max_pitch) {
      Copy2DOp c{to + off, from + off, pitch, width, (size_t)(k2 - k), dir, st};
      cudaError_t err = enq(do_copy2d, &c);
      if (err != cudaSuccess) return err;
    } else {
      for (int j = k; j < k2; ++j) {
        const int64_t o = b.seg_off[fi.field[j]] + e0 * eb;
        CopyOp c{to + o, from + o, width, dir, st};
        cudaError_t err = enq(do_copy, &c);
        if (err != cudaSuccess) return err;
      }
    }
    k = k2;
  }
  return cudaSuccess;
}

// LST_COPY_AUTO: one timed sub-chunk copy of a step (each direction of each
// sub-chunk, by the copy engines or the copy kernel; only the copy engines'
// copies are judged).
struct ChunkTiming {
  int64_t block;
  int chunk;
  int dir;  // 0 inbound, 1 outbound
  size_t ev;  // timers[ev] before the copies, timers[ev + 1] after
  int64_t bytes;
  bool engine;  // moved by the copy engines (judged), else by the copy kernel
};

static cudaError_t timer_pair(Engine* E, size_t* at, size_t* next) {
  while (E->timers.size() < *next + 2) {
    cudaEvent_t t = nullptr;
    const cudaError_t err = cudaEventCreateWithFlags(&t, cudaEventDefault);
    if (err != cudaSuccess) return err;
    E->timers.push_back(t);
  }
  *at = *next;
  *next += 2;
  return cudaSuccess;
}

// After a completed step: the summed copy time each way (the step's
// statistics) and the rate of every timed copy-engine sub-chunk copy; a
// sub-chunk whose copy took longer than its bytes at 0.4 of the best rate
// seen in its direction goes through the copy kernel from the next step on.
// (A slow part of a pinned allocation moves at 3-56 GB/s where the rest moves
// at 165-210; the threshold sits well between.) Copies under 4 MB are timed
// but neither set the best rate nor count as slow: a copy's fixed cost of a
// few microseconds dominates them.
constexpr int64_t kMinJudgedCopy = int64_t(4) << 20;

static void learn_from_timings(lst_layout* L, Engine* E, const std::vector<ChunkTiming>& timed) {
  const int inject_every = inject().kind.load() == 4 ? (int)inject().k.load() : 0;
  std::vector<double> gbs(timed.size(), -1.0);
  double busy_ms[2] = {0.0, 0.0};
  for (size_t j = 0; j < timed.size(); ++j) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, E->timers[timed[j].ev], E->timers[timed[j].ev + 1]) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    busy_ms[timed[j].dir] += ms;
    if (ms <= 0.0f || !timed[j].engine) continue;
    double r = (double)timed[j].bytes / (ms * 1e-3) / 1e9;
    if (inject_every > 0 && timed[j].block % inject_every == 0) r /= 100.0;  // test hook
    gbs[j] = r;
    if (timed[j].bytes >= kMinJudgedCopy && r > E->best_gbs[timed[j].dir]) E->best_gbs[timed[j].dir] = r;
  }
  for (size_t j = 0; j < timed.size(); ++j) {
    if (gbs[j] < 0.0) continue;
    const ChunkTiming& t = timed[j];
    LinkChoice& c = L->link[(size_t)t.block];
    c.measured = true;
    if (t.bytes < kMinJudgedCopy) continue;
    double& lo = t.dir == 0 ? c.engine_h2d_min : c.engine_d2h_min;
    double& hi = t.dir == 0 ? c.engine_h2d_max : c.engine_d2h_max;
    if (lo == 0.0 || gbs[j] < lo) lo = gbs[j];
    if (gbs[j] > hi) hi = gbs[j];
    if (gbs[j] < 0.4 * E->best_gbs[t.dir]) (t.dir == 0 ? c.slow_in : c.slow_out)[(size_t)t.chunk] = 1;
  }
  L->last_step.h2d_busy_ms = busy_ms[0];
  L->last_step.d2h_busy_ms = busy_ms[1];
}

static void drain(Engine* e) {
  cudaStreamSynchronize(e->h2d);
  cudaStreamSynchronize(e->compute);
  cudaStreamSynchronize(e->d2h);
}

}  // namespace lst

using namespace lst;

static lst_status stream_impl(const lst_layout* Lc, void* const* host_blocks, void* dev_buf0, void* dev_buf1,
                              const lst_adamw_hparams* hp, const lst_step_options* opts,
                              const void* const* dev_grads, void* const* grad_ready, const int64_t* order,
                              int64_t timeout_ms) {
  if (!Lc) return fail(LST_ERR_INVALID_ARG, "lst_stream_step: null layout");
  if (!hp) return fail(LST_ERR_INVALID_ARG, "lst_stream_step: null hparams");
  Scalars s;
  if (!make_scalars(*hp, &s))
    return fail(LST_ERR_INVALID_ARG,
                "lst_stream_step: hyperparameters outside their domain (step >= 1, 0 <= beta < 1, finite)");
  lst_layout* L = const_cast<lst_layout*>(Lc);  // engine cache and lock only
  std::vector<float> bc1, bc2;
  if (opts) {
    lst_status st = prepare_options(L, *hp, opts, &bc1, &bc2, "lst_stream_step");
    if (st != LST_OK) return st;
  }
  // The extended kernel is needed for per-block bias corrections or sums of
  // squares; a skip mask alone only changes which chunks are launched.
  const bool ex = opts != nullptr && (opts->block_steps != nullptr || opts->grad_sq != nullptr);
  const bool want_sq = opts && opts->grad_sq;
  auto skipped = [&](int64_t i) { return opts && opts->skip && opts->skip[i]; };
  const int64_t n = (int64_t)L->blocks.size();
  if (n == 0) return LST_OK;
  if (!host_blocks) return fail(LST_ERR_INVALID_ARG, "lst_stream_step: host_blocks is null");
  if (!dev_buf0 || !dev_buf1) return fail(LST_ERR_INVALID_ARG, "lst_stream_step: device buffer is null");
  if (reinterpret_cast<uintptr_t>(dev_buf0) % 256 || reinterpret_cast<uintptr_t>(dev_buf1) % 256)
    return fail(LST_ERR_ALIGNMENT, "lst_stream_step: device buffers must be 256-byte aligned");
  for (int64_t i = 0; i < n; ++i) {
    if (L->blocks[(size_t)i].bytes == 0 || skipped(i)) continue;
    if (!host_blocks[i])
      return fail(LST_ERR_INVALID_ARG, "lst_stream_step: host block %lld is null", (long long)i);
    if (reinterpret_cast<uintptr_t>(host_blocks[i]) % 4096)
      return fail(LST_ERR_ALIGNMENT, "lst_stream_step: host block %lld not 4096-byte aligned", (long long)i);
  }
  if (order) {  // a permutation of the blocks
    std::vector<char> seen((size_t)n, 0);
    for (int64_t k = 0; k < n; ++k) {
      const int64_t i = order[k];
      if (i < 0 || i >= n || seen[(size_t)i])
        return fail(LST_ERR_INVALID_ARG, "lst_stream_step: order is not a permutation of the %lld blocks (entry %lld)",
                    (long long)n, (long long)k);
      seen[(size_t)i] = 1;
    }
  }
  if (dev_grads) {
    for (int64_t i = 0; i < n; ++i) {
      if (L->blocks[(size_t)i].bytes == 0 || skipped(i)) continue;
      if (!dev_grads[i])
        return fail(LST_ERR_INVALID_ARG, "lst_stream_step: gradient of block %lld is null", (long long)i);
      if (reinterpret_cast<uintptr_t>(dev_grads[i]) % 16)
        return fail(LST_ERR_ALIGNMENT, "lst_stream_step: gradient of block %lld not 16-byte aligned", (long long)i);
    }
  }
  // Pinned / device checks (host-side driver queries, no device work), and
  // each host block's device mapping for the SM copies (null: none).
  std::vector<char*> mapped((size_t)n, nullptr);
  for (int64_t i = 0; i < n; ++i) {
    if (L->blocks[(size_t)i].bytes == 0 || skipped(i)) continue;
    cudaPointerAttributes a;
    cudaError_t err = cudaPointerGetAttributes(&a, host_blocks[i]);
    if (err != cudaSuccess) {
      cudaGetLastError();
      return fail(LST_ERR_NOT_PINNED, "lst_stream_step: host block %lld is not pinned", (long long)i);
    }
    if (a.type != cudaMemoryTypeHost)
      return fail(LST_ERR_NOT_PINNED, "lst_stream_step: host block %lld is not pinned host memory",
                  (long long)i);
    mapped[(size_t)i] = static_cast<char*>(a.devicePointer);
  }
  for (void* d : {dev_buf0, dev_buf1}) {
    cudaPointerAttributes a;
    cudaError_t err = cudaPointerGetAttributes(&a, d);
    if (err != cudaSuccess) {
      cudaGetLastError();
      return fail(LST_ERR_INVALID_ARG, "lst_stream_step: device buffer is not device memory");
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
      return fail(LST_ERR_INVALID_ARG, "lst_stream_step: device buffer is not device memory");
  }

  std::lock_guard<std::mutex> guard(L->stream_mu);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "lst_stream_step: cudaGetDevice");
  if (L->engine && L->engine->device != dev) {
    destroy_engine(L->engine);
    L->engine = nullptr;
  }
  if (!L->engine) {
    Engine* e = new (std::nothrow) Engine();
    if (!e) return fail(LST_ERR_OOM, "lst_stream_step: out of host memory");
    err = create(e, dev);
    if (err != cudaSuccess) {
      release(e);
      delete e;
      return cuda_fail(err, "lst_stream_step: creating streams/events");
    }
    L->engine = e;
  }
  Engine* E = L->engine;

  const FormatInfo& fi = format_info(L->fmt);
  char* bufs[2] = {static_cast<char*>(dev_buf0), static_cast<char*>(dev_buf1)};

  // LST_COPY_AUTO: per block, what earlier steps learned about its host
  // memory (reset where the pointer or size changed); this step times its
  // copy-engine sub-chunk copies.
  const bool auto_in = L->stream_copy_h2d == LST_COPY_AUTO;
  const bool auto_out = L->stream_copy_d2h == LST_COPY_AUTO;
  if ((auto_in || auto_out) && L->link.size() != (size_t)n) L->link.assign((size_t)n, LinkChoice());
  std::vector<ChunkTiming> timed;
  size_t next_timer = 0;
  lst_stream_stats step{};
  const auto t_start = std::chrono::steady_clock::now();
  Enqueuer enq{inject().kind.load(), inject().k.load()};
  bool used[2] = {false, false};
  const char* what = nullptr;

  // Blocks in processing order; the k-th block that is transferred is staged
  // in buffer k & 1.
  auto block_at = [&](int64_t k) { return order ? order[k] : k; };
  int64_t first_active = -1, last_active = -1;
  for (int64_t k = 0; k < n; ++k) {
    const int64_t i = block_at(k);
    if (skipped(i) || L->blocks[(size_t)i].padded == 0) continue;
    if (first_active < 0) first_active = i;
    last_active = i;
  }
  int64_t staged = 0;
  for (int64_t k = 0; k < n && !what; ++k) {
    const int64_t i = block_at(k);
    const Block& b = L->blocks[(size_t)i];
    if (skipped(i)) continue;  // a locked block: no transfer, no update
    if (b.padded == 0) {
      if (want_sq) {  // an empty block's sum of squares is 0
        LaunchOp l{L->fmt, block_run(*L, b, bufs[0], 0, 0), &s, E->compute, true, {}, opts->workspace,
                   opts->grad_sq};
        l.run_ex = RunEx{l.run, bc1[(size_t)i], bc2[(size_t)i], (int32_t)i, 0};
        if ((err = enq(do_launch, &l)) != cudaSuccess) { what = "launch update"; break; }
      }
      continue;
    }
    const int bi = (int)(staged++ & 1);
    char* buf = bufs[bi];
    char* host = static_cast<char*>(host_blocks[i]);
    // the SMs reach the host block through its device mapping
    const bool has_map = mapped[(size_t)i] != nullptr;
    if (used[bi]) {  // buffer-free: the last outbound copy from this buffer
      RecordOp w{E->buffer_free[bi], E->h2d};
      if ((err = enq(do_wait, &w)) != cudaSuccess) { what = "wait buffer-free"; break; }
    }
    used[bi] = true;
    if (grad_ready && grad_ready[i]) {  // Backward-Done: the block's gradient is complete
      RecordOp w{static_cast<cudaEvent_t>(grad_ready[i]), E->compute};
      if ((err = enq(do_wait, &w)) != cudaSuccess) { what = "wait gradient-ready"; break; }
    }
    const int64_t C = (L->stream_chunk > 0 && L->stream_chunk < b.padded) ? L->stream_chunk : b.padded;
    const bool whole = (C == b.padded);
    const std::vector<int64_t> cuts = chunk_cuts(b.padded, C, i == first_active, i == last_active);
    LinkChoice* lc = (auto_in || auto_out) ? &L->link[(size_t)i] : nullptr;
    if (lc && (lc->host != host_blocks[i] || lc->bytes != b.bytes || lc->cuts != cuts)) {
      *lc = LinkChoice();  // new memory or new sub-chunks: nothing learned yet
      lc->host = host_blocks[i];
      lc->bytes = b.bytes;
      lc->cuts = cuts;
      lc->slow_in.assign(cuts.size() - 1, 0);
      lc->slow_out.assign(cuts.size() - 1, 0);
    }
    for (size_t ci = 0; ci + 1 < cuts.size(); ++ci) {
      const int64_t e0 = cuts[ci], e1 = cuts[ci + 1];
      const bool sm_in = has_map && (L->stream_copy_h2d == LST_COPY_SM || (auto_in && lc->slow_in[ci]));
      const bool sm_out = has_map && (L->stream_copy_d2h == LST_COPY_SM || (auto_out && lc->slow_out[ci]));
      char* host_in = sm_in ? mapped[(size_t)i] : host;
      char* host_out = sm_out ? mapped[(size_t)i] : host;
      int64_t in_bytes = 0, out_bytes = 0;
      for (int k = dev_grads ? 1 : 0; k < fi.n_inputs; ++k) in_bytes += (e1 - e0) * fi.elem_bytes[k];
      for (int k = fi.first_output; k < fi.n_segments; ++k) out_bytes += (e1 - e0) * fi.elem_bytes[k];
      step.h2d_bytes += in_bytes;
      step.d2h_bytes += out_bytes;
      step.chunks += 1;
      step.kernel_in_chunks += sm_in ? 1 : 0;
      step.kernel_out_chunks += sm_out ? 1 : 0;
      const bool time_in = auto_in, time_out = auto_out;
      size_t ev_in = 0, ev_out = 0;
      if (time_in) {
        if ((err = timer_pair(E, &ev_in, &next_timer)) != cudaSuccess) { what = "timing event"; break; }
        RecordOp r0{E->timers[ev_in], E->h2d};
        if ((err = enq(do_record, &r0)) != cudaSuccess) { what = "record timing"; break; }
      }
      // StreamIn: the fields the update reads (all but G when the gradient is
      // already on the device; G is the first segment, so the rest is one range).
      const int first_in = dev_grads ? 1 : 0;
      if (whole) {
        const int64_t off = b.seg_off[fi.field[first_in]];
        const size_t nb = (size_t)(b.h2d_off + b.h2d_bytes - off);
        if (sm_in) {
          SmCopyOp c{buf + off, host_in + off, nb, nb, 1, E->h2d};
          err = enq(do_sm_copy, &c);
        } else {
          CopyOp c{buf + off, host + off, nb, cudaMemcpyHostToDevice, E->h2d};
          err = enq(do_copy, &c);
        }
        if (err != cudaSuccess) { what = "copy in"; break; }
      } else {
        err = enqueue_range(enq, E, fi, b, first_in, fi.n_inputs, e0, e1, buf, host_in, cudaMemcpyHostToDevice,
                            E->h2d, sm_in);
        if (err != cudaSuccess) { what = "copy in"; break; }
      }
      if (time_in) {
        RecordOp r0{E->timers[ev_in + 1], E->h2d};
        if ((err = enq(do_record, &r0)) != cudaSuccess) { what = "record timing"; break; }
        timed.push_back(ChunkTiming{i, (int)ci, 0, ev_in, in_bytes, !sm_in});
      }
      RecordOp r1{E->weights_ready[bi], E->h2d};
      if ((err = enq(do_record, &r1)) != cudaSuccess) { what = "record weights-ready"; break; }
      RecordOp w1{E->weights_ready[bi], E->compute};
      if ((err = enq(do_wait, &w1)) != cudaSuccess) { what = "wait weights-ready"; break; }
      // The update on the staged chunk.
      LaunchOp l{L->fmt, block_run(*L, b, buf, e0, e1), &s, E->compute, ex, {}, nullptr, nullptr};
      if (dev_grads)  // the update reads G from the caller's device gradient
        l.run.g = static_cast<const char*>(dev_grads[i]) + e0 * fi.elem_bytes[0];
      if (ex) {
        l.run_ex = RunEx{l.run, bc1[(size_t)i], bc2[(size_t)i], want_sq ? (int32_t)i : -1, e0 > 0 ? 1 : 0};
        l.workspace = want_sq ? opts->workspace : nullptr;
        l.grad_sq = want_sq ? opts->grad_sq : nullptr;
      }
      if ((err = enq(do_launch, &l)) != cudaSuccess) { what = "launch update"; break; }
      RecordOp r2{E->update_done[bi], E->compute};
      if ((err = enq(do_record, &r2)) != cudaSuccess) { what = "record update-done"; break; }
      RecordOp w2{E->update_done[bi], E->d2h};
      if ((err = enq(do_wait, &w2)) != cudaSuccess) { what = "wait update-done"; break; }
      if (time_out) {
        if ((err = timer_pair(E, &ev_out, &next_timer)) != cudaSuccess) { what = "timing event"; break; }
        RecordOp r0{E->timers[ev_out], E->d2h};
        if ((err = enq(do_record, &r0)) != cudaSuccess) { what = "record timing"; break; }
      }
      // StreamOut: the fields the update wrote.
      if (whole) {
        const size_t nb = (size_t)b.d2h_bytes;
        if (sm_out) {
          SmCopyOp c{host_out + b.d2h_off, buf + b.d2h_off, nb, nb, 1, E->d2h};
          err = enq(do_sm_copy, &c);
        } else {
          CopyOp c{host + b.d2h_off, buf + b.d2h_off, nb, cudaMemcpyDeviceToHost, E->d2h};
          err = enq(do_copy, &c);
        }
        if (err != cudaSuccess) { what = "copy out"; break; }
      } else {
        err = enqueue_range(enq, E, fi, b, fi.first_output, fi.n_segments, e0, e1, host_out, buf,
                            cudaMemcpyDeviceToHost, E->d2h, sm_out);
        if (err != cudaSuccess) { what = "copy out"; break; }
      }
      if (time_out) {
        RecordOp r0{E->timers[ev_out + 1], E->d2h};
        if ((err = enq(do_record, &r0)) != cudaSuccess) { what = "record timing"; break; }
        timed.push_back(ChunkTiming{i, (int)ci, 1, ev_out, out_bytes, !sm_out});
      }
    }
    if (what) break;
    RecordOp r3{E->buffer_free[bi], E->d2h};
    if ((err = enq(do_record, &r3)) != cudaSuccess) { what = "record buffer-free"; break; }
  }
  if (!what) {
    RecordOp rd{E->done, E->d2h};
    if ((err = enq(do_record, &rd)) != cudaSuccess) what = "record done";
  }
  if (what) {
    drain(E);  // nothing of this call stays in flight
    if (enq.injected)
      return fail(LST_ERR_CUDA, "lst_stream_step: %s: injected failure at enqueue %lld", what,
                  (long long)enq.k);
    return cuda_fail(err, what);
  }

  // Completion: poll the final event against the host-side deadline.
  const bool never_done = (enq.kind == 2);
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t q = never_done ? cudaErrorNotReady : cudaEventQuery(E->done);
    if (q == cudaSuccess) {
      step.steps_completed = L->last_step.steps_completed + 1;
      step.wall_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_start).count();
      step.timed = timed.empty() ? 0 : 1;
      L->last_step = step;
      if (!timed.empty()) learn_from_timings(L, E, timed);
      return LST_OK;
    }
    if (q != cudaErrorNotReady) {
      drain(E);
      return cuda_fail(q, "lst_stream_step: waiting for completion");
    }
    if (timeout_ms > 0 &&
        std::chrono::steady_clock::now() - t0 >= std::chrono::milliseconds(timeout_ms)) {
      if (never_done) drain(E);  // the simulated hang: the real work is finite
      return fail(LST_ERR_TIMEOUT, "lst_stream_step: not complete after %lld ms", (long long)timeout_ms);
    }
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

extern "C" lst_status lst_stream_step(const lst_layout* L, void* const* host_blocks, void* dev_buf0, void* dev_buf1,
                                      const lst_adamw_hparams* hp, int64_t timeout_ms) {
  clear_error();
  return stream_impl(L, host_blocks, dev_buf0, dev_buf1, hp, nullptr, nullptr, nullptr, nullptr, timeout_ms);
}

extern "C" lst_status lst_stream_step_ex(const lst_layout* L, void* const* host_blocks, void* dev_buf0,
                                         void* dev_buf1, const lst_adamw_hparams* hp, const lst_step_options* opts,
                                         int64_t timeout_ms) {
  clear_error();
  return stream_impl(L, host_blocks, dev_buf0, dev_buf1, hp, opts, nullptr, nullptr, nullptr, timeout_ms);
}

extern "C" lst_status lst_stream_step_devgrad(const lst_layout* L, void* const* host_blocks,
                                              const void* const* dev_grads, void* dev_buf0, void* dev_buf1,
                                              const lst_adamw_hparams* hp, const lst_step_options* opts,
                                              int64_t timeout_ms) {
  clear_error();
  if (L && !L->blocks.empty() && !dev_grads)
    return fail(LST_ERR_INVALID_ARG, "lst_stream_step_devgrad: dev_grads is null");
  return stream_impl(L, host_blocks, dev_buf0, dev_buf1, hp, opts, dev_grads, nullptr, nullptr, timeout_ms);
}

extern "C" lst_status lst_stream_step_devgrad_events(const lst_layout* L, void* const* host_blocks,
                                                     const void* const* dev_grads, void* const* grad_ready,
                                                     const int64_t* order, void* dev_buf0, void* dev_buf1,
                                                     const lst_adamw_hparams* hp, const lst_step_options* opts,
                                                     int64_t timeout_ms) {
  clear_error();
  if (L && !L->blocks.empty() && !dev_grads)
    return fail(LST_ERR_INVALID_ARG, "lst_stream_step_devgrad_events: dev_grads is null");
  return stream_impl(L, host_blocks, dev_buf0, dev_buf1, hp, opts, dev_grads, grad_ready, order, timeout_ms);
}
