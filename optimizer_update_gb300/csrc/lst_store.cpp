// File-backed block store: the storage tier under host memory.
//
// "Training 70B Models on Consumer Hardware" keeps the model state in files
// on an SSD (sections "How It Works" and "Storage": per-layer files,
// pre-allocated with fallocate so they stay contiguous (section "Limitations"),
// written through and flushed after every update (section "Verification",
// test 2); its safety note asks for checkpointed step counters and atomic
// writes or shadow copies, because a crash between the update and the flush
// corrupts state). The "MegaTrain" summary page names SSDs as the next tier
// below host memory. Here:
//   * one file per packed block: a 4 KB header (magic, layout fingerprint,
//     the block's step counter, a header checksum) then the block's bytes,
//     pre-allocated with fallocate;
//   * blocks move between file and pinned staging with direct I/O (no page
//     cache copy) when the file system allows it, buffered I/O otherwise;
//   * a step updates a block through lst_stream_step_ex and commits it as a
//     shadow file (written, fsync'd) renamed over the block file (then the
//     directory is fsync'd): a crash leaves every block either at its old or
//     at its new step, never torn;
//   * each block's step counter lives in its own header, so a step that was
//     interrupted is resumed by calling it again: blocks already at the step
//     are skipped, the rest are updated once.
//   * reading block k+1, updating block k and writing block k-1 overlap (a
//     reader thread, the caller's thread driving the GPU, a writer thread,
//     three pinned staging buffers).
#include <fcntl.h>
#include <sys/stat.h>
#include <sys/types.h>
#include <unistd.h>

#include <cerrno>
#include <condition_variable>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "lst_internal.h"

namespace lst {

constexpr int64_t kHeaderBytes = 4096;
constexpr uint64_t kMagic = 0x31304B4C4254534Cull;  // the bytes "LSTBLK01"
constexpr uint32_t kVersion = 1;

struct FileHeader {
  uint64_t magic;
  uint32_t version;
  uint32_t format;
  int64_t block;
  int64_t padded;
  int64_t bytes;
  int64_t params;
  int64_t step;
  uint64_t checksum;  // FNV-1a over the fields above
};

static uint64_t fnv1a(const void* p, size_t n) {
  const unsigned char* c = static_cast<const unsigned char*>(p);
  uint64_t h = 0xcbf29ce484222325ull;
  for (size_t i = 0; i < n; ++i) {
    h ^= c[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

static uint64_t header_checksum(const FileHeader& h) { return fnv1a(&h, offsetof(FileHeader, checksum)); }

}  // namespace lst

struct lst_store {
  const lst_layout* layout;
  std::string dir;
  std::vector<int64_t> steps;  // per block, as committed on disk
  bool direct_io = true;
};

namespace lst {

static std::string block_path(const lst_store* S, int64_t i, bool shadow) {
  char name[64];
  snprintf(name, sizeof(name), "/block_%06lld.lst%s", (long long)i, shadow ? ".new" : "");
  return S->dir + name;
}

static lst_status io_fail(const char* what, const std::string& path) {
  return fail(LST_ERR_IO, "%s %s: %s", what, path.c_str(), strerror(errno));
}

static lst_status full_pread(int fd, void* dst, int64_t n, int64_t off, const std::string& path) {
  char* d = static_cast<char*>(dst);
  while (n > 0) {
    ssize_t r = pread(fd, d, (size_t)(n > (1 << 30) ? (1 << 30) : n), off);
    if (r < 0 && errno == EINTR) continue;
    if (r <= 0) return r == 0 ? fail(LST_ERR_IO, "read %s: unexpected end of file", path.c_str())
                              : io_fail("read", path);
    d += r;
    off += r;
    n -= r;
  }
  return LST_OK;
}

static lst_status full_pwrite(int fd, const void* src, int64_t n, int64_t off, const std::string& path) {
  const char* s = static_cast<const char*>(src);
  while (n > 0) {
    ssize_t r = pwrite(fd, s, (size_t)(n > (1 << 30) ? (1 << 30) : n), off);
    if (r < 0 && errno == EINTR) continue;
    if (r <= 0) return io_fail("write", path);
    s += r;
    off += r;
    n -= r;
  }
  return LST_OK;
}

static lst_status fsync_dir(const std::string& dir) {
  int fd = open(dir.c_str(), O_RDONLY | O_DIRECTORY);
  if (fd < 0) return io_fail("open directory", dir);
  int r = fsync(fd);
  close(fd);
  if (r != 0) return io_fail("fsync directory", dir);
  return LST_OK;
}

// Opens for reading or writing, with direct I/O when allowed. Direct I/O needs
// page-aligned buffers, offsets and sizes, which the header and the blocks
// have; the staging buffers are checked by the callers.
static int open_block(const lst_store* S, const std::string& path, int flags) {
  int fd = -1;
#ifdef O_DIRECT
  if (S->direct_io) fd = open(path.c_str(), flags | O_DIRECT, 0644);
#endif
  if (fd < 0) fd = open(path.c_str(), flags, 0644);
  return fd;
}

static FileHeader make_header(const lst_store* S, int64_t i, int64_t step) {
  const Block& b = S->layout->blocks[(size_t)i];
  FileHeader h;
  memset(&h, 0, sizeof(h));
  h.magic = kMagic;
  h.version = kVersion;
  h.format = (uint32_t)S->layout->fmt;
  h.block = i;
  h.padded = b.padded;
  h.bytes = b.bytes;
  h.params = b.params;
  h.step = step;
  h.checksum = header_checksum(h);
  return h;
}

// Writes block i (its bytes from `src`, which must be page aligned) with step
// counter `step` as a shadow file, flushes it and renames it over the block
// file. `fail_before_rename` simulates a crash (test hook).
static lst_status commit_block(const lst_store* S, int64_t i, const void* src, int64_t step,
                               bool fail_before_rename) {
  const Block& b = S->layout->blocks[(size_t)i];
  const std::string tmp = block_path(S, i, true), dst = block_path(S, i, false);
  int fd = open_block(S, tmp, O_WRONLY | O_CREAT | O_TRUNC);
  if (fd < 0) return io_fail("create", tmp);
  lst_status st = LST_OK;
  if (posix_fallocate(fd, 0, kHeaderBytes + b.bytes) != 0) {
    // not every file system supports it; the write below allocates anyway
  }
  alignas(4096) static thread_local unsigned char hdr[kHeaderBytes];
  memset(hdr, 0, sizeof(hdr));
  FileHeader h = make_header(S, i, step);
  memcpy(hdr, &h, sizeof(h));
  st = full_pwrite(fd, hdr, kHeaderBytes, 0, tmp);
  if (st == LST_OK && b.bytes > 0) st = full_pwrite(fd, src, b.bytes, kHeaderBytes, tmp);
  if (st == LST_OK && fsync(fd) != 0) st = io_fail("fsync", tmp);
  close(fd);
  if (st != LST_OK) return st;
  if (fail_before_rename) return fail(LST_ERR_IO, "commit of block %lld: injected failure before rename", (long long)i);
  if (rename(tmp.c_str(), dst.c_str()) != 0) return io_fail("rename", tmp);
  return fsync_dir(S->dir);
}

static lst_status read_header(const lst_store* S, int64_t i, int64_t* step) {
  const std::string path = block_path(S, i, false);
  int fd = open_block(S, path, O_RDONLY);
  if (fd < 0) return io_fail("open", path);
  alignas(4096) static thread_local unsigned char hdr[kHeaderBytes];
  lst_status st = full_pread(fd, hdr, kHeaderBytes, 0, path);
  close(fd);
  if (st != LST_OK) return st;
  FileHeader h;
  memcpy(&h, hdr, sizeof(h));
  const Block& b = S->layout->blocks[(size_t)i];
  if (h.magic != kMagic || h.version != kVersion || h.checksum != header_checksum(h))
    return fail(LST_ERR_IO, "%s: not a block file, or a damaged header", path.c_str());
  if (h.format != (uint32_t)S->layout->fmt || h.block != i || h.padded != b.padded || h.bytes != b.bytes ||
      h.params != b.params)
    return fail(LST_ERR_INVALID_ARG, "%s: written for a different layout", path.c_str());
  *step = h.step;
  return LST_OK;
}

static lst_status read_block(const lst_store* S, int64_t i, void* dst) {
  const Block& b = S->layout->blocks[(size_t)i];
  if (b.bytes == 0) return LST_OK;
  const std::string path = block_path(S, i, false);
  int fd = open_block(S, path, O_RDONLY);
  if (fd < 0) return io_fail("open", path);
  lst_status st = full_pread(fd, dst, b.bytes, kHeaderBytes, path);
  close(fd);
  return st;
}

}  // namespace lst

using namespace lst;

extern "C" lst_status lst_store_create(const lst_layout* L, const char* dir, void* const* host_blocks, int64_t step,
                                       lst_store** out) {
  clear_error();
  if (!L || !dir || !out) return fail(LST_ERR_INVALID_ARG, "lst_store_create: null argument");
  *out = nullptr;
  if (step < 0) return fail(LST_ERR_INVALID_ARG, "lst_store_create: step must be >= 0");
  const int64_t n = (int64_t)L->blocks.size();
  for (int64_t i = 0; i < n; ++i)
    if (host_blocks && host_blocks[i] && reinterpret_cast<uintptr_t>(host_blocks[i]) % 4096)
      return fail(LST_ERR_ALIGNMENT, "lst_store_create: host block %lld not 4096-byte aligned", (long long)i);
  if (mkdir(dir, 0755) != 0 && errno != EEXIST) return io_fail("mkdir", dir);
  lst_store* S = new (std::nothrow) lst_store();
  if (!S) return fail(LST_ERR_OOM, "lst_store_create: out of host memory");
  S->layout = L;
  S->dir = dir;
  S->steps.assign((size_t)n, step);
  void* zeros = nullptr;
  for (int64_t i = 0; i < n; ++i) {
    const void* src = host_blocks ? host_blocks[i] : nullptr;
    if (!src && L->blocks[(size_t)i].bytes > 0) {
      if (!zeros) {
        if (posix_memalign(&zeros, 4096, (size_t)L->max_block_bytes) != 0) {
          delete S;
          return fail(LST_ERR_OOM, "lst_store_create: out of host memory");
        }
        memset(zeros, 0, (size_t)L->max_block_bytes);
      }
      src = zeros;
    }
    lst_status st = commit_block(S, i, src, step, false);
    if (st == LST_OK) continue;
    if (S->direct_io) {  // the file system may refuse direct I/O: retry buffered
      S->direct_io = false;
      st = commit_block(S, i, src, step, false);
    }
    if (st != LST_OK) {
      free(zeros);
      delete S;
      return st;
    }
  }
  free(zeros);
  *out = S;
  return LST_OK;
}

extern "C" lst_status lst_store_open(const lst_layout* L, const char* dir, lst_store** out) {
  clear_error();
  if (!L || !dir || !out) return fail(LST_ERR_INVALID_ARG, "lst_store_open: null argument");
  *out = nullptr;
  lst_store* S = new (std::nothrow) lst_store();
  if (!S) return fail(LST_ERR_OOM, "lst_store_open: out of host memory");
  S->layout = L;
  S->dir = dir;
  const int64_t n = (int64_t)L->blocks.size();
  S->steps.assign((size_t)n, 0);
  for (int64_t i = 0; i < n; ++i) {
    // A shadow file left by an interrupted commit was never renamed: the
    // block file still holds the committed state. Discard the shadow.
    unlink(block_path(S, i, true).c_str());
    lst_status st = read_header(S, i, &S->steps[(size_t)i]);
    if (st != LST_OK && S->direct_io) {
      S->direct_io = false;
      st = read_header(S, i, &S->steps[(size_t)i]);
    }
    if (st != LST_OK) {
      delete S;
      return st;
    }
  }
  *out = S;
  return LST_OK;
}

extern "C" void lst_store_close(lst_store* S) { delete S; }

extern "C" lst_status lst_store_block_step(const lst_store* S, int64_t layer, int64_t* step) {
  clear_error();
  if (!S || !step) return fail(LST_ERR_INVALID_ARG, "lst_store_block_step: null argument");
  if (layer < 0 || layer >= (int64_t)S->steps.size())
    return fail(LST_ERR_INVALID_ARG, "lst_store_block_step: block %lld out of range", (long long)layer);
  *step = S->steps[(size_t)layer];
  return LST_OK;
}

extern "C" lst_status lst_store_read(const lst_store* S, int64_t layer, void* host_dst) {
  clear_error();
  if (!S || !host_dst) return fail(LST_ERR_INVALID_ARG, "lst_store_read: null argument");
  if (layer < 0 || layer >= (int64_t)S->steps.size())
    return fail(LST_ERR_INVALID_ARG, "lst_store_read: block %lld out of range", (long long)layer);
  if (reinterpret_cast<uintptr_t>(host_dst) % 4096)
    return fail(LST_ERR_ALIGNMENT, "lst_store_read: destination not 4096-byte aligned");
  return read_block(S, layer, host_dst);
}

extern "C" lst_status lst_store_write(lst_store* S, int64_t layer, const void* host_src, int64_t step) {
  clear_error();
  if (!S || !host_src) return fail(LST_ERR_INVALID_ARG, "lst_store_write: null argument");
  if (layer < 0 || layer >= (int64_t)S->steps.size())
    return fail(LST_ERR_INVALID_ARG, "lst_store_write: block %lld out of range", (long long)layer);
  if (reinterpret_cast<uintptr_t>(host_src) % 4096)
    return fail(LST_ERR_ALIGNMENT, "lst_store_write: source not 4096-byte aligned");
  if (step < 0) return fail(LST_ERR_INVALID_ARG, "lst_store_write: step must be >= 0");
  const int kind = inject().kind.load();
  lst_status st = commit_block(S, layer, host_src, step, kind == 3 && inject().k.load() == layer + 1);
  if (st == LST_OK) S->steps[(size_t)layer] = step;
  return st;
}

namespace {

// The three-stage pipeline of lst_store_step.
struct Pipe {
  std::mutex mu;
  std::condition_variable cv;
  std::vector<int> state;  // per position in the work list: 0 pending, 1 read, 2 updated, 3 written
  lst_status err = LST_OK;
  std::string err_text;
  bool stop = false;

  void set_error(lst_status st) {
    std::lock_guard<std::mutex> g(mu);
    if (err == LST_OK) {
      err = st;
      err_text = lst_last_error();
    }
    stop = true;
    cv.notify_all();
  }
  // Waits until work[k] reached `want` (or the pipe stopped); returns false if stopped.
  bool wait_for(size_t k, int want) {
    std::unique_lock<std::mutex> g(mu);
    cv.wait(g, [&] { return stop || state[k] >= want; });
    return !stop;
  }
  bool wait_slot_free(size_t k, size_t slots) {  // slot of work k is free once work k - slots is written
    if (k < slots) return true;
    return wait_for(k - slots, 3);
  }
  void advance(size_t k, int to) {
    std::lock_guard<std::mutex> g(mu);
    state[k] = to;
    cv.notify_all();
  }
};

}  // namespace

extern "C" lst_status lst_store_step(lst_store* S, void* const* staging, void* dev_buf0, void* dev_buf1,
                                     const lst_adamw_hparams* hp, int64_t timeout_ms) {
  clear_error();
  if (!S || !staging || !hp) return fail(LST_ERR_INVALID_ARG, "lst_store_step: null argument");
  const lst_layout* L = S->layout;
  if (hp->step < 1) return fail(LST_ERR_INVALID_ARG, "lst_store_step: step must be >= 1");
  for (int k = 0; k < 3; ++k) {
    if (!staging[k]) return fail(LST_ERR_INVALID_ARG, "lst_store_step: staging buffer %d is null", k);
    if (reinterpret_cast<uintptr_t>(staging[k]) % 4096)
      return fail(LST_ERR_ALIGNMENT, "lst_store_step: staging buffer %d not 4096-byte aligned", k);
  }
  const int64_t n = (int64_t)L->blocks.size();
  // Blocks already at this step were committed by an earlier, interrupted
  // call: skip them. A block more than one step behind has missed a step.
  std::vector<int64_t> work;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t t = S->steps[(size_t)i];
    if (t >= hp->step) continue;
    if (t != hp->step - 1)
      return fail(LST_ERR_INVALID_ARG, "lst_store_step: block %lld is at step %lld, cannot apply step %lld",
                  (long long)i, (long long)t, (long long)hp->step);
    work.push_back(i);
  }
  if (work.empty()) return LST_OK;

  const size_t W = work.size();
  const size_t kSlots = 3;
  Pipe P;
  P.state.assign(W, 0);
  const int inject_kind = inject().kind.load();
  const int64_t inject_k = inject().k.load();

  std::thread reader([&] {
    for (size_t k = 0; k < W; ++k) {
      if (!P.wait_slot_free(k, kSlots)) return;
      lst_status st = read_block(S, work[k], staging[k % kSlots]);
      if (st != LST_OK) return P.set_error(st);
      P.advance(k, 1);
    }
  });
  std::thread writer([&] {
    for (size_t k = 0; k < W; ++k) {
      if (!P.wait_for(k, 2)) return;
      const int64_t i = work[k];
      lst_status st = commit_block(S, i, staging[k % kSlots], hp->step, inject_kind == 3 && inject_k == i + 1);
      if (st != LST_OK) return P.set_error(st);
      {
        std::lock_guard<std::mutex> g(P.mu);
        S->steps[(size_t)i] = hp->step;
      }
      P.advance(k, 3);
    }
  });

  // The caller's thread drives the device: one block at a time through the
  // streamed step (every other block marked as locked).
  std::vector<uint8_t> skip((size_t)n, 1);
  std::vector<void*> hb((size_t)n, nullptr);
  for (size_t k = 0; k < W; ++k) {
    if (!P.wait_for(k, 1)) break;
    const int64_t i = work[k];
    skip[(size_t)i] = 0;
    hb[(size_t)i] = staging[k % kSlots];
    lst_step_options o;
    o.block_steps = nullptr;
    o.skip = skip.data();
    o.grad_sq = nullptr;
    o.workspace = nullptr;
    lst_status st = lst_stream_step_ex(L, hb.data(), dev_buf0, dev_buf1, hp, &o, timeout_ms);
    skip[(size_t)i] = 1;
    hb[(size_t)i] = nullptr;
    if (st != LST_OK) {
      P.set_error(st);
      break;
    }
    P.advance(k, 2);
  }
  reader.join();
  writer.join();
  if (P.err != LST_OK) return fail(P.err, "%s", P.err_text.c_str());
  return LST_OK;
}
