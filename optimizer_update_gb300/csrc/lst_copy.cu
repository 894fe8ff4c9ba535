// StreamIn / StreamOut moved by the SMs instead of the copy engines.
//
// The streamed step ("MegaTrain" summary page, double-buffered pipeline and
// three-stream execution) moves each sub-chunk host -> device, updates it and
// moves it back. On a Grace host the pinned blocks are mapped into the
// device's address space, so the SMs can move those bytes with ordinary loads
// and stores over NVLink-C2C as well as the copy engines can by DMA. Measured
// on GB300 (per 0.7-1 GB block, GB/s, host -> device / device -> host): the
// copy engines 210 / 192 on most blocks but 3-15 / 190 on pinned allocations
// that the host backs badly (a third to a half of a process's blocks after
// other processes had pinned and freed ~160 GB), while this kernel ran every
// block at 210.5 / 193 in both states. The kernel runs on the engine's own
// copy streams, ordered by the same events, one launch per run of
// equal-width segment rows of a sub-chunk. In the whole streamed step (1.1 B
// mixed-layout parameters) the copy kernels compete with the update kernel
// for the SMs: on a host whose pinned memory copies at the link rate, copy
// engines both ways 92 ms, SM copies in 111 ms, both ways 117 ms; on a host
// with slow allocations 1.8-1.9 s, 1.4-1.6 s and 0.27-0.32 s. So the default
// mode (LST_COPY_AUTO, lst_layout_set_stream_copy) keeps the copy engines and
// takes this kernel only for a host block, and a direction, that the copy
// engines move at under half this kernel's rate (measured per block).
#include <mutex>

#include "lst_internal.h"

namespace lst {

// rows x row16 16-byte units; row r starts at r * pitch bytes on both sides.
// Every thread keeps four 16-byte loads in flight before it stores.
__global__ void __launch_bounds__(256) lst_stream_copy_kernel(const char* __restrict__ src, char* __restrict__ dst,
                                                             long long row16, long long pitch, int rows) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (int r = 0; r < rows; ++r) {
    const uint4* s = reinterpret_cast<const uint4*>(src + (long long)r * pitch);
    uint4* d = reinterpret_cast<uint4*>(dst + (long long)r * pitch);
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < row16; i += 4 * stride) {
      const uint4 a = s[i], b = s[i + stride], c = s[i + 2 * stride], e = s[i + 3 * stride];
      d[i] = a;
      d[i + stride] = b;
      d[i + 2 * stride] = c;
      d[i + 3 * stride] = e;
    }
    for (; i < row16; i += stride) d[i] = s[i];
  }
}

static int g_copy_sms[64];
static std::mutex g_copy_mu;

cudaError_t launch_stream_copy(const void* src, void* dst, size_t row_bytes, size_t pitch, int rows,
                               cudaStream_t stream) {
  if (rows <= 0 || row_bytes == 0) return cudaSuccess;
  if (row_bytes % 16 || pitch % 16 || reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = 0;
  {
    std::lock_guard<std::mutex> g(g_copy_mu);
    if (g_copy_sms[dev] == 0) {
      err = cudaDeviceGetAttribute(&g_copy_sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (err != cudaSuccess) return err;
    }
    sms = g_copy_sms[dev];
  }
  // one CTA of 256 threads per SM: enough bytes in flight for the host link,
  // and small enough to sit beside the update kernel's CTAs
  const long long row16 = (long long)(row_bytes / 16);
  long long grid = (row16 + 255) / 256;
  if (grid > sms) grid = sms;
  lst_stream_copy_kernel<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const char*>(src), static_cast<char*>(dst),
                                                              row16, (long long)pitch, rows);
  return cudaGetLastError();
}

}  // namespace lst
