/*
 * The seeded synthetic input generator of gen.c, on the GPU: a gradient
 * producer that stands in for a backward pass.
 *
 * This file produces INPUT data only. It holds none of the optimizer's
 * arithmetic, and neither the optimizer library nor the oracle includes or
 * links it. Value i of stream s under seed S is the same pure function of
 * (S, s, i) as in gen.c:
 *   key  = splitmix64(S ^ splitmix64(s))
 *   h    = splitmix64(key + i)
 *   k    = (h & 0xffff) + (h>>16 & 0xffff) + (h>>32 & 0xffff) + (h>>48) - 131070
 *   x    = (float)k * scale            (exact conversion, one IEEE fp32 multiply)
 * bf16 outputs are the upper 16 bits of x; the squared kind stores x * x.
 * Integer steps plus correctly rounded fp32 multiplies give the same bits on
 * the host and on the device (a GPU test checks this on sampled indices).
 *
 * splitmix64 is the published mixing function of Steele, Lea and Flood
 * ("Fast splittable pseudorandom number generators", OOPSLA 2014).
 *
 * A backward pass costs time on the SMs before a layer's gradient is ready.
 * `passes` > 1 makes the producer do passes - 1 extra rounds of the same hash
 * per element (folded into a value that is kept only in the practically
 * impossible case that it equals a runtime sentinel, so the compiler cannot
 * drop the rounds) before it writes the value: the written values do not
 * depend on `passes`. The loop is bounded; nothing waits on anything.
 *
 * Build: nvcc -O3 -shared -Xcompiler -fPIC -gencode arch=compute_103a,code=sm_103a
 *        -fmad=false gen_dev.cu -o libsynth_dev.so
 */
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__host__ __device__ inline uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

__device__ inline float draw(uint64_t key, uint64_t i, float scale) {
  const uint64_t h = splitmix64(key + i);
  const int k = (int)(h & 0xffffu) + (int)((h >> 16) & 0xffffu) + (int)((h >> 32) & 0xffffu) + (int)(h >> 48) -
                131070;
  return __fmul_rn(__int2float_rn(k), scale);
}

enum { KIND_F32 = 0, KIND_BF16 = 1, KIND_SQ_F32 = 2 };

__device__ unsigned long long g_sink;  // written only if the extra rounds hit the sentinel

__global__ void __launch_bounds__(256) synth_fill_kernel(int kind, uint64_t key, uint64_t start, long long n,
                                                         float scale, void* out, int passes, uint64_t sentinel) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t idx = start + (uint64_t)i;
    uint64_t acc = 0;
    for (int p = 1; p < passes; ++p) acc ^= splitmix64(key + idx + (uint64_t)p * 0x632BE59BD9B4E019ull);
    const float x = draw(key, idx, scale);
    if (kind == KIND_F32)
      static_cast<float*>(out)[i] = x;
    else if (kind == KIND_SQ_F32)
      static_cast<float*>(out)[i] = __fmul_rn(x, x);
    else
      static_cast<uint16_t*>(out)[i] = (uint16_t)(__float_as_uint(x) >> 16);
    if (passes > 1 && acc == sentinel) g_sink = acc;
  }
}

int g_sms[64];

}  // namespace

extern "C" {

/* Values start .. start+n-1 of the stream into device memory `out` (fp32
   for KIND_F32 / KIND_SQ_F32, bf16 bits for KIND_BF16), enqueued on
   cuda_stream. Returns 0 or the CUDA error code. */
__attribute__((visibility("default"))) int synth_dev_fill(int kind, uint64_t seed, uint64_t stream, uint64_t start,
                                                          int64_t n, float scale, void* out, int passes,
                                                          void* cuda_stream) {
  if (n < 0 || (n > 0 && !out) || kind < 0 || kind > 2 || passes < 1) return (int)cudaErrorInvalidValue;
  if (n == 0) return 0;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return (int)err;
  if (dev < 0 || dev >= 64) return (int)cudaErrorInvalidDevice;
  if (g_sms[dev] == 0) {
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return (int)err;
    g_sms[dev] = sms > 0 ? sms : 1;
  }
  // one CTA of 256 threads per SM at most: the producer leaves room on every
  // SM for the work that runs beside it, as a backward pass would share them
  long long grid = (n + 255) / 256;
  if (grid > g_sms[dev]) grid = g_sms[dev];
  const uint64_t key = splitmix64(seed ^ splitmix64(stream));
  synth_fill_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      kind, key, start, (long long)n, scale, out, passes, 0x5A5A5A5A5A5A5A5Aull ^ (uint64_t)passes);
  return (int)cudaGetLastError();
}

/* Zero `bytes` bytes of device memory on cuda_stream (the padding and the
   zero-valued fields of a block). Returns 0 or the CUDA error code. */
__attribute__((visibility("default"))) int synth_dev_zero(void* out, int64_t bytes, void* cuda_stream) {
  if (bytes < 0 || (bytes > 0 && !out)) return (int)cudaErrorInvalidValue;
  if (bytes == 0) return 0;
  return (int)cudaMemsetAsync(out, 0, (size_t)bytes, static_cast<cudaStream_t>(cuda_stream));
}

}  // extern "C"
