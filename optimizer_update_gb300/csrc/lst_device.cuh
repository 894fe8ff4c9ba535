// Device-side building blocks shared by the update kernels (not installed):
// the run table, the per-element arithmetic and the coalesced quad accesses.
#pragma once

#include <cuda_bf16.h>

#include "lst_internal.h"

namespace lst {

struct RunTable {
  int32_t n;
  int32_t pad_;
  struct Entry {
    const void* g;
    void* w;
    float* m;
    float* v;
    void* w16;
    long long tasks;       // elements / 256
    long long first_task;  // global index of this run's first task in the launch
  } r[kMaxRunsPerLaunch];
};
static_assert(sizeof(RunTable) < 30000, "kernel parameter space");

// ---- element math ---------------------------------------------------------

// Adam moments of one element: m' = b1 m + (1-b1) g, v' = b2 v + (1-b2) g^2.
__device__ __forceinline__ void adam_moments(float g, float& m, float& v, const Scalars& s) {
  m = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.one_minus_beta1, g));
  v = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.one_minus_beta2, __fmul_rn(g, g)));
}

// The IEEE division and square root (__fdiv_rn, __fsqrt_rn) leave their fast
// path for a zero operand, and exact zeros are common in optimizer state
// (zero-initialised moments, rows of an embedding that saw no gradient,
// padding): a zero-filled state ran at under half speed. For those operands
// the IEEE result is known exactly - (+-0) / positive = +-0 and sqrt(+0) = +0 -
// so the SAFE form gives each operation a harmless operand where the input is
// zero and selects the exact zero afterwards. The selects cost instructions,
// so callers use the SAFE form only for quads in which some lane of the warp
// holds a zero moment. 0 / 0 (eps = 0 and v = 0) keeps its true operands.
__device__ __forceinline__ float div_pos(float x, float d) {  // x / d for d > 0
  const bool z = (x == 0.0f);
  const float q = __fdiv_rn(z ? 1.0f : x, d);
  return z ? x : q;
}

__device__ __forceinline__ float sqrt_nonneg(float x) {  // sqrt(x) for x >= +0
  const bool z = (x == 0.0f);
  const float r = __fsqrt_rn(z ? 1.0f : x);
  return z ? 0.0f : r;
}

// Bias correction, normalised step and decoupled decay for one element whose
// moments m, v are already updated. Returns the new weight.
template <bool SAFE>
__device__ __forceinline__ float adamw_finish(float w, float m, float v, const Scalars& s) {
  float u;
  if (SAFE) {
    // bias corrections are > 0 (t >= 1, beta < 1)
    const float m_hat = div_pos(m, s.bias_correction1);
    const float v_hat = div_pos(v, s.bias_correction2);
    const float root = (v_hat >= 0.0f) ? sqrt_nonneg(v_hat) : __fsqrt_rn(v_hat);
    const float den = __fadd_rn(root, s.eps);
    u = (den > 0.0f) ? div_pos(m_hat, den) : __fdiv_rn(m_hat, den);
  } else {
    const float m_hat = __fdiv_rn(m, s.bias_correction1);
    const float v_hat = __fdiv_rn(v, s.bias_correction2);
    u = __fdiv_rn(m_hat, __fadd_rn(__fsqrt_rn(v_hat), s.eps));
  }
  return __fsub_rn(__fmul_rn(w, s.decay), __fmul_rn(s.lr, u));
}

__device__ __forceinline__ float sgd_elem(float g, float w, float lr) {
  return __fadd_rn(w, -__fmul_rn(lr, g));
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Two fp32 values -> two bf16 (round to nearest even), low half = first.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---- one quad (4 consecutive elements) per format --------------------------

enum { F_L12 = 0, F_L16M = 1, F_L16F = 2 };

template <int FMT, bool SGD>
struct Quad {
  float4 g, w, m, v;
};

template <int FMT, bool SGD>
__device__ __forceinline__ void load_quad(const RunTable::Entry& R, long long e, Quad<FMT, SGD>& q) {
  if (FMT == F_L16F) {
    q.g = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(R.g) + e));
    q.w = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(R.w) + e));
  } else {
    const uint2 gb = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(R.g) + e));
    q.g = make_float4(bf16_lo(gb.x), bf16_hi(gb.x), bf16_lo(gb.y), bf16_hi(gb.y));
    if (FMT == F_L12) {
      const uint2 wb = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(R.w) + e));
      q.w = make_float4(bf16_lo(wb.x), bf16_hi(wb.x), bf16_lo(wb.y), bf16_hi(wb.y));
    } else {
      q.w = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(R.w) + e));
    }
  }
  if (!SGD) {
    q.m = __ldcs(reinterpret_cast<const float4*>(R.m + e));
    q.v = __ldcs(reinterpret_cast<const float4*>(R.v + e));
  }
}

template <int FMT, bool SGD>
__device__ __forceinline__ void update_store_quad(const RunTable::Entry& R, long long e, Quad<FMT, SGD>& q,
                                                  const Scalars& s) {
  float4 w;
  if (SGD) {
    w.x = sgd_elem(q.g.x, q.w.x, s.lr);
    w.y = sgd_elem(q.g.y, q.w.y, s.lr);
    w.z = sgd_elem(q.g.z, q.w.z, s.lr);
    w.w = sgd_elem(q.g.w, q.w.w, s.lr);
  } else {
    adam_moments(q.g.x, q.m.x, q.v.x, s);
    adam_moments(q.g.y, q.m.y, q.v.y, s);
    adam_moments(q.g.z, q.m.z, q.v.z, s);
    adam_moments(q.g.w, q.m.w, q.v.w, s);
    // one vote per quad: the whole warp takes the zero-safe form if any lane
    // has a zero moment (all 32 lanes of a warp execute this together)
    const bool zero = (q.m.x == 0.0f) | (q.m.y == 0.0f) | (q.m.z == 0.0f) | (q.m.w == 0.0f) | (q.v.x == 0.0f) |
                      (q.v.y == 0.0f) | (q.v.z == 0.0f) | (q.v.w == 0.0f);
    if (__any_sync(0xffffffffu, zero)) {
      w.x = adamw_finish<true>(q.w.x, q.m.x, q.v.x, s);
      w.y = adamw_finish<true>(q.w.y, q.m.y, q.v.y, s);
      w.z = adamw_finish<true>(q.w.z, q.m.z, q.v.z, s);
      w.w = adamw_finish<true>(q.w.w, q.m.w, q.v.w, s);
    } else {
      w.x = adamw_finish<false>(q.w.x, q.m.x, q.v.x, s);
      w.y = adamw_finish<false>(q.w.y, q.m.y, q.v.y, s);
      w.z = adamw_finish<false>(q.w.z, q.m.z, q.v.z, s);
      w.w = adamw_finish<false>(q.w.w, q.m.w, q.v.w, s);
    }
    __stcs(reinterpret_cast<float4*>(R.m + e), q.m);
    __stcs(reinterpret_cast<float4*>(R.v + e), q.v);
  }
  if (FMT == F_L12) {
    uint2 wb = make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w));
    __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(R.w) + e), wb);
  } else {
    __stcs(reinterpret_cast<float4*>(static_cast<float*>(R.w) + e), w);
    if (FMT == F_L16M) {
      uint2 wb = make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w));
      __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(R.w16) + e), wb);
    }
  }
}

constexpr int kThreads = 256;

}  // namespace lst
