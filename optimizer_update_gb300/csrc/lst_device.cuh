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

__device__ __forceinline__ float adamw_elem(float g, float w, float& m, float& v, const Scalars& s) {
  const float m_new = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.one_minus_beta1, g));
  const float v_new = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.one_minus_beta2, __fmul_rn(g, g)));
  m = m_new;
  v = v_new;
  const float m_hat = __fdiv_rn(m_new, s.bias_correction1);
  const float v_hat = __fdiv_rn(v_new, s.bias_correction2);
  const float u = __fdiv_rn(m_hat, __fadd_rn(__fsqrt_rn(v_hat), s.eps));
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
    w.x = adamw_elem(q.g.x, q.w.x, q.m.x, q.v.x, s);
    w.y = adamw_elem(q.g.y, q.w.y, q.m.y, q.v.y, s);
    w.z = adamw_elem(q.g.z, q.w.z, q.m.z, q.v.z, s);
    w.w = adamw_elem(q.g.w, q.w.w, q.m.w, q.v.w, s);
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
