// Backward building blocks shared by the translation units of the backward
// kernels (register, ring and cluster forms): gamma as fp32, and the
// per-vector row sums and outputs in the paired fp32 instructions of sm_100+
// (__ffma2_rn / __fmul2_rn / __fadd2_rn: two independent fp32 operations per
// instruction, each rounded as its scalar form would be).
#pragma once

#include <type_traits>

#include "rmsnorm_device.cuh"
#include "rmsnorm_internal.h"

namespace rmsn {
namespace {

template <typename TW, int E>
__device__ __forceinline__ void load_gamma_vec(const void* gamma, int v, float (&g)[E]) {
  constexpr int GW = E * (int)sizeof(TW) / 16;
  const char* gp = static_cast<const char*>(gamma) + (size_t)v * GW * 16;
  if constexpr (std::is_same<TW, float>::value) {
#pragma unroll
    for (int w = 0; w < GW; ++w) {
      float t[4];
      unpack(ld_cached(gp + w * 16), t);
#pragma unroll
      for (int i = 0; i < 4; ++i) g[w * 4 + i] = t[i];
    }
  } else {
    unpack(ld_cached(gp), g);
  }
}

// Per-vector work of the register backward kernels with the paired fp32
// instructions.  Row sums: dot += sum g dy x over even / odd elements in two
// lanes (and ss += sum x^2 when the rstd is recomputed).
template <int E, bool SS>
__device__ __forceinline__ void bwd_vec_sums(const uint4& xv, const uint4& dv,
                                             const float (&g)[E], float2& dot, float2& ss) {
  float xf[E], df[E];
  unpack(xv, xf);
  unpack(dv, df);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    const float2 x2 = make_float2(xf[2 * i], xf[2 * i + 1]);
    const float2 gd = __fmul2_rn(make_float2(g[2 * i], g[2 * i + 1]),
                                 make_float2(df[2 * i], df[2 * i + 1]));
    dot = __ffma2_rn(gd, x2, dot);
    if (SS) ss = __ffma2_rn(x2, x2, ss);
  }
}
// dx = r (g dy - x c) (+ dres) and acc += dy x r, element by element with the
// same operations as the scalar form, two at a time.
template <int E, bool DRES>
__device__ __forceinline__ uint4 bwd_vec_apply(const uint4& xv, const uint4& dv,
                                               const uint4& rv, const float (&g)[E], float r,
                                               float c, float (&acc)[E]) {
  float xf[E], df[E], rf[E], o[E];
  unpack(xv, xf);
  unpack(dv, df);
  if (DRES) unpack(rv, rf);
  const float2 r2 = make_float2(r, r), nc = make_float2(-c, -c);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    const float2 x2 = make_float2(xf[2 * i], xf[2 * i + 1]);
    const float2 d2 = make_float2(df[2 * i], df[2 * i + 1]);
    const float2 gd = __fmul2_rn(make_float2(g[2 * i], g[2 * i + 1]), d2);
    float2 t = __fmul2_rn(__ffma2_rn(x2, nc, gd), r2);
    if (DRES) t = __fadd2_rn(t, make_float2(rf[2 * i], rf[2 * i + 1]));
    const float2 a = __ffma2_rn(__fmul2_rn(d2, x2), r2, make_float2(acc[2 * i], acc[2 * i + 1]));
    o[2 * i] = t.x;
    o[2 * i + 1] = t.y;
    acc[2 * i] = a.x;
    acc[2 * i + 1] = a.y;
  }
  return pack(o);
}

}  // namespace
}  // namespace rmsn
