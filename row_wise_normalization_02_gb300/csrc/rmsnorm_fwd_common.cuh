// Forward building blocks shared by the translation units of the forward
// kernels (plain and quantised outputs): dtype-pair constants, gamma
// unpacking, and the register slice of a row with its aligned load and its
// sum of squares (which, for the fused add, also forms, rounds and stores
// h = residual + x).
#pragma once

#include <type_traits>

#include "rmsnorm_device.cuh"
#include "rmsnorm_internal.h"

namespace rmsn {
namespace {

template <typename TX, typename TW>
struct Cfg {
  static constexpr int E = Elem<TX>::kPerVec;            // elements per x vector
  static constexpr int GW = E * (int)sizeof(TW) / 16;    // gamma vectors per x vector
  static_assert(GW >= 1, "unsupported dtype pair");
};

template <typename TW, int E, int GW>
__device__ __forceinline__ void unpack_gamma(const uint4 (&gw)[GW], float (&gf)[E]) {
  if constexpr (std::is_same<TW, float>::value) {
#pragma unroll
    for (int w = 0; w < GW; ++w) {
      float t[4];
      unpack(gw[w], t);
#pragma unroll
      for (int i = 0; i < 4; ++i) gf[w * 4 + i] = t[i];
    }
  } else {
    unpack(gw[0], gf);
  }
}

// Registers of one row slice: VPT vectors of x (and of the residual).
template <int VPT, bool FUSED>
struct Slice {
  uint4 x[VPT];
  uint4 r[FUSED ? VPT : 1];
};

template <typename TX, int VPT, bool FUSED>
__device__ __forceinline__ void load_aligned(Slice<VPT, FUSED>& s, const FwdParams& p,
                                             int64_t row, bool valid, int lane, int stride) {
  const size_t rb = (size_t)p.N * sizeof(TX);
  const char* xr = static_cast<const char*>(p.x) + row * rb;
  const char* rr = static_cast<const char*>(p.residual) + row * rb;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * stride;
    if (valid && v < p.nvec) {
      s.x[k] = ld_stream(xr + (size_t)v * 16);
      if (FUSED) s.r[k] = ld_rw(rr + (size_t)v * 16);
    } else {
      s.x[k] = make_uint4(0, 0, 0, 0);
      if (FUSED) s.r[k] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Sum of squares of this thread's part of the row.  Fused add: the vectors
// become h = round(r + x), which is written back over the residual and kept
// (packed) in s.x for the output pass.
template <typename TX, int VPT, bool FUSED>
__device__ __forceinline__ float slice_sumsq(Slice<VPT, FUSED>& s, char* res_row_vec0, int lane,
                                             int stride, int nvec_valid, bool valid) {
  constexpr int E = Elem<TX>::kPerVec;
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float f[E];
    unpack(s.x[k], f);
    if constexpr (FUSED) {
      float rf[E];
      unpack(s.r[k], rf);
#pragma unroll
      for (int e = 0; e < E; ++e) f[e] += rf[e];
      s.x[k] = pack(f);   // rounds to TX (nearest even)
      unpack(s.x[k], f);  // the stored h, exactly
      const int v = lane + k * stride;
      if (valid && v < nvec_valid) st_stream(res_row_vec0 + (size_t)v * 16, s.x[k]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(f[e], f[e], ss);
  }
  return ss;
}

}  // namespace
}  // namespace rmsn
