// Forward building blocks shared by the translation units of the forward
// kernels (plain, cluster and quantised outputs): dtype-pair constants, gamma
// unpacking, the register slice of a row with its aligned load and its sum of
// squares (which, for the fused add, also forms, rounds and stores
// h = residual + x), and the scaled output vector.
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

// bf16 rows straight from the packed words, with the mixed-precision FMA
// (bf16 sources, fp32 accumulate, one rounding): the squares of the 8 values
// of v into two accumulators (even / odd elements), no unpacking.
__device__ __forceinline__ void bf16x8_sumsq(const uint4& v, float& a0, float& a1) {
  asm("{\n\t.reg .b16 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      "mov.b32 {l0, h0}, %2;\n\t"
      "mov.b32 {l1, h1}, %3;\n\t"
      "mov.b32 {l2, h2}, %4;\n\t"
      "mov.b32 {l3, h3}, %5;\n\t"
      "fma.rn.f32.bf16 %0, l0, l0, %0;\n\t"
      "fma.rn.f32.bf16 %1, h0, h0, %1;\n\t"
      "fma.rn.f32.bf16 %0, l1, l1, %0;\n\t"
      "fma.rn.f32.bf16 %1, h1, h1, %1;\n\t"
      "fma.rn.f32.bf16 %0, l2, l2, %0;\n\t"
      "fma.rn.f32.bf16 %1, h2, h2, %1;\n\t"
      "fma.rn.f32.bf16 %0, l3, l3, %0;\n\t"
      "fma.rn.f32.bf16 %1, h3, h3, %1;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

// y = (x * g) * rs for 8 bf16 values x and gamma g: the products are exact in
// fp32 (formed from the packed halves by the mixed-precision FMA, addend -0
// to keep a zero product's sign), the scaling is a paired multiply, and each
// result is rounded once to bf16.
__device__ __forceinline__ uint4 bf16x8_scale(const uint4& x, const uint4& g, float rs) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, gw[4] = {g.x, g.y, g.z, g.w};
  float o[8];
  const float2 r2 = make_float2(rs, rs);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float p0, p1;
    asm("{\n\t.reg .b16 xl, xh, gl, gh;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "mov.b32 {gl, gh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, xl, gl, 0f80000000;\n\t"
        "fma.rn.f32.bf16 %1, xh, gh, 0f80000000;\n\t}"
        : "=f"(p0), "=f"(p1)
        : "r"(xw[i]), "r"(gw[i]));
    const float2 t = __fmul2_rn(make_float2(p0, p1), r2);
    o[2 * i] = t.x;
    o[2 * i + 1] = t.y;
  }
  return pack(o);
}

// Sum of squares of this thread's part of the row.  Fused add: the vectors
// become h = round(r + x), which is written back over the residual and kept
// (packed) in s.x for the output pass.
template <typename TX, int VPT, bool FUSED>
__device__ __forceinline__ float slice_sumsq(Slice<VPT, FUSED>& s, char* res_row_vec0, int lane,
                                             int stride, int nvec_valid, bool valid) {
  constexpr int E = Elem<TX>::kPerVec;
  float ss = 0.f, ss1 = 0.f;
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
    if constexpr (std::is_same<TX, bf16>::value) {
      bf16x8_sumsq(s.x[k], ss, ss1);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) ss = fmaf(f[e], f[e], ss);
    }
  }
  return ss + ss1;
}

// One output vector: y = x * rs * gamma, rounded once to TX (bf16 x and
// gamma: (x * gamma) * rs from the packed words, see bf16x8_scale).
template <typename TX, typename TW, int GW = Cfg<TX, TW>::GW>
__device__ __forceinline__ uint4 scale_vec(const uint4& xv, const uint4 (&gw)[GW], float rs) {
  if constexpr (std::is_same<TX, bf16>::value && std::is_same<TW, bf16>::value) {
    return bf16x8_scale(xv, gw[0], rs);
  } else {
    constexpr int E = Cfg<TX, TW>::E;
    float g[E], o[E];
    unpack_gamma<TW, E, GW>(gw, g);
    unpack(xv, o);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = o[e] * rs * g[e];
    return pack(o);
  }
}

}  // namespace
}  // namespace rmsn
