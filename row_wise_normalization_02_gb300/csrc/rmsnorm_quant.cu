// RMSNorm forward and fused residual-add forward with quantised outputs, for
// sm_103a.
//
// The quantised-output norms named in "TIRx kernels", Kernels list
// (flashinfer.norm: rmsnorm_quant, fused_add_rmsnorm_quant, rmsnorm_fp4quant,
// add_rmsnorm_fp4quant; the NVFP4 format of flashinfer.quantization:
// nvfp4_quantize) replace the forward's output y by
//   FP8    E4M3 codes q_ij = e4m3(y_ij / s_i) with one fp32 scale per row,
//          s_i = max_j |y_ij| / 448;
//   NVFP4  E2M1 codes q_j = e2m1(y_j * gs / S_b) in blocks of 16 consecutive
//          elements, with the block scale S_b = e4m3(gs * max_b |y| / 6)
//          stored as an E4M3 byte and gs the caller's global scale.
// The pages name these operations only; the formulas are the plain readings
// of the names.  Writes shrink from 2 bytes (bf16) to 1 (FP8) or 0.5625
// (NVFP4) per element; the kernels keep the plain forward's structure (one
// 16-byte-vector read of the row into registers, one reduction, vector
// stores of the codes), so they stay HBM-bound.
//
// FP8: y_ij / s_i equals x_ij gamma_j * 448 / max_k |x_ik gamma_k| exactly
// (rstd cancels), so the row reduction carries max |x gamma| beside the sum
// of squares and the codes come from x * gamma alone: one reduction per row,
// and codes untouched by the fp32 error of rstd.  s_i = rstd_i * max / 448.
// NVFP4: likewise y = (x gamma) * rstd, so the block maximum is taken over
// x * gamma (a block's 16 elements sit in 2 (bf16) or 4 (fp32) neighbouring
// lanes, whose maxima combine with xor shuffles) and scaled by rstd * gs / 6,
// and the codes are x * gamma * (rstd * gs / S_b), with gs / S_b looked up in
// a 128-entry table each CTA builds once (no division per block).  The lane
// holding the block's first vector writes its scale byte.  The ALU work per
// element is then unpack, one multiply, one max, one multiply and half a
// conversion; the multiplies, the sum of squares and the fused add run as
// paired fp32 instructions and the maxima as three-input max, which keeps the
// kernel under the issue rate the HBM stream allows.
//
// Conversions use the sm_100-family cvt.rn.satfinite forms (round to nearest
// even, saturate to the largest finite value), which are the reading's
// rounding.  An all-zero row (FP8) or block (NVFP4) gives scale 0 and codes 0.
#include "rmsnorm_fwd_common.cuh"
#include "rmsnorm_ring.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif

namespace rmsn {
namespace {

// ---------------------------------------------------------------- conversions

// In cvt's packed forms the first source lands in the upper half of the
// destination, the second in the lower half: element 0 is passed second so it
// ends up in the lowest byte (E4M3) or nibble (E2M1).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFFu;
}

// Value of a non-negative, non-NaN E4M3 code: exponent field e (bias 7) and
// 3 fraction bits f; e = 0 is subnormal, f * 2^-9.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, f = c & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (f << 20)) : (float)f * 0x1p-9f;
}

__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
        "f"(v[7]));
  return w;
}

__device__ __forceinline__ uint16_t e2m1x4(const float (&v)[4]) {
  uint16_t w;
  asm("{\n\t.reg .b8 b0, b1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "mov.b16 %0, {b0, b1};\n\t}"
      : "=h"(w)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]));
  return w;
}

__device__ __forceinline__ uint8_t e2m1x2(float lo, float hi) {
  float v[4] = {lo, hi, 0.f, 0.f};
  return (uint8_t)(e2m1x4(v) & 0xFFu);
}

// ---------------------------------------------------------------- stores

__device__ __forceinline__ void st_cs(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cs(void* p, uint16_t v) {
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}
__device__ __forceinline__ void st_cs(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// E4M3 codes of one vector's E values: E bytes at dst (E-byte aligned).
[[maybe_unused]] __device__ __forceinline__ void store_fp8(char* dst, const float (&o)[8]) {
  st_cs(dst, e4m3x4(o[0], o[1], o[2], o[3]), e4m3x4(o[4], o[5], o[6], o[7]));
}
[[maybe_unused]] __device__ __forceinline__ void store_fp8(char* dst, const float (&o)[4]) {
  st_cs(dst, e4m3x4(o[0], o[1], o[2], o[3]));
}
// E2M1 codes of one vector's E values: E / 2 bytes at dst, or zeros.
[[maybe_unused]] __device__ __forceinline__ void store_fp4(char* dst, const float (&o)[8], bool zero) {
  st_cs(dst, zero ? 0u : e2m1x8(o));
}
[[maybe_unused]] __device__ __forceinline__ void store_fp4(char* dst, const float (&o)[4], bool zero) {
  st_cs(dst, zero ? (uint16_t)0 : e2m1x4(o));
}

// ---------------------------------------------------------------- reductions

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// CTA-wide sum of s and maximum of m in one barrier (red: 2 x 64 floats,
// `parity` alternating between calls as in cta_sum).
__device__ __forceinline__ void cta_sum_max(float& s, float& m, float* red, int parity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  s = group_sum<32>(s);
  m = group_max<32>(m);
  float* buf = red + parity * 64;
  if (lane == 0) {
    buf[warp] = s;
    buf[32 + warp] = m;
  }
  __syncthreads();
  float ts = 0.f, tm = 0.f;
  for (int w = 0; w < nwarps; ++w) {
    ts += buf[w];
    tm = fmaxf(tm, buf[32 + w]);
  }
  s = ts;
  m = tm;
}

// Maximum of three values (the sm_100-family three-input form).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two bf16 values packed in x_word against the two in g_word, with the
// mixed-precision FMA (bf16 sources, fp32 result, one rounding): the products
// x * g, exact in fp32 (the addend -0 keeps the sign of a zero product), and
// acc += x * x for each.  No unpacking of either operand.
__device__ __forceinline__ void bf16_pair_products(uint32_t x_word, uint32_t g_word, float& p0,
                                                   float& p1, float& acc) {
  asm("{\n\t.reg .b16 xl, xh, gl, gh;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "mov.b32 {gl, gh}, %4;\n\t"
      "fma.rn.f32.bf16 %0, xl, gl, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %1, xh, gh, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %2, xl, xl, %2;\n\t"
      "fma.rn.f32.bf16 %2, xh, xh, %2;\n\t}"
      : "=f"(p0), "=f"(p1), "+f"(acc)
      : "r"(x_word), "r"(g_word));
}

// x * gamma of two bf16 pairs' worth of packed words (mixed-precision FMA,
// exact products, the addend -0 keeping a zero product's sign).
[[maybe_unused]] __device__ __forceinline__ void bf16_pair_mul(uint32_t x_word, uint32_t g_word, float& p0,
                                              float& p1) {
  asm("{\n\t.reg .b16 xl, xh, gl, gh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "mov.b32 {gl, gh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, xl, gl, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %1, xh, gh, 0f80000000;\n\t}"
      : "=f"(p0), "=f"(p1)
      : "r"(x_word), "r"(g_word));
}

// The products x * gamma of one vector, recomputed where the epilogue uses
// them: holding the row pass's products across the reduction would take
// 4 * E registers per thread and a third of the resident CTAs.
template <typename TX, typename TW, int E, int GW>
__device__ __forceinline__ void vec_products(uint4 xv, const uint4 (&gw)[GW],
                                             float2 (&pp)[E / 2]) {
  xv = opaque(xv);
  uint4 gk[GW];
#pragma unroll
  for (int w = 0; w < GW; ++w) gk[w] = opaque(gw[w]);
  if constexpr (std::is_same<TX, bf16>::value && std::is_same<TW, bf16>::value) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t gwd[4] = {gk[0].x, gk[0].y, gk[0].z, gk[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) bf16_pair_mul(xw[i], gwd[i], pp[i].x, pp[i].y);
  } else {
    float f[E], g[E];
    unpack(xv, f);
    unpack_gamma<TW, E, GW>(gk, g);
#pragma unroll
    for (int i = 0; i < E / 2; ++i)
      pp[i] = __fmul2_rn(make_float2(f[2 * i], f[2 * i + 1]), make_float2(g[2 * i], g[2 * i + 1]));
  }
}

// One pass over a thread's slice of the row, in pairs of elements with the
// paired fp32 instructions (each lane rounds exactly as the scalar op):
// fused add: h = round(r + x), stored over the residual; then the products
// p = x * gamma (kept for the epilogue), the maximum |p| of every vector, and
// the sum of squares of x in two partial sums added at the end.  bf16 x and
// gamma skip the unpacking: products and squares come from the packed words
// through the mixed-precision FMA.
// PROD = false (NVFP4: the block maxima are only needed after the row's
// reduction) skips the products and maxima: the pass is the sum of squares
// (and the fused add) alone.
// Vector of slot k of lane `lane` (L lanes per row): lane + k L, or with
// BV > 1 the BV consecutive vectors of one NVFP4 block per group of BV slots.
template <int BV>
__device__ __forceinline__ int qvec(int lane, int k, int L) {
  if constexpr (BV > 1) return BV * (lane + (k / BV) * L) + k % BV;
  else return lane + k * L;
}

template <typename TX, typename TW, int VPT, bool FUSED, bool PROD = true, int BV = 1,
          int E = Cfg<TX, TW>::E, int GW = Cfg<TX, TW>::GW>
__device__ __forceinline__ float quant_row_pass(Slice<VPT, FUSED>& s, const uint4 (&gw)[VPT][GW],
                                                float2 (&pr)[VPT][E / 2], float (&vmax)[VPT],
                                                char* hrow, int lane, int L, int nvec,
                                                bool valid) {
  float2 acc = make_float2(0.f, 0.f);
  float acc1 = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    float f[E], g[E];
    unpack(s.x[k], f);
    if constexpr (FUSED) {
      float rf[E];
      unpack(s.r[k], rf);
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        const float2 t = __fadd2_rn(make_float2(f[2 * i], f[2 * i + 1]),
                                    make_float2(rf[2 * i], rf[2 * i + 1]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
      }
      s.x[k] = pack(f);   // rounds to TX (nearest even)
      unpack(s.x[k], f);  // the stored h, exactly
      const int v = qvec<BV>(lane, k, L);
      if (valid && v < nvec) st_stream(hrow + (size_t)v * 16, s.x[k]);
    }
    float m = 0.f;
    if constexpr (!PROD && !FUSED && std::is_same<TX, bf16>::value) {
      bf16x8_sumsq(s.x[k], acc.x, acc.y);   // squares from the packed words
    } else if constexpr (!PROD) {
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        const float2 x2 = make_float2(f[2 * i], f[2 * i + 1]);
        acc = __ffma2_rn(x2, x2, acc);
      }
    } else if constexpr (std::is_same<TX, bf16>::value && std::is_same<TW, bf16>::value) {
      const uint32_t xw[4] = {s.x[k].x, s.x[k].y, s.x[k].z, s.x[k].w};
      const uint32_t gwd[4] = {gw[k][0].x, gw[k][0].y, gw[k][0].z, gw[k][0].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float p0, p1;
        bf16_pair_products(xw[i], gwd[i], p0, p1, acc1);
        pr[k][i] = make_float2(p0, p1);
        m = max3(m, fabsf(p0), fabsf(p1));
      }
    } else {
      unpack_gamma<TW, E, GW>(gw[k], g);
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        const float2 x2 = make_float2(f[2 * i], f[2 * i + 1]);
        acc = __ffma2_rn(x2, x2, acc);
        pr[k][i] = __fmul2_rn(x2, make_float2(g[2 * i], g[2 * i + 1]));
        m = max3(m, fabsf(pr[k][i].x), fabsf(pr[k][i].y));
      }
    }
    vmax[k] = m;
  }
  return acc.x + acc.y + acc1;
}

// ---------------------------------------------------------------------------
// Aligned rows: G lanes per row (G in 4..32, 256 / G rows per CTA iteration)
// or, with G = 0, the whole CTA per row; persistent grid, gamma in registers.
// PF: the next row's loads are issued before the current row is reduced.
// Registers: 128 caps the CTA form (up to 512 threads); the plain forms with
// 4 vectors per thread and prefetch are held to 80 so that three 256-thread
// CTAs fit an SM (NVFP4 otherwise takes 96 and two; no spills at 80).
// A row slice with the vectors of qvec<BV> (BV = 1: load_aligned's).
template <typename TX, int VPT, bool FUSED, int BV>
__device__ __forceinline__ void load_quant(Slice<VPT, FUSED>& s, const FwdParams& p, int64_t row,
                                           bool valid, int lane, int L) {
  if constexpr (BV == 1) {
    load_aligned<TX, VPT, FUSED>(s, p, row, valid, lane, L);
  } else {
    const size_t rb = (size_t)p.N * sizeof(TX);
    const char* xr = static_cast<const char*>(p.x) + row * rb;
    const char* rr = static_cast<const char*>(p.residual) + row * rb;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = qvec<BV>(lane, k, L);
      const bool in = valid && v < p.nvec;
      s.x[k] = in ? ld_stream(xr + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
      if (FUSED) s.r[k] = in ? ld_rw(rr + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
    }
  }
}

template <int G, int VPT, bool FUSED, int OUT, bool PF>
constexpr int quant_max_regs() {
  return G ? 255 : (VPT == 4 && PF && !FUSED) ? 80 : 128;
}

template <typename TX, typename TW, int G, int VPT, bool FUSED, int OUT, bool PF>
__global__ void __maxnreg__((quant_max_regs<G, VPT, FUSED, OUT, PF>()))
    fwd_quant_kernel(const FwdParams p) {
  {  // the first two iterations' rows into L2 while the previous kernel ends
    const int rpc0 = G ? kSubwarpThreads / G : 1;
    const int64_t b0 = (int64_t)blockIdx.x * rpc0, st = (int64_t)gridDim.x * rpc0;
    const size_t rb0 = (size_t)p.N * sizeof(TX);
    const void* r = FUSED ? p.residual : nullptr;
    l2_warm(p.x, r, nullptr, b0, rpc0, p.M, rb0);
    if (PF) l2_warm(p.x, r, nullptr, b0 + st, rpc0, p.M, rb0);
  }
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW;
  constexpr int VB = 16 / E;                       // vectors per NVFP4 block
  static_assert(G == 0 || G >= VB, "a block must sit inside one row group");
  __shared__ float red[128];
  const int L = G ? G : (int)blockDim.x;           // lanes per row
  const int lane = G ? (int)threadIdx.x % G : (int)threadIdx.x;
  const int rpc = G ? kSubwarpThreads / G : 1;
  const int grp = G ? (int)threadIdx.x / G : 0;
  // NVFP4 with one row per CTA: each thread holds whole blocks (BV
  // consecutive vectors), so a block's maximum, scale and codes need no
  // shuffle and are formed once (16384 x 8192 bf16: 0.89 -> 0.94 of the copy
  // peak).  Not for the fused add, whose h stores would then leave every
  // warp store half a sector at a time (0.98 against 1.0).
  constexpr int BV = (OUT == kOutNvfp4 && G == 0 && !FUSED && VPT % VB == 0) ? VB : 1;

  uint4 gw[VPT][GW];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = qvec<BV>(lane, k, L);
#pragma unroll
    for (int w = 0; w < GW; ++w)
      gw[k][w] = v < p.nvec ? ld_cached(static_cast<const char*>(p.gamma) +
                                        ((size_t)v * GW + w) * 16)
                            : make_uint4(0, 0, 0, 0);
  }
  const float gs = p.gs;
  const float gs6 = __fdiv_rn(gs, 6.f);
  // NVFP4: gs / S for every E4M3 code c below 0x80 (0 for c = 0)
  __shared__ float os_tab[128];
  if constexpr (OUT == kOutNvfp4) {
    for (int c = threadIdx.x; c < 128; c += blockDim.x)
      os_tab[c] = c ? __fdiv_rn(gs, e4m3_value((uint32_t)c)) : 0.f;
    __syncthreads();
  }
  const size_t rb = (size_t)p.N * sizeof(TX);
  const int64_t stride = (int64_t)gridDim.x * rpc;
  int parity = 0;

  int64_t base = (int64_t)blockIdx.x * rpc;
  Slice<VPT, FUSED> s, nxt;
  load_quant<TX, VPT, FUSED, BV>(s, p, base + grp, base + grp < p.M, lane, L);
  for (; base < p.M; base += stride) {
    const int64_t row = base + grp;
    const bool valid = row < p.M;
    const int64_t nrow = row + stride;
    if (PF) load_quant<TX, VPT, FUSED, BV>(nxt, p, nrow, nrow < p.M, lane, L);
    float2 pr[VPT][E / 2];
    float vmax[VPT];
    float ss = quant_row_pass<TX, TW, VPT, FUSED, OUT == kOutFp8, BV>(
        s, gw, pr, vmax, static_cast<char*>(p.residual) + row * rb, lane, L, p.nvec, valid);
    float mx = 0.f;
    if constexpr (OUT == kOutFp8) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) mx = fmaxf(mx, vmax[k]);
    }
    if constexpr (G != 0) {
      ss = group_sum<G>(ss);
      if constexpr (OUT == kOutFp8) mx = group_max<G>(mx);
    } else {
      if constexpr (OUT == kOutFp8) {
        cta_sum_max(ss, mx, red, parity);
      } else {
        float t[1] = {ss};
        cta_sum<1>(t, red, parity);
        ss = t[0];
      }
      parity ^= 1;
    }
    const float rs = rsqrtf(fmaf(ss, p.inv_n, p.eps));
    if (valid && lane == 0 && p.rstd != nullptr) p.rstd[row] = rs;

    if constexpr (OUT == kOutFp8) {
      const float inv = mx > 0.f ? __fdiv_rn(448.f, mx) : 0.f;
      const float2 inv2 = make_float2(inv, inv);
      if (valid && lane == 0)
        static_cast<float*>(p.qs)[row] = mx > 0.f ? __fdiv_rn(rs * mx, 448.f) : 0.f;
      char* qrow = static_cast<char*>(p.y) + row * (size_t)p.N;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lane + k * L;
        if (valid && v < p.nvec) {
          float o[E];
          float2 pp[E / 2];
          vec_products<TX, TW, E, GW>(s.x[k], gw[k], pp);
#pragma unroll
          for (int i = 0; i < E / 2; ++i) {
            const float2 t = __fmul2_rn(pp[i], inv2);
            o[2 * i] = t.x;
            o[2 * i + 1] = t.y;
          }
          store_fp8(qrow + (size_t)v * E, o);
        }
      }
    } else {
      char* qrow = static_cast<char*>(p.y) + row * (size_t)(p.N / 2);
      uint8_t* sfrow = static_cast<uint8_t*>(p.qs) + row * (size_t)(p.N / 16);
      const float rg6 = rs * gs6;
      if constexpr (BV > 1) {
        // whole blocks per thread: slots j BV .. j BV + BV - 1 are the block's
        // vectors v0 .. v0 + BV - 1
#pragma unroll
        for (int jb = 0; jb < VPT / BV; ++jb) {
          const int v0 = qvec<BV>(lane, jb * BV, L);
          float2 pp[BV][E / 2];
          float a = 0.f;
#pragma unroll
          for (int q = 0; q < BV; ++q) {
            vec_products<TX, TW, E, GW>(s.x[jb * BV + q], gw[jb * BV + q], pp[q]);
#pragma unroll
            for (int i = 0; i < E / 2; ++i) a = max3(a, fabsf(pp[q][i].x), fabsf(pp[q][i].y));
          }
          if (valid && v0 < p.nvec) {
            const uint32_t code = a > 0.f ? e4m3_code(a * rg6) : 0u;
            const float sc = rs * os_tab[code & 127u];
            const float2 sc2 = make_float2(sc, sc);
            sfrow[v0 / VB] = (uint8_t)code;
            uint32_t w[2];   // the block's 16 codes: 8 bytes
#pragma unroll
            for (int q = 0; q < BV; ++q) {
              float o[E];
#pragma unroll
              for (int i = 0; i < E / 2; ++i) {
                const float2 t = __fmul2_rn(pp[q][i], sc2);
                o[2 * i] = t.x;
                o[2 * i + 1] = t.y;
              }
              if constexpr (E == 8) {
                w[q] = e2m1x8(o);
              } else {
                const uint32_t h = e2m1x4(o);
                if (q % 2 == 0) w[q / 2] = h;
                else w[q / 2] |= h << 16;
              }
            }
            if (code == 0u) w[0] = w[1] = 0u;
            st_cs(qrow + (size_t)v0 * (E / 2), w[0], w[1]);
          }
        }
      } else {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lane + k * L;
        // the products, formed once here (lanes past the row hold zeros)
        float2 pp[E / 2];
        vec_products<TX, TW, E, GW>(s.x[k], gw[k], pp);
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < E / 2; ++i) a = max3(a, fabsf(pp[i].x), fabsf(pp[i].y));
        // every lane takes part: the block's other vectors are in lanes ^1 (^2)
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        if constexpr (VB == 4) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        // an all-zero block gets code 0 even when rstd is infinite (eps = 0)
        const uint32_t code = a > 0.f ? e4m3_code(a * rg6) : 0u;
        const float sc = rs * os_tab[code & 127u];
        const float2 sc2 = make_float2(sc, sc);
        if (valid && v < p.nvec) {
          if (v % VB == 0) sfrow[v / VB] = (uint8_t)code;
          float o[E];
#pragma unroll
          for (int i = 0; i < E / 2; ++i) {
            const float2 t = __fmul2_rn(pp[i], sc2);
            o[2 * i] = t.x;
            o[2 * i + 1] = t.y;
          }
          store_fp4(qrow + (size_t)v * (E / 2), o, code == 0u);
        }
      }
      }
    }
    if (PF) s = nxt;
    else load_quant<TX, VPT, FUSED, BV>(s, p, nrow, nrow < p.M, lane, L);
  }
}

// ---------------------------------------------------------------------------
// Staged: one row per CTA iteration as above, but the rows ([x], or [r | x]
// fused) arrive by bulk copies into the shared-memory ring of rmsnorm_ring.cuh,
// `stages` rows ahead of the CTA, so the bytes in flight per SM are set by the
// ring rather than by registers.  Every wait is bounded; a wait that runs out
// is voted on at the reduction barrier, the CTA stores nothing for that row
// and leaves, and thread 0 drains its copies and raises kStatusWaitTimeout.

// cta_sum_max whose barrier also votes on `pred` (true in every thread when
// true in any).
__device__ __forceinline__ bool cta_sum_max_vote(float& s, float& m, float* red, int parity,
                                                 bool pred) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  s = group_sum<32>(s);
  m = group_max<32>(m);
  float* buf = red + parity * 64;
  if (lane == 0) {
    buf[warp] = s;
    buf[32 + warp] = m;
  }
  const bool any = __syncthreads_or(pred ? 1 : 0) != 0;
  float ts = 0.f, tm = 0.f;
  for (int w = 0; w < nwarps; ++w) {
    ts += buf[w];
    tm = fmaxf(tm, buf[32 + w]);
  }
  s = ts;
  m = tm;
  return any;
}

template <typename TX, typename TW, int VPT, bool FUSED, int OUT>
__global__ void __launch_bounds__(kCtaMaxThreads) fwd_quant_staged_kernel(const FwdParams p) {
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW;
  constexpr int VB = 16 / E;
  constexpr int NS = FUSED ? 2 : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float os_tab[128];
  const Ring rg = ring_of(smem);
  const int tid = threadIdx.x, T = blockDim.x, S = p.stages;
  const size_t rb = (size_t)p.N * sizeof(TX);
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nrows = first < p.M ? (p.M - 1 - first) / stride + 1 : 0;
  const char* xs = static_cast<const char*>(p.x);
  const char* rsrc = static_cast<const char*>(p.residual);
  const float gs = p.gs;
  const float gs6 = __fdiv_rn(gs, 6.f);
  if constexpr (OUT == kOutNvfp4) {
    for (int c = tid; c < 128; c += T) os_tab[c] = c ? __fdiv_rn(gs, e4m3_value((uint32_t)c)) : 0.f;
  }
  // (the barrier inside ring_start also publishes os_tab)
  int64_t issued =
      ring_start<NS>(rg, S, nrows, first, stride, FUSED ? rsrc : xs, xs, nullptr, rb);

  uint4 gw[VPT][GW];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
#pragma unroll
    for (int w = 0; w < GW; ++w)
      gw[k][w] = v < p.nvec ? ld_cached(static_cast<const char*>(p.gamma) +
                                        ((size_t)v * GW + w) * 16)
                            : make_uint4(0, 0, 0, 0);
  }

  int parity = 0;
  int64_t i = 0;
  bool failed = false;
  for (; i < nrows; ++i) {
    const int st_i = (int)(i % S);
    const int64_t row = first + i * stride;
    const bool late =
        !mbar_wait_bounded(rg.full + st_i, (uint32_t)((i / S) & 1), p.wait_limit);
    const uint4* stg = reinterpret_cast<const uint4*>(rg.buf + (size_t)st_i * NS * rb);
    Slice<VPT, FUSED> sl;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      const bool in = v < p.nvec && !late;
      sl.x[k] = in ? stg[FUSED ? p.nvec + v : v] : make_uint4(0, 0, 0, 0);
      if constexpr (FUSED) sl.r[k] = in ? stg[v] : make_uint4(0, 0, 0, 0);
    }
    // h is stored only once the CTA knows that no wait ran out (below)
    float2 pr[VPT][E / 2];
    float vmax[VPT];
    float ss = quant_row_pass<TX, TW, VPT, FUSED>(sl, gw, pr, vmax, nullptr, tid, T, 0, false);
    float mx = 0.f;
    bool any_late;
    if constexpr (OUT == kOutFp8) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) mx = fmaxf(mx, vmax[k]);
      any_late = cta_sum_max_vote(ss, mx, rg.red, parity, late);
    } else {
      float t[1] = {ss};
      any_late = cta_sum_vote<1>(t, rg.red, parity, late);
      ss = t[0];
    }
    if (any_late) {
      failed = true;
      break;
    }
    parity ^= 1;
    // every thread is past its reads of this stage: refill it
    if (tid == 0 && issued < nrows) {
      fence_proxy_async_smem();
      issue_row<NS>(rg, issued, first, stride, S, FUSED ? rsrc : xs, xs, nullptr, rb);
      ++issued;
    }
    const float rs = rsqrtf(fmaf(ss, p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    if constexpr (FUSED) {
      char* hrow = static_cast<char*>(p.residual) + row * rb;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * T;
        if (v < p.nvec) st_stream(hrow + (size_t)v * 16, sl.x[k]);
      }
    }
    if constexpr (OUT == kOutFp8) {
      const float inv = mx > 0.f ? __fdiv_rn(448.f, mx) : 0.f;
      const float2 inv2 = make_float2(inv, inv);
      if (tid == 0) static_cast<float*>(p.qs)[row] = mx > 0.f ? __fdiv_rn(rs * mx, 448.f) : 0.f;
      char* qrow = static_cast<char*>(p.y) + row * (size_t)p.N;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * T;
        if (v < p.nvec) {
          float o[E];
#pragma unroll
          for (int j = 0; j < E / 2; ++j) {
            const float2 t = __fmul2_rn(pr[k][j], inv2);
            o[2 * j] = t.x;
            o[2 * j + 1] = t.y;
          }
          store_fp8(qrow + (size_t)v * E, o);
        }
      }
    } else {
      char* qrow = static_cast<char*>(p.y) + row * (size_t)(p.N / 2);
      uint8_t* sfrow = static_cast<uint8_t*>(p.qs) + row * (size_t)(p.N / 16);
      const float rg6 = rs * gs6;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * T;
        float a = vmax[k];
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        if constexpr (VB == 4) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        const uint32_t code = a > 0.f ? e4m3_code(a * rg6) : 0u;
        const float sc = rs * os_tab[code & 127u];
        const float2 sc2 = make_float2(sc, sc);
        if (v < p.nvec) {
          if (v % VB == 0) sfrow[v / VB] = (uint8_t)code;
          float o[E];
#pragma unroll
          for (int j = 0; j < E / 2; ++j) {
            const float2 t = __fmul2_rn(pr[k][j], sc2);
            o[2 * j] = t.x;
            o[2 * j + 1] = t.y;
          }
          store_fp4(qrow + (size_t)v * (E / 2), o, code == 0u);
        }
      }
    }
  }
  if (failed && tid == 0) {
    drain(rg, i, issued, S);
    atomicOr(p.status, kStatusWaitTimeout);
  }
}

// ---------------------------------------------------------------------------
// Any row: scalar, one row per CTA iteration, 256 threads.  Pass 1 reads the
// row (fused: forms, rounds and stores h) and reduces; pass 2 re-reads it and
// writes codes byte by byte (NVFP4: one 16-element block per thread).
template <typename TX, typename TW, bool FUSED, int OUT>
__global__ void __launch_bounds__(256) fwd_quant_generic_kernel(const FwdParams p) {
  pdl_begin();
  __shared__ float red[128];
  const int tid = threadIdx.x, T = blockDim.x;
  const int N = p.N;
  const TW* gam = static_cast<const TW*>(p.gamma);
  const float gs = p.gs;
  const float gs6 = __fdiv_rn(gs, 6.f);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const TX* xr = static_cast<const TX*>(p.x) + row * (int64_t)N;
    TX* hr = static_cast<TX*>(p.residual) + row * (int64_t)N;
    float ss = 0.f, mx = 0.f;
    for (int j = tid; j < N; j += T) {
      float v = ld_scalar(xr + j);
      if (FUSED) {
        v = round_to(ld_scalar(hr + j) + v, (TX*)nullptr);
        st_scalar(hr + j, v);
      }
      ss = fmaf(v, v, ss);
      if (OUT == kOutFp8) mx = fmaxf(mx, fabsf(v * ld_scalar_ro(gam + j)));
    }
    if constexpr (OUT == kOutFp8) {
      cta_sum_max(ss, mx, red, parity);
    } else {
      float t[1] = {ss};
      cta_sum<1>(t, red, parity);
      ss = t[0];
    }
    parity ^= 1;
    const float rs = rsqrtf(fmaf(ss, p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    // h written in pass 1 by other threads is visible after the barrier above
    auto in = [&](int j) { return FUSED ? ld_scalar(hr + j) : ld_scalar(xr + j); };
    if constexpr (OUT == kOutFp8) {
      const float inv = mx > 0.f ? __fdiv_rn(448.f, mx) : 0.f;
      if (tid == 0) static_cast<float*>(p.qs)[row] = mx > 0.f ? __fdiv_rn(rs * mx, 448.f) : 0.f;
      uint8_t* q = static_cast<uint8_t*>(p.y) + row * (int64_t)N;
      for (int j = tid; j < N; j += T)
        q[j] = (uint8_t)e4m3_code((in(j) * ld_scalar_ro(gam + j)) * inv);
    } else {
      uint8_t* q = static_cast<uint8_t*>(p.y) + row * (int64_t)(N / 2);
      uint8_t* sfrow = static_cast<uint8_t*>(p.qs) + row * (int64_t)(N / 16);
      for (int b = tid; b < N / 16; b += T) {
        float o[16];
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          o[e] = in(16 * b + e) * rs * ld_scalar_ro(gam + 16 * b + e);
          a = fmaxf(a, fabsf(o[e]));
        }
        const uint32_t code = e4m3_code(a * gs6);
        const float S = e4m3_value(code);
        const float os = S > 0.f ? __fdiv_rn(gs, S) : 0.f;
        sfrow[b] = (uint8_t)code;
#pragma unroll
        for (int e = 0; e < 16; e += 2)
          q[8 * b + e / 2] = S > 0.f ? e2m1x2(o[e] * os, o[e + 1] * os) : (uint8_t)0;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Instantiation table (one dtype pair per translation unit).

template <typename TX, typename TW, bool FUSED, int OUT, bool PF>
FwdKernel pick_shape(const FwdKey& k) {
  if (k.family == kCta) {
    switch (k.vpt) {
      case 1: return fwd_quant_kernel<TX, TW, 0, 1, FUSED, OUT, PF>;
      case 2: return fwd_quant_kernel<TX, TW, 0, 2, FUSED, OUT, PF>;
      case 4: return fwd_quant_kernel<TX, TW, 0, 4, FUSED, OUT, PF>;
      case 8: return PF ? nullptr : fwd_quant_kernel<TX, TW, 0, 8, FUSED, OUT, false>;
      default: return nullptr;
    }
  }
  if (k.family == kSubwarp) {
#define RMSN_Q(G_, V_) \
  if (k.g == G_ && k.vpt == V_) return fwd_quant_kernel<TX, TW, G_, V_, FUSED, OUT, PF>;
    RMSN_Q(4, 1) RMSN_Q(8, 1) RMSN_Q(16, 1) RMSN_Q(32, 1)
    RMSN_Q(8, 2) RMSN_Q(16, 2) RMSN_Q(32, 2) RMSN_Q(32, 3) RMSN_Q(32, 4)
#undef RMSN_Q
  }
  return nullptr;
}

template <typename TX, typename TW, bool FUSED, int OUT>
FwdKernel pick_out(const FwdKey& k) {
  if (k.family == kGeneric) return fwd_quant_generic_kernel<TX, TW, FUSED, OUT>;
  if (k.family == kStaged) {
    switch (k.vpt) {
      case 1: return fwd_quant_staged_kernel<TX, TW, 1, FUSED, OUT>;
      case 2: return fwd_quant_staged_kernel<TX, TW, 2, FUSED, OUT>;
      case 4: return fwd_quant_staged_kernel<TX, TW, 4, FUSED, OUT>;
      default: return nullptr;
    }
  }
  return k.prefetch ? pick_shape<TX, TW, FUSED, OUT, true>(k)
                    : pick_shape<TX, TW, FUSED, OUT, false>(k);
}

template <typename TX, typename TW>
FwdKernel pick_quant(const FwdKey& k) {
  if (k.strided) return nullptr;
  if (k.out == kOutFp8)
    return k.fused ? pick_out<TX, TW, true, kOutFp8>(k) : pick_out<TX, TW, false, kOutFp8>(k);
  if (k.out == kOutNvfp4)
    return k.fused ? pick_out<TX, TW, true, kOutNvfp4>(k) : pick_out<TX, TW, false, kOutNvfp4>(k);
  return nullptr;
}

}  // namespace

#if RMSN_PAIR == 0
FwdKernel get_fwd_quant_f32_f32(const FwdKey& k) { return pick_quant<float, float>(k); }
#elif RMSN_PAIR == 1
FwdKernel get_fwd_quant_bf16_bf16(const FwdKey& k) { return pick_quant<bf16, bf16>(k); }
#else
FwdKernel get_fwd_quant_bf16_f32(const FwdKey& k) { return pick_quant<bf16, float>(k); }
#endif

}  // namespace rmsn
