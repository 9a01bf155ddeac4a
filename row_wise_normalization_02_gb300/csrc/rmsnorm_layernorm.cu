// LayerNorm forward and backward kernels for sm_103a.
//
// y = (x - mean) / sqrt(var + eps) * gamma + beta per row ("Pre-built kernel
// library guide", section 1.1 LayerNorm: two passes, mean and then the
// variance; vector loads, XOR-shuffle and shared-memory reductions,
// non-temporal output stores).  The pages give no backward; with
// xhat = (x - mean) rstd and g = dy * gamma it is
//   dx = rstd (g - mean(g) - xhat mean(g xhat)),
//   dgamma = sum over rows of dy xhat,   dbeta = sum over rows of dy,
// with the saved mean and rstd when the caller passes them.
//
// Same skeleton as the RMSNorm kernels: the row is read once into registers
// with 16-byte loads, so the guide's second pass (the variance about the
// mean, with the corrected two-pass algorithm) runs over registers, not
// memory; G lanes per row for short rows or
// one CTA per row, persistent grid, next-row prefetch.  The per-element
// arithmetic uses the paired fp32 instructions.  The weight gradients follow
// the deterministic two-stage scheme of the RMSNorm backward: each CTA writes
// one partial row [dgamma | dbeta], and a column reduction sums the partial
// rows in a fixed order.
#include "rmsnorm_fwd_common.cuh"
#include "rmsnorm_ring.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif

namespace rmsn {
namespace {

// Scalar loads each thread issues per operand before using any, in the
// kernels for rows that are not 16-byte aligned (a warp keeps that many
// requests in flight instead of one).
constexpr int kGenericBatch = 4;

// Row reductions: G lanes (shuffles only) or, with G = 0, the whole CTA
// (shuffles, then shared memory; `parity` alternates per call).
template <int G>
__device__ __forceinline__ float row_sum(float v, float* red, int& parity) {
  if constexpr (G != 0) {
    return group_sum<G>(v);
  } else {
    float t[1] = {v};
    cta_sum<1>(t, red, parity);
    parity ^= 1;
    return t[0];
  }
}
template <int G>
__device__ __forceinline__ void row_sum2(float& a, float& b, float* red, int& parity) {
  if constexpr (G != 0) {
    a = group_sum<G>(a);
    b = group_sum<G>(b);
  } else {
    float t[2] = {a, b};
    cta_sum<2>(t, red, parity);
    parity ^= 1;
    a = t[0];
    b = t[1];
  }
}

// VPT 16-byte vectors of row `row` of a row-major activation (zeros beyond
// the row or for an invalid row).
template <typename TX, int VPT>
__device__ __forceinline__ void load_row(uint4 (&dst)[VPT], const void* base, int64_t row,
                                         bool valid, int lane, int L, int nvec, int N) {
  const char* r = static_cast<const char*>(base) + row * (size_t)N * sizeof(TX);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * L;
    dst[k] = (valid && v < nvec) ? ld_stream(r + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
  }
}

// The packed weight vectors matching activation vector v (kept packed in
// registers, unpacked where used).
template <int GW>
__device__ __forceinline__ void load_weight(uint4 (&w)[GW], const void* base, int v, bool on) {
#pragma unroll
  for (int i = 0; i < GW; ++i)
    w[i] = on ? ld_cached(static_cast<const char*>(base) + ((size_t)v * GW + i) * 16)
              : make_uint4(0, 0, 0, 0);
}

// Element arithmetic on bf16 rows straight from the packed words, with the
// mixed-precision FMA (bf16 sources, fp32 addend, one rounding): x * 1 + a is
// x + a rounded once, the same bits as unpacking and adding, in one
// instruction per element instead of an unpack and half a paired add.
// d = x - m for the 8 values of v.
[[maybe_unused]] __device__ __forceinline__ void bf16x8_minus(const uint4& v, float nm, float (&d)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n\t.reg .b16 l, h, one;\n\t"
        "mov.b16 one, 0x3F80;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "fma.rn.f32.bf16 %0, l, one, %3;\n\t"
        "fma.rn.f32.bf16 %1, h, one, %3;\n\t}"
        : "=f"(d[2 * i]), "=f"(d[2 * i + 1])
        : "r"(w[i]), "f"(nm));
}
// a0 += even elements of v, a1 += odd elements (in element order).
[[maybe_unused]] __device__ __forceinline__ void bf16x8_accumulate(const uint4& v, float& a0, float& a1) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n\t.reg .b16 l, h, one;\n\t"
        "mov.b16 one, 0x3F80;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "fma.rn.f32.bf16 %0, l, one, %0;\n\t"
        "fma.rn.f32.bf16 %1, h, one, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w[i]));
}
// p = a * b for 8 bf16 pairs: exact in fp32 (addend -0 keeps a zero
// product's sign), the same bits as unpacking both and multiplying.
[[maybe_unused]] __device__ __forceinline__ void bf16x8_products(const uint4& a, const uint4& b, float (&p)[8]) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, 0f80000000;\n\t"
        "fma.rn.f32.bf16 %1, ah, bh, 0f80000000;\n\t}"
        : "=f"(p[2 * i]), "=f"(p[2 * i + 1])
        : "r"(aw[i]), "r"(bw[i]));
}

// d = x - m for the E values of one activation vector (rounded once).
template <typename TX, int E>
__device__ __forceinline__ void vec_minus(const uint4& v, float nm, float (&d)[E]) {
  if constexpr (std::is_same<TX, bf16>::value) {
    bf16x8_minus(v, nm, d);
  } else {
    unpack(v, d);
    const float2 n2 = make_float2(nm, nm);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      const float2 t = __fadd2_rn(make_float2(d[2 * i], d[2 * i + 1]), n2);
      d[2 * i] = t.x;
      d[2 * i + 1] = t.y;
    }
  }
}
// g = dy * gamma for one activation vector (exact for bf16 pairs).
template <typename TX, typename TW, int E, int GW>
__device__ __forceinline__ void vec_dy_gamma(const uint4& dv, const uint4 (&gk)[GW],
                                             float (&g)[E]) {
  if constexpr (std::is_same<TX, bf16>::value && std::is_same<TW, bf16>::value) {
    bf16x8_products(dv, gk[0], g);
  } else {
    float d[E], w[E];
    unpack(dv, d);
    unpack_gamma<TW, E, GW>(gk, w);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      const float2 t = __fmul2_rn(make_float2(d[2 * i], d[2 * i + 1]),
                                  make_float2(w[2 * i], w[2 * i + 1]));
      g[2 * i] = t.x;
      g[2 * i + 1] = t.y;
    }
  }
}

// Sum of x over a slice (even and odd elements in two accumulators), then
// the sum of (x - m0) and of its square.
template <typename TX, int E, int VPT>
__device__ __forceinline__ float slice_sum(const uint4 (&s)[VPT]) {
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    if constexpr (std::is_same<TX, bf16>::value) {
      bf16x8_accumulate(s[k], acc.x, acc.y);
    } else {
      float f[E];
      unpack(s[k], f);
#pragma unroll
      for (int i = 0; i < E / 2; ++i) acc = __fadd2_rn(acc, make_float2(f[2 * i], f[2 * i + 1]));
    }
  }
  return acc.x + acc.y;
}
// Second pass about the first-pass mean m0: sum of d and of d^2, d = x - m0.
template <typename TX, int E, int VPT>
__device__ __forceinline__ void slice_dev(const uint4 (&s)[VPT], float m0, int lane, int L,
                                          int nvec, float& sd, float& sq) {
  float2 a1 = make_float2(0.f, 0.f), a2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    if (lane + k * L >= nvec) continue;   // padding lanes hold zeros, not x
    float f[E];
    vec_minus<TX, E>(s[k], -m0, f);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      const float2 d = make_float2(f[2 * i], f[2 * i + 1]);
      a1 = __fadd2_rn(a1, d);
      a2 = __ffma2_rn(d, d, a2);
    }
  }
  sd = a1.x + a1.y;
  sq = a2.x + a2.y;
}

// Row statistics by the corrected two-pass algorithm (Chan, Golub and
// LeVeque): m0 = sum(x) / N, then with d = x - m0 the correction
// c = sum(d) / N and var = sum(d^2) / N - c^2.  The fp32 rounding of the
// first sum moves m0 by a few ulp of the row's magnitude; c takes it back, so
// x - mean stays accurate for rows whose mean is large against their spread.
// Outputs use (x - m0) - c.
struct RowStats {
  float m0, c, rs;
};
template <int G, typename TX, int E, int VPT>
__device__ __forceinline__ RowStats row_stats(const uint4 (&s)[VPT], float* red, int& parity,
                                              int lane, int L, int nvec, float inv_n,
                                              float eps) {
  RowStats st;
  st.m0 = row_sum<G>(slice_sum<TX, E, VPT>(s), red, parity) * inv_n;
  float sd, sq;
  slice_dev<TX, E, VPT>(s, st.m0, lane, L, nvec, sd, sq);
  row_sum2<G>(sd, sq, red, parity);
  st.c = sd * inv_n;
  st.rs = rsqrtf(fmaxf(fmaf(sq, inv_n, -st.c * st.c), 0.f) + eps);
  return st;
}

// The rows [base, base + rows) of a row-major activation, from `ahead`
// iterations of the CTA's walk later, requested into L2 by one thread.
__device__ __forceinline__ void l2_ahead(const void* a, const LnParams& p, int64_t base,
                                         int64_t stride, int rows, size_t rb) {
  if (p.l2_rows <= 0 || threadIdx.x != 0) return;
  l2_prefetch_rows(a, base + (int64_t)p.l2_rows * stride, rows, p.M, rb);
}

// ---------------------------------------------------------------------------
// Forward: G lanes per row (G in 4..32) or, with G = 0, one CTA per row.
template <typename TX, typename TW, int G, int VPT, bool PF>
__global__ void __launch_bounds__(G ? kSubwarpThreads : kCtaMaxThreads)
    ln_fwd_kernel(const LnParams p) {
  {  // the first two iterations' rows into L2 while the previous kernel ends
    const int rpc0 = G ? kSubwarpThreads / G : 1;
    const int64_t b0 = (int64_t)blockIdx.x * rpc0, st = (int64_t)gridDim.x * rpc0;
    const size_t rb0 = (size_t)p.N * sizeof(TX);
    l2_warm(p.x, nullptr, nullptr, b0, rpc0, p.M, rb0);
    if (PF) l2_warm(p.x, nullptr, nullptr, b0 + st, rpc0, p.M, rb0);
  }
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  __shared__ float red[128];
  const int L = G ? G : (int)blockDim.x;
  const int lane = G ? (int)threadIdx.x % G : (int)threadIdx.x;
  const int rpc = G ? kSubwarpThreads / G : 1;
  const int grp = G ? (int)threadIdx.x / G : 0;

  constexpr int GW = Cfg<TX, TW>::GW;
  uint4 gw[VPT][GW], bw[VPT][GW];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * L;
    load_weight<GW>(gw[k], p.gamma, v, v < p.nvec);
    load_weight<GW>(bw[k], p.beta, v, v < p.nvec && p.beta != nullptr);
  }
  const int64_t stride = (int64_t)gridDim.x * rpc;
  const size_t rb = (size_t)p.N * sizeof(TX);
  int parity = 0;
  int64_t base = (int64_t)blockIdx.x * rpc;
  uint4 cur[VPT], nxt[VPT];
  load_row<TX, VPT>(cur, p.x, base + grp, base + grp < p.M, lane, L, p.nvec, p.N);
  for (; base < p.M; base += stride) {
    const int64_t row = base + grp;
    const bool valid = row < p.M;
    const int64_t nrow = row + stride;
    if (PF) load_row<TX, VPT>(nxt, p.x, nrow, nrow < p.M, lane, L, p.nvec, p.N);
    l2_ahead(p.x, p, base, stride, rpc, rb);
    // pass 1: the mean; pass 2: the variance about it (both over registers)
    const RowStats st = row_stats<G, TX, E, VPT>(cur, red, parity, lane, L, p.nvec, p.inv_n, p.eps);
    const float rs = st.rs;
    if (valid && lane == 0) {
      if (p.mean != nullptr) p.mean[row] = st.m0 + st.c;
      if (p.rstd != nullptr) p.rstd[row] = rs;
    }
    char* yr = static_cast<char*>(p.y) + row * rb;
    const float2 nc = make_float2(-st.c, -st.c), r2 = make_float2(rs, rs);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * L;
      if (valid && v < p.nvec) {
        float f[E], g[E], b[E];
        uint4 gk[GW], bk[GW];
#pragma unroll
        for (int w = 0; w < GW; ++w) {
          gk[w] = opaque(gw[k][w]);
          bk[w] = opaque(bw[k][w]);
        }
        vec_minus<TX, E>(opaque(cur[k]), -st.m0, f);
        unpack_gamma<TW, E, GW>(gk, g);
        unpack_gamma<TW, E, GW>(bk, b);
#pragma unroll
        for (int i = 0; i < E / 2; ++i) {
          const float2 t =
              __fmul2_rn(__fadd2_rn(make_float2(f[2 * i], f[2 * i + 1]), nc), r2);
          const float2 o = __ffma2_rn(t, make_float2(g[2 * i], g[2 * i + 1]),
                                      make_float2(b[2 * i], b[2 * i + 1]));
          f[2 * i] = o.x;
          f[2 * i + 1] = o.y;
        }
        st_stream(yr + (size_t)v * 16, pack(f));
      }
    }
    if (PF) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) cur[k] = nxt[k];
    } else {
      load_row<TX, VPT>(cur, p.x, nrow, nrow < p.M, lane, L, p.nvec, p.N);
    }
  }
}

// ---------------------------------------------------------------------------
// Backward per-vector work.  With t = x - m0 (the first-pass mean, or the
// saved mean with c = 0), xhat = (t - c) rstd and g = dy gamma:
//   row sums    S1 = sum g,  S2 = sum g (t - c)          (sum g xhat = rstd S2)
//   dx          = rstd g - rstd mean(g) - rstd xhat mean(g xhat)
//               = (dy rstd) gamma - (B t + C),  B = rstd^2 mean(g xhat),
//                                               C = rstd mean(g) - B c
//   dgamma     += (dy rstd)(t - c),   dbeta += dy
// all in pairs with the paired fp32 instructions: about a dozen instructions
// per element, down from eighteen in the direct form.
struct LnBwdRow {
  float2 nm, nc, r2, nb, ncc;   // -m0, -c, rstd, -B, -C (each in both lanes)
};

// C: the correction c is applied (recomputed statistics); with the saved
// statistics c = 0 and the add is left out.
template <typename TX, typename TW, int E, int GW, bool C>
__device__ __forceinline__ void ln_bwd_dot(const uint4& xv, const uint4& dv,
                                           const uint4 (&gk)[GW], float nm, float2 nc,
                                           float2& s1, float2& s2) {
  float t[E], g[E];
  vec_minus<TX, E>(xv, nm, t);
  vec_dy_gamma<TX, TW, E, GW>(dv, gk, g);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    float2 tc = make_float2(t[2 * i], t[2 * i + 1]);
    if (C) tc = __fadd2_rn(tc, nc);
    const float2 gg = make_float2(g[2 * i], g[2 * i + 1]);
    s1 = __fadd2_rn(s1, gg);
    s2 = __ffma2_rn(gg, tc, s2);
  }
}

// The row constants once S1 and S2 are known.
__device__ __forceinline__ LnBwdRow ln_bwd_row(float m0, float c, float rs, float S1, float S2,
                                               float inv_n) {
  const float mg = S1 * inv_n, mgx = rs * S2 * inv_n;
  const float B = rs * rs * mgx, C = fmaf(-B, c, rs * mg);
  LnBwdRow r;
  r.nm = make_float2(-m0, -m0);
  r.nc = make_float2(-c, -c);
  r.r2 = make_float2(rs, rs);
  r.nb = make_float2(-B, -B);
  r.ncc = make_float2(-C, -C);
  return r;
}

template <typename TX, typename TW, int E, int GW, bool C>
__device__ __forceinline__ uint4 ln_bwd_apply(const uint4& xv, const uint4& dv,
                                              const uint4 (&gk)[GW], const LnBwdRow& r,
                                              float2 (&ag)[E / 2], float2 (&ab)[E / 2]) {
  float f[E], d[E], g[E], o[E];
  vec_minus<TX, E>(xv, r.nm.x, f);
  unpack(dv, d);
  unpack_gamma<TW, E, GW>(gk, g);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    const float2 d2 = make_float2(d[2 * i], d[2 * i + 1]);
    const float2 t = make_float2(f[2 * i], f[2 * i + 1]);
    const float2 drs = __fmul2_rn(d2, r.r2);
    const float2 nu = __ffma2_rn(t, r.nb, r.ncc);                    // -(B t + C)
    const float2 dx = __ffma2_rn(drs, make_float2(g[2 * i], g[2 * i + 1]), nu);
    ag[i] = __ffma2_rn(drs, C ? __fadd2_rn(t, r.nc) : t, ag[i]);
    ab[i] = __fadd2_rn(ab[i], d2);
    o[2 * i] = dx.x;
    o[2 * i + 1] = dx.y;
  }
  return pack(o);
}

// One thread's columns of the partial row [dgamma | dbeta] (16-byte stores).
template <int E, int VPT>
__device__ __forceinline__ void write_partials(float* prow, int ld_half,
                                               const float2 (&ag)[VPT][E / 2],
                                               const float2 (&ab)[VPT][E / 2], int lane, int L,
                                               int nvec) {
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * L;
    if (v < nvec) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        reinterpret_cast<float4*>(prow + v * E)[q] =
            make_float4(ag[k][2 * q].x, ag[k][2 * q].y, ag[k][2 * q + 1].x, ag[k][2 * q + 1].y);
        reinterpret_cast<float4*>(prow + ld_half + v * E)[q] =
            make_float4(ab[k][2 * q].x, ab[k][2 * q].y, ab[k][2 * q + 1].x, ab[k][2 * q + 1].y);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Backward: same shapes.  dgamma / dbeta partials of this CTA's rows are kept
// in registers per thread; sub-warp groups are combined through shared memory
// in group order at the end, and one partial row [dgamma | dbeta] is written.
template <typename TX, typename TW, int G, int VPT, bool PF>
__global__ void __launch_bounds__(G ? kSubwarpThreads : kCtaMaxThreads)
    ln_bwd_kernel(const LnParams p) {
  {  // the first two iterations' rows into L2 while the previous kernel ends
    const int rpc0 = G ? kSubwarpThreads / G : 1;
    const int64_t b0 = (int64_t)blockIdx.x * rpc0, st = (int64_t)gridDim.x * rpc0;
    const size_t rb0 = (size_t)p.N * sizeof(TX);
    l2_warm(p.x, p.dy, nullptr, b0, rpc0, p.M, rb0);
    if (PF) l2_warm(p.x, p.dy, nullptr, b0 + st, rpc0, p.M, rb0);
  }
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  __shared__ float red[128];
  extern __shared__ float4 smem4[];                // sub-warp: [rpc][2 * nvec * E]
  float* sacc = reinterpret_cast<float*>(smem4);
  const int L = G ? G : (int)blockDim.x;
  const int lane = G ? (int)threadIdx.x % G : (int)threadIdx.x;
  const int rpc = G ? kSubwarpThreads / G : 1;
  const int grp = G ? (int)threadIdx.x / G : 0;
  const bool saved = p.mean != nullptr;

  constexpr int GW = Cfg<TX, TW>::GW;
  uint4 gw[VPT][GW];
  float2 ag[VPT][E / 2], ab[VPT][E / 2];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * L;
    load_weight<GW>(gw[k], p.gamma, v, v < p.nvec);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) ag[k][e] = ab[k][e] = make_float2(0.f, 0.f);
  }
  const int64_t stride = (int64_t)gridDim.x * rpc;
  const size_t rb = (size_t)p.N * sizeof(TX);
  int parity = 0;
  int64_t base = (int64_t)blockIdx.x * rpc;
  uint4 cx[VPT], cd[VPT], nx[VPT], nd[VPT];
  load_row<TX, VPT>(cx, p.x, base + grp, base + grp < p.M, lane, L, p.nvec, p.N);
  load_row<TX, VPT>(cd, p.dy, base + grp, base + grp < p.M, lane, L, p.nvec, p.N);
  // the saved statistics are loaded one row ahead, with the rows
  float sm = 0.f, sr = 0.f;
  if (saved && base + grp < p.M) {
    sm = p.mean[base + grp];
    sr = p.rstd[base + grp];
  }
  for (; base < p.M; base += stride) {
    const int64_t row = base + grp;
    const bool valid = row < p.M;
    const int64_t nrow = row + stride;
    float nsm = 0.f, nsr = 0.f;
    if (saved && nrow < p.M) {
      nsm = p.mean[nrow];
      nsr = p.rstd[nrow];
    }
    if (PF) {
      load_row<TX, VPT>(nx, p.x, nrow, nrow < p.M, lane, L, p.nvec, p.N);
      load_row<TX, VPT>(nd, p.dy, nrow, nrow < p.M, lane, L, p.nvec, p.N);
    }
    l2_ahead(p.x, p, base, stride, rpc, rb);
    l2_ahead(p.dy, p, base, stride, rpc, rb);
    // xhat = ((x - m0) - c) * rs: the saved statistics (c = 0), or recomputed
    RowStats st;
    if (saved) {
      st.m0 = sm;
      st.c = 0.f;
      st.rs = sr;
    } else {
      st = row_stats<G, TX, E, VPT>(cx, red, parity, lane, L, p.nvec, p.inv_n, p.eps);
    }
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
    const float2 nc = make_float2(-st.c, -st.c);
    auto dot = [&](auto corr) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {   // padding lanes hold zeros: g = 0
        uint4 gk[GW];
#pragma unroll
        for (int w = 0; w < GW; ++w) gk[w] = opaque(gw[k][w]);
        ln_bwd_dot<TX, TW, E, GW, decltype(corr)::value>(cx[k], cd[k], gk, -st.m0, nc, s1, s2);
      }
    };
    if (saved) dot(std::false_type{});
    else dot(std::true_type{});
    float a = s1.x + s1.y, b = s2.x + s2.y;
    row_sum2<G>(a, b, red, parity);
    const LnBwdRow rc = ln_bwd_row(st.m0, st.c, st.rs, a, b, p.inv_n);
    char* dxr = static_cast<char*>(p.y) + row * rb;
    auto apply = [&](auto corr) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lane + k * L;
        if (valid && v < p.nvec) {
          uint4 gk[GW];
#pragma unroll
          for (int w = 0; w < GW; ++w) gk[w] = opaque(gw[k][w]);
          st_stream(dxr + (size_t)v * 16,
                    ln_bwd_apply<TX, TW, E, GW, decltype(corr)::value>(
                        opaque(cx[k]), opaque(cd[k]), gk, rc, ag[k], ab[k]));
        }
      }
    };
    if (saved) apply(std::false_type{});
    else apply(std::true_type{});
    sm = nsm;
    sr = nsr;
    if (PF) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        cx[k] = nx[k];
        cd[k] = nd[k];
      }
    } else {
      load_row<TX, VPT>(cx, p.x, nrow, nrow < p.M, lane, L, p.nvec, p.N);
      load_row<TX, VPT>(cd, p.dy, nrow, nrow < p.M, lane, L, p.nvec, p.N);
    }
  }
  if (p.partial == nullptr) return;
  float* prow = p.partial + (size_t)blockIdx.x * 2 * p.ld_half;
  if constexpr (G != 0) {
    const int ncol = p.nvec * E;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * L;
      if (v < p.nvec) {
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          float* dg = sacc + (size_t)grp * 2 * ncol + v * E + 2 * e;
          dg[0] = ag[k][e].x;
          dg[1] = ag[k][e].y;
          dg[ncol] = ab[k][e].x;
          dg[ncol + 1] = ab[k][e].y;
        }
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < ncol; j += kSubwarpThreads) {
      float sg = 0.f, sb = 0.f;
      for (int q = 0; q < rpc; ++q) {
        sg += sacc[(size_t)q * 2 * ncol + j];
        sb += sacc[(size_t)q * 2 * ncol + ncol + j];
      }
      prow[j] = sg;
      prow[p.ld_half + j] = sb;
    }
  } else {
    write_partials<E, VPT>(prow, p.ld_half, ag, ab, lane, L, p.nvec);
  }
}

// ---------------------------------------------------------------------------
// Staged backward: one row per CTA iteration; the rows [x | dy] arrive by bulk
// copies into the shared-memory ring of rmsnorm_ring.cuh and are read from
// the stage twice (row sums, then dx) instead of being held in registers, so
// the registers hold only gamma and the two partial rows.  A stage is refilled
// one row late, at the next row's reduction barrier, which proves every thread
// has finished reading it -- no extra barrier per row.  Every wait is bounded;
// a wait that runs out is voted on at the row-sum barrier, the CTA stores
// nothing more and leaves, and thread 0 drains its copies and raises
// kStatusWaitTimeout.
template <typename TX, typename TW, int VPT>
__global__ void __launch_bounds__(kCtaMaxThreads) ln_bwd_staged_kernel(const LnParams p) {
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int GW = Cfg<TX, TW>::GW;
  extern __shared__ __align__(128) unsigned char smem[];
  const Ring rg = ring_of(smem);
  const int tid = threadIdx.x, T = blockDim.x, S = p.stages;
  const size_t rb = (size_t)p.N * sizeof(TX);
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nrows = first < p.M ? (p.M - 1 - first) / stride + 1 : 0;
  const char* xs = static_cast<const char*>(p.x);
  const char* ds = static_cast<const char*>(p.dy);
  int64_t issued = ring_start<2>(rg, S, nrows, first, stride, xs, ds, nullptr, rb);
  const bool saved = p.mean != nullptr;

  uint4 gw[VPT][GW];
  float2 ag[VPT][E / 2], ab[VPT][E / 2];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    load_weight<GW>(gw[k], p.gamma, v, v < p.nvec);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) ag[k][e] = ab[k][e] = make_float2(0.f, 0.f);
  }
  int parity = 0;
  int64_t i = 0;
  bool failed = false;
  // the saved statistics are loaded one row ahead
  float sm = 0.f, sr = 0.f;
  if (saved && nrows > 0) {
    sm = p.mean[first];
    sr = p.rstd[first];
  }
  for (; i < nrows; ++i) {
    const int st_i = (int)(i % S);
    const int64_t row = first + i * stride;
    float nsm = 0.f, nsr = 0.f;
    if (saved && i + 1 < nrows) {
      nsm = p.mean[row + stride];
      nsr = p.rstd[row + stride];
    }
    const bool late =
        !mbar_wait_bounded(rg.full + st_i, (uint32_t)((i / S) & 1), p.wait_limit);
    const uint4* stg = reinterpret_cast<const uint4*>(rg.buf + (size_t)st_i * 2 * rb);
    uint4 cx[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      cx[k] = (!late && v < p.nvec) ? stg[v] : make_uint4(0, 0, 0, 0);
    }
    RowStats st;
    if (saved) {
      st.m0 = sm;
      st.c = 0.f;
      st.rs = sr;
    } else {
      st = row_stats<0, TX, E, VPT>(cx, rg.red, parity, tid, T, p.nvec, p.inv_n, p.eps);
    }
    sm = nsm;
    sr = nsr;
    const float2 nc = make_float2(-st.c, -st.c);
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
    auto dot = [&](auto corr) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * T;
        if (late || v >= p.nvec) continue;
        uint4 gk[GW];
#pragma unroll
        for (int w = 0; w < GW; ++w) gk[w] = opaque(gw[k][w]);
        ln_bwd_dot<TX, TW, E, GW, decltype(corr)::value>(cx[k], stg[p.nvec + v], gk, -st.m0,
                                                          nc, s1, s2);
      }
    };
    if (saved) dot(std::false_type{});
    else dot(std::true_type{});
    float t[2] = {s1.x + s1.y, s2.x + s2.y};
    if (cta_sum_vote<2>(t, rg.red, parity, late)) {
      failed = true;
      break;
    }
    parity ^= 1;
    // every thread is past row i - 1's epilogue: its stage takes row i - 1 + S
    if (tid == 0 && i >= 1 && issued < nrows) {
      fence_proxy_async_smem();
      issue_row<2>(rg, issued, first, stride, S, xs, ds, nullptr, rb);
      ++issued;
    }
    const LnBwdRow rc = ln_bwd_row(st.m0, st.c, st.rs, t[0], t[1], p.inv_n);
    char* dxr = static_cast<char*>(p.y) + row * rb;
    auto apply = [&](auto corr) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * T;
        if (v < p.nvec) {
          uint4 gk[GW];
#pragma unroll
          for (int w = 0; w < GW; ++w) gk[w] = opaque(gw[k][w]);
          st_stream(dxr + (size_t)v * 16,
                    ln_bwd_apply<TX, TW, E, GW, decltype(corr)::value>(
                        stg[v], stg[p.nvec + v], gk, rc, ag[k], ab[k]));
        }
      }
    };
    if (saved) apply(std::false_type{});
    else apply(std::true_type{});
  }
  if (failed) {
    if (tid == 0) {
      drain(rg, i, issued, S);
      atomicOr(p.status, kStatusWaitTimeout);
    }
    return;
  }
  if (p.partial == nullptr) return;
  write_partials<E, VPT>(p.partial + (size_t)blockIdx.x * 2 * p.ld_half, p.ld_half, ag, ab, tid,
                         T, p.nvec);
}

// ---------------------------------------------------------------------------
// Short rows through the bulk-copy ring (staged with G lanes per row): a CTA
// iteration covers RPC = 256 / G consecutive rows, contiguous in memory, so
// one bulk copy per operand fills a ring stage ([x rows | dy rows]).  The row
// math is the sub-warp backward's (shuffle reductions within the G lanes);
// the vectors are read from the stage for the statistics, the row sums and
// dx rather than held in registers, which hold gamma (packed) and the two
// partial rows.  One CTA barrier per iteration votes on the bounded waits and
// proves that every thread has finished the previous iteration's stage,
// which thread 0 then refills.  The saved statistics are loaded one
// iteration ahead.  Held to two resident CTAs per SM (128 registers; the
// four-vector form would take 154 and one).
template <typename TX, typename TW, int G, int VPT>
__global__ void __launch_bounds__(kSubwarpThreads, 2) ln_bwd_rows_staged_kernel(const LnParams p) {
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int GW = Cfg<TX, TW>::GW;
  constexpr int RPC = kSubwarpThreads / G;
  const size_t rb = (size_t)p.N * sizeof(TX);
  {  // the rows of the first two iterations into L2 while the previous kernel ends
    const int64_t b0 = (int64_t)blockIdx.x * RPC, st0 = (int64_t)gridDim.x * RPC;
    l2_warm(p.x, p.dy, nullptr, b0, RPC, p.M, rb);
    l2_warm(p.x, p.dy, nullptr, b0 + st0, RPC, p.M, rb);
  }
  pdl_begin();
  extern __shared__ __align__(128) unsigned char smem[];
  const Ring rg = ring_of(smem);
  const int lane = threadIdx.x % G, grp = threadIdx.x / G, tid = threadIdx.x;
  const int S = p.stages;
  const size_t blk = (size_t)RPC * rb;              // one operand's rows of a stage
  const int64_t units = (p.M + RPC - 1) / RPC;      // CTA iterations of RPC rows
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nit = first < units ? (units - 1 - first) / stride + 1 : 0;
  const char* src[2] = {static_cast<const char*>(p.x), static_cast<const char*>(p.dy)};
  const bool saved = p.mean != nullptr;

  // thread 0: the rows of iteration j into stage j mod S (the last unit may
  // hold fewer than RPC rows)
  auto issue = [&](int64_t j) {
    const int s = (int)(j % S);
    const int64_t row0 = (first + j * stride) * RPC;
    const int64_t n = p.M - row0 < RPC ? p.M - row0 : RPC;
    const uint32_t bytes = (uint32_t)(n * (int64_t)rb);
    uint64_t* bar = rg.full + s;
    unsigned char* dst = rg.buf + (size_t)s * 2 * blk;
    mbar_arrive_expect_tx(bar, 2 * bytes);
#pragma unroll
    for (int q = 0; q < 2; ++q) bulk_copy_g2s(dst + q * blk, src[q] + row0 * rb, bytes, bar);
  };
  int64_t issued = 0;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(rg.full + s, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0)
    for (; issued < (nit < S ? nit : S); ++issued) issue(issued);

  uint4 gw[VPT][GW];
  float2 ag[VPT][E / 2], ab[VPT][E / 2];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * G;
    load_weight<GW>(gw[k], p.gamma, v, v < p.nvec);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) ag[k][e] = ab[k][e] = make_float2(0.f, 0.f);
  }
  // this thread's row statistics, one iteration ahead
  float sm = 0.f, sr = 0.f;
  if (saved && nit > 0) {
    const int64_t row = first * RPC + grp;
    if (row < p.M) {
      sm = p.mean[row];
      sr = p.rstd[row];
    }
  }
  int parity = 0;   // unused by the sub-warp reductions
  int64_t j = 0;
  bool failed = false;
  for (; j < nit; ++j) {
    const int s = (int)(j % S);
    const int64_t row = (first + j * stride) * RPC + grp;
    const bool valid = row < p.M;
    float nsm = 0.f, nsr = 0.f;
    if (saved && j + 1 < nit) {
      const int64_t nrow = (first + (j + 1) * stride) * RPC + grp;
      if (nrow < p.M) {
        nsm = p.mean[nrow];
        nsr = p.rstd[nrow];
      }
    }
    const bool late = !mbar_wait_bounded(rg.full + s, (uint32_t)((j / S) & 1), p.wait_limit);
    if (__syncthreads_or(late ? 1 : 0)) {
      failed = true;
      break;
    }
    // every thread is done with the previous iteration's stage: refill it
    if (tid == 0 && j > 0 && issued < nit) {
      fence_proxy_async_smem();
      issue(issued);
      ++issued;
    }
    const unsigned char* st = rg.buf + (size_t)s * 2 * blk + (size_t)grp * rb;
    const uint4* xs = reinterpret_cast<const uint4*>(st);
    const uint4* ds = reinterpret_cast<const uint4*>(st + blk);
    RowStats rst;
    if (saved) {
      rst.m0 = sm;
      rst.c = 0.f;
      rst.rs = sr;
    } else {
      uint4 cx[VPT];
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lane + k * G;
        cx[k] = (valid && v < p.nvec) ? xs[v] : make_uint4(0, 0, 0, 0);
      }
      rst = row_stats<G, TX, E, VPT>(cx, nullptr, parity, lane, G, p.nvec, p.inv_n, p.eps);
    }
    sm = nsm;
    sr = nsr;
    const float2 nc = make_float2(-rst.c, -rst.c);
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
    auto dot = [&](auto corr) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lane + k * G;
        if (!valid || v >= p.nvec) continue;
        uint4 gk[GW];
#pragma unroll
        for (int w = 0; w < GW; ++w) gk[w] = opaque(gw[k][w]);
        ln_bwd_dot<TX, TW, E, GW, decltype(corr)::value>(ld_shared_v4(xs + v), ld_shared_v4(ds + v),
                                                          gk, -rst.m0, nc, s1, s2);
      }
    };
    if (saved) dot(std::false_type{});
    else dot(std::true_type{});
    float a = s1.x + s1.y, b = s2.x + s2.y;
    row_sum2<G>(a, b, nullptr, parity);
    const LnBwdRow rc = ln_bwd_row(rst.m0, rst.c, rst.rs, a, b, p.inv_n);
    char* dxr = static_cast<char*>(p.y) + row * rb;
    auto apply = [&](auto corr) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = lane + k * G;
        if (valid && v < p.nvec) {
          uint4 gk[GW];
#pragma unroll
          for (int w = 0; w < GW; ++w) gk[w] = opaque(gw[k][w]);
          st_stream(dxr + (size_t)v * 16,
                    ln_bwd_apply<TX, TW, E, GW, decltype(corr)::value>(
                        ld_shared_v4(xs + v), ld_shared_v4(ds + v), gk, rc, ag[k], ab[k]));
        }
      }
    };
    if (saved) apply(std::false_type{});
    else apply(std::true_type{});
  }
  if (failed) {
    if (tid == 0) {
      drain(rg, j, issued, S);
      atomicOr(p.status, kStatusWaitTimeout);
    }
    return;
  }
  if (p.partial == nullptr) return;
  // the row groups' partial rows meet in shared memory (the ring is free:
  // every copy has been consumed), added in group order
  __syncthreads();
  float* sacc = reinterpret_cast<float*>(rg.buf);
  const int ncol = p.nvec * E;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * G;
    if (v < p.nvec) {
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        float* dg = sacc + (size_t)grp * 2 * ncol + v * E + 2 * e;
        dg[0] = ag[k][e].x;
        dg[1] = ag[k][e].y;
        dg[ncol] = ab[k][e].x;
        dg[ncol + 1] = ab[k][e].y;
      }
    }
  }
  __syncthreads();
  float* prow = p.partial + (size_t)blockIdx.x * 2 * p.ld_half;
  for (int c = tid; c < ncol; c += kSubwarpThreads) {
    float sg = 0.f, sb = 0.f;
    for (int q = 0; q < RPC; ++q) {
      sg += sacc[(size_t)q * 2 * ncol + c];
      sb += sacc[(size_t)q * 2 * ncol + ncol + c];
    }
    prow[c] = sg;
    prow[p.ld_half + c] = sb;
  }
}

// ---------------------------------------------------------------------------
// Any row (scalar, one row per CTA iteration, 256 threads): three passes over
// the row in global memory (mean, variance, output); the backward's partial
// row is accumulated in place in the workspace, each column by the one thread
// that owns it.
// The corrected two-pass statistics of a row in global memory (CTA-wide).
template <typename TX>
__device__ __forceinline__ RowStats generic_stats(const TX* xr, int N, float* red, int& parity,
                                                  float inv_n, float eps) {
  constexpr int U = kGenericBatch;
  const int tid = threadIdx.x, T = blockDim.x;
  RowStats st;
  float s = 0.f;
  for (int j0 = tid; j0 < N; j0 += U * T) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = j0 + u * T < N ? ld_scalar(xr + j0 + u * T) : 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) s += v[u];
  }
  st.m0 = row_sum<0>(s, red, parity) * inv_n;
  float sd = 0.f, sq = 0.f;
  for (int j0 = tid; j0 < N; j0 += U * T) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = j0 + u * T < N ? ld_scalar(xr + j0 + u * T) : st.m0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float d = v[u] - st.m0;   // 0 past the row
      sd += d;
      sq = fmaf(d, d, sq);
    }
  }
  row_sum2<0>(sd, sq, red, parity);
  st.c = sd * inv_n;
  st.rs = rsqrtf(fmaxf(fmaf(sq, inv_n, -st.c * st.c), 0.f) + eps);
  return st;
}

template <typename TX, typename TW>
__global__ void __launch_bounds__(256) ln_fwd_generic_kernel(const LnParams p) {
  pdl_begin();
  constexpr int U = kGenericBatch;
  __shared__ float red[128];
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const TW* gam = static_cast<const TW*>(p.gamma);
  const TW* bet = static_cast<const TW*>(p.beta);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const TX* xr = static_cast<const TX*>(p.x) + row * (int64_t)N;
    const RowStats st = generic_stats(xr, N, red, parity, p.inv_n, p.eps);
    if (tid == 0) {
      if (p.mean != nullptr) p.mean[row] = st.m0 + st.c;
      if (p.rstd != nullptr) p.rstd[row] = st.rs;
    }
    TX* yr = static_cast<TX*>(p.y) + row * (int64_t)N;
    for (int j0 = tid; j0 < N; j0 += U * T) {
      float xv[U], gv[U], bv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        const bool in = j < N;
        xv[u] = in ? ld_scalar(xr + j) : 0.f;
        gv[u] = in ? ld_scalar_ro(gam + j) : 0.f;
        bv[u] = (in && bet) ? ld_scalar_ro(bet + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        if (j >= N) continue;
        const float t = ((xv[u] - st.m0) - st.c) * st.rs;
        st_scalar(yr + j, fmaf(t, gv[u], bv[u]));
      }
    }
  }
}

template <typename TX, typename TW>
__global__ void __launch_bounds__(256) ln_bwd_generic_kernel(const LnParams p) {
  pdl_begin();
  constexpr int U = kGenericBatch;
  __shared__ float red[128];
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const TW* gam = static_cast<const TW*>(p.gamma);
  float* prow = p.partial ? p.partial + (size_t)blockIdx.x * 2 * p.ld_half : nullptr;
  if (prow)
    for (int j = tid; j < N; j += T) prow[j] = prow[p.ld_half + j] = 0.f;
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const TX* xr = static_cast<const TX*>(p.x) + row * (int64_t)N;
    const TX* dr = static_cast<const TX*>(p.dy) + row * (int64_t)N;
    RowStats st;
    if (p.mean != nullptr) {
      st.m0 = p.mean[row];
      st.c = 0.f;
      st.rs = p.rstd[row];
    } else {
      st = generic_stats(xr, N, red, parity, p.inv_n, p.eps);
    }
    const float rs = st.rs;
    float a = 0.f, b = 0.f;
    for (int j0 = tid; j0 < N; j0 += U * T) {
      float xv[U], dv[U], gv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        const bool in = j < N;
        xv[u] = in ? ld_scalar(xr + j) : 0.f;
        dv[u] = in ? ld_scalar(dr + j) : 0.f;
        gv[u] = in ? ld_scalar_ro(gam + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float xh = ((xv[u] - st.m0) - st.c) * rs;
        const float g = dv[u] * gv[u];   // 0 past the row
        a += g;
        b = fmaf(g, xh, b);
      }
    }
    row_sum2<0>(a, b, red, parity);
    const float mg = a * p.inv_n, mgx = b * p.inv_n;
    TX* dxr = static_cast<TX*>(p.y) + row * (int64_t)N;
    for (int j0 = tid; j0 < N; j0 += U * T) {
      float xv[U], dv[U], gv[U], pg[U], pb[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        const bool in = j < N;
        xv[u] = in ? ld_scalar(xr + j) : 0.f;
        dv[u] = in ? ld_scalar(dr + j) : 0.f;
        gv[u] = in ? ld_scalar_ro(gam + j) : 0.f;
        pg[u] = (prow && in) ? prow[j] : 0.f;
        pb[u] = (prow && in) ? prow[p.ld_half + j] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        if (j >= N) continue;
        const float xh = ((xv[u] - st.m0) - st.c) * rs;
        st_scalar(dxr + j, rs * (dv[u] * gv[u] - fmaf(xh, mgx, mg)));
        if (prow) {
          prow[j] = fmaf(dv[u], xh, pg[u]);
          prow[p.ld_half + j] = pb[u] + dv[u];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Instantiation table (one dtype pair per translation unit).

template <typename TX, typename TW, bool BWD, bool PF>
LnKernel pick_shape(const LnKey& k) {
  if (k.family == kCta) {
    switch (k.vpt) {
      case 1: return BWD ? ln_bwd_kernel<TX, TW, 0, 1, PF> : ln_fwd_kernel<TX, TW, 0, 1, PF>;
      case 2: return BWD ? ln_bwd_kernel<TX, TW, 0, 2, PF> : ln_fwd_kernel<TX, TW, 0, 2, PF>;
      // the backward keeps gamma and both partials in fp32 registers: at most
      // 2 vectors per thread
      case 4: return BWD ? nullptr : ln_fwd_kernel<TX, TW, 0, 4, PF>;
      case 8: return (BWD || PF) ? nullptr : ln_fwd_kernel<TX, TW, 0, 8, false>;
      default: return nullptr;
    }
  }
  if (k.family == kSubwarp) {
#define RMSN_LN(G_, V_)                                                                     \
  if (k.g == G_ && k.vpt == V_)                                                              \
    return BWD ? ln_bwd_kernel<TX, TW, G_, V_, PF> : ln_fwd_kernel<TX, TW, G_, V_, PF>;
    RMSN_LN(4, 1) RMSN_LN(8, 1) RMSN_LN(16, 1) RMSN_LN(32, 1)
    RMSN_LN(8, 2) RMSN_LN(16, 2) RMSN_LN(32, 2) RMSN_LN(32, 3) RMSN_LN(32, 4)
#undef RMSN_LN
  }
  return nullptr;
}

template <typename TX, typename TW>
LnKernel pick_ln(const LnKey& k) {
  if (k.family == kGeneric)
    return k.bwd ? ln_bwd_generic_kernel<TX, TW> : ln_fwd_generic_kernel<TX, TW>;
  if (k.family == kStaged && k.g > 0) {   // short rows through the ring
    if (!k.bwd) return nullptr;
#define RMSN_LNRS(G_, V_) \
  if (k.g == G_ && k.vpt == V_) return ln_bwd_rows_staged_kernel<TX, TW, G_, V_>;
    RMSN_LNRS(8, 1) RMSN_LNRS(16, 1) RMSN_LNRS(32, 1) RMSN_LNRS(16, 2) RMSN_LNRS(32, 2)
    RMSN_LNRS(32, 3) RMSN_LNRS(32, 4)
#undef RMSN_LNRS
    return nullptr;
  }
  if (k.family == kStaged) {
    if (!k.bwd) return nullptr;
    switch (k.vpt) {
      case 1: return ln_bwd_staged_kernel<TX, TW, 1>;
      case 2: return ln_bwd_staged_kernel<TX, TW, 2>;
      case 4: return ln_bwd_staged_kernel<TX, TW, 4>;
      default: return nullptr;
    }
  }
  if (k.bwd)
    return k.prefetch ? pick_shape<TX, TW, true, true>(k) : pick_shape<TX, TW, true, false>(k);
  return k.prefetch ? pick_shape<TX, TW, false, true>(k) : pick_shape<TX, TW, false, false>(k);
}


}  // namespace

#if RMSN_PAIR == 0
LnKernel get_ln_kernel_f32_f32(const LnKey& k) { return pick_ln<float, float>(k); }
#elif RMSN_PAIR == 1
LnKernel get_ln_kernel_bf16_bf16(const LnKey& k) { return pick_ln<bf16, bf16>(k); }
#else
LnKernel get_ln_kernel_bf16_f32(const LnKey& k) { return pick_ln<bf16, float>(k); }
#endif

}  // namespace rmsn
