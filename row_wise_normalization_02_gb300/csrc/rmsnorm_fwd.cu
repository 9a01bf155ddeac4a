// RMSNorm forward and fused residual-add forward kernels for sm_103a.
//
// y_ij = x_ij * rstd_i * gamma_j,  rstd_i = 1 / sqrt(mean_j x_ij^2 + eps)
// ("Pre-built kernel library guide", section 1.2 RMSNorm).  The fused variant
// first forms h = residual + x, rounds it to the activation dtype, writes it
// over the residual and normalises that stored h ("TIRx kernels", Kernels list:
// fused_add_rmsnorm among the flashinfer.norm ports).
//
// The operation moves 2 (or 4, fused) bytes of HBM traffic per activation
// byte and does ~4 flops per element, so every kernel here is an HBM-streaming
// kernel: each element is read once with 16-byte loads, the row stays in
// registers across the reduction (the register-resident fast path of the same
// guide's section 1.1, rather than its shared-memory row cache), and results
// leave through 16-byte evict-first stores.  Persistent grids walk rows with a
// fixed stride and issue the next row's loads before reducing the current one.
#include "rmsnorm_fwd_common.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif

namespace rmsn {
namespace {

// ---------------------------------------------------------------------------
// kSubwarp: G lanes per row, 256 / G rows per CTA iteration, persistent grid.
template <typename TX, typename TW, int G, int VPT, bool FUSED, bool PF>
__global__ void __launch_bounds__(kSubwarpThreads)
    fwd_subwarp_kernel(const FwdParams p) {
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW;
  constexpr int RPC = kSubwarpThreads / G;
  {  // the first two iterations' rows into L2 while the previous kernel ends
    const size_t rb = (size_t)p.N * sizeof(TX);
    const void* r = FUSED ? p.residual : nullptr;
    const int64_t b0 = (int64_t)blockIdx.x * RPC, st = (int64_t)gridDim.x * RPC;
    l2_warm(p.x, r, nullptr, b0, RPC, p.M, rb);
    if (PF) l2_warm(p.x, r, nullptr, b0 + st, RPC, p.M, rb);
  }
  pdl_begin();
  const int lane = threadIdx.x % G, grp = threadIdx.x / G;

  uint4 gw[VPT][GW];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * G;
#pragma unroll
    for (int w = 0; w < GW; ++w)
      gw[k][w] = v < p.nvec ? ld_cached(static_cast<const char*>(p.gamma) +
                                        ((size_t)v * GW + w) * 16)
                            : make_uint4(0, 0, 0, 0);
  }

  const int64_t stride = (int64_t)gridDim.x * RPC;
  int64_t base = (int64_t)blockIdx.x * RPC;
  Slice<VPT, FUSED> cur, nxt;
  load_aligned<TX, VPT, FUSED>(cur, p, base + grp, base + grp < p.M, lane, G);
  for (; base < p.M; base += stride) {
    const int64_t row = base + grp;
    const bool valid = row < p.M;
    const int64_t nrow = row + stride;
    if (PF) load_aligned<TX, VPT, FUSED>(nxt, p, nrow, nrow < p.M, lane, G);

    const size_t rb = (size_t)p.N * sizeof(TX);
    float ss = slice_sumsq<TX, VPT, FUSED>(cur, static_cast<char*>(p.residual) + row * rb, lane,
                                           G, p.nvec, valid);
    ss = group_sum<G>(ss);
    const float rs = rsqrtf(fmaf(ss, p.inv_n, p.eps));
    if (valid && lane == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    char* yr = static_cast<char*>(p.y) + row * rb;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * G;
      if (valid && v < p.nvec) st_stream(yr + (size_t)v * 16, scale_vec<TX, TW>(cur.x[k], gw[k], rs));
    }
    if (PF) cur = nxt;
    else load_aligned<TX, VPT, FUSED>(cur, p, nrow, nrow < p.M, lane, G);
  }
}

// ---------------------------------------------------------------------------
// kCta: one row per CTA iteration, blockDim.x threads, persistent; gamma
// vectors in registers for the whole kernel.
template <typename TX, typename TW, int VPT, bool FUSED, bool PF>
__global__ void __launch_bounds__(kCtaMaxThreads) fwd_cta_kernel(const FwdParams p) {
  {  // the first two rows into L2 while the previous kernel ends
    const size_t rb = (size_t)p.N * sizeof(TX);
    const void* r = FUSED ? p.residual : nullptr;
    l2_warm(p.x, r, nullptr, blockIdx.x, 1, p.M, rb);
    if (PF) l2_warm(p.x, r, nullptr, (int64_t)blockIdx.x + gridDim.x, 1, p.M, rb);
  }
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW;
  extern __shared__ float4 smem4[];
  float* red = reinterpret_cast<float*>(smem4);    // 2 x 32 warp partials
  const int tid = threadIdx.x, T = blockDim.x;

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
  Slice<VPT, FUSED> cur, nxt;
  int64_t row = blockIdx.x;
  const size_t rb = (size_t)p.N * sizeof(TX);
  if (row < p.M) load_aligned<TX, VPT, FUSED>(cur, p, row, true, tid, T);
  for (; row < p.M; row += gridDim.x) {
    const int64_t nrow = row + gridDim.x;
    if (PF && nrow < p.M) load_aligned<TX, VPT, FUSED>(nxt, p, nrow, true, tid, T);
    char* yrow = static_cast<char*>(p.y) + row * rb;
    char* hrow = static_cast<char*>(p.residual) + row * rb;
    float ss[1];
    ss[0] = slice_sumsq<TX, VPT, FUSED>(cur, hrow, tid, T, p.nvec, true);
    cta_sum<1>(ss, red, parity);
    parity ^= 1;
    const float rs = rsqrtf(fmaf(ss[0], p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < p.nvec) st_stream(yrow + (size_t)v * 16, scale_vec<TX, TW>(cur.x[k], gw[k], rs));
    }
    if (PF) cur = nxt;
    else if (nrow < p.M) load_aligned<TX, VPT, FUSED>(cur, p, nrow, true, tid, T);
  }
}

// ---------------------------------------------------------------------------
// Strided rows (per-head q/k norm, "TIRx kernels", Kernels list: qk_rmsnorm):
// row i = (t, h) of a [T, H, D] view.  Same per-row work as kSubwarp; each
// thread steps its (t, h) by the grid stride without dividing.
template <typename TX, typename TW, int G, int VPT, bool PF>
__global__ void __launch_bounds__(kSubwarpThreads) fwd_strided_kernel(const FwdParams p) {
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW;
  constexpr int RPC = kSubwarpThreads / G;
  const int lane = threadIdx.x % G, grp = threadIdx.x / G;
  const int64_t H = p.heads;

  uint4 gw[VPT][GW];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * G;
#pragma unroll
    for (int w = 0; w < GW; ++w)
      gw[k][w] = v < p.nvec ? ld_cached(static_cast<const char*>(p.gamma) +
                                        ((size_t)v * GW + w) * 16)
                            : make_uint4(0, 0, 0, 0);
  }
  const int64_t stride = (int64_t)gridDim.x * RPC;
  const int64_t dt = stride / H, dh = stride % H;
  int64_t base = (int64_t)blockIdx.x * RPC;
  int64_t t = (base + grp) / H, h = (base + grp) % H;
  const TX* x = static_cast<const TX*>(p.x);
  TX* y = static_cast<TX*>(p.y);

  auto load = [&](uint4 (&dst)[VPT], int64_t tt, int64_t hh, bool valid) {
    const TX* xr = x + tt * p.x_st + hh * p.x_sh;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * G;
      dst[k] = (valid && v < p.nvec) ? ld_stream(xr + v * E) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 cur[VPT], nxt[VPT];
  load(cur, t, h, base + grp < p.M);
  for (; base < p.M; base += stride) {
    const int64_t row = base + grp;
    const bool valid = row < p.M;
    int64_t tn = t + dt, hn = h + dh;
    if (hn >= H) {
      hn -= H;
      ++tn;
    }
    if (PF) load(nxt, tn, hn, row + stride < p.M);
    float ss = 0.f, ss1 = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if constexpr (std::is_same<TX, bf16>::value) {
        bf16x8_sumsq(cur[k], ss, ss1);
      } else {
        float f[E];
        unpack(cur[k], f);
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(f[e], f[e], ss);
      }
    }
    ss = group_sum<G>(ss + ss1);
    const float rs = rsqrtf(fmaf(ss, p.inv_n, p.eps));
    if (valid && lane == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    TX* yr = y + t * p.y_st + h * p.y_sh;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * G;
      if (valid && v < p.nvec) st_stream(yr + v * E, scale_vec<TX, TW>(cur[k], gw[k], rs));
    }
    if (PF) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) cur[k] = nxt[k];
    } else {
      load(cur, tn, hn, row + stride < p.M);
    }
    t = tn;
    h = hn;
  }
}

// Strided rows, any alignment and any D: one row per 256-thread CTA, scalar,
// two passes (the second re-reads the row, from L2 for rows of this size).
template <typename TX, typename TW>
__global__ void __launch_bounds__(256) fwd_strided_generic_kernel(const FwdParams p) {
  pdl_begin();
  __shared__ float red[64];
  const int tid = threadIdx.x, T = blockDim.x;
  const int D = p.N;
  const TW* g = static_cast<const TW*>(p.gamma);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const int64_t t = row / p.heads, h = row % p.heads;
    const TX* xr = static_cast<const TX*>(p.x) + t * p.x_st + h * p.x_sh;
    TX* yr = static_cast<TX*>(p.y) + t * p.y_st + h * p.y_sh;
    float ss[1] = {0.f};
    for (int j = tid; j < D; j += T) {
      const float v = ld_scalar(xr + j);
      ss[0] = fmaf(v, v, ss[0]);
    }
    cta_sum<1>(ss, red, parity);
    parity ^= 1;
    const float rs = rsqrtf(fmaf(ss[0], p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    for (int j = tid; j < D; j += T) st_scalar(yr + j, ld_scalar(xr + j) * rs * ld_scalar(g + j));
  }
}

// ---------------------------------------------------------------------------
// kGeneric: any N and any element-aligned pointers.  Pass 1 reads the row
// (fused: forms, rounds and stores h) and reduces; pass 2 re-reads it (from
// L2).  Each thread issues U scalar loads per operand before using any, so
// that a warp keeps U requests in flight instead of one (one load at a time
// left 8192 x 20000 bf16 at 0.29 of the copy bandwidth, latency-bound).
template <typename TX, typename TW, bool FUSED>
__global__ void __launch_bounds__(256) fwd_generic_kernel(const FwdParams p) {
  pdl_begin();
  constexpr int U = 8;
  __shared__ float red[64];
  const int tid = threadIdx.x, T = blockDim.x;
  const int N = p.N;
  const TW* g = static_cast<const TW*>(p.gamma);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const TX* xr = static_cast<const TX*>(p.x) + row * (int64_t)N;
    TX* hr = static_cast<TX*>(p.residual) + row * (int64_t)N;
    TX* yr = static_cast<TX*>(p.y) + row * (int64_t)N;
    float ss[1] = {0.f};
    for (int j0 = tid; j0 < N; j0 += U * T) {
      float v[U], r[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        v[u] = j < N ? ld_scalar(xr + j) : 0.f;
        if (FUSED) r[u] = j < N ? ld_scalar(hr + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        if (FUSED) {
          v[u] = round_to(r[u] + v[u], (TX*)nullptr);
          if (j < N) st_scalar(hr + j, v[u]);
        }
        ss[0] = fmaf(v[u], v[u], ss[0]);
      }
    }
    cta_sum<1>(ss, red, parity);
    parity ^= 1;
    const float rs = rsqrtf(fmaf(ss[0], p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    for (int j0 = tid; j0 < N; j0 += U * T) {
      float v[U], gv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        v[u] = j < N ? (FUSED ? ld_scalar(hr + j) : ld_scalar(xr + j)) : 0.f;
        gv[u] = j < N ? ld_scalar(g + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        if (j < N) st_scalar(yr + j, v[u] * rs * gv[u]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Instantiation table (one dtype pair per translation unit, see RMSN_PAIR).

template <typename TX, typename TW, bool FUSED, bool PF>
FwdKernel pick_subwarp(int g, int vpt) {
#define RMSN_SW(G_, V_) \
  if (g == G_ && vpt == V_) return fwd_subwarp_kernel<TX, TW, G_, V_, FUSED, PF>;
  RMSN_SW(4, 1) RMSN_SW(8, 1) RMSN_SW(16, 1) RMSN_SW(32, 1)
  RMSN_SW(8, 2) RMSN_SW(16, 2) RMSN_SW(32, 2) RMSN_SW(32, 3) RMSN_SW(32, 4)
#undef RMSN_SW
  return nullptr;
}

template <typename TX, typename TW, bool FUSED>
FwdKernel pick_cta(int vpt, bool pf) {
  switch (vpt) {
    case 1: return pf ? fwd_cta_kernel<TX, TW, 1, FUSED, true> : fwd_cta_kernel<TX, TW, 1, FUSED, false>;
    case 2: return pf ? fwd_cta_kernel<TX, TW, 2, FUSED, true> : fwd_cta_kernel<TX, TW, 2, FUSED, false>;
    case 4: return pf ? fwd_cta_kernel<TX, TW, 4, FUSED, true> : fwd_cta_kernel<TX, TW, 4, FUSED, false>;
    case 8: return pf ? nullptr : fwd_cta_kernel<TX, TW, 8, FUSED, false>;
    default: return nullptr;
  }
}

template <typename TX, typename TW, bool PF>
FwdKernel pick_strided(int g, int vpt) {
#define RMSN_ST(G_, V_) \
  if (g == G_ && vpt == V_) return fwd_strided_kernel<TX, TW, G_, V_, PF>;
  RMSN_ST(4, 1) RMSN_ST(8, 1) RMSN_ST(16, 1) RMSN_ST(32, 1)
  RMSN_ST(8, 2) RMSN_ST(16, 2) RMSN_ST(32, 2) RMSN_ST(32, 3) RMSN_ST(32, 4)
#undef RMSN_ST
  return nullptr;
}

template <typename TX, typename TW, bool FUSED>
FwdKernel pick_family(const FwdKey& k) {
  if (k.strided) {
    if (FUSED) return nullptr;
    if (k.family == kGeneric) return fwd_strided_generic_kernel<TX, TW>;
    if (k.family != kSubwarp) return nullptr;
    return k.prefetch ? pick_strided<TX, TW, true>(k.g, k.vpt)
                      : pick_strided<TX, TW, false>(k.g, k.vpt);
  }
  switch (k.family) {
    case kSubwarp:
      return k.prefetch ? pick_subwarp<TX, TW, FUSED, true>(k.g, k.vpt)
                        : pick_subwarp<TX, TW, FUSED, false>(k.g, k.vpt);
    case kCta: return pick_cta<TX, TW, FUSED>(k.vpt, k.prefetch);
    case kGeneric: return fwd_generic_kernel<TX, TW, FUSED>;
    default: return nullptr;
  }
}

template <typename TX, typename TW>
FwdKernel pick_fused(const FwdKey& k) {
  return k.fused ? pick_family<TX, TW, true>(k) : pick_family<TX, TW, false>(k);
}

}  // namespace

#if RMSN_PAIR == 0
FwdKernel get_fwd_kernel_f32_f32(const FwdKey& k) { return pick_fused<float, float>(k); }
#elif RMSN_PAIR == 1
FwdKernel get_fwd_kernel_bf16_bf16(const FwdKey& k) { return pick_fused<bf16, bf16>(k); }
#else
FwdKernel get_fwd_kernel_bf16_f32(const FwdKey& k) { return pick_fused<bf16, float>(k); }
#endif

}  // namespace rmsn
