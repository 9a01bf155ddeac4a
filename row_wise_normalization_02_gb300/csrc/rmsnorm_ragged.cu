// RMSNorm forward, fused add and backward for rows that do not start on a
// 16-byte boundary (for example N = 2049 bf16), sm_103a.
//
// Arithmetic as in rmsnorm_fwd.cu / rmsnorm_bwd.cu.  A row is split into a
// scalar head up to its first 16-byte boundary, a body of 16-byte vectors and
// a scalar tail ("Pre-built kernel library guide", section 1.1: vector body
// plus scalar tail for arbitrary N; here also a head, because the row start
// moves).  The split depends only on the row's start address modulo 16, which
// repeats with period P = 16 / gcd(N * size, 16) rows.  Each CTA therefore
// walks rows of one residue class modulo P: its head, body and tail -- and so
// the columns each thread touches -- are the same for every row it handles.
// Gamma is gathered into registers once per CTA and the backward's dgamma
// partials stay in registers, exactly as for aligned rows.
#include <type_traits>

#include "rmsnorm_bwd_common.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif

namespace rmsn {
namespace {

// Head scalars h, body vectors nb, tail scalars tl of a row starting at row0,
// and the column of the one head/tail scalar thread `tid` owns (-1: none):
// threads 0..h-1 own the head, threads 8..8+tl-1 the tail (h, tl < 8).
struct Layout {
  int h, nb, tl, scol;
};

template <typename TX>
__device__ __forceinline__ Layout layout_of(const void* row0, int N, int tid) {
  constexpr int E = Elem<TX>::kPerVec;
  Layout L;
  const int mis = (int)(reinterpret_cast<uintptr_t>(row0) & 15);
  int h = mis ? (16 - mis) / (int)sizeof(TX) : 0;
  if (h > N) h = N;
  L.h = h;
  L.nb = (N - h) / E;
  L.tl = N - h - L.nb * E;
  L.scol = tid < h ? tid : (tid >= 8 && tid - 8 < L.tl) ? h + L.nb * E + (tid - 8) : -1;
  return L;
}

// Rows of this CTA: residue class c = blockIdx mod P, then every
// (gridDim / P)-th row of that class (gridDim is a multiple of P).
struct Walk {
  int64_t first, stride, cls;
};
__device__ __forceinline__ Walk walk_of(int period, int64_t M) {
  const int c = blockIdx.x % period, j = blockIdx.x / period;
  const int per_class = gridDim.x / period;
  // a CTA beyond whole classes (never launched so) walks no rows
  const int64_t first = j < per_class ? c + (int64_t)period * j : M;
  return Walk{first, (int64_t)period * (per_class > 0 ? per_class : 1), c};
}

template <typename TW, typename TX, int VPT>
__device__ __forceinline__ void gather_gamma(const TW* gp, const Layout& L, int tid, int T,
                                             float (&g)[VPT][Elem<TX>::kPerVec], float& gs) {
  constexpr int E = Elem<TX>::kPerVec;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
#pragma unroll
    for (int e = 0; e < E; ++e) g[k][e] = v < L.nb ? ld_scalar_ro(gp + L.h + v * E + e) : 0.f;
  }
  gs = L.scol >= 0 ? ld_scalar_ro(gp + L.scol) : 0.f;
}

// Registers of one row: body vectors of x (and of dy or of the residual) and
// the one head/tail scalar of each.
template <int VPT, bool TWO, bool THREE = false>
struct RowRegs {
  uint4 a[VPT];
  uint4 b[TWO ? VPT : 1];
  uint4 c[THREE ? VPT : 1];
  float as, bs, cs;
};

// Load row `row` of up to two operands (b: the residual with `b_rw`, or dy).
template <typename TX, int VPT, bool TWO, bool B_RW, bool THREE = false>
__device__ __forceinline__ void load_row(RowRegs<VPT, TWO, THREE>& R, const TX* a, const TX* b,
                                         int64_t row, int N, const Layout& L, int tid, int T,
                                         const TX* c = nullptr) {
  constexpr int E = Elem<TX>::kPerVec;
  const TX* ar = a + row * (int64_t)N;
  const TX* br = b + row * (int64_t)N;
  const TX* cr = c + row * (int64_t)N;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    R.a[k] = v < L.nb ? ld_stream(ar + L.h + v * E) : make_uint4(0, 0, 0, 0);
    if constexpr (TWO) {
      if (B_RW) R.b[k] = v < L.nb ? ld_rw(br + L.h + v * E) : make_uint4(0, 0, 0, 0);
      else R.b[k] = v < L.nb ? ld_stream(br + L.h + v * E) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (THREE) R.c[k] = v < L.nb ? ld_rw(cr + L.h + v * E) : make_uint4(0, 0, 0, 0);
  }
  R.as = L.scol >= 0 ? ld_scalar(ar + L.scol) : 0.f;
  R.bs = (TWO && L.scol >= 0) ? ld_scalar(br + L.scol) : 0.f;
  R.cs = (THREE && L.scol >= 0) ? ld_scalar(cr + L.scol) : 0.f;
}

// Row `row` of a row-major array whose rows need not start on 16 bytes,
// requested into L2 by the calling thread: the 16-byte-aligned interior of
// the row only, so that every byte asked for lies inside it.
__device__ __forceinline__ void l2_prefetch_row_interior(const void* a, int64_t row, int64_t M,
                                                         size_t rb) {
  if (row >= M) return;
  const uintptr_t s = reinterpret_cast<uintptr_t>(a) + (uintptr_t)row * rb;
  const uintptr_t lo = (s + 15) & ~(uintptr_t)15, hi = (s + rb) & ~(uintptr_t)15;
  if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), (uint32_t)(hi - lo));
}

// ---------------------------------------------------------------------------
// Forward / fused add (b = residual, in r, out h).
template <typename TX, typename TW, int VPT, bool FUSED, bool PF>
__global__ void __launch_bounds__(kCtaMaxThreads) fwd_ragged_kernel(const FwdParams p) {
  if (threadIdx.x == 0) {   // the interiors of the first two rows into L2 before the wait
    const Walk w0 = walk_of(p.period, p.M);
    const size_t rb0 = (size_t)p.N * sizeof(TX);
    for (int k = 0; k < 2; ++k) {
      l2_prefetch_row_interior(p.x, w0.first + k * w0.stride, p.M, rb0);
      if (FUSED) l2_prefetch_row_interior(p.residual, w0.first + k * w0.stride, p.M, rb0);
    }
  }
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  extern __shared__ float4 smem4[];
  float* red = reinterpret_cast<float*>(smem4);
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const Walk w = walk_of(p.period, p.M);
  const TX* x = static_cast<const TX*>(p.x);
  TX* res = static_cast<TX*>(p.residual);
  TX* y = static_cast<TX*>(p.y);
  const Layout L = layout_of<TX>(x + w.cls * (int64_t)N, N, tid);
  float g[VPT][E], gs;
  gather_gamma<TW, TX, VPT>(static_cast<const TW*>(p.gamma), L, tid, T, g, gs);

  int parity = 0;
  RowRegs<VPT, FUSED> cur, nxt;
  if (w.first < p.M) load_row<TX, VPT, FUSED, true>(cur, x, res, w.first, N, L, tid, T);
  for (int64_t row = w.first; row < p.M; row += w.stride) {
    const int64_t nrow = row + w.stride;
    if (PF && nrow < p.M) load_row<TX, VPT, FUSED, true>(nxt, x, res, nrow, N, L, tid, T);
    if (PF && p.l2_rows > 0 && tid == 0) {   // the row l2_rows steps ahead in this walk
      const int64_t ahead = row + (int64_t)p.l2_rows * w.stride;
      l2_prefetch_row_interior(x, ahead, p.M, (size_t)N * sizeof(TX));
      if (FUSED) l2_prefetch_row_interior(res, ahead, p.M, (size_t)N * sizeof(TX));
    }
    TX* hr = res + row * (int64_t)N;
    TX* yr = y + row * (int64_t)N;
    float sv = cur.as;
    if (FUSED) {
      sv = round_to(cur.bs + sv, (TX*)nullptr);
      if (L.scol >= 0) st_scalar(hr + L.scol, sv);
    }
    float ss[1] = {sv * sv};
    uint4 hv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      float f[E];
      hv[k] = cur.a[k];
      unpack(hv[k], f);
      if constexpr (FUSED) {
        float rf[E];
        unpack(cur.b[k], rf);
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] += rf[e];
        hv[k] = pack(f);
        unpack(hv[k], f);
        if (v < L.nb) st_stream(hr + L.h + v * E, hv[k]);
      }
#pragma unroll
      for (int e = 0; e < E; ++e) ss[0] = fmaf(f[e], f[e], ss[0]);
    }
    cta_sum<1>(ss, red, parity);
    parity ^= 1;
    const float rs = rsqrtf(fmaf(ss[0], p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < L.nb) {
        float o[E];
        unpack(hv[k], o);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = o[e] * rs * g[k][e];
        st_stream(yr + L.h + v * E, pack(o));
      }
    }
    if (L.scol >= 0) st_scalar(yr + L.scol, sv * rs * gs);
    if (PF) cur = nxt;
    else if (nrow < p.M) load_row<TX, VPT, FUSED, true>(cur, x, res, nrow, N, L, tid, T);
  }
}

// ---------------------------------------------------------------------------
// Backward (a = x, b = dy; fused-add backward: c = dres, added to dx).
template <typename TX, typename TW, int VPT, bool HAS_RSTD, bool PF, bool DRES>
__global__ void __launch_bounds__(kCtaMaxThreads) bwd_ragged_kernel(const BwdParams p) {
  if (threadIdx.x == 0) {   // the interiors of the first two rows into L2 before the wait
    const Walk w0 = walk_of(p.period, p.M);
    const size_t rb0 = (size_t)p.N * sizeof(TX);
    for (int k = 0; k < 2; ++k) {
      l2_prefetch_row_interior(p.x, w0.first + k * w0.stride, p.M, rb0);
      l2_prefetch_row_interior(p.dy, w0.first + k * w0.stride, p.M, rb0);
      if (DRES) l2_prefetch_row_interior(p.dres, w0.first + k * w0.stride, p.M, rb0);
    }
  }
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int K = HAS_RSTD ? 1 : 2;
  extern __shared__ float4 smem4[];
  float* red = reinterpret_cast<float*>(smem4);
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const Walk w = walk_of(p.period, p.M);
  const TX* x = static_cast<const TX*>(p.x);
  const TX* dy = static_cast<const TX*>(p.dy);
  TX* dx = static_cast<TX*>(p.dx);
  const Layout L = layout_of<TX>(x + w.cls * (int64_t)N, N, tid);
  float g[VPT][E], gs;
  gather_gamma<TW, TX, VPT>(static_cast<const TW*>(p.gamma), L, tid, T, g, gs);
  float acc[VPT][E], acc_s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = 0.f;

  int parity = 0;
  RowRegs<VPT, true, DRES> cur, nxt;
  const TX* dres = static_cast<const TX*>(p.dres);
  if (w.first < p.M) load_row<TX, VPT, true, false, DRES>(cur, x, dy, w.first, N, L, tid, T, dres);
  for (int64_t row = w.first; row < p.M; row += w.stride) {
    const int64_t nrow = row + w.stride;
    if (PF && nrow < p.M) load_row<TX, VPT, true, false, DRES>(nxt, x, dy, nrow, N, L, tid, T, dres);
    if (PF && p.l2_rows > 0 && tid == 0) {
      const int64_t ahead = row + (int64_t)p.l2_rows * w.stride;
      l2_prefetch_row_interior(x, ahead, p.M, (size_t)N * sizeof(TX));
      l2_prefetch_row_interior(dy, ahead, p.M, (size_t)N * sizeof(TX));
      if (DRES) l2_prefetch_row_interior(dres, ahead, p.M, (size_t)N * sizeof(TX));
    }
    TX* dxr = dx + row * (int64_t)N;
    const float r_saved = HAS_RSTD ? __ldg(p.rstd + row) : 0.f;
    const float xs = cur.as, ds = cur.bs;
    float2 dot2 = make_float2(gs * ds * xs, 0.f), ss2 = make_float2(xs * xs, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) bwd_vec_sums<E, !HAS_RSTD>(cur.a[k], cur.b[k], g[k], dot2, ss2);
    float sums[K];
    sums[0] = dot2.x + dot2.y;
    if (!HAS_RSTD) sums[K - 1] = ss2.x + ss2.y;
    cta_sum<K>(sums, red, parity);
    parity ^= 1;
    const float r = HAS_RSTD ? r_saved : rsqrtf(fmaf(sums[K - 1], p.inv_n, p.eps));
    const float c = r * r * p.inv_n * sums[0];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < L.nb)
        st_stream(dxr + L.h + v * E, bwd_vec_apply<E, DRES>(cur.a[k], cur.b[k], cur.c[DRES ? k : 0],
                                                            g[k], r, c, acc[k]));
    }
    if (L.scol >= 0) {
      st_scalar(dxr + L.scol, r * fmaf(-xs, c, gs * ds) + (DRES ? cur.cs : 0.f));
      acc_s = fmaf(ds * xs, r, acc_s);
    }
    if (PF) cur = nxt;
    else if (nrow < p.M) load_row<TX, VPT, true, false, DRES>(cur, x, dy, nrow, N, L, tid, T, dres);
  }
  if (p.partial == nullptr) return;
  // every column of the partial row is written by exactly one thread
  float* prow = p.partial + (size_t)blockIdx.x * p.ld_partial;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    if (v < L.nb) {
#pragma unroll
      for (int e = 0; e < E; ++e) prow[L.h + v * E + e] = acc[k][e];
    }
  }
  if (L.scol >= 0) prow[L.scol] = acc_s;
}

template <typename TX, typename TW, bool FUSED>
FwdKernel pick_fwd(int vpt, bool pf) {
  switch (vpt) {
    case 1: return pf ? fwd_ragged_kernel<TX, TW, 1, FUSED, true> : fwd_ragged_kernel<TX, TW, 1, FUSED, false>;
    case 2: return pf ? fwd_ragged_kernel<TX, TW, 2, FUSED, true> : fwd_ragged_kernel<TX, TW, 2, FUSED, false>;
    case 4: return pf ? nullptr : fwd_ragged_kernel<TX, TW, 4, FUSED, false>;
    default: return nullptr;
  }
}

template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
BwdKernel pick_bwd(int vpt, bool pf) {
  switch (vpt) {
    case 1: return pf ? bwd_ragged_kernel<TX, TW, 1, HAS_RSTD, true, DRES>
                      : bwd_ragged_kernel<TX, TW, 1, HAS_RSTD, false, DRES>;
    case 2: return pf ? bwd_ragged_kernel<TX, TW, 2, HAS_RSTD, true, DRES>
                      : bwd_ragged_kernel<TX, TW, 2, HAS_RSTD, false, DRES>;
    case 4: return pf ? nullptr : bwd_ragged_kernel<TX, TW, 4, HAS_RSTD, false, DRES>;
    default: return nullptr;
  }
}

template <typename TX, typename TW>
FwdKernel ragged_fwd(const FwdKey& k) {
  return k.fused ? pick_fwd<TX, TW, true>(k.vpt, k.prefetch)
                 : pick_fwd<TX, TW, false>(k.vpt, k.prefetch);
}
template <typename TX, typename TW>
BwdKernel ragged_bwd(const BwdKey& k) {
  if (k.dres)
    return k.has_rstd ? pick_bwd<TX, TW, true, true>(k.vpt, k.prefetch)
                      : pick_bwd<TX, TW, false, true>(k.vpt, k.prefetch);
  return k.has_rstd ? pick_bwd<TX, TW, true, false>(k.vpt, k.prefetch)
                    : pick_bwd<TX, TW, false, false>(k.vpt, k.prefetch);
}

}  // namespace

#if RMSN_PAIR == 0
FwdKernel get_fwd_ragged_f32_f32(const FwdKey& k) { return ragged_fwd<float, float>(k); }
BwdKernel get_bwd_ragged_f32_f32(const BwdKey& k) { return ragged_bwd<float, float>(k); }
#elif RMSN_PAIR == 1
FwdKernel get_fwd_ragged_bf16_bf16(const FwdKey& k) { return ragged_fwd<bf16, bf16>(k); }
BwdKernel get_bwd_ragged_bf16_bf16(const BwdKey& k) { return ragged_bwd<bf16, bf16>(k); }
#else
FwdKernel get_fwd_ragged_bf16_f32(const FwdKey& k) { return ragged_fwd<bf16, float>(k); }
BwdKernel get_bwd_ragged_bf16_f32(const BwdKey& k) { return ragged_bwd<bf16, float>(k); }
#endif

}  // namespace rmsn
