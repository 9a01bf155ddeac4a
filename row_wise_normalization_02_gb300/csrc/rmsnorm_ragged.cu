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
//
// Mixed alignment (compiled with RMSN_MIX=1): the inputs x and dy need not
// start where the output does modulo 16.  The head / body / tail split is
// then the output's (y or h, dx), and an input whose rows lie s bytes past
// it (the same s for every row) is read in aligned 16-byte chunks: body
// vector v is the last 16 - s bytes of chunk v and the first s bytes of
// chunk v + 1, which the next lane holds (a warp shuffle).  A warp therefore
// owns 31 body vectors per slot; its lane 31 loads the chunk after them --
// the next warp's first -- and writes nothing.  The bytes each lane reads
// from HBM are unchanged; only 1 in 32 chunks is fetched twice (from L2).
#include <type_traits>

#include "rmsnorm_bwd_common.cuh"
#include "rmsnorm_fwd_common.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif
#ifndef RMSN_MIX
#define RMSN_MIX 0
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

// Body vector held by slot k of thread tid (T threads, a multiple of 32), and
// whether that thread owns it (computes and stores it).  Mixed alignment:
// 31 vectors per warp and slot, lane 31 carrying the next warp's first chunk.
template <bool MIX>
__device__ __forceinline__ int vec_of(int tid, int k, int T) {
  if constexpr (MIX) return ((tid >> 5) + k * (T >> 5)) * 31 + (tid & 31);
  else return tid + k * T;
}
template <bool MIX>
__device__ __forceinline__ bool owns(int v, int nb, int tid) {
  return v < nb && (!MIX || (tid & 31) != 31);
}

// Body vector v of an operand row (p: the vector's first element) whose rows
// start s bytes past the output's.  s == 0: the vector itself.  Otherwise the
// aligned chunk that holds the vector's first bytes, for v <= nb when the row
// has a body (nb > 0; only then is the body's start, and so p - s, on 16
// bytes): chunk nb still holds s bytes of the row, and an aligned 16-byte
// chunk never crosses a page.
template <bool MIX, bool RW, typename TX>
__device__ __forceinline__ uint4 ld_body(const TX* p, int v, int nb, int s) {
  if constexpr (MIX) {
    if (v < nb + (s != 0 && nb > 0 ? 1 : 0)) {
      const void* q = reinterpret_cast<const char*>(p) - s;
      return RW ? ld_rw(q) : ld_stream(q);
    }
    return make_uint4(0, 0, 0, 0);
  } else {
    return v < nb ? (RW ? ld_rw(p) : ld_stream(p)) : make_uint4(0, 0, 0, 0);
  }
}

// Chunks -> vectors: the 16 bytes that start s bytes (0 < s < 16) into this
// lane's chunk, i.e. its last 16 - s bytes and the next lane's first s.  All
// 32 lanes take part; lane 31's result is meaningless (its vector is not
// owned).
__device__ __forceinline__ uint4 realign(const uint4& c, int s) {
  const uint4 n = make_uint4(__shfl_down_sync(0xffffffffu, c.x, 1),
                             __shfl_down_sync(0xffffffffu, c.y, 1),
                             __shfl_down_sync(0xffffffffu, c.z, 1),
                             __shfl_down_sync(0xffffffffu, c.w, 1));
  return realign_pair(c, n, s);
}

// An input's body vector in slot k ready for use: realigned (mixed alignment,
// s != 0) and zero unless this thread owns it.  Uniform in s, so the
// shuffles run on full warps.
template <bool MIX>
__device__ __forceinline__ void settle(uint4& r, int s, int v, int nb, int tid) {
  if constexpr (MIX) {
    if (s != 0) r = realign(r, s);
    if (!owns<MIX>(v, nb, tid)) r = make_uint4(0, 0, 0, 0);
  }
}

template <typename TW, typename TX, int VPT, bool MIX>
__device__ __forceinline__ void gather_gamma(const TW* gp, const Layout& L, int tid, int T,
                                             float (&g)[VPT][Elem<TX>::kPerVec], float& gs) {
  constexpr int E = Elem<TX>::kPerVec;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = vec_of<MIX>(tid, k, T);
    const bool own = owns<MIX>(v, L.nb, tid);
#pragma unroll
    for (int e = 0; e < E; ++e) g[k][e] = own ? ld_scalar_ro(gp + L.h + v * E + e) : 0.f;
  }
  gs = L.scol >= 0 ? ld_scalar_ro(gp + L.scol) : 0.f;
}

// The same gamma packed like the activations (GW 16-byte words per body
// vector: bf16 weights exactly, fp32 weights as they are), for the forward's
// packed-word arithmetic; gathered by scalar loads once per CTA.
template <typename TX, typename TW, int VPT, bool MIX>
__device__ __forceinline__ void gather_gamma_packed(const TW* gp, const Layout& L, int tid, int T,
                                                    uint4 (&gw)[VPT][Cfg<TX, TW>::GW],
                                                    float& gs) {
  constexpr int E = Cfg<TX, TW>::E, GW = Cfg<TX, TW>::GW;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = vec_of<MIX>(tid, k, T);
    const bool own = owns<MIX>(v, L.nb, tid);
    float f[E];
#pragma unroll
    for (int e = 0; e < E; ++e) f[e] = own ? ld_scalar_ro(gp + L.h + v * E + e) : 0.f;
    if constexpr (std::is_same<TW, float>::value) {
#pragma unroll
      for (int q = 0; q < GW; ++q) {
        const float t[4] = {f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]};
        gw[k][q] = pack(t);
      }
    } else {
      gw[k][0] = pack(f);
    }
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

// Load row `row` of up to three operands (b: the residual with `b_rw`, or
// dy; c: dres).  sa, sb: the byte shifts of a and b against the output
// (mixed alignment only; c and a read-written b share the output's).
template <typename TX, int VPT, bool TWO, bool B_RW, bool THREE = false, bool MIX = false>
__device__ __forceinline__ void load_row(RowRegs<VPT, TWO, THREE>& R, const TX* a, const TX* b,
                                         int64_t row, int N, const Layout& L, int tid, int T,
                                         const TX* c = nullptr, int sa = 0, int sb = 0) {
  constexpr int E = Elem<TX>::kPerVec;
  const TX* ar = a + row * (int64_t)N;
  const TX* br = b + row * (int64_t)N;
  const TX* cr = c + row * (int64_t)N;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = vec_of<MIX>(tid, k, T);
    R.a[k] = ld_body<MIX, false>(ar + L.h + v * E, v, L.nb, sa);
    if constexpr (TWO) R.b[k] = ld_body<MIX, B_RW>(br + L.h + v * E, v, L.nb, sb);
    if constexpr (THREE) R.c[k] = ld_body<MIX, true>(cr + L.h + v * E, v, L.nb, 0);
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
// Forward / fused add (b = residual, in r, out h).  The body's arithmetic is
// the aligned kernels' (rmsnorm_fwd_common.cuh): gamma packed like the
// activations, bf16 squares and products straight from the packed words.
template <typename TX, typename TW, int VPT, bool FUSED, bool PF, bool MIX>
__device__ __forceinline__ void fwd_ragged_body(const FwdParams& p) {
  if (threadIdx.x == 0) {   // the interiors of the first two rows into L2 before the wait
    const Walk w0 = walk_of(p.period, p.M);
    const size_t rb0 = (size_t)p.N * sizeof(TX);
    for (int k = 0; k < 2; ++k) {
      l2_prefetch_row_interior(p.x, w0.first + k * w0.stride, p.M, rb0);
      if (FUSED) l2_prefetch_row_interior(p.residual, w0.first + k * w0.stride, p.M, rb0);
    }
  }
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW;
  extern __shared__ float4 smem4[];
  float* red = reinterpret_cast<float*>(smem4);
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const Walk w = walk_of(p.period, p.M);
  const TX* x = static_cast<const TX*>(p.x);
  TX* res = static_cast<TX*>(p.residual);
  TX* y = static_cast<TX*>(p.y);
  // the split follows the output (h over the residual for the fused add)
  const Layout L = layout_of<TX>((FUSED ? static_cast<const TX*>(res) : y) + w.cls * (int64_t)N,
                                 N, tid);
  const int sx = MIX ? p.x_shift : 0;
  uint4 gw[VPT][GW];
  float gs;
  gather_gamma_packed<TX, TW, VPT, MIX>(static_cast<const TW*>(p.gamma), L, tid, T, gw, gs);

  int parity = 0;
  RowRegs<VPT, FUSED> cur, nxt;
  if (w.first < p.M)
    load_row<TX, VPT, FUSED, true, false, MIX>(cur, x, res, w.first, N, L, tid, T, nullptr, sx);
  for (int64_t row = w.first; row < p.M; row += w.stride) {
    const int64_t nrow = row + w.stride;
    if (PF && nrow < p.M)
      load_row<TX, VPT, FUSED, true, false, MIX>(nxt, x, res, nrow, N, L, tid, T, nullptr, sx);
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
    float ss = sv * sv, ss1 = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = vec_of<MIX>(tid, k, T);
      settle<MIX>(cur.a[k], sx, v, L.nb, tid);
      if constexpr (FUSED) {   // h = round(r + x), stored over the residual
        settle<MIX>(cur.b[k], 0, v, L.nb, tid);
        float f[E], rf[E];
        unpack(cur.a[k], f);
        unpack(cur.b[k], rf);
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] += rf[e];
        cur.a[k] = pack(f);
        if (owns<MIX>(v, L.nb, tid)) st_stream(hr + L.h + v * E, cur.a[k]);
      }
      if constexpr (std::is_same<TX, bf16>::value) {
        bf16x8_sumsq(cur.a[k], ss, ss1);
      } else {
        float f[E];
        unpack(cur.a[k], f);
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(f[e], f[e], ss);
      }
    }
    float sums[1] = {ss + ss1};
    cta_sum<1>(sums, red, parity);
    parity ^= 1;
    const float rs = rsqrtf(fmaf(sums[0], p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = vec_of<MIX>(tid, k, T);
      if (owns<MIX>(v, L.nb, tid)) st_stream(yr + L.h + v * E, scale_vec<TX, TW>(cur.a[k], gw[k], rs));
    }
    if (L.scol >= 0) st_scalar(yr + L.scol, sv * rs * gs);
    if (PF) cur = nxt;
    else if (nrow < p.M)
      load_row<TX, VPT, FUSED, true, false, MIX>(cur, x, res, nrow, N, L, tid, T, nullptr, sx);
  }
}

template <typename TX, typename TW, int VPT, bool FUSED, bool PF, bool MIX>
__global__ void __launch_bounds__(kCtaMaxThreads) fwd_ragged_kernel(const FwdParams p) {
  fwd_ragged_body<TX, TW, VPT, FUSED, PF, MIX>(p);
}
// The same held to 72 registers, for the plain mixed form with 4 vectors per
// thread and prefetch: three CTAs of 288 threads (8192 bf16 rows) fit an SM
// (it takes 77 otherwise, and two); no spills.
template <typename TX, typename TW, int VPT, bool FUSED, bool PF, bool MIX>
__global__ void __maxnreg__(72) fwd_ragged_kernel_r72(const FwdParams p) {
  fwd_ragged_body<TX, TW, VPT, FUSED, PF, MIX>(p);
}

// ---------------------------------------------------------------------------
// Backward (a = x, b = dy; fused-add backward: c = dres, added to dx).
template <typename TX, typename TW, int VPT, bool HAS_RSTD, bool PF, bool DRES, bool MIX>
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
  // the split follows dx (and dres, which shares its alignment)
  const Layout L = layout_of<TX>(dx + w.cls * (int64_t)N, N, tid);
  const int sx = MIX ? p.x_shift : 0, sd = MIX ? p.dy_shift : 0;
  float g[VPT][E], gs;
  gather_gamma<TW, TX, VPT, MIX>(static_cast<const TW*>(p.gamma), L, tid, T, g, gs);
  float acc[VPT][E], acc_s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = 0.f;

  int parity = 0;
  RowRegs<VPT, true, DRES> cur, nxt;
  const TX* dres = static_cast<const TX*>(p.dres);
  if (w.first < p.M)
    load_row<TX, VPT, true, false, DRES, MIX>(cur, x, dy, w.first, N, L, tid, T, dres, sx, sd);
  for (int64_t row = w.first; row < p.M; row += w.stride) {
    const int64_t nrow = row + w.stride;
    if (PF && nrow < p.M)
      load_row<TX, VPT, true, false, DRES, MIX>(nxt, x, dy, nrow, N, L, tid, T, dres, sx, sd);
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
    for (int k = 0; k < VPT; ++k) {
      const int v = vec_of<MIX>(tid, k, T);
      settle<MIX>(cur.a[k], sx, v, L.nb, tid);
      settle<MIX>(cur.b[k], sd, v, L.nb, tid);
      bwd_vec_sums<E, !HAS_RSTD>(cur.a[k], cur.b[k], g[k], dot2, ss2);
    }
    float sums[K];
    sums[0] = dot2.x + dot2.y;
    if (!HAS_RSTD) sums[K - 1] = ss2.x + ss2.y;
    cta_sum<K>(sums, red, parity);
    parity ^= 1;
    const float r = HAS_RSTD ? r_saved : rsqrtf(fmaf(sums[K - 1], p.inv_n, p.eps));
    const float c = r * r * p.inv_n * sums[0];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = vec_of<MIX>(tid, k, T);
      if (owns<MIX>(v, L.nb, tid))
        st_stream(dxr + L.h + v * E, bwd_vec_apply<E, DRES>(cur.a[k], cur.b[k], cur.c[DRES ? k : 0],
                                                            g[k], r, c, acc[k]));
    }
    if (L.scol >= 0) {
      st_scalar(dxr + L.scol, r * fmaf(-xs, c, gs * ds) + (DRES ? cur.cs : 0.f));
      acc_s = fmaf(ds * xs, r, acc_s);
    }
    if (PF) cur = nxt;
    else if (nrow < p.M)
      load_row<TX, VPT, true, false, DRES, MIX>(cur, x, dy, nrow, N, L, tid, T, dres, sx, sd);
  }
  if (p.partial == nullptr) return;
  // every column of the partial row is written by exactly one thread
  float* prow = p.partial + (size_t)blockIdx.x * p.ld_partial;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = vec_of<MIX>(tid, k, T);
    if (owns<MIX>(v, L.nb, tid)) {
#pragma unroll
      for (int e = 0; e < E; ++e) prow[L.h + v * E + e] = acc[k][e];
    }
  }
  if (L.scol >= 0) prow[L.scol] = acc_s;
}

constexpr bool kMix = RMSN_MIX != 0;

template <typename TX, typename TW, bool FUSED>
FwdKernel pick_fwd(int vpt, bool pf) {
  switch (vpt) {
    case 1: return pf ? fwd_ragged_kernel<TX, TW, 1, FUSED, true, kMix>
                      : fwd_ragged_kernel<TX, TW, 1, FUSED, false, kMix>;
    case 2: return pf ? fwd_ragged_kernel<TX, TW, 2, FUSED, true, kMix>
                      : fwd_ragged_kernel<TX, TW, 2, FUSED, false, kMix>;
    case 4:
      if constexpr (kMix && !FUSED)
        if (pf) return fwd_ragged_kernel_r72<TX, TW, 4, FUSED, true, kMix>;
      return pf ? fwd_ragged_kernel<TX, TW, 4, FUSED, true, kMix>
                : fwd_ragged_kernel<TX, TW, 4, FUSED, false, kMix>;
    default: return nullptr;
  }
}

template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
BwdKernel pick_bwd(int vpt, bool pf) {
  switch (vpt) {
    case 1: return pf ? bwd_ragged_kernel<TX, TW, 1, HAS_RSTD, true, DRES, kMix>
                      : bwd_ragged_kernel<TX, TW, 1, HAS_RSTD, false, DRES, kMix>;
    case 2: return pf ? bwd_ragged_kernel<TX, TW, 2, HAS_RSTD, true, DRES, kMix>
                      : bwd_ragged_kernel<TX, TW, 2, HAS_RSTD, false, DRES, kMix>;
    case 4: return pf ? nullptr : bwd_ragged_kernel<TX, TW, 4, HAS_RSTD, false, DRES, kMix>;
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

#if RMSN_PAIR == 0 && !RMSN_MIX
FwdKernel get_fwd_ragged_f32_f32(const FwdKey& k) { return ragged_fwd<float, float>(k); }
BwdKernel get_bwd_ragged_f32_f32(const BwdKey& k) { return ragged_bwd<float, float>(k); }
#elif RMSN_PAIR == 1 && !RMSN_MIX
FwdKernel get_fwd_ragged_bf16_bf16(const FwdKey& k) { return ragged_fwd<bf16, bf16>(k); }
BwdKernel get_bwd_ragged_bf16_bf16(const BwdKey& k) { return ragged_bwd<bf16, bf16>(k); }
#elif !RMSN_MIX
FwdKernel get_fwd_ragged_bf16_f32(const FwdKey& k) { return ragged_fwd<bf16, float>(k); }
BwdKernel get_bwd_ragged_bf16_f32(const BwdKey& k) { return ragged_bwd<bf16, float>(k); }
#elif RMSN_PAIR == 0
FwdKernel get_fwd_ragged_mix_f32_f32(const FwdKey& k) { return ragged_fwd<float, float>(k); }
BwdKernel get_bwd_ragged_mix_f32_f32(const BwdKey& k) { return ragged_bwd<float, float>(k); }
#elif RMSN_PAIR == 1
FwdKernel get_fwd_ragged_mix_bf16_bf16(const FwdKey& k) { return ragged_fwd<bf16, bf16>(k); }
BwdKernel get_bwd_ragged_mix_bf16_bf16(const BwdKey& k) { return ragged_bwd<bf16, bf16>(k); }
#else
FwdKernel get_fwd_ragged_mix_bf16_f32(const FwdKey& k) { return ragged_fwd<bf16, float>(k); }
BwdKernel get_bwd_ragged_mix_bf16_f32(const BwdKey& k) { return ragged_bwd<bf16, float>(k); }
#endif

}  // namespace rmsn
