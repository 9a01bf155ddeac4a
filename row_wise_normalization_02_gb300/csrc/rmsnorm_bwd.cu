// RMSNorm backward kernels for sm_103a.
//
// The backward reads the forward's input, gamma, dy and the saved rstd, and
// writes dx and the weight gradient ("Pre-built kernel library guide", section
// 1.2 RMSNorm: Input, Gamma, DY, Rstd -> DX, DWeight; eps is folded into
// rstd).  The guide does not print the formula; differentiating
// y_j = gamma_j x_j r, r = (mean(x^2) + eps)^(-1/2) gives, per row,
//     c    = r^2 / N * sum_k gamma_k dy_k x_k
//     dx_j = r * (gamma_j dy_j - x_j c)
//     dgamma_j = sum over rows of dy_j x_j r.
//
// Where the guide's kernel atomically adds every row into DWeight, this
// library reduces dgamma in a fixed order so the result is bit-for-bit
// reproducible: stage 1 runs a persistent grid of P CTAs with a fixed
// row -> CTA map, each CTA accumulating its rows' dy*x*r per column in fp32
// and writing one partial row; stage 2 (colsum_kernel, built with the staged
// kernels) sums the P partial rows per column in a fixed order.  Like every
// kernel here, stage 2 is a programmatic dependent launch: its launch
// overlaps stage 1, and it waits for stage 1 to complete before reading the
// partial rows.
#include <type_traits>

#include "rmsnorm_bwd_common.cuh"
#include "rmsnorm_ring.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif

namespace rmsn {
namespace {

template <int VPT, bool DRES = false>
struct BSlice {
  uint4 x[VPT];
  uint4 dy[VPT];
  uint4 dr[DRES ? VPT : 1];   // fused-add backward: residual-path gradient
  float r;                    // saved rstd of the row
};

template <typename TX, int VPT, bool HAS_RSTD, bool DRES = false>
__device__ __forceinline__ void bload_aligned(BSlice<VPT, DRES>& s, const BwdParams& p,
                                              int64_t row, bool valid, int lane, int stride) {
  const size_t rb = (size_t)p.N * sizeof(TX);
  const char* xr = static_cast<const char*>(p.x) + row * rb;
  const char* dr = static_cast<const char*>(p.dy) + row * rb;
  const char* rr = static_cast<const char*>(p.dres) + row * rb;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * stride;
    if (valid && v < p.nvec) {
      s.x[k] = ld_stream(xr + (size_t)v * 16);
      s.dy[k] = ld_stream(dr + (size_t)v * 16);
      if (DRES) s.dr[k] = ld_rw(rr + (size_t)v * 16);
    } else {
      s.x[k] = make_uint4(0, 0, 0, 0);
      s.dy[k] = make_uint4(0, 0, 0, 0);
      if (DRES) s.dr[k] = make_uint4(0, 0, 0, 0);
    }
  }
  if (HAS_RSTD) s.r = valid ? __ldg(p.rstd + row) : 0.f;
}

// ---------------------------------------------------------------------------
// kSubwarp: G lanes per row, 256 / G rows per CTA iteration; gamma and the
// dgamma partials in registers; the row groups of a CTA are combined in
// shared memory (in group order) at the end.
template <typename TX, typename TW, int G, int VPT, bool HAS_RSTD, bool PF, bool DRES>
__device__ __forceinline__ void bwd_subwarp_body(const BwdParams& p) {
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int RPC = kSubwarpThreads / G;
  {  // the first two iterations' rows into L2 while the previous kernel ends
    const size_t rb = (size_t)p.N * sizeof(TX);
    const void* r = DRES ? p.dres : nullptr;
    const int64_t b0 = (int64_t)blockIdx.x * RPC, st = (int64_t)gridDim.x * RPC;
    l2_warm(p.x, p.dy, r, b0, RPC, p.M, rb);
    if (PF) l2_warm(p.x, p.dy, r, b0 + st, RPC, p.M, rb);
  }
  pdl_begin();
  extern __shared__ float4 smem4[];
  float* sacc = reinterpret_cast<float*>(smem4);   // [RPC][nvec * E]
  const int lane = threadIdx.x % G, grp = threadIdx.x / G;
  const bool want_dg = p.partial != nullptr;

  float g[VPT][E];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * G;
    if (v < p.nvec) load_gamma_vec<TW, E>(p.gamma, v, g[k]);
    else
#pragma unroll
      for (int e = 0; e < E; ++e) g[k][e] = 0.f;
  }
  float acc[VPT][E];
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = 0.f;

  const int64_t stride = (int64_t)gridDim.x * RPC;
  int64_t base = (int64_t)blockIdx.x * RPC;
  BSlice<VPT, DRES> cur, nxt;
  bload_aligned<TX, VPT, HAS_RSTD, DRES>(cur, p, base + grp, base + grp < p.M, lane, G);
  for (; base < p.M; base += stride) {
    const int64_t row = base + grp;
    const bool valid = row < p.M;
    const int64_t nrow = row + stride;
    if (PF) bload_aligned<TX, VPT, HAS_RSTD, DRES>(nxt, p, nrow, nrow < p.M, lane, G);
    // with the next rows in registers, the rows after them are requested
    // into L2 (compiled into the prefetching forms only: the others keep
    // their register budget)
    if (PF && p.l2_rows > 0 && threadIdx.x == 0) {
      const int64_t ahead = base + (int64_t)p.l2_rows * stride;
      const size_t rb = (size_t)p.N * sizeof(TX);
      l2_prefetch_rows(p.x, ahead, RPC, p.M, rb);
      l2_prefetch_rows(p.dy, ahead, RPC, p.M, rb);
      if (DRES) l2_prefetch_rows(p.dres, ahead, RPC, p.M, rb);
    }

    float2 dot2 = make_float2(0.f, 0.f), ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k)
      bwd_vec_sums<E, !HAS_RSTD>(cur.x[k], cur.dy[k], g[k], dot2, ss2);
    float dot = group_sum<G>(dot2.x + dot2.y), ss = ss2.x + ss2.y;
    float r;
    if constexpr (HAS_RSTD) {
      r = cur.r;
    } else {
      ss = group_sum<G>(ss);
      r = rsqrtf(fmaf(ss, p.inv_n, p.eps));
    }
    const float c = r * r * p.inv_n * dot;
    char* dxr = static_cast<char*>(p.dx) + row * (size_t)p.N * sizeof(TX);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * G;
      const uint4 o = bwd_vec_apply<E, DRES>(cur.x[k], cur.dy[k], cur.dr[DRES ? k : 0], g[k], r,
                                             c, acc[k]);
      if (valid && v < p.nvec) st_stream(dxr + (size_t)v * 16, o);
    }
    if (PF) cur = nxt;
    else bload_aligned<TX, VPT, HAS_RSTD, DRES>(cur, p, nrow, nrow < p.M, lane, G);
  }
  if (!want_dg) return;
  const int ncol = p.nvec * E;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * G;
    if (v < p.nvec) {
      float4* d = reinterpret_cast<float4*>(sacc + grp * ncol + v * E);
#pragma unroll
      for (int q = 0; q < E / 4; ++q)
        d[q] = make_float4(acc[k][4 * q], acc[k][4 * q + 1], acc[k][4 * q + 2],
                           acc[k][4 * q + 3]);
    }
  }
  __syncthreads();
  float* prow = p.partial + (size_t)blockIdx.x * p.ld_partial;
  for (int j = threadIdx.x; j < ncol; j += kSubwarpThreads) {
    float s = 0.f;
    for (int q = 0; q < RPC; ++q) s += sacc[q * ncol + j];
    prow[j] = s;
  }
}

// Two entry points: the compiler's own register choice, and one held to two
// resident 256-thread CTAs per SM (128 registers) for the plain backward with
// two or three vectors per thread, where the paired arithmetic would otherwise
// take the full-warp, three-vector form to 158 registers and one CTA.  (Asking
// every form for its minimum explicitly grows the one-vector forms from ~60
// to 72-95 registers, so the others keep the plain bound.)
template <typename TX, typename TW, int G, int VPT, bool HAS_RSTD, bool PF, bool DRES>
__global__ void __launch_bounds__(kSubwarpThreads) bwd_subwarp_kernel(const BwdParams p) {
  bwd_subwarp_body<TX, TW, G, VPT, HAS_RSTD, PF, DRES>(p);
}
template <typename TX, typename TW, int G, int VPT, bool HAS_RSTD, bool PF, bool DRES>
__global__ void __launch_bounds__(kSubwarpThreads, 2) bwd_subwarp_kernel_2cta(const BwdParams p) {
  bwd_subwarp_body<TX, TW, G, VPT, HAS_RSTD, PF, DRES>(p);
}

// ---------------------------------------------------------------------------
// Short rows through a bulk-copy ring (kStaged with G lanes per row): a CTA
// iteration covers RPC = 256 / G consecutive rows, which are contiguous in
// memory, so one cp.async.bulk per operand fills a stage of the ring; the
// CTA keeps stages - 1 iterations of rows in flight without holding them in
// registers.  The row math is the sub-warp kernel's (paired fp32, shuffle
// reduction within the G lanes of a row); gamma and the dgamma partials stay
// in registers.  One CTA barrier per iteration both votes on the bounded
// waits (so the whole CTA agrees to stop) and proves that every thread has
// finished the previous iteration's stage, which thread 0 then refills.
template <typename TX, typename TW, int G, int VPT, bool HAS_RSTD, bool DRES>
__global__ void __launch_bounds__(kSubwarpThreads)
    bwd_rows_staged_kernel(const BwdParams p) {
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int RPC = kSubwarpThreads / G;
  constexpr int NS = DRES ? 3 : 2;
  {  // the rows of the first two iterations into L2 while the previous kernel ends
    const size_t rb = (size_t)p.N * sizeof(TX);
    const int64_t b0 = (int64_t)blockIdx.x * RPC, st = (int64_t)gridDim.x * RPC;
    l2_warm(p.x, p.dy, DRES ? p.dres : nullptr, b0, RPC, p.M, rb);
    l2_warm(p.x, p.dy, DRES ? p.dres : nullptr, b0 + st, RPC, p.M, rb);
  }
  pdl_begin();
  extern __shared__ __align__(128) unsigned char smem[];
  const Ring rg = ring_of(smem);
  const int lane = threadIdx.x % G, grp = threadIdx.x / G, tid = threadIdx.x;
  const int S = p.stages;
  const size_t rb = (size_t)p.N * sizeof(TX);
  const size_t blk = (size_t)RPC * rb;              // one operand's rows of a stage
  const int64_t units = (p.M + RPC - 1) / RPC;      // CTA iterations of RPC rows
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nit = first < units ? (units - 1 - first) / stride + 1 : 0;
  const char* src[3] = {static_cast<const char*>(p.x), static_cast<const char*>(p.dy),
                        static_cast<const char*>(p.dres)};

  // thread 0: the rows of iteration j into stage j mod S (the last unit may
  // hold fewer than RPC rows)
  auto issue = [&](int64_t j) {
    const int s = (int)(j % S);
    const int64_t row0 = (first + j * stride) * RPC;
    const int64_t n = p.M - row0 < RPC ? p.M - row0 : RPC;
    const uint32_t bytes = (uint32_t)(n * (int64_t)rb);
    uint64_t* bar = rg.full + s;
    unsigned char* dst = rg.buf + (size_t)s * NS * blk;
    mbar_arrive_expect_tx(bar, NS * bytes);
#pragma unroll
    for (int q = 0; q < NS; ++q) bulk_copy_g2s(dst + q * blk, src[q] + row0 * rb, bytes, bar);
  };
  int64_t issued = 0;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(rg.full + s, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0)
    for (; issued < (nit < S ? nit : S); ++issued) issue(issued);

  float g[VPT][E], acc[VPT][E];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = lane + k * G;
    if (v < p.nvec) load_gamma_vec<TW, E>(p.gamma, v, g[k]);
    else
#pragma unroll
      for (int e = 0; e < E; ++e) g[k][e] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = 0.f;
  }

  // the saved rstd of this thread's row, one iteration ahead in a register
  float r_next = 0.f;
  if (HAS_RSTD && nit > 0) {
    const int64_t row = first * RPC + grp;
    r_next = row < p.M ? __ldg(p.rstd + row) : 0.f;
  }
  int64_t j = 0;
  bool failed = false;
  for (; j < nit; ++j) {
    const int s = (int)(j % S);
    const int64_t row = (first + j * stride) * RPC + grp;
    const bool valid = row < p.M;
    const float r_saved = r_next;
    if (HAS_RSTD && j + 1 < nit) {
      const int64_t nrow = (first + (j + 1) * stride) * RPC + grp;
      r_next = nrow < p.M ? __ldg(p.rstd + nrow) : 0.f;
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
    const unsigned char* st = rg.buf + (size_t)s * NS * blk + (size_t)grp * rb;
    const uint4* xs = reinterpret_cast<const uint4*>(st);
    const uint4* ds = reinterpret_cast<const uint4*>(st + blk);
    const uint4* rs = reinterpret_cast<const uint4*>(st + 2 * blk);
    float2 dot2 = make_float2(0.f, 0.f), ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * G;
      const bool in = valid && v < p.nvec;
      const uint4 xv = in ? xs[v] : make_uint4(0, 0, 0, 0);
      const uint4 dv = in ? ds[v] : make_uint4(0, 0, 0, 0);
      bwd_vec_sums<E, !HAS_RSTD>(xv, dv, g[k], dot2, ss2);
    }
    const float dot = group_sum<G>(dot2.x + dot2.y);
    float r;
    if constexpr (HAS_RSTD) {
      r = r_saved;
    } else {
      const float ss = group_sum<G>(ss2.x + ss2.y);
      r = rsqrtf(fmaf(ss, p.inv_n, p.eps));
    }
    const float c = r * r * p.inv_n * dot;
    char* dxr = static_cast<char*>(p.dx) + row * rb;
    // the vectors are read again from the stage (not held in registers
    // across the reduction: that would cost resident CTAs)
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + k * G;
      const bool in = valid && v < p.nvec;
      const uint4 xv = in ? ld_shared_v4(xs + v) : make_uint4(0, 0, 0, 0);
      const uint4 dv = in ? ld_shared_v4(ds + v) : make_uint4(0, 0, 0, 0);
      const uint4 rv = (DRES && in) ? ld_shared_v4(rs + v) : make_uint4(0, 0, 0, 0);
      const uint4 o = bwd_vec_apply<E, DRES>(xv, dv, rv, g[k], r, c, acc[k]);
      if (in) st_stream(dxr + (size_t)v * 16, o);
    }
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
      float4* d = reinterpret_cast<float4*>(sacc + grp * ncol + v * E);
#pragma unroll
      for (int q = 0; q < E / 4; ++q)
        d[q] = make_float4(acc[k][4 * q], acc[k][4 * q + 1], acc[k][4 * q + 2],
                           acc[k][4 * q + 3]);
    }
  }
  __syncthreads();
  float* prow = p.partial + (size_t)blockIdx.x * p.ld_partial;
  for (int c = tid; c < ncol; c += kSubwarpThreads) {
    float t = 0.f;
    for (int q = 0; q < RPC; ++q) t += sacc[q * ncol + c];
    prow[c] = t;
  }
}

// ---------------------------------------------------------------------------
// kCta: one row per CTA iteration.  dgamma partials live in registers
// (ACC_SMEM false) or in shared memory (ACC_SMEM, for wide rows).  A column is
// updated by one thread per row and rows are separated by the reduction
// barrier, so the shared-memory accumulation is race free and adds rows in
// order.
template <typename TX, typename TW, int VPT, bool HAS_RSTD, bool ACC_SMEM, bool PF>
__global__ void __launch_bounds__(kCtaMaxThreads) bwd_cta_kernel(const BwdParams p) {
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int K = HAS_RSTD ? 1 : 2;
  extern __shared__ float4 smem4[];
  float* red = reinterpret_cast<float*>(smem4);                // 2 * K * 32
  float* sacc = red + 128;                                     // [ld]
  const int tid = threadIdx.x, T = blockDim.x;
  const bool want_dg = p.partial != nullptr;

  if constexpr (ACC_SMEM) {
    for (int j = tid; j < p.ld_partial; j += T) sacc[j] = 0.f;
    __syncthreads();
  }
  float acc[ACC_SMEM ? 1 : VPT][E];
#pragma unroll
  for (int k = 0; k < (ACC_SMEM ? 1 : VPT); ++k)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = 0.f;

  int parity = 0;
  BSlice<VPT> cur, nxt;
  int64_t row = blockIdx.x;
  if (row < p.M) bload_aligned<TX, VPT, HAS_RSTD>(cur, p, row, true, tid, T);
  for (; row < p.M; row += gridDim.x) {
    const int64_t nrow = row + gridDim.x;
    if (PF && nrow < p.M) bload_aligned<TX, VPT, HAS_RSTD>(nxt, p, nrow, true, tid, T);
    float sums[K];
#pragma unroll
    for (int q = 0; q < K; ++q) sums[q] = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      float xf[E], df[E], g[E];
      unpack(cur.x[k], xf);
      unpack(cur.dy[k], df);
      if (v < p.nvec) load_gamma_vec<TW, E>(p.gamma, v, g);
      else
#pragma unroll
        for (int e = 0; e < E; ++e) g[e] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sums[0] = fmaf(g[e] * df[e], xf[e], sums[0]);
        if (!HAS_RSTD) sums[K - 1] = fmaf(xf[e], xf[e], sums[K - 1]);
      }
    }
    cta_sum<K>(sums, red, parity);
    parity ^= 1;
    const float r = HAS_RSTD ? cur.r : rsqrtf(fmaf(sums[K - 1], p.inv_n, p.eps));
    const float c = r * r * p.inv_n * sums[0];

    char* dxrow = static_cast<char*>(p.dx) + row * (size_t)p.N * sizeof(TX);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < p.nvec) {
        float xf[E], df[E], g[E], o[E];
        unpack(cur.x[k], xf);
        unpack(cur.dy[k], df);
        load_gamma_vec<TW, E>(p.gamma, v, g);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = r * fmaf(-xf[e], c, g[e] * df[e]);
        st_stream(dxrow + (size_t)v * 16, pack(o));
        if constexpr (ACC_SMEM) {
          float* a = sacc + v * E;
#pragma unroll
          for (int e = 0; e < E; ++e) a[e] = fmaf(df[e] * xf[e], r, a[e]);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) acc[k][e] = fmaf(df[e] * xf[e], r, acc[k][e]);
        }
      }
    }
    if (PF) cur = nxt;
    else if (nrow < p.M) bload_aligned<TX, VPT, HAS_RSTD>(cur, p, nrow, true, tid, T);
  }
  if (!want_dg) return;
  float* prow = p.partial + (size_t)blockIdx.x * p.ld_partial;
  if constexpr (ACC_SMEM) {
    __syncthreads();
    for (int j = tid; j < p.N; j += T) prow[j] = sacc[j];
  } else {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < p.nvec) {
        float4* d = reinterpret_cast<float4*>(prow + v * E);
#pragma unroll
        for (int q = 0; q < E / 4; ++q)
          d[q] = make_float4(acc[k][4 * q], acc[k][4 * q + 1], acc[k][4 * q + 2],
                             acc[k][4 * q + 3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// kGeneric: any N, any element-aligned pointers.  Pass 1 reduces, pass 2
// writes dx; the partial row of this CTA is accumulated in place in global
// memory, each column always by the same thread.  Each thread issues U
// scalar loads per operand before using any (U requests in flight per warp).
template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
__global__ void __launch_bounds__(256) bwd_generic_kernel(const BwdParams p) {
  pdl_begin();
  constexpr int K = HAS_RSTD ? 1 : 2;
  constexpr int U = 4;
  __shared__ float red[2 * 2 * 32];
  const int tid = threadIdx.x, T = blockDim.x;
  const int N = p.N;
  const TW* gp = static_cast<const TW*>(p.gamma);
  float* prow = p.partial ? p.partial + (size_t)blockIdx.x * p.ld_partial : nullptr;
  if (prow)
    for (int j = tid; j < N; j += T) prow[j] = 0.f;
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const TX* xr = static_cast<const TX*>(p.x) + row * (int64_t)N;
    const TX* dr = static_cast<const TX*>(p.dy) + row * (int64_t)N;
    TX* dxr = static_cast<TX*>(p.dx) + row * (int64_t)N;
    float sums[K];
#pragma unroll
    for (int q = 0; q < K; ++q) sums[q] = 0.f;
    for (int j0 = tid; j0 < N; j0 += U * T) {
      float xv[U], dv[U], gv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        xv[u] = j < N ? ld_scalar(xr + j) : 0.f;
        dv[u] = j < N ? ld_scalar(dr + j) : 0.f;
        gv[u] = j < N ? ld_scalar(gp + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        sums[0] = fmaf(gv[u] * dv[u], xv[u], sums[0]);
        if (!HAS_RSTD) sums[K - 1] = fmaf(xv[u], xv[u], sums[K - 1]);
      }
    }
    cta_sum<K>(sums, red, parity);
    parity ^= 1;
    const float r = HAS_RSTD ? __ldg(p.rstd + row) : rsqrtf(fmaf(sums[K - 1], p.inv_n, p.eps));
    const float c = r * r * p.inv_n * sums[0];
    const TX* rr = static_cast<const TX*>(p.dres) + row * (int64_t)N;
    for (int j0 = tid; j0 < N; j0 += U * T) {
      float xv[U], dv[U], gv[U], rv[U], pv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        const bool in = j < N;
        xv[u] = in ? ld_scalar(xr + j) : 0.f;
        dv[u] = in ? ld_scalar(dr + j) : 0.f;
        gv[u] = in ? ld_scalar(gp + j) : 0.f;
        rv[u] = (DRES && in) ? ld_scalar(rr + j) : 0.f;
        pv[u] = (prow && in) ? prow[j] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * T;
        if (j >= N) continue;
        float o = r * fmaf(-xv[u], c, gv[u] * dv[u]);
        if (DRES) o += rv[u];
        st_scalar(dxr + j, o);
        if (prow) prow[j] = fmaf(dv[u] * xv[u], r, pv[u]);
      }
    }
  }
}

template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
BwdKernel pick_subwarp(int g, int vpt, bool pf) {
#define RMSN_SW(G_, V_)                                                         \
  if (g == G_ && vpt == V_) {                                                   \
    if constexpr (V_ >= 2 && V_ <= 3 && !DRES)                                  \
      return pf ? bwd_subwarp_kernel_2cta<TX, TW, G_, V_, HAS_RSTD, true, DRES>  \
                : bwd_subwarp_kernel_2cta<TX, TW, G_, V_, HAS_RSTD, false, DRES>; \
    else                                                                        \
      return pf ? bwd_subwarp_kernel<TX, TW, G_, V_, HAS_RSTD, true, DRES>       \
                : bwd_subwarp_kernel<TX, TW, G_, V_, HAS_RSTD, false, DRES>;     \
  }
  RMSN_SW(4, 1) RMSN_SW(8, 1) RMSN_SW(16, 1) RMSN_SW(32, 1)
  RMSN_SW(8, 2) RMSN_SW(16, 2) RMSN_SW(32, 2) RMSN_SW(32, 3) RMSN_SW(32, 4)
#undef RMSN_SW
  return nullptr;
}

template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
BwdKernel pick_rows_staged(int g, int vpt) {
#define RMSN_RS(G_, V_) \
  if (g == G_ && vpt == V_) return bwd_rows_staged_kernel<TX, TW, G_, V_, HAS_RSTD, DRES>;
  RMSN_RS(4, 1) RMSN_RS(8, 1) RMSN_RS(16, 1) RMSN_RS(32, 1)
  RMSN_RS(8, 2) RMSN_RS(16, 2) RMSN_RS(32, 2) RMSN_RS(32, 3) RMSN_RS(32, 4)
#undef RMSN_RS
  return nullptr;
}

template <typename TX, typename TW, bool HAS_RSTD, bool ACC_SMEM>
BwdKernel pick_cta(int vpt, bool pf) {
  switch (vpt) {
    case 1: return pf ? bwd_cta_kernel<TX, TW, 1, HAS_RSTD, ACC_SMEM, true>
                      : bwd_cta_kernel<TX, TW, 1, HAS_RSTD, ACC_SMEM, false>;
    case 2: return pf ? bwd_cta_kernel<TX, TW, 2, HAS_RSTD, ACC_SMEM, true>
                      : bwd_cta_kernel<TX, TW, 2, HAS_RSTD, ACC_SMEM, false>;
    case 4: return pf ? bwd_cta_kernel<TX, TW, 4, HAS_RSTD, ACC_SMEM, true>
                      : bwd_cta_kernel<TX, TW, 4, HAS_RSTD, ACC_SMEM, false>;
    case 8: return pf ? nullptr : bwd_cta_kernel<TX, TW, 8, HAS_RSTD, ACC_SMEM, false>;
    default: return nullptr;
  }
}

template <typename TX, typename TW, bool HAS_RSTD>
BwdKernel pick_family(const BwdKey& k) {
  if (k.family == kStaged && k.g > 0)   // short rows through the bulk-copy ring
    return k.dres ? pick_rows_staged<TX, TW, HAS_RSTD, true>(k.g, k.vpt)
                  : pick_rows_staged<TX, TW, HAS_RSTD, false>(k.g, k.vpt);
  if (k.dres) {   // fused-add backward: subwarp rows or the generic kernel
    switch (k.family) {
      case kSubwarp: return pick_subwarp<TX, TW, HAS_RSTD, true>(k.g, k.vpt, k.prefetch);
      case kGeneric: return bwd_generic_kernel<TX, TW, HAS_RSTD, true>;
      default: return nullptr;
    }
  }
  switch (k.family) {
    case kSubwarp: return pick_subwarp<TX, TW, HAS_RSTD, false>(k.g, k.vpt, k.prefetch);
    case kCta:
      return k.acc_smem ? pick_cta<TX, TW, HAS_RSTD, true>(k.vpt, k.prefetch)
                        : pick_cta<TX, TW, HAS_RSTD, false>(k.vpt, k.prefetch);
    case kGeneric: return bwd_generic_kernel<TX, TW, HAS_RSTD, false>;
    default: return nullptr;
  }
}

template <typename TX, typename TW>
BwdKernel pick_rstd(const BwdKey& k) {
  return k.has_rstd ? pick_family<TX, TW, true>(k) : pick_family<TX, TW, false>(k);
}


}  // namespace

#if RMSN_PAIR == 0
BwdKernel get_bwd_kernel_f32_f32(const BwdKey& k) { return pick_rstd<float, float>(k); }
#elif RMSN_PAIR == 1
BwdKernel get_bwd_kernel_bf16_bf16(const BwdKey& k) { return pick_rstd<bf16, bf16>(k); }
#else
BwdKernel get_bwd_kernel_bf16_f32(const BwdKey& k) { return pick_rstd<bf16, float>(k); }
#endif

}  // namespace rmsn
