// Bulk-copy staged RMSNorm kernels (forward, fused add, backward) for sm_103a.
//
// Same arithmetic as the register-resident one-row-per-CTA kernels (see
// rmsnorm_fwd.cu / rmsnorm_bwd.cu for the formulas and their sources), but the
// rows of the streamed operands (x; r and x; x and dy) arrive through
// `cp.async.bulk` copies into a ring of `stages` shared-memory row buffers,
// each tracked by an mbarrier.  One thread keeps the ring `stages` rows ahead
// of the CTA, so the number of bytes in flight per SM is set by the ring, not
// by how many registers the row math needs -- the GB300 way to stream rows,
// where the pages' LDS-cached design ("Pre-built kernel library guide",
// section 1.2, pass 0: global -> LDS row cache) loads the row with the threads
// themselves.
//
// Pipeline of CTA row i (stage s = i mod stages):
//   wait(full[s])  ->  read own vectors from stage s  ->  CTA reduction
//   (its barrier also proves every thread is done with stage s)  ->  thread 0
//   refills stage s with row i + stages  ->  outputs from registers.
// Every wait is bounded by p.wait_limit clock cycles.  Whether any thread's
// wait ran out is voted on at the reduction barrier (__syncthreads_or), so the
// whole CTA agrees: it stores nothing for that row and leaves; thread 0 first
// waits (bounded) for the copies it has in flight, then raises
// kStatusWaitTimeout in p.status.
//
// Stage 2 of every backward (the fixed-order column sum of the weight
// gradients' partial rows, colsum_kernel) is built here too, once (RMSN_PAIR 0).
#include "rmsnorm_ring.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif

namespace rmsn {
namespace {

// ---------------------------------------------------------------------------
// Forward / fused add.  Stage layout: fused [r | x], forward [x].
template <typename TX, typename TW, int VPT, bool FUSED>
__global__ void __launch_bounds__(kCtaMaxThreads) fwd_staged_kernel(const FwdParams p) {
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int NS = FUSED ? 2 : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  const Ring rg = ring_of(smem);
  const int tid = threadIdx.x, T = blockDim.x, S = p.stages;
  const size_t rb = (size_t)p.N * sizeof(TX);
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nrows = first < p.M ? (p.M - 1 - first) / stride + 1 : 0;
  const char* xs = static_cast<const char*>(p.x);
  const char* rs_src = static_cast<const char*>(p.residual);
  int64_t issued =
      ring_start<NS>(rg, S, nrows, first, stride, FUSED ? rs_src : xs, xs, nullptr, rb);

  float g[VPT][E];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    if (v < p.nvec) gamma_f32<TW, E>(p.gamma, v, g[k]);
    else
#pragma unroll
      for (int e = 0; e < E; ++e) g[k][e] = 0.f;
  }

  int parity = 0;
  int64_t i = 0;
  bool failed = false;
  for (; i < nrows; ++i) {
    const int s = (int)(i % S);
    const int64_t row = first + i * stride;
    const bool late = !mbar_wait_bounded(rg.full + s, (uint32_t)((i / S) & 1), p.wait_limit);
    const uint4* st = reinterpret_cast<const uint4*>(rg.buf + (size_t)s * NS * rb);
    uint4 hv[VPT];
    float ss[1] = {0.f};
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      hv[k] = make_uint4(0, 0, 0, 0);
      if (v < p.nvec) {
        float f[E];
        if constexpr (FUSED) {
          float rf[E];
          unpack(st[v], rf);
          unpack(st[p.nvec + v], f);
#pragma unroll
          for (int e = 0; e < E; ++e) f[e] += rf[e];
          hv[k] = pack(f);      // h rounded to the activation dtype
          unpack(hv[k], f);
        } else {
          hv[k] = st[v];
          unpack(hv[k], f);
        }
#pragma unroll
        for (int e = 0; e < E; ++e) ss[0] = fmaf(f[e], f[e], ss[0]);
      }
    }
    if (cta_sum_vote<1>(ss, rg.red, parity, late)) {
      failed = true;
      break;
    }
    parity ^= 1;
    if (tid == 0 && issued < nrows) {
      fence_proxy_async_smem();
      issue_row<NS>(rg, issued, first, stride, S, FUSED ? rs_src : xs, xs, nullptr, rb);
      ++issued;
    }
    const float rs = rsqrtf(fmaf(ss[0], p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    char* yrow = static_cast<char*>(p.y) + row * rb;
    char* hrow = static_cast<char*>(p.residual) + row * rb;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < p.nvec) {
        if (FUSED) st_stream(hrow + (size_t)v * 16, hv[k]);
        float o[E];
        unpack(hv[k], o);
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = o[e] * rs * g[k][e];
        st_stream(yrow + (size_t)v * 16, pack(o));
      }
    }
  }
  if (failed && tid == 0) {
    drain(rg, i, issued, S);
    atomicOr(p.status, kStatusWaitTimeout);
  }
}

// ---------------------------------------------------------------------------
// Backward.  Stage layout [x | dy] (fused-add backward: [h | dy | dres]);
// dgamma partials of this CTA's rows in registers, written as one partial row
// at the end.  The fused-add backward reads dres from the stage in its output
// pass, so it refills the stage after that pass instead of right after the
// reduction.  MIX: x (h) and dy may start off dx's 16-byte alignment (dx,
// dres and gamma on 16 bytes, rows a multiple of 16 bytes): each shifted row
// arrives as its enclosing aligned span and its vectors are realigned from
// shared memory (slot_vec).
template <typename TX, typename TW, int VPT, bool HAS_RSTD, bool DRES, bool MIX>
__global__ void __launch_bounds__(kCtaMaxThreads) bwd_staged_kernel(const BwdParams p) {
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int K = HAS_RSTD ? 1 : 2;
  constexpr int NS = DRES ? 3 : 2;
  pdl_begin();
  extern __shared__ __align__(128) unsigned char smem[];
  const Ring rg = ring_of(smem);
  const int tid = threadIdx.x, T = blockDim.x, S = p.stages;
  const size_t rb = (size_t)p.N * sizeof(TX);
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nrows = first < p.M ? (p.M - 1 - first) / stride + 1 : 0;
  const char* xs = static_cast<const char*>(p.x);
  const char* ds = static_cast<const char*>(p.dy);
  const char* rs = static_cast<const char*>(p.dres);
  const int sx = MIX ? p.x_shift : 0, sd = MIX ? p.dy_shift : 0;
  const RowSpans sp{rb, MIX ? rb + 16 : rb, {sx, sd, 0}};
  int64_t issued = ring_start<NS>(rg, S, nrows, first, stride, xs, ds, rs, sp);

  float g[VPT][E], acc[VPT][E];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    if (v < p.nvec) gamma_f32<TW, E>(p.gamma, v, g[k]);
    else
#pragma unroll
      for (int e = 0; e < E; ++e) g[k][e] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = 0.f;
  }

  int parity = 0;
  int64_t i = 0;
  bool failed = false;
  for (; i < nrows; ++i) {
    const int s = (int)(i % S);
    const int64_t row = first + i * stride;
    const float r_saved = HAS_RSTD ? __ldg(p.rstd + row) : 0.f;
    const bool late = !mbar_wait_bounded(rg.full + s, (uint32_t)((i / S) & 1), p.wait_limit);
    const unsigned char* st = rg.buf + (size_t)s * NS * sp.slot;
    uint4 xv[VPT], dv[VPT];
    float sums[K];
#pragma unroll
    for (int q = 0; q < K; ++q) sums[q] = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      xv[k] = make_uint4(0, 0, 0, 0);
      dv[k] = make_uint4(0, 0, 0, 0);
      if (v < p.nvec) {
        xv[k] = slot_vec(st, v, sx);
        dv[k] = slot_vec(st + sp.slot, v, sd);
        float xf[E], df[E];
        unpack(xv[k], xf);
        unpack(dv[k], df);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          sums[0] = fmaf(g[k][e] * df[e], xf[e], sums[0]);
          if (!HAS_RSTD) sums[K - 1] = fmaf(xf[e], xf[e], sums[K - 1]);
        }
      }
    }
    if (cta_sum_vote<K>(sums, rg.red, parity, late)) {
      failed = true;
      break;
    }
    parity ^= 1;
    if (!DRES && tid == 0 && issued < nrows) {
      fence_proxy_async_smem();
      issue_row<NS>(rg, issued, first, stride, S, xs, ds, rs, sp);
      ++issued;
    }
    const float r = HAS_RSTD ? r_saved : rsqrtf(fmaf(sums[K - 1], p.inv_n, p.eps));
    const float c = r * r * p.inv_n * sums[0];
    char* dxrow = static_cast<char*>(p.dx) + row * rb;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < p.nvec) {
        float xf[E], df[E], o[E], rf[E];
        unpack(xv[k], xf);
        unpack(dv[k], df);
        if (DRES) unpack(reinterpret_cast<const uint4*>(st + 2 * sp.slot)[v], rf);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          o[e] = r * fmaf(-xf[e], c, g[k][e] * df[e]);
          if (DRES) o[e] += rf[e];
          acc[k][e] = fmaf(df[e] * xf[e], r, acc[k][e]);
        }
        st_stream(dxrow + (size_t)v * 16, pack(o));
      }
    }
    if (DRES) {
      // every thread has read this stage: refill it (the barrier orders the
      // reads before thread 0's bulk copy)
      __syncthreads();
      if (tid == 0 && issued < nrows) {
        fence_proxy_async_smem();
        issue_row<NS>(rg, issued, first, stride, S, xs, ds, rs, sp);
        ++issued;
      }
    }
  }
  if (failed) {
    if (tid == 0) {
      drain(rg, i, issued, S);
      atomicOr(p.status, kStatusWaitTimeout);
    }
    return;
  }
  if (p.partial == nullptr) return;
  float* prow = p.partial + (size_t)blockIdx.x * p.ld_partial;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    if (v < p.nvec) {
      float4* d = reinterpret_cast<float4*>(prow + v * E);
#pragma unroll
      for (int q = 0; q < E / 4; ++q)
        d[q] = make_float4(acc[k][4 * q], acc[k][4 * q + 1], acc[k][4 * q + 2], acc[k][4 * q + 3]);
    }
  }
}

template <typename TX, typename TW, bool FUSED>
FwdKernel pick_fwd(int vpt) {
  switch (vpt) {
    case 1: return fwd_staged_kernel<TX, TW, 1, FUSED>;
    case 2: return fwd_staged_kernel<TX, TW, 2, FUSED>;
    case 4: return fwd_staged_kernel<TX, TW, 4, FUSED>;
    case 8: return fwd_staged_kernel<TX, TW, 8, FUSED>;
    default: return nullptr;
  }
}

template <typename TX, typename TW, bool HAS_RSTD, bool DRES, bool MIX>
BwdKernel pick_bwd(int vpt) {
  switch (vpt) {
    case 1: return bwd_staged_kernel<TX, TW, 1, HAS_RSTD, DRES, MIX>;
    case 2: return bwd_staged_kernel<TX, TW, 2, HAS_RSTD, DRES, MIX>;
    case 4: return bwd_staged_kernel<TX, TW, 4, HAS_RSTD, DRES, MIX>;
    default: return nullptr;
  }
}
template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
BwdKernel pick_bwd(int vpt, bool mix) {
  return mix ? pick_bwd<TX, TW, HAS_RSTD, DRES, true>(vpt)
             : pick_bwd<TX, TW, HAS_RSTD, DRES, false>(vpt);
}

template <typename TX, typename TW>
FwdKernel staged_fwd(const FwdKey& k) {
  return k.fused ? pick_fwd<TX, TW, true>(k.vpt) : pick_fwd<TX, TW, false>(k.vpt);
}
template <typename TX, typename TW>
BwdKernel staged_bwd(const BwdKey& k) {
  if (k.dres)
    return k.has_rstd ? pick_bwd<TX, TW, true, true>(k.vpt, k.mix)
                      : pick_bwd<TX, TW, false, true>(k.vpt, k.mix);
  return k.has_rstd ? pick_bwd<TX, TW, true, false>(k.vpt, k.mix)
                    : pick_bwd<TX, TW, false, false>(k.vpt, k.mix);
}

#if RMSN_PAIR == 0
// Stage 2 of every backward: out_j = sum_b partial[b][j] over the P stage-1
// CTAs, in a fixed order, fp32 (or rounded once to bf16).  A CTA owns C
// float4 columns; its R = 256 / C row lanes each add the rows b = lane,
// lane + R, ... in sequence (loads issued sixteen ahead; the order of the
// adds does not change), then the R lane sums meet in a fixed binary tree in
// shared memory.  Launched as a programmatic dependent of stage 1:
// griddepcontrol.wait returns once stage 1 has completed and its writes are
// visible.
__device__ __forceinline__ void add4(float4& s, const float4& v) {
  s.x += v.x;
  s.y += v.y;
  s.z += v.z;
  s.w += v.w;
}

template <int C>
__global__ void __launch_bounds__(kColSumThreads)
    colsum_kernel(const float* partial, int P, int nq, ColSumOut o) {
  pdl_begin();
  constexpr int R = kColSumThreads / C;
  __shared__ float4 sh[R][C];
  const int tx = threadIdx.x % C, ty = threadIdx.x / C;
  const int q = blockIdx.x * C + tx;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (q < nq) {
    const float4* src = reinterpret_cast<const float4*>(partial) + q;
    // up to B rows per lane in flight at once (one round trip for P <= B R),
    // added in row order
    constexpr int B = 16;
    for (int b = ty; b < P; b += B * R) {
      float4 v[B];
#pragma unroll
      for (int u = 0; u < B; ++u)
        if (b + u * R < P) v[u] = __ldcs(src + (size_t)(b + u * R) * nq);
#pragma unroll
      for (int u = 0; u < B; ++u)
        if (b + u * R < P) add4(s, v[u]);
    }
  }
  sh[ty][tx] = s;
  __syncthreads();
#pragma unroll
  for (int h = R / 2; h > 0; h >>= 1) {
    if (ty < h) {
      float4 t = sh[ty][tx];
      add4(t, sh[ty + h][tx]);
      sh[ty][tx] = t;
    }
    __syncthreads();
  }
  if (ty == 0 && q < nq) {
    const float4 t = sh[0][tx];
    const bool second = q >= o.half_q;
    const int j = (second ? q - o.half_q : q) * 4;
    void* out = second ? o.out1 : o.out0;
    if (out == nullptr) return;
    const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (j + u < o.N) {
        if (o.bf16 && !second) static_cast<bf16*>(out)[j + u] = __float2bfloat16_rn(tv[u]);
        else static_cast<float*>(out)[j + u] = tv[u];
      }
    }
  }
}
#endif

}  // namespace

#if RMSN_PAIR == 0
ColSumKernel get_colsum_kernel(int c) {
  switch (c) {
    case 8: return colsum_kernel<8>;
    case 16: return colsum_kernel<16>;
    case 32: return colsum_kernel<32>;
    default: return nullptr;
  }
}
FwdKernel get_fwd_staged_f32_f32(const FwdKey& k) { return staged_fwd<float, float>(k); }
BwdKernel get_bwd_staged_f32_f32(const BwdKey& k) { return staged_bwd<float, float>(k); }
#elif RMSN_PAIR == 1
FwdKernel get_fwd_staged_bf16_bf16(const FwdKey& k) { return staged_fwd<bf16, bf16>(k); }
BwdKernel get_bwd_staged_bf16_bf16(const BwdKey& k) { return staged_bwd<bf16, bf16>(k); }
#else
FwdKernel get_fwd_staged_bf16_f32(const FwdKey& k) { return staged_fwd<bf16, float>(k); }
BwdKernel get_bwd_staged_bf16_f32(const BwdKey& k) { return staged_bwd<bf16, float>(k); }
#endif

}  // namespace rmsn
