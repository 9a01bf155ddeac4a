// RMSNorm forward, fused add, backward and fused-add backward for rows too
// long for one CTA, on thread-block clusters (sm_103a).
//
// Arithmetic as in rmsnorm_fwd.cu / rmsnorm_bwd.cu.  One row is handled by a
// cluster of C = 2, 4 or 8 CTAs: CTA rank r owns the contiguous slice of
// vectors [r * slice, (r + 1) * slice) of every row of the cluster's walk, so
// every element is still read once from HBM with 16-byte accesses and kept on
// chip until its output is written -- the register-resident path of the
// "Pre-built kernel library guide" (section 1.1) and the LDS row cache of its
// section 1.2 carried past the size of one CTA.  Where that guide combines
// the per-wave partial sums of a row inside one workgroup, a cluster combines
// the per-CTA sums through distributed shared memory: thread 0 of each CTA
// pushes its CTA's sum into a slot of every CTA of the cluster with st.async,
// each push completing on the receiving CTA's mbarrier, and every thread adds
// the C slots in rank order -- so every CTA obtains the same, fixed-order
// total without a cluster-wide barrier per row (a release at a cluster
// barrier would wait for every thread's outstanding global stores).
//
//   forward / fused add : the slice in registers, the next row's slice loaded
//                         before the current row is reduced (as kCta)
//   backward            : the slices of x and dy (and dres) through a ring of
//                         bulk copies (as kStaged); dgamma partials in
//                         registers, one partial row per cluster, each CTA
//                         writing its slice's columns
//
// The cluster meets at a hardware cluster barrier twice: once after the
// exchange barriers are initialised (no push may reach an uninitialised
// barrier) and once before leaving (no CTA's shared memory may disappear
// while a peer still pushes into it).  Every exchange wait is bounded; the
// bounded bulk-copy waits of the backward travel with the sums as a vote, so
// all CTAs of a cluster stop at the same row.
#include "rmsnorm_bwd_common.cuh"
#include "rmsnorm_fwd_common.cuh"
#include "rmsnorm_ring.cuh"

#ifndef RMSN_PAIR
#error "compile once per dtype pair with -DRMSN_PAIR=0 (f32/f32), 1 (bf16/bf16), 2 (bf16/f32)"
#endif

namespace rmsn {
namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives (release: its earlier
// shared-memory writes become visible to the cluster) and waits (acquire).
// Used twice per kernel: after the exchange barriers are initialised, and
// before leaving.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The shared::cluster address of `local` (this CTA's shared memory) in the
// CTA of `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(local)), "r"(rank));
  return a;
}
// Asynchronous 16-byte store into a peer's shared memory, counted as 16
// bytes of completed transactions on the peer's mbarrier.
__device__ __forceinline__ void st_async_peer(uint32_t addr, const float4& v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}

// Per-row exchange of one float4 per CTA across the cluster, without a
// cluster barrier: warp 0 pushes this CTA's value into slot[rank] of every
// CTA (itself included) with st.async, each push completing on the receiving
// CTA's mbarrier for this row's parity, which that CTA's thread 0 arms for C
// pushes (a push may land before the arming: the barrier's transaction count
// then runs below zero until it is armed).  Every thread waits (bounded) on its own barrier and adds the C
// slots in rank order, so all CTAs obtain the same total.  Slots and barriers
// alternate between rows: a CTA's slots of parity p are rewritten only by
// pushes for the row after next, which its peers send only after they have
// received this CTA's push for the next row -- sent after a CTA barrier that
// follows this CTA's last read of those slots.
struct Xchg {
  uint64_t* bar;   // [2]
  float4* slot;    // [2][8]
};

// Thread 0 initialises both barriers; the cluster then meets once, so that
// no push reaches a barrier before it is initialised.
__device__ __forceinline__ void xchg_init(const Xchg& x) {
  if (threadIdx.x == 0) {
    mbar_init(x.bar, 1);
    mbar_init(x.bar + 1, 1);
    mbar_init_fence();
  }
  cluster_sync();
}

// Exchange of row `it` of this CTA's walk; false if the wait gave up.  Lane r
// (< C) of warp 0 pushes v, which must be the same in all those lanes, to the
// CTA of rank r; out[k] receives the sum of component k (k < K).
template <int K>
__device__ __forceinline__ bool xchg_sum(const Xchg& x, const float4& v, int64_t it, uint32_t C,
                                         uint32_t rank, long long limit, float (&out)[K]) {
  const int p = (int)(it & 1);
  if (threadIdx.x < C) {
    if (threadIdx.x == 0) mbar_arrive_expect_tx(x.bar + p, C * 16u);
    // earlier generic reads of the slots (ordered before this by the CTA's
    // reduction barrier) come before the peers' asynchronous writes
    fence_proxy_async_smem();
    st_async_peer(peer_addr(x.slot + p * 8 + rank, threadIdx.x), v,
                  peer_addr(x.bar + p, threadIdx.x));
  }
  const bool ok = mbar_wait_bounded(x.bar + p, (uint32_t)((it >> 1) & 1), limit);
  const float* sl = reinterpret_cast<const float*>(x.slot + p * 8);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    float s = 0.f;
    for (uint32_t r = 0; r < C; ++r) s += sl[r * 4 + k];
    out[k] = s;
  }
  return ok;
}

// Vectors [v0, v0 + nv) of a row are this CTA's slice.
struct SliceOf {
  int v0, nv;
};
__device__ __forceinline__ SliceOf slice_of(int slice, int nvec, uint32_t rank) {
  const int v0 = (int)rank * slice;
  int nv = nvec - v0;
  nv = nv < 0 ? 0 : (nv > slice ? slice : nv);
  return SliceOf{v0, nv};
}

// ---------------------------------------------------------------------------
// Forward / fused add: the slice in registers, next-row prefetch (PF).
template <typename TX, typename TW, int VPT, bool FUSED, bool PF>
__global__ void __launch_bounds__(kCtaMaxThreads) fwd_cluster_kernel(const FwdParams p0) {
  if (threadIdx.x == 0) {   // this CTA's slice of its first two rows into L2 before the wait
    const uint32_t C0 = cluster_ctas();
    const SliceOf s0 = slice_of(p0.slice, p0.nvec, cluster_rank());
    const size_t rb0 = (size_t)p0.N * sizeof(TX), o0 = (size_t)s0.v0 * 16;
    const int64_t r0 = blockIdx.x / C0, st0 = gridDim.x / C0;
    for (int k = 0; k < 2 && s0.nv > 0; ++k) {
      const int64_t row = r0 + k * st0;
      if (row >= p0.M) break;
      bulk_prefetch_l2(static_cast<const char*>(p0.x) + row * rb0 + o0, (uint32_t)s0.nv * 16);
      if (FUSED)
        bulk_prefetch_l2(static_cast<const char*>(p0.residual) + row * rb0 + o0,
                         (uint32_t)s0.nv * 16);
    }
  }
  pdl_begin();
  using Cf = Cfg<TX, TW>;
  constexpr int E = Cf::E, GW = Cf::GW;
  __shared__ float red[2 * 32];
  __shared__ __align__(16) float4 slots[2 * 8];
  __shared__ __align__(8) uint64_t bars[2];
  const uint32_t C = cluster_ctas(), rank = cluster_rank();
  const Xchg xc{bars, slots};
  xchg_init(xc);
  const int tid = threadIdx.x, T = blockDim.x;
  const SliceOf sl = slice_of(p0.slice, p0.nvec, rank);
  // the parameters of this CTA's slice: operands shifted to its first vector
  FwdParams p = p0;
  const size_t off = (size_t)sl.v0 * 16;
  p.x = static_cast<const char*>(p0.x) + off;
  p.y = static_cast<char*>(p0.y) + off;
  if (FUSED) p.residual = static_cast<char*>(p0.residual) + off;
  p.nvec = sl.nv;
  const char* gp = static_cast<const char*>(p0.gamma) + (size_t)sl.v0 * GW * 16;

  uint4 gw[VPT][GW];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
#pragma unroll
    for (int w = 0; w < GW; ++w)
      gw[k][w] = v < sl.nv ? ld_cached(gp + ((size_t)v * GW + w) * 16) : make_uint4(0, 0, 0, 0);
  }

  const int64_t first = blockIdx.x / C, stride = gridDim.x / C;
  const size_t rb = (size_t)p.N * sizeof(TX);
  int parity = 0;
  bool failed = false;
  Slice<VPT, FUSED> cur, nxt;
  if (first < p.M) load_aligned<TX, VPT, FUSED>(cur, p, first, true, tid, T);
  int64_t it = 0;
  for (int64_t row = first; row < p.M; row += stride, ++it) {
    const int64_t nrow = row + stride;
    if (PF && nrow < p.M) load_aligned<TX, VPT, FUSED>(nxt, p, nrow, true, tid, T);
    // with the next row's slice in registers, the slice of the row l2_rows
    // steps ahead is requested into L2 (no registers held for it)
    if (PF && p.l2_rows > 0 && tid == 0 && sl.nv > 0) {
      const int64_t ahead = row + (int64_t)p.l2_rows * stride;
      if (ahead < p.M) {
        bulk_prefetch_l2(static_cast<const char*>(p.x) + ahead * rb, (uint32_t)sl.nv * 16);
        if (FUSED)
          bulk_prefetch_l2(static_cast<const char*>(p.residual) + ahead * rb, (uint32_t)sl.nv * 16);
      }
    }
    char* yrow = static_cast<char*>(p.y) + row * rb;
    char* hrow = static_cast<char*>(p.residual) + row * rb;
    float ss[1];
    ss[0] = slice_sumsq<TX, VPT, FUSED>(cur, hrow, tid, T, sl.nv, true);
    cta_sum<1>(ss, red, parity);
    parity ^= 1;
    if (!xchg_sum<1>(xc, make_float4(ss[0], 0.f, 0.f, 0.f), it, C, rank, p.wait_limit, ss)) {
      failed = true;   // a peer stopped answering: leave (it cannot happen while peers run)
      break;
    }
    const float rs = rsqrtf(fmaf(ss[0], p.inv_n, p.eps));
    if (rank == 0 && tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < sl.nv) st_stream(yrow + (size_t)v * 16, scale_vec<TX, TW>(cur.x[k], gw[k], rs));
    }
    if (PF) cur = nxt;
    else if (nrow < p.M) load_aligned<TX, VPT, FUSED>(cur, p, nrow, true, tid, T);
  }
  if (failed && tid == 0) atomicOr(p.status, kStatusWaitTimeout);
  cluster_sync();
}

// ---------------------------------------------------------------------------
// Backward (fused-add backward: DRES).  Stage layout [x | dy] ([h | dy | dres])
// of this CTA's slice of the row; the slice's dgamma partials in registers.
template <int NS>
__device__ __forceinline__ void issue_slice(const Ring& rg, int64_t i, int64_t first,
                                            int64_t stride, int S, const char* src0,
                                            const char* src1, const char* src2, size_t rb,
                                            uint32_t sb) {
  const int s = (int)(i % S);
  const int64_t row = first + i * stride;
  uint64_t* bar = rg.full + s;
  unsigned char* dst = rg.buf + (size_t)s * NS * sb;
  mbar_arrive_expect_tx(bar, NS * sb);
  if (sb == 0) return;
  bulk_copy_g2s(dst, src0 + row * rb, sb, bar);
  if (NS > 1) bulk_copy_g2s(dst + sb, src1 + row * rb, sb, bar);
  if (NS > 2) bulk_copy_g2s(dst + 2 * sb, src2 + row * rb, sb, bar);
}

template <typename TX, typename TW, int VPT, bool HAS_RSTD, bool DRES>
__global__ void __launch_bounds__(kCtaMaxThreads) bwd_cluster_kernel(const BwdParams p) {
  pdl_begin();
  constexpr int E = Elem<TX>::kPerVec;
  constexpr int K = HAS_RSTD ? 1 : 2;
  constexpr int NS = DRES ? 3 : 2;
  extern __shared__ __align__(128) unsigned char smem[];
  const Ring rg = ring_of(smem);
  // exchange barriers and slots in the header, after the ring's barriers and
  // reduction slots
  const Xchg xc{reinterpret_cast<uint64_t*>(smem + 640), reinterpret_cast<float4*>(smem + 768)};
  const uint32_t C = cluster_ctas(), rank = cluster_rank();
  const int tid = threadIdx.x, T = blockDim.x, S = p.stages;
  const SliceOf sl = slice_of(p.slice, p.nvec, rank);
  const size_t rb = (size_t)p.N * sizeof(TX);
  const uint32_t sb = (uint32_t)sl.nv * 16;
  const size_t off = (size_t)sl.v0 * 16;
  const int64_t first = blockIdx.x / C, stride = gridDim.x / C;
  const int64_t nrows = first < p.M ? (p.M - 1 - first) / stride + 1 : 0;
  const char* xs = static_cast<const char*>(p.x) + off;
  const char* ds = static_cast<const char*>(p.dy) + off;
  const char* rs = DRES ? static_cast<const char*>(p.dres) + off : nullptr;
  char* dxs = static_cast<char*>(p.dx) + off;

  int64_t issued = 0;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(rg.full + s, 1);
    mbar_init_fence();
  }
  xchg_init(xc);   // also orders the ring's barrier initialisation before use
  if (tid == 0) {
    const int64_t n0 = nrows < S ? nrows : S;
    for (; issued < n0; ++issued) issue_slice<NS>(rg, issued, first, stride, S, xs, ds, rs, rb, sb);
  }

  float g[VPT][E], acc[VPT][E];
  const char* gbase = static_cast<const char*>(p.gamma) + (size_t)sl.v0 * E * sizeof(TW);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    if (v < sl.nv) gamma_f32<TW, E>(gbase, v, g[k]);
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
    const uint4* st = reinterpret_cast<const uint4*>(rg.buf + (size_t)s * NS * sb);
    float2 dot2 = make_float2(0.f, 0.f), ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      const uint4 xv = v < sl.nv ? st[v] : make_uint4(0, 0, 0, 0);
      const uint4 dv = v < sl.nv ? st[sl.nv + v] : make_uint4(0, 0, 0, 0);
      bwd_vec_sums<E, !HAS_RSTD>(xv, dv, g[k], dot2, ss2);
    }
    float sums[K];
    sums[0] = dot2.x + dot2.y;
    if (K > 1) sums[K - 1] = ss2.x + ss2.y;
    // the CTA's sums and its vote, then the cluster's: every CTA of the
    // cluster sees the same sums and the same outcome of the waits
    const bool any_late = cta_sum_vote<K>(sums, rg.red, parity, late);
    parity ^= 1;
    float tot[3];
    const bool answered = xchg_sum<3>(xc, make_float4(sums[0], K > 1 ? sums[K - 1] : 0.f,
                                                      any_late ? 1.f : 0.f, 0.f),
                                      i, C, rank, p.wait_limit, tot);
    if (!answered || tot[2] != 0.f) {
      failed = true;
      break;
    }
    sums[0] = tot[0];
    if (K > 1) sums[K - 1] = tot[1];
    const float r = HAS_RSTD ? r_saved : rsqrtf(fmaf(sums[K - 1], p.inv_n, p.eps));
    const float c = r * r * p.inv_n * sums[0];
    char* dxrow = dxs + row * rb;
    // the vectors are read again from the stage rather than held across the
    // exchange (registers are what limits this kernel to one CTA per SM)
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * T;
      if (v < sl.nv) {
        const uint4 xv = ld_shared_v4(st + v), dv = ld_shared_v4(st + sl.nv + v);
        const uint4 rv = DRES ? ld_shared_v4(st + 2 * sl.nv + v) : make_uint4(0, 0, 0, 0);
        st_stream(dxrow + (size_t)v * 16, bwd_vec_apply<E, DRES>(xv, dv, rv, g[k], r, c, acc[k]));
      }
    }
    // every thread has read this stage (the output pass reads it again):
    // refill it
    __syncthreads();
    if (tid == 0 && issued < nrows) {
      fence_proxy_async_smem();
      issue_slice<NS>(rg, issued, first, stride, S, xs, ds, rs, rb, sb);
      ++issued;
    }
  }
  if (failed && tid == 0) {
    // every CTA of the cluster stops at the same row: wait (bounded) for the
    // copies still in flight, then report
    for (int64_t j = i; j < issued; ++j)
      mbar_wait_bounded(rg.full + (j % S), (uint32_t)((j / S) & 1), kDrainLimit);
    atomicOr(p.status, kStatusWaitTimeout);
  }
  cluster_sync();
  if (failed || p.partial == nullptr) return;
  float* prow = p.partial + (size_t)first * p.ld_partial + (size_t)sl.v0 * E;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * T;
    if (v < sl.nv) {
      float4* d = reinterpret_cast<float4*>(prow + v * E);
#pragma unroll
      for (int q = 0; q < E / 4; ++q)
        d[q] = make_float4(acc[k][4 * q], acc[k][4 * q + 1], acc[k][4 * q + 2], acc[k][4 * q + 3]);
    }
  }
}

template <typename TX, typename TW, bool FUSED>
FwdKernel pick_fwd(int vpt, bool pf) {
  switch (vpt) {
    case 2: return pf ? fwd_cluster_kernel<TX, TW, 2, FUSED, true>
                      : fwd_cluster_kernel<TX, TW, 2, FUSED, false>;
    case 4: return pf ? fwd_cluster_kernel<TX, TW, 4, FUSED, true>
                      : fwd_cluster_kernel<TX, TW, 4, FUSED, false>;
    case 8: return pf ? nullptr : fwd_cluster_kernel<TX, TW, 8, FUSED, false>;
    default: return nullptr;
  }
}

template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
BwdKernel pick_bwd(int vpt) {
  switch (vpt) {
    case 2: return bwd_cluster_kernel<TX, TW, 2, HAS_RSTD, DRES>;
    case 4: return bwd_cluster_kernel<TX, TW, 4, HAS_RSTD, DRES>;
    default: return nullptr;
  }
}

template <typename TX, typename TW>
FwdKernel cluster_fwd(const FwdKey& k) {
  if (k.family != kCluster || k.strided || k.out != kOutDtype) return nullptr;
  return k.fused ? pick_fwd<TX, TW, true>(k.vpt, k.prefetch)
                 : pick_fwd<TX, TW, false>(k.vpt, k.prefetch);
}
template <typename TX, typename TW>
BwdKernel cluster_bwd(const BwdKey& k) {
  if (k.family != kCluster) return nullptr;
  if (k.dres)
    return k.has_rstd ? pick_bwd<TX, TW, true, true>(k.vpt) : pick_bwd<TX, TW, false, true>(k.vpt);
  return k.has_rstd ? pick_bwd<TX, TW, true, false>(k.vpt) : pick_bwd<TX, TW, false, false>(k.vpt);
}

}  // namespace

#if RMSN_PAIR == 0
FwdKernel get_fwd_cluster_f32_f32(const FwdKey& k) { return cluster_fwd<float, float>(k); }
BwdKernel get_bwd_cluster_f32_f32(const BwdKey& k) { return cluster_bwd<float, float>(k); }
#elif RMSN_PAIR == 1
FwdKernel get_fwd_cluster_bf16_bf16(const FwdKey& k) { return cluster_fwd<bf16, bf16>(k); }
BwdKernel get_bwd_cluster_bf16_bf16(const BwdKey& k) { return cluster_bwd<bf16, bf16>(k); }
#else
FwdKernel get_fwd_cluster_bf16_f32(const FwdKey& k) { return cluster_fwd<bf16, float>(k); }
BwdKernel get_bwd_cluster_bf16_f32(const BwdKey& k) { return cluster_bwd<bf16, float>(k); }
#endif

}  // namespace rmsn
