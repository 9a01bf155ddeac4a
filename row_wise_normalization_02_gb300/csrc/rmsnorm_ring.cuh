// The shared-memory row ring of the staged kernels: rows of up to three
// streamed operands arrive by 1-D bulk copies (cp.async.bulk, the non-tensor
// form of TMA) into `stages` row buffers, each tracked by an mbarrier that
// thread 0 arms with the expected byte count.  Used by the staged forward,
// fused-add and backward kernels and by the staged quantised forward.
#pragma once

#include <type_traits>

#include "rmsnorm_device.cuh"
#include "rmsnorm_internal.h"

namespace rmsn {
namespace {

constexpr long long kDrainLimit = 1LL << 34;   // cycles: several seconds

struct Ring {
  uint64_t* full;       // kStagedMaxStages barriers
  float* red;           // 2 x 2 x 32 reduction slots
  unsigned char* buf;   // stages x NS x row bytes
};

__device__ __forceinline__ Ring ring_of(unsigned char* smem) {
  Ring r;
  r.full = reinterpret_cast<uint64_t*>(smem);
  r.red = reinterpret_cast<float*>(smem + 128);
  r.buf = smem + kStagedHeader;
  return r;
}

// Where the operands' rows lie: row bytes rb, and for an operand whose rows
// start sh[k] bytes past a 16-byte boundary (mixed alignment; rb a multiple
// of 16) the aligned span that holds the row -- sh[k] bytes before it and
// 16 - sh[k] after, both inside the row's first / last 16-byte chunk -- is
// copied instead, into slots of `slot` bytes (rb + 16; rb when no operand is
// shifted).
struct RowSpans {
  size_t rb, slot;
  int sh[3];
};
__device__ __forceinline__ RowSpans plain_spans(size_t rb) { return RowSpans{rb, rb, {0, 0, 0}}; }

// Thread 0: bulk-copy CTA row i of the NS streamed operands into its stage.
template <int NS>
__device__ __forceinline__ void issue_row(const Ring& rg, int64_t i, int64_t first, int64_t stride,
                                          int S, const char* src0, const char* src1,
                                          const char* src2, const RowSpans& sp) {
  const int s = (int)(i % S);
  const int64_t row = first + i * stride;
  uint64_t* bar = rg.full + s;
  unsigned char* dst = rg.buf + (size_t)s * NS * sp.slot;
  const char* src[3] = {src0, src1, src2};
  uint32_t n[3], total = 0;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    n[k] = (uint32_t)(sp.rb + (sp.sh[k] ? 16 : 0));
    total += n[k];
  }
  mbar_arrive_expect_tx(bar, total);
#pragma unroll
  for (int k = 0; k < NS; ++k)
    bulk_copy_g2s(dst + k * sp.slot, src[k] + row * sp.rb - sp.sh[k], n[k], bar);
}
template <int NS>
__device__ __forceinline__ void issue_row(const Ring& rg, int64_t i, int64_t first, int64_t stride,
                                          int S, const char* src0, const char* src1,
                                          const char* src2, size_t rb) {
  issue_row<NS>(rg, i, first, stride, S, src0, src1, src2, plain_spans(rb));
}

// Thread 0, error path: wait (bounded) for rows [from, issued) still in flight.
__device__ __forceinline__ void drain(const Ring& rg, int64_t from, int64_t issued, int S) {
  for (int64_t j = from; j < issued; ++j)
    mbar_wait_bounded(rg.full + (j % S), (uint32_t)((j / S) & 1), kDrainLimit);
}

// Prologue: barriers initialised, the first min(S, nrows) rows requested.
template <int NS>
__device__ __forceinline__ int64_t ring_start(const Ring& rg, int S, int64_t nrows, int64_t first,
                                              int64_t stride, const char* src0, const char* src1,
                                              const char* src2, const RowSpans& sp) {
  int64_t issued = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(rg.full + s, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t n0 = nrows < S ? nrows : S;
    for (; issued < n0; ++issued)
      issue_row<NS>(rg, issued, first, stride, S, src0, src1, src2, sp);
  }
  return issued;
}
template <int NS>
__device__ __forceinline__ int64_t ring_start(const Ring& rg, int S, int64_t nrows, int64_t first,
                                              int64_t stride, const char* src0, const char* src1,
                                              const char* src2, size_t rb) {
  return ring_start<NS>(rg, S, nrows, first, stride, src0, src1, src2, plain_spans(rb));
}

// Vector v of an operand slot: the slot's own vector, or (shifted by s bytes)
// the 16 bytes starting s into its chunks v and v + 1.
__device__ __forceinline__ uint4 slot_vec(const unsigned char* slot, int v, int s) {
  const uint4* c = reinterpret_cast<const uint4*>(slot);
  if (s == 0) return c[v];
  return realign_pair(c[v], c[v + 1], s);
}

template <typename TW, int E>
__device__ __forceinline__ void gamma_f32(const void* gamma, int v, float (&g)[E]) {
  constexpr int GW = E * (int)sizeof(TW) / 16;
  const char* gp = static_cast<const char*>(gamma) + (size_t)v * GW * 16;
  if constexpr (std::is_same<TW, float>::value) {
#pragma unroll
    for (int w = 0; w < GW; ++w) {
      float t[4];
      unpack(ld_cached(gp + w * 16), t);
#pragma unroll
      for (int i = 0; i < 4; ++i) g[w * 4 + i] = t[i];
    }
  } else {
    unpack(ld_cached(gp), g);
  }
}

}  // namespace
}  // namespace rmsn
