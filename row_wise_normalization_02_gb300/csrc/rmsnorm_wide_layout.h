// Index arithmetic of the wide kernels, as plain integer functions usable on
// the host and the device: the split of a row into a scalar head, a body of
// 16-byte vectors and a scalar tail; where another operand's bytes for a body
// vector lie; which thread takes each head and tail element; the shared-memory
// layout of the backward's partial rows; the span of a row requested into L2.
// The kernels in rmsnorm_wide.cu call these, and a host test checks them
// exhaustively against the buffers they address.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define RMSN_HD __host__ __device__ __forceinline__
#else
#define RMSN_HD inline
#endif

namespace rmsn {

// Elements of a row of N elements of es bytes, starting at byte address a
// (a multiple of es), before its first 16-byte boundary: at most N.
RMSN_HD int wide_head(uintptr_t a, int N, int es) {
  const int h = (int)(((16u - ((unsigned)a & 15u)) & 15u) / (unsigned)es);
  return h > N ? N : h;
}

// Whole 16-byte vectors after the head.
RMSN_HD int wide_nv(int N, int head, int es) {
  return (int)(((int64_t)(N - head) * es) >> 4);
}

// Another operand's row starting at byte address b, read in a frame whose
// head has `head` elements: body vector v of the frame covers its bytes
// [base + 16 v + s, base + 16 v + s + 16), base 16-byte aligned and s in
// [0, 16).  With s != 0 the vector spans the aligned chunks at base + 16 v
// and base + 16 v + 16.
struct WideSrc {
  uintptr_t base;
  int s;
};
RMSN_HD WideSrc wide_src(uintptr_t b, int head, int es) {
  const uintptr_t a = b + (uintptr_t)head * es;
  return WideSrc{a & ~(uintptr_t)15, (int)(a & 15)};
}

// The head or tail element thread tid (of T) takes, or -1: head elements on
// the first threads, tail elements on the last.
RMSN_HD int wide_edge_elem(int head, int nv, int E, int N, int tid, int T) {
  if (tid < head) return tid;
  const int t0 = head + nv * E;
  const int k = T - 1 - tid;
  return k < N - t0 ? t0 + k : -1;
}

// A partial row in shared memory for a split (head, nv): the head's columns
// at [0, E), then the body in groups of 32 vectors -- for each float4 w of a
// vector, the group's 32 float4s side by side, so a warp's access to 32
// consecutive vectors covers 512 contiguous bytes -- then the tail's columns.
// Float offset of float4 w of body vector v:
RMSN_HD int wide_acc_vec(int v, int w, int E) {
  return E + (v >> 5) * (32 * E) + w * 128 + (v & 31) * 4;
}
// Float offset of column j:
RMSN_HD int wide_acc_col(int j, int head, int nv, int E) {
  if (j < head) return j;
  const int b = j - head, v = b / E;
  if (v < nv) return wide_acc_vec(v, (b - v * E) >> 2, E) + ((b - v * E) & 3);
  return E + (nv + 31) / 32 * (32 * E) + (b - nv * E);
}
// Floats of the layout for rows of N elements, any split (nv <= N / E).
RMSN_HD constexpr int wide_acc_floats(int N, int E) {
  return 2 * E + (N / E + 32) / 32 * 32 * E;
}

// The span requested into L2 for a row of rb bytes at byte address a: its
// enclosing 16-byte span [lo, lo + bytes), or bytes = 0 beyond 16 MB (not
// requested).
RMSN_HD uintptr_t wide_l2_lo(uintptr_t a) { return a & ~(uintptr_t)15; }
RMSN_HD uint32_t wide_l2_bytes(uintptr_t a, uint64_t rb) {
  const uintptr_t lo = a & ~(uintptr_t)15, hi = (a + rb + 15) & ~(uintptr_t)15;
  return hi - lo <= (uintptr_t(1) << 24) ? (uint32_t)(hi - lo) : 0u;
}

}  // namespace rmsn
