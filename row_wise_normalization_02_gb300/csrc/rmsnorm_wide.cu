// kWide: RMSNorm and LayerNorm rows of any length whose operands start at
// any element-aligned offsets, read and written as 16-byte vectors.  One CTA
// per row (persistent walk over rows), each pass over a row working in the
// frame of one operand: that operand's row splits into a scalar head
// (elements before its first 16-byte boundary), a body of 16-byte vectors
// and a scalar tail.  Every other operand is read in the pass's frame: the
// frame's body vector v covers 16 bytes of that operand which start s bytes
// into one of its aligned chunks (s: the difference of the two rows' start
// addresses modulo 16), so two aligned chunk loads and one byte funnel give
// it.  No load or store is misaligned whatever the offsets; DRAM sees each
// byte once, later passes re-reading the row from L1 or L2 (a row of tens of
// KB, read moments before), and a shifted operand's second chunk is the
// neighbouring vector's first.  The index arithmetic is in
// rmsnorm_wide_layout.h.
//
// Forward: the reduction in x's frame (fused add: the residual's, which
// receives h), the output in y's.  Backward: both passes in dx's frame (rows
// a multiple of 16 bytes, so the split is the same for every row), pass 2 of
// a row fused with pass 1 of the CTA's next row; the weight-gradient partial
// rows accumulate in shared memory, each column always by the same thread in
// the CTA's row order, and are written to the workspace once, at the end.
//
// The arithmetic per element is that of the register kernels: the sum of
// squares (fused add: of h = round(r + x)), rs = 1/sqrt(ss/N + eps),
// y = x rs gamma (bf16 x and gamma: (x gamma) rs), one rounding per output;
// dx = r (gamma dy - x c) with c = r^2/N sum gamma dy x ("Pre-built kernel
// library guide", 1.2 RMSNorm; the backward derived from its forward).
// LayerNorm below.
#include <type_traits>

#include "rmsnorm_bwd_common.cuh"
#include "rmsnorm_device.cuh"
#include "rmsnorm_fwd_common.cuh"
#include "rmsnorm_internal.h"
#include "rmsnorm_wide_layout.h"

#ifndef RMSN_PAIR
#define RMSN_PAIR 1
#endif

namespace rmsn {
namespace {

// Split of a row of N elements of es bytes starting at `row`: x = elements
// before the first 16-byte boundary (at most N), y = whole 16-byte vectors
// after them; the rest is the tail.
__device__ __forceinline__ int2 split_row(const void* row, int N, int es) {
  const int head = wide_head(reinterpret_cast<uintptr_t>(row), N, es);
  return make_int2(head, wide_nv(N, head, es));
}

// An operand read in another row's frame: the frame's body vector v is the
// 16 bytes at c + 16 v + s (c 16-byte aligned, 0 <= s < 16).
struct Src {
  const char* c;
  int s;
};
__device__ __forceinline__ Src src_of(const void* row, int head, int es) {
  const WideSrc w = wide_src(reinterpret_cast<uintptr_t>(row), head, es);
  return Src{reinterpret_cast<const char*>(w.base), w.s};
}

// Read of a chunk: read-only data that pass 2 re-reads (L1 allocation),
// read-only data read once (no L1 allocation), or data this kernel writes
// (h; the residual-path gradient beside dx) on the coherent path.
enum Ld : int { kLdKeep = 0, kLdOnce = 1, kLdRw = 2 };
template <int LD>
__device__ __forceinline__ uint4 ld_chunk(const char* p) {
  if constexpr (LD == kLdKeep) return ld_cached(p);
  else if constexpr (LD == kLdOnce) return ld_stream(p);
  else return ld_rw(p);
}

// Body vector v of an operand in the frame.  The second chunk is read only
// when the operand is shifted: it then holds bytes of this row (the vector's
// last s bytes), so it lies in the row's enclosing 16-byte span.
template <int LD>
__device__ __forceinline__ uint4 vec_at(const Src& o, int v) {
  const char* p = o.c + (size_t)v * 16;
  const uint4 lo = ld_chunk<LD>(p);
  if (o.s == 0) return lo;
  return realign_pair(lo, ld_chunk<LD>(p + 16), o.s);
}

// The GW gamma chunks (E columns) of body vector v in the frame.
template <int GW>
__device__ __forceinline__ void gamma_at(const Src& g, int v, uint4 (&out)[GW]) {
  const char* p = g.c + (size_t)v * GW * 16;
  uint4 c[GW + 1];
#pragma unroll
  for (int w = 0; w < GW; ++w) c[w] = ld_cached(p + w * 16);
  if (g.s == 0) {
#pragma unroll
    for (int w = 0; w < GW; ++w) out[w] = c[w];
    return;
  }
  c[GW] = ld_cached(p + GW * 16);
#pragma unroll
  for (int w = 0; w < GW; ++w) out[w] = realign_pair(c[w], c[w + 1], g.s);
}

__device__ __forceinline__ void st_plain(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Scalar read of data this kernel wrote (h), through L2.
template <typename T>
__device__ __forceinline__ float ld_scalar_cg(const T* p) {
  if constexpr (std::is_same<T, float>::value) {
    return __ldcg(p);
  } else {
    const unsigned short b = __ldcg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float((uint32_t)b << 16);
  }
}

template <typename TX>
__device__ __forceinline__ void vec_sumsq(const uint4& v, float& a0, float& a1) {
  if constexpr (std::is_same<TX, bf16>::value) {
    bf16x8_sumsq(v, a0, a1);
  } else {
    float f[4];
    unpack(v, f);
    a0 = fmaf(f[0], f[0], a0);
    a1 = fmaf(f[1], f[1], a1);
    a0 = fmaf(f[2], f[2], a0);
    a1 = fmaf(f[3], f[3], a1);
  }
}

// The scalar form of scale_vec.
template <typename TX, typename TW>
__device__ __forceinline__ float scale_scalar(float x, float g, float rs) {
  if constexpr (std::is_same<TX, bf16>::value && std::is_same<TW, bf16>::value)
    return (x * g) * rs;
  else
    return x * rs * g;
}

// Element of the head or the tail of a split (head, nv) that thread tid
// handles, or -1: head elements on the first threads, tail elements on the
// last (both fewer than a vector's elements).
template <int E>
__device__ __forceinline__ int edge_elem(int2 f, int N, int tid, int T) {
  return wide_edge_elem(f.x, f.y, E, N, tid, T);
}

// Row q of a row-major operand (rows of rb bytes, any element-aligned base)
// requested into L2: its enclosing 16-byte span, by the bulk-copy unit.
__device__ __forceinline__ void l2_row(const void* base, int64_t q, size_t rb) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(base) + (uintptr_t)q * rb;
  const uint32_t bytes = wide_l2_bytes(a, rb);   // rows up to 16 MB
  if (bytes) bulk_prefetch_l2(reinterpret_cast<const void*>(wide_l2_lo(a)), bytes);
}

// L2 lookahead of the CTA's walk: thread 0 requests the input rows L steps
// ahead (at the first row also those 1 .. L-1 steps ahead), so that pass 1
// reads from L2 rather than waiting on DRAM row after row.
__device__ __forceinline__ void l2_ahead(int L, int64_t row, bool first, int64_t M,
                                         size_t rb, const void* a, const void* b,
                                         const void* c) {
  if (L <= 0 || threadIdx.x != 0) return;
  for (int k = first ? 1 : L; k <= L; ++k) {
    const int64_t q = row + (int64_t)k * gridDim.x;
    if (q >= M) break;
    if (a) l2_row(a, q, rb);
    if (b) l2_row(b, q, rb);
    if (c) l2_row(c, q, rb);
  }
}

// ---------------------------------------------------------------- forward
//
// Two passes per row.  Pass 1 reads x in its own frame (one aligned chunk a
// vector, four vectors in flight a thread); fusing pass 2 of a row with pass 1
// of the next, as the backward does, lost here (8192 x 20000 bf16, x off 16
// bytes: 0.59 of the copy peak against 0.75).

// The plain forward with gamma no wider than x fits 42 registers (three CTAs
// of 512 threads, six of 256, per SM); the others take 64.
template <typename TX, typename TW, bool FUSED>
__global__ void __launch_bounds__(kWideThreads, (FUSED || sizeof(TW) > sizeof(TX)) ? 2 : 3)
    fwd_wide_kernel(const FwdParams p) {
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW, ES = (int)sizeof(TX), WS = (int)sizeof(TW);
  constexpr int U1 = FUSED ? 2 : 4;   // vectors per thread in flight, pass 1
  constexpr int U2 = 2;               // and pass 2
  __shared__ float red[64];
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const size_t rb = (size_t)N * ES;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const char* xr = static_cast<const char*>(p.x) + row * rb;
    char* hr = FUSED ? static_cast<char*>(p.residual) + row * rb : nullptr;
    char* yr = static_cast<char*>(p.y) + row * rb;
    l2_ahead(p.l2_rows, row, row == blockIdx.x, p.M, rb, p.x, FUSED ? p.residual : nullptr,
             nullptr);
    float s0 = 0.f, s1 = 0.f;
    {  // pass 1: the sum of squares in the frame of x (fused: of the residual)
      const char* fr = FUSED ? hr : xr;
      const int2 f = split_row(fr, N, ES);
      const char* fb = fr + (size_t)f.x * ES;
      char* hb = FUSED ? hr + (size_t)f.x * ES : nullptr;
      if constexpr (!FUSED) {
        for (int v0 = tid; v0 < f.y; v0 += U1 * T) {
          uint4 a[U1];
#pragma unroll
          for (int u = 0; u < U1; ++u) {
            const int v = v0 + u * T;
            a[u] = v < f.y ? ld_cached(fb + (size_t)v * 16) : zero;
          }
#pragma unroll
          for (int u = 0; u < U1; ++u) vec_sumsq<TX>(a[u], s0, s1);
        }
      } else {
        const Src xs = src_of(xr, f.x, ES);
        for (int v0 = tid; v0 < f.y; v0 += U1 * T) {
          uint4 a[U1], r[U1];
#pragma unroll
          for (int u = 0; u < U1; ++u) {
            const int v = v0 + u * T;
            r[u] = v < f.y ? ld_rw(fb + (size_t)v * 16) : zero;
            a[u] = v < f.y ? vec_at<kLdOnce>(xs, v) : zero;
          }
#pragma unroll
          for (int u = 0; u < U1; ++u) {
            float hf[E], rf[E];
            unpack(a[u], hf);
            unpack(r[u], rf);
#pragma unroll
            for (int e = 0; e < E; ++e) hf[e] += rf[e];
            const uint4 h = pack(hf);   // rounds to TX (nearest even)
            const int v = v0 + u * T;
            if (v < f.y) st_plain(hb + (size_t)v * 16, h);
            vec_sumsq<TX>(h, s0, s1);
          }
        }
      }
      const int j = edge_elem<E>(f, N, tid, T);
      if (j >= 0) {
        float v = ld_scalar(reinterpret_cast<const TX*>(xr) + j);
        if (FUSED) {
          v = round_to(v + ld_scalar(reinterpret_cast<const TX*>(hr) + j), (TX*)nullptr);
          st_scalar(reinterpret_cast<TX*>(hr) + j, v);
        }
        s0 = fmaf(v, v, s0);
      }
    }
    float ss[1] = {s0 + s1};
    cta_sum<1>(ss, red, parity);   // its barrier also publishes h to the CTA
    parity ^= 1;
    const float rs = rsqrtf(fmaf(ss[0], p.inv_n, p.eps));
    if (tid == 0 && p.rstd != nullptr) p.rstd[row] = rs;
    {  // pass 2: y in its own frame
      const int2 f = split_row(yr, N, ES);
      char* yb = yr + (size_t)f.x * ES;
      const Src xs = src_of(FUSED ? hr : xr, f.x, ES);
      const Src gs = src_of(p.gamma, f.x, WS);
      for (int v0 = tid; v0 < f.y; v0 += U2 * T) {
        uint4 a[U2], g[U2][GW];
#pragma unroll
        for (int u = 0; u < U2; ++u) {
          const int v = v0 + u * T;
          if (v < f.y) {
            a[u] = vec_at<FUSED ? kLdRw : kLdKeep>(xs, v);
            gamma_at<GW>(gs, v, g[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < U2; ++u) {
          const int v = v0 + u * T;
          if (v < f.y) st_stream(yb + (size_t)v * 16, scale_vec<TX, TW>(a[u], g[u], rs));
        }
      }
      const int j = edge_elem<E>(f, N, tid, T);
      if (j >= 0) {
        const float v = FUSED ? ld_scalar_cg(reinterpret_cast<const TX*>(hr) + j)
                              : ld_scalar(reinterpret_cast<const TX*>(xr) + j);
        const float g = ld_scalar_ro(static_cast<const TW*>(p.gamma) + j);
        st_scalar(reinterpret_cast<TX*>(yr) + j, scale_scalar<TX, TW>(v, g, rs));
      }
    }
  }
}

// ---------------------------------------------------------------- backward
//
// A partial row in shared memory, for dx's split (head, nv): the head's
// columns at [0, E), then the body in groups of 32 vectors -- for each
// float4 w of a vector, the group's 32 float4s side by side, so that a warp's
// access to 32 consecutive vectors covers 512 contiguous bytes (no bank
// conflict; vectors laid end to end would put a warp's float4s 32 bytes
// apart for bf16, two to a bank group) -- then the tail's columns.
template <int E>
__device__ __forceinline__ int acc_vec(int v, int w) {
  return wide_acc_vec(v, w, E);
}
template <int E>
__device__ __forceinline__ int acc_col(int j, int2 f) {
  return wide_acc_col(j, f.x, f.y, E);
}
//
// Both passes in dx's frame (rows a multiple of 16 bytes: the same split, and
// the same shifts of x and dy against it, for every row), and pass 2 of a row
// fused with pass 1 of the CTA's next row: one loop over dx's vectors reads
// gamma once, the current row's x and dy again (from L1 or L2) and the next
// row's from DRAM, so every trip to memory carries both rows and the walk has
// one dependent chain per row, not two.

template <typename TX, typename TW, bool HAS_RSTD, bool DRES>
__global__ void __launch_bounds__(kWideBwdThreads, 2) bwd_wide_kernel(const BwdParams p) {
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW, ES = (int)sizeof(TX), WS = (int)sizeof(TW);
  constexpr int K = HAS_RSTD ? 1 : 2;
  // dgamma partial row, laid out by acc_col for dx's split
  extern __shared__ __align__(16) float acc_s[];
  __shared__ float red[2 * 2 * 32];
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const size_t rb = (size_t)N * ES;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const bool dg = p.partial != nullptr;
  const int2 fo = split_row(p.dx, N, ES);
  const Src gs = src_of(p.gamma, fo.x, WS);
  const int je = edge_elem<E>(fo, N, tid, T);   // this thread's head or tail element
  const TW* gp = static_cast<const TW*>(p.gamma);
  if (dg)
    for (int i = tid; i < wide_acc_floats(N, E); i += T) acc_s[i] = 0.f;
  const char* x0 = static_cast<const char*>(p.x);
  const char* d0 = static_cast<const char*>(p.dy);
  int64_t row = blockIdx.x;
  // pass 1 of the first row
  float2 dot = make_float2(0.f, 0.f), sq = make_float2(0.f, 0.f);
  if (row < p.M) {
    // (the walk reads the row after the current one as it goes: the
    // lookahead counts from there)
    l2_ahead(p.l2_rows, row + gridDim.x, true, p.M, rb, p.x, p.dy, DRES ? p.dres : nullptr);
    const Src xs = src_of(x0 + row * rb, fo.x, ES), ds = src_of(d0 + row * rb, fo.x, ES);
    for (int v = tid; v < fo.y; v += T) {
      uint4 g[GW];
      gamma_at<GW>(gs, v, g);
      const uint4 a = vec_at<kLdKeep>(xs, v), d = vec_at<kLdKeep>(ds, v);
      float gf[E];
      unpack_gamma<TW, E, GW>(g, gf);
      bwd_vec_sums<E, !HAS_RSTD>(a, d, gf, dot, sq);
    }
    if (je >= 0) {
      const float xv = ld_scalar(reinterpret_cast<const TX*>(x0 + row * rb) + je);
      const float dv = ld_scalar(reinterpret_cast<const TX*>(d0 + row * rb) + je);
      dot.x = fmaf(ld_scalar_ro(gp + je) * dv, xv, dot.x);
      if (!HAS_RSTD) sq.x = fmaf(xv, xv, sq.x);
    }
  }
  int parity = 0;
  for (; row < p.M; row += gridDim.x) {
    float sums[K];
    sums[0] = dot.x + dot.y;
    if (!HAS_RSTD) sums[K - 1] = sq.x + sq.y;
    cta_sum<K>(sums, red, parity);
    parity ^= 1;
    const float r = HAS_RSTD ? __ldg(p.rstd + row) : rsqrtf(fmaf(sums[K - 1], p.inv_n, p.eps));
    const float c = r * r * p.inv_n * sums[0];
    const int64_t nxt = row + gridDim.x;
    const bool more = nxt < p.M;   // the same in every thread
    l2_ahead(p.l2_rows, nxt, false, p.M, rb, p.x, p.dy, DRES ? p.dres : nullptr);
    const char* xr = x0 + row * rb;
    const char* dr = d0 + row * rb;
    char* dxr = static_cast<char*>(p.dx) + row * rb;
    const char* rr = DRES ? static_cast<const char*>(p.dres) + row * rb : nullptr;
    char* ob = dxr + (size_t)fo.x * ES;
    const Src xs = src_of(xr, fo.x, ES), ds = src_of(dr, fo.x, ES);
    const Src qs = DRES ? src_of(rr, fo.x, ES) : Src{nullptr, 0};
    const Src xn = src_of(x0 + (more ? nxt : row) * rb, fo.x, ES);
    const Src dn = src_of(d0 + (more ? nxt : row) * rb, fo.x, ES);
    dot = sq = make_float2(0.f, 0.f);
    for (int v = tid; v < fo.y; v += T) {
      uint4 g[GW];
      gamma_at<GW>(gs, v, g);
      const uint4 a = vec_at<kLdKeep>(xs, v), d = vec_at<kLdKeep>(ds, v);
      const uint4 q = DRES ? vec_at<kLdRw>(qs, v) : zero;
      uint4 an = zero, dnv = zero;
      if (more) {
        an = vec_at<kLdKeep>(xn, v);
        dnv = vec_at<kLdKeep>(dn, v);
      }
      float gf[E], acc[E];
      unpack_gamma<TW, E, GW>(g, gf);
#pragma unroll
      for (int w = 0; w < E / 4; ++w) {
        const float4 t = dg ? *reinterpret_cast<const float4*>(acc_s + acc_vec<E>(v, w))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        acc[4 * w] = t.x;
        acc[4 * w + 1] = t.y;
        acc[4 * w + 2] = t.z;
        acc[4 * w + 3] = t.w;
      }
      st_stream(ob + (size_t)v * 16, bwd_vec_apply<E, DRES>(a, d, q, gf, r, c, acc));
      if (dg) {
#pragma unroll
        for (int w = 0; w < E / 4; ++w)
          *reinterpret_cast<float4*>(acc_s + acc_vec<E>(v, w)) =
              make_float4(acc[4 * w], acc[4 * w + 1], acc[4 * w + 2], acc[4 * w + 3]);
      }
      if (more) bwd_vec_sums<E, !HAS_RSTD>(an, dnv, gf, dot, sq);
    }
    if (je >= 0) {
      const float gv = ld_scalar_ro(gp + je);
      const float xv = ld_scalar(reinterpret_cast<const TX*>(xr) + je);
      const float dv = ld_scalar(reinterpret_cast<const TX*>(dr) + je);
      float o = r * fmaf(-xv, c, gv * dv);
      if (DRES) o += ld_scalar_cg(reinterpret_cast<const TX*>(rr) + je);
      st_scalar(reinterpret_cast<TX*>(dxr) + je, o);
      if (dg) {
        float* a = acc_s + acc_col<E>(je, fo);
        *a = fmaf(dv * xv, r, *a);
      }
      if (more) {
        const float xv2 = ld_scalar(reinterpret_cast<const TX*>(x0 + nxt * rb) + je);
        const float dv2 = ld_scalar(reinterpret_cast<const TX*>(d0 + nxt * rb) + je);
        dot.x = fmaf(gv * dv2, xv2, dot.x);
        if (!HAS_RSTD) sq.x = fmaf(xv2, xv2, sq.x);
      }
    }
  }
  if (dg) {
    __syncthreads();
    float* prow = p.partial + (size_t)blockIdx.x * p.ld_partial;
    for (int j = tid; j < N; j += T) prow[j] = acc_s[acc_col<E>(j, fo)];
  }
}

// ---------------------------------------------------------------- LayerNorm
//
// The same frames for LayerNorm.  The statistics are taken in x's frame --
// m0 = sum x / N and, unless the moments about zero suffice (below), the
// corrected two-pass moments c = sum (x - m0) / N and
// rs = 1 / sqrt(sum (x - m0)^2 / N - c^2 + eps), the mean being m0 + c
// ("Pre-built kernel library guide", 1.1 LayerNorm) -- and the outputs in
// their own frame: y = ((x - m0) - c) rs gamma + beta; the backward's
// dx = rs (dy gamma - (mg + xh mgx)) with xh = ((x - m0) - c) rs, mg and mgx
// the row means of dy gamma and dy gamma xh, dgamma += dy xh, dbeta += dy.

// Sum of a vector's elements into two accumulators (even / odd elements);
// bf16 straight from the packed words by the mixed-precision FMA with 1 (one
// rounding, as the fp32 add of the exact value).
template <typename TX>
__device__ __forceinline__ void vec_sum(const uint4& v, float& s0, float& s1) {
  if constexpr (std::is_same<TX, bf16>::value) {
    asm("{\n\t.reg .b16 l0, h0, l1, h1, l2, h2, l3, h3, one;\n\t"
        "mov.b16 one, 0x3F80;\n\t"
        "mov.b32 {l0, h0}, %2;\n\t"
        "mov.b32 {l1, h1}, %3;\n\t"
        "mov.b32 {l2, h2}, %4;\n\t"
        "mov.b32 {l3, h3}, %5;\n\t"
        "fma.rn.f32.bf16 %0, l0, one, %0;\n\t"
        "fma.rn.f32.bf16 %1, h0, one, %1;\n\t"
        "fma.rn.f32.bf16 %0, l1, one, %0;\n\t"
        "fma.rn.f32.bf16 %1, h1, one, %1;\n\t"
        "fma.rn.f32.bf16 %0, l2, one, %0;\n\t"
        "fma.rn.f32.bf16 %1, h2, one, %1;\n\t"
        "fma.rn.f32.bf16 %0, l3, one, %0;\n\t"
        "fma.rn.f32.bf16 %1, h3, one, %1;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
  } else {
    float f[4];
    unpack(v, f);
    s0 += f[0];
    s1 += f[1];
    s0 += f[2];
    s1 += f[3];
  }
}

template <typename TX>
__device__ __forceinline__ void vec_dev(const uint4& v, float m0, float& sd, float& sq) {
  constexpr int E = Elem<TX>::kPerVec;
  float f[E];
  unpack(v, f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float d = f[e] - m0;
    sd += d;
    sq = fmaf(d, d, sq);
  }
}

// (m0, c, rs) of the row at xr, in x's frame; every thread of the CTA gets
// them.  Pass 1 sums x and x^2.  Where the row's mean is small against its
// spread (m0^2 <= sum x^2 / N - m0^2, so that the difference loses at most a
// factor two of its precision), rs comes from those sums with c = 0, and the
// row is read once; otherwise pass 2 forms the corrected moments about m0.
template <typename TX>
__device__ __forceinline__ float3 wide_ln_stats(const char* xr, int N, float* red, int& parity,
                                                float inv_n, float eps) {
  constexpr int E = Elem<TX>::kPerVec, ES = (int)sizeof(TX), U = 4;
  const int tid = threadIdx.x, T = blockDim.x;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const int2 f = split_row(xr, N, ES);
  const char* xb = xr + (size_t)f.x * ES;
  const int j = edge_elem<E>(f, N, tid, T);
  const TX* xe = reinterpret_cast<const TX*>(xr);
  float s0 = 0.f, s1 = 0.f, q0 = 0.f, q1 = 0.f;
  for (int v0 = tid; v0 < f.y; v0 += U * T) {
    uint4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * T;
      a[u] = v < f.y ? ld_cached(xb + (size_t)v * 16) : zero;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      vec_sum<TX>(a[u], s0, s1);
      vec_sumsq<TX>(a[u], q0, q1);
    }
  }
  if (j >= 0) {
    const float v = ld_scalar(xe + j);
    s0 += v;
    q0 = fmaf(v, v, q0);
  }
  float t1[2] = {s0 + s1, q0 + q1};
  cta_sum<2>(t1, red, parity);
  parity ^= 1;
  const float m0 = t1[0] * inv_n;
  const float var1 = fmaf(t1[1], inv_n, -m0 * m0);
  if (m0 * m0 <= var1) return make_float3(m0, 0.f, rsqrtf(var1 + eps));
  float sd = 0.f, sq = 0.f;
  for (int v0 = tid; v0 < f.y; v0 += U * T) {
    uint4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * T;
      a[u] = v < f.y ? ld_cached(xb + (size_t)v * 16) : zero;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (v0 + u * T < f.y) vec_dev<TX>(a[u], m0, sd, sq);
    }
  }
  if (j >= 0) {
    const float d = ld_scalar(xe + j) - m0;
    sd += d;
    sq = fmaf(d, d, sq);
  }
  float t2[2] = {sd, sq};
  cta_sum<2>(t2, red, parity);
  parity ^= 1;
  const float c = t2[0] * inv_n;
  return make_float3(m0, c, rsqrtf(fmaxf(fmaf(t2[1], inv_n, -c * c), 0.f) + eps));
}

template <typename TX, typename TW>
__global__ void __launch_bounds__(kWideThreads, 2) ln_fwd_wide_kernel(const LnParams p) {
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW, ES = (int)sizeof(TX), WS = (int)sizeof(TW);
  constexpr int U = GW == 2 ? 1 : 2;   // vectors in flight (gamma and beta in fp32: one)
  __shared__ float red[128];
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const size_t rb = (size_t)N * ES;
  const bool hb = p.beta != nullptr;
  const TW* gp = static_cast<const TW*>(p.gamma);
  const TW* bp = static_cast<const TW*>(p.beta);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
    const char* xr = static_cast<const char*>(p.x) + row * rb;
    char* yr = static_cast<char*>(p.y) + row * rb;
    l2_ahead(p.l2_rows, row, row == blockIdx.x, p.M, rb, p.x, nullptr, nullptr);
    const float3 st = wide_ln_stats<TX>(xr, N, red, parity, p.inv_n, p.eps);
    if (tid == 0) {
      if (p.mean != nullptr) p.mean[row] = st.x + st.y;
      if (p.rstd != nullptr) p.rstd[row] = st.z;
    }
    const int2 f = split_row(yr, N, ES);
    char* yb = yr + (size_t)f.x * ES;
    const Src xs = src_of(xr, f.x, ES), gs = src_of(p.gamma, f.x, WS),
              bs = src_of(hb ? p.beta : p.gamma, f.x, WS);
    for (int v0 = tid; v0 < f.y; v0 += U * T) {
      uint4 a[U], g[U][GW], b[U][GW];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * T;
        if (v < f.y) {
          a[u] = vec_at<kLdKeep>(xs, v);
          gamma_at<GW>(gs, v, g[u]);
          if (hb) gamma_at<GW>(bs, v, b[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * T;
        if (v >= f.y) continue;
        float xf[E], gf[E], bf[E];
        unpack(a[u], xf);
        unpack_gamma<TW, E, GW>(g[u], gf);
        if (hb) {
          unpack_gamma<TW, E, GW>(b[u], bf);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) bf[e] = 0.f;
        }
        // ((x - m0) - c) rs gamma + beta, two elements per paired instruction
        const float2 nm = make_float2(-st.x, -st.x), nc = make_float2(-st.y, -st.y),
                     r2 = make_float2(st.z, st.z);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 t = __fmul2_rn(
              __fadd2_rn(__fadd2_rn(make_float2(xf[e], xf[e + 1]), nm), nc), r2);
          const float2 o =
              __ffma2_rn(t, make_float2(gf[e], gf[e + 1]), make_float2(bf[e], bf[e + 1]));
          xf[e] = o.x;
          xf[e + 1] = o.y;
        }
        st_stream(yb + (size_t)v * 16, pack(xf));
      }
    }
    const int j = edge_elem<E>(f, N, tid, T);
    if (j >= 0) {
      const float t = ((ld_scalar(reinterpret_cast<const TX*>(xr) + j) - st.x) - st.y) * st.z;
      st_scalar(reinterpret_cast<TX*>(yr) + j,
                fmaf(t, ld_scalar_ro(gp + j), hb ? ld_scalar_ro(bp + j) : 0.f));
    }
  }
}

// Backward: rows a multiple of 16 bytes; the partial rows [dgamma | dbeta]
// in shared memory, each NA floats laid out as the RMSNorm backward's.

// Pass a of one vector: the row sums of g = dy gamma and g xh, even / odd
// elements apart, two per paired instruction.
template <typename TX, int E>
__device__ __forceinline__ void ln_sums_vec(const uint4& xv, const uint4& dv,
                                            const float (&gf)[E], float3 st, float2& a2,
                                            float2& b2) {
  float xf[E], df[E];
  unpack(xv, xf);
  unpack(dv, df);
  const float2 nm = make_float2(-st.x, -st.x), nc = make_float2(-st.y, -st.y),
               r2 = make_float2(st.z, st.z);
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 gd =
        __fmul2_rn(make_float2(df[e], df[e + 1]), make_float2(gf[e], gf[e + 1]));   // 0 past the row
    const float2 xh =
        __fmul2_rn(__fadd2_rn(__fadd2_rn(make_float2(xf[e], xf[e + 1]), nm), nc), r2);
    a2 = __fadd2_rn(a2, gd);
    b2 = __ffma2_rn(gd, xh, b2);
  }
}

// Pass b of body vector v: dx = rs (dy gamma - (mg + xh mgx)), and
// dgamma += dy xh, dbeta += dy in the partial rows (when dg).
template <typename TX, int E>
__device__ __forceinline__ uint4 ln_dx_vec(int v, const uint4& xv, const uint4& dv,
                                           const float (&gf)[E], float3 st, float mg,
                                           float mgx, float* acc_s, int NA, bool dg) {
  float xf[E], df[E], pg[E], pb[E];
  unpack(xv, xf);
  unpack(dv, df);
#pragma unroll
  for (int w = 0; w < E / 4; ++w) {
    const float* ag = acc_s + acc_vec<E>(v, w);
    const float4 tg = dg ? *reinterpret_cast<const float4*>(ag) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 tb = dg ? *reinterpret_cast<const float4*>(ag + NA)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    pg[4 * w] = tg.x; pg[4 * w + 1] = tg.y; pg[4 * w + 2] = tg.z; pg[4 * w + 3] = tg.w;
    pb[4 * w] = tb.x; pb[4 * w + 1] = tb.y; pb[4 * w + 2] = tb.z; pb[4 * w + 3] = tb.w;
  }
  const float2 nm = make_float2(-st.x, -st.x), nc = make_float2(-st.y, -st.y),
               r2 = make_float2(st.z, st.z), mgx2 = make_float2(mgx, mgx),
               mg2 = make_float2(mg, mg);
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 d2 = make_float2(df[e], df[e + 1]);
    const float2 xh =
        __fmul2_rn(__fadd2_rn(__fadd2_rn(make_float2(xf[e], xf[e + 1]), nm), nc), r2);
    const float2 f = __ffma2_rn(xh, mgx2, mg2);
    const float2 o = __fmul2_rn(
        r2, __fadd2_rn(__fmul2_rn(d2, make_float2(gf[e], gf[e + 1])), make_float2(-f.x, -f.y)));
    const float2 q = __ffma2_rn(d2, xh, make_float2(pg[e], pg[e + 1]));
    const float2 w = __fadd2_rn(make_float2(pb[e], pb[e + 1]), d2);
    xf[e] = o.x;
    xf[e + 1] = o.y;
    pg[e] = q.x;
    pg[e + 1] = q.y;
    pb[e] = w.x;
    pb[e + 1] = w.y;
  }
  if (dg) {
#pragma unroll
    for (int w = 0; w < E / 4; ++w) {
      float* ag = acc_s + acc_vec<E>(v, w);
      *reinterpret_cast<float4*>(ag) =
          make_float4(pg[4 * w], pg[4 * w + 1], pg[4 * w + 2], pg[4 * w + 3]);
      *reinterpret_cast<float4*>(ag + NA) =
          make_float4(pb[4 * w], pb[4 * w + 1], pb[4 * w + 2], pb[4 * w + 3]);
    }
  }
  return pack(xf);
}

// The head or tail element je of a row: pass a's sums, or pass b's dx and
// partials.
template <typename TX, typename TW>
__device__ __forceinline__ void ln_sums_edge(const char* xr, const char* dr, const TW* gp, int je,
                                             float3 st, float2& a2, float2& b2) {
  const float xh = ((ld_scalar(reinterpret_cast<const TX*>(xr) + je) - st.x) - st.y) * st.z;
  const float gd = ld_scalar(reinterpret_cast<const TX*>(dr) + je) * ld_scalar_ro(gp + je);
  a2.x += gd;
  b2.x = fmaf(gd, xh, b2.x);
}
template <typename TX, typename TW, int E>
__device__ __forceinline__ void ln_dx_edge(const char* xr, const char* dr, char* dxr,
                                           const TW* gp, int je, int2 fo, float3 st, float mg,
                                           float mgx, float* acc_s, int NA, bool dg) {
  const float dv = ld_scalar(reinterpret_cast<const TX*>(dr) + je);
  const float xh = ((ld_scalar(reinterpret_cast<const TX*>(xr) + je) - st.x) - st.y) * st.z;
  st_scalar(reinterpret_cast<TX*>(dxr) + je,
            st.z * (dv * ld_scalar_ro(gp + je) - fmaf(xh, mgx, mg)));
  if (dg) {
    float* ag = acc_s + acc_col<E>(je, fo);
    *ag = fmaf(dv, xh, *ag);
    ag[NA] += dv;
  }
}

// SAVED: the forward's mean and rstd are given; pass b of a row then runs
// fused with pass a of the CTA's next row (one loop over dx's vectors reads
// gamma once, the current row again and the next row from DRAM), as in the
// RMSNorm wide backward, in CTAs of at most kLnSavedThreads (80 registers a
// thread).  Otherwise the statistics, then pass a, then pass b.
template <typename TX, typename TW, bool SAVED>
__global__ void __launch_bounds__(SAVED ? kLnSavedThreads : kWideBwdThreads, 2)
    ln_bwd_wide_kernel(const LnParams p) {
  pdl_begin();
  using C = Cfg<TX, TW>;
  constexpr int E = C::E, GW = C::GW, ES = (int)sizeof(TX), WS = (int)sizeof(TW);
  constexpr int U = GW == 2 ? 1 : 2;   // vectors in flight, pass a of the unsaved form
  extern __shared__ __align__(16) float acc_s[];
  __shared__ float red[128];
  const int tid = threadIdx.x, T = blockDim.x, N = p.N;
  const int NA = wide_acc_floats(N, E);   // [dgamma | dbeta], each laid out by acc_col
  const size_t rb = (size_t)N * ES;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const bool dg = p.partial != nullptr;
  const int2 fo = split_row(p.y, N, ES);   // dx's split, the same for every row
  const Src gs = src_of(p.gamma, fo.x, WS);
  const int je = edge_elem<E>(fo, N, tid, T);
  const TW* gp = static_cast<const TW*>(p.gamma);
  const char* x0 = static_cast<const char*>(p.x);
  const char* d0 = static_cast<const char*>(p.dy);
  char* dx0 = static_cast<char*>(p.y);
  if (dg)
    for (int i = tid; i < 2 * NA; i += T) acc_s[i] = 0.f;
  int parity = 0;
  if constexpr (SAVED) {
    int64_t row = blockIdx.x;
    float2 a2 = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
    if (row < p.M) {   // pass a of the first row
      l2_ahead(p.l2_rows, row + gridDim.x, true, p.M, rb, p.x, p.dy, nullptr);
      const float3 st = make_float3(p.mean[row], 0.f, p.rstd[row]);
      const Src xs = src_of(x0 + row * rb, fo.x, ES), ds = src_of(d0 + row * rb, fo.x, ES);
      for (int v = tid; v < fo.y; v += T) {
        uint4 g[GW];
        gamma_at<GW>(gs, v, g);
        const uint4 xv = vec_at<kLdKeep>(xs, v), dv = vec_at<kLdKeep>(ds, v);
        float gf[E];
        unpack_gamma<TW, E, GW>(g, gf);
        ln_sums_vec<TX, E>(xv, dv, gf, st, a2, b2);
      }
      if (je >= 0) ln_sums_edge<TX, TW>(x0 + row * rb, d0 + row * rb, gp, je, st, a2, b2);
    }
    for (; row < p.M; row += gridDim.x) {
      float t[2] = {a2.x + a2.y, b2.x + b2.y};
      cta_sum<2>(t, red, parity);
      parity ^= 1;
      const float mg = t[0] * p.inv_n, mgx = t[1] * p.inv_n;
      const int64_t nxt = row + gridDim.x;
      const bool more = nxt < p.M;   // the same in every thread
      const int64_t qn = more ? nxt : row;
      l2_ahead(p.l2_rows, nxt, false, p.M, rb, p.x, p.dy, nullptr);
      const float3 st = make_float3(p.mean[row], 0.f, p.rstd[row]);
      const float3 sn = make_float3(p.mean[qn], 0.f, p.rstd[qn]);
      const char* xr = x0 + row * rb;
      const char* dr = d0 + row * rb;
      char* dxr = dx0 + row * rb;
      char* ob = dxr + (size_t)fo.x * ES;
      const Src xs = src_of(xr, fo.x, ES), ds = src_of(dr, fo.x, ES);
      const Src xn = src_of(x0 + qn * rb, fo.x, ES), dn = src_of(d0 + qn * rb, fo.x, ES);
      a2 = b2 = make_float2(0.f, 0.f);
      for (int v = tid; v < fo.y; v += T) {
        uint4 g[GW];
        gamma_at<GW>(gs, v, g);
        const uint4 xv = vec_at<kLdKeep>(xs, v), dv = vec_at<kLdKeep>(ds, v);
        uint4 xv2 = zero, dv2 = zero;
        if (more) {
          xv2 = vec_at<kLdKeep>(xn, v);
          dv2 = vec_at<kLdKeep>(dn, v);
        }
        float gf[E];
        unpack_gamma<TW, E, GW>(g, gf);
        st_stream(ob + (size_t)v * 16,
                  ln_dx_vec<TX, E>(v, xv, dv, gf, st, mg, mgx, acc_s, NA, dg));
        if (more) ln_sums_vec<TX, E>(xv2, dv2, gf, sn, a2, b2);
      }
      if (je >= 0) {
        ln_dx_edge<TX, TW, E>(xr, dr, dxr, gp, je, fo, st, mg, mgx, acc_s, NA, dg);
        if (more) ln_sums_edge<TX, TW>(x0 + nxt * rb, d0 + nxt * rb, gp, je, sn, a2, b2);
      }
    }
  } else {
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
      const char* xr = x0 + row * rb;
      const char* dr = d0 + row * rb;
      char* dxr = dx0 + row * rb;
      l2_ahead(p.l2_rows, row, row == blockIdx.x, p.M, rb, p.x, p.dy, nullptr);
      const float3 st = wide_ln_stats<TX>(xr, N, red, parity, p.inv_n, p.eps);
      const Src xs = src_of(xr, fo.x, ES), ds = src_of(dr, fo.x, ES);
      float2 a2 = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
      for (int v0 = tid; v0 < fo.y; v0 += U * T) {
        uint4 xv[U], dv[U], g[U][GW];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * T;
          if (v < fo.y) {
            xv[u] = vec_at<kLdKeep>(xs, v);
            dv[u] = vec_at<kLdKeep>(ds, v);
            gamma_at<GW>(gs, v, g[u]);
          } else {
            xv[u] = dv[u] = zero;
#pragma unroll
            for (int w = 0; w < GW; ++w) g[u][w] = zero;
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float gf[E];
          unpack_gamma<TW, E, GW>(g[u], gf);
          ln_sums_vec<TX, E>(xv[u], dv[u], gf, st, a2, b2);
        }
      }
      if (je >= 0) ln_sums_edge<TX, TW>(xr, dr, gp, je, st, a2, b2);
      float t[2] = {a2.x + a2.y, b2.x + b2.y};
      cta_sum<2>(t, red, parity);
      parity ^= 1;
      const float mg = t[0] * p.inv_n, mgx = t[1] * p.inv_n;
      char* ob = dxr + (size_t)fo.x * ES;
      for (int v = tid; v < fo.y; v += T) {
        uint4 g[GW];
        gamma_at<GW>(gs, v, g);
        const uint4 xv = vec_at<kLdKeep>(xs, v), dv = vec_at<kLdKeep>(ds, v);
        float gf[E];
        unpack_gamma<TW, E, GW>(g, gf);
        st_stream(ob + (size_t)v * 16,
                  ln_dx_vec<TX, E>(v, xv, dv, gf, st, mg, mgx, acc_s, NA, dg));
      }
      if (je >= 0) ln_dx_edge<TX, TW, E>(xr, dr, dxr, gp, je, fo, st, mg, mgx, acc_s, NA, dg);
    }
  }
  if (dg) {
    __syncthreads();
    float* prow = p.partial + (size_t)blockIdx.x * 2 * p.ld_half;
    for (int j = tid; j < N; j += T) {
      const int i = acc_col<E>(j, fo);
      prow[j] = acc_s[i];
      prow[p.ld_half + j] = acc_s[NA + i];
    }
  }
}

template <typename TX, typename TW>
LnKernel pick_ln(const LnKey& k) {
  if (k.family != kWide) return nullptr;
  if (!k.bwd) return ln_fwd_wide_kernel<TX, TW>;
  return k.saved ? ln_bwd_wide_kernel<TX, TW, true> : ln_bwd_wide_kernel<TX, TW, false>;
}

template <typename TX, typename TW>
FwdKernel pick_fwd(const FwdKey& k) {
  if (k.family != kWide || k.strided || k.out != kOutDtype) return nullptr;
  return k.fused ? fwd_wide_kernel<TX, TW, true> : fwd_wide_kernel<TX, TW, false>;
}

template <typename TX, typename TW>
BwdKernel pick_bwd(const BwdKey& k) {
  if (k.family != kWide) return nullptr;
  if (k.dres)
    return k.has_rstd ? bwd_wide_kernel<TX, TW, true, true> : bwd_wide_kernel<TX, TW, false, true>;
  return k.has_rstd ? bwd_wide_kernel<TX, TW, true, false> : bwd_wide_kernel<TX, TW, false, false>;
}

}  // namespace

#if RMSN_PAIR == 0
FwdKernel get_fwd_wide_f32_f32(const FwdKey& k) { return pick_fwd<float, float>(k); }
BwdKernel get_bwd_wide_f32_f32(const BwdKey& k) { return pick_bwd<float, float>(k); }
LnKernel get_ln_wide_f32_f32(const LnKey& k) { return pick_ln<float, float>(k); }
#elif RMSN_PAIR == 1
FwdKernel get_fwd_wide_bf16_bf16(const FwdKey& k) { return pick_fwd<bf16, bf16>(k); }
BwdKernel get_bwd_wide_bf16_bf16(const BwdKey& k) { return pick_bwd<bf16, bf16>(k); }
LnKernel get_ln_wide_bf16_bf16(const LnKey& k) { return pick_ln<bf16, bf16>(k); }
#else
FwdKernel get_fwd_wide_bf16_f32(const FwdKey& k) { return pick_fwd<bf16, float>(k); }
BwdKernel get_bwd_wide_bf16_f32(const BwdKey& k) { return pick_bwd<bf16, float>(k); }
LnKernel get_ln_wide_bf16_f32(const LnKey& k) { return pick_ln<bf16, float>(k); }
#endif

}  // namespace rmsn
