// Device building blocks shared by the RMSNorm kernels: 16-byte vector
// loads/stores with explicit cache policy, bf16 <-> fp32 conversion, and the
// two-level (warp shuffle, then CTA shared memory) sum.
//
// Prior art on the pages: 128-bit vector I/O and __shfl_xor_sync reductions
// ("GPU Kernel Suite (gks)", techniques list); XOR-shuffle reduction inside a
// wave followed by a shared-memory combine across waves, round-to-nearest-even
// bf16 packing, non-temporal output stores ("Pre-built kernel library guide",
// section 1.1 LayerNorm, algorithm and configuration constants, which RMSNorm
// shares); warp_sum / cta_sum and float22bfloat162_rn ("CUDA Authoring and
// Support APIs", CUDA helpers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- element types

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPerVec = 4;   // elements per 16-byte vector
  __device__ static __forceinline__ float to_f32(float v) { return v; }
};
template <> struct Elem<bf16> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }
};

// Unpack one 16-byte vector of T into fp32 values.
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack_word_bf16(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
  unpack_word_bf16(v.x, f[0], f[1]);
  unpack_word_bf16(v.y, f[2], f[3]);
  unpack_word_bf16(v.z, f[4], f[5]);
  unpack_word_bf16(v.w, f[6], f[7]);
}

// Pack fp32 values into one 16-byte vector; bf16 rounds to nearest even.
__device__ __forceinline__ uint4 pack(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
__device__ __forceinline__ uint32_t pack_word_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8]) {
  return make_uint4(pack_word_bf16(f[0], f[1]), pack_word_bf16(f[2], f[3]),
                    pack_word_bf16(f[4], f[5]), pack_word_bf16(f[6], f[7]));
}

__device__ __forceinline__ float round_to(float v, float*) { return v; }
__device__ __forceinline__ float round_to(float v, bf16*) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// ---------------------------------------------------------------- global memory

// Streaming read of data that this kernel never writes: read-only path, no L1
// allocation (each byte is used once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
// Read of data that this kernel later overwrites (the fused-add residual):
// coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_rw(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
// Read of small data every CTA re-reads (gamma): cached in L1.
__device__ __forceinline__ uint4 ld_cached(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
// Streaming write: evict-first in L2, the output is not re-read by this kernel.
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// A 16-byte shared-memory read the compiler may not merge with an earlier
// read of the same address (so the earlier value need not stay live).
__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return v;
}

// The 16 bytes that start s bytes (0 <= s < 16) into the 32-byte pair
// (lo, hi) of consecutive aligned chunks.  Words are picked by the two bits of
// s / 4 (selects, no indexing of a register array) and bytes by one byte
// permute per word; s == 0 gives lo.
__device__ __forceinline__ uint4 realign_pair(const uint4& lo, const uint4& hi, int s) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const int q = s >> 2;
  uint32_t t[6], u[5];
#pragma unroll
  for (int i = 0; i < 6; ++i) t[i] = (q & 2) ? w[i + 2] : w[i];
#pragma unroll
  for (int i = 0; i < 5; ++i) u[i] = (q & 1) ? t[i + 1] : t[i];
  const uint32_t sel = 0x3210u + 0x1111u * (uint32_t)(s & 3);
  return make_uint4(__byte_perm(u[0], u[1], sel), __byte_perm(u[1], u[2], sel),
                    __byte_perm(u[2], u[3], sel), __byte_perm(u[3], u[4], sel));
}

template <typename T>
__device__ __forceinline__ float ld_scalar(const T* p) {
  return Elem<T>::to_f32(*p);
}
// Scalar read of small read-only data (gamma), cached in L1.
template <typename T>
__device__ __forceinline__ float ld_scalar_ro(const T* p) {
  return Elem<T>::to_f32(__ldg(p));
}
__device__ __forceinline__ void st_scalar(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_scalar(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// An empty asm that claims to change v: the compiler must unpack v (or
// recompute what it feeds) again where it is used, instead of keeping fp32
// values derived from it live across a row's reductions or hoisting them out
// of the row loop -- which would cost registers and resident CTAs.
__device__ __forceinline__ uint4 opaque(uint4 v) {
  asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
  return v;
}

// ---------------------------------------------------------------- launch order

// Programmatic dependent launch: every kernel of the library is launched so
// that it may start while the previous kernel on the stream is finishing.
// Its first act is to wait until that kernel has completed and its writes are
// visible (no global memory is touched before), and then to allow the next
// kernel to launch the same way.  Without the launch attribute both
// instructions do nothing.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- reductions

// Sum over aligned groups of G consecutive lanes (G a power of two <= 32).
// Every lane of the warp must execute it; each lane receives its group's sum,
// combined in the same order for every lane of the group.
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// CTA-wide sum of K values per thread.  red: shared scratch of at least
// 2 * K * 32 floats; `parity` alternates between consecutive calls so one
// barrier per call suffices (a warp cannot re-enter the same half before every
// warp has left the previous call).  Every thread gets the same totals: the
// warp partials are added in warp order by every thread.
template <int K>
__device__ __forceinline__ void cta_sum(float (&v)[K], float* red, int parity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = group_sum<32>(v[k]);
  float* buf = red + parity * (K * 32);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) buf[k * 32 + warp] = v[k];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += buf[k * 32 + w];
    v[k] = s;
  }
}

// cta_sum whose barrier also takes a vote: returns true in every thread when
// `pred` is true in any thread (so a decision based on it is CTA-uniform).
template <int K>
__device__ __forceinline__ bool cta_sum_vote(float (&v)[K], float* red, int parity, bool pred) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = group_sum<32>(v[k]);
  float* buf = red + parity * (K * 32);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) buf[k * 32 + warp] = v[k];
  }
  const bool any = __syncthreads_or(pred ? 1 : 0) != 0;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += buf[k * 32 + w];
    v[k] = s;
  }
  return any;
}

// ---------------------------------------------------------------- bulk copies

// 1-D bulk copies global -> shared (the non-tensor form of TMA) completing on
// an mbarrier, and bounded waits on that barrier.  Every wait gives up after
// `limit` SM clock cycles and reports it, so no kernel can spin forever.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy accesses of shared memory before
// later bulk copies into it (the stage being refilled was just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and expect `bytes` of bulk-copy data on the barrier.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global
// to shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Ask for `bytes` of global memory (address 16-byte aligned, size a multiple
// of 16) to be brought into L2 ahead of use: a hint served by the bulk-copy
// unit, with nothing to wait for and no registers held.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Rows [first, first + rows) of a row-major array with rows of rb bytes
// (16-byte aligned), clipped to its M rows, requested into L2.
__device__ __forceinline__ void l2_prefetch_rows(const void* a, int64_t first, int64_t rows,
                                                 int64_t M, size_t rb) {
  if (first >= M) return;
  const int64_t n = M - first < rows ? M - first : rows;
  bulk_prefetch_l2(static_cast<const char*>(a) + first * rb, (uint32_t)(n * rb));
}

// Before a kernel waits for the previous one (pdl_begin), thread 0 may ask
// for the first rows the CTA will read to be brought into L2.  A prefetch
// returns nothing to the program, and L2 is where every write of the
// previous kernel lands, so reads after the wait still see those writes: the
// request only starts the DRAM traffic of the CTA's first rows while the
// previous kernel's last CTAs finish.  Rows [first, first + n) of up to three
// row-major operands with rows of rb bytes (16-byte aligned; null operands
// skipped), clipped to M rows.
__device__ __forceinline__ void l2_warm(const void* a, const void* b, const void* c,
                                        int64_t first, int64_t n, int64_t M, size_t rb) {
  if (threadIdx.x != 0) return;
  if (a) l2_prefetch_rows(a, first, n, M, rb);
  if (b) l2_prefetch_rows(b, first, n, M, rb);
  if (c) l2_prefetch_rows(c, first, n, M, rb);
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Potentially blocking test: the thread may be suspended up to about
// `hint_ns` nanoseconds waiting for the phase to complete.
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete; false once `limit`
// SM clock cycles have passed without completion (limit 0: only test once;
// limit < 0: give up at once without testing, so that every wait runs out --
// the deterministic form of the timeout path for tests).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit) {
  if (limit < 0) return false;
  if (mbar_test(bar, parity)) return true;
  if (limit <= 0) return false;
  const long long t0 = clock64();
  do {
    if (mbar_try(bar, parity, 2000u)) return true;
  } while (clock64() - t0 <= limit);
  return false;
}

}  // namespace rmsn
