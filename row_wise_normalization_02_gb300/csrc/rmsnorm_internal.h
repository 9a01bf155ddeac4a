// Internal interface between the kernel translation units and the C ABI /
// dispatch layer.  Nothing here is exported from the shared library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

enum DT : int { kF32 = 0, kBF16 = 1 };

// Kernel families.
//  kSubwarp : G (<= 32) lanes per row, several rows per 256-thread CTA,
//             reduction by shuffles only; rows must be 16-byte aligned.
//  kCta     : one row per CTA (blockDim chosen per N), row held in registers,
//             reduction by shuffles + shared memory; rows 16-byte aligned.
//  kRagged  : as kCta, for rows that are not 16-byte aligned (N * size % 16
//             != 0, or unaligned bases that agree modulo 16): per-row scalar
//             head and tail around an aligned vector body; each CTA walks
//             rows of one start-alignment class, so gamma and the dgamma
//             partials stay in registers.
//  kGeneric : any N, any element-aligned pointers; scalar two-pass loop.
//  kStaged  : as kCta, but rows arrive by bulk copies (the 1-D form of TMA)
//             into a ring of `stages` shared-memory row buffers, so several
//             rows per CTA are in flight independently of register pressure.
//  kCluster : one row per thread-block cluster of 2-8 CTAs, each CTA owning a
//             contiguous slice of `slice` vectors of every row (forward: in
//             registers; backward: through a bulk-copy ring); the CTAs' sums
//             meet in distributed shared memory.  For rows too long for one
//             CTA; rows 16-byte aligned.
//  kWide    : any N, any element-aligned pointers (backward: rows a multiple
//             of 16 bytes, the dgamma partial row in shared memory); two
//             passes of 16-byte vectors per row, each pass in the frame of one
//             operand's alignment with the others realigned to it.
enum Family : int { kSubwarp = 0, kCta = 1, kRagged = 2, kGeneric = 3, kStaged = 4,
                    kCluster = 5, kWide = 6 };

// Forward output kinds: y in the activation dtype, FP8 E4M3 codes with one
// scale per row, or NVFP4 (E2M1 codes, an E4M3 scale per 16 elements).
enum OutKind : int { kOutDtype = 0, kOutFp8 = 1, kOutNvfp4 = 2 };

// Shared-memory header of the staged kernels: barriers, reduction scratch
// and the error flag; the ring of row buffers starts after it.
constexpr int kStagedMaxStages = 8;
// Status bits a kernel may raise in the library's device status word.
constexpr unsigned kStatusWaitTimeout = 1u;
constexpr int kStagedHeader = 1024;

struct FwdParams {
  const void* x;
  void* residual;     // fused add only: in r, out h
  const void* gamma;
  void* y;
  float* rstd;        // may be null
  int64_t M;
  int N;
  int nvec;           // 16-byte vectors per row (aligned families)
  float eps;
  float inv_n;
  int stages;         // kStaged: row buffers in the shared-memory ring
  long long wait_limit;   // kStaged: clock cycles before a wait gives up
  unsigned* status;   // device status word (kStatus* bits)
  int period;         // kRagged: rows i and i + period start at the same address mod 16
  // strided rows (per-head q/k norm): row i = (t, h) = (i / heads, i % heads)
  // starts at element t * x_st + h * x_sh of x and t * y_st + h * y_sh of y
  int64_t heads;
  int64_t x_st, x_sh, y_st, y_sh;
  // quantised outputs: y holds the codes (E4M3 bytes, or E2M1 pairs), qs the
  // scales (fp32 per row for E4M3; E4M3 per 16 elements for NVFP4), gs the
  // NVFP4 global scale
  void* qs;
  float gs;
  int l2_rows;        // register kernels: rows of the CTA's walk fetched into L2
                      // this many iterations ahead (0: none)
  int slice;          // kCluster: vectors of each row per CTA of the cluster
  int x_shift;        // kRagged with mixed alignment: bytes (mod 16) by which x's
                      // rows start past the output's (y, or h for the fused add)
};

struct BwdParams {
  const void* dy;
  const void* x;
  const void* dres;   // fused-add backward: gradient reaching h on the residual path
                      // (dx then holds dx + dres, and may be the same buffer)
  const float* rstd;  // null: recompute from x and eps
  const void* gamma;
  void* dx;
  float* partial;     // [gridDim.x][ld_partial] fp32 dgamma partials, or null
  int64_t M;
  int N;
  int nvec;
  int ld_partial;     // row stride of partial, a multiple of 4 floats
  float eps;
  float inv_n;
  int stages;
  long long wait_limit;
  unsigned* status;
  int period;
  int l2_rows;        // register kernels: L2 lookahead in iterations (0: none)
  int slice;          // kCluster: vectors of each row per CTA of the cluster
  int x_shift;        // kRagged with mixed alignment: bytes (mod 16) by which the
  int dy_shift;       //   rows of x and of dy start past those of dx
};

// LayerNorm (forward and backward).
struct LnParams {
  const void* x;
  const void* dy;       // backward only
  const void* gamma;
  const void* beta;     // forward: may be null (no shift)
  void* y;              // forward: y; backward: dx
  float* mean;          // forward: optional outputs; backward: the saved
  float* rstd;          //   statistics (both given) or null (recomputed)
  float* partial;       // backward: [gridDim.x][2 * ld_half] fp32, [dgamma | dbeta]
  int64_t M;
  int N;
  int nvec;
  int ld_half;          // a multiple of 4 floats, >= N
  float eps;
  float inv_n;
  int stages;           // staged backward: row buffers in the shared-memory ring
  long long wait_limit; // staged backward: clock cycles before a wait gives up
  unsigned* status;     // device status word (kStatus* bits)
  int l2_rows;          // register kernels: rows of the CTA's walk fetched into L2
                        // this many iterations ahead (0: none)
};

using FwdKernel = void (*)(FwdParams);
using BwdKernel = void (*)(BwdParams);
// Stage 2 of every backward: column sums of the P x nq float4 partial rows
// (row stride nq float4), in a fixed order.  Float4 columns [0, half_q) go to
// out0 and [half_q, 2 half_q) to out1 (the LayerNorm backward's dgamma and
// dbeta); N valid columns per output; out0 in bf16 (rounded once) when bf16.
struct ColSumOut {
  void* out0;
  void* out1;
  int half_q;
  int N;
  int bf16;
};
using ColSumKernel = void (*)(const float*, int, int, ColSumOut);

struct FwdKey {
  int xd, wd;
  int family;
  int g;         // lanes per row (kSubwarp)
  int vpt;       // 16-byte vectors per thread
  bool fused;
  bool prefetch; // issue the next row's loads before reducing the current row
  bool strided;  // rows addressed through (heads, x_st, x_sh, y_st, y_sh)
  int out = kOutDtype;   // output kind (kOut*)
  bool mix = false;      // kRagged: x need not share the output's alignment
};

struct BwdKey {
  int xd, wd;
  int family;
  int g;
  int vpt;
  bool has_rstd;
  bool acc_smem; // kCta: dgamma partials in shared memory instead of registers
  bool prefetch;
  bool dres;     // fused-add backward (adds the residual-path gradient)
  bool mix = false;   // kRagged: x and dy need not share dx's alignment
};

// Kernel for a key, or nullptr when that instantiation does not exist.  Each
// dtype pair is instantiated in its own translation unit.
FwdKernel get_fwd_kernel_f32_f32(const FwdKey& k);
FwdKernel get_fwd_kernel_bf16_bf16(const FwdKey& k);
FwdKernel get_fwd_kernel_bf16_f32(const FwdKey& k);
BwdKernel get_bwd_kernel_f32_f32(const BwdKey& k);
BwdKernel get_bwd_kernel_bf16_bf16(const BwdKey& k);
BwdKernel get_bwd_kernel_bf16_f32(const BwdKey& k);
FwdKernel get_fwd_staged_f32_f32(const FwdKey& k);
FwdKernel get_fwd_staged_bf16_bf16(const FwdKey& k);
FwdKernel get_fwd_staged_bf16_f32(const FwdKey& k);
BwdKernel get_bwd_staged_f32_f32(const BwdKey& k);
BwdKernel get_bwd_staged_bf16_bf16(const BwdKey& k);
BwdKernel get_bwd_staged_bf16_f32(const BwdKey& k);
FwdKernel get_fwd_ragged_f32_f32(const FwdKey& k);
FwdKernel get_fwd_ragged_bf16_bf16(const FwdKey& k);
FwdKernel get_fwd_ragged_bf16_f32(const FwdKey& k);
BwdKernel get_bwd_ragged_f32_f32(const BwdKey& k);
BwdKernel get_bwd_ragged_bf16_bf16(const BwdKey& k);
BwdKernel get_bwd_ragged_bf16_f32(const BwdKey& k);
FwdKernel get_fwd_ragged_mix_f32_f32(const FwdKey& k);
FwdKernel get_fwd_ragged_mix_bf16_bf16(const FwdKey& k);
FwdKernel get_fwd_ragged_mix_bf16_f32(const FwdKey& k);
BwdKernel get_bwd_ragged_mix_f32_f32(const BwdKey& k);
BwdKernel get_bwd_ragged_mix_bf16_bf16(const BwdKey& k);
BwdKernel get_bwd_ragged_mix_bf16_f32(const BwdKey& k);
FwdKernel get_fwd_cluster_f32_f32(const FwdKey& k);
FwdKernel get_fwd_cluster_bf16_bf16(const FwdKey& k);
FwdKernel get_fwd_cluster_bf16_f32(const FwdKey& k);
BwdKernel get_bwd_cluster_f32_f32(const BwdKey& k);
BwdKernel get_bwd_cluster_bf16_bf16(const BwdKey& k);
BwdKernel get_bwd_cluster_bf16_f32(const BwdKey& k);
FwdKernel get_fwd_wide_f32_f32(const FwdKey& k);
FwdKernel get_fwd_wide_bf16_bf16(const FwdKey& k);
FwdKernel get_fwd_wide_bf16_f32(const FwdKey& k);
BwdKernel get_bwd_wide_f32_f32(const BwdKey& k);
BwdKernel get_bwd_wide_bf16_bf16(const BwdKey& k);
BwdKernel get_bwd_wide_bf16_f32(const BwdKey& k);
FwdKernel get_fwd_quant_f32_f32(const FwdKey& k);
FwdKernel get_fwd_quant_bf16_bf16(const FwdKey& k);
FwdKernel get_fwd_quant_bf16_f32(const FwdKey& k);
// Column sum with C float4 columns per 256-thread CTA (C = 8, 16 or 32).
ColSumKernel get_colsum_kernel(int c);

using LnKernel = void (*)(LnParams);
struct LnKey {
  int xd, wd;
  int family;    // kSubwarp, kCta or kGeneric
  int g, vpt;
  bool bwd;
  bool prefetch;
  bool saved = false;   // kWide backward: mean and rstd given (rows pipelined)
};
LnKernel get_ln_kernel_f32_f32(const LnKey& k);
LnKernel get_ln_kernel_bf16_bf16(const LnKey& k);
LnKernel get_ln_kernel_bf16_f32(const LnKey& k);
LnKernel get_ln_wide_f32_f32(const LnKey& k);
LnKernel get_ln_wide_bf16_bf16(const LnKey& k);
LnKernel get_ln_wide_bf16_f32(const LnKey& k);

// Threads per CTA of the subwarp families; upper bound of the per-row CTAs.
constexpr int kSubwarpThreads = 256;
constexpr int kCtaMaxThreads = 512;
// Most threads of a kWide CTA, built for two CTAs per SM (64 registers a
// thread).
constexpr int kWideThreads = 512;
constexpr int kWideBwdThreads = 512;
// Most threads of the wide LayerNorm backward with saved statistics, whose
// fused passes of two rows take 80 registers a thread at two CTAs per SM.
constexpr int kLnSavedThreads = 384;

// Threads of a stage-2 (column sum) CTA.
constexpr int kColSumThreads = 256;

}  // namespace rmsn
