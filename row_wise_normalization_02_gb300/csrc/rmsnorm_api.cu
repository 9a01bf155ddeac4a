// C ABI of the RMSNorm library: argument validation, the per-(op, dtype, N)
// dispatch table, grid sizing and launches.  No kernels live here.
//
// Dispatch (aligned rows = every base pointer 16-byte aligned and N * size a
// multiple of 16 bytes; E = elements per 16-byte vector; make_plan has the
// measured reasons):
//   N / E <= 128        kSubwarp  G lanes per row (4..32), VPT vectors per lane,
//                                 several rows per 256-thread CTA; the short-row
//                                 packing idea of the softmax kernel's
//                                 THREADS_PER_ROW / ROWS_PER_BLOCK knobs
//                                 ("Pre-built kernel library guide", 2.1); the
//                                 backward of 65-96 vectors through kStaged
//   N / E <= 2048/4096  kCta      one row per CTA of ceil(N / E / VPT) threads,
//                                 row in registers (backward: kStaged, rows by
//                                 bulk copies into a shared-memory ring)
//   longer              kCluster  one row per thread-block cluster
// Rows off 16 bytes whose operands agree modulo 16 bytes, and inputs off the
// outputs' alignment, take kRagged (its mixed form) or, for the backward,
// kStaged's mixed form; what none of these takes goes to kWide (two passes of
// 16-byte vectors, each operand realigned to the pass's frame) and, where
// that does not apply either, kGeneric.  Grids are persistent: min(rows, SMs
// x resident CTAs per SM).
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/rmsnorm.h"
#include "rmsnorm_internal.h"
#include "rmsnorm_wide_layout.h"

namespace rmsn {
namespace {

constexpr int64_t kMaxN = int64_t(1) << 30;
constexpr int kRaggedMaxN = 24576;
// Shared memory of a staged CTA: aim for two CTAs per SM, allow one.
constexpr int64_t kStagedSmemBudget = 110 * 1024;
constexpr int64_t kStagedSmemMax = 226 * 1024;
constexpr long long kDefaultWaitLimit = 1LL << 32;   // clock cycles (about 2 s)

int esize(int dt) { return dt == kF32 ? 4 : 2; }
int per_vec(int dt) { return 16 / esize(dt); }

bool dtype_pair_ok(int xd, int wd) {
  return (xd == kF32 && wd == kF32) || (xd == kBF16 && (wd == kBF16 || wd == kF32));
}

FwdKernel fwd_kernel(const FwdKey& k) {
  if (k.out != kOutDtype) {
    if (k.xd == kF32 && k.wd == kF32) return get_fwd_quant_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16) return get_fwd_quant_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32) return get_fwd_quant_bf16_f32(k);
    return nullptr;
  }
  if (k.family == kRagged) {
    if (k.xd == kF32 && k.wd == kF32)
      return k.mix ? get_fwd_ragged_mix_f32_f32(k) : get_fwd_ragged_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16)
      return k.mix ? get_fwd_ragged_mix_bf16_bf16(k) : get_fwd_ragged_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32)
      return k.mix ? get_fwd_ragged_mix_bf16_f32(k) : get_fwd_ragged_bf16_f32(k);
    return nullptr;
  }
  if (k.family == kWide) {
    if (k.xd == kF32 && k.wd == kF32) return get_fwd_wide_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16) return get_fwd_wide_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32) return get_fwd_wide_bf16_f32(k);
    return nullptr;
  }
  if (k.family == kCluster) {
    if (k.xd == kF32 && k.wd == kF32) return get_fwd_cluster_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16) return get_fwd_cluster_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32) return get_fwd_cluster_bf16_f32(k);
    return nullptr;
  }
  const bool st = k.family == kStaged;
  if (k.xd == kF32 && k.wd == kF32) return st ? get_fwd_staged_f32_f32(k) : get_fwd_kernel_f32_f32(k);
  if (k.xd == kBF16 && k.wd == kBF16)
    return st ? get_fwd_staged_bf16_bf16(k) : get_fwd_kernel_bf16_bf16(k);
  if (k.xd == kBF16 && k.wd == kF32)
    return st ? get_fwd_staged_bf16_f32(k) : get_fwd_kernel_bf16_f32(k);
  return nullptr;
}
BwdKernel bwd_kernel(const BwdKey& k) {
  if (k.family == kRagged) {
    if (k.xd == kF32 && k.wd == kF32)
      return k.mix ? get_bwd_ragged_mix_f32_f32(k) : get_bwd_ragged_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16)
      return k.mix ? get_bwd_ragged_mix_bf16_bf16(k) : get_bwd_ragged_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32)
      return k.mix ? get_bwd_ragged_mix_bf16_f32(k) : get_bwd_ragged_bf16_f32(k);
    return nullptr;
  }
  if (k.family == kWide) {
    if (k.xd == kF32 && k.wd == kF32) return get_bwd_wide_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16) return get_bwd_wide_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32) return get_bwd_wide_bf16_f32(k);
    return nullptr;
  }
  if (k.family == kCluster) {
    if (k.xd == kF32 && k.wd == kF32) return get_bwd_cluster_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16) return get_bwd_cluster_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32) return get_bwd_cluster_bf16_f32(k);
    return nullptr;
  }
  const bool st = k.family == kStaged && k.g == 0;   // staged short rows live with the others
  if (k.xd == kF32 && k.wd == kF32) return st ? get_bwd_staged_f32_f32(k) : get_bwd_kernel_f32_f32(k);
  if (k.xd == kBF16 && k.wd == kBF16)
    return st ? get_bwd_staged_bf16_bf16(k) : get_bwd_kernel_bf16_bf16(k);
  if (k.xd == kBF16 && k.wd == kF32)
    return st ? get_bwd_staged_bf16_f32(k) : get_bwd_kernel_bf16_f32(k);
  return nullptr;
}

// ---------------------------------------------------------------- status word

// Bits raised by kernels (kStatusWaitTimeout: a bounded wait gave up).  Read
// and cleared by rmsnorm_check_device.  Its device address is looked up once
// per device: in host code the name is only a host-side stand-in.
static __device__ unsigned int g_device_status;

// ---------------------------------------------------------------- errors

// Text of the last CUDA failure seen by this thread's calls into the library.
thread_local char g_last_error[256] = "";

rmsnorm_status_t cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorString(e),
           cudaGetErrorName(e));
  return RMSNORM_ERR_CUDA;
}

// ---------------------------------------------------------------- device info

struct DevInfo {
  int sms = 0;
  int max_smem_optin = 0;
  unsigned* status = nullptr;
};

std::mutex g_mu;
DevInfo g_dev[64];

cudaError_t device_info(int device, DevInfo* out) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev[device].sms == 0) {
    int sms = 0, smem = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    void* st = nullptr;
    e = cudaGetSymbolAddress(&st, g_device_status);
    if (e != cudaSuccess) return e;
    g_dev[device].sms = sms;
    g_dev[device].max_smem_optin = smem;
    g_dev[device].status = static_cast<unsigned*>(st);
  }
  *out = g_dev[device];
  return cudaSuccess;
}

// Dynamic shared memory limit of each (kernel, device): the attribute is a
// maximum, so it is only ever raised, to the largest size any launch of that
// kernel has needed (lowering it for a smaller launch would break a later,
// larger launch whose occupancy is already cached).
struct SmemEntry {
  const void* fn;
  int device, limit;
};
SmemEntry g_smem[256];
int g_nsmem = 0;

cudaError_t ensure_smem(const void* fn, int device, int smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  std::lock_guard<std::mutex> lk(g_mu);
  SmemEntry* ent = nullptr;
  for (int i = 0; i < g_nsmem; ++i)
    if (g_smem[i].fn == fn && g_smem[i].device == device) ent = &g_smem[i];
  if (ent && ent->limit >= smem) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (ent) ent->limit = smem;
  else if (g_nsmem < 256) g_smem[g_nsmem++] = SmemEntry{fn, device, smem};
  return cudaSuccess;
}

// Resident CTAs per SM of (kernel, threads, smem) -- or, for a cluster size
// > 0, clusters of that size the whole device holds at once -- cached.
struct OccEntry {
  const void* fn;
  int device, threads, smem, cluster, blocks;
};
OccEntry g_occ[512];
int g_nocc = 0;

cudaError_t occupancy(const void* fn, int device, int threads, int smem, int* blocks,
                      int cluster = 0) {
  cudaError_t e = ensure_smem(fn, device, smem);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_nocc; ++i)
    if (g_occ[i].fn == fn && g_occ[i].device == device && g_occ[i].threads == threads &&
        g_occ[i].smem == smem && g_occ[i].cluster == cluster) {
      *blocks = g_occ[i].blocks;
      return cudaSuccess;
    }
  int b = 0;
  if (cluster > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&b, fn, &cfg);
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem);
  }
  if (e != cudaSuccess) return e;
  if (b < 1) return cudaErrorInvalidConfiguration;
  if (g_nocc < 512) g_occ[g_nocc++] = OccEntry{fn, device, threads, smem, cluster, b};
  *blocks = b;
  return cudaSuccess;
}

// ---------------------------------------------------------------- plans

enum Op { kFwd = 0, kFused = 1, kBwd = 2, kFusedBwd = 3 };

struct Plan {
  int family = kGeneric;
  int g = 0, vpt = 0;
  bool prefetch = false, acc_smem = false;
  int threads = 256;
  int smem = 0;
  int stages = 0;            // kStaged: ring of row buffers
  int rows_per_cta = 1;      // rows one CTA iteration covers
  int min_rows = 0;          // backward: rows per CTA at least this many (bounds
                             // the dgamma partial rows), unless below 1 CTA/SM
  int period = 1;            // kRagged: the grid is a multiple of it
  bool mix = false;          // kRagged: inputs off the outputs' alignment
  int cta_per_sm_cap = 0;    // 0: occupancy limit
  int l2_ahead = 0;          // LayerNorm register kernels: L2 lookahead in iterations
  int cluster = 0;           // kCluster: CTAs per cluster (one row per cluster)
  int slice = 0;             // kCluster: vectors of each row per CTA
  int64_t ahead_bytes = 0;   // kWide: input bytes of one row of every CTA's walk,
                             // per grid CTA (sizes the L2 lookahead once the grid
                             // is known; 0: lookahead as set)
  const void* fn = nullptr;
  FwdKernel fwd = nullptr;
  BwdKernel bwd = nullptr;
  int grid = 0;
};

int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Subwarp shape for nvec 16-byte vectors per row.
void subwarp_shape(int nvec, int* g, int* vpt) {
  if (nvec <= 4) { *g = 4; *vpt = 1; }
  else if (nvec <= 8) { *g = 8; *vpt = 1; }
  else if (nvec <= 16) { *g = 8; *vpt = 2; }
  else if (nvec <= 32) { *g = 16; *vpt = 2; }
  else if (nvec <= 64) { *g = 32; *vpt = 2; }
  else if (nvec <= 96) { *g = 32; *vpt = 3; }
  else { *g = 32; *vpt = 4; }
}

// Vectors per thread for a row of nvec vectors in one CTA, and the CTA size.
// op kQuantFwd: the quantised forwards, whose longer epilogues are best with
// more vectors per thread (measured at 16384 x 8192 and 32768 x 4096 bf16).
constexpr int kQuantFwd = 100;
bool cta_shape(int op, int nvec, int* vpt, int* threads) {
  // forward and fused add: 4 vectors per thread first -- with the bf16
  // arithmetic done from the packed words (62 registers at VPT 4 with
  // prefetch, four 256-thread CTAs per SM) this beats VPT 2 / 512 threads
  // (16384 x 8192 forward 0.96 vs 0.90, 32768 x 4096 fused add 0.98 vs 0.95)
  static const int pref_fwd[] = {4, 2, 8, 1};
  static const int pref_fused[] = {4, 2, 1, 8};
  static const int pref_bwd[] = {4, 2, 1, 8};
  static const int pref_qfwd[] = {4, 2, 8, 1};
  const int* pref = op == kFwd ? pref_fwd : op == kFused ? pref_fused
                  : op == kQuantFwd ? pref_qfwd : pref_bwd;
  for (int i = 0; i < 4; ++i) {
    const int v = pref[i];
    const int t = round_up((nvec + v - 1) / v, 32);
    if (t >= 64 && t <= kCtaMaxThreads) {
      *vpt = v;
      *threads = t;
      return true;
    }
  }
  // very short rows: smallest CTA
  if (nvec <= 64) {
    *vpt = 1;
    *threads = 64;
    return true;
  }
  return false;
}

// Cluster shape for a row of nvec vectors: the fewest CTAs (2, 4 or 8) whose
// slices hold at most 2048 vectors (4 per thread, up to 512 threads) -- fewer
// CTAs per row exchange less and pack better into the GPCs (2048 x 65536
// bf16: forward 0.91 of the copy peak with 4 CTAs of 2048 vectors against
// 0.86 with 8 of 1024; backward 0.77 against 0.52) -- or, forward only, 8
// CTAs with up to 4096 vectors (8 per thread, no next-row prefetch).  cl > 0
// fixes the cluster size.  False when the row is too long.
bool cluster_shape(bool bwd, int nvec, int cl, int* c_out, int* slice, int* vpt, int* threads) {
  int c = cl;
  if (c <= 0)
    for (c = 2; c < 8 && (nvec + c - 1) / c > 2048; c *= 2) {
    }
  if (c < 1 || c > 8) return false;
  const int sl = (nvec + c - 1) / c;
  const int v = sl <= 2048 ? 4 : 8;
  if (v == 8 && bwd) return false;
  const int t = round_up((sl + v - 1) / v, 32);
  if (t > kCtaMaxThreads) return false;
  *c_out = c;
  *slice = sl;
  *vpt = v;
  *threads = t < 64 ? 64 : t;
  return true;
}

// Vectors a ragged CTA of `threads` holds at `vpt` per thread: 32 per warp
// and slot, 31 with mixed alignment (lane 31 carries the next warp's chunk).
int64_t ragged_capacity(int threads, int vpt, bool mix) {
  return (int64_t)(threads / 32) * (mix ? 31 : 32) * vpt;
}

// Vectors per thread (1, 2 or 4) and CTA size for a ragged row of at most
// nvec vectors; false when the row needs more than 4 vectors x 512 threads.
bool ragged_shape(int nvec, bool mix, int* vpt, int* threads) {
  static const int pref[] = {2, 4, 1};
  const int per_warp = mix ? 31 : 32;
  for (int i = 0; i < 3; ++i) {
    const int v = pref[i];
    int t = 32 * ((nvec + per_warp * v - 1) / (per_warp * v));
    if (t < 64) t = 64;
    if (t <= kCtaMaxThreads) {
      *vpt = v;
      *threads = t;
      return true;
    }
  }
  return false;
}

// Rows i and i + P start at the same address modulo 16 for a row of `bytes`:
// P = 16 / gcd(bytes, 16).
int ragged_period(int64_t bytes) {
  int g = 1;
  while (g < 16 && bytes % (2 * g) == 0) g *= 2;
  return 16 / g;
}

// Debug and A/B knobs, read from the environment once when the library is
// loaded and again only by rmsnorm_reload_debug_env -- never on the launch
// path:
//  RMSNORM_FORCE_VARIANT="family[:key=value...]" with family one of subwarp,
//    cta, ragged, generic, staged, cluster and keys g, vpt, t (threads), pf
//    (0/1), acc (0/1 shared-memory dgamma partials), cps (CTAs per SM cap),
//    st (stages), mr (backward: minimum rows per CTA, 0 = none), l2 (L2
//    lookahead), cl (CTAs per cluster).  For profiling A/B runs; a forced
//    variant that cannot serve the call is an argument error.
//  RMSNORM_WAIT_LIMIT_CYCLES: clock cycles a bulk-copy wait lasts before it
//    gives up (a test knob; a negative value makes every wait give up at
//    once), else about 2 s.
//  RMSNORM_NO_PDL=1: launch without programmatic dependent launch.
struct Force {
  bool on = false;
  int family = -1, g = 0, vpt = 0, threads = 0, pf = -1, acc = -1, cps = 0, st = 0, mr = -1,
      l2 = -1, cl = 0;
};

struct DebugEnv {
  Force force;
  long long wait_limit = kDefaultWaitLimit;
  bool no_pdl = false;
};

Force parse_force(const char* s) {
  Force f;
  if (!s || !*s) return f;
  f.on = true;
  char buf[128];
  strncpy(buf, s, sizeof buf - 1);
  buf[sizeof buf - 1] = 0;
  char* save = nullptr;
  char* tok = strtok_r(buf, ":", &save);
  if (!tok) return f;
  if (!strcmp(tok, "subwarp")) f.family = kSubwarp;
  else if (!strcmp(tok, "cta")) f.family = kCta;
  else if (!strcmp(tok, "ragged")) f.family = kRagged;
  else if (!strcmp(tok, "generic")) f.family = kGeneric;
  else if (!strcmp(tok, "staged")) f.family = kStaged;
  else if (!strcmp(tok, "cluster")) f.family = kCluster;
  else if (!strcmp(tok, "wide")) f.family = kWide;
  while ((tok = strtok_r(nullptr, ":", &save))) {
    char* eq = strchr(tok, '=');
    if (!eq) continue;
    *eq = 0;
    const int v = atoi(eq + 1);
    if (!strcmp(tok, "g")) f.g = v;
    else if (!strcmp(tok, "vpt")) f.vpt = v;
    else if (!strcmp(tok, "t")) f.threads = v;
    else if (!strcmp(tok, "pf")) f.pf = v;
    else if (!strcmp(tok, "acc")) f.acc = v;
    else if (!strcmp(tok, "cps")) f.cps = v;
    else if (!strcmp(tok, "st")) f.st = v;
    else if (!strcmp(tok, "mr")) f.mr = v;
    else if (!strcmp(tok, "l2")) f.l2 = v;
    else if (!strcmp(tok, "cl")) f.cl = v;
  }
  return f;
}

DebugEnv read_debug_env() {
  DebugEnv e;
  e.force = parse_force(getenv("RMSNORM_FORCE_VARIANT"));
  const char* w = getenv("RMSNORM_WAIT_LIMIT_CYCLES");
  if (w && *w) e.wait_limit = atoll(w);
  const char* off = getenv("RMSNORM_NO_PDL");
  e.no_pdl = off && *off && *off != '0';
  return e;
}

// Initialised when the library is loaded; replaced by rmsnorm_reload_debug_env.
DebugEnv g_env = read_debug_env();

const Force& read_force() { return g_env.force; }
long long wait_limit() { return g_env.wait_limit; }

// kWide: the backward keeps its dgamma partial row (N columns, laid out in
// groups of 32 vectors with the head and tail of dx's split beside them) in
// shared memory, and needs dx's split to be the same for every row.
int64_t wide_smem(int N, int xd) { return wide_acc_floats(N, per_vec(xd)) * 4LL; }
bool wide_ok(bool bwd, int N, int xd) {
  return !bwd || (((int64_t)N * esize(xd)) % 16 == 0 && wide_smem(N, xd) <= kStagedSmemMax);
}
// Threads of a wide CTA: about two vectors of the row per thread, from 64 to
// 256 for the forward (four CTAs per SM beat two of 512 threads: 32768 x 4096
// bf16 fused add with y off the residual 0.93 of the copy peak against 0.62)
// and to 512 for the backward (its shared-memory dgamma row allows few CTAs
// per SM).
int wide_threads(bool bwd, int N, int E) {
  const int t = round_up((N / E + 2) / 2, 32), cap = bwd ? kWideBwdThreads : 256;
  return t < 64 ? 64 : (t > cap ? cap : t);
}
// Bytes of input rows the grid of a wide kernel may have requested into L2
// ahead of its walk (8192 x 20000 bf16 forward, 608 CTAs: 0.75 of the copy
// peak without lookahead, 0.71 one step ahead, 0.60 two; 32768 x 4096 bf16
// fused add: 0.87 / 0.93 / 0.92; 8192 x 20000 backward, 304 CTAs: 0.58 /
// 0.55 / 0.49).
constexpr int64_t kWideAheadBudget = 12 << 20;

// Choose the variant.  aligned16: all base pointers 16-byte aligned;
// same_mod16: all activation base pointers agree modulo 16 bytes.
// mix_ok: the outputs agree modulo 16 (y with h over the residual; dx with
// dres) while an input (x, dy) need not -- the ragged kernels' mixed form;
// frame16: the outputs and gamma are moreover on 16 bytes.
rmsnorm_status_t make_plan(int op, int64_t M, int N, int xd, int wd, bool aligned16,
                           bool same_mod16, bool has_rstd, Plan* pl, bool mix_ok = false,
                           bool frame16 = false) {
  const bool bwd = op == kBwd || op == kFusedBwd;
  const bool dres = op == kFusedBwd;
  const int E = per_vec(xd);
  const bool rows_aligned = aligned16 && ((int64_t)N * esize(xd)) % 16 == 0;
  // inputs off the outputs' alignment while the outputs' rows (and gamma) lie
  // on 16 bytes: the backward's ring copies each input row's enclosing span
  const bool mixed_rows =
      !same_mod16 && mix_ok && frame16 && ((int64_t)N * esize(xd)) % 16 == 0;
  const int nvec = rows_aligned || mixed_rows ? N / E : 0;
  Plan p;
  if (rows_aligned && nvec <= 128) {
    p.family = kSubwarp;
    subwarp_shape(nvec, &p.g, &p.vpt);
    p.threads = kSubwarpThreads;
    p.rows_per_cta = kSubwarpThreads / p.g;
    p.prefetch = !(bwd && p.g == 32);   // full-warp rows: more CTAs beat prefetch
    if (op == kBwd && p.g == 32 && p.vpt == 3) {
      // rows of 65-96 vectors: the CTA's eight rows through a three-stage
      // bulk-copy ring rather than in registers (65536 x 768 bf16: 0.90 of
      // the copy peak against 0.83; the register form spills at two CTAs per
      // SM)
      p.family = kStaged;
      p.prefetch = false;
      p.stages = 3;
    }
  } else if (rows_aligned && bwd && nvec <= 4 * kCtaMaxThreads) {
    // backward: rows streamed by bulk copies, two stages, up to 4 vectors
    // per thread (the dgamma partials and gamma stay in registers)
    p.family = kStaged;
    if (!cta_shape(kBwd, nvec, &p.vpt, &p.threads) || p.vpt > 4) p.family = kGeneric;
    // the fused-add backward streams three rows per stage (dy, h, dres): one
    // more stage in flight pays for its longer epilogue (measured at
    // 32768 x 4096 bf16: 0.83 -> 1.0 of the copy bandwidth); the plain
    // backward is best at two
    p.stages = dres && kStagedHeader + 3 * 3 * (int64_t)N * esize(xd) <= kStagedSmemMax ? 3 : 2;
  } else if (rows_aligned && bwd) {
    // longer rows: one row per cluster, each CTA streaming its slice through
    // a two-stage bulk-copy ring
    p.family = kCluster;
    if (!cluster_shape(true, nvec, 0, &p.cluster, &p.slice, &p.vpt, &p.threads))
      p.family = kGeneric;
    // as many stages as fit one CTA per SM, at most three
    p.stages = (int)((kStagedSmemMax - kStagedHeader) / ((dres ? 3 : 2) * (int64_t)p.slice * 16));
    if (p.stages > 3) p.stages = 3;
    if (p.stages < 2) p.stages = 2;
  } else if (rows_aligned && nvec <= (op == kFwd ? 2048 : 4096)) {
    // one row per CTA; beyond 2048 vectors the forward does better on two-CTA
    // clusters (4096 x 32768 bf16: 0.92 of the copy peak against 0.84 at 8
    // vectors per thread), the fused add does not (0.93 against 0.95)
    p.family = kCta;
    if (!cta_shape(op, nvec, &p.vpt, &p.threads)) p.family = kGeneric;
    p.prefetch = op == kFwd ? p.vpt <= 4 : (op == kFused ? p.vpt != 2 && p.vpt <= 4 : p.vpt <= 2);
  } else if (rows_aligned) {
    // longer rows: one row per cluster, each CTA holding its slice in
    // registers with the next row's slice in flight
    p.family = kCluster;
    if (!cluster_shape(false, nvec, 0, &p.cluster, &p.slice, &p.vpt, &p.threads))
      p.family = kGeneric;
    p.prefetch = p.vpt <= 4;
  } else if (mixed_rows && bwd && nvec > 128 && nvec <= 4 * kCtaMaxThreads &&
             cta_shape(kBwd, nvec, &p.vpt, &p.threads) && p.vpt <= 4) {
    // as the aligned backward, the shifted inputs' rows arriving as their
    // enclosing 16-byte spans (4096 and 8192 bf16: see the measurements)
    p.family = kStaged;
    p.mix = true;
    p.stages = dres && kStagedHeader + 3 * 3 * ((int64_t)N * esize(xd) + 16) <= kStagedSmemMax
                   ? 3 : 2;
  } else if ((same_mod16 || mix_ok) && N <= kRaggedMaxN) {
    // rows off 16 bytes, or inputs off the outputs' alignment (x a view at an
    // odd element offset, say): vector body plus scalar head and tail
    p.family = kRagged;
    p.mix = !same_mod16;
    if (!ragged_shape(N / E + 1, p.mix, &p.vpt, &p.threads)) p.family = kGeneric;
    p.period = ragged_period((int64_t)N * esize(xd));
    // next-row prefetch up to 4 vectors per thread for the plain forward
    // (64 / 72 registers with packed gamma), up to 2 for the others -- but not
    // for the mixed fused add, whose extra CTAs beat it (32768 x 4096 bf16,
    // x off 16 bytes: 0.96 of the copy peak without, 0.90 with)
    p.prefetch = op == kFwd || (p.vpt <= 2 && !(op == kFused && p.mix));
  } else {
    p.family = kGeneric;
  }
  // what the register, ring and cluster kernels do not take: two passes of
  // 16-byte vectors (every operand realigned to the pass's frame) where that
  // kernel applies, else the scalar one
  if (p.family == kGeneric && wide_ok(bwd, N, xd)) p.family = kWide;
  if (p.family == kGeneric) {
    p.threads = 256;
    p.g = p.vpt = 0;
    p.prefetch = false;
    p.mix = false;
    p.period = 1;
  }
  if (p.family == kWide) {
    p.threads = wide_threads(bwd, N, E);
    p.g = p.vpt = 0;
    p.prefetch = false;
    p.mix = false;
    p.period = 1;
  }

  const Force& f = read_force();
  if (f.on) {
    if (f.family >= 0) p.family = f.family;
    if (f.g) p.g = f.g;
    if (f.vpt) p.vpt = f.vpt;
    if (f.threads) p.threads = f.threads;
    if (f.pf >= 0) p.prefetch = f.pf != 0;
    if (f.acc >= 0) p.acc_smem = f.acc != 0;
    p.cta_per_sm_cap = f.cps;
    if (p.family == kSubwarp) {
      p.threads = kSubwarpThreads;
      if (!rows_aligned || p.g < 1 || p.g > 32 || p.g * p.vpt * 1LL < nvec) return RMSNORM_ERR_INVALID_ARG;
      p.rows_per_cta = kSubwarpThreads / p.g;
    } else if (p.family == kCta) {
      if (!rows_aligned) return RMSNORM_ERR_INVALID_ARG;
      if (!f.threads) p.threads = round_up((nvec + p.vpt - 1) / (p.vpt ? p.vpt : 1), 32);
      if (p.vpt < 1 || (int64_t)p.threads * p.vpt < nvec) return RMSNORM_ERR_INVALID_ARG;
    } else if (p.family == kRagged) {
      if (!(same_mod16 || mix_ok) || N > kRaggedMaxN) return RMSNORM_ERR_INVALID_ARG;
      p.mix = !same_mod16;
      if (!p.vpt) p.vpt = 2;
      if (!f.threads) {
        const int per = (p.mix ? 31 : 32) * p.vpt;
        p.threads = 32 * ((N / E + 1 + per - 1) / per);
        if (p.threads < 64) p.threads = 64;
      }
      if (ragged_capacity(p.threads, p.vpt, p.mix) < N / E) return RMSNORM_ERR_INVALID_ARG;
      p.period = ragged_period((int64_t)N * esize(xd));
    } else if (p.family == kStaged && bwd && (f.g > 0 || (f.family < 0 && p.g > 0))) {
      // short backward rows through the ring: g lanes per row, 256 / g rows
      // per CTA iteration
      if (!f.vpt) p.vpt = (nvec + p.g - 1) / p.g;
      if (!rows_aligned || p.g > 32 || (int64_t)p.g * p.vpt < nvec) return RMSNORM_ERR_INVALID_ARG;
      p.threads = kSubwarpThreads;
      p.rows_per_cta = kSubwarpThreads / p.g;
      p.prefetch = false;
      if (f.st > 0) p.stages = f.st;
      else if (f.family == kStaged) p.stages = 0;   // as many as the budget holds
    } else if (p.family == kStaged) {
      if (!rows_aligned && !(mixed_rows && bwd)) return RMSNORM_ERR_INVALID_ARG;
      p.mix = !rows_aligned;
      p.g = 0;
      if (!p.vpt) p.vpt = 4;
      if (!f.threads) p.threads = round_up((nvec + p.vpt - 1) / p.vpt, 32);
      if ((int64_t)p.threads * p.vpt < nvec) return RMSNORM_ERR_INVALID_ARG;
      // st= sets the ring depth; without it a forced staged plan keeps the
      // default's depth, or takes as many stages as fit when the default is
      // another family
      if (f.st > 0 || f.family == kStaged) p.stages = f.st;
    } else if (p.family == kCluster) {
      if (!rows_aligned) return RMSNORM_ERR_INVALID_ARG;
      if (f.cl || f.family == kCluster) {
        if (!cluster_shape(bwd, nvec, f.cl, &p.cluster, &p.slice, &p.vpt, &p.threads))
          return RMSNORM_ERR_INVALID_ARG;
        if (f.vpt) p.vpt = f.vpt;
        p.threads = f.threads ? f.threads : round_up((p.slice + p.vpt - 1) / p.vpt, 32);
        if (f.pf < 0) p.prefetch = !bwd && p.vpt <= 4;
      }
      if (p.vpt < 1 || (int64_t)p.threads * p.vpt < p.slice) return RMSNORM_ERR_INVALID_ARG;
      if (bwd) {
        p.prefetch = false;
        if (f.st > 0) p.stages = f.st;
        if (p.stages < 2) p.stages = 2;
      }
    } else if (p.family == kGeneric) {
      if (!f.threads) p.threads = 256;
      if (p.threads != 256) return RMSNORM_ERR_INVALID_ARG;
    } else if (p.family == kWide) {
      if (!wide_ok(bwd, N, xd)) return RMSNORM_ERR_INVALID_ARG;
      if (!f.threads) p.threads = wide_threads(bwd, N, E);
      if (p.threads > (bwd ? kWideBwdThreads : kWideThreads)) return RMSNORM_ERR_INVALID_ARG;
      p.g = p.vpt = 0;
      p.prefetch = false;
    }
    if (p.family != kCluster) p.cluster = p.slice = 0;
    if (p.family != kSubwarp && !(p.family == kStaged && p.g > 0)) p.rows_per_cta = 1;
    if (p.family != kRagged) p.period = 1;
    if (p.family != kRagged && !(p.family == kStaged && p.g == 0)) p.mix = false;
    if (p.threads < 32 || p.threads > kCtaMaxThreads || p.threads % 32) return RMSNORM_ERR_INVALID_ARG;
  }

  // L2 lookahead (rows two iterations ahead, see the LayerNorm plan): in the
  // sub-warp backward with next-row prefetch only (262144 x 128 bf16: 0.80 ->
  // 0.85 of the copy peak); the forward kernels lost with it (16384 x 8192:
  // 0.97 -> 0.93), so they are built without it
  // The ragged kernels (rows not on 16 bytes) request the aligned interior
  // of the rows two steps ahead in their walk (4096 x 2049 bf16: bwd 0.372 ->
  // 0.385, fwd 0.546 -> 0.551; their few rows per CTA leave the pipeline's
  // fill and drain, not the bytes in flight, as the limit).
  const bool l2_able = p.prefetch && ((bwd && p.family == kSubwarp) || p.family == kRagged ||
                                      (!bwd && p.family == kCluster));
  // cluster forward: the slice of the row two steps ahead (2048 x 65536 bf16:
  // 0.77 -> 0.91 of the copy peak)
  if (l2_able) p.l2_ahead = 2;
  // the wide kernel: input rows requested into L2 up to two steps ahead of
  // the CTA's walk, as many steps as keep the requests of the whole grid
  // within kWideAheadBudget (set by size_grid)
  if (p.family == kWide)
    p.ahead_bytes = (int64_t)N * esize(xd) * (op == kFwd ? 1 : (op == kFusedBwd ? 3 : 2));
  if (f.on && f.l2 >= 0) {
    p.l2_ahead = f.l2;
    p.ahead_bytes = 0;
  }
  if (!l2_able && p.family != kWide) p.l2_ahead = 0;

  // kernel and shared memory
  if (p.family == kStaged) {
    // ring of row buffers: as many stages as fit a half-SM budget (two CTAs
    // per SM), at least two, at most kStagedMaxStages
    const int ns = op == kFwd ? 1 : (op == kFusedBwd ? 3 : 2);
    // a stage holds one row per operand, or the rows_per_cta rows of a CTA
    // iteration of short rows
    const int64_t stage_bytes =
        (int64_t)ns * ((int64_t)N * esize(xd) + (p.mix ? 16 : 0)) * (p.g > 0 ? p.rows_per_cta : 1);
    if (p.stages <= 0) {
      int64_t st = (kStagedSmemBudget - kStagedHeader) / stage_bytes;
      if (st < 2) st = (kStagedSmemMax - kStagedHeader) / stage_bytes;
      p.stages = (int)(st > kStagedMaxStages ? kStagedMaxStages : st);
    }
    if (p.stages < 2 || p.stages > kStagedMaxStages ||
        kStagedHeader + p.stages * stage_bytes > kStagedSmemMax)
      return RMSNORM_ERR_INVALID_ARG;
    p.smem = (int)(kStagedHeader + p.stages * stage_bytes);
    if (p.g == 0) p.rows_per_cta = 1;
  }
  if (bwd) {
    // each CTA writes one dgamma partial row (N fp32); keep that traffic to a
    // few percent of the rows it reads
    p.min_rows = 8 / p.rows_per_cta > 0 ? 8 / p.rows_per_cta : 1;
    const Force& fr = read_force();
    if (fr.on && fr.mr >= 0) p.min_rows = fr.mr;
    if (dres && p.family == kCta) return RMSNORM_ERR_INVALID_ARG;
    BwdKey k{xd, wd, p.family, p.g, p.vpt, has_rstd, p.acc_smem, p.prefetch, dres, p.mix};
    p.bwd = bwd_kernel(k);
    p.fn = reinterpret_cast<const void*>(p.bwd);
    const int ld = round_up(N, 4);
    if (p.family == kSubwarp) p.smem = p.rows_per_cta * nvec * E * 4;
    else if (p.family == kCta) p.smem = 512 + (p.acc_smem ? ld * 4 : 0);
    else if (p.family == kRagged) p.smem = 512;
    else if (p.family == kWide) p.smem = (int)wide_smem(N, xd);
    else if (p.family == kCluster) {
      // ring of the slice of [x | dy] ([h | dy | dres]) rows
      const int64_t bytes = kStagedHeader + (int64_t)p.stages * (dres ? 3 : 2) * p.slice * 16;
      if (p.stages > kStagedMaxStages || bytes > kStagedSmemMax) return RMSNORM_ERR_INVALID_ARG;
      p.smem = (int)bytes;
    } else if (p.family != kStaged) p.smem = 0;
  } else {
    FwdKey k{xd, wd, p.family, p.g, p.vpt, op == kFused, p.prefetch, false};
    k.mix = p.mix;
    p.fwd = fwd_kernel(k);
    p.fn = reinterpret_cast<const void*>(p.fwd);
    if (p.family == kCta) p.smem = 256;
    else if (p.family == kRagged) p.smem = 256;
    else if (p.family != kStaged) p.smem = 0;
  }
  if (p.fn == nullptr) return RMSNORM_ERR_INVALID_ARG;
  *pl = p;
  return RMSNORM_OK;
}

// Grid of a plan on a device: persistent, at most SMs x resident CTAs.
rmsnorm_status_t size_grid(Plan* p, int64_t M, int device, unsigned** status = nullptr) {
  DevInfo di;
  cudaError_t e = device_info(device, &di);
  if (e != cudaSuccess) return cuda_fail(e, "device attributes");
  if (status) *status = di.status;
  if (p->smem > di.max_smem_optin) return RMSNORM_ERR_INVALID_ARG;
  if (p->cluster > 0) {
    // one row per cluster: as many clusters as the device holds at once (the
    // occupancy query accounts for how clusters pack into the GPCs)
    int clusters = 0;
    if ((e = occupancy(p->fn, device, p->threads, p->smem, &clusters, p->cluster)) !=
        cudaSuccess)
      return cuda_fail(e, "cluster occupancy query");
    int64_t cap = clusters;
    if (p->cta_per_sm_cap > 0) {
      const int64_t lim = (int64_t)di.sms * p->cta_per_sm_cap / p->cluster;
      if (cap > lim) cap = lim > 0 ? lim : 1;
    }
    if (p->min_rows > 0) {
      const int64_t want = (M + p->min_rows - 1) / p->min_rows;
      const int64_t floor_cap = di.sms / p->cluster < cap ? di.sms / p->cluster : cap;
      cap = want < floor_cap ? floor_cap : (want < cap ? want : cap);
    }
    int64_t n = M < cap ? M : cap;
    if (n < 1) n = 1;
    p->grid = (int)n * p->cluster;
    return RMSNORM_OK;
  }
  int per_sm = 0;
  if ((e = occupancy(p->fn, device, p->threads, p->smem, &per_sm)) != cudaSuccess)
    return cuda_fail(e, "occupancy query");
  if (p->cta_per_sm_cap > 0 && per_sm > p->cta_per_sm_cap) per_sm = p->cta_per_sm_cap;
  const int64_t units = (M + p->rows_per_cta - 1) / p->rows_per_cta;
  int64_t cap = (int64_t)di.sms * per_sm;
  if (p->min_rows > 0) {
    const int64_t want = (units + p->min_rows - 1) / p->min_rows;
    const int64_t floor_cap = di.sms < cap ? di.sms : cap;
    cap = want < floor_cap ? floor_cap : (want < cap ? want : cap);
  }
  p->grid = (int)(units < cap ? units : cap);
  if (p->grid < 1) p->grid = 1;
  if (p->family == kWide && p->ahead_bytes > 0) {
    const int64_t step = p->ahead_bytes * p->grid;
    const int64_t n = kWideAheadBudget / step;
    p->l2_ahead = n > 2 ? 2 : (int)n;
  }
  if (p->period > 1) {   // whole residue classes: a multiple of the period
    p->grid = p->grid / p->period * p->period;
    if (p->grid < p->period) p->grid = p->period;
  }
  return RMSNORM_OK;
}

const char* family_name(int f) {
  switch (f) {
    case kSubwarp: return "subwarp";
    case kCta: return "cta";
    case kRagged: return "ragged";
    case kStaged: return "staged";
    case kCluster: return "cluster";
    case kWide: return "wide";
    default: return "generic";
  }
}

void describe(int op, const Plan& p, char* buf, size_t len) {
  static const char* ops[] = {"fwd",     "fused_add",     "bwd",       "fused_add_bwd",
                              "fwd_strided", "fwd_fp8",   "fused_add_fp8", "fwd_nvfp4",
                              "fused_add_nvfp4", "layernorm_fwd", "layernorm_bwd"};
  const bool bwd = op == kBwd || op == kFusedBwd;
  char l2[24] = "";
  if (p.l2_ahead > 0) snprintf(l2, sizeof l2, "/l2ahead%d", p.l2_ahead);
  char cl[32] = "";
  if (p.cluster > 0) snprintf(cl, sizeof cl, "/cl%d/slice%d", p.cluster, p.slice);
  snprintf(buf, len, "%s/%s%s/g%d/vpt%d/t%d/pf%d/st%d/per%d%s/grid%d/smem%d%s%s", ops[op],
           family_name(p.family), p.mix ? "_mix" : "", p.g, p.vpt, p.threads, p.prefetch ? 1 : 0, p.stages, p.period,
           bwd ? (p.acc_smem ? "/acc_smem" : "/acc_reg") : "", p.grid, p.smem, l2, cl);
}

// ---------------------------------------------------------------- launches

// Every kernel is launched as a programmatic dependent of the previous work on
// the stream (the kernels wait for it at entry, see pdl_begin), so the launch
// of one call overlaps the end of the previous one.  RMSNORM_NO_PDL=1 (read
// with the other debug knobs) turns the attribute off for A/B measurements.
template <typename... Args>
cudaError_t launch_in_clusters(int cluster, void (*kernel)(Args...), int grid, int threads,
                               int smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (!g_env.no_pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 0) {   // thread-block clusters of `cluster` consecutive CTAs
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
template <typename... Args>
cudaError_t launch(void (*kernel)(Args...), int grid, int threads, int smem,
                   cudaStream_t stream, Args... args) {
  return launch_in_clusters(0, kernel, grid, threads, smem, stream, args...);
}

// Stage 2 of a backward (column sums of P partial rows of nq float4): eight
// float4 columns per CTA (32 row lanes), or -- for the few partial rows of
// clusters and short walks -- sixteen (P <= 256) or thirty-two (P <= 128), so
// that lanes are not left idle over a wide grid (2048 x 65536 bf16, 36
// partial rows: 2048 CTAs at eight columns).  A grid wider than eight columns
// per CTA gives lost badly behind the fused-add backward's three-CTA-per-SM
// ring when launched as a programmatic dependent (32768 x 4096 bf16: 259 /
// 219 us per call at two / four columns against 159 at eight; 161 at any
// width without the dependent launch); stage 2 costs its latency, not its
// bytes.
cudaError_t launch_colsum(const float* part, int P, int nq, const ColSumOut& o,
                          cudaStream_t stream) {
  const int c = P <= 128 ? 32 : (P <= 256 ? 16 : 8);
  return launch(get_colsum_kernel(c), (nq + c - 1) / c, kColSumThreads, 0, stream, part, P, nq,
                o);
}

// ---------------------------------------------------------------- validation

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || !na || !nb) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

rmsnorm_status_t check_sizes(int64_t M, int64_t N, float eps) {
  if (M < 0 || N < 1 || N > kMaxN) return RMSNORM_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || isinf(eps)) return RMSNORM_ERR_INVALID_ARG;
  return RMSNORM_OK;
}

rmsnorm_status_t current_device(int* dev) {
  const cudaError_t e = cudaGetDevice(dev);
  return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e, "cudaGetDevice");
}

// ---------------------------------------------------------------- forward

rmsnorm_status_t fwd_impl(int op, const void* x, void* residual, const void* gamma, void* y,
                          float* rstd, int64_t M, int64_t N, float eps, int xd, int wd,
                          cudaStream_t stream) {
  rmsnorm_status_t st = check_sizes(M, N, eps);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok(xd, wd)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if (M == 0) return RMSNORM_OK;
  if (!x || !gamma || !y || (op == kFused && !residual)) return RMSNORM_ERR_INVALID_ARG;
  const size_t xs = (size_t)esize(xd), ws = (size_t)esize(wd);
  if (!aligned_to(x, xs) || !aligned_to(y, xs) || !aligned_to(gamma, ws) ||
      (residual && !aligned_to(residual, xs)) || (rstd && !aligned_to(rstd, 4)))
    return RMSNORM_ERR_MISALIGNED;
  const size_t act = (size_t)M * (size_t)N * xs, gb = (size_t)N * ws, rb = (size_t)M * 4;
  if (overlap(y, act, x, act) || overlap(y, act, gamma, gb) || overlap(y, act, rstd, rb) ||
      overlap(rstd, rb, x, act) || overlap(rstd, rb, gamma, gb))
    return RMSNORM_ERR_INVALID_ARG;
  if (op == kFused && (overlap(residual, act, x, act) || overlap(residual, act, y, act) ||
                       overlap(residual, act, gamma, gb) || overlap(residual, act, rstd, rb)))
    return RMSNORM_ERR_INVALID_ARG;

  const uintptr_t mx = reinterpret_cast<uintptr_t>(x) & 15;
  const uintptr_t my = reinterpret_cast<uintptr_t>(y) & 15;
  // the outputs (y, and h over the residual) agree modulo 16; x may not
  const bool out_same = op != kFused || (reinterpret_cast<uintptr_t>(residual) & 15) == my;
  const bool same = out_same && my == mx;
  const bool aligned16 = same && mx == 0 && aligned_to(gamma, 16);

  int dev;
  if ((st = current_device(&dev)) != RMSNORM_OK) return st;
  Plan pl;
  if ((st = make_plan(op, M, (int)N, xd, wd, aligned16, same, false, &pl, out_same)) !=
      RMSNORM_OK)
    return st;
  unsigned* status = nullptr;
  if ((st = size_grid(&pl, M, dev, &status)) != RMSNORM_OK) return st;

  FwdParams prm = {};
  prm.x = x;
  prm.residual = residual;
  prm.gamma = gamma;
  prm.y = y;
  prm.rstd = rstd;
  prm.M = M;
  prm.N = (int)N;
  prm.nvec = (int)(N / per_vec(xd));
  prm.eps = eps;
  prm.inv_n = 1.0f / (float)N;
  prm.stages = pl.stages;
  prm.wait_limit = wait_limit();
  prm.status = status;
  prm.period = pl.period;
  prm.l2_rows = pl.l2_ahead;
  prm.slice = pl.slice;
  prm.x_shift = (int)((mx - my) & 15);
  const cudaError_t e =
      launch_in_clusters(pl.cluster, pl.fwd, pl.grid, pl.threads, pl.smem, stream, prm);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "forward kernel launch");
  }
  return RMSNORM_OK;
}

// ---------------------------------------------------------------- strided rows

// Rows (t, h) of a [T, H, D] view with element strides (st, sh): non-negative,
// rows inside a token do not overlap, tokens do not overlap.
bool strided_layout_ok(int64_t T, int64_t H, int64_t D, int64_t st, int64_t sh) {
  if (st < 0 || sh < 0) return false;
  if (H > 1 && sh < D) return false;
  if (T > 1 && st < (H - 1) * sh + D) return false;
  return true;
}

// Plan of the strided forward: a row of at most 128 16-byte vectors with every
// pointer and stride 16-byte aligned goes to the sub-warp kernel (G lanes walk
// the (token, head) rows), anything else to the scalar kernel.
rmsnorm_status_t strided_plan(int64_t D, int xd, int wd, bool vec_ok, Plan* out) {
  const int nvec = vec_ok ? (int)(D / per_vec(xd)) : 0;
  Plan p;
  if (vec_ok && nvec <= 128) {
    p.family = kSubwarp;
    subwarp_shape(nvec, &p.g, &p.vpt);
    p.threads = kSubwarpThreads;
    p.rows_per_cta = kSubwarpThreads / p.g;
    // next-row prefetch (q norm at 32768 tokens x 32 heads x 128: 0.92 with,
    // 0.90 without, since the bf16 arithmetic runs from the packed words)
    p.prefetch = true;
  } else {
    p.family = kGeneric;
    p.threads = 256;
  }
  const Force& f = read_force();
  if (f.on) {
    if (f.family == kGeneric) {
      p.family = kGeneric;
      p.threads = 256;
      p.rows_per_cta = 1;
    } else if (f.family == kSubwarp) {
      if (!vec_ok || !f.g || !f.vpt || f.g * f.vpt < nvec) return RMSNORM_ERR_INVALID_ARG;
      p.g = f.g;
      p.vpt = f.vpt;
      p.rows_per_cta = kSubwarpThreads / p.g;
    } else if (f.family >= 0) {
      return RMSNORM_ERR_INVALID_ARG;
    }
    if (f.pf >= 0) p.prefetch = f.pf != 0;
    p.cta_per_sm_cap = f.cps;
  }
  FwdKey k{xd, wd, p.family, p.g, p.vpt, false, p.prefetch, true};
  p.fwd = fwd_kernel(k);
  p.fn = reinterpret_cast<const void*>(p.fwd);
  p.smem = 0;
  if (p.fn == nullptr) return RMSNORM_ERR_INVALID_ARG;
  *out = p;
  return RMSNORM_OK;
}

rmsnorm_status_t fwd_strided_impl(const void* x, int64_t x_st, int64_t x_sh, const void* gamma,
                                  void* y, int64_t y_st, int64_t y_sh, float* rstd, int64_t T,
                                  int64_t H, int64_t D, float eps, int xd, int wd,
                                  cudaStream_t stream) {
  if (T < 0 || H < 0) return RMSNORM_ERR_INVALID_ARG;
  rmsnorm_status_t st = check_sizes(T * H, D, eps);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok(xd, wd)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  const int64_t M = T * H;
  if (M == 0) return RMSNORM_OK;
  if (!x || !gamma || !y) return RMSNORM_ERR_INVALID_ARG;
  if (!strided_layout_ok(T, H, D, x_st, x_sh) || !strided_layout_ok(T, H, D, y_st, y_sh))
    return RMSNORM_ERR_INVALID_ARG;
  const size_t xs = (size_t)esize(xd), ws = (size_t)esize(wd);
  if (!aligned_to(x, xs) || !aligned_to(y, xs) || !aligned_to(gamma, ws) ||
      (rstd && !aligned_to(rstd, 4)))
    return RMSNORM_ERR_MISALIGNED;
  const size_t xspan = (size_t)((T - 1) * x_st + (H - 1) * x_sh + D) * xs;
  const size_t yspan = (size_t)((T - 1) * y_st + (H - 1) * y_sh + D) * xs;
  const size_t gb = (size_t)D * ws, rb = (size_t)M * 4;
  const bool in_place = x == y && x_st == y_st && x_sh == y_sh;
  if ((!in_place && overlap(x, xspan, y, yspan)) || overlap(y, yspan, gamma, gb) ||
      overlap(y, yspan, rstd, rb) || overlap(rstd, rb, x, xspan) || overlap(rstd, rb, gamma, gb))
    return RMSNORM_ERR_INVALID_ARG;

  const bool vec_ok = aligned_to(x, 16) && aligned_to(y, 16) && aligned_to(gamma, 16) &&
                      (D * (int64_t)xs) % 16 == 0 && (x_st * (int64_t)xs) % 16 == 0 &&
                      (x_sh * (int64_t)xs) % 16 == 0 && (y_st * (int64_t)xs) % 16 == 0 &&
                      (y_sh * (int64_t)xs) % 16 == 0;
  Plan p;
  if ((st = strided_plan(D, xd, wd, vec_ok, &p)) != RMSNORM_OK) return st;
  const int nvec = vec_ok ? (int)(D / per_vec(xd)) : 0;
  int dev;
  if ((st = current_device(&dev)) != RMSNORM_OK) return st;
  unsigned* status = nullptr;
  if ((st = size_grid(&p, M, dev, &status)) != RMSNORM_OK) return st;

  FwdParams prm = {};
  prm.x = x;
  prm.gamma = gamma;
  prm.y = y;
  prm.rstd = rstd;
  prm.M = M;
  prm.N = (int)D;
  prm.nvec = nvec;
  prm.eps = eps;
  prm.inv_n = 1.0f / (float)D;
  prm.status = status;
  prm.period = 1;
  prm.heads = H;
  prm.x_st = x_st;
  prm.x_sh = x_sh;
  prm.y_st = y_st;
  prm.y_sh = y_sh;
  const cudaError_t e = launch(p.fwd, p.grid, p.threads, p.smem, stream, prm);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "strided forward launch");
  }
  return RMSNORM_OK;
}

// ---------------------------------------------------------------- quantised outputs

// Plan of the quantised forward (out = kOutFp8 or kOutNvfp4): rows of at most
// 128 16-byte vectors take the sub-warp form, rows of at most 4096 vectors the
// CTA-per-row form, both needing 16-byte aligned rows and codes that can be
// stored a vector at a time; anything else the scalar kernel.  Every shape
// issues the next row's loads before reducing the current one (register
// prefetch): the epilogue is long enough that without it too few bytes stay
// in flight (16384 x 8192 bf16 FP8: 0.62 -> 0.85 of the copy bandwidth;
// 32768 x 4096 fused add: 0.94-0.96 -> 0.97-0.99).  The staged form (rows
// through the bulk-copy ring) is available as a forced variant; it measured
// no better here (0.83 / 0.67 plain, 0.93 / 0.79 fused), the kernels being
// bound by instruction issue rather than by bytes in flight.
rmsnorm_status_t quant_plan(int out, bool fused, int64_t N, int xd, int wd, bool vec_ok,
                            Plan* res) {
  const int nvec = vec_ok ? (int)(N / per_vec(xd)) : 0;
  Plan p;
  if (vec_ok && nvec <= 128) {
    p.family = kSubwarp;
    subwarp_shape(nvec, &p.g, &p.vpt);
    p.threads = kSubwarpThreads;
    p.rows_per_cta = kSubwarpThreads / p.g;
    p.prefetch = true;
  } else if (vec_ok && cta_shape(kQuantFwd, nvec, &p.vpt, &p.threads)) {
    p.family = kCta;
    p.prefetch = p.vpt <= 4;
  } else {
    p.family = kGeneric;
    p.threads = 256;
  }
  const Force& f = read_force();
  if (f.on) {
    if (f.family == kGeneric) {
      p.family = kGeneric;
      p.threads = 256;
      p.rows_per_cta = 1;
    } else if (f.family == kSubwarp) {
      if (!vec_ok || !f.g || !f.vpt || f.g * f.vpt < nvec) return RMSNORM_ERR_INVALID_ARG;
      p.family = kSubwarp;
      p.g = f.g;
      p.vpt = f.vpt;
      p.threads = kSubwarpThreads;
      p.rows_per_cta = kSubwarpThreads / p.g;
    } else if (f.family == kCta) {
      if (!vec_ok || !f.vpt) return RMSNORM_ERR_INVALID_ARG;
      p.family = kCta;
      p.vpt = f.vpt;
      p.threads = f.threads ? f.threads : round_up((nvec + p.vpt - 1) / p.vpt, 32);
      if (p.threads < 32 || p.threads > kCtaMaxThreads || p.threads % 32 ||
          (int64_t)p.threads * p.vpt < nvec)
        return RMSNORM_ERR_INVALID_ARG;
      p.rows_per_cta = 1;
    } else if (f.family == kStaged) {
      if (!vec_ok) return RMSNORM_ERR_INVALID_ARG;
      p.family = kStaged;
      p.vpt = f.vpt ? f.vpt : 4;
      p.threads = f.threads ? f.threads : round_up((nvec + p.vpt - 1) / p.vpt, 32);
      if (p.threads < 32 || p.threads > kCtaMaxThreads || p.threads % 32 ||
          (int64_t)p.threads * p.vpt < nvec)
        return RMSNORM_ERR_INVALID_ARG;
      p.stages = f.st;
      p.rows_per_cta = 1;
    } else if (f.family >= 0) {
      return RMSNORM_ERR_INVALID_ARG;
    }
    if (f.pf >= 0) p.prefetch = f.pf != 0;
    if (p.family == kGeneric || p.family == kStaged) p.prefetch = false;
    p.cta_per_sm_cap = f.cps;
  }
  FwdKey k{xd, wd, p.family, p.g, p.vpt, fused, p.prefetch, false, out};
  p.fwd = fwd_kernel(k);
  p.fn = reinterpret_cast<const void*>(p.fwd);
  p.smem = 0;
  if (p.fn == nullptr) return RMSNORM_ERR_INVALID_ARG;
  if (p.family == kStaged) {
    // ring of row buffers ([x], or [r | x] fused): as many stages as fit the
    // half-SM budget (two CTAs per SM), at least two, at most kStagedMaxStages
    const int64_t stage_bytes = (fused ? 2 : 1) * N * esize(xd);
    if (p.stages <= 0) {
      int64_t st = (kStagedSmemBudget - kStagedHeader) / stage_bytes;
      if (st < 2) st = (kStagedSmemMax - kStagedHeader) / stage_bytes;
      p.stages = (int)(st > kStagedMaxStages ? kStagedMaxStages : st);
    }
    if (p.stages < 2 || p.stages > kStagedMaxStages ||
        kStagedHeader + p.stages * stage_bytes > kStagedSmemMax)
      return RMSNORM_ERR_INVALID_ARG;
    p.smem = (int)(kStagedHeader + p.stages * stage_bytes);
  }
  *res = p;
  return RMSNORM_OK;
}

// q: codes (FP8: M x N bytes; NVFP4: M x N/2); qs: scales (FP8: M fp32;
// NVFP4: M x N/16 E4M3 bytes); gs: NVFP4 global scale.
rmsnorm_status_t fwd_quant_impl(int out, const void* x, void* residual, const void* gamma,
                                float gs, void* q, void* qs, float* rstd, int64_t M, int64_t N,
                                float eps, int xd, int wd, cudaStream_t stream) {
  rmsnorm_status_t st = check_sizes(M, N, eps);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok(xd, wd)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if (out == kOutNvfp4 && (N % 16 != 0 || !(gs > 0.f) || isinf(gs)))
    return RMSNORM_ERR_INVALID_ARG;
  if (M == 0) return RMSNORM_OK;
  if (!x || !gamma || !q || !qs) return RMSNORM_ERR_INVALID_ARG;
  const size_t xs = (size_t)esize(xd), ws = (size_t)esize(wd);
  if (!aligned_to(x, xs) || !aligned_to(gamma, ws) || (residual && !aligned_to(residual, xs)) ||
      (rstd && !aligned_to(rstd, 4)) || (out == kOutFp8 && !aligned_to(qs, 4)))
    return RMSNORM_ERR_MISALIGNED;
  const size_t act = (size_t)M * (size_t)N * xs, gb = (size_t)N * ws, rb = (size_t)M * 4;
  const size_t qb = out == kOutFp8 ? (size_t)M * N : (size_t)M * (N / 2);
  const size_t sb = out == kOutFp8 ? (size_t)M * 4 : (size_t)M * (N / 16);
  const void* bufs[6] = {x, residual, gamma, q, qs, rstd};
  const size_t lens[6] = {act, act, gb, qb, sb, rb};
  for (int i = 0; i < 6; ++i)
    for (int j = i + 1; j < 6; ++j)
      if (overlap(bufs[i], lens[i], bufs[j], lens[j])) return RMSNORM_ERR_INVALID_ARG;

  const bool vec_ok = aligned_to(x, 16) && aligned_to(gamma, 16) &&
                      (!residual || aligned_to(residual, 16)) && (N * (int64_t)xs) % 16 == 0 &&
                      aligned_to(q, 8);
  Plan p;
  if ((st = quant_plan(out, residual != nullptr, N, xd, wd, vec_ok, &p)) != RMSNORM_OK)
    return st;
  int dev;
  if ((st = current_device(&dev)) != RMSNORM_OK) return st;
  unsigned* status = nullptr;
  if ((st = size_grid(&p, M, dev, &status)) != RMSNORM_OK) return st;

  FwdParams prm = {};
  prm.x = x;
  prm.residual = residual;
  prm.gamma = gamma;
  prm.y = q;
  prm.stages = p.stages;
  prm.wait_limit = wait_limit();
  prm.status = status;
  prm.rstd = rstd;
  prm.M = M;
  prm.N = (int)N;
  prm.nvec = vec_ok ? (int)(N / per_vec(xd)) : 0;
  prm.eps = eps;
  prm.inv_n = 1.0f / (float)N;
  prm.period = 1;
  prm.qs = qs;
  prm.gs = gs;
  const cudaError_t e = launch(p.fwd, p.grid, p.threads, p.smem, stream, prm);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "quantised forward launch");
  }
  return RMSNORM_OK;
}

// ---------------------------------------------------------------- LayerNorm

LnKernel ln_kernel(const LnKey& k) {
  if (k.family == kWide) {
    if (k.xd == kF32 && k.wd == kF32) return get_ln_wide_f32_f32(k);
    if (k.xd == kBF16 && k.wd == kBF16) return get_ln_wide_bf16_bf16(k);
    if (k.xd == kBF16 && k.wd == kF32) return get_ln_wide_bf16_f32(k);
    return nullptr;
  }
  if (k.xd == kF32 && k.wd == kF32) return get_ln_kernel_f32_f32(k);
  if (k.xd == kBF16 && k.wd == kBF16) return get_ln_kernel_bf16_bf16(k);
  if (k.xd == kBF16 && k.wd == kF32) return get_ln_kernel_bf16_f32(k);
  return nullptr;
}

// The wide LayerNorm backward keeps its two partial rows in shared memory
// (each N + 2E floats, rounded to 4) and needs dx's split to be the same for
// every row.
int64_t ln_wide_smem(int N, int xd) { return 2 * wide_smem(N, xd); }
bool ln_wide_ok(bool bwd, int64_t N, int xd) {
  return !bwd || ((N * esize(xd)) % 16 == 0 && ln_wide_smem((int)N, xd) <= kStagedSmemMax);
}

// Plan of the LayerNorm kernels: rows of at most 128 16-byte vectors take the
// sub-warp form; longer aligned rows one CTA per row with next-row prefetch --
// the forward with up to 4 vectors per thread (16384 x 8192 bf16: VPT 4 0.84
// of the copy bandwidth, VPT 2 / 512 threads 0.69: two row barriers per row
// cost more in a larger CTA), the backward with up to 2 (0.80; it holds gamma
// and two partial rows per thread).  The staged backward with one row per
// CTA (rows through the bulk-copy ring) is a forced variant only: at 4
// vectors per thread it spills (0.70), at 2 it fits one CTA per SM (0.63);
// the backward of rows of 65-128 vectors takes the ring with eight rows of 32
// lanes per stage.  Anything else: the scalar kernel.
rmsnorm_status_t ln_plan(bool bwd, int64_t M, int64_t N, int xd, int wd, bool vec_ok,
                         Plan* res, bool saved = false) {
  const int E = per_vec(xd);
  const int nvec = vec_ok ? (int)(N / E) : 0;
  Plan p;
  p.family = kGeneric;
  p.threads = 256;
  // sub-warp rows up to 128 vectors; the backward takes one CTA per row
  // from 128 vectors on (65536 x 1024 bf16: 64-thread CTAs at 2 vectors per
  // thread 0.84 against 0.83 for 32 lanes at 4, both with the L2 lookahead)
  if (vec_ok && (bwd ? nvec < 128 : nvec <= 128)) {
    p.family = kSubwarp;
    subwarp_shape(nvec, &p.g, &p.vpt);
    p.threads = kSubwarpThreads;
    p.rows_per_cta = kSubwarpThreads / p.g;
    p.prefetch = true;
  } else if (vec_ok) {
    static const int pref_fwd[] = {4, 2, 1}, pref_bwd[] = {2, 1};
    const int* pref = bwd ? pref_bwd : pref_fwd;
    for (int i = 0; i < (bwd ? 2 : 3); ++i) {
      const int t = round_up((nvec + pref[i] - 1) / pref[i], 32);
      if (t >= 64 && t <= kCtaMaxThreads) {
        p.family = kCta;
        p.vpt = pref[i];
        p.threads = t;
        p.prefetch = true;
        break;
      }
    }
  }
  // backward rows of 65-128 vectors: the CTA's eight rows of 32 lanes through
  // a bulk-copy ring, one copy per operand per stage (65536 x 1024 bf16: 0.94
  // of the copy peak with three stages, against 0.88 for one 64-thread CTA per
  // row; two stages 0.88, four 0.67 at one CTA per SM).  Not for bf16
  // activations with fp32 weights at 4 vectors per lane, whose form spills.
  if (bwd && vec_ok && nvec > 64 && nvec <= 128 &&
      !(xd == kBF16 && wd == kF32 && (nvec + 31) / 32 == 4)) {
    p.family = kStaged;
    p.g = 32;
    p.vpt = (nvec + 31) / 32;
    p.threads = kSubwarpThreads;
    p.rows_per_cta = kSubwarpThreads / 32;
    p.prefetch = false;
    p.stages = 0;
  }
  // what those do not take -- rows or operands off 16 bytes, forward rows
  // beyond 2048 vectors, backward rows beyond 1024 -- goes to the wide
  // kernel where it applies, else to the scalar one
  if (p.family == kGeneric && ln_wide_ok(bwd, N, xd)) {
    p.family = kWide;
    p.threads = wide_threads(bwd, (int)N, E);
  }
  const Force& f = read_force();
  if (f.on) {
    if (f.family == kGeneric) {
      p.family = kGeneric;
      p.threads = 256;
      p.rows_per_cta = 1;
    } else if (f.family == kWide) {
      if (!ln_wide_ok(bwd, N, xd)) return RMSNORM_ERR_INVALID_ARG;
      p.family = kWide;
      p.threads = f.threads ? f.threads : wide_threads(bwd, (int)N, E);
      if (p.threads < 64 || p.threads % 32 || p.threads > (bwd ? kWideBwdThreads : kWideThreads))
        return RMSNORM_ERR_INVALID_ARG;
      p.rows_per_cta = 1;
      p.stages = 0;
    } else if (f.family == kSubwarp) {
      if (!vec_ok || !f.g || !f.vpt || f.g * f.vpt < nvec) return RMSNORM_ERR_INVALID_ARG;
      p.family = kSubwarp;
      p.g = f.g;
      p.vpt = f.vpt;
      p.threads = kSubwarpThreads;
      p.rows_per_cta = kSubwarpThreads / p.g;
    } else if (f.family == kCta) {
      if (!vec_ok || !f.vpt) return RMSNORM_ERR_INVALID_ARG;
      p.family = kCta;
      p.vpt = f.vpt;
      p.threads = f.threads ? f.threads : round_up((nvec + p.vpt - 1) / p.vpt, 32);
      if (p.threads < 32 || p.threads > kCtaMaxThreads || p.threads % 32 ||
          (int64_t)p.threads * p.vpt < nvec)
        return RMSNORM_ERR_INVALID_ARG;
      p.rows_per_cta = 1;
    } else if (f.family == kStaged && f.g > 0) {
      // short rows through the ring: g lanes per row, 256 / g rows per stage
      if (!vec_ok || !bwd || f.g > 32) return RMSNORM_ERR_INVALID_ARG;
      p.family = kStaged;
      p.g = f.g;
      p.vpt = f.vpt ? f.vpt : (nvec + f.g - 1) / f.g;
      if ((int64_t)p.g * p.vpt < nvec) return RMSNORM_ERR_INVALID_ARG;
      p.threads = kSubwarpThreads;
      p.rows_per_cta = kSubwarpThreads / p.g;
      p.stages = f.st;
    } else if (f.family == kStaged) {
      if (!vec_ok || !bwd) return RMSNORM_ERR_INVALID_ARG;
      p.family = kStaged;
      p.g = 0;
      p.vpt = f.vpt ? f.vpt : 4;
      p.threads = f.threads ? f.threads : round_up((nvec + p.vpt - 1) / p.vpt, 32);
      if (p.threads < 32 || p.threads > kCtaMaxThreads || p.threads % 32 ||
          (int64_t)p.threads * p.vpt < nvec)
        return RMSNORM_ERR_INVALID_ARG;
      p.rows_per_cta = 1;
      p.stages = f.st;
    } else if (f.family >= 0) {
      return RMSNORM_ERR_INVALID_ARG;
    }
    if (f.pf >= 0) p.prefetch = f.pf != 0;
    p.cta_per_sm_cap = f.cps;
  }
  // register kernels: besides the next row held in registers, the rows two
  // iterations ahead are requested into L2, doubling the bytes in flight per
  // SM without holding registers for them (measured, 16384 x 8192 bf16: fwd
  // 0.88 -> 0.93, bwd 0.82 -> 0.92 of the copy peak; 65536 x 1024: bwd 0.77 ->
  // 0.83, but the sub-warp forward loses, 0.93 -> 0.84, so it goes without)
  if (p.prefetch && (p.family == kCta || (p.family == kSubwarp && bwd))) p.l2_ahead = 2;
  if (f.on && f.l2 >= 0) p.l2_ahead = f.l2;
  if (p.family == kGeneric || p.family == kWide) {
    p.g = p.vpt = 0;
    p.prefetch = false;
    p.rows_per_cta = 1;
  }
  if (p.family == kGeneric || p.family == kStaged) p.l2_ahead = 0;
  // the wide kernel's lookahead, sized to the grid by size_grid
  if (p.family == kWide && !(f.on && f.l2 >= 0)) {
    p.l2_ahead = 0;
    p.ahead_bytes = N * esize(xd) * (bwd ? 2 : 1);
  }
  if (p.family == kStaged) {
    p.prefetch = false;
    // ring of [x | dy] row pairs (of the CTA's rows_per_cta rows for short
    // rows): as many stages as fit the half-SM budget (two CTAs per SM), at
    // least two, at most kStagedMaxStages
    const int64_t stage_bytes = 2 * N * esize(xd) * p.rows_per_cta;
    if (p.stages <= 0) {
      int64_t st = (kStagedSmemBudget - kStagedHeader) / stage_bytes;
      if (st < 2) st = (kStagedSmemMax - kStagedHeader) / stage_bytes;
      p.stages = (int)(st > kStagedMaxStages ? kStagedMaxStages : st);
    }
    if (p.stages < 2 || p.stages > kStagedMaxStages ||
        kStagedHeader + p.stages * stage_bytes > kStagedSmemMax)
      return RMSNORM_ERR_INVALID_ARG;
  }
  if (p.family != kSubwarp && p.family != kStaged) p.g = 0;
  // the wide backward with saved statistics: the pipelined form, smaller CTAs
  const bool wide_saved = bwd && saved && p.family == kWide;
  if (wide_saved && p.threads > kLnSavedThreads) {
    if (f.on && f.threads) return RMSNORM_ERR_INVALID_ARG;
    p.threads = kLnSavedThreads;
  }
  LnKey k{xd, wd, p.family, p.g, p.vpt, bwd, p.prefetch};
  k.saved = wide_saved;
  LnKernel fn = ln_kernel(k);
  if (fn == nullptr) return RMSNORM_ERR_INVALID_ARG;
  p.fn = reinterpret_cast<const void*>(fn);
  // sub-warp backward: the groups' partial rows meet in shared memory;
  // staged: the ring
  p.smem = (bwd && p.family == kSubwarp) ? p.rows_per_cta * 2 * nvec * E * 4 : 0;
  if (p.family == kStaged)
    p.smem = (int)(kStagedHeader + p.stages * 2 * N * esize(xd) * p.rows_per_cta);
  if (p.family == kWide && bwd) p.smem = (int)ln_wide_smem((int)N, xd);
  if (bwd) {
    p.min_rows = 8 / p.rows_per_cta > 0 ? 8 / p.rows_per_cta : 1;
    const Force& fr = read_force();
    if (fr.on && fr.mr >= 0) p.min_rows = fr.mr;
  }
  (void)M;
  *res = p;
  return RMSNORM_OK;
}

rmsnorm_status_t ln_fwd_impl(const void* x, const void* gamma, const void* beta, void* y,
                             float* mean, float* rstd, int64_t M, int64_t N, float eps, int xd,
                             int wd, cudaStream_t stream) {
  rmsnorm_status_t st = check_sizes(M, N, eps);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok(xd, wd)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if (M == 0) return RMSNORM_OK;
  if (!x || !gamma || !y) return RMSNORM_ERR_INVALID_ARG;
  const size_t xs = (size_t)esize(xd), ws = (size_t)esize(wd);
  if (!aligned_to(x, xs) || !aligned_to(y, xs) || !aligned_to(gamma, ws) ||
      (beta && !aligned_to(beta, ws)) || (mean && !aligned_to(mean, 4)) ||
      (rstd && !aligned_to(rstd, 4)))
    return RMSNORM_ERR_MISALIGNED;
  const size_t act = (size_t)M * (size_t)N * xs, gb = (size_t)N * ws, rb = (size_t)M * 4;
  const void* outs[3] = {y, mean, rstd};
  const size_t olen[3] = {act, rb, rb};
  const void* ins[3] = {x, gamma, beta};
  const size_t ilen[3] = {act, gb, gb};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], olen[i], ins[j], ilen[j])) return RMSNORM_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], olen[i], outs[j], olen[j])) return RMSNORM_ERR_INVALID_ARG;
  }
  const bool vec_ok = aligned_to(x, 16) && aligned_to(y, 16) && aligned_to(gamma, 16) &&
                      (!beta || aligned_to(beta, 16)) && (N * (int64_t)xs) % 16 == 0;
  Plan p;
  if ((st = ln_plan(false, M, N, xd, wd, vec_ok, &p)) != RMSNORM_OK) return st;
  int dev;
  if ((st = current_device(&dev)) != RMSNORM_OK) return st;
  if ((st = size_grid(&p, M, dev)) != RMSNORM_OK) return st;
  LnParams prm = {};
  prm.x = x;
  prm.gamma = gamma;
  prm.beta = beta;
  prm.y = y;
  prm.mean = mean;
  prm.rstd = rstd;
  prm.M = M;
  prm.N = (int)N;
  prm.nvec = vec_ok ? (int)(N / per_vec(xd)) : 0;
  prm.eps = eps;
  prm.inv_n = 1.0f / (float)N;
  prm.l2_rows = p.l2_ahead;
  const cudaError_t e =
      launch(reinterpret_cast<LnKernel>(const_cast<void*>(p.fn)), p.grid, p.threads, p.smem,
             stream, prm);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "LayerNorm forward launch");
  }
  return RMSNORM_OK;
}

// Stage-1 CTA count bound of the LayerNorm backward for these sizes (the
// grid of the plan for 16-byte aligned operands; every launch clamps to it).
rmsnorm_status_t ln_partial_rows(int64_t M, int N, int xd, int wd, int device, int* rows) {
  Plan pl;
  rmsnorm_status_t st = ln_plan(true, M, N, xd, wd, (int64_t)N * esize(xd) % 16 == 0, &pl);
  if (st != RMSNORM_OK) return st;
  if ((st = size_grid(&pl, M, device)) != RMSNORM_OK) return st;
  *rows = pl.grid;
  // operands off 16 bytes may take the wide kernel, whose grid the aligned
  // plan's need not bound
  Plan pw;
  if (ln_plan(true, M, N, xd, wd, false, &pw) == RMSNORM_OK && pw.family == kWide &&
      size_grid(&pw, M, device) == RMSNORM_OK && pw.grid > *rows)
    *rows = pw.grid;
  return RMSNORM_OK;
}

rmsnorm_status_t ln_bwd_impl(const void* dy, const void* x, const float* mean,
                             const float* rstd, const void* gamma, void* dx, float* dgamma,
                             float* dbeta, void* workspace, size_t workspace_bytes, int64_t M,
                             int64_t N, float eps, int xd, int wd, cudaStream_t stream) {
  rmsnorm_status_t st = check_sizes(M, N, eps);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok(xd, wd)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if ((mean == nullptr) != (rstd == nullptr)) return RMSNORM_ERR_INVALID_ARG;
  if (M == 0) {
    for (float* out : {dgamma, dbeta})
      if (out) {
        const cudaError_t e = cudaMemsetAsync(out, 0, (size_t)N * 4, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync of a weight gradient");
      }
    return RMSNORM_OK;
  }
  if (!dy || !x || !gamma || !dx) return RMSNORM_ERR_INVALID_ARG;
  const size_t xs = (size_t)esize(xd), ws = (size_t)esize(wd);
  if (!aligned_to(dy, xs) || !aligned_to(x, xs) || !aligned_to(dx, xs) ||
      !aligned_to(gamma, ws) || (mean && (!aligned_to(mean, 4) || !aligned_to(rstd, 4))) ||
      (dgamma && !aligned_to(dgamma, 4)) || (dbeta && !aligned_to(dbeta, 4)))
    return RMSNORM_ERR_MISALIGNED;
  const size_t act = (size_t)M * (size_t)N * xs, gb = (size_t)N * ws, rb = (size_t)M * 4,
               db = (size_t)N * 4;
  const bool want = dgamma || dbeta;
  const int ld_half = round_up((int)N, 4);
  const void* outs[4] = {dx, dgamma, dbeta, nullptr};   // [3]: the workspace, once sized
  size_t olen[4] = {act, db, db, 0};
  const void* ins[5] = {dy, x, gamma, mean, rstd};
  const size_t ilen[5] = {act, act, gb, rb, rb};
  auto overlaps = [&]() {
    for (int i = 0; i < 4; ++i) {
      for (int j = 0; j < 5; ++j)
        if (overlap(outs[i], olen[i], ins[j], ilen[j])) return true;
      for (int j = i + 1; j < 4; ++j)
        if (overlap(outs[i], olen[i], outs[j], olen[j])) return true;
    }
    return false;
  };
  if (overlaps()) return RMSNORM_ERR_INVALID_ARG;
  if (want && (!workspace || !aligned_to(workspace, 16))) return RMSNORM_ERR_WORKSPACE;
  int dev;
  if ((st = current_device(&dev)) != RMSNORM_OK) return st;
  int prows = 0;
  if (want) {
    if ((st = ln_partial_rows(M, (int)N, xd, wd, dev, &prows)) != RMSNORM_OK) return st;
    const size_t need = (size_t)prows * 2 * ld_half * 4;
    if (workspace_bytes < need) return RMSNORM_ERR_WORKSPACE;
    outs[3] = workspace;
    olen[3] = need;
    if (overlaps()) return RMSNORM_ERR_INVALID_ARG;
  }
  const bool vec_ok = aligned_to(x, 16) && aligned_to(dy, 16) && aligned_to(dx, 16) &&
                      aligned_to(gamma, 16) && (N * (int64_t)xs) % 16 == 0;
  Plan p;
  if ((st = ln_plan(true, M, N, xd, wd, vec_ok, &p, mean != nullptr)) != RMSNORM_OK) return st;
  unsigned* status = nullptr;
  if ((st = size_grid(&p, M, dev, &status)) != RMSNORM_OK) return st;
  if (want && p.grid > prows) p.grid = prows;
  LnParams prm = {};
  prm.x = x;
  prm.dy = dy;
  prm.gamma = gamma;
  prm.y = dx;
  prm.mean = const_cast<float*>(mean);
  prm.rstd = const_cast<float*>(rstd);
  prm.partial = want ? static_cast<float*>(workspace) : nullptr;
  prm.M = M;
  prm.N = (int)N;
  prm.nvec = vec_ok ? (int)(N / per_vec(xd)) : 0;
  prm.ld_half = ld_half;
  prm.eps = eps;
  prm.inv_n = 1.0f / (float)N;
  prm.stages = p.stages;
  prm.wait_limit = wait_limit();
  prm.status = status;
  prm.l2_rows = p.l2_ahead;
  cudaError_t e = launch(reinterpret_cast<LnKernel>(const_cast<void*>(p.fn)), p.grid, p.threads,
                         p.smem, stream, prm);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "LayerNorm backward stage-1 launch");
  }
  if (!want) return RMSNORM_OK;
  // stage 2: both halves of the partial rows, summed per column in a fixed order
  const float* part = static_cast<const float*>(workspace);
  e = launch_colsum(part, p.grid, 2 * ld_half / 4,
                    ColSumOut{dgamma, dbeta, ld_half / 4, (int)N, 0}, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "LayerNorm backward stage-2 launch");
  }
  return RMSNORM_OK;
}

// ---------------------------------------------------------------- backward

// Stage-1 CTA count bound for these sizes: the grid of the plan for 16-byte
// aligned operands.  Every launch clamps its stage-1 grid to it, so the
// workspace query does not need the pointers.
// aligned_rows (optional): the aligned plan's bound alone.
rmsnorm_status_t bwd_partial_rows(int64_t M, int N, int xd, int wd, int device, int* rows,
                                  int* aligned_rows = nullptr) {
  Plan pl;
  rmsnorm_status_t st = make_plan(kBwd, M, N, xd, wd, true, true, true, &pl);
  if (st != RMSNORM_OK) {
    // a forced variant that does not fit aligned operands: fall back to the
    // unforced plan for the bound
    return st;
  }
  if ((st = size_grid(&pl, M, device)) != RMSNORM_OK) return st;
  *rows = pl.cluster > 0 ? pl.grid / pl.cluster : pl.grid;   // a partial row per cluster
  if (aligned_rows) *aligned_rows = *rows;
  // operands at other offsets may take the wide kernel, whose grid (one row
  // per CTA, several CTAs per SM) the aligned plan's need not bound
  Plan pw;
  if (make_plan(kBwd, M, N, xd, wd, false, false, true, &pw) == RMSNORM_OK &&
      pw.family == kWide && size_grid(&pw, M, device) == RMSNORM_OK && pw.grid > *rows)
    *rows = pw.grid;
  return RMSNORM_OK;
}

// Backward and fused-add backward.  dres (fused-add backward only) is the
// residual-path gradient; its result dh = dx + dres goes to dx, which is then
// the same buffer.  dgamma is fp32, or bf16 when dgamma_bf16.  fit: a
// workspace of fixed size (the allocation-free entry point's scratch) that
// holds the aligned plan's partial rows but not the wide kernel's bounds the
// stage-1 grid instead of failing.
rmsnorm_status_t bwd_impl(const void* dy, const void* x, const float* rstd, const void* gamma,
                          void* dx, const void* dres, void* dgamma, bool dgamma_bf16,
                          void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                          float eps, int xd, int wd, cudaStream_t stream, bool fit = false) {
  rmsnorm_status_t st = check_sizes(M, N, eps);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok(xd, wd)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  const size_t gsz = dgamma_bf16 ? 2 : 4;
  if (M == 0) {
    if (dgamma) {
      const cudaError_t e = cudaMemsetAsync(dgamma, 0, (size_t)N * gsz, stream);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync of dgamma");
    }
    return RMSNORM_OK;
  }
  if (!dy || !x || !gamma || !dx) return RMSNORM_ERR_INVALID_ARG;
  const size_t xs = (size_t)esize(xd), ws = (size_t)esize(wd);
  if (!aligned_to(dy, xs) || !aligned_to(x, xs) || !aligned_to(dx, xs) ||
      !aligned_to(gamma, ws) || (rstd && !aligned_to(rstd, 4)) ||
      (dgamma && !aligned_to(dgamma, gsz)) || (dres && !aligned_to(dres, xs)))
    return RMSNORM_ERR_MISALIGNED;
  const size_t act = (size_t)M * (size_t)N * xs, gb = (size_t)N * ws, rb = (size_t)M * 4,
               db = (size_t)N * gsz;
  if (overlap(dx, act, dy, act) || overlap(dx, act, x, act) || overlap(dx, act, gamma, gb) ||
      overlap(dx, act, rstd, rb) || overlap(dx, act, dgamma, db) ||
      overlap(dgamma, db, dy, act) || overlap(dgamma, db, x, act) ||
      overlap(dgamma, db, gamma, gb) || overlap(dgamma, db, rstd, rb))
    return RMSNORM_ERR_INVALID_ARG;
  if (dres && dres != dx && overlap(dres, act, dx, act)) return RMSNORM_ERR_INVALID_ARG;

  int dev;
  if ((st = current_device(&dev)) != RMSNORM_OK) return st;
  const int ld = round_up((int)N, 4);
  int prows = 0, prows_aligned = 0;
  if (dgamma) {
    if ((st = bwd_partial_rows(M, (int)N, xd, wd, dev, &prows, &prows_aligned)) != RMSNORM_OK)
      return st;
    size_t need = (size_t)prows * ld * 4;
    if (fit && workspace_bytes < need && workspace_bytes >= (size_t)prows_aligned * ld * 4) {
      prows = (int)(workspace_bytes / ((size_t)ld * 4));
      need = (size_t)prows * ld * 4;
    }
    if (!workspace || workspace_bytes < need || !aligned_to(workspace, 16))
      return RMSNORM_ERR_WORKSPACE;
    if (overlap(workspace, need, dx, act) || overlap(workspace, need, dgamma, db) ||
        overlap(workspace, need, dy, act) || overlap(workspace, need, x, act) ||
        overlap(workspace, need, gamma, gb) || overlap(workspace, need, rstd, rb))
      return RMSNORM_ERR_INVALID_ARG;
  }

  const uintptr_t mx = reinterpret_cast<uintptr_t>(x) & 15;
  const uintptr_t mdy = reinterpret_cast<uintptr_t>(dy) & 15;
  const uintptr_t mdx = reinterpret_cast<uintptr_t>(dx) & 15;
  // the output dx (and dres, read where dh is written) set the alignment
  const bool out_same = !dres || (reinterpret_cast<uintptr_t>(dres) & 15) == mdx;
  const bool same = out_same && mdy == mx && mdx == mx;
  const bool aligned16 = same && mx == 0 && aligned_to(gamma, 16);
  Plan pl;
  const bool frame16 = mdx == 0 && aligned_to(gamma, 16);
  if ((st = make_plan(dres ? kFusedBwd : kBwd, M, (int)N, xd, wd, aligned16, same,
                      rstd != nullptr, &pl, out_same, frame16)) != RMSNORM_OK)
    return st;
  unsigned* status = nullptr;
  if ((st = size_grid(&pl, M, dev, &status)) != RMSNORM_OK) return st;
  if (pl.cluster > 0) {
    if (dgamma && pl.grid / pl.cluster > prows) pl.grid = prows * pl.cluster;
  } else if (dgamma && pl.grid > prows) {
    pl.grid = prows;
  }
  if (pl.period > 1) {   // ragged rows: whole residue classes only
    pl.grid = pl.grid / pl.period * pl.period;
    if (pl.grid < pl.period) return RMSNORM_ERR_WORKSPACE;
  }

  BwdParams prm = {};
  prm.dy = dy;
  prm.x = x;
  prm.dres = dres;
  prm.rstd = rstd;
  prm.gamma = gamma;
  prm.dx = dx;
  prm.partial = dgamma ? static_cast<float*>(workspace) : nullptr;
  prm.M = M;
  prm.N = (int)N;
  prm.nvec = (int)(N / per_vec(xd));
  prm.ld_partial = ld;
  prm.eps = eps;
  prm.inv_n = 1.0f / (float)N;
  prm.stages = pl.stages;
  prm.wait_limit = wait_limit();
  prm.status = status;
  prm.period = pl.period;
  prm.l2_rows = pl.l2_ahead;
  prm.slice = pl.slice;
  prm.x_shift = (int)((mx - mdx) & 15);
  prm.dy_shift = (int)((mdy - mdx) & 15);
  cudaError_t e =
      launch_in_clusters(pl.cluster, pl.bwd, pl.grid, pl.threads, pl.smem, stream, prm);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "backward stage-1 launch");
  }
  if (!dgamma) return RMSNORM_OK;
  // stage 2: the P partial rows summed per column in a fixed order
  const float* part = static_cast<const float*>(workspace);
  e = launch_colsum(part, pl.cluster > 0 ? pl.grid / pl.cluster : pl.grid, ld / 4,
                    ColSumOut{dgamma, nullptr, ld / 4, (int)N, dgamma_bf16 ? 1 : 0}, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "backward stage-2 launch");
  }
  return RMSNORM_OK;
}

// ---------------------------------------------------------------- backward
// without allocation

// Scratch for the dgamma partial rows of rmsnorm_bwd_noalloc.  It lives in
// the library's device image, so every GPU that loads the library holds it
// until the process exits; calls share it and it keeps the last call's
// partial rows (each call overwrites every partial it later reads).
static __device__ __align__(256) unsigned char g_noalloc_scratch[RMSNORM_BWD_NOALLOC_SCRATCH_BYTES];

void* g_noalloc_addr[64];

// Device address of the scratch on `device` (the current device), looked up
// once per device with cudaGetSymbolAddress: in host code the array's name is
// only a host-side stand-in and must never be handed to a kernel.
rmsnorm_status_t noalloc_scratch(int device, void** out) {
  if (device < 0 || device >= 64) return RMSNORM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_addr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return cuda_fail(e, "cudaGetSymbolAddress of the scratch");
    }
    g_noalloc_addr[device] = p;
  }
  *out = g_noalloc_addr[device];
  return RMSNORM_OK;
}

}  // namespace
}  // namespace rmsn

// ======================================================================= C ABI

using namespace rmsn;

extern "C" {

rmsnorm_status_t rmsnorm_fwd(const void* x, const void* gamma, void* y, float* rstd, int64_t M,
                             int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                             rmsnorm_dtype_t w_dtype, cudaStream_t stream) {
  return fwd_impl(kFwd, x, nullptr, gamma, y, rstd, M, N, eps, (int)x_dtype, (int)w_dtype,
                  stream);
}

rmsnorm_status_t rmsnorm_fused_add_fwd(const void* x, void* residual, const void* gamma, void* y,
                                       float* rstd, int64_t M, int64_t N, float eps,
                                       rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                       cudaStream_t stream) {
  return fwd_impl(kFused, x, residual, gamma, y, rstd, M, N, eps, (int)x_dtype, (int)w_dtype,
                  stream);
}

rmsnorm_status_t rmsnorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype_t x_dtype,
                                            rmsnorm_dtype_t w_dtype, int device,
                                            size_t* bytes) {
  if (!bytes) return RMSNORM_ERR_INVALID_ARG;
  *bytes = 0;
  rmsnorm_status_t st = check_sizes(M, N, 0.f);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok((int)x_dtype, (int)w_dtype)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if (M == 0) return RMSNORM_OK;
  if (device < 0 && (st = current_device(&device)) != RMSNORM_OK) return st;
  int rows = 0;
  if ((st = bwd_partial_rows(M, (int)N, (int)x_dtype, (int)w_dtype, device, &rows)) !=
      RMSNORM_OK)
    return st;
  *bytes = (size_t)rows * (size_t)round_up((int)N, 4) * 4;
  return RMSNORM_OK;
}

rmsnorm_status_t rmsnorm_bwd(const void* dy, const void* x, const float* rstd, const void* gamma,
                             void* dx, float* dgamma, void* workspace, size_t workspace_bytes,
                             int64_t M, int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                             rmsnorm_dtype_t w_dtype, cudaStream_t stream) {
  return bwd_impl(dy, x, rstd, gamma, dx, nullptr, dgamma, false, workspace, workspace_bytes, M,
                  N, eps, (int)x_dtype, (int)w_dtype, stream);
}

rmsnorm_status_t rmsnorm_fwd_strided(const void* x, int64_t x_stride_token,
                                     int64_t x_stride_head, const void* gamma, void* y,
                                     int64_t y_stride_token, int64_t y_stride_head, float* rstd,
                                     int64_t T, int64_t H, int64_t D, float eps,
                                     rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                     cudaStream_t stream) {
  return fwd_strided_impl(x, x_stride_token, x_stride_head, gamma, y, y_stride_token,
                          y_stride_head, rstd, T, H, D, eps, (int)x_dtype, (int)w_dtype, stream);
}

rmsnorm_status_t layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y,
                               float* mean, float* rstd, int64_t M, int64_t N, float eps,
                               rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                               cudaStream_t stream) {
  return ln_fwd_impl(x, gamma, beta, y, mean, rstd, M, N, eps, (int)x_dtype, (int)w_dtype,
                     stream);
}

rmsnorm_status_t layernorm_bwd_workspace_size(int64_t M, int64_t N, rmsnorm_dtype_t x_dtype,
                                              rmsnorm_dtype_t w_dtype, int device,
                                              size_t* bytes) {
  if (!bytes) return RMSNORM_ERR_INVALID_ARG;
  *bytes = 0;
  rmsnorm_status_t st = check_sizes(M, N, 0.f);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok((int)x_dtype, (int)w_dtype)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if (M == 0) return RMSNORM_OK;
  if (device < 0 && (st = current_device(&device)) != RMSNORM_OK) return st;
  int rows = 0;
  if ((st = ln_partial_rows(M, (int)N, (int)x_dtype, (int)w_dtype, device, &rows)) !=
      RMSNORM_OK)
    return st;
  *bytes = (size_t)rows * 2 * (size_t)round_up((int)N, 4) * 4;
  return RMSNORM_OK;
}

rmsnorm_status_t layernorm_bwd(const void* dy, const void* x, const float* mean,
                               const float* rstd, const void* gamma, void* dx, float* dgamma,
                               float* dbeta, void* workspace, size_t workspace_bytes, int64_t M,
                               int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                               rmsnorm_dtype_t w_dtype, cudaStream_t stream) {
  return ln_bwd_impl(dy, x, mean, rstd, gamma, dx, dgamma, dbeta, workspace, workspace_bytes, M,
                     N, eps, (int)x_dtype, (int)w_dtype, stream);
}

rmsnorm_status_t rmsnorm_fwd_fp8(const void* x, void* residual, const void* gamma, void* q,
                                 float* scale, float* rstd, int64_t M, int64_t N, float eps,
                                 rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                 cudaStream_t stream) {
  return fwd_quant_impl(kOutFp8, x, residual, gamma, 0.f, q, scale, rstd, M, N, eps,
                        (int)x_dtype, (int)w_dtype, stream);
}

rmsnorm_status_t rmsnorm_fwd_nvfp4(const void* x, void* residual, const void* gamma,
                                   float global_scale, void* q, void* block_scale, float* rstd,
                                   int64_t M, int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                                   rmsnorm_dtype_t w_dtype, cudaStream_t stream) {
  return fwd_quant_impl(kOutNvfp4, x, residual, gamma, global_scale, q, block_scale, rstd, M, N,
                        eps, (int)x_dtype, (int)w_dtype, stream);
}

rmsnorm_status_t rmsnorm_fused_add_bwd(const void* dy, const void* h, const float* rstd,
                                       const void* gamma, void* dres, void* dgamma,
                                       rmsnorm_dtype_t dgamma_dtype, void* workspace,
                                       size_t workspace_bytes, int64_t M, int64_t N, float eps,
                                       rmsnorm_dtype_t x_dtype, rmsnorm_dtype_t w_dtype,
                                       cudaStream_t stream) {
  if (dgamma_dtype != RMSNORM_F32 && dgamma_dtype != RMSNORM_BF16)
    return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if (M > 0 && dres == nullptr) return RMSNORM_ERR_INVALID_ARG;
  return bwd_impl(dy, h, rstd, gamma, dres, dres, dgamma, dgamma_dtype == RMSNORM_BF16,
                  workspace, workspace_bytes, M, N, eps, (int)x_dtype, (int)w_dtype, stream);
}

rmsnorm_status_t rmsnorm_bwd_noalloc(const void* dy, const void* x, const float* rstd,
                                     const void* gamma, void* dx, float* dgamma, int64_t M,
                                     int64_t N, float eps, rmsnorm_dtype_t x_dtype,
                                     rmsnorm_dtype_t w_dtype, cudaStream_t stream) {
  void* scratch = nullptr;
  if (dgamma != nullptr && M > 0 && check_sizes(M, N, eps) == RMSNORM_OK) {
    int dev;
    rmsnorm_status_t st = current_device(&dev);
    if (st != RMSNORM_OK) return st;
    if ((st = noalloc_scratch(dev, &scratch)) != RMSNORM_OK) return st;
  }
  // the workspace entry point with the static scratch as its workspace: a
  // shape whose aligned plan's partial rows exceed the scratch gets
  // RMSNORM_ERR_WORKSPACE; the wide kernel's larger grid is bounded to it
  return bwd_impl(dy, x, rstd, gamma, dx, nullptr, dgamma, false, scratch,
                  scratch ? (size_t)RMSNORM_BWD_NOALLOC_SCRATCH_BYTES : 0, M, N, eps,
                  (int)x_dtype, (int)w_dtype, stream, true);
}

rmsnorm_status_t rmsnorm_check_device(cudaStream_t stream) {
  int dev;
  rmsnorm_status_t st = current_device(&dev);
  if (st != RMSNORM_OK) return st;
  DevInfo di;
  cudaError_t e = device_info(dev, &di);
  if (e != cudaSuccess) return cuda_fail(e, "device attributes");
  unsigned flags = 0;
  if ((e = cudaMemcpyAsync(&flags, di.status, sizeof flags, cudaMemcpyDeviceToHost, stream)) !=
          cudaSuccess ||
      (e = cudaMemsetAsync(di.status, 0, sizeof flags, stream)) != cudaSuccess ||
      (e = cudaStreamSynchronize(stream)) != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "reading the device status word");
  }
  return (flags & kStatusWaitTimeout) ? RMSNORM_ERR_TIMEOUT : RMSNORM_OK;
}

const char* rmsnorm_last_error(void) { return g_last_error; }

void rmsnorm_reload_debug_env(void) { g_env = read_debug_env(); }

const char* rmsnorm_status_string(rmsnorm_status_t status) {
  switch (status) {
    case RMSNORM_OK: return "ok";
    case RMSNORM_ERR_INVALID_ARG: return "invalid argument";
    case RMSNORM_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype pair";
    case RMSNORM_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case RMSNORM_ERR_WORKSPACE: return "workspace missing or too small";
    case RMSNORM_ERR_CUDA: return "CUDA runtime error";
    case RMSNORM_ERR_TIMEOUT: return "a kernel gave up waiting for its own bulk copies";
    default: return "unknown status";
  }
}

rmsnorm_status_t rmsnorm_describe_plan(int op, int64_t M, int64_t N, rmsnorm_dtype_t x_dtype,
                                       rmsnorm_dtype_t w_dtype, int aligned16, int device,
                                       char* buf, size_t len) {
  if (!buf || len == 0 || op < 0 || op > 10) return RMSNORM_ERR_INVALID_ARG;
  buf[0] = 0;
  rmsnorm_status_t st = check_sizes(M, N, 0.f);
  if (st != RMSNORM_OK) return st;
  if (!dtype_pair_ok((int)x_dtype, (int)w_dtype)) return RMSNORM_ERR_UNSUPPORTED_DTYPE;
  if (device < 0 && (st = current_device(&device)) != RMSNORM_OK) return st;
  Plan pl;
  if (op >= 9) {
    if ((st = ln_plan(op == 10, M, N, (int)x_dtype, (int)w_dtype,
                      aligned16 != 0 && (N * esize((int)x_dtype)) % 16 == 0, &pl,
                      op == 10)) != RMSNORM_OK)
      return st;
  } else if (op >= 5) {
    const int out = op <= 6 ? kOutFp8 : kOutNvfp4;
    if (out == kOutNvfp4 && N % 16 != 0) return RMSNORM_ERR_INVALID_ARG;
    if ((st = quant_plan(out, op == 6 || op == 8, N, (int)x_dtype, (int)w_dtype,
                         aligned16 != 0 && (N * esize((int)x_dtype)) % 16 == 0, &pl)) !=
        RMSNORM_OK)
      return st;
  } else if (op == 4) {
    if ((st = strided_plan(N, (int)x_dtype, (int)w_dtype,
                           aligned16 != 0 && (N * esize((int)x_dtype)) % 16 == 0, &pl)) !=
        RMSNORM_OK)
      return st;
  } else if (aligned16 == 2) {   // outputs on 16 bytes, x (and dy) off them
    if ((st = make_plan(op, M, (int)N, (int)x_dtype, (int)w_dtype, false, false, true, &pl,
                        true, true)) != RMSNORM_OK)
      return st;
  } else if ((st = make_plan(op, M, (int)N, (int)x_dtype, (int)w_dtype, aligned16 != 0,
                             aligned16 != 0, true, &pl)) != RMSNORM_OK) {
    return st;
  }
  if ((st = size_grid(&pl, M > 0 ? M : 1, device)) != RMSNORM_OK) return st;
  describe(op, pl, buf, len);
  return RMSNORM_OK;
}

}  // extern "C"
