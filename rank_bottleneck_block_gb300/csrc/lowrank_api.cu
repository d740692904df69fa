// C ABI of liblowrank.so: argument validation, workspace layout and the
// launch sequence of each entry point (declared and documented in
// include/lowrank.h).  Every step of the path runs in this library's kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/lowrank.h"
#include "common.cuh"
#include "gemm.h"
#include "attn_kernels.cuh"
#include "small_kernels.cuh"

namespace lr {

// ------------------------------------------------------------------ errors
static thread_local std::string t_last_error;

static lr_status fail(lr_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

#define LR_CUDA(expr)                                                                       \
  do {                                                                                      \
    cudaError_t e_ = (expr);                                                                \
    if (e_ != cudaSuccess) return fail(LR_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

#define LR_TRY(expr)                   \
  do {                                 \
    lr_status s_ = (expr);             \
    if (s_ != LR_OK) return s_;        \
  } while (0)

// --------------------------------------------------------- device state
// The device error word: kernels OR bits into it instead of trapping.
__device__ unsigned g_device_error_word;

static constexpr int kMaxDevices = 64;
static unsigned* s_err_ptr[kMaxDevices];
static int s_sms[kMaxDevices];
static std::mutex s_dev_mu;

static lr_status current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(LR_ERR_UNSUPPORTED, "no CUDA device: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return fail(LR_ERR_UNSUPPORTED, "device ordinal %d out of range", *dev);
  return LR_OK;
}

// Looked up once per device with that device current; later calls reuse it.
static lr_status device_error_word(unsigned** out) {
  int dev;
  LR_TRY(current_device(&dev));
  std::lock_guard<std::mutex> lk(s_dev_mu);
  if (!s_err_ptr[dev]) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(LR_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                  minor);
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_device_error_word);
    if (e != cudaSuccess) return fail(LR_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
    s_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = s_err_ptr[dev];
  return LR_OK;
}

int device_sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 1;
  if (!s_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    s_sms[dev] = n > 0 ? n : 1;
  }
  return s_sms[dev];
}

// ------------------------------------------------------------- profiling
// Every launch of the library increments a counter.  While profiling is on,
// each launch is also bracketed by two CUDA events recorded on its stream,
// tagged with the kernel's name and its algorithmic FLOPs / bytes; stopping
// synchronises the events and aggregates per name.
static std::atomic<unsigned long long> s_launches{0};

struct ProfRec {
  std::string name;
  cudaEvent_t a, b;
  double flops, bytes;
};
struct ProfAgg {
  std::string name;
  long long n;
  double ms, flops, bytes;
};
static std::mutex s_prof_mu;
static bool s_prof_on = false;
static std::string s_prof_filter;  // record only kernels whose name starts with this (empty: all)
static std::vector<ProfRec> s_prof;
static std::vector<cudaEvent_t> s_event_pool;
static std::vector<ProfAgg> s_prof_result;

static cudaEvent_t pool_event() {
  if (!s_event_pool.empty()) {
    cudaEvent_t e = s_event_pool.back();
    s_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

struct LaunchScope {
  bool on;
  ProfRec rec;
  cudaStream_t st;
  LaunchScope(const std::string& name, cudaStream_t s, double flops, double bytes) : on(false), st(s) {
    s_launches.fetch_add(1, std::memory_order_relaxed);
    std::lock_guard<std::mutex> lk(s_prof_mu);
    if (!s_prof_on) return;
    if (!s_prof_filter.empty() && name.compare(0, s_prof_filter.size(), s_prof_filter) != 0) return;
    on = true;
    rec.name = name;
    rec.flops = flops;
    rec.bytes = bytes;
    rec.a = pool_event();
    rec.b = pool_event();
    cudaEventRecord(rec.a, st);
  }
  ~LaunchScope() {
    if (!on) return;
    cudaEventRecord(rec.b, st);
    std::lock_guard<std::mutex> lk(s_prof_mu);
    s_prof.push_back(rec);
  }
};

// ----------------------------------------------------------- GEMM dispatch
struct Ctx {
  lr_dtype dt;
  int act;    // pair activation: 0 SiLU, 1 identity
  size_t es;  // element size of the storage dtype
  cudaStream_t st;
  unsigned* err;
  int sms;
  int chunk;  // row-partial chunk width of the engine
};

// A second stream for work that can run beside the caller's stream within one entry point, with the
// events that fork it from and join it back to the caller's stream (under CUDA graph capture the
// fork makes it part of the capture).  One per host thread and device, created on first use and kept.
struct SideStream {
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

static lr_status side_stream(SideStream** out) {
  thread_local SideStream per_dev[32];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 32) return fail(LR_ERR_CUDA, "no current device");
  SideStream& s = per_dev[dev];
  if (!s.st) {
    if (cudaStreamCreateWithFlags(&s.st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess)
      return fail(LR_ERR_CUDA, "side stream: %s", cudaGetErrorString(cudaGetLastError()));
  }
  *out = &s;
  return LR_OK;
}

// Tile width of the SwiGLU dual GEMM (two accumulators: 256 fills TMEM with one buffer,
// 128 keeps two buffers).
static constexpr int kSwigluBn = 256;

// Tile width from waves of pair tiles (256 rows, one per SM pair); a 128-wide tile costs
// about 0.75 of a 256-wide one (its shared-memory traffic per FLOP is 1.5x higher).
static int pick_bn(const GemmCall& g, int sms) {
  if (g.N <= 128) return 128;
  const long long slots = std::max(1, sms / 2);
  const long long mp = (g.M + 255) / 256;
  const long long t256 = mp * ((g.N + 255) / 256) * g.batches * std::max(1, g.ksplit);
  const long long t128 = mp * ((g.N + 127) / 128) * g.batches * std::max(1, g.ksplit);
  const double c256 = static_cast<double>((t256 + slots - 1) / slots);
  const double c128 = 0.75 * static_cast<double>((t128 + slots - 1) / slots);
  return c128 < c256 ? 128 : 256;
}

template <EpiKind K, bool A_MN, bool B_MN, bool RB = false>
static cudaError_t umma_bn(const GemmCall& g, cudaStream_t st) {
  if (g.bn == 128) return launch_umma<K, 128, A_MN, B_MN, RB>(g, st);
  return launch_umma<K, 256, A_MN, B_MN, RB>(g, st);
}

// Row-batched calls (the attention GEMMs over all heads) run the kernels built for them.
static cudaError_t dispatch_rowbatch(EpiKind k, GemmCall& g, cudaStream_t st) {
  const bool kk = !g.a_mn && !g.b_mn, km = !g.a_mn && g.b_mn, mm = g.a_mn && g.b_mn;
  switch (k) {
    case EPI_F32: if (kk) return umma_bn<EPI_F32, false, false, true>(g, st); break;
    case EPI_STORE:
      if (km) return umma_bn<EPI_STORE, false, true, true>(g, st);
      if (mm) return umma_bn<EPI_STORE, true, true, true>(g, st);
      break;
    case EPI_ATTN_BWD:
      if (kk && g.nacc == 2) return launch_umma<EPI_ATTN_BWD, 256, false, false, true>(g, st);
      break;
    default: break;
  }
  return cudaErrorNotSupported;
}

static cudaError_t dispatch_bf16(EpiKind k, GemmCall& g, cudaStream_t st, int sms) {
  (void)sms;
  if (g.rowbatch) return dispatch_rowbatch(k, g, st);
  const bool kk = !g.a_mn && !g.b_mn, km = !g.a_mn && g.b_mn, mm = g.a_mn && g.b_mn;
  switch (k) {
    case EPI_NORM_SILU: if (kk) return umma_bn<EPI_NORM_SILU, false, false>(g, st); break;
    case EPI_SILU: if (kk) return umma_bn<EPI_SILU, false, false>(g, st); break;
    case EPI_STORE:
      if (kk) return umma_bn<EPI_STORE, false, false>(g, st);
      if (km) return umma_bn<EPI_STORE, false, true>(g, st);
      break;
    case EPI_RESID: if (kk) return umma_bn<EPI_RESID, false, false>(g, st); break;
    case EPI_SWIGLU:
      if (kk && g.nacc == 2) return umma_bn<EPI_SWIGLU, false, false>(g, st);
      break;
    case EPI_SWIGLU_H:
      if (kk && g.nacc == 2) return launch_umma<EPI_SWIGLU_H, 256, false, false>(g, st);
      break;
    case EPI_NORM_SWIGLU:
      if (kk && g.nacc == 2) return launch_umma<EPI_NORM_SWIGLU, 256, false, false>(g, st);
      break;
    case EPI_SWIGLU_BWD_NORM: if (km) return umma_bn<EPI_SWIGLU_BWD_NORM, false, true>(g, st); break;
    case EPI_F32_SS: if (kk && g.ksplit == 1) return umma_bn<EPI_F32_SS, false, false>(g, st); break;
    case EPI_DSILU: if (km) return umma_bn<EPI_DSILU, false, true>(g, st); break;
    case EPI_DSILU_Z: if (km) return umma_bn<EPI_DSILU_Z, false, true>(g, st); break;
    case EPI_DSILU_NORM: if (km) return umma_bn<EPI_DSILU_NORM, false, true>(g, st); break;
    case EPI_SWIGLU_BWD: if (km) return umma_bn<EPI_SWIGLU_BWD, false, true>(g, st); break;
    case EPI_SWIGLU_REBWD:
      if (kk && g.nacc == 3) return launch_umma<EPI_SWIGLU_REBWD, 256, false, false>(g, st);
      break;
    case EPI_DX_NORM: if (km) return umma_bn<EPI_DX_NORM, false, true>(g, st); break;
    case EPI_F32:
      if (mm) return umma_bn<EPI_F32, true, true>(g, st);
      break;
    default: break;
  }
  return cudaErrorNotSupported;
}

static cudaError_t dispatch_f32(EpiKind k, GemmCall& g, cudaStream_t st) {
  switch (k) {
    case EPI_NORM_SILU: return launch_simt<EPI_NORM_SILU>(g, st);
    case EPI_SILU: return launch_simt<EPI_SILU>(g, st);
    case EPI_STORE: return launch_simt<EPI_STORE>(g, st);
    case EPI_RESID: return launch_simt<EPI_RESID>(g, st);
    case EPI_SWIGLU: return launch_simt<EPI_SWIGLU>(g, st);
    case EPI_DSILU: return launch_simt<EPI_DSILU>(g, st);
    case EPI_DSILU_NORM: return launch_simt<EPI_DSILU_NORM>(g, st);
    case EPI_SWIGLU_BWD: return launch_simt<EPI_SWIGLU_BWD>(g, st);
    case EPI_DX_NORM: return launch_simt<EPI_DX_NORM>(g, st);
    case EPI_F32: return launch_simt<EPI_F32>(g, st);
    case EPI_NORM_SWIGLU: return launch_simt<EPI_NORM_SWIGLU>(g, st);
    case EPI_SWIGLU_BWD_NORM: return launch_simt<EPI_SWIGLU_BWD_NORM>(g, st);
    case EPI_F32_SS: return launch_simt<EPI_F32_SS>(g, st);
    default: return cudaErrorNotSupported;
  }
}

static const char* epi_name(EpiKind k) {
  static const char* names[] = {"norm_silu", "silu",       "store",  "resid",       "swiglu",        "dsilu",
                                "dsilu_norm", "swiglu_bwd", "dx_norm", "f32", "norm_swiglu", "swiglu_bwd_norm",
                                "f32_ss", "attn_bwd", "swiglu_rebwd", "swiglu", "dsilu_z"};
  return (k >= 0 && k < EPI_COUNT) ? names[k] : "?";
}

static lr_status gemm(const Ctx& c, EpiKind k, GemmCall& g, double extra_bytes = 0) {
  g.err = c.err;
  if (g.nacc < 1) g.nacc = 1;
  if (g.batches < 1) g.batches = 1;
  if (g.ksplit < 1) g.ksplit = 1;
  g.ep.M = g.M;
  g.ep.N = g.N;
  g.ep.act = c.act;
  if (c.dt == LR_BF16) {
    if (k == EPI_SWIGLU || k == EPI_SWIGLU_H) g.bn = kSwigluBn;
    else if (k == EPI_NORM_SWIGLU || k == EPI_ATTN_BWD) g.bn = 256;  // split-phase dual-accumulator kernels
    else if (k == EPI_SWIGLU_REBWD) g.bn = 256;  // three accumulators take two TMEM regions in turn
    else if (g.bn != 128 && g.bn != 256) g.bn = pick_bn(g, c.sms);
  } else {
    g.bn = 0;
  }
  std::string name = std::string(c.dt == LR_BF16 ? "umma_" : "simt_") + epi_name(k);
  if (g.bn) name += "_bn" + std::to_string(g.bn);
  double flops = 2.0 * g.M * g.N * static_cast<double>(g.K) * g.nacc * g.batches;
  if (g.causal) {  // every causal mode computes the pair tiles (or K ranges) on or below the diagonal
    const double mp = g.M / 256.0;
    flops *= (mp + 1.0) / (2.0 * mp);
  }
  if (g.grouped) {
    flops = 0.0;
    for (int b = 0; b < g.batches; ++b) flops += 2.0 * g.gM[b] * g.gN[b] * static_cast<double>(g.K);
  }
  LaunchScope scope(name, c.st, flops, extra_bytes);
  cudaError_t e = (c.dt == LR_BF16) ? dispatch_bf16(k, g, c.st, c.sms) : dispatch_f32(k, g, c.st);
  if (e != cudaSuccess)
    return fail(LR_ERR_CUDA, "GEMM %s (M=%d N=%d K=%d) launch failed: %s", epi_name(k), g.M, g.N, g.K,
                cudaGetErrorString(e));
  return LR_OK;
}

static GemmCall new_call(int M, int N, int K) {
  GemmCall g;
  memset(&g, 0, sizeof(g));
  g.M = M;
  g.N = N;
  g.K = K;
  g.nacc = 1;
  g.batches = 1;
  g.ksplit = 1;
  return g;
}

static inline const void* off(const void* p, size_t bytes) { return static_cast<const char*>(p) + bytes; }
static inline void* off(void* p, size_t bytes) { return static_cast<char*>(p) + bytes; }

// --------------------------------------------------- weight gradients
// A weight gradient is dW = X^T dY over K = tokens: a small output with a long
// reduction.  The planner picks the tile width (128 or 256) and a split of K
// over CTAs from a cost model: waves of persistent tiles times the per-tile
// MMA work, plus the fp32 partial traffic of the fixed-order reduction.  At
// most 8 splits, each at least 8 k-blocks long; the device-independent bound
// min(8, max(1, kb / 8)) sizes the workspace.
static int wgrad_split_bound(int K) {
  const int kb = (K + 63) / 64;
  return std::max(1, std::min(8, kb / 8));
}

struct WgradPlan {
  int bn, ksplit;
  double t;  // modelled time (relative units)
};

static int normalise_split(int K, int ks) {
  const int kb = (K + 63) / 64;
  const int per = (kb + ks - 1) / ks;
  return (kb + per - 1) / per;
}

// Modelled time of one pair tile of a weight-gradient GEMM over K / ks tokens.
static double wgrad_tile_time(int bn, int K, int ks) {
  const double per_sm_flops = 2.25e15 / 152.0 * 0.65;  // sustained MMA rate per SM (relative units suffice)
  return 2.0 * 128 * bn * (static_cast<double>(K) / ks) / per_sm_flops * (bn == 128 ? 1.33 : 1.0);
}

static WgradPlan wgrad_plan(const Ctx& c, int M, int N, int K, bool needs_pass) {
  if (c.dt != LR_BF16) return {0, 1, 0.0};
  const double reduce_bw = 4.0e12;  // bytes/s of the partial reduction
  WgradPlan best{256, 1, 1e30};
  const long long slots = std::max(1, c.sms / 2);  // SM pairs
  for (int bn : {256, 128}) {
    const long long tiles = 1LL * ((M + 255) / 256) * ((N + bn - 1) / bn);  // pair tiles
    for (int ks = 1; ks <= wgrad_split_bound(K); ++ks) {
      const int ksn = normalise_split(K, ks);
      if (ksn != ks) continue;
      const long long waves = (tiles * ks + slots - 1) / slots;
      double t = waves * wgrad_tile_time(bn, K, ks);
      if (ks > 1 || needs_pass) t += (static_cast<double>(ks) + 1.0) * M * N * 4.0 / reduce_bw;
      if (t < best.t * 0.98) best = {bn, ks, t};
    }
  }
  return best;
}

static size_t wgrad_part_bytes(lr_dtype dt, int M, int N, int K) {
  const int ks = dt == LR_BF16 ? wgrad_split_bound(K) : 1;
  return static_cast<size_t>(ks) * M * N * sizeof(float);
}

// dst = (A^T B) over K tokens, both operands stored [K, .] row-major (MN-major),
// reduced over splits in a fixed order, times the optional column scale, and the
// optional dg partial sums over row blocks.  Without a split, a scale or dg, the
// GEMM writes the fp32 result straight into the single destination.
// With `pairs` > 0 the GEMM runs without a split on 256-wide tiles and at most that many SM pairs (a
// share of the GPU beside another stream's kernel).
static lr_status wgrad(const Ctx& c, int M, int N, int K, Operand A, Operand B, WgradDst dst, int rows_each,
                       const void* colscale, float* dgpart, float* wpart, int pairs = 0) {
  const bool needs_pass = colscale != nullptr || dgpart != nullptr || rows_each != M;
  const WgradPlan plan = pairs > 0 ? WgradPlan{256, 1, 0.0} : wgrad_plan(c, M, N, K, needs_pass);
  GemmCall g = new_call(M, N, K);
  g.a_mn = g.b_mn = true;
  g.A[0] = A;
  g.B[0] = B;
  g.bn = plan.bn;
  g.ksplit = plan.ksplit;
  g.max_pairs = pairs;
  const bool direct = !needs_pass && plan.ksplit == 1;
  g.ep.out0[0] = direct ? static_cast<void*>(dst.dst[0]) : static_cast<void*>(wpart);
  g.ep.ldo0 = N;
  g.ep.split_stride = 1LL * M * N;
  LR_TRY(gemm(c, EPI_F32, g));
  if (direct) return LR_OK;
  LaunchScope scope("wgrad_reduce", c.st, 0, 4.0 * g.ksplit * M * N + 4.0 * M * N);
  cudaError_t e = (c.dt == LR_BF16)
                      ? launch_wgrad_reduce<bf16>(wpart, g.ksplit, 1LL * M * N, M, N,
                                                  static_cast<const bf16*>(colscale), dst, rows_each, dgpart, c.st)
                      : launch_wgrad_reduce<float>(wpart, g.ksplit, 1LL * M * N, M, N,
                                                   static_cast<const float*>(colscale), dst, rows_each, dgpart, c.st);
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "wgrad reduce: %s", cudaGetErrorString(e));
  return LR_OK;
}

// One plain weight gradient (no column scale, no dg, one destination) of a group sharing K.
struct WgradJob {
  int M, N;
  Operand A, B;
  float* dst;
};

// Weight gradients that share K (tokens) and need no pass after the GEMM: one grouped launch whose
// tiles fill the SM pairs together, without split-K (fp32 results stored directly), when the cost
// model prefers it to planning each GEMM alone; else each on its own.
static lr_status wgrad_group(const Ctx& c, int K, int n, const WgradJob* jobs, float* wpart) {
  bool grouped = c.dt == LR_BF16 && n >= 2 && n <= kMaxBatch;
  if (grouped) {
    const long long slots = std::max(1, c.sms / 2);
    long long tiles = 0;
    double alone = 0.0;
    for (int i = 0; i < n; ++i) {
      tiles += 1LL * ((jobs[i].M + 255) / 256) * ((jobs[i].N + 255) / 256);
      alone += wgrad_plan(c, jobs[i].M, jobs[i].N, K, false).t;
    }
    grouped = ((tiles + slots - 1) / slots) * wgrad_tile_time(256, K, 1) < alone;
  }
  if (!grouped) {
    for (int i = 0; i < n; ++i) {
      WgradDst dst = {{jobs[i].dst, nullptr, nullptr}, {nullptr, nullptr, nullptr}};
      LR_TRY(wgrad(c, jobs[i].M, jobs[i].N, K, jobs[i].A, jobs[i].B, dst, jobs[i].M, nullptr, nullptr, wpart));
    }
    return LR_OK;
  }
  GemmCall g = new_call(jobs[0].M, jobs[0].N, K);
  g.a_mn = g.b_mn = true;
  g.bn = 256;
  g.batches = n;
  g.grouped = true;
  for (int i = 0; i < n; ++i) {
    g.A[i] = jobs[i].A;
    g.B[i] = jobs[i].B;
    g.gM[i] = jobs[i].M;
    g.gN[i] = jobs[i].N;
    g.gldo[i] = jobs[i].N;
    g.ep.out0[i] = jobs[i].dst;
  }
  g.ep.ldo0 = jobs[0].N;
  return gemm(c, EPI_F32, g);
}

// ------------------------------------------------------------ small ops
static lr_status fold(const Ctx& c, void* out, StackSrc src, int nsrc, int rows_each, int cols, const void* g) {
  LaunchScope scope("fold", c.st, 0, 2.0 * c.es * nsrc * rows_each * cols);
  cudaError_t e = (c.dt == LR_BF16) ? launch_fold<bf16>(static_cast<bf16*>(out), src, nsrc, rows_each, cols,
                                                        static_cast<const bf16*>(g), c.st)
                                    : launch_fold<float>(static_cast<float*>(out), src, nsrc, rows_each, cols,
                                                         static_cast<const float*>(g), c.st);
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "fold: %s", cudaGetErrorString(e));
  return LR_OK;
}

static lr_status rstd(const Ctx& c, const void* x, int T, int d, float eps, float* s) {
  LaunchScope scope("rstd", c.st, 0, static_cast<double>(c.es) * T * d + 4.0 * T);
  cudaError_t e = (c.dt == LR_BF16) ? launch_rstd<bf16>(static_cast<const bf16*>(x), T, d, eps, s, c.st)
                                    : launch_rstd<float>(static_cast<const float*>(x), T, d, eps, s, c.st);
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "rstd: %s", cudaGetErrorString(e));
  return LR_OK;
}

static lr_status silu_slabs(const Ctx& c, SiluSlab a, SiluSlab b, int T) {
  LaunchScope scope("silu", c.st, 0, 2.0 * c.es * T * (a.n + b.n));
  cudaError_t e = (c.dt == LR_BF16) ? launch_silu<bf16>(a, b, T, c.st) : launch_silu<float>(a, b, T, c.st);
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "silu: %s", cudaGetErrorString(e));
  return LR_OK;
}

static lr_status dg_finalize(const Ctx& c, const float* dgpart, int nparts, int N, float* dg) {
  LaunchScope scope("dg_finalize", c.st, 0, 4.0 * nparts * N + 4.0 * N);
  cudaError_t e = launch_dg_finalize(dgpart, nparts, N, dg, c.st);
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "dg: %s", cudaGetErrorString(e));
  return LR_OK;
}

// ---------------------------------------------------------------- arena
// Bump allocator over a caller buffer; with base == nullptr it only measures.
struct Arena {
  char* base;
  size_t off;
  explicit Arena(void* b) : base(static_cast<char*>(b)), off(0) {}
  void* take(size_t bytes) {
    off = (off + 255) & ~size_t(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
  size_t size() const { return (off + 255) & ~size_t(255); }
};

static size_t esize(lr_dtype dt) { return dt == LR_BF16 ? 2 : 4; }
static int chunk_width(lr_dtype dt) { return dt == LR_BF16 ? kChunkUmma : kChunkSimt; }
static int cdiv(int a, int b) { return (a + b - 1) / b; }

// ============================================================ MLP block
struct MlpSaved {
  void *u_gu, *u_d;
  float* s;
  void *z_gu, *z_d, *a, *b, *h;  // LR_SAVE_FULL only
};

static size_t mlp_saved_layout(lr_dtype dt, lr_mode mode, int T, int d, int f, int r, void* base, MlpSaved* S) {
  (void)d;
  const size_t es = esize(dt);
  Arena ar(base);
  MlpSaved tmp;
  if (!S) S = &tmp;
  memset(S, 0, sizeof(*S));
  S->u_gu = ar.take(es * T * 2 * r);
  S->u_d = ar.take(es * T * r);
  S->s = static_cast<float*>(ar.take(sizeof(float) * T));
  if (mode == LR_SAVE_FULL) {
    S->z_gu = ar.take(es * T * 2 * r);
    S->z_d = ar.take(es * T * r);
    S->a = ar.take(es * T * f);
    S->b = ar.take(es * T * f);
    S->h = ar.take(es * T * f);
  }
  return ar.size();
}

struct MlpFwdWs {
  void *Af, *z_gu, *z_d, *h;
};

static size_t mlp_fwd_ws_layout(lr_dtype dt, lr_mode mode, int T, int d, int f, int r, void* base, MlpFwdWs* W) {
  const size_t es = esize(dt);
  Arena ar(base);
  MlpFwdWs tmp;
  if (!W) W = &tmp;
  memset(W, 0, sizeof(*W));
  W->Af = ar.take(es * 2 * r * d);
  if (mode == LR_SAVE_CKPT) {
    W->z_gu = ar.take(es * T * 2 * r);
    W->z_d = ar.take(es * T * r);
    W->h = ar.take(es * T * f);
  }
  return ar.size();
}

struct MlpBwdWs {
  void *Af, *z_gu, *z_d, *a, *b, *h;  // z/a/b/h: LR_SAVE_CKPT recompute only (a, b: fp32 engine)
  void *du_d, *da, *db, *du_s;
  float *rowpart, *wpart, *dgpart;
};

static size_t mlp_bwd_ws_layout(lr_dtype dt, lr_mode mode, int T, int d, int f, int r, void* base, MlpBwdWs* W) {
  const size_t es = esize(dt);
  Arena ar(base);
  MlpBwdWs tmp;
  if (!W) W = &tmp;
  memset(W, 0, sizeof(*W));
  W->Af = ar.take(es * 2 * r * d);
  if (mode == LR_SAVE_CKPT) {
    W->z_gu = ar.take(es * T * 2 * r);
    W->z_d = ar.take(es * T * r);
    if (dt != LR_BF16) {  // bf16: a and b live only in TMEM (the fused re-forward + SwiGLU backward)
      W->a = ar.take(es * T * f);
      W->b = ar.take(es * T * f);
    }
    W->h = ar.take(es * T * f);
  }
  W->du_d = ar.take(es * T * r);
  W->da = ar.take(es * T * f);
  W->db = ar.take(es * T * f);
  W->du_s = ar.take(es * T * 2 * r);
  W->rowpart = static_cast<float*>(ar.take(sizeof(float) * 2 * cdiv(r, chunk_width(dt)) * T));
  size_t wp = std::max({wgrad_part_bytes(dt, d, r, T), wgrad_part_bytes(dt, r, f, T), wgrad_part_bytes(dt, f, r, T),
                        wgrad_part_bytes(dt, 2 * r, d, T)});
  W->wpart = static_cast<float*>(ar.take(wp));
  W->dgpart = static_cast<float*>(ar.take(sizeof(float) * cdiv(2 * r, kReduceRows) * d));
  return ar.size();
}

// The SwiGLU dual GEMM: a = z_g B_gate^T, b = z_u B_up^T, h = SiLU(a) * b.
static lr_status swiglu_gemm(const Ctx& c, int T, int f, int r, const void* z_gu, const void* Bg, const void* Bu,
                             void* h, void* a, void* b) {
  // h alone (the checkpointed forward) runs the kernel built for one output: one more operand stage.
  const EpiKind kind = (a || b || c.dt != LR_BF16) ? EPI_SWIGLU : EPI_SWIGLU_H;
  GemmCall g = new_call(T, f, r);
  g.nacc = 2;
  g.A[0] = {z_gu, 2LL * r};
  g.A[1] = {off(z_gu, c.es * r), 2LL * r};
  g.B[0] = {Bg, r};
  g.B[1] = {Bu, r};
  g.ep.out0[0] = h;
  g.ep.out1[0] = a;
  g.ep.out2[0] = b;
  g.ep.ldo0 = g.ep.ldo1 = g.ep.ldo2 = f;
  return gemm(c, kind, g);
}

static lr_status mlp_fwd_impl(const Ctx& c, lr_mode mode, int T, int d, int f, int r, float eps, const void* x,
                              const void* g, lr_pair gate, lr_pair up, lr_pair down, void* out, void* saved,
                              void* ws) {
  MlpSaved S;
  MlpFwdWs W;
  mlp_saved_layout(c.dt, mode, T, d, f, r, saved, &S);
  mlp_fwd_ws_layout(c.dt, mode, T, d, f, r, ws, &W);
  void* z_gu = mode == LR_SAVE_FULL ? S.z_gu : W.z_gu;
  void* z_d = mode == LR_SAVE_FULL ? S.z_d : W.z_d;
  void* h = mode == LR_SAVE_FULL ? S.h : W.h;

  // Online-RMSNorm (technical summary §2.2): gain folded into the stacked [A_gate; A_up] ...
  StackSrc src = {{gate.A, up.A, nullptr}};
  LR_TRY(fold(c, W.Af, src, 2, r, d, g));
  // ... the row sum of squares of x accumulated in the same pass as the grouped gate/up GEMM
  // (tcgen05 path: statistics warps read the x tiles of the GEMM's own shared-memory ring;
  // fp32 path: a separate row pass), and 1/rms applied as a row scale in its epilogue, SiLU fused.
  if (c.dt != LR_BF16) LR_TRY(rstd(c, x, T, d, eps, S.s));
  {
    GemmCall k = new_call(T, 2 * r, d);
    k.A[0] = {x, d};
    k.B[0] = {W.Af, d};
    k.ep.out0[0] = S.u_gu;
    k.ep.out1[0] = z_gu;
    k.ep.ldo0 = k.ep.ldo1 = 2 * r;
    k.ep.rowscale = S.s;
    k.ep.rowscale_out = S.s;
    k.ep.coef = 1.f / static_cast<float>(d);
    k.ep.eps = eps;
    LR_TRY(gemm(c, EPI_NORM_SILU, k));
  }
  // B_gate / B_up with the SwiGLU product fused.
  LR_TRY(swiglu_gemm(c, T, f, r, z_gu, gate.B, up.B, h, mode == LR_SAVE_FULL ? S.a : nullptr,
                     mode == LR_SAVE_FULL ? S.b : nullptr));
  // A_down with SiLU fused (reads h right after the SwiGLU GEMM wrote it: start on the last tiles).
  {
    GemmCall k = new_call(T, r, f);
    k.reverse = true;
    k.A[0] = {h, f};
    k.B[0] = {down.A, f};
    k.ep.out0[0] = S.u_d;
    k.ep.out1[0] = z_d;
    k.ep.ldo0 = k.ep.ldo1 = r;
    LR_TRY(gemm(c, EPI_SILU, k));
  }
  // B_down with the residual fused.
  {
    GemmCall k = new_call(T, d, r);
    k.A[0] = {z_d, r};
    k.B[0] = {down.B, r};
    k.ep.out0[0] = out;
    k.ep.ldo0 = d;
    k.ep.aux0[0] = x;
    k.ep.lda0 = d;
    LR_TRY(gemm(c, EPI_RESID, k));
  }
  return LR_OK;
}

static lr_status mlp_bwd_impl(const Ctx& c, lr_mode mode, int T, int d, int f, int r, float eps, const void* x,
                              const void* g, lr_pair gate, lr_pair up, lr_pair down, const void* saved,
                              const void* G, void* dx, float* dg, lr_pair_grad dgate, lr_pair_grad dup,
                              lr_pair_grad ddown, void* ws) {
  (void)eps;
  MlpSaved S;
  MlpBwdWs W;
  mlp_saved_layout(c.dt, mode, T, d, f, r, const_cast<void*>(saved), &S);
  mlp_bwd_ws_layout(c.dt, mode, T, d, f, r, ws, &W);
  const int ch = chunk_width(c.dt);

  StackSrc src = {{gate.A, up.A, nullptr}};
  void *z_gu, *z_d, *a, *b, *h;
  z_gu = W.z_gu;
  z_d = W.z_d;
  // Checkpointed bf16: the gain fold and the re-forward of z_gate;up from the saved u run on a second
  // stream beside du_down's GEMM, which leaves SM pairs free (it fills them in fewer waves than it has
  // pairs); joined before the re-forward GEMM.  z_down comes from du_down's own epilogue, which reads
  // u_down anyway.
  const bool side = mode == LR_SAVE_CKPT && c.dt == LR_BF16 && !c.act;
  SideStream* ss = nullptr;
  if (side) {
    LR_TRY(side_stream(&ss));
    Ctx cs = c;
    cs.st = ss->st;
    if (cudaEventRecord(ss->fork, c.st) != cudaSuccess || cudaStreamWaitEvent(ss->st, ss->fork, 0) != cudaSuccess)
      return fail(LR_ERR_CUDA, "fork: %s", cudaGetErrorString(cudaGetLastError()));
    LR_TRY(fold(cs, W.Af, src, 2, r, d, g));
    LR_TRY(silu_slabs(cs, {S.u_gu, 2LL * r, z_gu, 2LL * r, 2 * r}, {S.u_d, r, z_d, r, 0}, T));
    if (cudaEventRecord(ss->join, ss->st) != cudaSuccess)
      return fail(LR_ERR_CUDA, "join: %s", cudaGetErrorString(cudaGetLastError()));
  } else {
    LR_TRY(fold(c, W.Af, src, 2, r, d, g));
  }

  // du_down = (G B_down) * SiLU'(u_down): needs only dout and the saved u_down, so it runs first
  // and the SwiGLU backward can follow the re-forward while a, b are still in L2
  {
    GemmCall k = new_call(T, r, d);
    k.b_mn = true;
    k.A[0] = {G, d};
    k.B[0] = {down.B, r};
    k.ep.aux0[0] = S.u_d;
    k.ep.lda0 = r;
    k.ep.out0[0] = W.du_d;
    k.ep.ldo0 = r;
    if (side) {  // z_down = SiLU(u_down) from the same operand tiles
      k.ep.out1[0] = z_d;
      k.ep.ldo1 = r;
    }
    LR_TRY(gemm(c, side ? EPI_DSILU_Z : EPI_DSILU, k));
  }
  if (mode == LR_SAVE_CKPT) {
    // Low-rank activation checkpointing (technical summary §2.2): re-forward inside the block
    // from the saved [T, r] pre-activations; no other state is needed.
    a = W.a;
    b = W.b;
    h = W.h;
    if (c.act) {  // sigma = identity: z is u itself
      z_gu = S.u_gu;
      z_d = S.u_d;
    } else if (side) {
      if (cudaStreamWaitEvent(c.st, ss->join, 0) != cudaSuccess)
        return fail(LR_ERR_CUDA, "join: %s", cudaGetErrorString(cudaGetLastError()));
    } else {
      LR_TRY(silu_slabs(c, {S.u_gu, 2LL * r, z_gu, 2LL * r, 2 * r}, {S.u_d, r, z_d, r, r}, T));
    }
    if (c.dt == LR_BF16) {
      // One launch recomputes a = z_g B_gate^T and b = z_u B_up^T and computes dh = du_down A_down
      // for each tile in three TMEM accumulators; its epilogue writes h (for dA_down) and the
      // SwiGLU backward's da, db.  a and b never reach memory.  A_down [r, f] is read in its stored
      // orientation (MN-major), B_gate and B_up K-major.
      GemmCall k = new_call(T, f, r);
      k.nacc = 3;
      k.A[0] = {z_gu, 2LL * r};
      k.A[1] = {off(z_gu, c.es * r), 2LL * r};
      k.A[2] = {W.du_d, r};
      k.B[0] = {gate.B, r};
      k.B[1] = {up.B, r};
      k.B[2] = {down.A, f};
      k.ep.out0[0] = h;
      k.ep.out1[0] = W.da;
      k.ep.out2[0] = W.db;
      k.ep.ldo0 = k.ep.ldo1 = k.ep.ldo2 = f;
      LR_TRY(gemm(c, EPI_SWIGLU_REBWD, k));
    } else {
      LR_TRY(swiglu_gemm(c, T, f, r, z_gu, gate.B, up.B, h, a, b));
    }
  } else {
    z_gu = S.z_gu;
    z_d = S.z_d;
    a = S.a;
    b = S.b;
    h = S.h;
  }

  // dh = du_down A_down; SwiGLU backward fused: da = dh b SiLU'(a), db = dh SiLU(a)
  if (!(mode == LR_SAVE_CKPT && c.dt == LR_BF16)) {
    GemmCall k = new_call(T, f, r);
    k.reverse = mode == LR_SAVE_CKPT;  // a, b were just written by the re-forward: start on the last tiles
    k.b_mn = true;
    k.A[0] = {W.du_d, r};
    k.B[0] = {down.A, f};
    k.ep.aux0[0] = a;
    k.ep.aux1[0] = b;
    k.ep.lda0 = k.ep.lda1 = f;
    k.ep.out0[0] = W.da;
    k.ep.out1[0] = W.db;
    k.ep.ldo0 = k.ep.ldo1 = f;
    LR_TRY(gemm(c, EPI_SWIGLU_BWD, k));
  }
  // dB_gate = da^T z_gate, dB_up = db^T z_up, dA_down = du_down^T h, dB_down = G^T z_down: four
  // weight gradients over the same T tokens, one grouped launch (da, db first: just written)
  {
    const WgradJob jobs[4] = {{f, r, {W.da, f}, {z_gu, 2LL * r}, static_cast<float*>(dgate.dB)},
                              {f, r, {W.db, f}, {off(z_gu, c.es * r), 2LL * r}, static_cast<float*>(dup.dB)},
                              {r, f, {W.du_d, r}, {h, f}, static_cast<float*>(ddown.dA)},
                              {d, r, {G, d}, {z_d, r}, static_cast<float*>(ddown.dB)}};
    LR_TRY(wgrad_group(c, T, 4, jobs, W.wpart));
  }
  // du_{gate,up} = (d{a,b} B) * SiLU'(u), stored pre-scaled by s; rho partials = sum du * u.
  {
    GemmCall k = new_call(T, r, f);
    k.reverse = true;  // da, db were written tile by tile by the SwiGLU backward (after dB_gate, dB_up)
    k.b_mn = true;
    k.batches = 2;
    k.A[0] = {W.da, f};
    k.A[1] = {W.db, f};
    k.B[0] = {gate.B, r};
    k.B[1] = {up.B, r};
    k.ep.aux0[0] = S.u_gu;
    k.ep.aux0[1] = off(S.u_gu, c.es * r);
    k.ep.lda0 = 2 * r;
    k.ep.out0[0] = W.du_s;
    k.ep.out0[1] = off(W.du_s, c.es * r);
    k.ep.ldo0 = 2 * r;
    k.ep.rowscale = S.s;
    k.ep.rowpart = W.rowpart;
    k.ep.rowpart_chunks = cdiv(r, ch);
    LR_TRY(gemm(c, EPI_DSILU_NORM, k));
  }
  // dA'_{gate;up} = (s du)^T x; dA = dA' * g; dg_j = sum_i dA'_ij A_ij.  dA' and dx below are independent:
  // on the checkpointed bf16 path, when dA' (one 256 x 256 tile per SM pair, K = T, no split) needs at most
  // half of the pairs, it runs with its pass and dg's final sum on the second stream on that many pairs,
  // and dx on the others (the split-K alternative leaves pairs idle and adds the partials' reduction).
  const int all_pairs = std::max(1, c.sms / 2);
  const int wg_pairs = cdiv(2 * r, 256) * cdiv(d, 256);
  const bool beside = side && T >= 8192 && 2 * wg_pairs <= all_pairs;
  {
    WgradDst dst = {{dgate.dA, dup.dA, nullptr}, {gate.A, up.A, nullptr}};
    if (beside) {
      Ctx cs = c;
      cs.st = ss->st;
      if (cudaEventRecord(ss->fork, c.st) != cudaSuccess || cudaStreamWaitEvent(ss->st, ss->fork, 0) != cudaSuccess)
        return fail(LR_ERR_CUDA, "fork: %s", cudaGetErrorString(cudaGetLastError()));
      LR_TRY(wgrad(cs, 2 * r, d, T, {W.du_s, 2LL * r}, {x, d}, dst, r, g, W.dgpart, W.wpart, wg_pairs));
      LR_TRY(dg_finalize(cs, W.dgpart, cdiv(2 * r, kReduceRows), d, dg));
      if (cudaEventRecord(ss->join, ss->st) != cudaSuccess)
        return fail(LR_ERR_CUDA, "join: %s", cudaGetErrorString(cudaGetLastError()));
    } else {
      LR_TRY(wgrad(c, 2 * r, d, T, {W.du_s, 2LL * r}, {x, d}, dst, r, g, W.dgpart, W.wpart));
      LR_TRY(dg_finalize(c, W.dgpart, cdiv(2 * r, kReduceRows), d, dg));
    }
  }
  // dx = G + (s du) A' - (s^2 / d) rho x  (one GEMM with K = 2r: gate and up sum inside the MMA)
  {
    GemmCall k = new_call(T, d, 2 * r);
    k.b_mn = true;
    k.A[0] = {W.du_s, 2LL * r};
    k.B[0] = {W.Af, d};
    k.ep.aux0[0] = G;
    k.ep.aux1[0] = x;
    k.ep.lda0 = k.ep.lda1 = d;
    k.ep.rowscale = S.s;
    k.ep.rowpart_in = W.rowpart;
    k.ep.rowpart_in_chunks = 2 * cdiv(r, ch);
    k.ep.coef = 1.f / static_cast<float>(d);
    k.ep.out0[0] = dx;
    k.ep.ldo0 = d;
    if (beside) k.max_pairs = all_pairs - wg_pairs;
    LR_TRY(gemm(c, EPI_DX_NORM, k));
  }
  if (beside && cudaStreamWaitEvent(c.st, ss->join, 0) != cudaSuccess)
    return fail(LR_ERR_CUDA, "join: %s", cudaGetErrorString(cudaGetLastError()));
  return LR_OK;
}

// ====================================================== dense MLP block
// The full-rank SwiGLU MLP block the low-rank block replaces, on the same kernels, for a
// same-device comparison: n = RMSNorm(x), a = W_gate n, b = W_up n, h = SiLU(a) b,
// out = x + W_down h.  RMSNorm is folded the same way (W' = W * g, 1/rms as a row scale;
// the statistics come from a row pass), gate and up are one dual-accumulator GEMM with the
// SwiGLU product fused, and the backward mirrors the low-rank one with the pairs replaced by
// single matrices: dh = dout W_down with the SwiGLU backward, 1/rms scaling and rho partials
// fused; dW = (s du)^T x with the gain unfold and dg; dx in one GEMM with K = 2f.
struct DenseSaved {
  void *a, *b, *h;
  float* s;
};

static size_t dense_saved_layout(lr_dtype dt, int T, int f, void* base, DenseSaved* S) {
  const size_t es = esize(dt);
  Arena ar(base);
  DenseSaved tmp;
  if (!S) S = &tmp;
  S->a = ar.take(es * T * f);
  S->b = ar.take(es * T * f);
  S->h = ar.take(es * T * f);
  S->s = static_cast<float*>(ar.take(sizeof(float) * T));
  return ar.size();
}

struct DenseWs {
  void *Wf, *du_s;
  float *rowpart, *wpart, *dgpart;
};

static size_t dense_ws_layout(lr_dtype dt, bool bwd, int T, int d, int f, void* base, DenseWs* W) {
  const size_t es = esize(dt);
  Arena ar(base);
  DenseWs tmp;
  if (!W) W = &tmp;
  memset(W, 0, sizeof(*W));
  W->Wf = ar.take(es * 2 * f * d);
  if (bwd) {
    W->du_s = ar.take(es * T * 2 * f);
    W->rowpart = static_cast<float*>(ar.take(sizeof(float) * cdiv(f, chunk_width(dt)) * T));
    W->wpart = static_cast<float*>(
        ar.take(std::max(wgrad_part_bytes(dt, d, f, T), wgrad_part_bytes(dt, 2 * f, d, T))));
    W->dgpart = static_cast<float*>(ar.take(sizeof(float) * cdiv(2 * f, kReduceRows) * d));
  }
  return ar.size();
}

static lr_status dense_fwd_impl(const Ctx& c, int T, int d, int f, float eps, const void* x, const void* g,
                                const void* Wg, const void* Wu, const void* Wd, void* out, void* saved, void* ws) {
  DenseSaved S;
  DenseWs W;
  dense_saved_layout(c.dt, T, f, saved, &S);
  dense_ws_layout(c.dt, false, T, d, f, ws, &W);
  StackSrc src = {{Wg, Wu, nullptr}};
  LR_TRY(fold(c, W.Wf, src, 2, f, d, g));
  LR_TRY(rstd(c, x, T, d, eps, S.s));
  {
    GemmCall k = new_call(T, f, d);
    k.nacc = 2;
    k.A[0] = {x, d};
    k.A[1] = {x, d};
    k.B[0] = {W.Wf, d};
    k.B[1] = {off(W.Wf, c.es * f * d), d};
    k.ep.out0[0] = S.h;
    k.ep.out1[0] = S.a;
    k.ep.out2[0] = S.b;
    k.ep.ldo0 = k.ep.ldo1 = k.ep.ldo2 = f;
    k.ep.rowscale = S.s;
    LR_TRY(gemm(c, EPI_NORM_SWIGLU, k));
  }
  {
    GemmCall k = new_call(T, d, f);
    k.A[0] = {S.h, f};
    k.B[0] = {Wd, f};
    k.ep.out0[0] = out;
    k.ep.ldo0 = d;
    k.ep.aux0[0] = x;
    k.ep.lda0 = d;
    LR_TRY(gemm(c, EPI_RESID, k));
  }
  return LR_OK;
}

static lr_status dense_bwd_impl(const Ctx& c, int T, int d, int f, const void* x, const void* g, const void* Wg,
                                const void* Wu, const void* Wd, const void* saved, const void* G, void* dx, float* dg,
                                float* dWg, float* dWu, float* dWd, void* ws) {
  DenseSaved S;
  DenseWs W;
  dense_saved_layout(c.dt, T, f, const_cast<void*>(saved), &S);
  dense_ws_layout(c.dt, true, T, d, f, ws, &W);
  const int ch = chunk_width(c.dt);
  StackSrc src = {{Wg, Wu, nullptr}};
  LR_TRY(fold(c, W.Wf, src, 2, f, d, g));
  // dh = dout W_down; da = dh b SiLU'(a), db = dh SiLU(a); du_s = s [da | db]; rho partials
  {
    GemmCall k = new_call(T, f, d);
    k.b_mn = true;
    k.A[0] = {G, d};
    k.B[0] = {Wd, f};
    k.ep.aux0[0] = S.a;
    k.ep.aux1[0] = S.b;
    k.ep.lda0 = k.ep.lda1 = f;
    k.ep.out0[0] = W.du_s;
    k.ep.out1[0] = off(W.du_s, c.es * f);
    k.ep.ldo0 = k.ep.ldo1 = 2LL * f;
    k.ep.rowscale = S.s;
    k.ep.rowpart = W.rowpart;
    k.ep.rowpart_chunks = cdiv(f, ch);
    LR_TRY(gemm(c, EPI_SWIGLU_BWD_NORM, k));
  }
  // dW_down = dout^T h
  {
    WgradDst dst = {{dWd, nullptr, nullptr}, {nullptr, nullptr, nullptr}};
    LR_TRY(wgrad(c, d, f, T, {G, d}, {S.h, f}, dst, d, nullptr, nullptr, W.wpart));
  }
  // dW'_{gate;up} = (s du)^T x; dW = dW' * g; dg_j = sum_i dW'_ij W_ij
  {
    WgradDst dst = {{dWg, dWu, nullptr}, {Wg, Wu, nullptr}};
    LR_TRY(wgrad(c, 2 * f, d, T, {W.du_s, 2LL * f}, {x, d}, dst, f, g, W.dgpart, W.wpart));
    LR_TRY(dg_finalize(c, W.dgpart, cdiv(2 * f, kReduceRows), d, dg));
  }
  // dx = dout + (s du) W' - (s^2 / d) rho x
  {
    GemmCall k = new_call(T, d, 2 * f);
    k.b_mn = true;
    k.A[0] = {W.du_s, 2LL * f};
    k.B[0] = {W.Wf, d};
    k.ep.aux0[0] = G;
    k.ep.aux1[0] = x;
    k.ep.lda0 = k.ep.lda1 = d;
    k.ep.rowscale = S.s;
    k.ep.rowpart_in = W.rowpart;
    k.ep.rowpart_in_chunks = cdiv(f, ch);
    k.ep.coef = 1.f / static_cast<float>(d);
    k.ep.out0[0] = dx;
    k.ep.ldo0 = d;
    LR_TRY(gemm(c, EPI_DX_NORM, k));
  }
  return LR_OK;
}

// ============================================== BTP row-parallel normed group
// Bottleneck-aware tensor parallelism (technical summary §2.1) keeps activations sharded
// along d and makes a normed group of A's row-parallel: each rank computes fp32 partial
// sums over its d-shard, and the only collective is one all-reduce at the bottleneck
// width.  Online-RMSNorm (§2.2) puts the statistics on that same all-reduce: the payload
// is [acc (T x group*r) | ss (T)], the shard's sums of squares of x appended.
static size_t btp_ws_layout(lr_dtype dt, int d_shard, int r, int group, void* base, void** Af) {
  Arena ar(base);
  void* a = ar.take(esize(dt) * group * r * d_shard);
  if (Af) *Af = a;
  return ar.size();
}

static lr_status btp_partial_impl(const Ctx& c, int T, int d_shard, int r, int group, const lr_pair* pairs,
                                  const void* g, const void* x, float* payload, void* ws) {
  void* Af = nullptr;
  btp_ws_layout(c.dt, d_shard, r, group, ws, &Af);
  StackSrc src = {{nullptr, nullptr, nullptr}};
  for (int i = 0; i < group; ++i) src.src[i] = pairs[i].A;
  LR_TRY(fold(c, Af, src, group, r, d_shard, g));
  const int R = group * r;
  float* ss = payload + static_cast<size_t>(T) * R;
  if (c.dt != LR_BF16) {  // fp32 path: the sums of squares from a row pass
    LaunchScope scope("rowss", c.st, 0, static_cast<double>(c.es) * T * d_shard + 4.0 * T);
    cudaError_t e = launch_rstd<float>(static_cast<const float*>(x), T, d_shard, 0.f, ss, c.st, true);
    if (e != cudaSuccess) return fail(LR_ERR_CUDA, "row sums of squares: %s", cudaGetErrorString(e));
  }
  GemmCall k = new_call(T, R, d_shard);
  k.A[0] = {x, d_shard};
  k.B[0] = {Af, d_shard};
  k.ep.out0[0] = payload;
  k.ep.ldo0 = R;
  k.ep.split_stride = static_cast<long long>(T) * R;
  k.ep.rowscale_out = c.dt == LR_BF16 ? ss : nullptr;  // tcgen05: the statistics warps write ss
  k.ep.coef = 1.f;
  return gemm(c, EPI_F32_SS, k);
}

static lr_status btp_finish_impl(const Ctx& c, int T, int d, int R, const float* payload, float eps, void* u, void* z,
                                 float* s) {
  const float* ss = payload + static_cast<size_t>(T) * R;
  LaunchScope scope("norm_finish", c.st, 0, 4.0 * T * R + 4.0 * T + 2.0 * c.es * T * R + 4.0 * T);
  const float coef = 1.f / static_cast<float>(d);
  cudaError_t e = (c.dt == LR_BF16)
                      ? launch_norm_finish<bf16>(payload, ss, T, R, coef, eps, c.act, static_cast<bf16*>(u),
                                                 static_cast<bf16*>(z), s, c.st)
                      : launch_norm_finish<float>(payload, ss, T, R, coef, eps, c.act, static_cast<float*>(u),
                                                  static_cast<float*>(z), s, c.st);
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "norm finish: %s", cudaGetErrorString(e));
  return LR_OK;
}

// ======================================================= projection group
struct ProjSaved {
  void *u, *z;
  float* s;
};

static size_t proj_saved_layout(lr_dtype dt, int T, int r, int group, int norm, void* base, ProjSaved* S) {
  const size_t es = esize(dt);
  Arena ar(base);
  ProjSaved tmp;
  if (!S) S = &tmp;
  S->u = ar.take(es * T * group * r);
  S->z = ar.take(es * T * group * r);
  S->s = norm ? static_cast<float*>(ar.take(sizeof(float) * T)) : nullptr;
  return ar.size();
}

struct ProjWs {
  void *Af, *du;
  float *rowpart, *wpart, *dgpart;
};

static size_t proj_ws_layout(lr_dtype dt, bool bwd, int T, int d_in, int d_out, int r, int group, int norm,
                             void* base, ProjWs* W) {
  const size_t es = esize(dt);
  Arena ar(base);
  ProjWs tmp;
  if (!W) W = &tmp;
  memset(W, 0, sizeof(*W));
  W->Af = ar.take(es * group * r * d_in);
  if (bwd) {
    W->du = ar.take(es * T * group * r);
    if (norm) W->rowpart = static_cast<float*>(ar.take(sizeof(float) * group * cdiv(r, chunk_width(dt)) * T));
    W->wpart = static_cast<float*>(
        ar.take(std::max(wgrad_part_bytes(dt, d_out, r, T), wgrad_part_bytes(dt, group * r, d_in, T))));
    if (norm) W->dgpart = static_cast<float*>(ar.take(sizeof(float) * cdiv(group * r, kReduceRows) * d_in));
  }
  return ar.size();
}

// resid (group 1, d_out == d_in, or null): outs[0] = resid + LR(x), the residual fused into the B GEMM.
static lr_status proj_fwd_impl(const Ctx& c, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                               const void* g, float eps, const void* x, void* const* outs, void* saved, void* ws,
                               const void* resid = nullptr) {
  const int norm = g != nullptr;
  ProjSaved S;
  ProjWs W;
  proj_saved_layout(c.dt, T, r, group, norm, saved, &S);
  proj_ws_layout(c.dt, false, T, d_in, d_out, r, group, norm, ws, &W);
  StackSrc src = {{nullptr, nullptr, nullptr}};
  for (int i = 0; i < group; ++i) src.src[i] = pairs[i].A;
  if (!norm) {
    // Without the norm there is no gain to fold: the A's are read where they are, one batch per pair
    // writing its columns of u and z (the same tiles as one GEMM over the stacked A's).
    GemmCall k = new_call(T, r, d_in);
    k.batches = group;
    for (int i = 0; i < group; ++i) {
      k.A[i] = {x, d_in};
      k.B[i] = {pairs[i].A, d_in};
      k.ep.out0[i] = off(S.u, c.es * i * r);
      k.ep.out1[i] = off(S.z, c.es * i * r);
    }
    k.ep.ldo0 = k.ep.ldo1 = 1LL * group * r;
    LR_TRY(gemm(c, EPI_SILU, k));
  } else {
    LR_TRY(fold(c, W.Af, src, group, r, d_in, g));
    if (c.dt != LR_BF16) LR_TRY(rstd(c, x, T, d_in, eps, S.s));
    GemmCall k = new_call(T, group * r, d_in);
    k.A[0] = {x, d_in};
    k.B[0] = {W.Af, d_in};
    k.ep.out0[0] = S.u;
    k.ep.out1[0] = S.z;
    k.ep.ldo0 = k.ep.ldo1 = 1LL * group * r;
    k.ep.rowscale = S.s;
    k.ep.rowscale_out = S.s;
    k.ep.coef = 1.f / static_cast<float>(d_in);
    k.ep.eps = eps;
    LR_TRY(gemm(c, EPI_NORM_SILU, k));
  }
  {
    // The B's have distinct inputs: one batched GEMM (technical summary §2.2).
    GemmCall k = new_call(T, d_out, r);
    k.batches = group;
    for (int i = 0; i < group; ++i) {
      k.A[i] = {off(S.z, c.es * i * r), 1LL * group * r};
      k.B[i] = {pairs[i].B, r};
      k.ep.out0[i] = outs[i];
    }
    k.ep.ldo0 = d_out;
    if (resid) {
      k.ep.aux0[0] = resid;
      k.ep.lda0 = d_out;
    }
    LR_TRY(gemm(c, resid ? EPI_RESID : EPI_STORE, k));
  }
  return LR_OK;
}

// dres (normed groups, or null): the gradient reaching x through a residual, added into dx by the
// dx GEMM's epilogue.
static lr_status proj_bwd_impl(const Ctx& c, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                               const void* g, const void* x, const void* saved, const void* const* douts, void* dx,
                               float* dg, const lr_pair_grad* grads, void* ws, const void* dres = nullptr) {
  const int norm = g != nullptr;
  ProjSaved S;
  ProjWs W;
  proj_saved_layout(c.dt, T, r, group, norm, const_cast<void*>(saved), &S);
  proj_ws_layout(c.dt, true, T, d_in, d_out, r, group, norm, ws, &W);
  const int ch = chunk_width(c.dt);
  const long long ldg = 1LL * group * r;
  StackSrc src = {{nullptr, nullptr, nullptr}};
  for (int i = 0; i < group; ++i) src.src[i] = pairs[i].A;
  // dx reads the stacked (and, with the norm, gain-folded) A's; a single pair without the norm is read in place.
  const bool stack = norm || group > 1;
  if (stack) LR_TRY(fold(c, W.Af, src, group, r, d_in, g));
  for (int i = 0; i < group; ++i) {
    WgradDst dst = {{grads[i].dB, nullptr, nullptr}, {nullptr, nullptr, nullptr}};
    LR_TRY(wgrad(c, d_out, r, T, {douts[i], d_out}, {off(S.z, c.es * i * r), ldg}, dst, d_out, nullptr, nullptr,
                 W.wpart));
  }
  {
    GemmCall k = new_call(T, r, d_out);
    k.b_mn = true;
    k.batches = group;
    for (int i = 0; i < group; ++i) {
      k.A[i] = {douts[i], d_out};
      k.B[i] = {pairs[i].B, r};
      k.ep.aux0[i] = off(S.u, c.es * i * r);
      k.ep.out0[i] = off(W.du, c.es * i * r);
    }
    k.ep.lda0 = k.ep.ldo0 = ldg;
    k.ep.rowscale = S.s;
    k.ep.rowpart = W.rowpart;
    k.ep.rowpart_chunks = cdiv(r, ch);
    LR_TRY(gemm(c, norm ? EPI_DSILU_NORM : EPI_DSILU, k));
  }
  {
    WgradDst dst = {{nullptr, nullptr, nullptr}, {nullptr, nullptr, nullptr}};
    for (int i = 0; i < group; ++i) {
      dst.dst[i] = grads[i].dA;
      dst.aw[i] = norm ? pairs[i].A : nullptr;
    }
    LR_TRY(wgrad(c, group * r, d_in, T, {W.du, ldg}, {x, d_in}, dst, r, g, norm ? W.dgpart : nullptr, W.wpart));
    if (norm) LR_TRY(dg_finalize(c, W.dgpart, cdiv(group * r, kReduceRows), d_in, dg));
  }
  {
    GemmCall k = new_call(T, d_in, group * r);
    k.b_mn = true;
    k.A[0] = {W.du, ldg};
    k.B[0] = stack ? Operand{W.Af, d_in} : Operand{pairs[0].A, d_in};
    k.ep.out0[0] = dx;
    k.ep.ldo0 = d_in;
    if (norm) {
      k.ep.aux0[0] = dres;
      k.ep.lda0 = d_in;
      k.ep.aux1[0] = x;
      k.ep.lda1 = d_in;
      k.ep.rowscale = S.s;
      k.ep.rowpart_in = W.rowpart;
      k.ep.rowpart_in_chunks = group * cdiv(r, ch);
      k.ep.coef = 1.f / static_cast<float>(d_in);
    }
    LR_TRY(gemm(c, norm ? EPI_DX_NORM : EPI_STORE, k));
  }
  return LR_OK;
}

// ============================================================ causal attention
// Each GEMM runs once over all b*H heads in row-batched mode; head n = bi*H + h is batch n.
// q, k, v, o and their gradients stay token-major ([b*s, H*dh]: head (bi, h) is rows bi*s ..
// bi*s + s - 1, columns h*dh .. h*dh + dh - 1), read and written in place through per-head row
// and column offsets.  The s x s score tensors (S, P, dS) are head-major ([b*H*s, s]: head n is
// rows n*s .. n*s + s - 1), as are lse and D.
// The head widths with kernels that keep the scores on chip (attn_flash*.cu) need only the work-item
// counter, the stored scale dS^T (bf16 [b*H*s keys, s queries]) and D; the others S, P, dS and D.
struct AttnWs {
  float *S, *D;
  bf16 *P, *dS;  // dS takes the first half of S's bytes (S is the forward's, dS the backward's)
  unsigned* sched;  // flash kernels: the counter of work items
  bf16* dST;        // flash backward: scale dS^T
};

static size_t attn_ws_layout(int b, int s, int H, int dh, void* base, AttnWs* W) {
  Arena ar(base);
  AttnWs tmp;
  if (!W) W = &tmp;
  memset(W, 0, sizeof(*W));
  const size_t R = static_cast<size_t>(b) * H * s;
  if (attn_flash_fwd_supported(dh)) {
    W->sched = static_cast<unsigned*>(ar.take(256));
    W->dST = static_cast<bf16*>(ar.take(R * s * sizeof(bf16)));
  } else {
    W->S = static_cast<float*>(ar.take(R * s * sizeof(float)));
    W->P = static_cast<bf16*>(ar.take(R * s * sizeof(bf16)));
    W->dS = reinterpret_cast<bf16*>(W->S);
  }
  W->D = static_cast<float*>(ar.take(R * sizeof(float)));
  return ar.size();
}

struct AttnDims {
  int b, s, H, dh;
};

// Places operand X of head n = bi*H + h: token-major (rows bi*s, columns h*dh of a [b*s, H*dh]
// tensor) or head-major (rows n*s of a [b*H*s, *] tensor).
static void attn_place(const AttnDims& a, bool tok, int& rb, int& rl, int& cb, long long& rows, long long& cols) {
  if (tok) {
    rb = a.s, rl = 0, cb = a.dh, rows = 1LL * a.b * a.s, cols = 1LL * a.H * a.dh;
  } else {
    rb = a.H * a.s, rl = a.s, cb = 0, rows = 1LL * a.b * a.H * a.s, cols = 0;
  }
}

// One GEMM over all heads.  tok_*: whether A, B, the output are token-major (else head-major).
static GemmCall attn_call(const AttnDims& a, int M, int N, int K, bool a_tok, bool b_tok, bool o_tok, int causal) {
  GemmCall g = new_call(M, N, K);
  g.causal = causal;
  g.batches = a.b * a.H;
  g.rowbatch = true;
  g.bh = a.H;
  attn_place(a, a_tok, g.rb_a, g.rl_a, g.cb_a, g.rows_a, g.cols_a);
  attn_place(a, b_tok, g.rb_b, g.rl_b, g.cb_b, g.rows_b, g.cols_b);
  attn_place(a, o_tok, g.rb_o, g.rl_o, g.cb_o, g.rows_o, g.cols_o);
  g.bn = N % 256 == 0 ? 256 : 128;
  return g;
}

static lr_status attn_gemm(const Ctx& c, EpiKind k, const AttnDims& a, int M, int N, int K, Operand A, bool a_mn,
                           bool a_tok, Operand B, bool b_mn, bool b_tok, void* out, long long ldo, bool o_tok,
                           int causal) {
  GemmCall g = attn_call(a, M, N, K, a_tok, b_tok, o_tok, causal);
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  g.A[0] = A;
  g.B[0] = B;
  g.ep.out0[0] = out;
  g.ep.ldo0 = ldo;
  g.ep.split_stride = ldo * g.rows_o;
  return gemm(c, k, g);
}

static lr_status attn_fwd_impl(const Ctx& c, int b, int s, int H, int dh, float scale, const void* q, const void* k,
                               const void* v, void* o, float* lse, void* ws) {
  AttnWs W;
  attn_ws_layout(b, s, H, dh, ws, &W);
  const AttnDims a{b, s, H, dh};
  const int R = b * H * s, d = H * dh;
  if (attn_flash_fwd_supported(dh)) {
    // One persistent launch over the (head, 128 queries) items: S and O in TMEM, the softmax in the
    // epilogue warps; no scores in memory (one word of the workspace counts the items taken).
    // Algorithmic FLOPs: Q K^T and P V over the causal half.
    const double causal = 2.0 * 2.0 * b * H * static_cast<double>(s) * s * dh * 0.5;
    LaunchScope scope("attn_flash_fwd", c.st, causal, 8.0 * b * s * d + 4.0 * R);
    cudaError_t e = launch_attn_flash_fwd(static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                          static_cast<const bf16*>(v), static_cast<bf16*>(o), b, s, H, dh, scale,
                                          lse, W.sched, c.err, c.st);
    if (e != cudaSuccess) return fail(LR_ERR_CUDA, "attention forward: %s", cudaGetErrorString(e));
    return LR_OK;
  }
  // S = Q K^T (fp32, head-major), both operands K-major (K = dh) in their token-major rows
  LR_TRY(attn_gemm(c, EPI_F32, a, s, s, dh, {q, d}, false, true, {k, d}, false, true, W.S, s, false, 1));
  {
    double row_bytes = 0.0;  // S read up to the diagonal, P written up to the end of the key tile
    for (int i = 0; i < s; ++i) row_bytes += 4.0 * (i + 1) + 2.0 * std::min(s, (i / 256 + 1) * 256);
    LaunchScope scope("attn_softmax", c.st, 0, row_bytes * b * H);
    cudaError_t e = launch_attn_softmax_fwd(W.S, R, s, scale, W.P, lse, c.st);
    if (e != cudaSuccess) return fail(LR_ERR_CUDA, "attention softmax: %s", cudaGetErrorString(e));
  }
  // O = P V: P K-major (K = keys), V read MN-major in its stored [keys, dh] columns; O token-major
  return attn_gemm(c, EPI_STORE, a, s, dh, s, {W.P, s}, false, false, {v, d}, true, true, o, d, true, 2);
}

static lr_status attn_bwd_impl(const Ctx& c, int b, int s, int H, int dh, float scale, const void* q, const void* k,
                               const void* v, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                               void* dv, void* ws) {
  AttnWs W;
  attn_ws_layout(b, s, H, dh, ws, &W);
  const AttnDims a{b, s, H, dh};
  const int R = b * H * s, d = H * dh;
  {
    LaunchScope scope("attn_rowdot", c.st, 0, 4.0 * R * dh + 4.0 * R);
    cudaError_t e = launch_attn_rowdot(static_cast<const bf16*>(dout), static_cast<const bf16*>(o), b, s, H, dh,
                                       W.D, c.st);
    if (e != cudaSuccess) return fail(LR_ERR_CUDA, "attention row dot: %s", cudaGetErrorString(e));
  }
  if (attn_flash_fwd_supported(dh)) {
    // dK and dV in one persistent launch over (head, 128 keys) items (S^T, dP^T, dV, dK in TMEM; P^T and
    // dS^T as the TMEM A operands of dV and dK), which also stores scale dS^T (bf16, head-major, in the
    // workspace); then dQ = dS K as one GEMM that reads it MN-major.  Algorithmic FLOPs: four products
    // over the causal half; bytes: q, k, v, dO read, dk, dv and the causal half of dS^T written.
    bf16* dst = W.dST;
    {
      const double causal4 = 4.0 * 2.0 * b * H * static_cast<double>(s) * s * dh * 0.5;
      LaunchScope scope("attn_flash_bwd", c.st, causal4, 12.0 * b * s * d + 1.0 * R * s + 8.0 * R);
      cudaError_t e = launch_attn_flash_bwd(
          static_cast<const bf16*>(q), static_cast<const bf16*>(k), static_cast<const bf16*>(v),
          static_cast<const bf16*>(dout), lse, W.D, dst, static_cast<bf16*>(dk), static_cast<bf16*>(dv), b, s, H, dh,
          scale, W.sched, c.err, c.st);
      if (e != cudaSuccess) return fail(LR_ERR_CUDA, "attention backward: %s", cudaGetErrorString(e));
    }
    return attn_gemm(c, EPI_STORE, a, s, dh, s, {dst, s}, true, false, {k, d}, true, true, dq, d, true, 2);
  }
  {
    // One dual-accumulator launch per tile of every head: S = Q K^T again (only its log-sum-exp
    // was kept) and dP = dO V^T, turned in the epilogue into P = exp(scale S - lse) and
    // dS = scale P (dP - D), stored bf16 (head-major) up to the end of each row's 256-key tile.
    GemmCall g = attn_call(a, s, s, dh, true, true, false, 1);
    g.nacc = 2;
    g.A[0] = {q, d};
    g.B[0] = {k, d};
    g.A[1] = {dout, d};
    g.B[1] = {v, d};
    g.ep.out0[0] = W.P;
    g.ep.out1[0] = W.dS;
    g.ep.ldo0 = g.ep.ldo1 = s;
    g.ep.rowscale = lse;
    g.ep.rowpart_in = W.D;
    g.ep.rowpart_in_chunks = 1;
    g.ep.coef = scale;
    LR_TRY(gemm(c, EPI_ATTN_BWD, g, 8.0 * R));
  }
  // dV = P^T dO (P read MN-major: keys index its columns), dQ = dS K, dK = dS^T Q (dS holds scale);
  // the gradients land token-major in place
  LR_TRY(attn_gemm(c, EPI_STORE, a, s, dh, s, {W.P, s}, true, false, {dout, d}, true, true, dv, d, true, 3));
  LR_TRY(attn_gemm(c, EPI_STORE, a, s, dh, s, {W.dS, s}, false, false, {k, d}, true, true, dq, d, true, 2));
  return attn_gemm(c, EPI_STORE, a, s, dh, s, {W.dS, s}, true, false, {q, d}, true, true, dk, d, true, 3);
}

// ============================================================ transformer block
// Pre-norm low-rank transformer block: [q; k; v] = normed group (gain g_attn), causal attention,
// x1 = x + LR_o(o) (residual fused into the o-projection's B GEMM), out = MLP block(x1) in
// checkpoint mode.  bf16.  The saved set keeps q, k, v, o and x1 besides the pieces' own sets.
struct BlockSaved {
  void *qkv, *q, *k, *v, *o, *oproj, *x1, *mlp;
  float* lse;
};

static size_t block_saved_layout(int b, int s, int H, int dh, int f, int ra, int rm, void* base, BlockSaved* S) {
  Arena ar(base);
  BlockSaved tmp;
  if (!S) S = &tmp;
  const int T = b * s, d = H * dh;
  const size_t act = sizeof(bf16) * static_cast<size_t>(T) * d;
  S->qkv = ar.take(proj_saved_layout(LR_BF16, T, ra, 3, 1, nullptr, nullptr));
  S->q = ar.take(act);
  S->k = ar.take(act);
  S->v = ar.take(act);
  S->o = ar.take(act);
  S->lse = static_cast<float*>(ar.take(sizeof(float) * static_cast<size_t>(b) * H * s));
  S->oproj = ar.take(proj_saved_layout(LR_BF16, T, ra, 1, 0, nullptr, nullptr));
  S->x1 = ar.take(act);
  S->mlp = ar.take(mlp_saved_layout(LR_BF16, LR_SAVE_CKPT, T, d, f, rm, nullptr, nullptr));
  return ar.size();
}

struct BlockWs {
  void* sub;  // the workspace of whichever piece runs
  void *dx1, *dO, *dq, *dk, *dv;
};

static size_t block_ws_layout(int b, int s, int H, int dh, int f, int ra, int rm, void* base, BlockWs* W) {
  Arena ar(base);
  BlockWs tmp;
  if (!W) W = &tmp;
  const int T = b * s, d = H * dh;
  const size_t act = sizeof(bf16) * static_cast<size_t>(T) * d;
  const size_t sub = std::max({proj_ws_layout(LR_BF16, true, T, d, d, ra, 3, 1, nullptr, nullptr),
                               proj_ws_layout(LR_BF16, true, T, d, d, ra, 1, 0, nullptr, nullptr),
                               attn_ws_layout(b, s, H, dh, nullptr, nullptr),
                               mlp_fwd_ws_layout(LR_BF16, LR_SAVE_CKPT, T, d, f, rm, nullptr, nullptr),
                               mlp_bwd_ws_layout(LR_BF16, LR_SAVE_CKPT, T, d, f, rm, nullptr, nullptr)});
  W->sub = ar.take(sub);
  void** bufs[5] = {&W->dx1, &W->dO, &W->dq, &W->dk, &W->dv};
  for (void** p : bufs) *p = ar.take(act);
  return ar.size();
}

static lr_status block_fwd_impl(const Ctx& c, int b, int s, int H, int dh, int f, int ra, int rm, float eps,
                                const void* x, const lr_block_weights& w, void* out, void* saved, void* ws) {
  BlockSaved S;
  BlockWs W;
  block_saved_layout(b, s, H, dh, f, ra, rm, saved, &S);
  block_ws_layout(b, s, H, dh, f, ra, rm, ws, &W);
  const int T = b * s, d = H * dh;
  const lr_pair qkv[3] = {w.q, w.k, w.v};
  void* const outs[3] = {S.q, S.k, S.v};
  LR_TRY(proj_fwd_impl(c, T, d, d, ra, 3, qkv, w.g_attn, eps, x, outs, S.qkv, W.sub));
  LR_TRY(attn_fwd_impl(c, b, s, H, dh, 1.f / sqrtf(static_cast<float>(dh)), S.q, S.k, S.v, S.o, S.lse, W.sub));
  void* const x1[1] = {S.x1};
  LR_TRY(proj_fwd_impl(c, T, d, d, ra, 1, &w.o, nullptr, eps, S.o, x1, S.oproj, W.sub, x));
  return mlp_fwd_impl(c, LR_SAVE_CKPT, T, d, f, rm, eps, S.x1, w.g_mlp, w.gate, w.up, w.down, out, S.mlp, W.sub);
}

static lr_status block_bwd_impl(const Ctx& c, int b, int s, int H, int dh, int f, int ra, int rm, float eps,
                                const void* x, const lr_block_weights& w, const void* saved, const void* dout,
                                void* dx, const lr_block_grads& gr, void* ws) {
  BlockSaved S;
  BlockWs W;
  block_saved_layout(b, s, H, dh, f, ra, rm, const_cast<void*>(saved), &S);
  block_ws_layout(b, s, H, dh, f, ra, rm, ws, &W);
  const int T = b * s, d = H * dh;
  // MLP block: dx1 already holds the gradient its residual passes through
  LR_TRY(mlp_bwd_impl(c, LR_SAVE_CKPT, T, d, f, rm, eps, S.x1, w.g_mlp, w.gate, w.up, w.down, S.mlp, dout, W.dx1,
                      gr.dg_mlp, gr.gate, gr.up, gr.down, W.sub));
  // o-projection: its output's gradient is dx1; its dx is dL/do
  const void* const d1[1] = {W.dx1};
  LR_TRY(proj_bwd_impl(c, T, d, d, ra, 1, &w.o, nullptr, S.o, S.oproj, d1, W.dO, nullptr, &gr.o, W.sub));
  LR_TRY(attn_bwd_impl(c, b, s, H, dh, 1.f / sqrtf(static_cast<float>(dh)), S.q, S.k, S.v, S.o, S.lse, W.dO, W.dq,
                       W.dk, W.dv, W.sub));
  // q/k/v group, with the residual's gradient dx1 added into dx
  const lr_pair qkv[3] = {w.q, w.k, w.v};
  const void* const dqkv[3] = {W.dq, W.dk, W.dv};
  const lr_pair_grad gq[3] = {gr.q, gr.k, gr.v};
  return proj_bwd_impl(c, T, d, d, ra, 3, qkv, w.g_attn, x, S.qkv, dqkv, dx, gr.dg_attn, gq, W.sub, W.dx1);
}

// ============================================================ block stack
struct StackWs {
  void* acts;   // x_1 .. x_L, [L][T, d]
  void* saved;  // [L][mlp saved]
  size_t saved_each;
  void* scratch;  // max(mlp fwd ws, mlp bwd ws)
  void *dy0, *dy1;
  float* mse_part;
};

static size_t stack_ws_layout(lr_dtype dt, lr_mode mode, int L, int T, int d, int f, int r, void* base,
                              StackWs* W) {
  const size_t es = esize(dt);
  Arena ar(base);
  StackWs tmp;
  if (!W) W = &tmp;
  W->acts = ar.take(es * L * T * d);
  W->saved_each = mlp_saved_layout(dt, mode, T, d, f, r, nullptr, nullptr);
  W->saved = ar.take(W->saved_each * L);
  W->scratch = ar.take(std::max(mlp_fwd_ws_layout(dt, mode, T, d, f, r, nullptr, nullptr),
                                mlp_bwd_ws_layout(dt, mode, T, d, f, r, nullptr, nullptr)));
  W->dy0 = ar.take(es * T * d);
  W->dy1 = ar.take(es * T * d);
  W->mse_part = static_cast<float*>(ar.take(sizeof(float) * kMseParts));
  return ar.size();
}

static lr_status stack_impl(const Ctx& c, lr_mode mode, int L, int T, int d, int f, int r, float eps, const void* x,
                            const void* target, const void* const* gs, const lr_pair* pairs, float* loss, void* dx,
                            float* const* dgs, const lr_pair_grad* grads, void* ws) {
  StackWs W;
  stack_ws_layout(c.dt, mode, L, T, d, f, r, ws, &W);
  const size_t act_bytes = c.es * T * d;
  auto act = [&](int l) -> void* { return l == 0 ? const_cast<void*>(x) : off(W.acts, act_bytes * (l - 1)); };
  auto sv = [&](int l) -> void* { return off(W.saved, W.saved_each * l); };
  for (int l = 0; l < L; ++l)
    LR_TRY(mlp_fwd_impl(c, mode, T, d, f, r, eps, act(l), gs[l], pairs[3 * l], pairs[3 * l + 1], pairs[3 * l + 2],
                        act(l + 1), sv(l), W.scratch));
  {
    const long long n = 1LL * T * d;
    LaunchScope scope("mse", c.st, 0, 3.0 * c.es * n);
    cudaError_t e = (c.dt == LR_BF16)
                        ? launch_mse<bf16>(static_cast<const bf16*>(act(L)), static_cast<const bf16*>(target), n,
                                           static_cast<bf16*>(W.dy0), W.mse_part, kMseParts, loss, c.st)
                        : launch_mse<float>(static_cast<const float*>(act(L)), static_cast<const float*>(target), n,
                                            static_cast<float*>(W.dy0), W.mse_part, kMseParts, loss, c.st);
    if (e != cudaSuccess) return fail(LR_ERR_CUDA, "mse: %s", cudaGetErrorString(e));
  }
  void* dcur = W.dy0;
  void* dnext = W.dy1;
  for (int l = L - 1; l >= 0; --l) {
    void* dst = (l == 0 && dx) ? dx : dnext;
    LR_TRY(mlp_bwd_impl(c, mode, T, d, f, r, eps, act(l), gs[l], pairs[3 * l], pairs[3 * l + 1], pairs[3 * l + 2],
                        sv(l), dcur, dst, dgs[l], grads[3 * l], grads[3 * l + 1], grads[3 * l + 2], W.scratch));
    std::swap(dcur, dnext);
  }
  return LR_OK;
}

// ============================================================ validation
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static lr_status check_ptr(const void* p, const char* name) {
  if (!p) return fail(LR_ERR_NULL, "%s is NULL", name);
  if (!aligned16(p)) return fail(LR_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return LR_OK;
}

static lr_status check_dim(int v, const char* name, bool mult8) {
  if (v <= 0) return fail(LR_ERR_SHAPE, "%s = %d must be positive", name, v);
  if (v > (1 << 24)) return fail(LR_ERR_SHAPE, "%s = %d exceeds 16777216", name, v);
  if (mult8 && (v % 8)) return fail(LR_ERR_SHAPE, "%s = %d must be a multiple of 8", name, v);
  return LR_OK;
}

static lr_status check_dtype(lr_dtype dt) {
  if (dt != LR_F32 && dt != LR_BF16) return fail(LR_ERR_DTYPE, "unknown dtype %d", static_cast<int>(dt));
  return LR_OK;
}

static lr_status check_mode(lr_mode m) {
  if (m != LR_SAVE_FULL && m != LR_SAVE_CKPT) return fail(LR_ERR_DTYPE, "unknown mode %d", static_cast<int>(m));
  return LR_OK;
}

static lr_status check_act(lr_act a) {
  if (a != LR_ACT_SILU && a != LR_ACT_IDENTITY) return fail(LR_ERR_DTYPE, "unknown act %d", static_cast<int>(a));
  return LR_OK;
}

static lr_status check_size(size_t have, size_t need, const char* name) {
  if (have < need) return fail(LR_ERR_WORKSPACE, "%s has %zu bytes, needs %zu", name, have, need);
  return LR_OK;
}

static lr_status make_ctx(lr_dtype dt, void* stream, Ctx* c, lr_act act = LR_ACT_SILU) {
  c->dt = dt;
  c->act = act == LR_ACT_IDENTITY ? 1 : 0;
  c->es = esize(dt);
  c->st = static_cast<cudaStream_t>(stream);
  LR_TRY(device_error_word(&c->err));
  c->sms = device_sm_count();
  c->chunk = chunk_width(dt);
  return LR_OK;
}

static lr_status check_mlp_dims(int T, int d, int f, int r) {
  LR_TRY(check_dim(T, "T", false));
  LR_TRY(check_dim(d, "d", true));
  LR_TRY(check_dim(f, "f", true));
  LR_TRY(check_dim(r, "r", true));
  return LR_OK;
}

static lr_status check_proj_dims(int T, int d_in, int d_out, int r, int group) {
  LR_TRY(check_dim(T, "T", false));
  LR_TRY(check_dim(d_in, "d_in", true));
  LR_TRY(check_dim(d_out, "d_out", true));
  LR_TRY(check_dim(r, "r", true));
  if (group < 1 || group > kMaxStack) return fail(LR_ERR_SHAPE, "group = %d must be 1..%d", group, kMaxStack);
  return LR_OK;
}

// ================================================== allocation-free variant
// Scratch of lr_proj_fwd_noalloc: the folded, stacked A' = [A_1; ...; A_group] * g
// (the only workspace a projection-group forward needs).  It lives in a
// file-scope device array, so every GPU that loads this library holds it until
// the process exits, and every call shares it.
static constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(LR_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
static void* s_noalloc_scratch[kMaxDevices];

// The host-side name g_noalloc_scratch is only a stand-in for the array: its
// device address is looked up once per device, with that device current.
static lr_status noalloc_scratch(void** out) {
  int dev;
  LR_TRY(current_device(&dev));
  std::lock_guard<std::mutex> lk(s_dev_mu);
  if (!s_noalloc_scratch[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
      return fail(LR_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch): %s", cudaGetErrorString(e));
    s_noalloc_scratch[dev] = p;
  }
  *out = s_noalloc_scratch[dev];
  return LR_OK;
}

}  // namespace lr

using namespace lr;

// ================================================================== C ABI
extern "C" {

int lr_version(void) { return 100; }

unsigned long long lr_launch_count(void) { return s_launches.load(); }

lr_status lr_profile_start(void) {
  std::lock_guard<std::mutex> lk(s_prof_mu);
  for (auto& r : s_prof) {
    s_event_pool.push_back(r.a);
    s_event_pool.push_back(r.b);
  }
  s_prof.clear();
  s_prof_result.clear();
  s_prof_on = true;
  return LR_OK;
}

lr_status lr_profile_filter(const char* prefix) {
  std::lock_guard<std::mutex> lk(s_prof_mu);
  s_prof_filter = prefix ? prefix : "";
  return LR_OK;
}

lr_status lr_profile_stop(void) {
  std::lock_guard<std::mutex> lk(s_prof_mu);
  s_prof_on = false;
  s_prof_result.clear();
  for (auto& r : s_prof) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return fail(LR_ERR_CUDA, "profile event: %s", cudaGetErrorString(e));
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    auto it = std::find_if(s_prof_result.begin(), s_prof_result.end(),
                           [&](const ProfAgg& a) { return a.name == r.name; });
    if (it == s_prof_result.end()) {
      s_prof_result.push_back({r.name, 0, 0.0, 0.0, 0.0});
      it = s_prof_result.end() - 1;
    }
    it->n += 1;
    it->ms += ms;
    it->flops += r.flops;
    it->bytes += r.bytes;
  }
  return LR_OK;
}

int lr_profile_count(void) {
  std::lock_guard<std::mutex> lk(s_prof_mu);
  return static_cast<int>(s_prof_result.size());
}

lr_status lr_profile_entry(int i, char* name, size_t name_len, long long* launches, double* total_ms, double* flops,
                           double* bytes) {
  std::lock_guard<std::mutex> lk(s_prof_mu);
  if (i < 0 || i >= static_cast<int>(s_prof_result.size())) return fail(LR_ERR_SHAPE, "profile entry %d", i);
  const ProfAgg& a = s_prof_result[i];
  if (name && name_len) {
    strncpy(name, a.name.c_str(), name_len - 1);
    name[name_len - 1] = 0;
  }
  if (launches) *launches = a.n;
  if (total_ms) *total_ms = a.ms;
  if (flops) *flops = a.flops;
  if (bytes) *bytes = a.bytes;
  return LR_OK;
}

const char* lr_last_error(void) { return t_last_error.c_str(); }

size_t lr_mlp_saved_bytes(lr_dtype dt, lr_mode mode, int T, int d, int f, int r) {
  if (check_dtype(dt) || check_mode(mode) || check_mlp_dims(T, d, f, r)) return 0;
  return mlp_saved_layout(dt, mode, T, d, f, r, nullptr, nullptr);
}

size_t lr_mlp_fwd_workspace_bytes(lr_dtype dt, lr_mode mode, int T, int d, int f, int r) {
  if (check_dtype(dt) || check_mode(mode) || check_mlp_dims(T, d, f, r)) return 0;
  return mlp_fwd_ws_layout(dt, mode, T, d, f, r, nullptr, nullptr);
}

size_t lr_mlp_bwd_workspace_bytes(lr_dtype dt, lr_mode mode, int T, int d, int f, int r) {
  if (check_dtype(dt) || check_mode(mode) || check_mlp_dims(T, d, f, r)) return 0;
  return mlp_bwd_ws_layout(dt, mode, T, d, f, r, nullptr, nullptr);
}

static lr_status check_pair(lr_pair p, const char* name) {
  char buf[64];
  snprintf(buf, sizeof(buf), "%s.A", name);
  LR_TRY(check_ptr(p.A, buf));
  snprintf(buf, sizeof(buf), "%s.B", name);
  return check_ptr(p.B, buf);
}

static lr_status check_grad(lr_pair_grad p, const char* name) {
  char buf[64];
  snprintf(buf, sizeof(buf), "%s.dA", name);
  LR_TRY(check_ptr(p.dA, buf));
  snprintf(buf, sizeof(buf), "%s.dB", name);
  return check_ptr(p.dB, buf);
}

lr_status lr_mlp_fwd(lr_dtype dt, lr_mode mode, lr_act act, int T, int d, int f, int r, float eps, const void* x,
                     const void* g, lr_pair gate, lr_pair up, lr_pair down, void* out, void* saved,
                     size_t saved_bytes, void* ws, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_mode(mode));
  LR_TRY(check_act(act));
  LR_TRY(check_mlp_dims(T, d, f, r));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(g, "g"));
  LR_TRY(check_pair(gate, "gate"));
  LR_TRY(check_pair(up, "up"));
  LR_TRY(check_pair(down, "down"));
  LR_TRY(check_ptr(out, "out"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, mlp_saved_layout(dt, mode, T, d, f, r, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, mlp_fwd_ws_layout(dt, mode, T, d, f, r, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c, act));
  return mlp_fwd_impl(c, mode, T, d, f, r, eps, x, g, gate, up, down, out, saved, ws);
}

lr_status lr_mlp_bwd(lr_dtype dt, lr_mode mode, lr_act act, int T, int d, int f, int r, float eps, const void* x,
                     const void* g, lr_pair gate, lr_pair up, lr_pair down, const void* saved, size_t saved_bytes,
                     const void* dout, void* dx, float* dg, lr_pair_grad dgate, lr_pair_grad dup, lr_pair_grad ddown,
                     void* ws, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_mode(mode));
  LR_TRY(check_act(act));
  LR_TRY(check_mlp_dims(T, d, f, r));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(g, "g"));
  LR_TRY(check_pair(gate, "gate"));
  LR_TRY(check_pair(up, "up"));
  LR_TRY(check_pair(down, "down"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(dout, "dout"));
  LR_TRY(check_ptr(dx, "dx"));
  LR_TRY(check_ptr(dg, "dg"));
  LR_TRY(check_grad(dgate, "dgate"));
  LR_TRY(check_grad(dup, "dup"));
  LR_TRY(check_grad(ddown, "ddown"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, mlp_saved_layout(dt, mode, T, d, f, r, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, mlp_bwd_ws_layout(dt, mode, T, d, f, r, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c, act));
  return mlp_bwd_impl(c, mode, T, d, f, r, eps, x, g, gate, up, down, saved, dout, dx, dg, dgate, dup, ddown, ws);
}

size_t lr_proj_saved_bytes(lr_dtype dt, int T, int d_in, int d_out, int r, int group, int norm) {
  if (check_dtype(dt) || check_proj_dims(T, d_in, d_out, r, group)) return 0;
  return proj_saved_layout(dt, T, r, group, norm != 0, nullptr, nullptr);
}

size_t lr_proj_fwd_workspace_bytes(lr_dtype dt, int T, int d_in, int d_out, int r, int group, int norm) {
  if (check_dtype(dt) || check_proj_dims(T, d_in, d_out, r, group)) return 0;
  return proj_ws_layout(dt, false, T, d_in, d_out, r, group, norm != 0, nullptr, nullptr);
}

size_t lr_proj_bwd_workspace_bytes(lr_dtype dt, int T, int d_in, int d_out, int r, int group, int norm) {
  if (check_dtype(dt) || check_proj_dims(T, d_in, d_out, r, group)) return 0;
  return proj_ws_layout(dt, true, T, d_in, d_out, r, group, norm != 0, nullptr, nullptr);
}

lr_status lr_proj_fwd(lr_dtype dt, lr_act act, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                      const void* g, float eps, const void* x, void* const* outs, void* saved, size_t saved_bytes,
                      void* ws, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_act(act));
  LR_TRY(check_proj_dims(T, d_in, d_out, r, group));
  if (!pairs || !outs) return fail(LR_ERR_NULL, "pairs / outs is NULL");
  for (int i = 0; i < group; ++i) {
    LR_TRY(check_pair(pairs[i], "pairs[i]"));
    LR_TRY(check_ptr(outs[i], "outs[i]"));
  }
  if (g) LR_TRY(check_ptr(g, "g"));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, proj_saved_layout(dt, T, r, group, g != nullptr, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, proj_ws_layout(dt, false, T, d_in, d_out, r, group, g != nullptr, nullptr, nullptr),
                    "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c, act));
  return proj_fwd_impl(c, T, d_in, d_out, r, group, pairs, g, eps, x, outs, saved, ws);
}

lr_status lr_proj_bwd(lr_dtype dt, lr_act act, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                      const void* g, float eps, const void* x, const void* saved, size_t saved_bytes,
                      const void* const* douts, void* dx, float* dg, const lr_pair_grad* grads, void* ws,
                      size_t ws_bytes, void* stream) {
  (void)eps;
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_act(act));
  LR_TRY(check_proj_dims(T, d_in, d_out, r, group));
  if (!pairs || !douts || !grads) return fail(LR_ERR_NULL, "pairs / douts / grads is NULL");
  for (int i = 0; i < group; ++i) {
    LR_TRY(check_pair(pairs[i], "pairs[i]"));
    LR_TRY(check_ptr(douts[i], "douts[i]"));
    LR_TRY(check_grad(grads[i], "grads[i]"));
  }
  if (g) {
    LR_TRY(check_ptr(g, "g"));
    LR_TRY(check_ptr(dg, "dg"));
  }
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(dx, "dx"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, proj_saved_layout(dt, T, r, group, g != nullptr, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, proj_ws_layout(dt, true, T, d_in, d_out, r, group, g != nullptr, nullptr, nullptr),
                    "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c, act));
  return proj_bwd_impl(c, T, d_in, d_out, r, group, pairs, g, x, saved, douts, dx, dg, grads, ws);
}

size_t lr_dense_saved_bytes(lr_dtype dt, int T, int d, int f) {
  if (check_dtype(dt) || check_dim(T, "T", false) || check_dim(d, "d", true) || check_dim(f, "f", true)) return 0;
  return dense_saved_layout(dt, T, f, nullptr, nullptr);
}

size_t lr_dense_fwd_workspace_bytes(lr_dtype dt, int T, int d, int f) {
  if (check_dtype(dt) || check_dim(T, "T", false) || check_dim(d, "d", true) || check_dim(f, "f", true)) return 0;
  return dense_ws_layout(dt, false, T, d, f, nullptr, nullptr);
}

size_t lr_dense_bwd_workspace_bytes(lr_dtype dt, int T, int d, int f) {
  if (check_dtype(dt) || check_dim(T, "T", false) || check_dim(d, "d", true) || check_dim(f, "f", true)) return 0;
  return dense_ws_layout(dt, true, T, d, f, nullptr, nullptr);
}

lr_status lr_dense_fwd(lr_dtype dt, int T, int d, int f, float eps, const void* x, const void* g, const void* W_gate,
                       const void* W_up, const void* W_down, void* out, void* saved, size_t saved_bytes, void* ws,
                       size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_mlp_dims(T, d, f, 8));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(g, "g"));
  LR_TRY(check_ptr(W_gate, "W_gate"));
  LR_TRY(check_ptr(W_up, "W_up"));
  LR_TRY(check_ptr(W_down, "W_down"));
  LR_TRY(check_ptr(out, "out"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, dense_saved_layout(dt, T, f, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, dense_ws_layout(dt, false, T, d, f, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  return dense_fwd_impl(c, T, d, f, eps, x, g, W_gate, W_up, W_down, out, saved, ws);
}

lr_status lr_dense_bwd(lr_dtype dt, int T, int d, int f, float eps, const void* x, const void* g, const void* W_gate,
                       const void* W_up, const void* W_down, const void* saved, size_t saved_bytes, const void* dout,
                       void* dx, float* dg, float* dW_gate, float* dW_up, float* dW_down, void* ws, size_t ws_bytes,
                       void* stream) {
  (void)eps;
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_mlp_dims(T, d, f, 8));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(g, "g"));
  LR_TRY(check_ptr(W_gate, "W_gate"));
  LR_TRY(check_ptr(W_up, "W_up"));
  LR_TRY(check_ptr(W_down, "W_down"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(dout, "dout"));
  LR_TRY(check_ptr(dx, "dx"));
  LR_TRY(check_ptr(dg, "dg"));
  LR_TRY(check_ptr(dW_gate, "dW_gate"));
  LR_TRY(check_ptr(dW_up, "dW_up"));
  LR_TRY(check_ptr(dW_down, "dW_down"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, dense_saved_layout(dt, T, f, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, dense_ws_layout(dt, true, T, d, f, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  return dense_bwd_impl(c, T, d, f, x, g, W_gate, W_up, W_down, saved, dout, dx, dg, dW_gate, dW_up, dW_down, ws);
}

static lr_status check_attn(lr_dtype dt, int b, int s, int H, int dh) {
  LR_TRY(check_dtype(dt));
  if (dt != LR_BF16) return fail(LR_ERR_UNSUPPORTED, "attention: bf16 only");
  if (b < 1 || H < 1 || s < 256 || s % 256 || dh < 128 || dh % 128)
    return fail(LR_ERR_SHAPE, "attention: b = %d, H = %d >= 1, s = %d a multiple of 256, dh = %d of 128 needed", b,
                H, s, dh);
  // Tokens b*s and channels H*dh are formed in int by the callers of this check: bound them first.
  if (1LL * b * s > (1 << 24) || 1LL * H * dh > (1 << 24))
    return fail(LR_ERR_SHAPE, "attention: b*s = %lld tokens and H*dh = %lld channels must not exceed 16777216",
                1LL * b * s, 1LL * H * dh);
  if (1LL * b * H * s * s > (1LL << 40) || 1LL * b * H * s > (1LL << 30))
    return fail(LR_ERR_SHAPE, "attention: b*H*s*s or b*H*s too large");
  return LR_OK;
}

size_t lr_attn_saved_bytes(int b, int s, int H, int dh) {
  if (check_attn(LR_BF16, b, s, H, dh)) return 0;
  return static_cast<size_t>(b) * H * s * sizeof(float);
}

size_t lr_attn_workspace_bytes(int b, int s, int H, int dh) {
  if (check_attn(LR_BF16, b, s, H, dh)) return 0;
  return attn_ws_layout(b, s, H, dh, nullptr, nullptr);
}

lr_status lr_attn_fwd(lr_dtype dt, int b, int s, int H, int dh, float scale, const void* q, const void* k,
                      const void* v, void* o, void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                      void* stream) {
  t_last_error.clear();
  LR_TRY(check_attn(dt, b, s, H, dh));
  LR_TRY(check_ptr(q, "q"));
  LR_TRY(check_ptr(k, "k"));
  LR_TRY(check_ptr(v, "v"));
  LR_TRY(check_ptr(o, "o"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, lr_attn_saved_bytes(b, s, H, dh), "saved"));
  LR_TRY(check_size(ws_bytes, attn_ws_layout(b, s, H, dh, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  PdlOff serial;  // see lr_block_fwd
  return attn_fwd_impl(c, b, s, H, dh, scale, q, k, v, o, static_cast<float*>(saved), ws);
}

lr_status lr_attn_bwd(lr_dtype dt, int b, int s, int H, int dh, float scale, const void* q, const void* k,
                      const void* v, const void* o, const void* saved, const void* dout, void* dq, void* dk,
                      void* dv, void* ws, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_attn(dt, b, s, H, dh));
  const void* ptrs[] = {q, k, v, o, saved, dout, dq, dk, dv, ws};
  const char* names[] = {"q", "k", "v", "o", "saved", "dout", "dq", "dk", "dv", "ws"};
  for (int i = 0; i < 10; ++i) LR_TRY(check_ptr(ptrs[i], names[i]));
  LR_TRY(check_size(ws_bytes, attn_ws_layout(b, s, H, dh, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  PdlOff serial;  // see lr_block_fwd
  return attn_bwd_impl(c, b, s, H, dh, scale, q, k, v, o, static_cast<const float*>(saved), dout, dq, dk, dv, ws);
}

static lr_status check_block(lr_dtype dt, int b, int s, int H, int dh, int f, int ra, int rm) {
  LR_TRY(check_attn(dt, b, s, H, dh));
  LR_TRY(check_mlp_dims(b * s, H * dh, f, rm));
  return check_mlp_dims(b * s, H * dh, H * dh, ra);
}

size_t lr_block_saved_bytes(int b, int s, int H, int dh, int f, int ra, int rm) {
  if (check_block(LR_BF16, b, s, H, dh, f, ra, rm)) return 0;
  return block_saved_layout(b, s, H, dh, f, ra, rm, nullptr, nullptr);
}

size_t lr_block_workspace_bytes(int b, int s, int H, int dh, int f, int ra, int rm) {
  if (check_block(LR_BF16, b, s, H, dh, f, ra, rm)) return 0;
  return block_ws_layout(b, s, H, dh, f, ra, rm, nullptr, nullptr);
}

static lr_status check_block_weights(const lr_block_weights* w) {
  LR_TRY(check_ptr(w, "w"));
  const void* ptrs[] = {w->g_attn, w->q.A, w->q.B, w->k.A, w->k.B, w->v.A, w->v.B, w->o.A, w->o.B,
                        w->g_mlp, w->gate.A, w->gate.B, w->up.A, w->up.B, w->down.A, w->down.B};
  for (const void* p : ptrs) LR_TRY(check_ptr(p, "block weight"));
  return LR_OK;
}

lr_status lr_block_fwd(lr_dtype dt, int b, int s, int H, int dh, int f, int ra, int rm, float eps, const void* x,
                       const lr_block_weights* w, void* out, void* saved, size_t saved_bytes, void* ws,
                       size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_block(dt, b, s, H, dh, f, ra, rm));
  LR_TRY(check_block_weights(w));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(out, "out"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, block_saved_layout(b, s, H, dh, f, ra, rm, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, block_ws_layout(b, s, H, dh, f, ra, rm, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  // Without programmatic dependent launch: with it, three fwd+bwd steps of the block issued back to
  // back stopped making progress on the GPU (one or two did not; the cause is not known).
  PdlOff serial;
  return block_fwd_impl(c, b, s, H, dh, f, ra, rm, eps, x, *w, out, saved, ws);
}

lr_status lr_block_bwd(lr_dtype dt, int b, int s, int H, int dh, int f, int ra, int rm, float eps, const void* x,
                       const lr_block_weights* w, const void* saved, size_t saved_bytes, const void* dout, void* dx,
                       const lr_block_grads* g, void* ws, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_block(dt, b, s, H, dh, f, ra, rm));
  LR_TRY(check_block_weights(w));
  LR_TRY(check_ptr(g, "g"));
  const void* gp[] = {g->dg_attn, g->q.dA, g->q.dB, g->k.dA, g->k.dB, g->v.dA, g->v.dB, g->o.dA, g->o.dB,
                      g->dg_mlp, g->gate.dA, g->gate.dB, g->up.dA, g->up.dB, g->down.dA, g->down.dB};
  for (const void* p : gp) LR_TRY(check_ptr(p, "block gradient"));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_ptr(dout, "dout"));
  LR_TRY(check_ptr(dx, "dx"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(saved_bytes, block_saved_layout(b, s, H, dh, f, ra, rm, nullptr, nullptr), "saved"));
  LR_TRY(check_size(ws_bytes, block_ws_layout(b, s, H, dh, f, ra, rm, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  PdlOff serial;  // see lr_block_fwd
  return block_bwd_impl(c, b, s, H, dh, f, ra, rm, eps, x, *w, saved, dout, dx, *g, ws);
}

size_t lr_btp_payload_floats(int T, int r, int group) {
  if (check_dim(T, "T", false) || check_dim(r, "r", true) || group < 1 || group > kMaxStack) return 0;
  return static_cast<size_t>(T) * group * r + static_cast<size_t>(T);
}

size_t lr_btp_workspace_bytes(lr_dtype dt, int d_shard, int r, int group) {
  if (check_dtype(dt) || check_dim(d_shard, "d_shard", true) || check_dim(r, "r", true) || group < 1 ||
      group > kMaxStack)
    return 0;
  return btp_ws_layout(dt, d_shard, r, group, nullptr, nullptr);
}

lr_status lr_btp_partial(lr_dtype dt, int T, int d_shard, int r, int group, const lr_pair* pairs, const void* g_shard,
                         const void* x_shard, float* payload, void* ws, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_proj_dims(T, d_shard, 8, r, group));
  if (!pairs) return fail(LR_ERR_NULL, "pairs is NULL");
  for (int i = 0; i < group; ++i) LR_TRY(check_ptr(pairs[i].A, "pairs[i].A"));
  LR_TRY(check_ptr(g_shard, "g_shard"));
  LR_TRY(check_ptr(x_shard, "x_shard"));
  LR_TRY(check_ptr(payload, "payload"));
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(ws_bytes, btp_ws_layout(dt, d_shard, r, group, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  return btp_partial_impl(c, T, d_shard, r, group, pairs, g_shard, x_shard, payload, ws);
}

lr_status lr_btp_finish(lr_dtype dt, lr_act act, int T, int d, int r, int group, const float* payload, float eps,
                        void* u, void* z, float* s, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_act(act));
  LR_TRY(check_proj_dims(T, d, 8, r, group));
  LR_TRY(check_ptr(payload, "payload"));
  LR_TRY(check_ptr(u, "u"));
  LR_TRY(check_ptr(z, "z"));
  LR_TRY(check_ptr(s, "s"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c, act));
  return btp_finish_impl(c, T, d, group * r, payload, eps, u, z, s);
}

size_t lr_stack_workspace_bytes(lr_dtype dt, lr_mode mode, int nblocks, int T, int d, int f, int r) {
  if (check_dtype(dt) || check_mode(mode) || check_mlp_dims(T, d, f, r) || nblocks < 1) return 0;
  return stack_ws_layout(dt, mode, nblocks, T, d, f, r, nullptr, nullptr);
}

lr_status lr_stack_step(lr_dtype dt, lr_mode mode, int nblocks, int T, int d, int f, int r, float eps, const void* x,
                        const void* target, const void* const* gs, const lr_pair* pairs, float* loss, void* dx,
                        float* const* dgs, const lr_pair_grad* grads, void* ws, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_mode(mode));
  LR_TRY(check_mlp_dims(T, d, f, r));
  if (nblocks < 1 || nblocks > 4096) return fail(LR_ERR_SHAPE, "nblocks = %d must be 1..4096", nblocks);
  if (!gs || !pairs || !dgs || !grads) return fail(LR_ERR_NULL, "gs / pairs / dgs / grads is NULL");
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(target, "target"));
  LR_TRY(check_ptr(loss, "loss"));
  if (dx) LR_TRY(check_ptr(dx, "dx"));
  for (int l = 0; l < nblocks; ++l) {
    LR_TRY(check_ptr(gs[l], "gs[l]"));
    LR_TRY(check_ptr(dgs[l], "dgs[l]"));
    for (int k = 0; k < 3; ++k) {
      LR_TRY(check_pair(pairs[3 * l + k], "pairs[i]"));
      LR_TRY(check_grad(grads[3 * l + k], "grads[i]"));
    }
  }
  LR_TRY(check_ptr(ws, "ws"));
  LR_TRY(check_size(ws_bytes, stack_ws_layout(dt, mode, nblocks, T, d, f, r, nullptr, nullptr), "ws"));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  return stack_impl(c, mode, nblocks, T, d, f, r, eps, x, target, gs, pairs, loss, dx, dgs, grads, ws);
}

lr_status lr_proj_fwd_noalloc(lr_dtype dt, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                              const void* g, float eps, const void* x, void* const* outs, void* saved,
                              size_t saved_bytes, void* stream) {
  t_last_error.clear();
  LR_TRY(check_dtype(dt));
  LR_TRY(check_proj_dims(T, d_in, d_out, r, group));
  if (!pairs || !outs) return fail(LR_ERR_NULL, "pairs / outs is NULL");
  for (int i = 0; i < group; ++i) {
    LR_TRY(check_pair(pairs[i], "pairs[i]"));
    LR_TRY(check_ptr(outs[i], "outs[i]"));
  }
  if (g) LR_TRY(check_ptr(g, "g"));
  LR_TRY(check_ptr(x, "x"));
  LR_TRY(check_ptr(saved, "saved"));
  LR_TRY(check_size(saved_bytes, proj_saved_layout(dt, T, r, group, g != nullptr, nullptr, nullptr), "saved"));
  const size_t need = proj_ws_layout(dt, false, T, d_in, d_out, r, group, g != nullptr, nullptr, nullptr);
  if (need > kNoAllocScratchBytes)
    return fail(LR_ERR_WORKSPACE,
                "lr_proj_fwd_noalloc: group * r * d_in weights need %zu bytes of scratch, more than its fixed "
                "%zu-byte device array; use lr_proj_fwd with a caller workspace",
                need, kNoAllocScratchBytes);
  {
    std::lock_guard<std::mutex> lk(s_prof_mu);
    if (s_prof_on)
      return fail(LR_ERR_UNSUPPORTED,
                  "lr_proj_fwd_noalloc does not run while profiling is on (the profiler creates CUDA events)");
  }
  void* scratch = nullptr;
  LR_TRY(noalloc_scratch(&scratch));
  Ctx c;
  LR_TRY(make_ctx(dt, stream, &c));
  return proj_fwd_impl(c, T, d_in, d_out, r, group, pairs, g, eps, x, outs, saved, scratch);
}

lr_status lr_check_device_error(void* stream) {
  unsigned* p = nullptr;
  LR_TRY(device_error_word(&p));
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
  unsigned word = 0;
  e = cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
  if (word) {
    const unsigned zero = 0;
    cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    return fail(LR_ERR_TIMEOUT, "device error word 0x%x (1 producer, 2 mma, 4 epilogue, 8 self-test timeout)", word);
  }
  return LR_OK;
}

lr_status lr_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  t_last_error.clear();
  unsigned* p = nullptr;
  LR_TRY(device_error_word(&p));
  if (limit_ns > 5000000000ull) return fail(LR_ERR_SHAPE, "limit_ns must be <= 5e9");
  cudaError_t e = launch_wait_selftest(p, limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(LR_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return LR_OK;
}

}  // extern "C"
