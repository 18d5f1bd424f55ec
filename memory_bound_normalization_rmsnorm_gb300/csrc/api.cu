// api.cu -- the C ABI declared in include/gbnorm.h: argument validation,
// the per-shape launch plan, and the kernel launches.
//
// Launch plan (variant choice by row length N).  Rows are cut into 16-byte
// chunks; a group of `tpr` threads owns one row and each thread K chunks of
// it, in registers.  Short rows (N <= 256) use a group of up to one warp,
// so a warp holds one or several rows and reduces with shuffles only; longer
// rows use several warps per row (shuffles plus a named-barrier fold); rows
// too long for one CTA are split across a thread-block cluster whose CTAs
// exchange partial statistics through distributed shared memory.  The
// persistent-reduction threshold of about 1024 elements named in "PyTorch
// atinge desempenho SOTA em normalizacao com torch.compile" (paragraph on
// Inductor) is where the warp-per-row regime ends here as well
// (N <= 2048 for the forward pass, whose rows sit in registers).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "../../include/gbnorm.h"
#include "common.cuh"

namespace gbn {
namespace {

__device__ unsigned g_device_error;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  unsigned *err = nullptr;
  unsigned long long ctx = 0;  // context the cached addresses belong to
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::set<std::pair<int, const void *>> g_attr_done;
std::map<std::tuple<int, int, int64_t, int, int>, Plan> g_plans;
void *g_noalloc_ptr[kMaxDevices];  // scratch array address per device, guarded by g_mu

// Unique identity (for the life of the process) of the calling thread's
// current CUDA context -- the device's primary context for runtime-API
// callers -- or 0 when there is none yet.  Every per-device cache of this
// library (device error word and scratch addresses, kernel attributes,
// plans) belongs to one context; cudaDeviceReset destroys it, and the next
// call sees a new identity and sets the device up again.  `*ok` is false
// when the driver offers no context identities (the caches are then kept
// for the life of the process).
unsigned long long current_context_id(bool *ok) {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    cudaGetLastError();
  });
  *ok = get_cur && get_id;
  if (!*ok) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

norm_status_t device_info(DeviceInfo *out, int *dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return NORM_ERR_UNSUPPORTED;
  bool ids = false;
  const unsigned long long ctx = current_context_id(&ids);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (d.sms == 0 || (ids && ctx != d.ctx)) {
    int sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return NORM_ERR_CUDA;
    }
    // (makes the device's primary context current if none was)
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
      cudaGetLastError();
      return NORM_ERR_CUDA;
    }
    // Kernel attributes, plans (which were made with them) and the scratch
    // address of an earlier context of this device are void.
    for (auto it = g_attr_done.begin(); it != g_attr_done.end();)
      it = it->first == dev ? g_attr_done.erase(it) : std::next(it);
    for (auto it = g_plans.begin(); it != g_plans.end();)
      it = std::get<0>(it->first) == dev ? g_plans.erase(it) : std::next(it);
    g_noalloc_ptr[dev] = nullptr;
    d.err = static_cast<unsigned *>(p);
    d.smem_optin = optin;
    d.sms = sms;
    d.ctx = ids ? current_context_id(&ids) : 0;
  }
  *out = d;
  *dev_out = dev;
  return NORM_OK;
}

// Sets the per-function attributes a launch needs (once per device).
norm_status_t prepare_function(int dev, const void *fn, int smem_optin) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_attr_done.count({dev, fn})) return NORM_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) !=
          cudaSuccess ||
      cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  g_attr_done.insert({dev, fn});
  return NORM_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int pow2ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Optional plan override for tuning sweeps: GBNORM_PLAN="C=2,tpr=256,rpg=1,S=4"
// (any subset).  Fields left out keep the heuristic's choice.  grid=P caps
// the persistent grid at P CTAs (clusters), i.e. the backward's partial rows.
struct Override {
  int C = 0, tpr = 0, rpg = 0, S = 0, G = 0, ctas = 0, lng = -1, K = 0, gsm = -1, grid = 0;
  int split = -1;  // 1: the two-pass path at any N; 0: never
  int W = 0;       // two-pass path: segment width (a multiple of 1024)
  int S1 = 0, S2 = 0;  // two-pass path: stages of its first / second pass
  int hint = -1;       // register-resident forward: suspend hint of its stage waits (ns)
  int stream = -1;     // backward: 1 the streaming long-row kernel where it applies, 0 never,
                       // -1 where it measured faster (stream_default)
  bool any = false;
};

Override read_override() {
  Override o;
  const char *s = std::getenv("GBNORM_PLAN");
  if (!s || !*s) return o;
  char buf[256];
  std::snprintf(buf, sizeof buf, "%s", s);
  // Fields separated by commas, walked with a local cursor (no hidden state:
  // several host threads may plan at once).
  for (char *tok = buf; tok && *tok;) {
    char *comma = std::strchr(tok, ',');
    if (comma) *comma = '\0';
    char *cur = tok;
    tok = comma ? comma + 1 : nullptr;
    char key[32];
    int val = 0;
    if (std::sscanf(cur, "%31[^=]=%d", key, &val) != 2) continue;
    if (!std::strcmp(key, "C")) o.C = val;
    else if (!std::strcmp(key, "tpr")) o.tpr = val;
    else if (!std::strcmp(key, "rpg")) o.rpg = val;
    else if (!std::strcmp(key, "S")) o.S = val;
    else if (!std::strcmp(key, "G")) o.G = val;
    else if (!std::strcmp(key, "ctas")) o.ctas = val;
    else if (!std::strcmp(key, "long")) o.lng = val;
    else if (!std::strcmp(key, "K")) o.K = val;
    else if (!std::strcmp(key, "gsm")) o.gsm = val;
    else if (!std::strcmp(key, "grid")) o.grid = val;
    else if (!std::strcmp(key, "split")) o.split = val;
    else if (!std::strcmp(key, "W")) o.W = val;
    else if (!std::strcmp(key, "S1")) o.S1 = val;
    else if (!std::strcmp(key, "S2")) o.S2 = val;
    else if (!std::strcmp(key, "stream")) o.stream = val;
    else if (!std::strcmp(key, "hint")) o.hint = val;
    o.any = true;
  }
  return o;
}

int round_k(int K, bool bwd) {
  if (bwd) return K;  // 1..4 all compiled
  return K == 7 ? 8 : K;
}

// Offline-tuned plans for row lengths measured on GB300 (a search over
// threads per row, rows per group and stages, keeping changes that beat the
// heuristic by more than ~5 %; then a search over the stage count alone,
// keeping gains above 1 %: fewer tiles in flight than fit -- 2 to 5 -- are
// often faster).  Like any plan they fix the reduction order, so results
// stay bitwise reproducible; shapes not listed use the heuristic.
struct TunedPlan {
  int mode;  // kRMS / kLayer
  int bwd;   // 0 forward, 1 backward
  int N;
  int tpr, rpg, S;  // 0 = heuristic's choice
  int gsm = 0;      // forward: gamma/beta staged in shared memory, 8 chunks per thread
  int lng = 0;      // 1: the long-row kernels (slice re-read from the stage)
  int G = 0;        // row groups per CTA (0 = heuristic's choice)
  int hint = 0;     // forward: suspend hint (ns) of the stage waits, 0 none
};
constexpr TunedPlan kTuned[] = {
    {kRMS, 0, 256, 32, 2, 2},     {kRMS, 0, 512, 32, 1, 2},    {kRMS, 0, 768, 32, 0, 3},
    {kRMS, 0, 1024, 64, 1, 0},    {kRMS, 0, 2048, 128, 1, 2},  {kRMS, 0, 3072, 192, 1, 3},
    {kRMS, 0, 5120, 160, 0, 3},   {kRMS, 0, 8192, 256, 0, 3},  {kRMS, 0, 16384, 512, 0, 4},
    {kRMS, 0, 32768, 0, 0, 2},
    // LayerNorm 4096 forward: its four 128-thread row groups per CTA wait
    // for stages with a 2 us suspend hint, so a waiting group leaves the
    // issue slots to the others (93.8 -> 96.0 % of measured; the same hint
    // cost most other plans 0.1-1.9 %, so they keep the default polls).
    {kLayer, 0, 2048, 64, 0, 5},  {kLayer, 0, 3072, 0, 0, 0, 1},
    {kLayer, 0, 4096, 0, 0, 4, 0, 0, 0, 2000},
    {kLayer, 0, 5120, 0, 0, 3, 1}, {kLayer, 0, 8192, 0, 0, 0, 1},
    {kRMS, 1, 256, 32, 2, 5},     {kRMS, 1, 512, 64, 0, 0},    {kRMS, 1, 768, 64, 4, 0},
    {kRMS, 1, 1024, 64, 1, 5},    {kRMS, 1, 2048, 128, 1, 5},  {kRMS, 1, 5120, 256, 2, 0},
    {kRMS, 1, 16384, 0, 0, 2},
    {kLayer, 1, 3072, 192, 4, 0},
    // LayerNorm backward at 5120 / 8192: the long-row kernel with 4 chunks
    // per thread and 3 / 2 row groups (15 / 16 warps) beats the register
    // kernel's 2 chunks per thread (10 / 16 warps, 8 / 16 warps per row):
    // 195 -> 173 us and 274 -> 265 us at 32768 rows; two stages instead of
    // three gain another 2-3 %.
    {kLayer, 1, 5120, 0, 0, 2, 0, 1, 3}, {kLayer, 1, 8192, 0, 0, 2, 0, 1, 2},
};

// Ring and tile sizing shared by both plan kinds: rows per tile and the
// number of stages that fit in shared memory (at least two).
norm_status_t size_ring(Plan &p, bool bwd, int smem_optin, const Override &ov, int64_t M,
                        int s_cap = 0) {
  // (the long-row fused residual backward reads dh into registers: not staged)
  const int ntensors = (bwd ? 2 : 1) + (p.resid && !(bwd && p.long_rows) ? 1 : 0);
  const int C = p.C;
  int G = p.G;
  const int row_bytes = p.NS * 2;
  int rpg = 1;
  if (C == 1) rpg = std::max(1, (32 * 1024) / (row_bytes * G));
  if (ov.rpg) rpg = ov.rpg;
  if (rpg < 1 || (C > 1 && rpg != 1)) return NORM_ERR_UNSUPPORTED;
  const int budget = smem_optin - 1024;
  int S = 0;
  for (;;) {
    const SmemLayout L1 = make_layout(G * rpg, p.NS, 1, G, p.tpr, ntensors, bwd, C, p.par_bpc);
    const SmemLayout L2 = make_layout(G * rpg, p.NS, 2, G, p.tpr, ntensors, bwd, C, p.par_bpc);
    const int per_stage = static_cast<int>(L2.total - L1.total);
    const int fixed = static_cast<int>(L1.total) - per_stage;
    S = (budget - fixed) / per_stage;
    if (S >= 2 || ov.rpg || ov.G || (rpg == 1 && G == 1)) break;
    if (rpg > 1) rpg = (rpg + 1) / 2;
    else G = (G + 1) / 2;
  }
  S = std::min(S, 8);
  if (s_cap) S = std::min(S, s_cap);
  if (ov.S) S = ov.S;
  if (S < 2) return NORM_ERR_UNSUPPORTED;
  p.G = G;
  p.rpg = rpg;
  p.RT = G * rpg;
  p.S = S;
  p.threads = G * p.tpr;
  if (p.threads % 32) return NORM_ERR_UNSUPPORTED;
  const SmemLayout L = make_layout(p.RT, p.NS, S, G, p.tpr, ntensors, bwd, C, p.par_bpc);
  if (static_cast<int64_t>(L.total) > budget) return NORM_ERR_UNSUPPORTED;
  if (L.stage_bytes >= (1u << 20)) return NORM_ERR_UNSUPPORTED;
  if (bwd && static_cast<int64_t>(2) * G * p.NS * 4 > static_cast<int64_t>(S) * L.stage_bytes)
    return NORM_ERR_UNSUPPORTED;
  p.smem = L.total;
  p.ntiles = (M + p.RT - 1) / p.RT;
  return NORM_OK;
}

// Plan for the long-row kernels: K chunks per thread (8 forward, 4
// backward), two row groups of up to 256 threads per CTA when the slice
// allows, and the smallest power-of-two cluster whose slices fit.
norm_status_t long_plan(int mode, bool bwd, int64_t M, int N, int smem_optin, const Override &ov,
                        Plan *out, bool resid = false, bool fp8 = false) {
  const int nc = N / 8;
  // 8 chunks per thread for the forward (RMSNorm without spilling;
  // LayerNorm with a few spilled registers when one CTA owns the row and
  // none in clusters, and still faster than 4: 60 -> 73 % of measured at
  // 32768 columns, 58 -> 86 % at 65536, 48 -> 83 % at 131072; with the fused
  // residual add 94 -> 96, 91 -> 98, 76 -> 83 %; with E4M3 output, of its
  // minimal bytes, MX 42 -> 44, 41 -> 60, 33 -> 58 %, per-row 34 -> 40,
  // 32 -> 33, 26 -> 32 %, the last two now 47 and 45 % with one exchange
  // round per row); 4 for the backward.
  const int K = ov.K ? ov.K : (!bwd ? 8 : 4);
  if (K != 2 && K != 4 && K != 8) return NORM_ERR_UNSUPPORTED;
  // Slices up to kMaxThreads threads x K chunks per CTA; clusters when the
  // row is wider, or when a stage of the CTA's slice (x, and dy and / or the
  // residual tensor) would not leave room for two stages.  Without a
  // cluster, up to two row groups per CTA overlap each other's reductions;
  // in a cluster one group of up to kMaxThreads threads per CTA, the
  // cross-CTA exchange being overlapped by the kernel's software pipeline.
  int C = 1;
  while (C < 16 && ceil_div(nc, C) > kMaxThreads * K) C <<= 1;
  if (ov.C) C = ov.C;
  for (;; C <<= 1) {
    if (C < 1 || C > 16) return NORM_ERR_UNSUPPORTED;
    Plan p;
    p.long_rows = true;
    p.resid = resid;
    p.C = C;
    // E4M3 output: slices start on a 32-column MX block (4 chunks)
    p.nsc = fp8 ? 4 * ceil_div(nc, 4 * C) : ceil_div(nc, C);
    p.NS = p.nsc * 8;
    if ((C - 1) * p.nsc >= nc) return NORM_ERR_UNSUPPORTED;
    const int tpr = ov.tpr ? ov.tpr : 32 * ceil_div(ceil_div(p.nsc, K), 32);
    if (tpr < 32 || tpr > kMaxThreads || tpr % 32) return NORM_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(tpr) * K < p.nsc) return NORM_ERR_UNSUPPORTED;
    p.tpr = tpr;
    p.K = K;
    p.exact = (nc % C == 0) && (tpr * K == p.nsc);
    p.G = ov.G ? ov.G : (C > 1 ? 1 : std::max(1, std::min(2, kMaxThreads / tpr)));
    if (p.G * tpr > kMaxThreads || p.G > 15) return NORM_ERR_UNSUPPORTED;
    if (C > 1 && p.G != 1) return NORM_ERR_UNSUPPORTED;  // one row per CTA per tile
    norm_status_t st = size_ring(p, bwd, smem_optin, ov, M);
    if (st != NORM_OK) {
      if (ov.C) return st;
      continue;  // a wider cluster halves the slice
    }
    if (fp8 ? !long_fp8_kernel_ptr(mode, p.K, p.C > 1, p.exact, resid, kOutFp8Mx)
            : !long_kernel_ptr(mode, p.K, p.C > 1, p.exact, bwd, resid))
      return NORM_ERR_UNSUPPORTED;
    *out = p;
    return NORM_OK;
  }
}

// Plans of the streaming long-row kernels (stream.cu): rows of C slices, a
// cluster of C CTAs per row (one CTA when C = 1), one row group of
// kStreamThreads threads per CTA, slices streamed as pieces of
// stream_piece_cols(kp) columns with as many pieces in flight as fit (up to
// kStreamMaxStages).  Pieces of 16384 columns (kp = 4), or of 8192 (kp =
// 2) for the fused residual backward, whose third tensor would leave only
// two 96 KB stages: from 8192- to 16384-column pieces (fewer waits and
// refills per byte) the RMSNorm backward at 131072 columns went from 85.9 to
// 93.0 % of measured, LayerNorm's from 74.0 to 83.0 % (its dx pass moves the
// dgamma / dbeta accumulators through registers in two batches of two
// chunks), the fused residual RMSNorm backward's from 98.8 down to 96.0 %.
// The override W= sets the piece width (8192 or 16384).
constexpr int kStreamMaxStages = 12;

int stream_kp(const Override &ov, bool resid) {
  if (ov.W == stream_piece_cols(2)) return 2;
  if (ov.W == stream_piece_cols(4)) return 4;
  return resid ? 2 : 4;
}

// The streaming forward's pieces: 16384 columns for RMSNorm, 8192 for
// LayerNorm (the instantiated variants).
int stream_fwd_kp(int mode, const Override &ov) {
  if (ov.W == stream_piece_cols(2)) return 2;
  if (ov.W == stream_piece_cols(4)) return 4;
  return mode == kRMS ? 4 : 2;
}

bool stream_applies(int N) { return N % kStreamSlice == 0 && N / kStreamSlice <= 16; }

// Row widths, in slices of kStreamSlice columns, where the streaming
// backward measured faster on GB300 (1024 to 4096 rows) than the resident
// long-row kernel or, beyond NORM_MAX_N_ONEPASS, the two-pass path, in % of
// the measured copy bandwidth: 1, 2, 4 and 8 slices (RMSNorm 87.2 -> 91.9,
// 86.9 -> 93.6, 74.3 -> 93.5, 66.1 -> 83.0; LayerNorm 75.0 -> 82.5,
// 72.7 -> 83.4, 61.7 -> 83.0, 53.0 -> 72.2: the resident kernel's clusters
// of 8 and 16 occupy only 120 and 112 SMs) and 16 (two-pass RMSNorm
// 58.4 -> 77.1, LayerNorm 57.8 -> 64.1).  Slice counts that are not powers
// of two keep the resident kernel (clusters of 3 measured ~40 %).  The fused residual
// backward (dh streamed once with the dx pass) takes it at the same widths
// (1, 2, 4 and 8 slices; the fused entry points stop at 262144 columns):
// RMSNorm 80.9 -> 95.9, 80.2 -> 98.5, 70.3 -> 98.6, 64.7 -> 86.3 %,
// LayerNorm 63.6 -> 90.6, 57.8 -> 90.1, 48.2 -> 88.8, 45.0 -> 74.0 %.
bool stream_default(int mode, int C) {
  (void)mode;
  return C == 1 || C == 2 || C == 4 || C == 8 || C == 16;
}

// Whether the backward of rows of N columns takes the streaming kernel:
// forced by the override stream=1, or by default where it measured faster
// (not under other override fields, which pin the plan they describe).
bool use_stream(int N, int mode, const Override &ov) {
  if (!stream_applies(N) || ov.stream == 0) return false;
  if (ov.stream == 1) return true;
  return !ov.any && stream_default(mode, N / kStreamSlice);
}

// The part of a streaming plan both passes share.
norm_status_t stream_common(int64_t M, int N, int slice, int kp, int ntensors, int smem_optin,
                            const Override &ov, Plan *out) {
  Plan p;
  p.stream = true;
  p.piece_kp = kp;
  p.C = N / slice;
  if (ov.C && ov.C != p.C) return NORM_ERR_UNSUPPORTED;
  p.NS = slice;
  p.nsc = slice / 8;
  p.tpr = kStreamThreads;
  p.K = p.nsc / kStreamThreads;
  p.exact = true;
  p.G = 1;
  p.rpg = 1;
  p.RT = 1;
  p.threads = kStreamThreads;
  const int64_t budget = smem_optin - 1024;
  auto bytes = [&](int S) {
    return static_cast<int64_t>(stream_layout(S, p.C, ntensors, kp).total);
  };
  int S = ov.S ? ov.S : kStreamMaxStages;
  while (!ov.S && S > 2 && bytes(S) > budget) --S;
  if (S < 2 || bytes(S) > budget) return NORM_ERR_UNSUPPORTED;
  p.S = S;
  p.smem = stream_layout(S, p.C, ntensors, kp).total;
  p.ntiles = M;
  *out = p;
  return NORM_OK;
}

norm_status_t stream_plan(int64_t M, int N, int mode, int smem_optin, const Override &ov,
                          Plan *out, bool resid = false) {
  if (!stream_applies(N)) return NORM_ERR_UNSUPPORTED;
  const int kp = stream_kp(ov, resid);
  if (!stream_kernel_ptr(mode, kp, N > kStreamSlice, resid)) return NORM_ERR_UNSUPPORTED;
  const norm_status_t st =
      stream_common(M, N, kStreamSlice, kp, resid ? 3 : 2, smem_optin, ov, out);
  if (st == NORM_OK) out->resid = resid;
  return st;
}

// The streaming forward: by default for RMSNorm rows wider than
// NORM_MAX_N_ONEPASS, in place of the two-pass path (which reads x twice
// from HBM), with 65536-column slices where at most 16 make a row, else
// 32768 (RMSNorm 4096 x 524288: two-pass 63.3 %, 32768-column slices in
// clusters of 16 72.1 %, 65536-column slices in clusters of 8 78.2 %;
// 1024 x 1048576: 63.4 -> 70.3 %).  The LayerNorm forward keeps the
// two-pass path there (42.6 against 60.4 % at 2048 x 524288).  Forced by
// stream=1 at any width it takes (K=8: 32768-column slices, K=16: 65536).
int stream_fwd_np(int N, int mode, const Override &ov) {
  if (ov.stream == 0) return 0;
  const bool forced = ov.stream == 1;
  if (!forced && (ov.any || N <= NORM_MAX_N_ONEPASS || mode != kRMS)) return 0;
  const int kp = stream_fwd_kp(mode, ov);
  auto fits = [&](int np) {
    const int slice = np * stream_piece_cols(kp);
    const int C = N / slice;
    return np >= 1 && N % slice == 0 && C >= 1 && C <= 16 && (forced || (C & (C - 1)) == 0) &&
           stream_fwd_kernel_ptr(mode, kp, np, C > 1) != nullptr;
  };
  const int np1 = kStreamSlice / stream_piece_cols(kp);  // 32768-column slices
  if (ov.K == 8) return fits(np1) ? np1 : 0;
  if (ov.K == 16) return fits(2 * np1) ? 2 * np1 : 0;
  if (!forced && fits(2 * np1)) return 2 * np1;
  if (fits(np1)) return np1;
  return fits(2 * np1) ? 2 * np1 : 0;
}

norm_status_t stream_fwd_plan(int64_t M, int N, int mode, int np, int smem_optin,
                              const Override &ov, Plan *out) {
  const int kp = stream_fwd_kp(mode, ov);
  return stream_common(M, N, np * stream_piece_cols(kp), kp, 1, smem_optin, ov, out);
}

// Shape part of the plan for one pass: everything except the grid size.
// Pure host arithmetic (no CUDA call).  `bwd` selects the backward kernel
// (two tensors per stage, at most kMaxKBwd chunks per thread).
norm_status_t shape_plan(int mode, bool bwd, int64_t M, int N, int smem_optin,
                         const Override &ov_in, Plan *out, bool resid = false,
                         bool fp8 = false) {
  Override ov = ov_in;
  bool tuned_gsm = false;
  if (!ov.any && !resid && !fp8) {
    for (const TunedPlan &tp : kTuned) {
      if (tp.mode == mode && tp.bwd == (bwd ? 1 : 0) && tp.N == N) {
        ov.tpr = tp.tpr;
        ov.rpg = tp.rpg;
        ov.S = tp.S;
        ov.G = tp.G;
        if (tp.lng) ov.lng = 1;
        if (tp.hint) ov.hint = tp.hint;
        tuned_gsm = tp.gsm != 0;
        break;
      }
    }
  }
  if (bwd && !fp8 && use_stream(N, mode, ov))
    return stream_plan(M, N, mode, smem_optin, ov, out, resid);
  if (!bwd && !resid && !fp8) {
    const int np = stream_fwd_np(N, mode, ov);
    if (np) return stream_fwd_plan(M, N, mode, np, smem_optin, ov, out);
  }
  const int kmax = bwd ? kMaxKBwd : kMaxKFwd;
  const int nc = N / 8;
  Plan p;
  p.resid = resid;

  // Preferred chunks per thread, and the most that still fit in registers
  // without spilling (ptxas -v: forward LayerNorm 4, RMSNorm 6; backward
  // LayerNorm 2, RMSNorm 3); up to kmax only when a row needs it.
  const int kpref = bwd ? 2 : 4;
  const int klim = bwd ? (mode == kLayer ? 2 : 3) : (mode == kLayer ? 4 : 6);

  // Rows wider than one CTA's register capacity (kMaxThreads x klim chunks)
  // go to the long-row kernels, which keep the row in shared memory.
  if (ov.lng == 1 || (ov.lng != 0 && nc > kMaxThreads * klim)) {
    return long_plan(mode, bwd, M, N, smem_optin, ov, out, resid, fp8 && !bwd);
  }

  // Column split: the smallest power-of-two cluster (up to 8) whose per-CTA
  // slice fits kMaxThreads threads x kpref chunks, else the smallest (up to
  // 16) that fits klim, else kmax chunks.  Slices are ceil(nc / C) chunks;
  // the last CTA of a cluster takes the remainder.
  // (The fused residual add has no register-resident cluster variants: it
  // keeps C = 1 up to klim chunks per thread; wider rows took the long-row
  // path above.)
  int C = 1;
  if (!resid) {
    while (C < 8 && ceil_div(nc, C) > kMaxThreads * kpref) C <<= 1;
    while (C < 16 && ceil_div(nc, C) > kMaxThreads * klim) C <<= 1;
    while (C <= 16 && ceil_div(nc, C) > kMaxThreads * kmax) C <<= 1;
  }
  if (ov.C) C = ov.C;
  if (C < 1 || C > 16 || (resid && C != 1)) return NORM_ERR_UNSUPPORTED;
  p.C = C;
  p.nsc = ceil_div(nc, C);
  p.NS = p.nsc * 8;
  if ((C - 1) * p.nsc >= nc) return NORM_ERR_UNSUPPORTED;  // a CTA would own nothing

  // Threads per row.  Preferred: an exact split of the slice into K chunks
  // per thread over tpr = nsc / K threads, tpr a multiple of 32 (the EXACT
  // kernels, which test no chunk ownership), with the largest K <= kpref,
  // else the smallest K <= kmax.  Otherwise power-of-two groups with a
  // ragged last chunk column.
  const bool even = (nc % C) == 0;
  int tpr = 0, K = 0;
  bool exact = false;
  auto try_exact = [&](int k, bool gsm) {
    if (!even || p.nsc % k || (p.nsc / k) % 32 || p.nsc / k > kMaxThreads) return false;
    if (!(bwd ? bwd_kernel_ptr(mode, k, C > 1, true, resid)
              : fwd_kernel_ptr(mode, k, C > 1, true, resid, gsm)))
      return false;
    tpr = p.nsc / k;
    K = k;
    exact = true;
    return true;
  };
  // Forward with gamma/beta in shared memory, 8 chunks per thread, exact
  // split: forced by the override, or preferred for E4M3 output (whose
  // per-row amax costs a reduction round that fewer, fuller warps per row
  // amortise) and for tuned shapes; otherwise the register-resident plan.
  bool want_gsm = !bwd && (ov.gsm == 1 || (ov.gsm == -1 && !ov.tpr && (fp8 || tuned_gsm)));
  if (want_gsm && !ov.tpr) {
    bool found = false;
    for (int k : {8, 6, 5}) {
      if (!found) found = try_exact(k, true);
    }
    if (!found) {
      if (ov.gsm == 1) return NORM_ERR_UNSUPPORTED;
      want_gsm = false;
    }
  }
  if (want_gsm && !ov.tpr) {
    // K and tpr set by try_exact
  } else if (ov.tpr) {
    tpr = ov.tpr;
    K = round_k(ceil_div(p.nsc, tpr), bwd);
    exact = even && tpr % 32 == 0 && K * tpr == p.nsc;
  } else {
    bool found = false;
    // E4M3 output of short rows: the per-row amax and scale cost the same
    // per row whatever the row length, so give each thread as many chunks as
    // registers allow and let sub-warp groups (down to 4 threads, the MX
    // block width in chunks) cover the row (RMSNorm 256: 54 -> 85 % of
    // measured, 768: 88 -> 93 %).
    if (fp8 && !bwd && C == 1) {
      for (int k = klim; k >= 1 && !found; --k) {
        if (p.nsc % k) continue;
        const int t = p.nsc / k;
        if (t < 4 || t >= 32 || 32 % t) continue;
        if (!fwd_fp8_kernel_ptr(mode, k, false, resid, kOutFp8Row)) continue;
        tpr = t;
        K = k;
        found = true;
      }
    }
    for (int k = kpref; k >= 1 && !found; --k) found = try_exact(k, false);
    for (int k = kpref + 1; k <= klim && !found; ++k) found = try_exact(k, false);
    if (!found) {
      if (p.nsc <= 32) tpr = pow2ceil(p.nsc);
      else tpr = std::min(kMaxThreads, std::max(32, pow2ceil(ceil_div(p.nsc, kpref))));
      K = round_k(ceil_div(p.nsc, tpr), bwd);
    }
  }
  if (tpr < 1 || tpr > kMaxThreads || (tpr > 32 && tpr % 32) || (tpr < 32 && 32 % tpr))
    return NORM_ERR_UNSUPPORTED;
  if (K > kmax) return NORM_ERR_UNSUPPORTED;
  p.tpr = tpr;
  p.K = K;
  p.exact = exact;
  if (want_gsm) {
    if (!exact || (K != 8 && K != 6 && K != 5) || C != 1) return NORM_ERR_UNSUPPORTED;
    p.gsm = true;
    p.par_bpc = param_bytes_per_col(mode, fp8);
  }

  int G = kMaxThreads / tpr;
  if (tpr > 32) G = std::min(G, 8);
  if (ov.G) G = ov.G;
  if (G < 1 || G * tpr > kMaxThreads || (tpr > 32 && G > 15))
    return NORM_ERR_UNSUPPORTED;

  p.G = G;
  // Fewer tiles in flight than fit, measured per variant on every workload
  // width: two for the fused residual add (two or three tensors per stage;
  // 3-8 % faster than three or four), at most four for the E4M3 output of
  // sub-warp rows and three with staged parameters (2-4 %).
  const int s_cap = resid ? 2 : (fp8 ? (p.gsm ? 3 : 4) : 0);
  norm_status_t st = size_ring(p, bwd, smem_optin, ov, M, s_cap);
  if (st != NORM_OK) return st;
  if (!bwd && ov.hint > 0 && fwd_kernel_ptr(mode, p.K, p.C > 1, p.exact, resid, p.gsm, true))
    p.wait_ns = std::min(ov.hint, 1000000);
  *out = p;
  return NORM_OK;
}

const void *kernel_for(const Plan &p, int mode, bool bwd) {
  if (p.split) return split_kernel_ptr(mode, p.phase, p.K);
  if (p.stream)
    return bwd ? stream_kernel_ptr(mode, p.piece_kp, p.C > 1, p.resid)
               : stream_fwd_kernel_ptr(mode, p.piece_kp, p.NS / stream_piece_cols(p.piece_kp),
                                       p.C > 1);
  if (p.long_rows) return long_kernel_ptr(mode, p.K, p.C > 1, p.exact, bwd, p.resid);
  return bwd ? bwd_kernel_ptr(mode, p.K, p.C > 1, p.exact, p.resid)
             : fwd_kernel_ptr(mode, p.K, p.C > 1, p.exact, p.resid, p.gsm, p.wait_ns > 0);
}

void set_grid(Plan &p, int64_t resident_clusters) {
  const int64_t clusters = std::min<int64_t>(resident_clusters, p.ntiles);
  p.P = static_cast<int>(clusters);
  p.grid = static_cast<int>(clusters * p.C);
}

norm_status_t finish_plan(const DeviceInfo &d, int dev, int mode, bool bwd, const Override &ov,
                          Plan *pp);

// Full plan on the current device: shape part plus the occupancy-derived
// grid (persistent: as many CTAs or clusters as can be resident at once).
// `no_stream`: a backward plan without the streaming kernel (the resident
// long-row kernel or the two-pass path instead; fewer partial rows).
norm_status_t make_plan(const DeviceInfo &d, int dev, int mode, bool bwd, int64_t M, int N,
                        Plan *out, bool resid = false, bool fp8 = false,
                        bool no_stream = false) {
  Override ov = read_override();
  if (no_stream) ov.stream = 0;
  const auto key = std::make_tuple(dev, mode * 2 + (bwd ? 1 : 0), M, N,
                                   (resid ? 1 : 0) | (fp8 ? 2 : 0) | (no_stream ? 4 : 0));
  if (!ov.any) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      *out = it->second;
      return NORM_OK;
    }
  }
  Plan p;
  norm_status_t st = shape_plan(mode, bwd, M, N, d.smem_optin, ov, &p, resid, fp8);
  if (st != NORM_OK) return st;
  st = finish_plan(d, dev, mode, bwd, ov, &p);
  if (st != NORM_OK) return st;

  if (!ov.any) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_plans[key] = p;
  }
  *out = p;
  return NORM_OK;
}

// The device-dependent part of a plan: kernel attributes and the persistent
// grid from the occupancy of the chosen kernel.
norm_status_t finish_plan(const DeviceInfo &d, int dev, int mode, bool bwd, const Override &ov,
                          Plan *pp) {
  Plan &p = *pp;
  norm_status_t st;
  const void *fn = kernel_for(p, mode, bwd);
  if (!fn) return NORM_ERR_UNSUPPORTED;
  st = prepare_function(dev, fn, d.smem_optin);
  if (st != NORM_OK) return st;

  int64_t resident = 0;
  if (p.C == 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, p.threads, p.smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return NORM_ERR_CUDA;
    }
    if (ov.ctas) per_sm = std::min(per_sm, ov.ctas);
    resident = static_cast<int64_t>(per_sm) * d.sms;
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = p.C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(p.C * 64);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, fn, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return NORM_ERR_CUDA;
    }
    resident = nclusters;
  }
  if (ov.grid > 0) resident = std::min<int64_t>(resident, ov.grid);
  if (resident < 1) return NORM_ERR_UNSUPPORTED;
  set_grid(p, resident);
  return NORM_OK;
}

// ------------------------------------------------------ two-pass path
// Rows wider than NORM_MAX_N_ONEPASS (or any row, with the plan override
// split=1) are cut into segments of kSplitW columns (override W=); see
// split.cu.  Each pass has its own plan: rows of RT = G * rpg per unit, S
// units in flight, and a persistent grid of at most one CTA per unit.
constexpr int kSplitW = 4096;

// (rows the streaming kernels take do not: the backward's, and the
// forward's beyond NORM_MAX_N_ONEPASS)
bool use_split(int N, const Override &ov, int mode, bool bwd) {
  if (bwd ? use_stream(N, mode, ov) : stream_fwd_np(N, mode, ov) != 0) return false;
  return ov.split == 1 || (ov.split != 0 && N > NORM_MAX_N_ONEPASS);
}

// Shape part of a pass's plan (no CUDA call): threads per row and chunks per
// thread from the segment width (K = 4, or 2 for the dx pass, which holds
// the column sums), G row groups of up to 512 threads, and the stages that
// fit in `smem_optin` bytes.
norm_status_t split_shape(int mode, int phase, int64_t M, int N, int smem_optin,
                          const Override &ov, Plan *out) {
  const int W = ov.W ? ov.W : kSplitW;
  const int K = phase == kSplitBwdDx ? 2 : 4;
  const int nc = W / 8;
  if (W < 1024 || W % 1024 || nc % K) return NORM_ERR_UNSUPPORTED;
  const int tpr = nc / K;
  if (tpr < 32 || tpr > kMaxThreads || tpr % 32) return NORM_ERR_UNSUPPORTED;
  if (!split_kernel_ptr(mode, phase, K)) return NORM_ERR_UNSUPPORTED;
  Plan p;
  p.split = true;
  p.phase = phase;
  p.C = 1;
  p.NS = W;
  p.nsc = nc;
  p.tpr = tpr;
  p.K = K;
  p.exact = false;
  p.nseg = (N + W - 1) / W;
  int G = kMaxThreads / tpr;
  if (tpr > 32) G = std::min(G, 8);
  if (ov.G) G = ov.G;
  if (G < 1 || G * tpr > kMaxThreads || (tpr > 32 && G > 15)) return NORM_ERR_UNSUPPORTED;
  const int nt = phase >= kSplitBwdDots ? 2 : 1;
  int rpg = ov.rpg ? ov.rpg : std::max(1, 4 / G);
  const int budget = smem_optin - 1024;
  int S = 0;
  for (;;) {
    const SmemLayout L1 = split_smem_layout(G * rpg, W, 1, G, tpr, nt);
    const SmemLayout L2 = split_smem_layout(G * rpg, W, 2, G, tpr, nt);
    const int per_stage = static_cast<int>(L2.total - L1.total);
    const int fixed = static_cast<int>(L1.total) - per_stage;
    S = (budget - fixed) / per_stage;
    if (S >= 2 || rpg == 1 || ov.rpg) break;
    rpg = (rpg + 1) / 2;
  }
  // units in flight: three (two for the dx pass, whose units hold x and dy
  // and write dx), measured the fastest of 2 to 8 per pass
  S = std::min(S, phase == kSplitBwdDx ? 2 : 3);
  const bool first = phase == kSplitFwdStats || phase == kSplitBwdDots;
  if (ov.S) S = ov.S;
  if (first && ov.S1) S = ov.S1;
  if (!first && ov.S2) S = ov.S2;
  if (S < 2) return NORM_ERR_UNSUPPORTED;
  const SmemLayout L = split_smem_layout(G * rpg, W, S, G, tpr, nt);
  if (static_cast<int64_t>(L.total) > budget) return NORM_ERR_UNSUPPORTED;
  p.G = G;
  p.rpg = rpg;
  p.RT = G * rpg;
  p.S = S;
  p.threads = G * tpr;
  if (p.threads % 32) return NORM_ERR_UNSUPPORTED;
  p.smem = L.total;
  p.ntiles = (M + p.RT - 1) / p.RT;
  *out = p;
  return NORM_OK;
}

// Units of a pass: row tiles x segments.  The grid never exceeds them, so
// every CTA owns at least one unit (the dgamma/dbeta reduction relies on it).
void split_grid(Plan &p, int64_t resident) {
  const int64_t units = p.ntiles * p.nseg;
  p.grid = static_cast<int>(std::min<int64_t>(resident, units));
  p.P = p.grid;
}

// Plans of the two passes of the two-pass path: [0] statistics (forward) or
// dot products (backward), [1] output or dx.  Cached like the one-pass plans.
norm_status_t make_split_plans(const DeviceInfo &d, int dev, int mode, bool bwd, int64_t M,
                               int N, Plan out[2]) {
  const Override ov = read_override();
  for (int i = 0; i < 2; ++i) {
    const int phase = (bwd ? kSplitBwdDots : kSplitFwdStats) + i;
    const auto key = std::make_tuple(dev, mode * 2 + (bwd ? 1 : 0), M, N, 8 + phase);
    if (!ov.any) {
      std::lock_guard<std::mutex> lk(g_mu);
      auto it = g_plans.find(key);
      if (it != g_plans.end()) {
        out[i] = it->second;
        continue;
      }
    }
    Plan p;
    norm_status_t st = split_shape(mode, phase, M, N, d.smem_optin, ov, &p);
    if (st != NORM_OK) return st;
    const void *fn = split_kernel_ptr(mode, phase, p.K);
    if ((st = prepare_function(dev, fn, d.smem_optin)) != NORM_OK) return st;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, p.threads, p.smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return NORM_ERR_CUDA;
    }
    if (ov.ctas) per_sm = std::min(per_sm, ov.ctas);
    int64_t resident = static_cast<int64_t>(per_sm) * d.sms;
    if (ov.grid > 0) resident = std::min<int64_t>(resident, ov.grid);
    if (resident < 1) return NORM_ERR_UNSUPPORTED;
    split_grid(p, resident);
    if (!ov.any) {
      std::lock_guard<std::mutex> lk(g_mu);
      g_plans[key] = p;
    }
    out[i] = p;
  }
  return NORM_OK;
}

// Workspace of the two-pass backward: the dgamma (and dbeta) slots, one
// segment wide, for every (CTA, segment) pair of the dx pass (CTA b's slot
// of segment s is b + s, since a CTA's units cover consecutive segments),
// then the per-(row, segment) dot products and the per-row totals.
struct SplitWs {
  size_t slots = 0, rowp = 0, rowt = 0, total = 0;
};
SplitWs split_ws(const Plan &dx, int64_t M, int mode) {
  SplitWs w;
  const size_t k = mode == kLayer ? 2 : 1;
  const size_t nslots = static_cast<size_t>(dx.grid) + static_cast<size_t>(dx.nseg);
  w.slots = 0;
  w.rowp = k * nslots * static_cast<size_t>(dx.NS) * sizeof(float);
  w.rowt = w.rowp + ((static_cast<size_t>(M) * dx.nseg * 2 * sizeof(float) + 15) & ~size_t(15));
  w.total = w.rowt + ((static_cast<size_t>(M) * 2 * sizeof(float) + 15) & ~size_t(15));
  return w;
}

norm_status_t launch(const void *fn, const Plan &p, const NormArgs &args, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  // Every kernel waits (griddepcontrol.wait) before its first global access,
  // so it may be launched while the previous kernel of the stream drains.
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (p.C > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p.C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  NormArgs a = args;
  void *kargs[] = {&a};
  if (cudaLaunchKernelExC(&cfg, fn, kargs) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  return NORM_OK;
}

// The fixed-order reduction of the backward partials into dgamma (and dbeta
// when given), on `s` after the row kernel.
norm_status_t launch_reduce(const float *ws, int P, int n, float *dgamma, float *dbeta,
                            cudaStream_t s) {
  const int nparts = dbeta ? 2 : 1;
  void *rargs[] = {&ws, &P, &n, &dgamma, &dbeta};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + 127) / 128, nparts);
  cfg.blockDim = dim3(reduce_threads());
  cfg.stream = s;
  cudaLaunchAttribute rattr;
  rattr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  rattr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &rattr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelExC(&cfg, reduce_kernel_ptr(), rargs) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  return NORM_OK;
}

// A launch with programmatic stream serialisation allowed (the kernel waits
// for its predecessor before touching global memory).
norm_status_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  return NORM_OK;
}

// The per-row fold of the two-pass path: one warp per row, 8 rows per block.
norm_status_t launch_fold(int mode, bool bwd, const NormArgs &args, cudaStream_t s) {
  NormArgs a = args;
  void *kargs[] = {&a};
  const int64_t blocks = (a.M + 7) / 8;
  if (blocks > 0x7fffffff) return NORM_ERR_SHAPE;
  return launch_pdl(split_fold_kernel_ptr(mode, bwd), dim3(static_cast<unsigned>(blocks)),
                    dim3(256), kargs, s);
}

// dgamma (and dbeta) from the two-pass dx pass's slots.
norm_status_t launch_split_reduce(const NormArgs &args, int grid, float *dgamma, float *dbeta,
                                  cudaStream_t s) {
  NormArgs a = args;
  void *kargs[] = {&a, &grid, &dgamma, &dbeta};
  const int64_t threads = (static_cast<int64_t>(a.N) + 3) / 4;
  return launch_pdl(split_reduce_kernel_ptr(),
                    dim3(static_cast<unsigned>((threads + 255) / 256), dbeta ? 2 : 1), dim3(256),
                    kargs, s);
}

norm_status_t check_common(int64_t M, int64_t N, norm_mode_t mode,
                           int64_t max_n = NORM_MAX_N) {
  if (mode != NORM_RMS && mode != NORM_LAYER) return NORM_ERR_MODE;
  if (M < 1 || N < 8 || N > max_n || (N % 8) != 0) return NORM_ERR_SHAPE;
  if (M > (int64_t(1) << 40)) return NORM_ERR_SHAPE;
  return NORM_OK;
}

NormArgs base_args(const Plan &p, int64_t M, int N) {
  NormArgs a;
  std::memset(&a, 0, sizeof a);
  a.M = M;
  a.N = N;
  a.NS = p.NS;
  a.nsc = p.nsc;
  a.tpr = p.tpr;
  a.G = p.G;
  a.rpg = p.rpg;
  a.RT = p.RT;
  a.S = p.S;
  a.P = p.P;
  a.C = p.C;
  a.ntiles = p.ntiles;
  a.nseg = p.nseg;
  a.invN = 1.0f / static_cast<float>(N);
  a.wait_ns = static_cast<unsigned>(p.wait_ns);
  return a;
}

void fill_plan(const Plan &p, norm_plan_t *out) {
  out->cluster = p.C;
  out->cols_per_cta = p.NS;
  out->threads_per_row = p.tpr;
  out->chunks_per_thread = p.K;
  out->groups = p.G;
  out->rows_per_group = p.rpg;
  out->rows_per_tile = p.RT;
  out->stages = p.S;
  out->threads = p.threads;
  out->smem_bytes = static_cast<int32_t>(p.smem);
  out->tiles = p.ntiles;
  out->grid = p.grid;
  out->partials = p.P;
  out->exact = p.exact ? 1 : 0;
  out->long_rows = p.long_rows ? 1 : 0;
  out->param_smem_bytes = p.par_bpc * p.NS;
  out->split_segments = p.split ? p.nseg : 0;
  out->streamed = p.stream ? 1 : 0;
  out->piece_cols = p.stream ? stream_piece_cols(p.piece_kp) : 0;
  out->wait_hint_ns = p.wait_ns;
}

// ------------------------------------------------------------ plan tuning
// The pages name the split size and the number of pipeline stages as the
// levers an autotuner turns for these kernels; here the candidates are the
// single-CTA plans of one pass: every threads-per-row value that splits the
// row (exactly, or raggedly over a power of two) within the compiled chunk
// counts, rows per group 1, 2, 4 or the heuristic's, the long-row kernels
// with 1 to 8 row groups, and for the forward pass the staged-parameter
// plans.  Rows that need a cluster keep their plan.
std::vector<Override> tune_candidates(bool bwd, int N) {
  std::vector<Override> v;
  const int nsc = N / 8;
  const int kmax = bwd ? kMaxKBwd : kMaxKFwd;
  std::vector<int> tprs;
  for (int k = 1; k <= kmax; ++k) {
    if (nsc % k) continue;
    const int t = nsc / k;
    if ((t <= 32 && 32 % t == 0) || (t % 32 == 0 && t <= kMaxThreads)) tprs.push_back(t);
  }
  for (int t = 1; t <= kMaxThreads; t *= 2)
    if (ceil_div(nsc, t) <= kmax && t <= pow2ceil(nsc)) tprs.push_back(t);
  std::sort(tprs.begin(), tprs.end());
  tprs.erase(std::unique(tprs.begin(), tprs.end()), tprs.end());
  for (int t : tprs) {
    for (int rpg : {0, 1, 2, 4}) {
      Override o;
      o.any = true;
      o.tpr = t;
      o.rpg = rpg;
      o.gsm = 0;
      o.lng = 0;
      o.C = 1;
      v.push_back(o);
    }
  }
  // the long-row kernels at this width (slice re-read from the stage):
  // 1 to 8 row groups per CTA
  for (int G = 1; G <= 8; ++G) {
    Override o;
    o.any = true;
    o.lng = 1;
    o.C = 1;
    o.G = G;
    v.push_back(o);
  }
  if (!bwd) {
    for (int k : {5, 6, 8}) {
      if (nsc % k || (nsc / k) % 32 || nsc / k > kMaxThreads) continue;
      for (int rpg : {0, 1, 2}) {
        Override o;
        o.any = true;
        o.tpr = nsc / k;
        o.rpg = rpg;
        o.gsm = 1;
        o.lng = 0;
        o.C = 1;
        v.push_back(o);
      }
    }
  }
  return v;
}

bool same_plan(const Plan &a, const Plan &b) {
  return a.C == b.C && a.tpr == b.tpr && a.K == b.K && a.G == b.G && a.rpg == b.rpg &&
         a.S == b.S && a.gsm == b.gsm && a.long_rows == b.long_rows && a.grid == b.grid &&
         a.stream == b.stream && a.piece_kp == b.piece_kp && a.wait_ns == b.wait_ns;
}

// Times `run` (one launch of the pass with the plan installed in the cache
// under `key`) for every candidate and leaves the fastest installed.
template <typename Run>
norm_status_t tune_pass(int mode, bool bwd, int64_t M, int N, size_t ws_bytes, int iters,
                        cudaStream_t stream, Run run, norm_plan_t *chosen) {
  if (iters < 1 || iters > 100000) return NORM_ERR_ARG;
  if (read_override().any) return NORM_ERR_ARG;  // a plan override bypasses the cache
  norm_status_t st = run();                      // validates, caches the default plan
  if (st != NORM_OK) return st;
  if (use_split(N, Override(), mode, bwd)) {  // the two-pass path keeps its plan
    if (chosen) {
      norm_plan_t pl;
      if ((st = norm_plan(M, N, static_cast<norm_mode_t>(mode), bwd ? 1 : 0, 0, 0, &pl)) !=
          NORM_OK)
        return st;
      *chosen = pl;
    }
    return NORM_OK;
  }
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  Plan def;
  if ((st = make_plan(d, dev, mode, bwd, M, N, &def)) != NORM_OK) return st;
  const auto key = std::make_tuple(dev, mode * 2 + (bwd ? 1 : 0), M, N, 0);
  auto install = [&](const Plan &p) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_plans[key] = p;
  };
  std::vector<Plan> cands{def};
  if (def.C == 1) {
    for (const Override &o : tune_candidates(bwd, N)) {
      Plan p;
      if (shape_plan(mode, bwd, M, N, d.smem_optin, o, &p) != NORM_OK) continue;
      if (p.C != 1) continue;
      if (finish_plan(d, dev, mode, bwd, o, &p) != NORM_OK) continue;
      const size_t need = static_cast<size_t>(p.P) * N * 4 * (mode == kLayer ? 2 : 1);
      if (bwd && need > ws_bytes) continue;
      bool dup = false;
      for (const Plan &q : cands) dup = dup || same_plan(p, q);
      if (!dup) cands.push_back(p);
    }
  }
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  float best_ms = 0.f;
  int best = -1;
  for (size_t i = 0; i < cands.size(); ++i) {
    install(cands[i]);
    bool ok = run() == NORM_OK && run() == NORM_OK;  // warm-up
    ok = ok && cudaEventRecord(e0, stream) == cudaSuccess;
    for (int it = 0; it < iters && ok; ++it) ok = run() == NORM_OK;
    ok = ok && cudaEventRecord(e1, stream) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess;
    float ms = 0.f;
    ok = ok && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      continue;
    }
    if (best < 0 || ms < best_ms) {
      best_ms = ms;
      best = static_cast<int>(i);
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  install(cands[best < 0 ? 0 : best]);
  if ((st = run()) != NORM_OK) return st;  // outputs of the chosen plan
  if (chosen) fill_plan(cands[best < 0 ? 0 : best], chosen);
  return best < 0 ? NORM_ERR_CUDA : NORM_OK;
}

}  // namespace

// Fixed-order column sum of P fp32 rows [P][n] (and, with dbeta, of the P
// rows that follow them) into dgamma (dbeta), on `s`.
norm_status_t reduce_rows(const float *rows, int P, int n, float *dgamma, float *dbeta,
                          cudaStream_t s) {
  return launch_reduce(rows, P, n, dgamma, dbeta, s);
}

// Ordinal, SM count, opt-in shared memory per block, device error word and
// context identity (0 if unknown) of the current device (cached per device
// and context).
norm_status_t device_context(int *dev, int *sms, int *smem_optin, unsigned **err,
                             unsigned long long *ctx) {
  DeviceInfo d;
  int dv = 0;
  norm_status_t st = device_info(&d, &dv);
  if (st != NORM_OK) return st;
  *dev = dv;
  *sms = d.sms;
  *smem_optin = d.smem_optin;
  *err = d.err;
  if (ctx) *ctx = d.ctx;
  return NORM_OK;
}

}  // namespace gbn

// ---------------------------------------------------------------------------
// Allocation-free backward: the scratch lives in a fixed device array of this
// file.  Host code cannot use the array's name as a device address (on the
// host it names a stand-in), so the address is looked up once per device
// with cudaGetSymbolAddress, that device current, and cached (until the
// device's context is destroyed: see device_info).
static __device__ __align__(256) unsigned char g_noalloc_workspace[NORM_NOALLOC_WORKSPACE_BYTES];

using namespace gbn;

extern "C" {

norm_status_t norm_fwd(const void *x, const void *gamma, const void *beta, int64_t M,
                       int64_t N, float eps, norm_mode_t mode, void *y, float *rstd,
                       float *mean, norm_stream_t stream) {
  if (!x || !gamma || !y || !rstd) return NORM_ERR_NULL;
  norm_status_t st = check_common(M, N, mode);
  if (st != NORM_OK) return st;
  if (mode == NORM_RMS && (beta || mean)) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && !mean) return NORM_ERR_MODE;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return NORM_ERR_ARG;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(y) || !aligned16(rstd) ||
      (beta && !aligned16(beta)) || (mean && !aligned16(mean)))
    return NORM_ERR_ALIGN;
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  const bool split = use_split(static_cast<int>(N), read_override(), mode, false);
  Plan sp[2];
  Plan &p = sp[0];
  if (split) {
    if ((st = make_split_plans(d, dev, mode, false, M, static_cast<int>(N), sp)) != NORM_OK)
      return st;
  } else if ((st = make_plan(d, dev, mode, false, M, static_cast<int>(N), &p)) != NORM_OK) {
    return st;
  }
  NormArgs a = base_args(p, M, static_cast<int>(N));
  a.x = static_cast<const uint16_t *>(x);
  a.gamma = static_cast<const uint16_t *>(gamma);
  a.beta = static_cast<const uint16_t *>(beta);
  a.out = static_cast<uint16_t *>(y);
  a.rstd = rstd;
  a.mean = mean;
  a.err = d.err;
  a.eps = eps;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!split) return launch(kernel_for(p, mode, false), p, a, s);
  // statistics into y, their fold into rstd / mean, then y
  if ((st = launch(kernel_for(sp[0], mode, false), sp[0], a, s)) != NORM_OK) return st;
  if ((st = launch_fold(mode, false, a, s)) != NORM_OK) return st;
  NormArgs b = base_args(sp[1], M, static_cast<int>(N));
  b.x = a.x;
  b.gamma = a.gamma;
  b.beta = a.beta;
  b.out = a.out;
  b.rstd = rstd;
  b.mean = mean;
  b.err = d.err;
  b.eps = eps;
  return launch(kernel_for(sp[1], mode, false), sp[1], b, s);
}

// Workspace of the backward's plan (`no_stream`: the plan without the
// streaming kernel).
static norm_status_t bwd_workspace(int64_t M, int64_t N, norm_mode_t mode, bool no_stream,
                                   size_t *bytes) {
  if (!bytes) return NORM_ERR_NULL;
  norm_status_t st = check_common(M, N, mode);
  if (st != NORM_OK) return st;
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  Override ov = read_override();
  if (no_stream) ov.stream = 0;
  if (use_split(static_cast<int>(N), ov, mode, true)) {
    Plan sp[2];
    if ((st = make_split_plans(d, dev, mode, true, M, static_cast<int>(N), sp)) != NORM_OK)
      return st;
    *bytes = split_ws(sp[1], M, mode).total;
    return NORM_OK;
  }
  Plan p;
  if ((st = make_plan(d, dev, mode, true, M, static_cast<int>(N), &p, false, false,
                      no_stream)) != NORM_OK)
    return st;
  *bytes = static_cast<size_t>(p.P) * static_cast<size_t>(N) * sizeof(float) *
           (mode == NORM_LAYER ? 2u : 1u);
  return NORM_OK;
}

norm_status_t norm_bwd_workspace_bytes(int64_t M, int64_t N, norm_mode_t mode, size_t *bytes) {
  return bwd_workspace(M, N, mode, false, bytes);
}

static norm_status_t bwd_run(const void *dy, const void *x, const void *gamma, const float *rstd,
                             const float *mean, int64_t M, int64_t N, norm_mode_t mode,
                             void *dx, float *dgamma, float *dbeta, void *workspace,
                             size_t workspace_bytes, norm_stream_t stream, bool no_stream) {
  if (!dy || !x || !gamma || !rstd || !dx || !dgamma) return NORM_ERR_NULL;
  norm_status_t st = check_common(M, N, mode);
  if (st != NORM_OK) return st;
  if (mode == NORM_RMS && (mean || dbeta)) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && !mean) return NORM_ERR_MODE;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(rstd) ||
      !aligned16(dx) || !aligned16(dgamma) || (mean && !aligned16(mean)) ||
      (dbeta && !aligned16(dbeta)) || (workspace && !aligned16(workspace)))
    return NORM_ERR_ALIGN;
  if (!workspace) return NORM_ERR_WORKSPACE;
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Override ov = read_override();
  if (no_stream) ov.stream = 0;
  if (use_split(static_cast<int>(N), ov, mode, true)) {
    Plan sp[2];
    if ((st = make_split_plans(d, dev, mode, true, M, static_cast<int>(N), sp)) != NORM_OK)
      return st;
    const SplitWs w = split_ws(sp[1], M, mode);
    if (workspace_bytes < w.total) return NORM_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    NormArgs a[2];
    for (int i = 0; i < 2; ++i) {
      a[i] = base_args(sp[i], M, static_cast<int>(N));
      a[i].x = static_cast<const uint16_t *>(x);
      a[i].dy = static_cast<const uint16_t *>(dy);
      a[i].gamma = static_cast<const uint16_t *>(gamma);
      a[i].out = static_cast<uint16_t *>(dx);
      a[i].rstd = const_cast<float *>(rstd);
      a[i].mean = const_cast<float *>(mean);
      a[i].ws = reinterpret_cast<float *>(ws + w.slots);
      a[i].rowp = reinterpret_cast<float *>(ws + w.rowp);
      a[i].rowt = reinterpret_cast<float *>(ws + w.rowt);
      a[i].err = d.err;
    }
    // dot products per (row, segment), their per-row fold, dx with the
    // dgamma / dbeta slots, and the slots' fixed-order reduction
    if ((st = launch(kernel_for(sp[0], mode, true), sp[0], a[0], s)) != NORM_OK) return st;
    if ((st = launch_fold(mode, true, a[0], s)) != NORM_OK) return st;
    if ((st = launch(kernel_for(sp[1], mode, true), sp[1], a[1], s)) != NORM_OK) return st;
    return launch_split_reduce(a[1], sp[1].grid, dgamma, mode == NORM_LAYER ? dbeta : nullptr,
                               s);
  }
  Plan p;
  if ((st = make_plan(d, dev, mode, true, M, static_cast<int>(N), &p, false, false,
                      no_stream)) != NORM_OK)
    return st;
  const size_t need = static_cast<size_t>(p.P) * static_cast<size_t>(N) * sizeof(float) *
                      (mode == NORM_LAYER ? 2u : 1u);
  if (workspace_bytes < need) return NORM_ERR_WORKSPACE;
  NormArgs a = base_args(p, M, static_cast<int>(N));
  a.x = static_cast<const uint16_t *>(x);
  a.dy = static_cast<const uint16_t *>(dy);
  a.gamma = static_cast<const uint16_t *>(gamma);
  a.out = static_cast<uint16_t *>(dx);
  a.rstd = const_cast<float *>(rstd);
  a.mean = const_cast<float *>(mean);
  a.ws = static_cast<float *>(workspace);
  a.err = d.err;
  if ((st = launch(kernel_for(p, mode, true), p, a, s)) != NORM_OK) return st;

  return launch_reduce(static_cast<const float *>(workspace), p.P, static_cast<int>(N), dgamma,
                       (mode == NORM_LAYER) ? dbeta : nullptr, s);
}

norm_status_t norm_bwd(const void *dy, const void *x, const void *gamma, const float *rstd,
                       const float *mean, int64_t M, int64_t N, norm_mode_t mode, void *dx,
                       float *dgamma, float *dbeta, void *workspace, size_t workspace_bytes,
                       norm_stream_t stream) {
  return bwd_run(dy, x, gamma, rstd, mean, M, N, mode, dx, dgamma, dbeta, workspace,
                 workspace_bytes, stream, false);
}

norm_status_t norm_add_fwd(const void *x, const void *r, const void *gamma, const void *beta,
                           int64_t M, int64_t N, float eps, norm_mode_t mode, void *h, void *y,
                           float *rstd, float *mean, norm_stream_t stream) {
  if (!x || !r || !gamma || !h || !y || !rstd) return NORM_ERR_NULL;
  norm_status_t st = check_common(M, N, mode, NORM_MAX_N_FUSED);
  if (st != NORM_OK) return st;
  if (mode == NORM_RMS && (beta || mean)) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && !mean) return NORM_ERR_MODE;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return NORM_ERR_ARG;
  if (!aligned16(x) || !aligned16(r) || !aligned16(gamma) || !aligned16(h) || !aligned16(y) ||
      !aligned16(rstd) || (beta && !aligned16(beta)) || (mean && !aligned16(mean)))
    return NORM_ERR_ALIGN;
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  Plan p;
  if ((st = make_plan(d, dev, mode, false, M, static_cast<int>(N), &p, true)) != NORM_OK)
    return st;
  NormArgs a = base_args(p, M, static_cast<int>(N));
  a.x = static_cast<const uint16_t *>(x);
  a.res = static_cast<const uint16_t *>(r);
  a.gamma = static_cast<const uint16_t *>(gamma);
  a.beta = static_cast<const uint16_t *>(beta);
  a.h = static_cast<uint16_t *>(h);
  a.out = static_cast<uint16_t *>(y);
  a.rstd = rstd;
  a.mean = mean;
  a.err = d.err;
  a.eps = eps;
  return launch(kernel_for(p, mode, false), p, a, reinterpret_cast<cudaStream_t>(stream));
}

norm_status_t norm_add_bwd_workspace_bytes(int64_t M, int64_t N, norm_mode_t mode,
                                           size_t *bytes) {
  if (!bytes) return NORM_ERR_NULL;
  norm_status_t st = check_common(M, N, mode, NORM_MAX_N_FUSED);
  if (st != NORM_OK) return st;
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  Plan p;
  if ((st = make_plan(d, dev, mode, true, M, static_cast<int>(N), &p, true)) != NORM_OK)
    return st;
  *bytes = static_cast<size_t>(p.P) * static_cast<size_t>(N) * sizeof(float) *
           (mode == NORM_LAYER ? 2u : 1u);
  return NORM_OK;
}

norm_status_t norm_add_bwd(const void *dy, const void *dh, const void *h, const void *gamma,
                           const float *rstd, const float *mean, int64_t M, int64_t N,
                           norm_mode_t mode, void *dx, float *dgamma, float *dbeta,
                           void *workspace, size_t workspace_bytes, norm_stream_t stream) {
  if (!dy || !dh || !h || !gamma || !rstd || !dx || !dgamma) return NORM_ERR_NULL;
  norm_status_t st = check_common(M, N, mode, NORM_MAX_N_FUSED);
  if (st != NORM_OK) return st;
  if (mode == NORM_RMS && (mean || dbeta)) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && !mean) return NORM_ERR_MODE;
  if (!aligned16(dy) || !aligned16(dh) || !aligned16(h) || !aligned16(gamma) ||
      !aligned16(rstd) || !aligned16(dx) || !aligned16(dgamma) || (mean && !aligned16(mean)) ||
      (dbeta && !aligned16(dbeta)) || (workspace && !aligned16(workspace)))
    return NORM_ERR_ALIGN;
  if (!workspace) return NORM_ERR_WORKSPACE;
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  Plan p;
  if ((st = make_plan(d, dev, mode, true, M, static_cast<int>(N), &p, true)) != NORM_OK)
    return st;
  const size_t need = static_cast<size_t>(p.P) * static_cast<size_t>(N) * sizeof(float) *
                      (mode == NORM_LAYER ? 2u : 1u);
  if (workspace_bytes < need) return NORM_ERR_WORKSPACE;
  NormArgs a = base_args(p, M, static_cast<int>(N));
  a.x = static_cast<const uint16_t *>(h);
  a.dy = static_cast<const uint16_t *>(dy);
  a.res = static_cast<const uint16_t *>(dh);
  a.gamma = static_cast<const uint16_t *>(gamma);
  a.out = static_cast<uint16_t *>(dx);
  a.rstd = const_cast<float *>(rstd);
  a.mean = const_cast<float *>(mean);
  a.ws = static_cast<float *>(workspace);
  a.err = d.err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch(kernel_for(p, mode, true), p, a, s)) != NORM_OK) return st;
  return launch_reduce(static_cast<const float *>(workspace), p.P, static_cast<int>(N), dgamma,
                       (mode == NORM_LAYER) ? dbeta : nullptr, s);
}

norm_status_t norm_fwd_fp8(const void *x, const void *r, const void *gamma, const void *beta,
                           int64_t M, int64_t N, float eps, norm_mode_t mode,
                           norm_fp8_scaling_t scaling, void *h, void *q, void *scale,
                           float *rstd, float *mean, norm_stream_t stream) {
  if (!x || !gamma || !q || !scale || !rstd) return NORM_ERR_NULL;
  if (r && !h) return NORM_ERR_NULL;
  if (!r && h) return NORM_ERR_ARG;
  if (scaling != NORM_FP8_ROW && scaling != NORM_FP8_MX) return NORM_ERR_ARG;
  norm_status_t st = check_common(M, N, mode, NORM_MAX_N_FUSED);
  if (st != NORM_OK) return st;
  if (scaling == NORM_FP8_MX && N % kMxBlock != 0) return NORM_ERR_SHAPE;
  if (mode == NORM_RMS && (beta || mean)) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && !mean) return NORM_ERR_MODE;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return NORM_ERR_ARG;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(q) || !aligned16(scale) ||
      !aligned16(rstd) || (r && !aligned16(r)) || (h && !aligned16(h)) ||
      (beta && !aligned16(beta)) || (mean && !aligned16(mean)))
    return NORM_ERR_ALIGN;
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != NORM_OK) return st;
  const bool resid = r != nullptr;
  Plan p;
  if ((st = make_plan(d, dev, mode, false, M, static_cast<int>(N), &p, resid, true)) != NORM_OK)
    return st;
  // MX blocks need quads of lanes.
  if (scaling == NORM_FP8_MX && p.tpr % 4 != 0) return NORM_ERR_UNSUPPORTED;
  const int out = scaling == NORM_FP8_ROW ? kOutFp8Row : kOutFp8Mx;
  const void *fn = p.long_rows ? long_fp8_kernel_ptr(mode, p.K, p.C > 1, p.exact, resid, out)
                               : fwd_fp8_kernel_ptr(mode, p.K, p.exact, resid, out, p.gsm);
  if (!fn) return NORM_ERR_UNSUPPORTED;
  if ((st = prepare_function(dev, fn, d.smem_optin)) != NORM_OK) return st;
  NormArgs a = base_args(p, M, static_cast<int>(N));
  a.x = static_cast<const uint16_t *>(x);
  a.res = static_cast<const uint16_t *>(r);
  a.gamma = static_cast<const uint16_t *>(gamma);
  a.beta = static_cast<const uint16_t *>(beta);
  a.h = static_cast<uint16_t *>(h);
  a.q = static_cast<uint8_t *>(q);
  if (scaling == NORM_FP8_ROW) a.qscale = static_cast<float *>(scale);
  else a.qexp = static_cast<uint8_t *>(scale);
  a.rstd = rstd;
  a.mean = mean;
  a.err = d.err;
  a.eps = eps;
  return launch(fn, p, a, reinterpret_cast<cudaStream_t>(stream));
}

norm_status_t norm_plan(int64_t M, int64_t N, norm_mode_t mode, int backward, int sm_count,
                        int smem_optin_bytes, norm_plan_t *out) {
  if (!out) return NORM_ERR_NULL;
  norm_status_t st = check_common(M, N, mode);
  if (st != NORM_OK) return st;
  if (backward & ~15) return NORM_ERR_ARG;
  const bool bwd = (backward & 1) != 0;
  const bool resid = (backward & 2) != 0;
  const bool fp8 = (backward & 4) != 0;
  const bool other = (backward & 8) != 0;  // two-pass path: its other pass
  if (fp8 && bwd) return NORM_ERR_ARG;
  if ((resid || fp8) && N > NORM_MAX_N_FUSED) return NORM_ERR_SHAPE;
  Plan p;
  const Override ov = read_override();
  if (!resid && !fp8 && use_split(static_cast<int>(N), ov, mode, bwd)) {
    // the two-pass path: its statistics (forward) or dx (backward) pass,
    // or with bit 3 the output (forward) or dot-product (backward) pass
    const int phase = bwd ? (other ? kSplitBwdDots : kSplitBwdDx)
                          : (other ? kSplitFwdOut : kSplitFwdStats);
    if (sm_count > 0) {
      if (smem_optin_bytes <= 0) return NORM_ERR_ARG;
      if ((st = split_shape(mode, phase, M, static_cast<int>(N), smem_optin_bytes, ov, &p)) !=
          NORM_OK)
        return st;
      split_grid(p, sm_count);
    } else {
      DeviceInfo d;
      int dev = 0;
      if ((st = device_info(&d, &dev)) != NORM_OK) return st;
      Plan sp[2];
      if ((st = make_split_plans(d, dev, mode, bwd, M, static_cast<int>(N), sp)) != NORM_OK)
        return st;
      p = sp[(phase == kSplitBwdDx || phase == kSplitFwdOut) ? 1 : 0];
    }
    fill_plan(p, out);
    if (phase == kSplitBwdDx) out->partials = p.grid + p.nseg;  // slots, one segment wide
    return NORM_OK;
  }
  if (sm_count > 0) {
    if (smem_optin_bytes <= 0) return NORM_ERR_ARG;
    if ((st = shape_plan(mode, bwd, M, static_cast<int>(N), smem_optin_bytes, read_override(),
                         &p, resid, fp8)) != NORM_OK)
      return st;
    set_grid(p, static_cast<int64_t>(sm_count) / p.C);
    if (p.grid < 1) return NORM_ERR_UNSUPPORTED;
  } else {
    DeviceInfo d;
    int dev = 0;
    if ((st = device_info(&d, &dev)) != NORM_OK) return st;
    if ((st = make_plan(d, dev, mode, bwd, M, static_cast<int>(N), &p, resid, fp8)) != NORM_OK)
      return st;
  }
  fill_plan(p, out);
  return NORM_OK;
}

norm_status_t norm_tune_fwd(const void *x, const void *gamma, const void *beta, int64_t M,
                            int64_t N, float eps, norm_mode_t mode, void *y, float *rstd,
                            float *mean, int iters, norm_plan_t *chosen, norm_stream_t stream) {
  auto run = [&]() { return norm_fwd(x, gamma, beta, M, N, eps, mode, y, rstd, mean, stream); };
  norm_status_t st = check_common(M, N, mode);
  if (st != NORM_OK) return st;
  return tune_pass(mode, false, M, static_cast<int>(N), 0, iters,
                   reinterpret_cast<cudaStream_t>(stream), run, chosen);
}

norm_status_t norm_tune_bwd(const void *dy, const void *x, const void *gamma, const float *rstd,
                            const float *mean, int64_t M, int64_t N, norm_mode_t mode, void *dx,
                            float *dgamma, float *dbeta, void *workspace,
                            size_t workspace_bytes, int iters, norm_plan_t *chosen,
                            norm_stream_t stream) {
  auto run = [&]() {
    return norm_bwd(dy, x, gamma, rstd, mean, M, N, mode, dx, dgamma, dbeta, workspace,
                    workspace_bytes, stream);
  };
  norm_status_t st = check_common(M, N, mode);
  if (st != NORM_OK) return st;
  return tune_pass(mode, true, M, static_cast<int>(N), workspace_bytes, iters,
                   reinterpret_cast<cudaStream_t>(stream), run, chosen);
}

norm_status_t norm_tune_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_plans.clear();
  return NORM_OK;
}

norm_status_t norm_bwd_noalloc(const void *dy, const void *x, const void *gamma,
                               const float *rstd, const float *mean, int64_t M, int64_t N,
                               norm_mode_t mode, void *dx, float *dgamma, float *dbeta,
                               norm_stream_t stream) {
  // Size check first: nothing is launched for a shape that does not fit.
  // The streaming backward writes a partial row per cluster (up to 152);
  // where that exceeds the array, the resident long-row kernel's plan (fewer
  // partial rows) runs instead.
  size_t need = 0;
  norm_status_t st = bwd_workspace(M, N, mode, false, &need);
  if (st != NORM_OK) return st;
  bool no_stream = false;
  if (need > NORM_NOALLOC_WORKSPACE_BYTES) {
    if ((st = bwd_workspace(M, N, mode, true, &need)) != NORM_OK) return st;
    if (need > NORM_NOALLOC_WORKSPACE_BYTES) return NORM_ERR_WORKSPACE;
    no_stream = true;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return NORM_ERR_UNSUPPORTED;
  void *ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = p;
    }
    ws = g_noalloc_ptr[dev];
  }
  return bwd_run(dy, x, gamma, rstd, mean, M, N, mode, dx, dgamma, dbeta, ws,
                 NORM_NOALLOC_WORKSPACE_BYTES, stream, no_stream);
}

norm_status_t norm_selftest_wait_timeout(uint32_t polls, norm_stream_t stream) {
  if (polls < 1 || polls > (1u << 20)) return NORM_ERR_ARG;
  DeviceInfo d;
  int dev = 0;
  norm_status_t st = device_info(&d, &dev);
  if (st != NORM_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  unsigned *err = d.err;
  void *args[] = {&err, &polls};
  if (cudaLaunchKernelExC(&cfg, selftest_kernel_ptr(), args) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  return NORM_OK;
}

const char *norm_strerror(norm_status_t s) {
  switch (s) {
    case NORM_OK: return "success";
    case NORM_ERR_NULL: return "a required pointer is NULL";
    case NORM_ERR_SHAPE: return "unsupported shape (need M >= 1, 8 <= N <= NORM_MAX_N, N % 8 == 0)";
    case NORM_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case NORM_ERR_MODE: return "mode/argument mismatch (beta, mean, dbeta only for LayerNorm; mean required there)";
    case NORM_ERR_WORKSPACE: return "workspace missing or too small";
    case NORM_ERR_UNSUPPORTED: return "shape cannot be scheduled on this device";
    case NORM_ERR_CUDA: return "CUDA runtime error";
    case NORM_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait on an asynchronous copy";
    case NORM_ERR_ARG: return "eps must be finite and >= 0 (or a numeric argument is out of range)";
    case NORM_ERR_MEMORY: return "a pointer is not device memory of the current device";
  }
  return "unknown status";
}

norm_status_t norm_get_device_error(norm_stream_t stream) {
  DeviceInfo d;
  int dev = 0;
  norm_status_t st = device_info(&d, &dev);
  if (st != NORM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned h = 0;
  if (cudaMemcpyAsync(&h, d.err, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(d.err, 0, sizeof h, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  return h ? NORM_ERR_DEVICE_TIMEOUT : NORM_OK;
}

}  // extern "C"
