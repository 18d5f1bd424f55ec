// common.cuh -- types shared by the kernels and the host launcher.
#pragma once
#include <cstdint>

namespace gbn {

constexpr int kRMS = 0;
constexpr int kLayer = 1;

// Largest chunk counts per thread that are compiled (a chunk is 8 bf16 =
// 16 bytes of one row).
constexpr int kMaxKFwd = 8;
constexpr int kMaxKBwd = 4;
// Largest CTA (the kernels are compiled for at most this many threads, which
// lets the compiler give each thread up to 128 registers).
constexpr int kMaxThreads = 512;
// Cross-CTA exchange buffers (rounds use them in turn; four allow a round to
// be pushed before the previous one is consumed).
constexpr int kXchBuffers = 4;

// Kernel arguments.  A "tile" is RT consecutive rows restricted to the
// column slice [col0, col0 + NS) that one CTA of a cluster owns (the whole
// row when the cluster has one CTA).  Each row of a tile is processed by a
// group of `tpr` threads; a CTA has G groups; each group takes rpg rows of
// every tile (RT = G * rpg).
struct NormArgs {
  const uint16_t *x;      // bf16 [M, N]
  const uint16_t *dy;     // bf16 [M, N] (backward)
  const uint16_t *gamma;  // bf16 [N]
  const uint16_t *beta;   // bf16 [N] or null (forward, LayerNorm)
  const uint16_t *res;    // fused residual: r (forward) or dh (backward), bf16 [M, N]
  uint16_t *h;            // fused residual forward: h = bf16(x + r), bf16 [M, N]
  uint16_t *out;          // y (forward) or dx (backward), bf16 [M, N]
  uint8_t *q;             // FP8 forward: E4M3 codes of y [M, N]
  float *qscale;          // FP8 forward, per-row scaling: dequantisation scale [M]
  uint8_t *qexp;          // FP8 forward, MX scaling: E8M0 block exponents [M, N / 32]
  float *rstd;            // [M]: written by forward, read by backward
  float *mean;            // [M]: same, LayerNorm only
  float *ws;              // backward partial sums [P, N] (+ [P, N] for dbeta); on the
                          // two-pass path the per-(CTA, segment) slots
  float *rowp;            // two-pass backward: per-(row, segment) dot products [M, nseg, 2]
  float *rowt;            // two-pass backward: per-row dot-product totals [M, 2]
  unsigned *err;          // device error word
  int64_t M;
  int64_t ntiles;
  int N;    // row length
  int NS;   // columns per CTA slice (N / cluster size)
  int nsc;  // 16-byte chunks per slice (NS / 8)
  int tpr;  // threads per row
  int G;    // row groups per CTA
  int rpg;  // rows per group per tile
  int RT;   // rows per tile
  int S;    // pipeline stages
  int P;    // partial rows (backward) = number of clusters in the grid
  int C;    // CTAs per cluster
  int nseg; // two-pass path: segments of NS columns per row (the last one ragged)
  float eps;
  float invN;
  unsigned wait_ns;  // register-resident forward: suspend hint of its stage waits (0: none)
};

// Byte offsets of the dynamic shared memory regions (all 16-byte aligned).
struct SmemLayout {
  uint32_t tensor_bytes;  // one tensor's share of a stage: RT * NS * 2
  uint32_t stage_bytes;   // ntensors * tensor_bytes
  uint32_t par_off;       // forward with gamma (and beta) staged in shared memory
  uint32_t stats_off;     // backward: [S][RT][2] floats (rstd, mean)
  uint32_t red_off;       // [2][G][W][4] floats, cross-warp group partials
                          // (W = tpr / 32; only when tpr > 32)
  uint32_t xch_off;       // clusters only: [kXchBuffers][RT][C][4] floats of
                          // cross-CTA partials, then one mbarrier per buffer
  uint32_t bar_off;       // [S] mbarriers
  uint32_t flag_off;      // abort flag (int), then [S] ints: warps done per stage
  uint32_t total;
};

__host__ __device__ inline int64_t min64(int64_t a, int64_t b) {
  return a < b ? a : b;
}

__host__ __device__ inline uint32_t align16(uint32_t v) {
  return (v + 15u) & ~15u;
}

// C: CTAs per cluster (1: no cluster exchange region).  par_bpc: bytes per
// column of the parameters staged in shared memory by the forward kernels
// that read them per row (param_bytes_per_col; 0 for the others).
__host__ __device__ inline SmemLayout make_layout(int RT, int NS, int S, int G,
                                                  int tpr, int ntensors,
                                                  bool stats, int C, int par_bpc = 0) {
  SmemLayout L;
  L.tensor_bytes = static_cast<uint32_t>(RT) * static_cast<uint32_t>(NS) * 2u;
  L.stage_bytes = L.tensor_bytes * static_cast<uint32_t>(ntensors);
  uint32_t off = L.stage_bytes * static_cast<uint32_t>(S);
  L.par_off = off;
  off = align16(off + static_cast<uint32_t>(par_bpc) * static_cast<uint32_t>(NS));
  L.stats_off = off;
  if (stats) off = align16(off + static_cast<uint32_t>(S * RT * 2) * 4u);
  L.red_off = off;
  if (tpr > 32) off = align16(off + static_cast<uint32_t>(2 * G * (tpr / 32) * 4) * 4u);
  L.xch_off = off;
  if (C > 1) off = align16(off + static_cast<uint32_t>(kXchBuffers * RT * C * 4) * 4u +
                           8u * kXchBuffers);
  L.bar_off = off;
  off = align16(off + static_cast<uint32_t>(S) * 8u);
  L.flag_off = off;
  off = align16(off + 4u + 4u * static_cast<uint32_t>(S));
  L.total = off;
  return L;
}

// Host-side launch plan.
struct Plan {
  int C = 1;       // CTAs per cluster (column split)
  int NS = 0;      // columns per CTA
  int nsc = 0;     // chunks per CTA slice
  int tpr = 0;     // threads per row
  int K = 0;       // chunks per thread
  bool exact = false; // slices divide evenly into K chunks x tpr threads, tpr >= 32
  bool long_rows = false; // long-row kernels (row re-read from the stage)
  bool resid = false;     // fused residual add variant
  bool gsm = false;       // forward: gamma/beta read per row from shared memory
  int par_bpc = 0;        // gsm: staged parameter bytes per column
  int G = 0;       // groups per CTA
  int rpg = 1;     // rows per group per tile
  int RT = 0;      // rows per tile
  int S = 0;       // stages
  int threads = 0; // G * tpr
  uint32_t smem = 0;
  int64_t ntiles = 0;
  int grid = 0;    // CTAs
  int P = 0;       // clusters in the grid (partial rows in backward)
  bool split = false;  // two-pass path: rows cut into nseg segments of NS columns
  int nseg = 0;
  int phase = 0;       // two-pass path: which of its passes (kSplit*)
  bool stream = false; // the streaming long-row kernels (stream.cu)
  int piece_kp = 0;    // streaming: chunks per thread per piece
  int wait_ns = 0;     // register-resident forward: suspend hint of its stage waits
};

// Kernel entry points, by (mode, K, cluster, exact, fused residual).
// Return nullptr when that combination is not compiled (the fused residual
// variants exist without clusters only).
// Bytes per column of the parameters a staged-parameter forward kernel keeps
// in shared memory: gamma (and beta for LayerNorm), as fp32 for bf16 output
// (no unpacking per row) and as bf16 for E4M3 output (less shared-memory
// traffic next to the heavier epilogue; measured faster for each).
__host__ __device__ constexpr int param_bytes_per_col(int mode, bool fp8_out) {
  return (mode == 1 ? 2 : 1) * (fp8_out ? 2 : 4);
}

// Forward output kinds: bf16 y, or E4M3 codes with a per-row fp32 scale, or
// E4M3 codes with one E8M0 exponent per 32-column block (MX).
constexpr int kOutBf16 = 0;
constexpr int kOutFp8Row = 1;
constexpr int kOutFp8Mx = 2;
constexpr int kMxBlock = 32;
// Phases of the long-row forward's per-row E4M3 output pass: amax then codes
// (one CTA per row), or in a cluster this CTA's slice amax alone, and later
// the codes with the row amax the exchange returned.
constexpr int kFp8Whole = 0;
constexpr int kFp8Amax = 1;
constexpr int kFp8Codes = 2;

// gsm: gamma (and beta) staged in shared memory and read per row, which frees
// the registers that hold them otherwise (exact splits, no cluster, K in
// {5, 6, 8}; see fwd_gsm_kernel_ptr).
// sleep: the variant whose stage waits carry the plan's suspend hint (exact,
// no cluster, no residual, no staged parameters, K in {2, 4}).
const void *fwd_kernel_ptr(int mode, int K, bool cluster, bool exact, bool resid = false,
                           bool gsm = false, bool sleep = false);
// E4M3 output variants (no cluster variants); nullptr if not instantiated.
const void *fwd_fp8_kernel_ptr(int mode, int K, bool exact, bool resid, int out,
                               bool gsm = false);
// Forward kernels with gamma/beta staged in shared memory (exact splits, no
// cluster), K in {5, 6, 8}, any output kind; nullptr otherwise.
const void *fwd_gsm_kernel_ptr(int mode, int K, bool resid, int out);
const void *bwd_kernel_ptr(int mode, int K, bool cluster, bool exact, bool resid = false);
const void *reduce_kernel_ptr();
// Long-row kernels (row slice re-read from shared memory), K in {4, 8}.
const void *long_kernel_ptr(int mode, int K, bool cluster, bool exact, bool bwd,
                            bool resid = false);
const void *long_resid_kernel_ptr(int mode, int K, bool cluster, bool exact, bool bwd);
// Long-row forward with E4M3 output (kOutFp8Row or kOutFp8Mx, with or
// without a cluster); nullptr if not instantiated.
const void *long_fp8_kernel_ptr(int mode, int K, bool cluster, bool exact, bool resid, int out);
int reduce_threads();
const void *selftest_kernel_ptr();

// The two-pass path for rows longer than one cluster holds (split.cu).
constexpr int kSplitFwdStats = 0;  // per-(row, segment) statistics into y
constexpr int kSplitFwdOut = 1;    // y from the folded statistics
constexpr int kSplitBwdDots = 2;   // per-(row, segment) dot products
constexpr int kSplitBwdDx = 3;     // dx and the dgamma / dbeta slots
// Kernels by (mode, pass, chunks per thread); nullptr if not instantiated
// (K = 4 for the first three passes, 2 for the dx pass).
const void *split_kernel_ptr(int mode, int phase, int K);
const void *split_fold_kernel_ptr(int mode, bool bwd);
const void *split_reduce_kernel_ptr();
SmemLayout split_smem_layout(int RT, int NS, int S, int G, int tpr, int ntensors);

// The streaming long-row kernels (stream.cu): one row group of
// kStreamThreads threads per CTA, each CTA owning a slice of a row
// (kStreamSlice columns in the backward, a cluster of N / kStreamSlice CTAs;
// that or twice as many in the forward), streamed twice through a ring of
// pieces of kStreamThreads x kp x 8 columns (kp 16-byte chunks per thread).
constexpr int kStreamThreads = 512;
constexpr int kStreamSlice = 32768;
__host__ __device__ constexpr int stream_piece_cols(int kp) { return kStreamThreads * kp * 8; }
// Their shared memory: S stages of `ntensors` pieces -- x (forward), x and dy
// (backward), x, dy and dh (fused residual backward; only the dx pass loads
// dh) -- the per-warp row partials ([kXchBuffers][warps][2] floats for the
// backward's two sums, [..][4] for the forward's (mean, M2) pairs, then
// kXchBuffers arrival counters), the exchange slots and their mbarriers
// ([kXchBuffers][C] float4, also for C = 1), the stage mbarriers, then the
// abort flag, the per-stage warp counters and the tensor-memory address slot.
__host__ __device__ inline SmemLayout stream_layout(int S, int C, int ntensors, int kp) {
  SmemLayout L;
  L.tensor_bytes = static_cast<uint32_t>(stream_piece_cols(kp)) * 2u;
  L.stage_bytes = static_cast<uint32_t>(ntensors) * L.tensor_bytes;
  uint32_t off = L.stage_bytes * static_cast<uint32_t>(S);
  L.par_off = off;
  L.stats_off = off;
  L.red_off = off;
  const int per_warp = ntensors == 1 ? 4 : 2;
  off = align16(off + static_cast<uint32_t>(kXchBuffers * (kStreamThreads / 32) * per_warp) * 4u +
                4u * kXchBuffers);
  L.xch_off = off;
  off = align16(off + static_cast<uint32_t>(kXchBuffers * C * 4) * 4u + 8u * kXchBuffers);
  L.bar_off = off;
  off = align16(off + static_cast<uint32_t>(S) * 8u);
  L.flag_off = off;
  off = align16(off + 4u + 4u * static_cast<uint32_t>(S) + 4u);
  L.total = off;
  return L;
}
// Backward kernel by (mode, chunks per thread per piece: 2 or 4, cluster or
// single CTA, fused residual); nullptr if not instantiated.
const void *stream_kernel_ptr(int mode, int kp, bool cluster, bool resid = false);
// Forward kernel by (mode, kp, pieces per slice, cluster); nullptr if not
// instantiated.
const void *stream_fwd_kernel_ptr(int mode, int kp, int np, bool cluster);

}  // namespace gbn
