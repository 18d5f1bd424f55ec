/*
 * gbnorm.h -- C ABI of the GB300 (sm_103a) RMSNorm / LayerNorm library.
 *
 * The operation (page "PyTorch atinge desempenho SOTA em normalizacao com
 * torch.compile", matsubara.tec.br; paragraphs on LayerNorm/RMSNorm, on the
 * forward pass and on the backward pass):
 *   forward   a reduction along the contiguous last dimension of each row
 *             (mean and variance for LayerNorm, mean square for RMSNorm),
 *             then pointwise normalisation and the trainable scale gamma
 *             (plus the shift beta for LayerNorm);
 *   backward  dX from per-row dot products, dW (dgamma) and, for LayerNorm,
 *             dB (dbeta) from a column reduction over all rows.
 * Definitions used (the page prints none; the textbook reading):
 *   LayerNorm  mean = sum(x)/N, var = sum((x-mean)^2)/N (population),
 *              rstd = 1/sqrt(var + eps), y = (x-mean)*rstd*gamma + beta
 *   RMSNorm    rstd = 1/sqrt(sum(x^2)/N + eps), y = x*rstd*gamma
 *   backward   g = dy*gamma, xhat = (x-mean)*rstd (mean = 0 for RMSNorm),
 *              c = sum(g*xhat)/N, a = sum(g)/N (LayerNorm; 0 for RMSNorm),
 *              dx = rstd*(g - a - xhat*c),
 *              dgamma = column sums of dy*xhat, dbeta = column sums of dy.
 *
 * Data layout.  x, y, dy, dx: bf16 [M, N], row-major, rows contiguous (row
 * stride N elements).  gamma, beta: bf16 [N].  rstd, mean: fp32 [M].
 * dgamma, dbeta: fp32 [N].  All arithmetic is fp32; bf16 results are
 * rounded to nearest even.
 *
 * Ownership.  Every pointer is a DEVICE pointer owned by the caller.  The
 * library allocates no device memory; the backward pass takes a caller
 * workspace (see norm_bwd_workspace_bytes).  Outputs must not alias inputs.
 *
 * Requirements.  M >= 1, 8 <= N <= NORM_MAX_N, N % 8 == 0, and every
 * pointer 16-byte aligned (so each row starts on a 16-byte boundary and is
 * moved by 16-byte bulk copies and 128-bit loads/stores).  There is no
 * slow path for other shapes: they are rejected with a status code.
 *
 * Execution.  Calls are asynchronous on `stream` (NULL = the legacy default
 * stream) and thread-safe.  The library caches per device and per CUDA
 * context what it looks up once (SM count, kernel attributes, launch plans,
 * the addresses of its device error word and scratch array, its internal
 * copy streams); after the context is destroyed (cudaDeviceReset) the next
 * call on that device sees a new context and sets it up again, dropping
 * the plans of the old one (tuned plans included).  The return value
 * reports argument validation and launch errors.  Execution errors surface
 * at the caller's next synchronisation, or, for the library's own bounded
 * waits, through norm_get_device_error.  Results are bitwise reproducible run to run for a
 * given shape and device: every reduction, including the dgamma/dbeta
 * column sums, is done in a fixed order without atomics.
 */
#ifndef GBNORM_H
#define GBNORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that callers need no CUDA
 * header. */
struct CUstream_st;
typedef struct CUstream_st *norm_stream_t;

/* Largest row length (columns) of norm_fwd / norm_bwd and of their
 * allocation-free and host-tensor variants.  Rows of up to
 * NORM_MAX_N_ONEPASS columns are normalised in one pass over HBM (rows held
 * in registers, or in the shared memory of one CTA or of a thread-block
 * cluster of up to 16 CTAs); wider rows take a two-pass path that cuts each
 * row into 4096-column segments and reads x (and dy) twice. */
#define NORM_MAX_N (1 << 24)
#define NORM_MAX_N_ONEPASS 262144
/* Largest row length of the fused variants (norm_add_fwd / norm_add_bwd,
 * norm_fwd_fp8) and of the normalisation-GEMM's K: the one-pass limit. */
#define NORM_MAX_N_FUSED NORM_MAX_N_ONEPASS

typedef enum {
    NORM_RMS = 0,   /* RMSNorm: no mean, no beta */
    NORM_LAYER = 1  /* LayerNorm */
} norm_mode_t;

typedef enum {
    NORM_OK = 0,
    NORM_ERR_NULL = 1,           /* a required pointer is NULL */
    NORM_ERR_SHAPE = 2,          /* M < 1, N < 8, N % 8 != 0, or N above the
                                    entry point's limit (NORM_MAX_N, or
                                    NORM_MAX_N_FUSED for the fused variants) */
    NORM_ERR_ALIGN = 3,          /* a pointer is not 16-byte aligned */
    NORM_ERR_MODE = 4,           /* unknown mode, or a pointer given that the
                                    mode forbids (beta/mean/dbeta for RMS) or
                                    missing that it needs (mean for LAYER) */
    NORM_ERR_WORKSPACE = 5,      /* workspace NULL or smaller than required */
    NORM_ERR_UNSUPPORTED = 6,    /* shape cannot be scheduled on this device */
    NORM_ERR_CUDA = 7,           /* a CUDA runtime call failed */
    NORM_ERR_DEVICE_TIMEOUT = 8, /* a kernel gave up a bounded wait */
    NORM_ERR_ARG = 9,            /* eps is negative or not finite (or
                                    another numeric argument out of range) */
    NORM_ERR_MEMORY = 10         /* a pointer that a tensor copy reads or
                                    writes is not device memory of the
                                    current device (norm_gemm_fwd) */
} norm_status_t;

/*
 * norm_fwd -- forward pass.
 *   x      bf16 [M, N] input
 *   gamma  bf16 [N] scale
 *   beta   bf16 [N] shift; LAYER only (NULL means zero); must be NULL for RMS
 *   eps    added to the variance (LAYER) or mean square (RMS) inside the
 *          square root; finite and >= 0
 *   y      bf16 [M, N] output
 *   rstd   fp32 [M] output, 1/sqrt(var + eps) or 1/sqrt(meansq + eps)
 *   mean   fp32 [M] output; required for LAYER, must be NULL for RMS
 * One kernel for N <= NORM_MAX_N_ONEPASS.  Wider rows take three: the
 * per-segment statistics (written into y as scratch, 8 bytes per segment of
 * each row), their fixed-order fold into rstd / mean, and the output.
 */
norm_status_t norm_fwd(const void *x, const void *gamma, const void *beta,
                       int64_t M, int64_t N, float eps, norm_mode_t mode,
                       void *y, float *rstd, float *mean,
                       norm_stream_t stream);

/*
 * norm_bwd_workspace_bytes -- size of the workspace norm_bwd needs for this
 * shape on the CURRENT device (it holds one fp32 row of dgamma partial sums,
 * and for LAYER one of dbeta partial sums, per column-reduction split).
 */
norm_status_t norm_bwd_workspace_bytes(int64_t M, int64_t N, norm_mode_t mode,
                                       size_t *bytes);

/*
 * norm_bwd -- backward pass, reusing the statistics saved by norm_fwd.
 *   dy      bf16 [M, N] gradient of y
 *   x       bf16 [M, N] forward input
 *   gamma   bf16 [N]
 *   rstd    fp32 [M] from norm_fwd
 *   mean    fp32 [M] from norm_fwd; required for LAYER, NULL for RMS
 *   dx      bf16 [M, N] output
 *   dgamma  fp32 [N] output
 *   dbeta   fp32 [N] output for LAYER (NULL skips it); must be NULL for RMS
 *   workspace, workspace_bytes  device scratch of at least
 *           norm_bwd_workspace_bytes(M, N, mode) bytes, 16-byte aligned; its
 *           contents on entry are ignored.  Two calls that overlap in time
 *           must not share a workspace.
 * Two kernels run on `stream`: the fused row pass (dx plus per-CTA partial
 * column sums written to the workspace) and a fixed-order reduction of the
 * partials into dgamma/dbeta.  Rows wider than NORM_MAX_N_ONEPASS take four:
 * the per-(row, segment) dot products (into the workspace), their per-row
 * fold, dx with the dgamma/dbeta sums of each CTA's segments (into the
 * workspace), and a fixed-order reduction of those.
 */
norm_status_t norm_bwd(const void *dy, const void *x, const void *gamma,
                       const float *rstd, const float *mean, int64_t M,
                       int64_t N, norm_mode_t mode, void *dx, float *dgamma,
                       float *dbeta, void *workspace, size_t workspace_bytes,
                       norm_stream_t stream);

/*
 * Fused residual add + norm.  The same page credits the normalisation
 * kernels' automatic fusion with surrounding operations, and "Otimizacao de
 * Performance de GPU" (introl.com, paragraph on kernel fusion) the saving of
 * intermediate HBM traffic; the usual pre-norm transformer block adds a
 * residual right before the norm.  One pass reads x and r and writes both
 * the updated residual stream and the normalised output:
 *   h = bf16(x + r)   (sum in fp32, rounded to nearest even)
 *   y = norm(h)       (as norm_fwd, on the bf16 values of h)
 * and the backward pass adds the gradient dh that reaches h through the
 * residual path:  dx = (norm_bwd's dx at h) + dh  (sum in fp32, one rounding);
 * dx is the gradient of both x and r.  dgamma / dbeta as norm_bwd.
 * Shapes: as norm_fwd / norm_bwd but N up to NORM_MAX_N_FUSED; rows wider than one
 * CTA's registers use the long-row kernels (and thread-block clusters) with
 * the residual tensor in the same shared-memory stage.  Other requirements
 * as norm_fwd / norm_bwd.
 *
 * norm_add_fwd:  x, r bf16 [M, N] inputs; h, y bf16 [M, N] outputs; rstd,
 *                mean (LAYER) fp32 [M] outputs; gamma, beta as norm_fwd.
 * norm_add_bwd:  dy, dh, h bf16 [M, N]; rstd, mean from norm_add_fwd; dx bf16
 *                [M, N]; workspace of norm_add_bwd_workspace_bytes bytes.
 */
norm_status_t norm_add_fwd(const void *x, const void *r, const void *gamma,
                           const void *beta, int64_t M, int64_t N, float eps,
                           norm_mode_t mode, void *h, void *y, float *rstd,
                           float *mean, norm_stream_t stream);

norm_status_t norm_add_bwd_workspace_bytes(int64_t M, int64_t N,
                                           norm_mode_t mode, size_t *bytes);

norm_status_t norm_add_bwd(const void *dy, const void *dh, const void *h,
                           const void *gamma, const float *rstd,
                           const float *mean, int64_t M, int64_t N,
                           norm_mode_t mode, void *dx, float *dgamma,
                           float *dbeta, void *workspace,
                           size_t workspace_bytes, norm_stream_t stream);

/*
 * FP8 output.  The page "Otimizacao de Performance de GPU" (introl.com,
 * December 2025 update) reports FP8 training as production ready on
 * Blackwell; the next consumer of a norm's output is usually a GEMM, which
 * on this GPU reads E4M3 operands.  norm_fwd_fp8 computes y exactly as
 * norm_fwd (or norm_add_fwd when r is given) and writes it as E4M3 codes
 * (OCP 8-bit floating point E4M3FN: bias 7, 3 mantissa bits, largest finite
 * 448, no infinities) rounded to nearest even with saturation, after one of
 * two scalings:
 *   NORM_FP8_ROW  per row: amax = max_j |y_ij| (fp32), codes of
 *                 y * (448 / amax); scale[i] = amax / 448 (fp32 [M]) so that
 *                 y ~= decode(q) * scale; a row of zeros has scale 1.  Both
 *                 quotients are formed in fp32 within 2 ulp.
 *   NORM_FP8_MX   per 32-column block (OCP Microscaling Formats v1.0, section
 *                 6.3): X = 2^e, e = floor(log2 amax_block) - 8, clamped
 *                 below at -127; codes of y / X (exact); scale holds the
 *                 E8M0 byte e + 127 per block, row-major uint8 [M, N / 32].
 *                 N must be a multiple of 32 (else NORM_ERR_SHAPE).
 * Arguments:
 *   x, gamma, beta, M, N, eps, mode, rstd, mean   as norm_fwd;
 *   r     bf16 [M, N] residual, or NULL for a plain norm; with r, h (bf16
 *         [M, N]) receives bf16(x + r) and the norm is taken of h, as
 *         norm_add_fwd (h must be NULL when r is);
 *   q     uint8 [M, N] E4M3 codes of y;
 *   scale float [M] (NORM_FP8_ROW) or uint8 [M, N / 32] (NORM_FP8_MX).
 * All pointers are device pointers owned by the caller, 16-byte aligned.
 * Every N up to NORM_MAX_N_FUSED is supported (rows wider than one CTA use the
 * long-row kernels and clusters; with per-row scaling the CTAs of a cluster
 * exchange their slice maxima); an unknown scaling returns NORM_ERR_ARG.
 * One kernel on `stream`.  The backward pass of an FP8-output forward is
 * norm_bwd / norm_add_bwd (it reads x or h and the saved rstd / mean).
 */
typedef enum { NORM_FP8_ROW = 0, NORM_FP8_MX = 1 } norm_fp8_scaling_t;

norm_status_t norm_fwd_fp8(const void *x, const void *r, const void *gamma,
                           const void *beta, int64_t M, int64_t N, float eps,
                           norm_mode_t mode, norm_fp8_scaling_t scaling,
                           void *h, void *q, void *scale, float *rstd,
                           float *mean, norm_stream_t stream);

/*
 * Forward + backward on HOST tensors.  For callers whose activations live in
 * host memory (offloaded activations, data-loader output, tests): one call
 * copies the inputs in, runs norm_fwd and norm_bwd, and copies every output
 * back, with the rows cut into chunks that stream through a few device
 * buffers so that host-to-device copies, kernels and device-to-host copies
 * of different chunks overlap on three streams (the copy engines of the two
 * directions work at the same time).  The computation is that of norm_fwd /
 * norm_bwd: y, rstd, mean and dx equal theirs bit for bit; dgamma / dbeta
 * are summed per chunk and then over chunks in chunk order (bitwise
 * reproducible for a given chunk_rows, equal to norm_bwd's within
 * rounding).
 *
 * norm_host_workspace_bytes: device workspace norm_fwd_bwd_host needs for
 *   this shape and chunk size (chunk_rows = 0: the library's default, about
 *   16 MB of x per chunk): three chunks of x, dy, y and dx, plus rstd (and
 *   mean) of all M rows, which go back to the host in one copy each after
 *   the last chunk.
 * norm_fwd_bwd_host:
 *   x, dy          HOST bf16 [M, N] inputs (page-locked memory, e.g. from
 *                  cudaHostAlloc, for the copies to overlap; pageable memory
 *                  works but serialises);
 *   gamma, beta    HOST bf16 [N] (beta NULL: zero; RMS: NULL);
 *   y, dx          HOST bf16 [M, N] outputs; rstd, mean HOST fp32 [M]
 *                  (mean LAYER only); dgamma, dbeta HOST fp32 [N] (dbeta
 *                  LAYER only, may be NULL);
 *   chunk_rows     rows per chunk (0: default; rounded up to a multiple of
 *                  4 when smaller than M);
 *   workspace      DEVICE memory of norm_host_workspace_bytes bytes, 256-byte
 *                  aligned, owned by the caller (NORM_ERR_WORKSPACE if NULL or
 *                  short, NORM_ERR_ALIGN if misaligned).
 * Asynchronous: the call enqueues everything behind the work already on
 * `stream` and returns; the host outputs are complete once `stream` is
 * synchronised.  The host buffers must stay valid until then.  Calls on one
 * device are serialised while they enqueue; the library's two internal copy
 * streams are created on first use.
 */
norm_status_t norm_host_workspace_bytes(int64_t M, int64_t N, norm_mode_t mode,
                                        int64_t chunk_rows, size_t *bytes);

norm_status_t norm_fwd_bwd_host(const void *x, const void *dy, const void *gamma,
                                const void *beta, int64_t M, int64_t N, float eps,
                                norm_mode_t mode, void *y, void *dx, float *rstd,
                                float *mean, float *dgamma, float *dbeta,
                                int64_t chunk_rows, void *workspace,
                                size_t workspace_bytes, norm_stream_t stream);

/*
 * norm_plan -- the launch plan the library uses for one pass (backward = 0
 * for norm_fwd, 1 for norm_bwd, 2 for norm_add_fwd, 3 for norm_add_bwd, 4
 * for norm_fwd_fp8 without and 6 with a residual; for rows on the two-pass
 * path, 0 / 1 report its statistics / dx pass and 8 / 9 its output /
 * dot-product pass) of an [M, N] problem: how rows are split
 * across threads, CTAs and clusters, and how many tiles are kept in flight.
 * With sm_count <= 0 it describes the CURRENT device (occupancy queried
 * through the CUDA runtime) and equals what norm_fwd / norm_bwd launch.
 * With sm_count > 0 and smem_optin_bytes > 0 it computes the plan for that
 * hypothetical device without any CUDA call, assuming one resident CTA per
 * SM (for host-side checks and planning).
 */
typedef struct {
    int32_t cluster;           /* CTAs per thread-block cluster; each owns
                                  N / cluster consecutive columns */
    int32_t cols_per_cta;      /* N / cluster */
    int32_t threads_per_row;   /* threads cooperating on one row (slice) */
    int32_t chunks_per_thread; /* 16-byte chunks of a row per thread */
    int32_t groups;            /* rows processed concurrently per CTA */
    int32_t rows_per_group;    /* rows each group takes from a tile */
    int32_t rows_per_tile;     /* groups * rows_per_group */
    int32_t stages;            /* tiles in flight per CTA */
    int32_t threads;           /* CTA size */
    int32_t smem_bytes;        /* dynamic shared memory per CTA */
    int64_t tiles;             /* ceil(M / rows_per_tile) */
    int32_t grid;              /* CTAs launched */
    int32_t partials;          /* clusters launched = partial rows written
                                  by the backward pass */
    int32_t exact;             /* 1: every CTA slice is exactly
                                  threads_per_row * chunks_per_thread chunks
                                  (kernels without ownership tests) */
    int32_t long_rows;         /* 1: long-row kernels (the row slice is read
                                  twice from shared memory instead of being
                                  held in registers) */
    int32_t param_smem_bytes;  /* forward only: bytes of gamma (and beta for
                                  LAYER) staged in shared memory and read per
                                  row instead of being held in registers
                                  (fp32 for bf16 output, bf16 for E4M3
                                  output); 0 if none */
    int32_t split_segments;    /* two-pass path (rows wider than
                                  NORM_MAX_N_ONEPASS): segments of
                                  cols_per_cta columns per row; the fields
                                  above describe its statistics (forward) or
                                  dx (backward) pass, whose rows_per_tile
                                  rows of one segment make a unit, `tiles`
                                  counting the row tiles; 0 otherwise */
    int32_t streamed;          /* 1 when the row slices (cols_per_cta
                                  columns each) are streamed twice through
                                  shared memory, the second read served from
                                  L2: statistics then y (forward), dot
                                  products then dx with the dgamma / dbeta
                                  column sums held in tensor memory
                                  (backward); 0 otherwise */
    int32_t wait_hint_ns;      /* forward, register-resident rows: suspend
                                  hint (ns) of the waits for a stage, so that
                                  a waiting row group issues nothing; 0: the
                                  hardware's default interval */
    int32_t piece_cols;        /* streamed plans: columns of a slice moved
                                  per shared-memory stage; 0 otherwise */
} norm_plan_t;

norm_status_t norm_plan(int64_t M, int64_t N, norm_mode_t mode, int backward,
                        int sm_count, int smem_optin_bytes, norm_plan_t *out);

/*
 * Normalisation fused into a GEMM.  Item 4 of the page "Towards Free
 * Normalization: Fusing Normalization into GEMM and Attention Kernels"
 * names the Lazy Pre-Norm fusion; its items 9 and 10 give the obstacle it
 * removes (the normalisation needs whole rows, a GEMM tiles rows and
 * columns).  The operation is a pre-norm linear layer:
 *
 *   out = norm(x) W^T    x bf16 [M, K]; W bf16 [Nout, K], one row per
 *                        output feature; out bf16 [M, Nout], row-major
 *
 * with norm the forward definition at the top of this file over the K
 * columns of x (gamma, beta bf16 [K]).  The library applies the
 * normalisation after the contraction, which is linear in the normalised
 * row:
 *
 *   out_ik = rstd_i * (sum_j x_ij W'_kj - mean_i * u_k) + v_k
 *   W'_kj = bf16(W_kj * gamma_j) (nearest even), u_k = sum_j W'_kj,
 *   v_k = sum_j W_kj * beta_j    (mean = 0 and v = 0 for RMSNorm)
 *
 * norm_gemm_prepare makes W', u and v from the weights (once per weight
 * update).  norm_gemm_fwd is one tcgen05 tensor-core GEMM on the raw x that
 * takes each row's statistics from the tiles it streams and applies rstd
 * and the mean correction in its epilogue; the normalised rows are never
 * written.  Accumulation is fp32; out is rounded to nearest even.  Numerics
 * differ from rounding norm(x) to bf16 before a bf16 GEMM: here x enters
 * exactly and W * gamma is rounded once.  Results are bitwise reproducible
 * for a given shape and device.
 *
 * norm_gemm_prepare: w [Nout, K]; gamma [K]; beta [K] or NULL (LAYER only,
 *   NULL = 0; non-NULL with RMS is NORM_ERR_MODE); wg [Nout, K] bf16 out
 *   (W'); u, v [Nout] fp32 out, required for LAYER (else NORM_ERR_MODE),
 *   optional for RMS.
 * norm_gemm_fwd: x [M, K]; wg, u, v from norm_gemm_prepare (u and v are
 *   not read for RMS; required for LAYER); out [M, Nout]; rstd [M] fp32 out
 *   (required); mean [M] fp32 out, required for LAYER and NULL for RMS
 *   (else NORM_ERR_MODE); eps finite and >= 0 (else NORM_ERR_ARG).
 * Both: device pointers owned by the caller, 16-byte aligned (else
 *   NORM_ERR_ALIGN); outputs must not alias inputs; K % 64 == 0 with
 *   64 <= K <= NORM_MAX_N_FUSED, Nout % 32 == 0 with 32 <= Nout <= 2^20, and
 *   1 <= M <= 8388480 (65535 tiles of 128 rows), else NORM_ERR_SHAPE.
 *   norm_gemm_fwd moves x, wg and out with tiled tensor copies, whose
 *   descriptors take addresses this GPU reaches directly: each must be
 *   device memory of the current device (or managed memory), else
 *   NORM_ERR_MEMORY before anything is built or launched.
 *   Asynchronous on `stream`; a lost asynchronous copy or MMA surfaces
 *   through norm_get_device_error.
 */
norm_status_t norm_gemm_prepare(const void *w, const void *gamma, const void *beta,
                                int64_t K, int64_t Nout, norm_mode_t mode, void *wg,
                                float *u, float *v, norm_stream_t stream);

norm_status_t norm_gemm_fwd(const void *x, const void *wg, const float *u,
                            const float *v, int64_t M, int64_t K, int64_t Nout,
                            float eps, norm_mode_t mode, void *out, float *rstd,
                            float *mean, norm_stream_t stream);

/*
 * Plan tuning.  The first page names the split size and the number of
 * pipeline stages as what Inductor's autotuner searches for these kernels;
 * the library's default plan comes from a heuristic and a table measured
 * offline.  norm_tune_fwd / norm_tune_bwd measure, on the caller's buffers
 * and stream, every single-CTA plan of that pass (each threads-per-row
 * value that splits the row within the compiled chunk counts, rows per
 * group 1, 2, 4 or the heuristic's, the long-row kernels with 1 to 8 row
 * groups, and for the forward pass the plans with gamma/beta staged in
 * shared memory), each `iters` times after two warm-up
 * launches, and install the fastest in the process's plan cache for this
 * (device, mode, pass, M, N): later norm_fwd / norm_bwd calls of that shape
 * use it and norm_plan reports it (written to *chosen when not NULL).  Rows
 * that need a cluster keep their plan.  The outputs
 * hold the chosen plan's results.  The call blocks until its measurements
 * are done.
 *
 * A plan fixes the order of every floating-point reduction, so results are
 * bitwise reproducible for a given plan; tuning can change the plan (and so
 * the last bits of rstd, y, dx, dgamma, dbeta) from one process to the
 * next.  norm_tune_reset drops every cached plan, tuned or not.
 *
 * Arguments as norm_fwd / norm_bwd (the backward candidates are limited to
 * those whose partial rows fit workspace_bytes); iters in [1, 100000], else
 * NORM_ERR_ARG; NORM_ERR_ARG also when the GBNORM_PLAN override is set
 * (which bypasses the cache).
 */
norm_status_t norm_tune_fwd(const void *x, const void *gamma, const void *beta,
                            int64_t M, int64_t N, float eps, norm_mode_t mode,
                            void *y, float *rstd, float *mean, int iters,
                            norm_plan_t *chosen, norm_stream_t stream);

norm_status_t norm_tune_bwd(const void *dy, const void *x, const void *gamma,
                            const float *rstd, const float *mean, int64_t M,
                            int64_t N, norm_mode_t mode, void *dx,
                            float *dgamma, float *dbeta, void *workspace,
                            size_t workspace_bytes, int iters,
                            norm_plan_t *chosen, norm_stream_t stream);

norm_status_t norm_tune_reset(void);

/*
 * norm_bwd_noalloc -- norm_bwd for callers that cannot allocate device
 * memory.  (An addition of this library; the normalisation pages describe
 * no such entry point.)
 *
 * Some callers may not call cudaMalloc or any allocator at all: code whose
 * device memory is owned entirely by a framework's pool or a pre-reserved
 * arena, latency-critical paths where an allocation (which can synchronise
 * the device) is not acceptable, and plugin interfaces that are handed only
 * the input and output pointers.  This entry point takes exactly the
 * arguments of norm_bwd minus the workspace and uses, as its scratch space,
 * a fixed array of NORM_NOALLOC_WORKSPACE_BYTES (16 MiB) that the library
 * declares in device memory; every GPU that loads the library holds that
 * array until the process exits.  It calls no allocation routine.
 *
 *   - The scratch need is norm_bwd_workspace_bytes(M, N, mode) (the number
 *     of partial rows times N times 4 bytes, twice for LAYER).  Where the
 *     plan norm_bwd takes is the streaming long-row kernel (norm_plan's
 *     `streamed`, one partial row per cluster) and its need exceeds the
 *     array, this entry point runs the resident long-row plan instead (the
 *     plan norm_bwd takes under GBNORM_PLAN=stream=0); a shape whose need
 *     still exceeds NORM_NOALLOC_WORKSPACE_BYTES is rejected with
 *     NORM_ERR_WORKSPACE before anything is launched.
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - All calls on a device share the one array and it keeps the last
 *     call's contents.  Nothing in it needs clearing (each call writes
 *     every partial it later reads), but two calls that overlap on the GPU
 *     (different streams, or different host threads) race on it and must
 *     be serialised by the caller.
 */
#define NORM_NOALLOC_WORKSPACE_BYTES (16u << 20)

norm_status_t norm_bwd_noalloc(const void *dy, const void *x, const void *gamma,
                               const float *rstd, const float *mean,
                               int64_t M, int64_t N, norm_mode_t mode,
                               void *dx, float *dgamma, float *dbeta,
                               norm_stream_t stream);

/*
 * norm_selftest_wait_timeout -- exercises the failure path of the kernels'
 * bounded waits.  Launches one CTA whose thread waits, with the same
 * give-up logic as every wait in the library, on an mbarrier phase that
 * nothing completes, polling at most `polls` times (1 <= polls <= 2^20).
 * The wait gives up, the kernel records the timeout in the device error word
 * and returns normally, so the context stays usable.  A following
 * norm_get_device_error returns NORM_ERR_DEVICE_TIMEOUT (and clears it).
 * Asynchronous on `stream`; returns argument or launch errors.
 */
norm_status_t norm_selftest_wait_timeout(uint32_t polls, norm_stream_t stream);

/* Static, human-readable description of a status code. */
const char *norm_strerror(norm_status_t status);

/*
 * norm_get_device_error -- synchronises `stream`, then reads and clears the
 * current device's error word, which kernels set when one of their bounded
 * waits on an asynchronous copy gives up.  Returns NORM_OK or
 * NORM_ERR_DEVICE_TIMEOUT (or NORM_ERR_CUDA).
 */
norm_status_t norm_get_device_error(norm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBNORM_H */
