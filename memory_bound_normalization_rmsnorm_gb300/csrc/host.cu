// host.cu -- forward + backward on host-resident tensors (norm_fwd_bwd_host
// in include/gbnorm.h): the rows are cut into chunks that stream through a
// few device buffers, with the host-to-device copies, the kernels and the
// device-to-host copies of different chunks on three streams, so the two
// copy directions and the compute overlap.  Only orchestration lives here;
// every step of the computation runs in the kernels behind norm_fwd /
// norm_bwd and the fixed-order partial reduction.
//
// dgamma / dbeta: each chunk's backward reduces its rows into one row of a
// [2][chunks][N] array (its own fixed-order partial sum), and a last
// reduction sums those rows in chunk order, so the result is bitwise
// reproducible for a given chunk size.
//
// rstd and mean of every row stay on the device until the last chunk is
// done and go back in one copy each: a copy has a fixed cost of several
// microseconds on the host link, which per chunk added up to more than the
// statistics' own bytes.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/gbnorm.h"
#include "common.cuh"

namespace gbn {
norm_status_t reduce_rows(const float *rows, int P, int n, float *dgamma, float *dbeta,
                          cudaStream_t s);
norm_status_t device_context(int *dev, int *sms, int *smem_optin, unsigned **err,
                             unsigned long long *ctx);
}

namespace {

constexpr int kDepth = 3;           // chunks in flight
constexpr int kMaxDev = 64;
constexpr size_t kAlign = 256;
constexpr size_t kChunkBytes = size_t(16) << 20;  // default: ~16 MB of x per chunk

size_t up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

struct Pipe {
  bool ready = false;
  unsigned long long ctx = 0;  // the context its streams and events belong to
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start, fin, end;
  cudaEvent_t in_done[kDepth], comp_done[kDepth], out_done[kDepth];
};
Pipe g_pipe[kMaxDev];
std::mutex g_pipe_mu[kMaxDev];

bool make_pipe(Pipe &p) {
  if (p.ready) return true;
  if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess)
    return false;
  cudaEvent_t *all[] = {&p.start, &p.fin, &p.end};
  for (cudaEvent_t *e : all)
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
  for (int i = 0; i < kDepth; ++i) {
    if (cudaEventCreateWithFlags(&p.in_done[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.comp_done[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.out_done[i], cudaEventDisableTiming) != cudaSuccess)
      return false;
  }
  p.ready = true;
  return true;
}

int64_t default_chunk_rows(int64_t M, int64_t N) {
  const int64_t r = std::max<int64_t>(1, static_cast<int64_t>(kChunkBytes) / (N * 2));
  return std::min(r, M);
}

// Byte layout of the device workspace.
struct Layout {
  int64_t R = 0, nch = 0;
  size_t gamma = 0, beta = 0, slot0 = 0, slot_bytes = 0, x = 0, dy = 0, y = 0, dx = 0,
         rstd = 0, mean = 0, bws = 0, bws_bytes = 0, rows = 0, dg = 0, db = 0, total = 0;
  // rstd / mean: [M] fp32 arrays of the whole call (not per slot)
};

norm_status_t layout(int64_t M, int64_t N, norm_mode_t mode, int64_t chunk_rows, Layout *L) {
  Layout l;
  l.R = chunk_rows > 0 ? std::min(chunk_rows, M) : default_chunk_rows(M, N);
  // a chunk's first row indexes the [M] statistics arrays, whose pointers the
  // kernels take 16-byte aligned: chunks start at multiples of 4 rows
  if (l.R < M) l.R = std::min(M, (l.R + 3) / 4 * 4);
  l.nch = (M + l.R - 1) / l.R;
  if (l.nch > (int64_t(1) << 20)) return NORM_ERR_SHAPE;
  size_t bws = 0;
  norm_status_t st = norm_bwd_workspace_bytes(l.R, N, mode, &bws);
  if (st != NORM_OK) return st;
  const size_t t = static_cast<size_t>(l.R) * N * 2, s = static_cast<size_t>(M) * 4;
  size_t off = 0;
  l.gamma = off; off = up(off + N * 2);
  l.beta = off; off = up(off + N * 2);
  l.rstd = off; off = up(off + s);
  l.mean = off; off = up(off + (mode == NORM_LAYER ? s : 0));
  l.x = 0; l.dy = up(t); l.y = l.dy + up(t); l.dx = l.y + up(t);
  l.slot_bytes = l.dx + up(t);
  l.slot0 = off; off += kDepth * l.slot_bytes;
  l.bws = off; l.bws_bytes = std::max<size_t>(bws, 16); off = up(off + l.bws_bytes);
  l.rows = off; off = up(off + size_t(2) * l.nch * N * 4);
  l.dg = off; off = up(off + N * 4);
  l.db = off; off = up(off + N * 4);
  l.total = off;
  *L = l;
  return NORM_OK;
}

}  // namespace

extern "C" {

norm_status_t norm_host_workspace_bytes(int64_t M, int64_t N, norm_mode_t mode,
                                        int64_t chunk_rows, size_t *bytes) {
  if (!bytes) return NORM_ERR_NULL;
  if (mode != NORM_RMS && mode != NORM_LAYER) return NORM_ERR_MODE;
  if (M < 1 || N < 8 || N > NORM_MAX_N || N % 8 || chunk_rows < 0) return NORM_ERR_SHAPE;
  Layout L;
  norm_status_t st = layout(M, N, mode, chunk_rows, &L);
  if (st != NORM_OK) return st;
  *bytes = L.total;
  return NORM_OK;
}

norm_status_t norm_fwd_bwd_host(const void *x, const void *dy, const void *gamma,
                                const void *beta, int64_t M, int64_t N, float eps,
                                norm_mode_t mode, void *y, void *dx, float *rstd, float *mean,
                                float *dgamma, float *dbeta, int64_t chunk_rows,
                                void *workspace, size_t workspace_bytes,
                                norm_stream_t stream) {
  if (!x || !dy || !gamma || !y || !dx || !rstd || !dgamma) return NORM_ERR_NULL;
  if (mode != NORM_RMS && mode != NORM_LAYER) return NORM_ERR_MODE;
  if (M < 1 || N < 8 || N > NORM_MAX_N || N % 8 || chunk_rows < 0) return NORM_ERR_SHAPE;
  if (mode == NORM_RMS && (beta || mean || dbeta)) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && !mean) return NORM_ERR_MODE;
  if (!(eps >= 0.0f) || !(eps <= 3.4e38f)) return NORM_ERR_ARG;
  Layout L;
  norm_status_t st = layout(M, N, mode, chunk_rows, &L);
  if (st != NORM_OK) return st;
  if (!workspace || workspace_bytes < L.total) return NORM_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return NORM_ERR_ALIGN;
  int dev = 0, sms = 0, optin = 0;
  unsigned *err = nullptr;
  unsigned long long ctx = 0;
  if ((st = gbn::device_context(&dev, &sms, &optin, &err, &ctx)) != NORM_OK) return st;
  if (dev >= kMaxDev) return NORM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
  Pipe &P = g_pipe[dev];
  // Streams and events of a destroyed context (cudaDeviceReset) went with
  // it: make new ones.
  if (P.ready && P.ctx != ctx) P = Pipe();
  P.ctx = ctx;
  if (!make_pipe(P)) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  const bool ln = mode == NORM_LAYER;
  const unsigned char *hx = static_cast<const unsigned char *>(x);
  const unsigned char *hdy = static_cast<const unsigned char *>(dy);
  unsigned char *hy = static_cast<unsigned char *>(y);
  unsigned char *hdx = static_cast<unsigned char *>(dx);
  float *rows = reinterpret_cast<float *>(ws + L.rows);
  const size_t row_bytes = static_cast<size_t>(N) * 2;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };

  // Nothing of this call starts before earlier work on `stream`.
  chk(cudaEventRecord(P.start, cs));
  chk(cudaStreamWaitEvent(P.h2d, P.start, 0));
  chk(cudaStreamWaitEvent(P.d2h, P.start, 0));
  chk(cudaMemcpyAsync(ws + L.gamma, gamma, N * 2, h2d, P.h2d));
  if (ln && beta) chk(cudaMemcpyAsync(ws + L.beta, beta, N * 2, h2d, P.h2d));
  const void *dbeta_dev = (ln && beta) ? ws + L.beta : nullptr;

  for (int64_t c = 0; c < L.nch && ok; ++c) {
    const int s = static_cast<int>(c % kDepth);
    const int64_t r0 = c * L.R, nr = std::min(L.R, M - r0);
    unsigned char *slot = ws + L.slot0 + s * L.slot_bytes;
    const size_t bytes = static_cast<size_t>(nr) * row_bytes, off = r0 * row_bytes;
    // inputs: the slot's previous chunk must be done computing
    if (c >= kDepth) chk(cudaStreamWaitEvent(P.h2d, P.comp_done[s], 0));
    chk(cudaMemcpyAsync(slot + L.x, hx + off, bytes, h2d, P.h2d));
    chk(cudaMemcpyAsync(slot + L.dy, hdy + off, bytes, h2d, P.h2d));
    chk(cudaEventRecord(P.in_done[s], P.h2d));
    // compute: inputs in, and the slot's previous outputs copied out
    chk(cudaStreamWaitEvent(cs, P.in_done[s], 0));
    if (c >= kDepth) chk(cudaStreamWaitEvent(cs, P.out_done[s], 0));
    float *rs = reinterpret_cast<float *>(ws + L.rstd) + r0;
    float *mu = ln ? reinterpret_cast<float *>(ws + L.mean) + r0 : nullptr;
    st = norm_fwd(slot + L.x, ws + L.gamma, dbeta_dev, nr, N, eps, mode, slot + L.y, rs, mu,
                  stream);
    if (st != NORM_OK) return st;
    st = norm_bwd(slot + L.dy, slot + L.x, ws + L.gamma, rs, mu, nr, N, mode, slot + L.dx,
                  rows + c * N, ln ? rows + (L.nch + c) * N : nullptr, ws + L.bws, L.bws_bytes,
                  stream);
    if (st != NORM_OK) return st;
    chk(cudaEventRecord(P.comp_done[s], cs));
    // outputs
    chk(cudaStreamWaitEvent(P.d2h, P.comp_done[s], 0));
    chk(cudaMemcpyAsync(hy + off, slot + L.y, bytes, d2h, P.d2h));
    chk(cudaMemcpyAsync(hdx + off, slot + L.dx, bytes, d2h, P.d2h));
    chk(cudaEventRecord(P.out_done[s], P.d2h));
  }
  if (!ok) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  // chunk rows -> dgamma / dbeta in chunk order, then to the host
  float *dg = reinterpret_cast<float *>(ws + L.dg);
  float *db = ln ? reinterpret_cast<float *>(ws + L.db) : nullptr;
  st = gbn::reduce_rows(rows, static_cast<int>(L.nch), static_cast<int>(N), dg, db, cs);
  if (st != NORM_OK) return st;
  chk(cudaEventRecord(P.fin, cs));
  chk(cudaStreamWaitEvent(P.d2h, P.fin, 0));
  chk(cudaMemcpyAsync(dgamma, dg, N * 4, d2h, P.d2h));
  if (ln && dbeta) chk(cudaMemcpyAsync(dbeta, db, N * 4, d2h, P.d2h));
  chk(cudaMemcpyAsync(rstd, ws + L.rstd, M * 4, d2h, P.d2h));
  if (ln) chk(cudaMemcpyAsync(mean, ws + L.mean, M * 4, d2h, P.d2h));
  // `stream` ends after the last copy
  chk(cudaEventRecord(P.end, P.d2h));
  chk(cudaStreamWaitEvent(cs, P.end, 0));
  if (!ok) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  return NORM_OK;
}

}  // extern "C"
