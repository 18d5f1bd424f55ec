// tiles.cuh -- issuing one tile of the shared-memory ring: bulk
// asynchronous copies of the tile's rows (the CTA's column slice of each)
// into stage s, completing on the stage's mbarrier.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace gbn {

// Forward: x (and, with RESID, the residual r at the next tensor slot of
// the stage).  Called by one thread.
template <bool CLUSTER, bool RESID = false>
__device__ __forceinline__ void issue_fwd_tile(const NormArgs &a, const SmemLayout &L,
                                               unsigned char *smem, int64_t tile, int s,
                                               int col0, int nsc_me, uint64_t pol) {
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off) + s;
  unsigned char *dst = smem + static_cast<size_t>(s) * L.stage_bytes;
  const int64_t row0 = tile * a.RT;
  const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
  const uint32_t nt = RESID ? 2u : 1u;
  if (!CLUSTER) {
    const uint32_t bytes = static_cast<uint32_t>(nrows) * a.N * 2u;
    mbar_arrive_expect_tx(full, nt * bytes);
    bulk_g2s(dst, a.x + row0 * a.N, bytes, full, pol);
    if (RESID) bulk_g2s(dst + L.tensor_bytes, a.res + row0 * a.N, bytes, full, pol);
  } else {
    // Row r of the tile lands at r * NS * 2 (slice stride), nsc_me chunks.
    const uint32_t bytes = static_cast<uint32_t>(nsc_me) * 16u;
    const uint32_t stride = static_cast<uint32_t>(a.NS) * 2u;
    mbar_arrive_expect_tx(full, nt * bytes * nrows);
    for (int r = 0; r < nrows; ++r) {
      bulk_g2s(dst + r * stride, a.x + (row0 + r) * a.N + col0, bytes, full, pol);
      if (RESID)
        bulk_g2s(dst + L.tensor_bytes + r * stride, a.res + (row0 + r) * a.N + col0, bytes,
                 full, pol);
    }
  }
}

// Issues tile `tile` into stage `s`: the rows' statistics with 4-byte
// cp.async copies (one completion arrival per lane), then x and dy (and,
// with RESID, dh at the third tensor slot) with bulk copies.  Must be called
// by all 32 lanes of one warp.
template <int MODE, bool CLUSTER, bool RESID = false>
__device__ __forceinline__ void issue_bwd_tile(const NormArgs &a, const SmemLayout &L,
                                               unsigned char *smem, int64_t tile, int s,
                                               int col0, int nsc_me, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off) + s;
  unsigned char *dst = smem + static_cast<size_t>(s) * L.stage_bytes;
  float *stats = reinterpret_cast<float *>(smem + L.stats_off) + static_cast<size_t>(s) * a.RT * 2;
  const int64_t row0 = tile * a.RT;
  const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
  for (int r = lane; r < nrows; r += 32) {
    cp_async_4(stats + 2 * r, a.rstd + row0 + r);
    if (MODE == kLayer) cp_async_4(stats + 2 * r + 1, a.mean + row0 + r);
  }
  cp_async_mbar_arrive(full);
  __syncwarp();
  if (lane == 0) {
    const uint32_t nt = RESID ? 3u : 2u;
    if (!CLUSTER) {
      const uint32_t bytes = static_cast<uint32_t>(nrows) * a.N * 2u;
      mbar_arrive_expect_tx(full, nt * bytes);
      bulk_g2s(dst, a.x + row0 * a.N, bytes, full, pol);
      bulk_g2s(dst + L.tensor_bytes, a.dy + row0 * a.N, bytes, full, pol);
      if (RESID) bulk_g2s(dst + 2 * L.tensor_bytes, a.res + row0 * a.N, bytes, full, pol);
    } else {
      const uint32_t bytes = static_cast<uint32_t>(nsc_me) * 16u;
      const uint32_t stride = static_cast<uint32_t>(a.NS) * 2u;
      mbar_arrive_expect_tx(full, nt * bytes * nrows);
      for (int r = 0; r < nrows; ++r) {
        const int64_t off = (row0 + r) * a.N + col0;
        bulk_g2s(dst + r * stride, a.x + off, bytes, full, pol);
        bulk_g2s(dst + L.tensor_bytes + r * stride, a.dy + off, bytes, full, pol);
        if (RESID) bulk_g2s(dst + 2 * L.tensor_bytes + r * stride, a.res + off, bytes, full, pol);
      }
    }
  }
}

// Backward epilogue: fold the column accumulators of the G row groups of this
// CTA in group order through shared memory (the ring is idle: every issued
// tile was consumed), then write one partial row slice (and one for dbeta)
// per CTA to the workspace.  Called by all threads.
template <int MODE, int K, bool EXACT>
__device__ __forceinline__ void write_column_partials(const NormArgs &a, unsigned char *smem,
                                                      const float2 (&accg)[K][4],
                                                      const float2 (&accb)[K][4], int g, int t,
                                                      int nsc_me, int64_t cid, int col0) {
  const int tid = threadIdx.x;
  __syncthreads();
  float *accs = reinterpret_cast<float *>(smem);  // [G][NS] dgamma, [G][NS] dbeta
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int c = t + k * a.tpr;
    if (c < nsc_me) {
      float4 *dg = reinterpret_cast<float4 *>(accs + static_cast<size_t>(g) * a.NS + c * 8);
      dg[0] = make_float4(accg[k][0].x, accg[k][0].y, accg[k][1].x, accg[k][1].y);
      dg[1] = make_float4(accg[k][2].x, accg[k][2].y, accg[k][3].x, accg[k][3].y);
      if (MODE == kLayer) {
        float4 *db = reinterpret_cast<float4 *>(accs + static_cast<size_t>(a.G + g) * a.NS + c * 8);
        db[0] = make_float4(accb[k][0].x, accb[k][0].y, accb[k][1].x, accb[k][1].y);
        db[1] = make_float4(accb[k][2].x, accb[k][2].y, accb[k][3].x, accb[k][3].y);
      }
    }
  }
  __syncthreads();
  const int nq = nsc_me * 2;       // float4s of this CTA's columns
  const int nq_stride = a.NS / 4;  // float4s per group row in shared memory
  const int nparts = (MODE == kLayer) ? 2 : 1;
  for (int w = 0; w < nparts; ++w) {
    const float4 *src = reinterpret_cast<const float4 *>(accs + static_cast<size_t>(w) * a.G * a.NS);
    float4 *dst = reinterpret_cast<float4 *>(a.ws + (static_cast<size_t>(w) * a.P + cid) * a.N + col0);
    for (int j = tid; j < nq; j += blockDim.x) {
      float4 acc = src[j];
      for (int q = 1; q < a.G; ++q) {
        const float4 v = src[static_cast<size_t>(q) * nq_stride + j];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      dst[j] = acc;
    }
  }
}

}  // namespace gbn
