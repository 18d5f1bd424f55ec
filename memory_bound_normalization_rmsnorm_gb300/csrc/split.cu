// split.cu -- the multi-CTA two-pass path for rows too long for one
// thread-block cluster (more columns than 16 CTAs hold in registers or
// shared memory).
//
// "PyTorch atinge desempenho SOTA em normalizacao com torch.compile"
// (matsubara.tec.br) contrasts the persistent reduction, which keeps a whole
// row on chip, with the looped reduction that walks a long row in pieces,
// and names very large dimensions as where generated kernels regress.  Here
// each row is cut into segments of NS columns (the last one ragged) and a
// persistent grid walks units of (segment, RT consecutive rows); a CTA takes
// one contiguous, balanced range of units in segment-major order, so it
// stays on one or two segments and reads its rows' slices of them through
// the same bulk-copy ring as the one-pass kernels.  The row reduction
// becomes two passes joined by a per-row fold:
//
//   forward   1. statistics of each (row, segment): sum x^2 (RMSNorm), or
//               the segment's mean and sum of squared deviations from it
//               (LayerNorm, two-pass inside the segment), written into the
//               row's own output y as scratch (the forward takes no
//               workspace; y is overwritten by step 3);
//             2. one warp per row folds the row's segment partials in a
//               fixed order (Chan's merge for LayerNorm) into rstd and mean;
//             3. y = (x - mean) * rstd * gamma + beta per unit.
//   backward  1. per (row, segment): sum g and sum g * xhat, with the saved
//               rstd / mean (g = dy * gamma), into the workspace;
//             2. one warp per row folds them into the row's totals;
//             3. dx per unit, and dgamma / dbeta accumulated in registers
//               for the CTA's current segment; when its range moves to the
//               next segment (and at the end) the row groups add their sums
//               in group order into the CTA's slot of that segment;
//             4. a fixed-order reduction of the slots: for the columns of
//               segment s, the slots of the CTAs whose ranges touch s, in
//               CTA order.
// Every pass reads its tiles from HBM (or L2 when the tensors fit): x is read
// twice by the forward, x and dy twice by the backward.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"

namespace gbn {

namespace {

// Shared-memory layout of a split-path kernel: S stages of NT tensors, then
// per stage and row of a tile four floats of row data (rstd, mean and, for
// the backward dx pass, the row's two dot-product totals), the cross-warp
// scratch of the group sums, the stage mbarriers and the flags.
__host__ __device__ inline SmemLayout split_layout(int RT, int NS, int S, int G, int tpr,
                                                   int ntensors) {
  SmemLayout L;
  L.tensor_bytes = static_cast<uint32_t>(RT) * static_cast<uint32_t>(NS) * 2u;
  L.stage_bytes = L.tensor_bytes * static_cast<uint32_t>(ntensors);
  uint32_t off = L.stage_bytes * static_cast<uint32_t>(S);
  L.par_off = off;
  L.stats_off = off;
  off = align16(off + static_cast<uint32_t>(S * RT * 4) * 4u);
  L.red_off = off;
  if (tpr > 32) off = align16(off + static_cast<uint32_t>(2 * G * (tpr / 32) * 4) * 4u);
  L.xch_off = off;
  L.bar_off = off;
  off = align16(off + static_cast<uint32_t>(S) * 8u);
  L.flag_off = off;
  off = align16(off + 4u + 4u * static_cast<uint32_t>(S));
  L.total = off;
  return L;
}

// Unit u of the walk: segment u / T, row tile u % T (T = a.ntiles row
// tiles).  The range of CTA b of `grid` CTAs is [U b / grid, U (b+1) / grid).
__device__ __forceinline__ int64_t unit_begin(int64_t U, int64_t b, int64_t grid) {
  return U * b / grid;
}

// L2 policy of the first read of a tensor on this path (its second read
// comes one kernel later and may still find it in L2) and of the last.
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Segment and row tile of a unit, advanced without division.
struct UnitPos {
  int64_t seg, rt;
};
__device__ __forceinline__ void unit_advance(UnitPos &p, int64_t by, int64_t T) {
  p.rt += by;
  while (p.rt >= T) {
    p.rt -= T;
    ++p.seg;
  }
}

// Issues the unit at `pos` into stage s: the tile's row slices of x (and
// dy), each one bulk copy, and for the passes that need them the rows' saved
// statistics (and the backward's dot-product totals) by 4-byte copies.
// Called by all 32 lanes of one warp.
template <int MODE, int PHASE>
__device__ __forceinline__ void issue_unit(const NormArgs &a, const SmemLayout &L,
                                           unsigned char *smem, UnitPos pos, int s,
                                           uint64_t pol) {
  constexpr int NT = PHASE >= kSplitBwdDots ? 2 : 1;
  const int lane = threadIdx.x & 31;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off) + s;
  unsigned char *dst = smem + static_cast<size_t>(s) * L.stage_bytes;
  const int64_t seg = pos.seg;
  const int64_t row0 = pos.rt * a.RT;
  const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
  const int64_t col0 = seg * a.NS;
  const int nsc_me = static_cast<int>(min64(a.nsc, a.N / 8 - seg * a.nsc));
  if (PHASE != kSplitFwdStats) {
    float *st = reinterpret_cast<float *>(smem + L.stats_off) + static_cast<size_t>(s) * a.RT * 4;
    for (int r = lane; r < nrows; r += 32) {
      cp_async_4(st + 4 * r, a.rstd + row0 + r);
      if (MODE == kLayer) cp_async_4(st + 4 * r + 1, a.mean + row0 + r);
      if (PHASE == kSplitBwdDx) {
        cp_async_4(st + 4 * r + 2, a.rowt + 2 * (row0 + r));
        cp_async_4(st + 4 * r + 3, a.rowt + 2 * (row0 + r) + 1);
      }
    }
    cp_async_mbar_arrive(full);
  }
  __syncwarp();
  if (lane == 0) {
    const uint32_t bytes = static_cast<uint32_t>(nsc_me) * 16u;
    const uint32_t stride = static_cast<uint32_t>(a.NS) * 2u;
    mbar_arrive_expect_tx(full, NT * bytes * static_cast<uint32_t>(nrows));
    for (int r = 0; r < nrows; ++r) {
      const int64_t off = (row0 + r) * a.N + col0;
      bulk_g2s(dst + r * stride, a.x + off, bytes, full, pol);
      if (NT == 2) bulk_g2s(dst + L.tensor_bytes + r * stride, a.dy + off, bytes, full, pol);
    }
  }
}

// One pass of the split path (PHASE: kSplitFwdStats, kSplitFwdOut,
// kSplitBwdDots, kSplitBwdDx) over this CTA's range of units.  Row groups of
// tpr threads, K 16-byte chunks per thread: NS = tpr * K * 8 columns.
template <int MODE, int PHASE, int K>
__global__ void __launch_bounds__(kMaxThreads, 1) norm_split_kernel(const NormArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NT = PHASE >= kSplitBwdDots ? 2 : 1;
  const SmemLayout L = split_layout(a.RT, a.NS, a.S, a.G, a.tpr, NT);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag_off);
  int *done_cnt = reinterpret_cast<int *>(smem + L.flag_off) + 1;

  const int tid = threadIdx.x;
  const int g = tid / a.tpr;
  const int t = tid - g * a.tpr;
  const int nwarps = blockDim.x >> 5;
  const int64_t T = a.ntiles;
  const int64_t U = T * a.nseg;
  const int64_t u0 = unit_begin(U, blockIdx.x, gridDim.x);
  const int64_t u1 = unit_begin(U, blockIdx.x + 1, gridDim.x);

  if (tid == 0) {
    for (int s = 0; s < a.S; ++s) {
      mbar_init(full + s, 1);
      done_cnt[s] = 0;
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Programmatic dependent launch, as in the one-pass kernels.
  grid_launch_dependents();
  grid_dependency_wait();

  const uint64_t pol = (PHASE == kSplitFwdStats || PHASE == kSplitBwdDots)
                           ? l2_evict_normal_policy()
                           : l2_evict_first_policy();
  // position of the first unit (one division per CTA), then advanced
  UnitPos first;
  first.seg = u0 / T;
  first.rt = u0 - first.seg * T;
  if (tid < 32) {
    __syncwarp();
    UnitPos ip = first;
    for (int j = 0; j < a.S; ++j) {
      if (u0 + j < u1) issue_unit<MODE, PHASE>(a, L, smem, ip, j, pol);
      unit_advance(ip, 1, T);
    }
  }

  // Per-segment state: gamma (fp32 pairs) and beta (packed) of this
  // thread's chunks, and for the dx pass the column accumulators.
  float2 gf[K][4], accg[K][4], accb[K][4];
  uint4 bv[K];
  int64_t cur = -1;   // segment the state belongs to
  int nsc_me = 0;     // chunks of that segment
  const float invN = a.invN;

  // dgamma / dbeta of segment `seg` accumulated by this CTA: the G row
  // groups add their sums into slot (blockIdx.x + seg) one group at a time
  // (a CTA barrier orders each group's global writes before the next
  // group's reads), so the slot gets them in group order.
  auto flush = [&](int64_t seg) {
    const int64_t nslots = static_cast<int64_t>(gridDim.x) + a.nseg;
    float *sg = a.ws + (static_cast<int64_t>(blockIdx.x) + seg) * a.NS;
    float *sb = a.ws + (nslots + static_cast<int64_t>(blockIdx.x) + seg) * a.NS;
    for (int gg = 0; gg < a.G; ++gg) {
      __syncthreads();
      if (g == gg) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int c = t + k * a.tpr;
          if (c < nsc_me) {
            float4 *dg = reinterpret_cast<float4 *>(sg + c * 8);
            float4 v0 = make_float4(accg[k][0].x, accg[k][0].y, accg[k][1].x, accg[k][1].y);
            float4 v1 = make_float4(accg[k][2].x, accg[k][2].y, accg[k][3].x, accg[k][3].y);
            if (gg > 0) {
              const float4 o0 = dg[0], o1 = dg[1];
              v0 = make_float4(o0.x + v0.x, o0.y + v0.y, o0.z + v0.z, o0.w + v0.w);
              v1 = make_float4(o1.x + v1.x, o1.y + v1.y, o1.z + v1.z, o1.w + v1.w);
            }
            dg[0] = v0;
            dg[1] = v1;
            if (MODE == kLayer) {
              float4 *db = reinterpret_cast<float4 *>(sb + c * 8);
              float4 w0 = make_float4(accb[k][0].x, accb[k][0].y, accb[k][1].x, accb[k][1].y);
              float4 w1 = make_float4(accb[k][2].x, accb[k][2].y, accb[k][3].x, accb[k][3].y);
              if (gg > 0) {
                const float4 o0 = db[0], o1 = db[1];
                w0 = make_float4(o0.x + w0.x, o0.y + w0.y, o0.z + w0.z, o0.w + w0.w);
                w1 = make_float4(o1.x + w1.x, o1.y + w1.y, o1.z + w1.z, o1.w + w1.w);
              }
              db[0] = w0;
              db[1] = w1;
            }
          }
        }
      }
    }
    __syncthreads();
  };

  __syncthreads();
  int rpar = 0;
  int s = 0;
  uint32_t par = 0;
  UnitPos pos = first;
  for (int64_t u = u0; u < u1; ++u, unit_advance(pos, 1, T)) {
    const int64_t seg = pos.seg;
    if (seg != cur) {
      if (PHASE == kSplitBwdDx && cur >= 0) flush(cur);
      cur = seg;
      nsc_me = static_cast<int>(min64(a.nsc, a.N / 8 - seg * a.nsc));
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int c = t + k * a.tpr;
        uint4 gv = make_uint4(0, 0, 0, 0);
        bv[k] = make_uint4(0, 0, 0, 0);
        if (PHASE != kSplitFwdStats && c < nsc_me) {
          gv = ld_global_nc_v4(a.gamma + seg * a.NS + c * 8);
          if (PHASE == kSplitFwdOut && MODE == kLayer && a.beta != nullptr)
            bv[k] = ld_global_nc_v4(a.beta + seg * a.NS + c * 8);
        }
        chunk_to_f2(gv, gf[k]);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          accg[k][p] = splat2(0.f);
          accb[k][p] = splat2(0.f);
        }
      }
    }
    mbar_wait(full + s, par, a.err, abort_flag);
    const int64_t row0 = pos.rt * a.RT;
    const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
    const unsigned char *stx = smem + static_cast<size_t>(s) * L.stage_bytes;
    const float *stats = reinterpret_cast<const float *>(smem + L.stats_off) +
                         static_cast<size_t>(s) * a.RT * 4;

    for (int q = 0; q < a.rpg; ++q) {
      const int r = g + q * a.G;
      const bool active = r < nrows;
      const unsigned char *rowp = stx + static_cast<size_t>(r) * a.NS * 2 + t * 16;
      float2 xf[K][4];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const bool ok = active && t + k * a.tpr < nsc_me;
        const uint4 v = ok ? *reinterpret_cast<const uint4 *>(rowp + k * a.tpr * 16)
                           : make_uint4(0, 0, 0, 0);
        chunk_to_f2(v, xf[k]);
      }

      if (PHASE == kSplitFwdStats) {
        // The row's partial over this segment, into y's own row as scratch.
        float *scratch = reinterpret_cast<float *>(a.out + (row0 + r) * a.N);
        if (MODE == kRMS) {
          float2 q0 = splat2(0.f), q1 = splat2(0.f);
#pragma unroll
          for (int k = 0; k < K; ++k) {
            q0 = fma2(xf[k][0], xf[k][0], fma2(xf[k][1], xf[k][1], q0));
            q1 = fma2(xf[k][2], xf[k][2], fma2(xf[k][3], xf[k][3], q1));
          }
          const float2 qt = add2(q0, q1);
          float v[1] = {qt.x + qt.y};
          group_sum<1, true>(v, a.tpr, g, a.G, t, red, rpar);
          if (active && t == 0) scratch[seg] = v[0];
        } else {
          // two passes inside the segment: its mean, then the sum of
          // squared deviations from it over the owned chunks
          float2 acc = splat2(0.f);
#pragma unroll
          for (int k = 0; k < K; ++k)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc = add2(acc, xf[k][p]);
          float v1[1] = {acc.x + acc.y};
          group_sum<1, true>(v1, a.tpr, g, a.G, t, red, rpar);
          const float mseg = v1[0] / static_cast<float>(nsc_me * 8);
          const float2 nm = splat2(-mseg);
          float2 q2 = splat2(0.f);
#pragma unroll
          for (int k = 0; k < K; ++k) {
            if (t + k * a.tpr < nsc_me) {
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const float2 d = add2(xf[k][p], nm);
                q2 = fma2(d, d, q2);
              }
            }
          }
          float v2[1] = {q2.x + q2.y};
          group_sum<1, true>(v2, a.tpr, g, a.G, t, red, rpar);
          if (active && t == 0)
            reinterpret_cast<float2 *>(scratch)[seg] = make_float2(mseg, v2[0]);
        }
      } else if (PHASE == kSplitFwdOut) {
        if (active) {
          const float rs = stats[4 * r];
          const float mu = MODE == kLayer ? stats[4 * r + 1] : 0.f;
          const float2 rs2 = splat2(rs), nmu = splat2(-mu);
          uint16_t *yrow = a.out + (row0 + r) * a.N + seg * a.NS + t * 8;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            if (t + k * a.tpr < nsc_me) {
              float2 o[4], bf[4];
              if (MODE == kLayer) chunk_to_f2(bv[k], bf);
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const float2 xh = mul2(MODE == kLayer ? add2(xf[k][p], nmu) : xf[k][p], rs2);
                o[p] = MODE == kLayer ? fma2(xh, gf[k][p], bf[p]) : mul2(xh, gf[k][p]);
              }
              st_global_cs_v4(yrow + k * a.tpr * 8, f2_to_chunk(o));
            }
          }
        }
      } else {
        // backward passes: xhat and g = dy * gamma of the owned chunks
        const float rs = active ? stats[4 * r] : 0.f;
        const float mu = (active && MODE == kLayer) ? stats[4 * r + 1] : 0.f;
        const float2 rs2 = splat2(rs), nmu = splat2(-mu);
        float2 xh[K][4], gg[K][4], df[K][4];
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const bool ok = active && t + k * a.tpr < nsc_me;
          const uint4 dv = ok ? *reinterpret_cast<const uint4 *>(rowp + L.tensor_bytes +
                                                                 k * a.tpr * 16)
                              : make_uint4(0, 0, 0, 0);
          chunk_to_f2(dv, df[k]);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            xh[k][p] = mul2(MODE == kLayer ? add2(xf[k][p], nmu) : xf[k][p], rs2);
            gg[k][p] = mul2(df[k][p], gf[k][p]);
          }
        }
        if (PHASE == kSplitBwdDots) {
          float2 s1 = splat2(0.f), s2 = splat2(0.f);
#pragma unroll
          for (int k = 0; k < K; ++k)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              s1 = add2(s1, gg[k][p]);
              s2 = fma2(gg[k][p], xh[k][p], s2);
            }
          float v[2] = {s1.x + s1.y, s2.x + s2.y};
          group_sum<2, true>(v, a.tpr, g, a.G, t, red, rpar);
          if (active && t == 0)
            reinterpret_cast<float2 *>(a.rowp)[(row0 + r) * a.nseg + seg] = make_float2(v[0], v[1]);
        } else if (active) {
          // dx = rstd (g - a - xhat c) = rstd g - rstd a - (rstd c) xhat
          const float2 nra = splat2(MODE == kLayer ? -rs * (stats[4 * r + 2] * invN) : 0.f);
          const float2 nrc = splat2(-rs * (stats[4 * r + 3] * invN));
          uint16_t *dxrow = a.out + (row0 + r) * a.N + seg * a.NS + t * 8;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            if (t + k * a.tpr < nsc_me) {
              float2 o[4];
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                o[p] = fma2(xh[k][p], nrc,
                            MODE == kLayer ? fma2(gg[k][p], rs2, nra) : mul2(gg[k][p], rs2));
                accg[k][p] = fma2(df[k][p], xh[k][p], accg[k][p]);
                if (MODE == kLayer) accb[k][p] = add2(accb[k][p], df[k][p]);
              }
              st_global_cs_v4(dxrow + k * a.tpr * 8, f2_to_chunk(o));
            }
          }
        }
      }
    }

    // This warp is done with the stage; the last warp refills it.
    if (last_warp_done(done_cnt, s, nwarps)) {
      const int64_t next = u + a.S;
      if (next < u1) {
        if ((tid & 31) == 0) fence_proxy_async_smem();
        __syncwarp();
        UnitPos np = pos;
        unit_advance(np, a.S, T);
        issue_unit<MODE, PHASE>(a, L, smem, np, s, pol);
      }
    }
    if (++s == a.S) {
      s = 0;
      par ^= 1u;
    }
  }
  if (PHASE == kSplitBwdDx && cur >= 0) flush(cur);
}

// Fold of a row's segment partials, one warp per row, in a fixed order: each
// lane folds segments lane, lane + 32, ... in increasing order, then the
// lanes combine by a butterfly (for LayerNorm Chan's merge with the lower
// lane's partial first, so both partners compute the same bits).
//   forward:  RMSNorm sums the segments' sum x^2; LayerNorm merges their
//             (count, mean, M2).  Writes rstd (and mean).  The partials are
//             read from the row of y where the statistics pass left them.
//   backward: sums the (sum g, sum g * xhat) pairs into the row's totals.
template <int MODE, bool BWD>
__global__ void __launch_bounds__(256) norm_split_fold_kernel(const NormArgs a) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= a.M) return;
  const int nseg = a.nseg;
  if (BWD) {
    const float2 *p = reinterpret_cast<const float2 *>(a.rowp) + row * nseg;
    float s1 = 0.f, s2 = 0.f;
    for (int sg = lane; sg < nseg; sg += 32) {
      const float2 v = p[sg];
      s1 += v.x;
      s2 += v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    if (lane == 0) {
      a.rowt[2 * row] = s1;
      a.rowt[2 * row + 1] = s2;
    }
    return;
  }
  const float *p = reinterpret_cast<const float *>(a.out + row * a.N);
  if (MODE == kRMS) {
    float acc = 0.f;
    for (int sg = lane; sg < nseg; sg += 32) acc += p[sg];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.rstd[row] = rsqrtf(acc * a.invN + a.eps);
  } else {
    const float2 *p2 = reinterpret_cast<const float2 *>(p);
    float n = 0.f, m = 0.f, q = 0.f;
    for (int sg = lane; sg < nseg; sg += 32) {
      const float ns = static_cast<float>(sg == nseg - 1 ? a.N - sg * a.NS : a.NS);
      const float2 v = p2[sg];
      nms_merge(n, m, q, ns, v.x, v.y);
    }
    int rpar = 0;
    group_nmeanvar(n, m, q, 32, 0, 1, lane, nullptr, rpar);
    if (lane == 0) {
      a.mean[row] = m;
      a.rstd[row] = rsqrtf(q * a.invN + a.eps);
    }
  }
}

// dgamma (blockIdx.y = 0) and dbeta (blockIdx.y = 1) from the slots of the
// dx pass: columns j of segment s get the slots (b + s) of the CTAs b whose
// unit ranges touch segment s, added in increasing b.  Each thread owns 4
// consecutive columns (NS is a multiple of 8, so they share a segment).
__global__ void __launch_bounds__(256) norm_split_reduce_kernel(const NormArgs a, int grid,
                                                                float *dgamma, float *dbeta) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int64_t col = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (col >= a.N) return;
  const int64_t T = a.ntiles;
  const int64_t U = T * a.nseg;
  const int64_t seg = col / a.NS;
  const int64_t j = col - seg * a.NS;
  // CTA whose range holds unit v: floor(((v + 1) grid - 1) / U)
  const int64_t b_lo = ((seg * T + 1) * grid - 1) / U;
  const int64_t b_hi = (((seg + 1) * T) * grid - 1) / U;
  const int64_t nslots = static_cast<int64_t>(grid) + a.nseg;
  const float *src = a.ws + (blockIdx.y ? nslots * a.NS : 0);
  float4 acc = *reinterpret_cast<const float4 *>(src + (b_lo + seg) * a.NS + j);
  for (int64_t b = b_lo + 1; b <= b_hi; ++b) {
    const float4 v = *reinterpret_cast<const float4 *>(src + (b + seg) * a.NS + j);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  *reinterpret_cast<float4 *>((blockIdx.y ? dbeta : dgamma) + col) = acc;
}

template <int MODE>
const void *pick_split(int phase, int K) {
  switch (phase) {
    case kSplitFwdStats:
      return K == 4 ? reinterpret_cast<const void *>(&norm_split_kernel<MODE, kSplitFwdStats, 4>)
                    : nullptr;
    case kSplitFwdOut:
      return K == 4 ? reinterpret_cast<const void *>(&norm_split_kernel<MODE, kSplitFwdOut, 4>)
                    : nullptr;
    case kSplitBwdDots:
      return K == 4 ? reinterpret_cast<const void *>(&norm_split_kernel<MODE, kSplitBwdDots, 4>)
                    : nullptr;
    case kSplitBwdDx:
      return K == 2 ? reinterpret_cast<const void *>(&norm_split_kernel<MODE, kSplitBwdDx, 2>)
                    : nullptr;
    default:
      return nullptr;
  }
}

}  // namespace

const void *split_kernel_ptr(int mode, int phase, int K) {
  return mode == kRMS ? pick_split<kRMS>(phase, K) : pick_split<kLayer>(phase, K);
}

const void *split_fold_kernel_ptr(int mode, bool bwd) {
  if (mode == kRMS)
    return bwd ? reinterpret_cast<const void *>(&norm_split_fold_kernel<kRMS, true>)
               : reinterpret_cast<const void *>(&norm_split_fold_kernel<kRMS, false>);
  return bwd ? reinterpret_cast<const void *>(&norm_split_fold_kernel<kLayer, true>)
             : reinterpret_cast<const void *>(&norm_split_fold_kernel<kLayer, false>);
}

const void *split_reduce_kernel_ptr() {
  return reinterpret_cast<const void *>(&norm_split_reduce_kernel);
}

SmemLayout split_smem_layout(int RT, int NS, int S, int G, int tpr, int ntensors) {
  return split_layout(RT, NS, S, G, tpr, ntensors);
}

}  // namespace gbn
