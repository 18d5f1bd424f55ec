// long_kernel.cuh -- forward and backward kernels for long rows, included
// by the translation units that instantiate them (long.cu: plain, and
// long_resid.cu: fused residual add).
//
// Same pipeline as fwd.cu / bwd.cu (persistent grid, bulk-copy ring of S
// stages, last-warp refill, fixed-order reductions, cluster column split
// with DSMEM pushes), with two differences:
//   - the row slice is NOT copied into registers: it is read from the
//     shared-memory stage twice (statistics or dot products, then outputs),
//     so registers hold only per-column state (gamma, beta, the dgamma/dbeta
//     accumulators) and a CTA can own a wide slice (up to 8 chunks of 8
//     columns per thread);
//   - in a cluster the cross-CTA exchange is software-pipelined: the partial
//     of the current tile's row is pushed to the peers, and only then is the
//     previous tile finished (wait for its exchange, outputs, stage
//     release), so the DSMEM round trip overlaps a full statistics pass.
// LayerNorm statistics use one exchange round of (count, mean, M2) merges.
//
// What is computed follows the same page paragraphs as fwd.cu and bwd.cu
// ("PyTorch atinge desempenho SOTA em normalizacao com torch.compile":
// LayerNorm/RMSNorm definitions, forward reduction + pointwise pass, fused
// backward with split column reduction).
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"
#include "tiles.cuh"

namespace gbn {


__device__ __forceinline__ uint4 lds_chunk(const unsigned char *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

// State of a tile whose statistics are pushed but whose outputs are not
// written yet.
struct Pending {
  int64_t tile;
  int s;
  float a, b, c;  // this row group's partial (also the total without a cluster)
};

// RESID: fused residual add -- the stage also holds r; the statistics pass
// forms h = bf16(x + r) (sum in binary32, round to nearest even), writes it
// over x in the stage, and the output pass writes h out beside y.
// OUT: bf16 y (kOutBf16), or E4M3 codes with a per-row scale (kOutFp8Row:
// RMSNorm's amax is rstd times the largest |x gamma|, taken in the
// statistics pass; LayerNorm's needs y, and in a cluster the CTAs' slice
// maxima of a row travel in the next row's exchange round, so its codes are
// written one round later) or with per-32-column E8M0 exponents
// (kOutFp8Mx; slices start on a block).
template <int MODE, int K, bool CLUSTER, bool EXACT, bool RESID, int OUT = kOutBf16>
__global__ void __launch_bounds__(kMaxThreads, 1) norm_fwd_long_kernel(const NormArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout L = make_layout(a.RT, a.NS, a.S, a.G, a.tpr, RESID ? 2 : 1, false, a.C);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag_off);
  int *done_cnt = reinterpret_cast<int *>(smem + L.flag_off) + 1;

  const int tid = threadIdx.x;
  const int g = tid / a.tpr;
  const int t = tid - g * a.tpr;
  const int nwarps = blockDim.x >> 5;
  const int crank = CLUSTER ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t cid = CLUSTER ? static_cast<int64_t>(cluster_id_x()) : blockIdx.x;
  const int64_t ncl = CLUSTER ? static_cast<int64_t>(ncluster_x()) : gridDim.x;
  const int col0 = crank * a.NS;
  const int nsc_me = min(a.nsc, a.N / 8 - crank * a.nsc);

  if (tid == 0) {
    for (int s = 0; s < a.S; ++s) {
      mbar_init(full + s, 1);
      done_cnt[s] = 0;
    }
    if (CLUSTER) {
      uint64_t *xb = xch_bars(smem, L, a.RT, a.C);
      for (int b = 0; b < kXchBuffers; ++b) mbar_init(xb + b, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Programmatic dependent launch: let the next kernel in the stream start
  // its prologue as our CTAs retire, and touch no global memory before the
  // previous kernel's writes are complete and visible.
  grid_launch_dependents();
  grid_dependency_wait();

  // Per-column state: gamma and beta of this thread's chunks, packed bf16.
  uint4 gv[K], bv[K];
  int nown = 0;  // chunks this thread owns
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int c = t + k * a.tpr;
    gv[k] = make_uint4(0, 0, 0, 0);
    bv[k] = make_uint4(0, 0, 0, 0);
    if (c < nsc_me) {
      ++nown;
      gv[k] = ld_global_nc_v4(a.gamma + col0 + c * 8);
      if (MODE == kLayer && a.beta != nullptr) bv[k] = ld_global_nc_v4(a.beta + col0 + c * 8);
    }
  }

  if (CLUSTER) cluster_sync(); else __syncthreads();

  const uint64_t pol = l2_evict_first_policy();
  if (tid == 0) {
    for (int j = 0; j < a.S; ++j) {
      const int64_t tile = cid + j * ncl;
      if (tile < a.ntiles) issue_fwd_tile<CLUSTER, RESID>(a, L, smem, tile, j, col0, nsc_me, pol);
    }
  }

  const float invN = a.invN;
  const int cstep = a.tpr * 16;
  int rpar = 0;
  ClusterXch xch = make_xch(smem, L, a.RT, CLUSTER ? a.C : 1, crank);

  // First read of chunk k of a row slot: x, or with RESID h = bf16(x + r),
  // which replaces x in the stage for the later passes (each chunk is read
  // and written by its one owning thread only).
  auto first_chunk = [&](const unsigned char *rowp, int k) -> uint4 {
    const unsigned char *p = rowp + k * cstep;
    if (!RESID) return lds_chunk(p);
    float2 xs[4], rs_[4];
    chunk_to_f2(lds_chunk(p), xs);
    chunk_to_f2(lds_chunk(p + L.tensor_bytes), rs_);
#pragma unroll
    for (int q = 0; q < 4; ++q) xs[q] = add2(xs[q], rs_[q]);
    const uint4 h = f2_to_chunk(xs);
    *reinterpret_cast<uint4 *>(const_cast<unsigned char *>(p)) = h;
    return h;
  };

  // Statistics pass of row slot r of the stage at `st`: this row group's
  // partial, (n, mean, M2) for LayerNorm or (sum x^2) for RMSNorm.
  auto stats_pass = [&](const unsigned char *st, int r, bool active, float &pa, float &pb,
                        float &pc) {
    const unsigned char *rowp = st + static_cast<size_t>(r) * a.NS * 2 + t * 16;
    if (MODE == kLayer) {
      float2 a0 = splat2(0.f), a1 = splat2(0.f);
      if (active) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          if (EXACT || t + k * a.tpr < nsc_me) {
            float2 xf[4];
            chunk_to_f2(first_chunk(rowp, k), xf);
            a0 = add2(a0, add2(xf[0], xf[1]));
            a1 = add2(a1, add2(xf[2], xf[3]));
          }
        }
      }
      const float2 at = add2(a0, a1);
      float n = active ? 8.f * static_cast<float>(nown) : 0.f;
      // exact slices: every thread holds 8 K values (no division per row)
      float m = EXACT ? (at.x + at.y) * (1.f / (8.f * K)) : (n > 0.f ? (at.x + at.y) / n : 0.f);
      const float2 nm = splat2(-m);
      float2 q0 = splat2(0.f), q1 = splat2(0.f);
      if (active) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          if (EXACT || t + k * a.tpr < nsc_me) {
            float2 xf[4];
            chunk_to_f2(lds_chunk(rowp + k * cstep), xf);
            const float2 d0 = add2(xf[0], nm), d1 = add2(xf[1], nm);
            const float2 d2 = add2(xf[2], nm), d3 = add2(xf[3], nm);
            q0 = fma2(d0, d0, fma2(d1, d1, q0));
            q1 = fma2(d2, d2, fma2(d3, d3, q1));
          }
        }
      }
      const float2 qt = add2(q0, q1);
      float q = qt.x + qt.y;
      // Exact slices: every partial of the row group covers the same count,
      // so the merges are the equal-count ones (constant weights, no
      // division, no empty-partial tests); ragged slices need the
      // count-weighted merge.  (With it on exact slices the LayerNorm
      // forward ran at 20-34 % of measured from 32768 columns on.)
      if (EXACT)
        group_meanvar(m, q, 8.f * K, a.tpr, g, a.G, t, red, rpar);
      else
        group_nmeanvar(n, m, q, a.tpr, g, a.G, t, red, rpar);
      pa = m;
      pb = q;
      pc = n;
    } else {
      float2 q0 = splat2(0.f), q1 = splat2(0.f);
      float mx = 0.f;  // per-row E4M3: the largest |x gamma| of the slice
      if (active) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
          if (EXACT || t + k * a.tpr < nsc_me) {
            float2 xf[4];
            chunk_to_f2(first_chunk(rowp, k), xf);
            q0 = fma2(xf[0], xf[0], fma2(xf[1], xf[1], q0));
            q1 = fma2(xf[2], xf[2], fma2(xf[3], xf[3], q1));
            if (OUT == kOutFp8Row) {
              float2 gf[4];
              chunk_to_f2(gv[k], gf);
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const float2 pr = mul2(xf[p], gf[p]);
                mx = fmaxf(mx, fmaxf(fabsf(pr.x), fabsf(pr.y)));
              }
            }
          }
        }
      }
      const float2 qt = add2(q0, q1);
      float v[1] = {qt.x + qt.y};
      group_sum<1, EXACT>(v, a.tpr, g, a.G, t, red, rpar);
      pa = v[0];
      pb = OUT == kOutFp8Row ? group_max<true>(mx, a.tpr, g, a.G, t, red, rpar) : 0.f;
      pc = 0.f;
    }
  };

  // Output pass of row slot r given the row totals; writes y and the
  // statistics.  Per-row E4M3, LayerNorm, runs in one of three phases:
  // kFp8Whole (no cluster: the row amax, then the codes), kFp8Amax (cluster:
  // returns this CTA's slice amax, stores nothing) or kFp8Codes (cluster:
  // the codes with the row amax `am_row`, then the statistics); RMSNorm
  // always writes the codes, `am_row` being the row's largest |x gamma|.
  auto output_pass = [&](const unsigned char *st, int64_t row0, int r, float ta, float tb,
                         int phase = kFp8Whole, float am_row = 0.f) -> float {
    float rs, mu = 0.f;
    if (MODE == kLayer) {
      mu = ta;
      rs = rsqrtf(tb * invN + a.eps);
    } else {
      rs = rsqrtf(ta * invN + a.eps);
    }
    const unsigned char *rowp = st + static_cast<size_t>(r) * a.NS * 2 + t * 16;
    const float2 rs2 = splat2(rs), nmu = splat2(-mu);
    uint16_t *hrow = RESID ? a.h + (row0 + r) * a.N + col0 + t * 8 : nullptr;
    // y of chunk k (owned chunks only); with `store_h` also streams h out.
    auto ychunk = [&](int k, float2 (&o)[4], bool store_h) {
      float2 xf[4], gf[4], bf[4];
      const uint4 hv = lds_chunk(rowp + k * cstep);
      if (RESID && store_h) st_global_cs_v4(hrow + k * a.tpr * 8, hv);
      chunk_to_f2(hv, xf);
      chunk_to_f2(gv[k], gf);
      if (MODE == kLayer) chunk_to_f2(bv[k], bf);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 xh = mul2(MODE == kLayer ? add2(xf[p], nmu) : xf[p], rs2);
        o[p] = (MODE == kLayer) ? fma2(xh, gf[p], bf[p]) : mul2(xh, gf[p]);
      }
    };
    if (OUT == kOutBf16) {
      uint16_t *yrow = a.out + (row0 + r) * a.N + col0 + t * 8;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (EXACT || t + k * a.tpr < nsc_me) {
          float2 o[4];
          ychunk(k, o, true);
          st_global_cs_v4(yrow + k * a.tpr * 8, f2_to_chunk(o));
        }
      }
    } else if (OUT == kOutFp8Row) {
      // amax of the row (of this CTA's slice in a cluster), then the codes
      uint8_t *qrow = a.q + (row0 + r) * a.N + col0 + t * 8;
      float am = am_row;
      if (MODE == kRMS) {
        // y = x rstd gamma with rstd > 0: the row's amax is rstd times the
        // largest |x gamma|, which the statistics pass took (am_row), so
        // there is no y pass for it and, in a cluster, no second exchange.
        am = rs * am_row;
      } else if (phase != kFp8Codes) {
        am = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          if (EXACT || t + k * a.tpr < nsc_me) {
            float2 o[4];
            ychunk(k, o, false);
#pragma unroll
            for (int p = 0; p < 4; ++p) am = fmaxf(am, fmaxf(fabsf(o[p].x), fabsf(o[p].y)));
          }
        }
        am = group_max<true>(am, a.tpr, g, a.G, t, red, rpar);
        if (phase == kFp8Amax) return am;
      }
      const float2 inv = splat2(am > 0.f ? __fdividef(448.f, am) : 1.f);
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (EXACT || t + k * a.tpr < nsc_me) {
          float2 o[4];
          ychunk(k, o, true);
          uint32_t w[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 v = mul2(o[p], inv);
            w[p] = cvt_e4m3x2(v.x, v.y);
          }
          st_global_cs_v2(qrow + k * a.tpr * 8,
                          make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16)));
        }
      }
      if (t == 0 && crank == 0) a.qscale[row0 + r] = am > 0.f ? am * (1.0f / 448.0f) : 1.f;
    } else {
      // MX: a block is 4 consecutive chunks of 4 consecutive lanes (tpr is a
      // multiple of 32 and the slice starts on a block), so its amax is two
      // butterfly steps; every lane takes part in the shuffles.
      uint8_t *qrow = a.q + (row0 + r) * a.N + col0 + t * 8;
      uint8_t *erow = a.qexp + (row0 + r) * (a.N / kMxBlock) + col0 / kMxBlock;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const bool own = EXACT || t + k * a.tpr < nsc_me;
        float2 o[4] = {splat2(0.f), splat2(0.f), splat2(0.f), splat2(0.f)};
        if (own) ychunk(k, o, true);
        float m = 0.f;
#pragma unroll
        for (int p = 0; p < 4; ++p) m = fmaxf(m, fmaxf(fabsf(o[p].x), fabsf(o[p].y)));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int eb = static_cast<int>(__float_as_uint(m) >> 23);
        const float2 inv =
            splat2(__uint_as_float(static_cast<uint32_t>(min(262 - eb, 254)) << 23));
        if (own) {
          uint32_t w[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 v = mul2(o[p], inv);
            w[p] = cvt_e4m3x2(v.x, v.y);
          }
          st_global_cs_v2(qrow + k * a.tpr * 8,
                          make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16)));
          st_global_u8_if(erow + ((t + k * a.tpr) >> 2), static_cast<uint32_t>(max(eb - 8, 0)),
                          (t & 3) == 0);
        }
      }
    }
    if (t == 0 && crank == 0) {
      a.rstd[row0 + r] = rs;
      if (MODE == kLayer) a.mean[row0 + r] = mu;
    }
    return 0.f;
  };

  // Stage s is consumed: the last warp refills it with the tile S ahead.
  auto release = [&](int64_t tile, int s) {
    if (last_warp_done(done_cnt, s, nwarps) && (tid & 31) == 0) {
      const int64_t next = tile + static_cast<int64_t>(a.S) * ncl;
      if (next < a.ntiles) {
        fence_proxy_async_smem();
        issue_fwd_tile<CLUSTER, RESID>(a, L, smem, next, s, col0, nsc_me, pol);
      }
    }
  };

  // Finish a pending cluster tile: wait for its exchange, fold in rank
  // order, write outputs, release the stage.  (Cluster tiles hold one row
  // per group: rows_per_group is 1.)
  // Row totals of an exchange round's C slots, folded in rank order.
  auto fold_totals = [&](const float *row, float &ta, float &tb) {
    if (MODE == kLayer) {
      float n, m, q;
      if (EXACT) {
        // equal counts (NS columns per CTA), merged in rank order
        rank_fold_meanvar(row, xch.C, static_cast<float>(a.NS), m, q);
      } else {
        fold_nmeanvar(row, xch.C, n, m, q);
      }
      ta = m;
      tb = q;
    } else {
      float v[1];
      fold_sum<1>(row, xch.C, v);
      ta = v[0];
      tb = 0.f;
    }
  };
  auto finish = [&](const Pending &p) {
    const int64_t row0 = p.tile * a.RT;
    const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
    const int r = g;
    float ta, tb;
    const float *row = cluster_wait_row(r, xch, a.err, abort_flag);
    fold_totals(row, ta, tb);
    float mx = 0.f;  // per-row E4M3 (RMSNorm): the row's largest |x gamma|
    if (OUT == kOutFp8Row && MODE == kRMS) {
      mx = row[1];
      for (int q = 1; q < xch.C; ++q) mx = fmaxf(mx, row[q * 4 + 1]);
    }
    if (r < nrows)
      output_pass(smem + static_cast<size_t>(p.s) * L.stage_bytes, row0, r, ta, tb, kFp8Codes,
                  mx);
    release(p.tile, p.s);
  };
  // Per-row E4M3 in a cluster, LayerNorm: one exchange round per tile
  // carries the tile's statistics partial and, in its fourth float, this
  // CTA's slice amax of the previous tile, whose codes are written once the
  // round is in.  (Two rounds per tile -- statistics, then amax -- cannot
  // overlap the next tile's statistics, since rounds are consumed in push
  // order.)  RMSNorm's amax travels with its statistics (second float) and
  // takes the pipelined path of the other outputs.
  float pend_ta = 0.f, pend_tb = 0.f, pend_am = 0.f;
  auto fp8_codes = [&](const Pending &p, const float *row) {
    const int64_t row0 = p.tile * a.RT;
    const int r = g;
    float am = row[3];
    for (int q = 1; q < xch.C; ++q) am = fmaxf(am, row[q * 4 + 3]);
    if (r < static_cast<int>(min64(a.RT, a.M - row0)))
      output_pass(smem + static_cast<size_t>(p.s) * L.stage_bytes, row0, r, pend_ta, pend_tb,
                  kFp8Codes, am);
    release(p.tile, p.s);
  };

  int s = 0;
  uint32_t par = 0;
  Pending pend;
  bool have_pend = false;
  for (int64_t tile = cid; tile < a.ntiles; tile += ncl) {
    mbar_wait(full + s, par, a.err, abort_flag);
    const int64_t row0 = tile * a.RT;
    const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
    const unsigned char *st = smem + static_cast<size_t>(s) * L.stage_bytes;
    if (CLUSTER) {
      const int r = g;
      Pending cur;
      cur.tile = tile;
      cur.s = s;
      stats_pass(st, r, r < nrows, cur.a, cur.b, cur.c);
      if (OUT == kOutFp8Row && MODE == kLayer) {
        cluster_push(cur.a, cur.b, cur.c, r, t, xch, have_pend ? pend_am : 0.f);
        const float *row = cluster_wait_row(r, xch, a.err, abort_flag);
        float ta, tb;
        fold_totals(row, ta, tb);
        if (have_pend) fp8_codes(pend, row);
        pend = cur;
        pend_ta = ta;
        pend_tb = tb;
        pend_am = r < nrows ? output_pass(st, row0, r, ta, tb, kFp8Amax) : 0.f;
        have_pend = true;
      } else {
        cluster_push(cur.a, cur.b, cur.c, r, t, xch);
        if (have_pend) finish(pend);
        pend = cur;
        have_pend = true;
      }
    } else {
      for (int q = 0; q < a.rpg; ++q) {
        const int r = g + q * a.G;
        const bool active = r < nrows;
        float pa, pb, pc;
        stats_pass(st, r, active, pa, pb, pc);
        if (active) output_pass(st, row0, r, pa, pb, kFp8Whole, pb);
      }
      release(tile, s);
    }
    if (++s == a.S) {
      s = 0;
      par ^= 1u;
    }
  }
  if (CLUSTER) {
    if (have_pend) {
      if (OUT == kOutFp8Row && MODE == kLayer) {
        // a last round with the last tile's slice maxima only
        cluster_push(0.f, 0.f, 0.f, g, t, xch, pend_am);
        fp8_codes(pend, cluster_wait_row(g, xch, a.err, abort_flag));
      } else {
        finish(pend);
      }
    }
    cluster_sync();
  }
}

// RESID: fused residual add -- dx = (norm backward at h) + dh, summed in
// fp32 and rounded once.  dh is needed by the dx pass only, so it is not
// staged: each thread loads its chunks of a row's dh into registers one step
// ahead of that row's dx pass (before the dot pass without a cluster; after
// the previous tile's push in a cluster), so the stage holds h and dy like
// the plain backward and takes the same (narrower) clusters.
template <int MODE, int K, bool CLUSTER, bool EXACT, bool RESID>
__global__ void __launch_bounds__(kMaxThreads, 1) norm_bwd_long_kernel(const NormArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout L = make_layout(a.RT, a.NS, a.S, a.G, a.tpr, 2, true, a.C);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag_off);
  int *done_cnt = reinterpret_cast<int *>(smem + L.flag_off) + 1;

  const int tid = threadIdx.x;
  const int g = tid / a.tpr;
  const int t = tid - g * a.tpr;
  const int nwarps = blockDim.x >> 5;
  const int crank = CLUSTER ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t cid = CLUSTER ? static_cast<int64_t>(cluster_id_x()) : blockIdx.x;
  const int64_t ncl = CLUSTER ? static_cast<int64_t>(ncluster_x()) : gridDim.x;
  const int col0 = crank * a.NS;
  const int nsc_me = min(a.nsc, a.N / 8 - crank * a.nsc);

  if (tid == 0) {
    for (int s = 0; s < a.S; ++s) {
      mbar_init(full + s, 1);
      done_cnt[s] = 0;
    }
    if (CLUSTER) {
      uint64_t *xb = xch_bars(smem, L, a.RT, a.C);
      for (int b = 0; b < kXchBuffers; ++b) mbar_init(xb + b, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Programmatic dependent launch: let the next kernel in the stream start
  // its prologue as our CTAs retire, and touch no global memory before the
  // previous kernel's writes are complete and visible.
  grid_launch_dependents();
  grid_dependency_wait();

  // Per-column state: gamma (packed bf16) and the fp32 column accumulators.
  uint4 gv[K];
  float2 accg[K][4], accb[K][4];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int c = t + k * a.tpr;
    gv[k] = (c < nsc_me) ? ld_global_nc_v4(a.gamma + col0 + c * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      accg[k][p] = splat2(0.f);
      accb[k][p] = splat2(0.f);
    }
  }

  if (CLUSTER) cluster_sync(); else __syncthreads();

  const uint64_t pol = l2_evict_first_policy();
  if (tid < 32) {
    for (int j = 0; j < a.S; ++j) {
      const int64_t tile = cid + j * ncl;
      if (tile < a.ntiles)
        issue_bwd_tile<MODE, CLUSTER, false>(a, L, smem, tile, j, col0, nsc_me, pol);
    }
  }

  const float invN = a.invN;
  const int cstep = a.tpr * 16;
  int rpar = 0;
  ClusterXch xch = make_xch(smem, L, a.RT, CLUSTER ? a.C : 1, crank);
  const float *stats_all = reinterpret_cast<const float *>(smem + L.stats_off);

  // Dot-product pass of row slot r of stage s: sum(g) and sum(g * xhat) of
  // this row group (group totals), and the column accumulators.
  auto dot_pass = [&](int s, int r, bool active, float &pa, float &pb) {
    const unsigned char *xrow = smem + static_cast<size_t>(s) * L.stage_bytes +
                                static_cast<size_t>(r) * a.NS * 2 + t * 16;
    const float *stats = stats_all + static_cast<size_t>(s) * a.RT * 2;
    float rs = 0.f, mu = 0.f;
    if (active) {
      rs = stats[2 * r];
      if (MODE == kLayer) mu = stats[2 * r + 1];
    }
    const float2 rs2 = splat2(rs), nmu = splat2(-mu);
    float2 s1 = splat2(0.f), s2 = splat2(0.f), s1b = splat2(0.f), s2b = splat2(0.f);
    if (active) {
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (EXACT || t + k * a.tpr < nsc_me) {
          float2 xf[4], df[4], gf[4];
          chunk_to_f2(lds_chunk(xrow + k * cstep), xf);
          chunk_to_f2(lds_chunk(xrow + L.tensor_bytes + k * cstep), df);
          chunk_to_f2(gv[k], gf);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 xh = mul2(MODE == kLayer ? add2(xf[p], nmu) : xf[p], rs2);
            const float2 gg = mul2(df[p], gf[p]);
            if (p & 1) {
              s2b = fma2(gg, xh, s2b);
              if (MODE == kLayer) s1b = add2(s1b, gg);
            } else {
              s2 = fma2(gg, xh, s2);
              if (MODE == kLayer) s1 = add2(s1, gg);
            }
            accg[k][p] = fma2(df[p], xh, accg[k][p]);
            if (MODE == kLayer) accb[k][p] = add2(accb[k][p], df[p]);
          }
        }
      }
    }
    s1 = add2(s1, s1b);
    s2 = add2(s2, s2b);
    float v[2] = {s1.x + s1.y, s2.x + s2.y};
    if (MODE == kLayer) {
      group_sum<2, EXACT>(v, a.tpr, g, a.G, t, red, rpar);
    } else {
      float w1[1] = {v[1]};
      group_sum<1, EXACT>(w1, a.tpr, g, a.G, t, red, rpar);
      v[1] = w1[0];
    }
    pa = v[0];
    pb = v[1];
  };

  // RESID: this thread's chunks of dh for the row whose dx pass comes next.
  uint4 dhr[RESID ? K : 1];
  auto load_dh = [&](int64_t row0, int r, bool active) {
#pragma unroll
    for (int k = 0; k < (RESID ? K : 0); ++k) {
      const int c = t + k * a.tpr;
      dhr[k] = (active && (EXACT || c < nsc_me))
                   ? ld_global_nc_v4(a.res + (row0 + r) * a.N + col0 + c * 8)
                   : make_uint4(0, 0, 0, 0);
    }
  };

  // dx pass of row slot r of stage s given the row totals.
  auto dx_pass = [&](int s, int64_t row0, int r, float tsum_g, float tsum_gx) {
    const unsigned char *xrow = smem + static_cast<size_t>(s) * L.stage_bytes +
                                static_cast<size_t>(r) * a.NS * 2 + t * 16;
    const float *stats = stats_all + static_cast<size_t>(s) * a.RT * 2;
    const float rs = stats[2 * r];
    const float mu = (MODE == kLayer) ? stats[2 * r + 1] : 0.f;
    const float2 rs2 = splat2(rs), nmu = splat2(-mu);
    // dx = rstd (g - a - xhat c) = rstd g - rstd a - rstd^2 c (x - mean):
    // the row constants -rstd a and -rstd^2 c leave three (RMSNorm) or four
    // (LayerNorm) packed operations per pair
    const float2 nra = splat2((MODE == kLayer) ? -rs * (tsum_g * invN) : 0.f);
    const float2 nk1 = splat2(-rs * rs * (tsum_gx * invN));
    uint16_t *dxrow = a.out + (row0 + r) * a.N + col0 + t * 8;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (EXACT || t + k * a.tpr < nsc_me) {
        float2 xf[4], df[4], gf[4], o[4];
        chunk_to_f2(lds_chunk(xrow + k * cstep), xf);
        chunk_to_f2(lds_chunk(xrow + L.tensor_bytes + k * cstep), df);
        chunk_to_f2(gv[k], gf);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 gg = mul2(df[p], gf[p]);
          const float2 xc = MODE == kLayer ? add2(xf[p], nmu) : xf[p];
          o[p] = fma2(xc, nk1, MODE == kLayer ? fma2(gg, rs2, nra) : mul2(gg, rs2));
        }
        if (RESID) {
          float2 hf[4];
          chunk_to_f2(dhr[RESID ? k : 0], hf);
#pragma unroll
          for (int p = 0; p < 4; ++p) o[p] = add2(o[p], hf[p]);
        }
        st_global_cs_v4(dxrow + k * a.tpr * 8, f2_to_chunk(o));
      }
    }
  };

  auto release = [&](int64_t tile, int s) {
    if (last_warp_done(done_cnt, s, nwarps)) {
      const int64_t next = tile + static_cast<int64_t>(a.S) * ncl;
      if (next < a.ntiles) {
        if ((tid & 31) == 0) fence_proxy_async_smem();
        __syncwarp();
        issue_bwd_tile<MODE, CLUSTER, false>(a, L, smem, next, s, col0, nsc_me, pol);
      }
    }
  };

  auto finish = [&](const Pending &p) {
    const int64_t row0 = p.tile * a.RT;
    const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
    const int r = g;
    const float *row = cluster_wait_row(r, xch, a.err, abort_flag);
    float v[2];
    fold_sum<2>(row, xch.C, v);
    if (r < nrows) dx_pass(p.s, row0, r, v[0], v[1]);
    release(p.tile, p.s);
  };

  int s = 0;
  uint32_t par = 0;
  Pending pend;
  bool have_pend = false;
  for (int64_t tile = cid; tile < a.ntiles; tile += ncl) {
    mbar_wait(full + s, par, a.err, abort_flag);
    const int64_t row0 = tile * a.RT;
    const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
    if (CLUSTER) {
      const int r = g;
      Pending cur;
      cur.tile = tile;
      cur.s = s;
      cur.c = 0.f;
      dot_pass(s, r, r < nrows, cur.a, cur.b);
      cluster_push(cur.a, cur.b, 0.f, r, t, xch);
      if (have_pend) finish(pend);  // its dh arrived during this tile's dot pass
      if (RESID) load_dh(row0, r, r < nrows);
      pend = cur;
      have_pend = true;
    } else {
      for (int q = 0; q < a.rpg; ++q) {
        const int r = g + q * a.G;
        const bool active = r < nrows;
        float pa, pb;
        if (RESID) load_dh(row0, r, active);  // in flight during the dot pass
        dot_pass(s, r, active, pa, pb);
        if (active) dx_pass(s, row0, r, pa, pb);
      }
      release(tile, s);
    }
    if (++s == a.S) {
      s = 0;
      par ^= 1u;
    }
  }
  if (CLUSTER && have_pend) finish(pend);

  write_column_partials<MODE, K, EXACT>(a, smem, accg, accb, g, t, nsc_me, cid, col0);
  if (CLUSTER) cluster_sync();
}

}  // namespace gbn
