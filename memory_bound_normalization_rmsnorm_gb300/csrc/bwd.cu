// bwd.cu -- backward RMSNorm / LayerNorm: one fused row pass (dx, plus
// per-CTA partial column sums for dgamma and dbeta) and a fixed-order
// reduction of those partials.
//
// Follows the backward-pass paragraphs of "PyTorch atinge desempenho SOTA
// em normalizacao com torch.compile" (matsubara.tec.br):
//   - dX, dW and dB computed in ONE kernel so that dy and x are read once
//     (the fused-reduction paragraph);
//   - the column reduction split across CTAs, each CTA summing many rows
//     into a partial row of a workspace that a second kernel reduces,
//     without atomics (the split-reduction paragraph);
//   - rows per partial set by how many CTAs run (the SPLIT_SIZE paragraph)
//     and several loads kept in flight (the num_stages paragraph).
// The saved rstd (and mean) of the forward pass are reused, not recomputed.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"
#include "tiles.cuh"

namespace gbn {

namespace {

// EXACT: every CTA's slice is exactly K * tpr chunks and tpr >= 32, so no
// chunk needs an ownership test and the warp butterfly is full width.
// RESID: fused residual add -- x is h, and the stage also holds dh, added to
// dx (in fp32, before rounding): dx = norm backward + dh.
template <int MODE, int K, bool CLUSTER, bool EXACT, bool RESID>
__global__ void __launch_bounds__(kMaxThreads, 1) norm_bwd_kernel(const NormArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout L = make_layout(a.RT, a.NS, a.S, a.G, a.tpr, RESID ? 3 : 2, true, a.C);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  const float *stats_all = reinterpret_cast<const float *>(smem + L.stats_off);
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
  // Chunks this CTA owns (the last CTA of a cluster may own fewer).
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

  // The first S tiles are requested before anything else, so that their
  // DRAM round trip overlaps the parameter loads below (warp 0, whose lane 0
  // initialised the barriers, issues them after a warp sync).
  const uint64_t pol = l2_evict_first_policy();
  if (tid < 32) {
    __syncwarp();
    for (int j = 0; j < a.S; ++j) {
      const int64_t tile = cid + j * ncl;
      if (tile < a.ntiles) issue_bwd_tile<MODE, CLUSTER, RESID>(a, L, smem, tile, j, col0, nsc_me, pol);
    }
  }

  // gamma (fp32 pairs) and the column accumulators of this thread's chunks
  // live in registers for the whole kernel.
  float2 gf[K][4], accg[K][4], accb[K][4];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int c = t + k * a.tpr;
    const uint4 gv = (c < nsc_me) ? ld_global_nc_v4(a.gamma + col0 + c * 8) : make_uint4(0, 0, 0, 0);
    chunk_to_f2(gv, gf[k]);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      accg[k][p] = splat2(0.f);
      accb[k][p] = splat2(0.f);
    }
  }

  if (CLUSTER) cluster_sync(); else __syncthreads();

  const float invN = a.invN;
  int rpar = 0;
  ClusterXch xch = make_xch(smem, L, a.RT, CLUSTER ? a.C : 1, crank);
  // Stage s and its phase parity advance with the tile count (no division).
  int s = 0;
  uint32_t par = 0;
  for (int64_t tile = cid; tile < a.ntiles; tile += ncl) {
    mbar_wait(full + s, par, a.err, abort_flag);
    const int64_t row0 = tile * a.RT;
    const int nrows = static_cast<int>(min64(a.RT, a.M - row0));
    const unsigned char *stx = smem + static_cast<size_t>(s) * L.stage_bytes;
    const float *stats = stats_all + static_cast<size_t>(s) * a.RT * 2;

    for (int q = 0; q < a.rpg; ++q) {
      const int r = g + q * a.G;
      const bool active = r < nrows;
      float rs = 0.f, mu = 0.f;
      if (active) {
        rs = stats[2 * r];
        if (MODE == kLayer) mu = stats[2 * r + 1];
      }
      const float2 rs2 = splat2(rs);
      const float2 nmu = splat2(-mu);
      const unsigned char *xrow = stx + static_cast<size_t>(r) * a.NS * 2 + t * 16;
      // xhat and g = dy * gamma stay in registers between the two passes.
      float2 xh[K][4], gg[K][4];
      float2 s1 = splat2(0.f), s2 = splat2(0.f), s1b = splat2(0.f), s2b = splat2(0.f);
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const bool ok = active && (EXACT || t + k * a.tpr < nsc_me);
        uint4 xv = make_uint4(0, 0, 0, 0), dv = make_uint4(0, 0, 0, 0);
        if (ok) {
          xv = *reinterpret_cast<const uint4 *>(xrow + k * a.tpr * 16);
          dv = *reinterpret_cast<const uint4 *>(xrow + L.tensor_bytes + k * a.tpr * 16);
        }
        float2 xf[4], df[4];
        chunk_to_f2(xv, xf);
        chunk_to_f2(dv, df);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          xh[k][p] = mul2(MODE == kLayer ? add2(xf[p], nmu) : xf[p], rs2);
          gg[k][p] = mul2(df[p], gf[k][p]);
          // two independent accumulator pairs shorten the dependency chains
          if (p & 1) {
            s2b = fma2(gg[k][p], xh[k][p], s2b);
            if (MODE == kLayer) s1b = add2(s1b, gg[k][p]);
          } else {
            s2 = fma2(gg[k][p], xh[k][p], s2);
            if (MODE == kLayer) s1 = add2(s1, gg[k][p]);
          }
          accg[k][p] = fma2(df[p], xh[k][p], accg[k][p]);
          if (MODE == kLayer) accb[k][p] = add2(accb[k][p], df[p]);
        }
      }
      s1 = add2(s1, s1b);
      s2 = add2(s2, s2b);
      float v[2] = {s1.x + s1.y, s2.x + s2.y};
      if (MODE == kLayer) {
        group_sum<2, EXACT>(v, a.tpr, g, a.G, t, red, rpar);
        if (CLUSTER) cluster_sum<2>(v, r, t, xch, a.err, abort_flag);
      } else {
        float w1[1] = {v[1]};
        group_sum<1, EXACT>(w1, a.tpr, g, a.G, t, red, rpar);
        if (CLUSTER) cluster_sum<1>(w1, r, t, xch, a.err, abort_flag);
        v[1] = w1[0];
      }
      // dx = rstd (g - a - xhat c) = rstd g - rstd a - (rstd c) xhat
      const float2 nra = splat2((MODE == kLayer) ? -rs * (v[0] * invN) : 0.f);
      const float2 nrc = splat2(-rs * (v[1] * invN));

      if (active) {
        uint16_t *dxrow = a.out + (row0 + r) * a.N + col0 + t * 8;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          if (EXACT || t + k * a.tpr < nsc_me) {
            float2 o[4];
#pragma unroll
            for (int p = 0; p < 4; ++p)
              o[p] = fma2(xh[k][p], nrc,
                          MODE == kLayer ? fma2(gg[k][p], rs2, nra) : mul2(gg[k][p], rs2));
            if (RESID) {
              float2 dh[4];
              chunk_to_f2(*reinterpret_cast<const uint4 *>(stx + 2 * L.tensor_bytes +
                                                           static_cast<size_t>(r) * a.NS * 2 +
                                                           (t + k * a.tpr) * 16),
                          dh);
#pragma unroll
              for (int p = 0; p < 4; ++p) o[p] = add2(o[p], dh[p]);
            }
            st_global_cs_v4(dxrow + k * a.tpr * 8, f2_to_chunk(o));
          }
        }
      }
    }

    if (last_warp_done(done_cnt, s, nwarps)) {
      const int64_t next = tile + static_cast<int64_t>(a.S) * ncl;
      if (next < a.ntiles) {
        if ((tid & 31) == 0) fence_proxy_async_smem();
        __syncwarp();
        issue_bwd_tile<MODE, CLUSTER, RESID>(a, L, smem, next, s, col0, nsc_me, pol);
      }
    }
    if (++s == a.S) {
      s = 0;
      par ^= 1u;
    }
  }

  write_column_partials<MODE, K, EXACT>(a, smem, accg, accb, g, t, nsc_me, cid, col0);
  if (CLUSTER) cluster_sync();
}

// Self-test of the bounded-wait failure path: waits on phase 0 of an
// mbarrier that expects one arrival which never comes.
__global__ void selftest_wait_kernel(unsigned *err, uint32_t polls) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, err, &abort_flag, polls);
}

constexpr int kReduceWarps = 32;
constexpr int kReduceBatch = 8;  // partial rows a lane loads before adding

// dgamma[j] = sum over p of ws[p][j] (blockIdx.y = 0) and dbeta[j] = sum
// over p of ws[P + p][j] (blockIdx.y = 1).  Warp w of the block sums the
// contiguous range p in [P*w/32, P*(w+1)/32) in increasing p (loads of a
// batch issued together, then added in order); the 32 warp sums are then
// added in warp order: a fixed order for a given P, so the result is bitwise
// reproducible.  Each lane owns 4 consecutive columns.
__global__ void __launch_bounds__(kReduceWarps * 32) reduce_partials_kernel(
    const float *__restrict__ ws, int P, int N, float *__restrict__ dgamma,
    float *__restrict__ dbeta) {
  __shared__ float4 part[kReduceWarps][32];
  grid_launch_dependents();
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const float *src = ws + static_cast<size_t>(blockIdx.y) * P * N;
  float *dst = blockIdx.y ? dbeta : dgamma;
  const int col = (blockIdx.x * 32 + lane) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col < N) {
    const int p0 = static_cast<int>((static_cast<int64_t>(P) * w) / kReduceWarps);
    const int p1 = static_cast<int>((static_cast<int64_t>(P) * (w + 1)) / kReduceWarps);
    for (int p = p0; p < p1; p += kReduceBatch) {
      float4 v[kReduceBatch];
#pragma unroll
      for (int u = 0; u < kReduceBatch; ++u)
        v[u] = (p + u < p1) ? __ldcg(reinterpret_cast<const float4 *>(
                                  src + static_cast<size_t>(p + u) * N + col))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < kReduceBatch; ++u) {
        if (p + u < p1) {
          acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
        }
      }
    }
  }
  part[w][lane] = acc;
  __syncthreads();
  if (w == 0 && col < N) {
    float4 s = part[0][lane];
#pragma unroll
    for (int u = 1; u < kReduceWarps; ++u) {
      s.x += part[u][lane].x; s.y += part[u][lane].y;
      s.z += part[u][lane].z; s.w += part[u][lane].w;
    }
    *reinterpret_cast<float4 *>(dst + col) = s;
  }
}

template <int MODE, int K, bool CLUSTER, bool RESID>
const void *pick_exact(bool e) {
  return e ? reinterpret_cast<const void *>(&norm_bwd_kernel<MODE, K, CLUSTER, true, RESID>)
           : reinterpret_cast<const void *>(&norm_bwd_kernel<MODE, K, CLUSTER, false, RESID>);
}

template <int MODE, int K, bool CLUSTER>
const void *pick_variant(bool e, bool r) {
  if (r) return CLUSTER ? nullptr : pick_exact<MODE, K, false, true>(e);  // no cluster variants
  return pick_exact<MODE, K, CLUSTER, false>(e);
}

template <int MODE, bool CLUSTER>
const void *pick_bwd(int K, bool e, bool r) {
  switch (K) {
    case 1: return pick_variant<MODE, 1, CLUSTER>(e, r);
    case 2: return pick_variant<MODE, 2, CLUSTER>(e, r);
    case 3: return pick_variant<MODE, 3, CLUSTER>(e, r);
    case 4: return pick_variant<MODE, 4, CLUSTER>(e, r);
    default: return nullptr;
  }
}

}  // namespace

const void *bwd_kernel_ptr(int mode, int K, bool cluster, bool exact, bool resid) {
  if (mode == kRMS)
    return cluster ? pick_bwd<kRMS, true>(K, exact, resid) : pick_bwd<kRMS, false>(K, exact, resid);
  return cluster ? pick_bwd<kLayer, true>(K, exact, resid)
                 : pick_bwd<kLayer, false>(K, exact, resid);
}

const void *reduce_kernel_ptr() {
  return reinterpret_cast<const void *>(&reduce_partials_kernel);
}

int reduce_threads() { return kReduceWarps * 32; }

const void *selftest_kernel_ptr() {
  return reinterpret_cast<const void *>(&selftest_wait_kernel);
}

}  // namespace gbn
