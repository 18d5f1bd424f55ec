// stream.cu -- the streaming long-row kernels.  Backward: rows of 32768
// columns per CTA (a cluster of C = N / 32768 CTAs per row), each row slice
// streamed through a shared-memory ring twice -- once for the per-row dot
// products, once for dx -- instead of being held in shared memory, with the
// dgamma / dbeta column sums accumulated in tensor memory (TMEM).  Forward
// (further down): the same piece sequence for rows wider than a 16-CTA
// cluster holds, pass 1 the statistics, pass 2 y.
//
// "PyTorch atinge desempenho SOTA em normalizacao com torch.compile"
// (matsubara.tec.br) places the backward's difficulty at very large
// dimensions: a row no longer fits on chip, and a kernel that keeps its
// slice resident needs so many CTAs per row that whole clusters stop
// fitting on the GPU's processor clusters (at 131072 columns the resident
// long-row backward needs clusters of 8 CTAs, of which 15 fit: 120 of 152
// SMs).  Here a CTA keeps on chip only what a row does not need twice: the
// packed gamma of its slice (registers) and the column accumulators (TMEM,
// 128 KB for RMSNorm, 256 KB with dbeta).  Its 32768-column slice of x and
// dy passes through a ring of 16384-column pieces (8192 for the fused
// residual backward, whose dh is a third tensor of the dx pass's pieces):
//
//   pass 1 (row j)    sum g and sum g (x - mean) over the slice (g = dy *
//                     gamma), summed over the CTA, then over the cluster
//                     (DSMEM exchange, the same rank-order fold as the
//                     resident long-row kernel); x and dy come from HBM;
//   pass 2 (row j-1)  dx = rstd g - rstd a - rstd^2 c (x - mean) with the
//                     row totals, and dgamma += dy xhat, dbeta += dy read,
//                     updated and written back in TMEM; x and dy come again
//                     -- from L2, where pass 1 left them one row earlier.
//
// The pieces are issued in the order pass 1 of row j, pass 2 of row j-1, so
// the cross-CTA exchange of row j-1 completes while row j streams in, and
// the L2 holds about two slices per CTA between their two reads (~40 MB on
// the whole GPU at 131072 columns).  The column sums leave TMEM once, at the
// end, as this cluster's partial row of the workspace; the fixed-order
// reduce kernel adds the partial rows as for the other backward kernels, so
// results stay bitwise reproducible.
#include "common.cuh"
#include "ptx.cuh"
#include "rowops.cuh"
#include "tcgen05.cuh"

namespace gbn {

namespace {


// L2 policy of pass 1's reads (their data is read again by pass 2).
__device__ __forceinline__ uint64_t l2_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 lds_v4(const unsigned char *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

// Piece q of a CTA's sequence over its nr rows (np pieces per slice):
// pass 1 of row 0, then for j = 1 .. nr-1 pass 1 of row j and pass 2 of
// row j-1, then pass 2 of row nr-1.
__device__ __forceinline__ void piece_at(int64_t q, int np, int64_t nr, int &pass, int64_t &j,
                                         int &p) {
  if (q < np) {
    pass = 0;
    j = 0;
    p = static_cast<int>(q);
    return;
  }
  const int64_t q2 = q - np;
  const int64_t b = q2 / (2 * np);
  const int w = static_cast<int>(q2 - b * 2 * np);
  if (b < nr - 1) {
    if (w < np) {
      pass = 0;
      j = b + 1;
      p = w;
    } else {
      pass = 1;
      j = b;
      p = w - np;
    }
  } else {
    pass = 1;
    j = nr - 1;
    p = w;
  }
}

// Publishes a CTA's row totals (a, b) into exchange round x.push_buf, by one
// thread: with a cluster, the round's expected bytes on this CTA's mbarrier
// and an asynchronous store into slot [crank] of every CTA of the cluster;
// alone, a store into its own slot and an arrival (release) on its mbarrier.
template <bool CLUSTER>
__device__ __forceinline__ void xch_publish(float a, float b, const ClusterXch &x) {
  const int bsel = x.push_buf;
  float *mine = x.slots + (static_cast<size_t>(bsel) * x.C + x.crank) * 4;
  uint64_t *bar = x.bars + bsel;
  const float4 val = make_float4(a, b, 0.f, 0.f);
  if (CLUSTER) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(x.C * 16));
    for (int q = 0; q < x.C; ++q) st_async_f32x4(mapa_shared(mine, q), val, mapa_shared(bar, q));
  } else {
    *reinterpret_cast<float4 *>(mine) = val;
    mbar_arrive(bar);
  }
}

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// One CTA per (row, 32768-column slice); NP pieces of kW columns per slice.
// RESID: the fused residual backward, dx = (norm backward at h) + dh, dh
// streamed once with the dx pass's pieces (a.x holds h, a.res dh).
template <int MODE, int KP, bool CLUSTER, bool RESID>
__global__ void __launch_bounds__(kStreamThreads, 1) norm_bwd_stream_kernel(const NormArgs a) {
  constexpr int kKP = KP;                          // 16-byte chunks per thread per piece
  constexpr int kW = stream_piece_cols(KP);        // piece width (columns)
  constexpr int NP = kStreamSlice / kW;            // pieces per slice
  constexpr int NACC = MODE == kLayer ? 2 : 1;          // dgamma (and dbeta)
  constexpr int CPC = 8 * NACC;                          // TMEM columns per chunk
  constexpr int TCW = NP * kKP * CPC;                    // columns per warp quarter group
  constexpr uint32_t kCols = pow2_at_least(4 * TCW);     // 16 warps: 4 per lane quarter
  static_assert(4 * TCW <= 512, "accumulators exceed tensor memory");
  constexpr int kNW = kStreamThreads / 32;
  constexpr int kStride = kStreamThreads * 16;           // bytes between a thread's chunks

  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout L = stream_layout(a.S, CLUSTER ? a.C : 1, RESID ? 3 : 2, KP);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *wred = reinterpret_cast<float *>(smem + L.red_off);  // [buffer][warp][2]
  int *wcnt = reinterpret_cast<int *>(wred + kXchBuffers * kNW * 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag_off);
  int *done_cnt = reinterpret_cast<int *>(smem + L.flag_off) + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.flag_off) + 1 + a.S;

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int crank = CLUSTER ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t cid = CLUSTER ? static_cast<int64_t>(cluster_id_x()) : blockIdx.x;
  const int64_t ncl = CLUSTER ? static_cast<int64_t>(ncluster_x()) : gridDim.x;
  const int64_t col0 = static_cast<int64_t>(crank) * a.NS;
  const int64_t nr = cid < a.M ? (a.M - cid + ncl - 1) / ncl : 0;  // rows of this cluster
  const int64_t total = 2 * NP * nr;                                 // pieces

  if (t == 0) {
    for (int s = 0; s < a.S; ++s) {
      mbar_init(full + s, 1);
      done_cnt[s] = 0;
    }
    uint64_t *xb = xch_bars(smem, L, 1, CLUSTER ? a.C : 1);
    for (int b = 0; b < kXchBuffers; ++b) {
      mbar_init(xb + b, 1);
      wcnt[b] = 0;
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  // Programmatic dependent launch: no global access before the previous
  // kernel's writes are visible.
  grid_launch_dependents();
  grid_dependency_wait();

  // This thread's chunks of gamma: piece p, chunk k at column
  // col0 + p * kW + (k * threads + t) * 8.
  uint4 gv[NP][kKP];
#pragma unroll
  for (int p = 0; p < NP; ++p)
#pragma unroll
    for (int k = 0; k < kKP; ++k)
      gv[p][k] = ld_global_nc_v4(a.gamma + col0 + p * kW + (k * kStreamThreads + t) * 8);

  tc_fence_before();
  if (CLUSTER) cluster_sync(); else __syncthreads();
  tc_fence_after();
  // Warp w reaches TMEM lanes 32 (w % 4) ..; the four warps sharing them
  // take consecutive groups of TCW columns.
  const uint32_t tq = *tmem_slot + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                      static_cast<uint32_t>((warp >> 2) * TCW);
  {
    uint32_t z[CPC];
#pragma unroll
    for (int i = 0; i < CPC; ++i) z[i] = 0u;
#pragma unroll
    for (int c = 0; c < NP * kKP; ++c) tmem_st_n<CPC>(tq + c * CPC, z);
  }

  const uint64_t pol1 = l2_normal_policy();
  const uint64_t pol2 = l2_evict_first_policy();
  // Issues piece q of the sequence into stage s (one thread).
  auto issue = [&](int64_t q, int s) {
    int pass, p;
    int64_t j;
    piece_at(q, NP, nr, pass, j, p);
    const int64_t off = (cid + j * ncl) * a.N + col0 + static_cast<int64_t>(p) * kW;
    uint64_t *bar = full + s;
    unsigned char *dst = smem + static_cast<size_t>(s) * L.stage_bytes;
    const uint64_t pol = pass ? pol2 : pol1;
    const bool with_dh = RESID && pass == 1;
    mbar_arrive_expect_tx(bar, (with_dh ? 3u : 2u) * L.tensor_bytes);
    bulk_g2s(dst, a.x + off, L.tensor_bytes, bar, pol);
    bulk_g2s(dst + L.tensor_bytes, a.dy + off, L.tensor_bytes, bar, pol);
    if (with_dh) bulk_g2s(dst + 2 * L.tensor_bytes, a.res + off, L.tensor_bytes, bar, pol2);
  };
  if (t == 0) {
    for (int64_t q = 0; q < total && q < a.S; ++q) issue(q, static_cast<int>(q));
  }
  // After every warp has read stage s for piece q, the last one refills it
  // with piece q + S.
  auto release = [&](int64_t q, int s) {
    if (last_warp_done(done_cnt, s, kNW)) {
      const int64_t next = q + a.S;
      if (next < total && (t & 31) == 0) {
        fence_proxy_async_smem();
        issue(next, s);
      }
    }
  };

  auto load_stats = [&](int64_t j, float &rs, float &mu) {
    rs = 0.f;
    mu = 0.f;
    if (j < nr) {
      const int64_t row = cid + j * ncl;
      rs = __ldg(a.rstd + row);
      if (MODE == kLayer) mu = __ldg(a.mean + row);
    }
  };

  ClusterXch xch = make_xch(smem, L, 1, CLUSTER ? a.C : 1, crank);
  const float invN = a.invN;
  int s = 0;
  uint32_t par = 0;
  int64_t q = 0;
  auto advance = [&]() {
    ++q;
    if (++s == a.S) {
      s = 0;
      par ^= 1u;
    }
  };
  float rs_prev = 0.f, mu_prev = 0.f, rs_cur, mu_cur, rs_next, mu_next;
  load_stats(0, rs_cur, mu_cur);
  load_stats(1, rs_next, mu_next);

  for (int64_t j = 0; j <= nr; ++j) {
    if (j < nr) {
      // ---- pass 1 of row j: sum g and sum g (x - mean) over the slice
      const float2 nmu = splat2(-mu_cur);
      float2 s1 = splat2(0.f), s2 = splat2(0.f), s1b = splat2(0.f), s2b = splat2(0.f);
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        mbar_wait(full + s, par, a.err, abort_flag);
        const unsigned char *st = smem + static_cast<size_t>(s) * L.stage_bytes + t * 16;
#pragma unroll
        for (int k = 0; k < kKP; ++k) {
          float2 xf[4], df[4], gf[4];
          chunk_to_f2(lds_v4(st + k * kStride), xf);
          chunk_to_f2(lds_v4(st + L.tensor_bytes + k * kStride), df);
          chunk_to_f2(gv[p][k], gf);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 gg = mul2(df[e], gf[e]);
            const float2 xc = MODE == kLayer ? add2(xf[e], nmu) : xf[e];
            if (e & 1) {
              s2b = fma2(gg, xc, s2b);
              if (MODE == kLayer) s1b = add2(s1b, gg);
            } else {
              s2 = fma2(gg, xc, s2);
              if (MODE == kLayer) s1 = add2(s1, gg);
            }
          }
        }
        release(q, s);
        advance();
      }
      s1 = add2(s1, s1b);
      s2 = add2(s2, s2b);
      // The row's totals without a CTA-wide barrier: each warp posts its
      // butterfly-summed partial; the last warp to post adds the partials
      // in warp order and publishes the CTA total (to every CTA of the
      // cluster, or to this CTA's own exchange slot) while the other warps
      // go on to the next pass.  Same additions in the same order as a
      // barrier-synchronised group sum.
      float v0 = s1.x + s1.y, v1 = s2.x + s2.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (MODE == kLayer) v0 += __shfl_xor_sync(0xffffffffu, v0, o);
        v1 += __shfl_xor_sync(0xffffffffu, v1, o);
      }
      const int rb = xch.push_buf;
      float *slots = wred + rb * kNW * 2;
      if ((t & 31) == 0) {
        slots[2 * warp] = v0;
        slots[2 * warp + 1] = v1;
      }
      if (last_warp_done(wcnt, rb, kNW) && (t & 31) == 0) {
        float A = slots[0], U = slots[1];
        for (int w = 1; w < kNW; ++w) {
          A += slots[2 * w];
          U += slots[2 * w + 1];
        }
        xch_publish<CLUSTER>(A, U, xch);
      }
      xch.push_buf = (rb + 1) % kXchBuffers;
    }
    if (j >= 1) {
      // ---- pass 2 of row j - 1: dx and the column sums
      float A, U;
      {
        const float *row = cluster_wait_row(0, xch, a.err, abort_flag);
        float v[2];
        fold_sum<2>(row, xch.C, v);
        A = v[0];
        U = v[1];
      }
      const float rs = rs_prev;
      // c = mean(g xhat) = rstd U / N; dx = rstd g - rstd a - rstd^2 c (x - mean)
      const float chat = rs * (U * invN);
      const float2 nk1 = splat2(-(rs * rs) * chat);
      const float2 nra = splat2(MODE == kLayer ? -rs * (A * invN) : 0.f);
      const float2 rs2 = splat2(rs), nmu = splat2(-mu_prev);
      uint16_t *dxrow = a.out + (cid + (j - 1) * ncl) * a.N + col0 + t * 8;
      __syncwarp();
      tmem_wait_st();  // the previous pass 2's accumulator stores are complete
      // The accumulators of a piece go through registers in batches of KB
      // chunks (32 registers at most): LayerNorm's dgamma and dbeta take 16
      // TMEM columns per chunk, so its 16384-column pieces take two batches.
      constexpr int KB = (kKP * CPC <= 32) ? kKP : 32 / CPC;
      constexpr int NBAT = kKP / KB;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        uint32_t acc[KB * CPC];
        __syncwarp();
#pragma unroll
        for (int k = 0; k < KB; ++k)
          tmem_ld_n<CPC>(tq + (p * kKP + k) * CPC,
                         *reinterpret_cast<uint32_t(*)[CPC]>(acc + k * CPC));
        mbar_wait(full + s, par, a.err, abort_flag);
        const unsigned char *st = smem + static_cast<size_t>(s) * L.stage_bytes + t * 16;
#pragma unroll
        for (int b = 0; b < NBAT; ++b) {
          __syncwarp();
          if (b > 0) {
#pragma unroll
            for (int k = 0; k < KB; ++k)
              tmem_ld_n<CPC>(tq + (p * kKP + b * KB + k) * CPC,
                             *reinterpret_cast<uint32_t(*)[CPC]>(acc + k * CPC));
          }
          if constexpr (KB * CPC == 16) {
            tmem_wait_ld_n<16>(*reinterpret_cast<uint32_t(*)[16]>(acc));
          } else {
            tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(acc));
          }
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            const int k = b * KB + kb;
            float2 xf[4], df[4], gf[4], o[4];
            chunk_to_f2(lds_v4(st + k * kStride), xf);
            chunk_to_f2(lds_v4(st + L.tensor_bytes + k * kStride), df);
            chunk_to_f2(gv[p][k], gf);
            uint32_t *ak = acc + kb * CPC;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 gg = mul2(df[e], gf[e]);
              const float2 xc = MODE == kLayer ? add2(xf[e], nmu) : xf[e];
              o[e] = fma2(xc, nk1, MODE == kLayer ? fma2(gg, rs2, nra) : mul2(gg, rs2));
              const float2 xh = mul2(xc, rs2);
              float2 ag = make_float2(__uint_as_float(ak[2 * e]), __uint_as_float(ak[2 * e + 1]));
              ag = fma2(df[e], xh, ag);
              ak[2 * e] = __float_as_uint(ag.x);
              ak[2 * e + 1] = __float_as_uint(ag.y);
              if (MODE == kLayer) {
                float2 ab = make_float2(__uint_as_float(ak[8 + 2 * e]),
                                        __uint_as_float(ak[8 + 2 * e + 1]));
                ab = add2(ab, df[e]);
                ak[8 + 2 * e] = __float_as_uint(ab.x);
                ak[8 + 2 * e + 1] = __float_as_uint(ab.y);
              }
            }
            if (RESID) {
              float2 hf[4];
              chunk_to_f2(lds_v4(st + 2 * L.tensor_bytes + k * kStride), hf);
#pragma unroll
              for (int e = 0; e < 4; ++e) o[e] = add2(o[e], hf[e]);
            }
            st_global_cs_v4(dxrow + p * kW + k * kStreamThreads * 8, f2_to_chunk(o));
          }
          __syncwarp();
#pragma unroll
          for (int kb = 0; kb < KB; ++kb)
            tmem_st_n<CPC>(tq + (p * kKP + b * KB + kb) * CPC,
                           *reinterpret_cast<const uint32_t(*)[CPC]>(acc + kb * CPC));
        }
        release(q, s);
        advance();
      }
    }
    rs_prev = rs_cur;
    mu_prev = mu_cur;
    rs_cur = rs_next;
    mu_cur = mu_next;
    load_stats(j + 2, rs_next, mu_next);
  }

  // This cluster's partial row of the workspace: [P][N] dgamma, then
  // [P][N] dbeta (LayerNorm).
  __syncwarp();
  tmem_wait_st();
#pragma unroll
  for (int p = 0; p < NP; ++p) {
#pragma unroll
    for (int k = 0; k < kKP; ++k) {
      uint32_t acc[CPC];
      __syncwarp();
      tmem_ld_n<CPC>(tq + (p * kKP + k) * CPC, acc);
      tmem_wait_ld_n<CPC>(acc);
      const int64_t col = col0 + p * kW + (k * kStreamThreads + t) * 8;
#pragma unroll
      for (int w = 0; w < NACC; ++w) {
        float4 *dst = reinterpret_cast<float4 *>(a.ws + (w * a.P + cid) * a.N + col);
        dst[0] = make_float4(__uint_as_float(acc[8 * w + 0]), __uint_as_float(acc[8 * w + 1]),
                             __uint_as_float(acc[8 * w + 2]), __uint_as_float(acc[8 * w + 3]));
        dst[1] = make_float4(__uint_as_float(acc[8 * w + 4]), __uint_as_float(acc[8 * w + 5]),
                             __uint_as_float(acc[8 * w + 6]), __uint_as_float(acc[8 * w + 7]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, kCols);
  }
  if (CLUSTER) cluster_sync();
}

// Streaming forward for rows too wide for a resident slice: the same piece
// sequence over 32768-column slices (65536 for RMSNorm's 8-piece variant),
// pass 1 the row statistics from HBM, pass 2 y from the L2 copy pass 1 left.
// Statistics per thread: sum x^2 (RMSNorm), or per piece (16 values in
// registers) its mean and sum of squared deviations, merged into a running
// (mean, M2) weighted by counts (LayerNorm); then an equal-count butterfly
// over the warp, the last warp to finish the row folds the 16 warp partials
// pairwise and publishes the CTA's, and the cluster merges its CTAs' in rank
// order.  gamma (and beta) stay in registers.
template <int MODE, int KP, int NP, bool CLUSTER>
__global__ void __launch_bounds__(kStreamThreads, 1) norm_fwd_stream_kernel(const NormArgs a) {
  constexpr int kKP = KP;
  constexpr int kW = stream_piece_cols(KP);
  constexpr int kNW = kStreamThreads / 32;
  constexpr int kStride = kStreamThreads * 16;
  constexpr int kPW = 4;  // floats per warp partial

  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout L = stream_layout(a.S, CLUSTER ? a.C : 1, 1, KP);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  float *wred = reinterpret_cast<float *>(smem + L.red_off);  // [buffer][warp][4]
  int *wcnt = reinterpret_cast<int *>(wred + kXchBuffers * kNW * kPW);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag_off);
  int *done_cnt = reinterpret_cast<int *>(smem + L.flag_off) + 1;

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int crank = CLUSTER ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t cid = CLUSTER ? static_cast<int64_t>(cluster_id_x()) : blockIdx.x;
  const int64_t ncl = CLUSTER ? static_cast<int64_t>(ncluster_x()) : gridDim.x;
  const int64_t col0 = static_cast<int64_t>(crank) * a.NS;
  const int64_t nr = cid < a.M ? (a.M - cid + ncl - 1) / ncl : 0;
  const int64_t total = 2 * NP * nr;

  if (t == 0) {
    for (int s = 0; s < a.S; ++s) {
      mbar_init(full + s, 1);
      done_cnt[s] = 0;
    }
    uint64_t *xb = xch_bars(smem, L, 1, CLUSTER ? a.C : 1);
    for (int b = 0; b < kXchBuffers; ++b) {
      mbar_init(xb + b, 1);
      wcnt[b] = 0;
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  grid_launch_dependents();
  grid_dependency_wait();

  uint4 gv[NP][kKP], bv[NP][kKP];
#pragma unroll
  for (int p = 0; p < NP; ++p)
#pragma unroll
    for (int k = 0; k < kKP; ++k) {
      const int64_t c = col0 + p * kW + (k * kStreamThreads + t) * 8;
      gv[p][k] = ld_global_nc_v4(a.gamma + c);
      bv[p][k] = (MODE == kLayer && a.beta != nullptr) ? ld_global_nc_v4(a.beta + c)
                                                      : make_uint4(0, 0, 0, 0);
    }

  if (CLUSTER) cluster_sync(); else __syncthreads();

  const uint64_t pol1 = l2_normal_policy();
  const uint64_t pol2 = l2_evict_first_policy();
  auto issue = [&](int64_t q, int s) {
    int pass, p;
    int64_t j;
    piece_at(q, NP, nr, pass, j, p);
    const int64_t off = (cid + j * ncl) * a.N + col0 + static_cast<int64_t>(p) * kW;
    uint64_t *bar = full + s;
    mbar_arrive_expect_tx(bar, L.tensor_bytes);
    bulk_g2s(smem + static_cast<size_t>(s) * L.stage_bytes, a.x + off, L.tensor_bytes, bar,
             pass ? pol2 : pol1);
  };
  if (t == 0) {
    for (int64_t q = 0; q < total && q < a.S; ++q) issue(q, static_cast<int>(q));
  }
  auto release = [&](int64_t q, int s) {
    if (last_warp_done(done_cnt, s, kNW)) {
      const int64_t next = q + a.S;
      if (next < total && (t & 31) == 0) {
        fence_proxy_async_smem();
        issue(next, s);
      }
    }
  };

  ClusterXch xch = make_xch(smem, L, 1, CLUSTER ? a.C : 1, crank);
  const float invN = a.invN;
  constexpr float kPerThread = 8.f * kKP * NP;  // elements of a row slice per thread
  int s = 0;
  uint32_t par = 0;
  int64_t q = 0;
  auto advance = [&]() {
    ++q;
    if (++s == a.S) {
      s = 0;
      par ^= 1u;
    }
  };

  for (int64_t j = 0; j <= nr; ++j) {
    if (j < nr) {
      // ---- pass 1 of row j: this thread's statistics, then the CTA's
      float m = 0.f, m2 = 0.f;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        mbar_wait(full + s, par, a.err, abort_flag);
        const unsigned char *st = smem + static_cast<size_t>(s) * L.stage_bytes + t * 16;
        float2 xf[kKP][4];
#pragma unroll
        for (int k = 0; k < kKP; ++k) chunk_to_f2(lds_v4(st + k * kStride), xf[k]);
        release(q, s);
        advance();
        if (MODE == kLayer) {
          float2 s0 = splat2(0.f), s1 = splat2(0.f);
#pragma unroll
          for (int k = 0; k < kKP; ++k) {
            s0 = add2(s0, add2(xf[k][0], xf[k][1]));
            s1 = add2(s1, add2(xf[k][2], xf[k][3]));
          }
          const float2 st2 = add2(s0, s1);
          const float mp = (st2.x + st2.y) * (1.f / (8.f * kKP));
          const float2 nm = splat2(-mp);
          float2 q0 = splat2(0.f), q1 = splat2(0.f);
#pragma unroll
          for (int k = 0; k < kKP; ++k) {
            const float2 d0 = add2(xf[k][0], nm), d1 = add2(xf[k][1], nm);
            const float2 d2 = add2(xf[k][2], nm), d3 = add2(xf[k][3], nm);
            q0 = fma2(d0, d0, fma2(d1, d1, q0));
            q1 = fma2(d2, d2, fma2(d3, d3, q1));
          }
          const float2 qt = add2(q0, q1);
          const float qp = qt.x + qt.y;
          if (p == 0) {
            m = mp;
            m2 = qp;
          } else {
            // running partial over p pieces merged with piece p (counts 16p, 16)
            ms_merge(m, m2, mp, qp, 1.f / static_cast<float>(p + 1),
                     8.f * kKP * static_cast<float>(p) / static_cast<float>(p + 1));
          }
        } else {
          float2 q0 = splat2(0.f), q1 = splat2(0.f);
#pragma unroll
          for (int k = 0; k < kKP; ++k) {
            q0 = fma2(xf[k][0], xf[k][0], fma2(xf[k][1], xf[k][1], q0));
            q1 = fma2(xf[k][2], xf[k][2], fma2(xf[k][3], xf[k][3], q1));
          }
          const float2 qt = add2(q0, q1);
          m2 += qt.x + qt.y;
        }
      }
      // warp: butterfly (equal counts for LayerNorm's merges)
      float h = 0.5f * kPerThread;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float qo = __shfl_xor_sync(0xffffffffu, m2, o);
        if (MODE == kLayer) {
          const float mo = __shfl_xor_sync(0xffffffffu, m, o);
          ms_merge_equal(m, m2, mo, qo, h);
          h *= 2.f;
        } else {
          m2 += qo;
        }
      }
      const int rb = xch.push_buf;
      float *slots = wred + rb * kNW * kPW;
      if ((t & 31) == 0) {
        slots[kPW * warp] = m;
        slots[kPW * warp + 1] = m2;
      }
      if (last_warp_done(wcnt, rb, kNW) && (t & 31) == 0) {
        float M = 0.f, Q = 0.f;
        if (MODE == kLayer) {
          tree_fold<kNW>(slots, 32.f * kPerThread, M, Q);
        } else {
          Q = slots[1];
          for (int w = 1; w < kNW; ++w) Q += slots[kPW * w + 1];
        }
        xch_publish<CLUSTER>(M, Q, xch);
      }
      xch.push_buf = (rb + 1) % kXchBuffers;
    }
    if (j >= 1) {
      // ---- pass 2 of row j - 1: y
      const float *rowx = cluster_wait_row(0, xch, a.err, abort_flag);
      float mu = 0.f, rs;
      if (MODE == kLayer) {
        float mm, qq;
        rank_fold_meanvar(rowx, xch.C, static_cast<float>(a.NS), mm, qq);
        mu = mm;
        rs = rsqrtf(qq * invN + a.eps);
      } else {
        float v[1];
        fold_sum<1>(rowx + 1, xch.C, v);
        rs = rsqrtf(v[0] * invN + a.eps);
      }
      const int64_t row = cid + (j - 1) * ncl;
      if (t == 0 && crank == 0) {
        a.rstd[row] = rs;
        if (MODE == kLayer) a.mean[row] = mu;
      }
      const float2 rs2 = splat2(rs), nmu = splat2(-mu);
      uint16_t *yrow = a.out + row * a.N + col0 + t * 8;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        mbar_wait(full + s, par, a.err, abort_flag);
        const unsigned char *st = smem + static_cast<size_t>(s) * L.stage_bytes + t * 16;
#pragma unroll
        for (int k = 0; k < kKP; ++k) {
          float2 xf[4], gf[4], bf[4], o[4];
          chunk_to_f2(lds_v4(st + k * kStride), xf);
          chunk_to_f2(gv[p][k], gf);
          if (MODE == kLayer) chunk_to_f2(bv[p][k], bf);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 xh = mul2(MODE == kLayer ? add2(xf[e], nmu) : xf[e], rs2);
            o[e] = (MODE == kLayer) ? fma2(xh, gf[e], bf[e]) : mul2(xh, gf[e]);
          }
          st_global_cs_v4(yrow + p * kW + k * kStreamThreads * 8, f2_to_chunk(o));
        }
        release(q, s);
        advance();
      }
    }
  }
  if (CLUSTER) cluster_sync();
}

template <int MODE, int KP, int NP>
const void *stream_fwd_ptr(bool cluster) {
  return cluster ? reinterpret_cast<const void *>(&norm_fwd_stream_kernel<MODE, KP, NP, true>)
                 : reinterpret_cast<const void *>(&norm_fwd_stream_kernel<MODE, KP, NP, false>);
}

template <int MODE, int KP, bool RESID>
const void *stream_ptr(bool cluster) {
  return cluster ? reinterpret_cast<const void *>(&norm_bwd_stream_kernel<MODE, KP, true, RESID>)
                 : reinterpret_cast<const void *>(&norm_bwd_stream_kernel<MODE, KP, false, RESID>);
}

}  // namespace

// Instantiated: 4 chunks per thread per piece (16384-column pieces, the
// default of the plain backward; LayerNorm's dx pass moves its dgamma and
// dbeta accumulators through registers in batches) and 2 (8192, the fused
// residual backward's default and the W=8192 override) for both modes.
const void *stream_kernel_ptr(int mode, int kp, bool cluster, bool resid) {
  if (mode == kLayer) {
    if (kp == 4) return resid ? stream_ptr<kLayer, 4, true>(cluster) : stream_ptr<kLayer, 4, false>(cluster);
    if (kp == 2) return resid ? stream_ptr<kLayer, 2, true>(cluster) : stream_ptr<kLayer, 2, false>(cluster);
    return nullptr;
  }
  if (kp == 4) return resid ? stream_ptr<kRMS, 4, true>(cluster) : stream_ptr<kRMS, 4, false>(cluster);
  if (kp == 2) return resid ? stream_ptr<kRMS, 2, true>(cluster) : stream_ptr<kRMS, 2, false>(cluster);
  return nullptr;
}

// Forward: RMSNorm with 16384-column pieces, two or four per slice (32768 or
// 65536 columns); LayerNorm with four 8192-column pieces.
const void *stream_fwd_kernel_ptr(int mode, int kp, int np, bool cluster) {
  if (mode == kLayer) return (kp == 2 && np == 4) ? stream_fwd_ptr<kLayer, 2, 4>(cluster) : nullptr;
  if (kp != 4) return nullptr;
  if (np == 2) return stream_fwd_ptr<kRMS, 4, 2>(cluster);
  if (np == 4) return stream_fwd_ptr<kRMS, 4, 4>(cluster);
  return nullptr;
}

}  // namespace gbn
