// gemm.cu -- normalisation fused into the prologue of a tcgen05 GEMM
// (norm_gemm_prepare / norm_gemm_fwd in include/gbnorm.h).
//
// out = norm(x) W^T with x [M, K] and W [Nout, K] in bf16 (one W row per
// output feature), out bf16 [M, Nout].  Item 4 of the page "Towards Free
// Normalization: Fusing Normalization into GEMM and Attention Kernels" names
// the Lazy Pre-Norm fusion, and its items 9 and 10 the obstacle: the
// normalisation wants whole rows while a GEMM tiles rows and columns.  Here
// the normalisation is moved past the contraction, which is linear in the
// normalised row:
//
//   out_ik = rstd_i * (sum_j x_ij W'_kj - mean_i * u_k) + v_k
//   W' = bf16(W * gamma) (gamma scales the columns j), u = W' 1, v = W beta
//
// (mean = 0 and v = 0 for RMSNorm).  W', u and v depend on the weights only
// and are made once by norm_gemm_prepare.  The GEMM then streams raw x
// tiles through shared memory; four warps take each row's statistics from
// the same tiles the tensor cores read, and the epilogue applies rstd and
// the mean correction while it drains the fp32 accumulator from tensor
// memory.  x reaches the SM once per output tile column (mostly from L2),
// and the normalised rows are never written.
//
// A persistent grid (one CTA per SM, 12 warps) walks the output tiles in
// units of 1 to 8 consecutive column tiles of one row block, dealt
// round-robin in the grouped order of tile_coords.  By default 2-CTA
// clusters (PAIR) share 256 x 256 tiles with cta_group::2 MMAs, each CTA
// holding 128 x rows and 128 W' rows per stage (6 stages); the single-CTA
// form takes 128 x 256 tiles (4 stages).  Per CTA:
//   warp 0      (lane 0) issues the tiled TMA loads of the x and W' tiles
//               into the stage ring (128-byte swizzle);
//   warp 1      (lane 0; rank 0 of a pair) issues the tcgen05.mma
//               instructions, 4 per 64-wide K block, into one of two
//               256-column fp32 accumulators in tensor memory, and commits
//               each stage back to the producers;
//   warp 2      allocates (and at the end frees) the 512 TMEM columns;
//   warps 8-11  the statistics of the current unit's 128 rows, from the x
//               tiles of its first tile, handed to the epilogue through a
//               shared-memory slot;
//   warps 4-7   the epilogue of the previous tile, on TMEM lane t = row t,
//               while the tensor cores fill the other accumulator; output
//               through two swizzled staging buffers and TMA tensor stores.
// Row statistics use shifted sums: the mean of the row's first 64 values,
// rounded to bf16, is the shift c, and sum(x - c), sum((x - c)^2) give the
// mean and the population variance without the cancellation of raw power
// sums.
// Every wait is bounded: a lost copy or MMA sets the device error word, the
// CTA still waits (bounded) for its own copies and MMAs in flight, frees its
// tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <tuple>
#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/gbnorm.h"
#include "common.cuh"
#include "rowops.cuh"
#include "tcgen05.cuh"

namespace gbn {

// Device error word and shape of the current device (api.cu).
norm_status_t device_context(int *dev, int *sms, int *smem_optin, unsigned **err,
                             unsigned long long *ctx);

namespace {

constexpr int kBM = 128;       // rows per CTA (TMEM lanes)
constexpr int kBN = 256;       // tile columns (fp32 TMEM columns per accumulator)
constexpr int kBK = 64;        // K block: one 128-byte swizzle row of bf16
constexpr int kUK = 16;        // K per tcgen05.mma of kind::f16
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;   // warps 4-7: TMEM lane quarters 0-3
constexpr int kStatWarp0 = 8;  // warps 8-11
constexpr uint32_t kATile = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kTmemCols = 2 * kBN;     // two accumulators: all 512 columns
constexpr int kOutCols = 64;                  // output columns per TMA store box
constexpr uint32_t kOutTile = kBM * kOutCols * 2;  // 16 KB per staging buffer (two)

// Per-CTA geometry.  One CTA holds all 256 W' rows of its tile (4 stages of
// 48 KB); in a CTA pair each holds 128 of them (6 stages of 32 KB).  Shared
// memory: ring, two output staging buffers, mbarriers, TMEM address slot
// and abort flag, one slot of per-row (rstd, mean); plus slack to align the
// ring to 1024 bytes (the 128-byte swizzle atom is 8 rows of 128 bytes).
// Kernel forms: one CTA per 128 x 256 tile, or a CTA pair sharing one
// cta_group::2 MMA per 256 x 256 tile.
constexpr int kFormSingle = 0;
constexpr int kFormPair = 1;

template <int FORM>
struct Geo {
  static constexpr int kCtas = FORM == kFormSingle ? 1 : 2;  // CTAs per cluster
  static constexpr int kStages = FORM == kFormPair ? 6 : 4;
  // W' rows held per CTA and stage (the pair splits the tile's 256 rows)
  static constexpr int kBRows = FORM == kFormPair ? kBN / 2 : kBN;
  static constexpr uint32_t kBTile = kBRows * kBK * 2;
  static constexpr uint32_t kStageBytes = kATile + kBTile;
  static constexpr int kNumBars = 2 * kStages + 8 + 1;
  static constexpr uint32_t kSmemBytes =
      1024 + kStages * kStageBytes + 2 * kOutTile + 256 + kBM * 8;
  static_assert(kNumBars * 8 + 8 <= 256, "barrier region");
};

static_assert(kBK * 2 == 128, "one K block is one 128-byte swizzled row");
static_assert(kBN % 32 == 0 && kBN <= 256 && kBM == 128, "tcgen05 tile shape");

// Tile walk: groups of row blocks spanning kGroupRows rows (16 blocks of
// 128 rows for the single CTA, 8 of 256 for a pair), each group taken
// column by column (row block fastest).  The tiles in flight then cover a
// block of about 2048 rows x 2400 columns instead of a few whole row
// blocks, so the x and W' tiles they read stay in L2 even when W' is larger
// than L2.  (Pairs over 16 blocks of 256 rows read 1.9x the algorithmic
// bytes from DRAM at 32768 x 4096 x 4096, over 8 blocks 1.5x, 1-2 % faster.)
constexpr int kGroupRows = 2048;

__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int gm,
                                            int &m_blk, int &n_blk) {
  const int per_group = gm * n_tiles;
  const int group = tile / per_group;
  const int first = group * gm;
  const int rows = min(gm, m_tiles - first);
  const int idx = tile - group * per_group;
  m_blk = first + idx % rows;
  n_blk = idx / rows;
}

// PAIR: the grid is made of 2-CTA clusters; each pair computes 256 x 256
// tiles with cta_group::2 MMAs issued by rank 0 (M = 256: 128 rows and 128
// W' rows per CTA).  All four loads of a stage count on rank 0's full
// barrier; the MMA commit frees the stage in both CTAs and also completes
// rank 1's full barrier, after which rank 1's statistics warps read its x
// tile (the MMA has read it, so it has landed).  Rank 1's epilogue warps
// release the accumulator on rank 0.
template <int MODE, int FORM>
__global__ void __launch_bounds__(kThreads, 1)
    norm_gemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_out, const float *__restrict__ u,
                     const float *__restrict__ v,
                     float *__restrict__ rstd, float *__restrict__ mean, int M, int K, int Nout,
                     float eps, uint32_t tx_bytes, int rgrp, int gm, unsigned *err) {
  constexpr bool PAIR = FORM == kFormPair;
  constexpr bool CLUSTER = FORM != kFormSingle;
  using G = Geo<FORM>;
  constexpr int kStages = G::kStages;
  constexpr uint32_t kBTile = G::kBTile;
  constexpr uint32_t kStageBytes = G::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t *ring = smem_raw + pad;
  uint8_t *a_tiles = ring;
  uint8_t *b_tiles = ring + kStages * kATile;
  uint8_t *staging = ring + kStages * kStageBytes;  // [2][kOutTile]
  uint64_t *full = reinterpret_cast<uint64_t *>(staging + 2 * kOutTile);
  uint64_t *empty = full + kStages;      // [kStages]
  uint64_t *acc_full = empty + kStages;  // [2] accumulator complete
  uint64_t *acc_empty = acc_full + 2;    // [2] accumulator drained
  uint64_t *st_full = acc_empty + 2;     // row statistics of a tile written
  uint64_t *st_empty = st_full + 1;      // ... and read by the epilogue
  uint64_t *done = st_empty + 1;         // every MMA of the CTA finished
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float2 *stats = reinterpret_cast<float2 *>(staging + 2 * kOutTile + 256);  // [kBM]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = CLUSTER ? cluster_ctarank() : 0u;
  const int unit0 = blockIdx.x / G::kCtas;  // this CTA's (cluster's) first unit
  const int nunits = gridDim.x / G::kCtas;  // unit stride
  const int nk = K / kBK;
  const int n_tiles = (Nout + kBN - 1) / kBN;
  const int m_tiles = (M + kBM * G::kCtas - 1) / (kBM * G::kCtas);
  // A unit is rgrp consecutive column tiles of one row block (rgrp divides
  // n_tiles); units are dealt to the CTAs (pairs) round-robin in the
  // grouped order of tile_coords, and each takes its unit's tiles in turn,
  // so the row statistics are computed once per unit.  tile_at gives the
  // j-th tile of this CTA (false past the last one).
  const int n_groups = n_tiles / rgrp;
  const int nunits_all = m_tiles * n_groups;
  auto tile_at = [&](int j, int &mb, int &nb) {
    const int unit = unit0 + (j / rgrp) * nunits;
    if (unit >= nunits_all) return false;
    int ngb;
    tile_coords(unit, m_tiles, n_groups, gm, mb, ngb);
    nb = ngb * rgrp + j % rgrp;
    return true;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // its producer's arrival with the byte count of the stage (rank 1 of
      // a pair: rank 0's MMA commit instead)
      mbar_init(&full[s], 1);
      // the MMA commit and one arrival per statistics warp
      mbar_init(&empty[s], 1 + 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      // rank 1's four epilogue warps also release rank 0's accumulator slot
      mbar_init(&acc_empty[b], PAIR ? 128 + 4 : 128);
    }
    mbar_init(st_full, 128);
    mbar_init(st_empty, 128);
    mbar_init(done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (CLUSTER)
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = l2_evict_last_policy();
      int g = 0;  // K blocks issued by this CTA (all tiles)
      bool ok = true;
      const uint32_t full_rank0 = PAIR ? mapa_shared(full, 0) : 0u;
      int mb, nb;
      for (int j = 0; ok && tile_at(j, mb, nb); ++j) {
        const int m0 = (mb * G::kCtas + int(rank)) * kBM;
        // this CTA's W' rows: all 256 (single), or its half (pair)
        const int n0 = nb * kBN + (CLUSTER ? int(rank) * (kBN / 2) : 0);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % kStages;
          if (g >= kStages) {
            if (!mbar_wait(&empty[s], (g / kStages - 1) & 1, err, abort)) {
              ok = false;
              break;
            }
            // The statistics warps read the stage through the generic
            // proxy; order those reads before the asynchronous-proxy refill.
            fence_proxy_async_smem();
          }
          if (PAIR && rank != 0) {  // counted on rank 0's barrier, where the MMA waits
            tma_load_2d_pair(a_tiles + s * kATile, &tm_x, kb * kBK, m0,
                             full_rank0 + uint32_t(s * 8));
            tma_load_2d_pair(b_tiles + s * kBTile, &tm_w, kb * kBK, n0,
                             full_rank0 + uint32_t(s * 8));
          } else {
            // W' tiles are read again by every row block: kept in L2 ahead
            // of the x stream and of the output (written once, evict-first)
            mbar_arrive_expect_tx(&full[s], tx_bytes);
            tma_load_2d(a_tiles + s * kATile, &tm_x, kb * kBK, m0, &full[s]);
            tma_load_2d_hint(b_tiles + s * kBTile, &tm_w, kb * kBK, n0, &full[s], pol_w);
          }
        }
      }
      // No copy may still be landing in shared memory when the CTA exits.
      volatile int never = 0;
      for (int s = 0; s < kStages && s < g; ++s) {
        const int loads = (g - s + kStages - 1) / kStages;
        mbar_wait(&full[s], (loads - 1) & 1, err, &never);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0 && (!PAIR || rank == 0)) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM * (PAIR ? 2 : 1), kBN);
      auto commit = [&](uint64_t *bar) {
        if (PAIR)
          mma_commit_pair(bar, 0x3);
        else
          mma_commit(bar);
      };
      bool ok = true;
      int mb, nb;
      // One thread issues every MMA and the tensor pipe holds only a few
      // queued instructions, so the per-K-block bookkeeping of this loop is
      // on the critical path: descriptors and barrier addresses are formed
      // by one add each from values taken once.
      const uint64_t adesc0 = desc_sw128(smem_addr(a_tiles));
      const uint64_t bdesc0 = desc_sw128(smem_addr(b_tiles));
      const uint32_t full0 = smem_addr(full), empty0 = smem_addr(empty);
      int s = 0;
      uint32_t ph = 0;
      for (int j = 0; ok && tile_at(j, mb, nb); ++j) {
        const int b = j & 1;
        // rank 1's epilogue also releases this slot (a generic arrival from
        // the other CTA: acquired at cluster scope)
        if (j >= 2 && !(PAIR ? mbar_wait_cluster(&acc_empty[b], ((j >> 1) - 1) & 1, err, abort)
                             : mbar_wait(&acc_empty[b], ((j >> 1) - 1) & 1, err, abort)))
          break;
        tc_fence_after();
        const uint32_t d = tmem + uint32_t(b * kBN);
        for (int kb = 0; kb < nk; ++kb) {
          const uint32_t fb = full0 + 8u * uint32_t(s);
          if (!mbar_try_wait_sa(fb, ph) && !mbar_wait_sa(fb, ph, err, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // start address field (bits 0-13, address / 16): + stage offset,
          // + 2 per 16-element K step (32 bytes)
          const uint64_t ad = adesc0 + uint32_t(s * int(kATile >> 4));
          const uint64_t bd = bdesc0 + uint32_t(s * int(kBTile >> 4));
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k) {
            if (PAIR)
              mma_bf16_ss_pair(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
            else
              mma_bf16_ss(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
          }
          // the stage is free once these MMAs have read it
          if (PAIR) {
            mma_commit_pair_sa(empty0 + 8u * uint32_t(s), 0x3);
            mma_commit_pair_sa(fb, 0x2);  // rank 1's x tile: readable now
          } else {
            mma_commit_sa(empty0 + 8u * uint32_t(s));
          }
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) commit(&acc_full[b]);
      }
      commit(done);  // arrives when every MMA issued above has completed
    }
    __syncwarp();
  } else if (warp >= kStatWarp0) {
    // ------------------------------------------------ row statistics
    // Warp w of the four takes rows 32w .. 32w + 31.  In each 64-wide K
    // block, load i (0..7) has lane l read 16-byte chunk l % 8 of row
    // 32w + 4i + l / 8: eight lanes read one whole 128-byte row line, so the
    // lanes of a load never share a bank, whatever the swizzle.  Each lane
    // keeps partial sums of its chunk for its eight rows; the eight lanes of
    // a row combine them once per tile (and once for the LayerNorm shift).
    // The chunk order within a row does not matter to a sum.
    const int sw = warp - kStatWarp0;
    const int sub = lane >> 3;  // row within each group of four
    const int part = lane & 7;  // chunk of the row line
    int g = 0;
    int mb, nb;
    float r[8], mu[8];  // statistics of the current unit's rows
    for (int j = 0; tile_at(j, mb, nb); ++j) {
      const bool fresh = (j % rgrp) == 0;  // first tile of a unit: take the statistics
      float2 s1[8], s2[8];
      float c[8];  // shift (LayerNorm): mean of the row's first 64 values
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        s1[i] = s2[i] = make_float2(0.f, 0.f);
        c[i] = 0.f;
      }
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int s = g % kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (g / kStages) & 1, err, abort));
        if (!ok) break;
        if (!fresh) {  // statistics already known: just hand the stage back
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          continue;
        }
        const uint8_t *base = a_tiles + s * kATile + (32 * sw + sub) * 128 + part * 16;
        uint4 q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = *reinterpret_cast<const uint4 *>(base + i * 4 * 128);
        if (MODE == kLayer && kb == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float2 f[4];
            chunk_to_f2(q[i], f);
            const float2 a2 = add2(add2(f[0], f[1]), add2(f[2], f[3]));
            float a = a2.x + a2.y;
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            // Rounded to bf16, so that x - c is exact in fp32 (two 8-bit
            // significands less than 2^16 apart in magnitude); an fp32
            // shift would round every difference the same way and bias the
            // sum.
            c[i] = __bfloat162float(__float2bfloat16_rn(a * (1.f / kBK)));
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float2 f[4];
          chunk_to_f2(q[i], f);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (MODE == kRMS) {
              s2[i] = fma2(f[e], f[e], s2[i]);
            } else {
              const float2 dv = add2(f[e], splat2(-c[i]));
              s1[i] = add2(s1[i], dv);
              s2[i] = fma2(dv, dv, s2[i]);
            }
          }
        }
        // The stage is released only after its values have been consumed:
        // an arrival right after the loads were issued let the refill land
        // under loads still in flight.
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (!ok) break;
      const float invK = 1.f / float(K);
#pragma unroll
      for (int i = 0; i < 8 && fresh; ++i) {
        float q2 = s2[i].x + s2[i].y;
        q2 += __shfl_xor_sync(0xffffffffu, q2, 1);
        q2 += __shfl_xor_sync(0xffffffffu, q2, 2);
        q2 += __shfl_xor_sync(0xffffffffu, q2, 4);
        float var;
        mu[i] = 0.f;
        if (MODE == kRMS) {
          var = q2 * invK;
        } else {
          float q1 = s1[i].x + s1[i].y;
          q1 += __shfl_xor_sync(0xffffffffu, q1, 1);
          q1 += __shfl_xor_sync(0xffffffffu, q1, 2);
          q1 += __shfl_xor_sync(0xffffffffu, q1, 4);
          const float d1 = q1 * invK;  // mean - c
          var = fmaxf(fmaf(-d1, d1, q2 * invK), 0.f);
          mu[i] = c[i] + d1;
        }
        r[i] = rsqrtf(var + eps);
      }
      // one slot: the epilogue has read the previous tile's statistics
      if (j >= 1 &&
          !__all_sync(0xffffffffu, mbar_wait(st_empty, (j - 1) & 1, err, abort)))
        break;
      const int m0 = (mb * G::kCtas + int(rank)) * kBM;
      if (part == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = 32 * sw + 4 * i + sub;
          stats[t] = make_float2(r[i], mu[i]);
          if (nb == 0 && m0 + t < M) {
            rstd[m0 + t] = r[i];
            if (MODE == kLayer) mean[m0 + t] = mu[i];
          }
        }
      }
      mbar_arrive(st_full);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------ epilogue
    // Thread t drains TMEM lane t (row t of the tile) 64 columns at a time
    // into a 128-byte-swizzled staging buffer (chunk q of row t at position
    // q ^ (t % 8)), from which one thread writes the 128 x 64 box with a TMA
    // store; rows beyond M and columns beyond Nout are clipped by the store.
    const int t = threadIdx.x - kEpiWarp0 * 32;  // row of the tile = TMEM lane
    const uint64_t pol_out = l2_evict_first_policy();
    const int quarter = warp - kEpiWarp0;        // == warp % 4: TMEM lanes 32q .. 32q + 31
    const uint32_t acc_empty_rank0 = PAIR ? mapa_shared(acc_empty, 0) : 0u;
    int mb, nb;
    int slice = 0;  // 64-column slices stored so far (staging buffer slice % 2)
    for (int j = 0; tile_at(j, mb, nb); ++j) {
      const int b = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      // The four epilogue warps meet at named barriers below, so they never
      // leave the loop early: after a lost wait (error recorded, abort
      // raised, later waits give up at once) they carry on with whatever
      // the accumulator holds.
      mbar_wait(&acc_full[b], ph, err, abort);
      mbar_wait(st_full, j & 1, err, abort);
      __syncwarp();
      tc_fence_after();
      const float2 rm = stats[t];
      mbar_arrive(st_empty);
      const float r = rm.x, mu = rm.y;
      const int m0 = (mb * G::kCtas + int(rank)) * kBM;
      const int n0 = nb * kBN;
      const uint32_t t_lane = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(b * kBN);
#pragma unroll 1
      for (int h = 0; h < kBN / kOutCols; ++h) {
        const int n = n0 + h * kOutCols;
        if (n >= Nout) break;  // the same for the whole CTA
        uint32_t pk[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t acc[32];
          tmem_ld32(t_lane + h * kOutCols + half * 32, acc);
          tmem_wait_ld(acc);
          if (n + half * 32 >= Nout) {  // Nout % 64 == 32: nothing to read or store here
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[half * 16 + e] = 0u;
          } else if (MODE == kRMS) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[half * 16 + e] = f2_to_bf2(mul2(
                  splat2(r), make_float2(__uint_as_float(acc[2 * e]), __uint_as_float(acc[2 * e + 1]))));
          } else {
            const float4 *u4 = reinterpret_cast<const float4 *>(u + n + half * 32);
            const float4 *v4 = reinterpret_cast<const float4 *>(v + n + half * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 uu = __ldg(u4 + q);
              const float4 vv = __ldg(v4 + q);
              const float2 a0 = make_float2(__uint_as_float(acc[4 * q]),
                                            __uint_as_float(acc[4 * q + 1]));
              const float2 a1 = make_float2(__uint_as_float(acc[4 * q + 2]),
                                            __uint_as_float(acc[4 * q + 3]));
              const float2 o0 = fma2(splat2(r), fma2(splat2(-mu), make_float2(uu.x, uu.y), a0),
                                     make_float2(vv.x, vv.y));
              const float2 o1 = fma2(splat2(r), fma2(splat2(-mu), make_float2(uu.z, uu.w), a1),
                                     make_float2(vv.z, vv.w));
              pk[half * 16 + 2 * q] = f2_to_bf2(o0);
              pk[half * 16 + 2 * q + 1] = f2_to_bf2(o1);
            }
          }
        }
        if (h == kBN / kOutCols - 1 || n + kOutCols >= Nout) {
          // this lane's accumulator columns are all read
          tc_fence_before();
          if (PAIR && rank != 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc_empty_rank0 + uint32_t(b * 8));
          } else {
            mbar_arrive(&acc_empty[b]);
          }
        }
        // Two staging buffers in turn: the one about to be written is free
        // once the store issued from it two slices ago has read it.
        uint8_t *sbuf = staging + (slice & 1) * kOutTile;
        ++slice;
        if (t == 0) bulk_wait_read_but_one();
        named_bar_sync(1, 128);
        uint8_t *srow = sbuf + t * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4 *>(srow + ((q ^ (t & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        fence_proxy_async_smem();  // generic writes -> the store's async-proxy reads
        named_bar_sync(1, 128);
        if (t == 0 && m0 < M) {  // rank 1 of a pair may own no row of a short last tile
          tma_store_2d_hint(&tm_out, n, m0, sbuf, pol_out);
          bulk_commit();
        }
      }
    }
    if (t == 0) bulk_wait_all();  // every output store is complete before exit
  }

  // Teardown: every MMA has finished before the tensor memory is freed, and
  // (pair) neither CTA exits while the other may still signal it.
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    if (lane == 0) {
      volatile int never = 0;
      mbar_wait(done, 0, err, &never);
    }
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
  if (CLUSTER) cluster_sync();
}

// W' = bf16(W * gamma) per column, u = row sums of W' and v = W beta (fp32,
// fixed order: each lane strides the row in 8-element chunks, then a
// butterfly over the warp).  One warp per W row.
__global__ void __launch_bounds__(256)
    norm_gemm_prepare_kernel(const uint16_t *__restrict__ w, const uint16_t *__restrict__ gamma,
                             const uint16_t *__restrict__ beta, int K, int Nout,
                             uint16_t *__restrict__ wg, float *__restrict__ u,
                             float *__restrict__ v) {
  const int o = blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (o >= Nout) return;
  const uint16_t *wr = w + size_t(o) * K;
  uint16_t *gr = wg + size_t(o) * K;
  float su = 0.f, sv = 0.f;
  for (int j = lane * 8; j < K; j += 256) {
    float2 wv[4], gv[4], p[4], pr[4];
    chunk_to_f2(ld_global_nc_v4(wr + j), wv);
    chunk_to_f2(ld_global_nc_v4(gamma + j), gv);
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = mul2(wv[e], gv[e]);  // exact: 8-bit x 8-bit significands
    const uint4 pc = f2_to_chunk(p);
    *reinterpret_cast<uint4 *>(gr + j) = pc;
    chunk_to_f2(pc, pr);
#pragma unroll
    for (int e = 0; e < 4; ++e) su = (su + pr[e].x) + pr[e].y;
    if (beta) {
      float2 bv[4];
      chunk_to_f2(ld_global_nc_v4(beta + j), bv);
#pragma unroll
      for (int e = 0; e < 4; ++e) sv = fmaf(wv[e].y, bv[e].y, fmaf(wv[e].x, bv[e].x, sv));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    su += __shfl_xor_sync(0xffffffffu, su, off);
    sv += __shfl_xor_sync(0xffffffffu, sv, off);
  }
  if (lane == 0) {
    if (u) u[o] = su;
    if (v) v[o] = sv;
  }
}

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::set<std::pair<unsigned long long, const void *>> g_attr_done;  // (context, kernel)

norm_status_t encoder(PFN_cuTensorMapEncodeTiled_v12000 *out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      return NORM_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return NORM_OK;
}

// Row-major bf16 [rows, cols] with boxes of box_rows x 64 columns, 128-byte
// swizzle, zero fill outside the tensor.
norm_status_t make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                       uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  norm_status_t st = encoder(&enc);
  if (st != NORM_OK) return st;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {cuuint32_t(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NORM_OK : NORM_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// x, W' and out are moved by tiled tensor copies, whose tensor maps take a
// global address this GPU can reach: device memory of the current device
// (or managed memory).  Host memory, another device's memory and addresses
// unknown to CUDA are refused before a map is built.
norm_status_t check_device_memory(const void *p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_MEMORY;
  }
  if (a.type == cudaMemoryTypeManaged) return NORM_OK;
  return (a.type == cudaMemoryTypeDevice && a.device == dev) ? NORM_OK : NORM_ERR_MEMORY;
}

// Kernel form: the CTA pair (cta_group::2) by default, GBNORM_GEMM_CTAS=1
// the single-CTA kernel.  Measured on GB300 at M = 32768, K = Nout from 2048
// to 8192 (one box, TF/s): RMSNorm pair 1498-1578 against single 1453-1497,
// LayerNorm 1407-1528 against 1364-1462.  The pair's per-SM operand traffic
// (shared-memory writes by TMA and reads by the tensor core) is two thirds
// of the single CTA's, and once the MMA issuer's per-K-block bookkeeping was
// cut (it is one thread on the critical path) that is what showed.
int gemm_form() {
  const char *s = std::getenv("GBNORM_GEMM_CTAS");
  if (s && std::strcmp(s, "1") == 0) return kFormSingle;
  return kFormPair;
}

uint32_t form_smem(int form) {
  return form == kFormPair ? Geo<kFormPair>::kSmemBytes : Geo<kFormSingle>::kSmemBytes;
}

// Co-resident 2-CTA clusters of a cluster form, per (device, mode, form)
// (GBNORM_GEMM_PAIRS=n launches n clusters instead, for sweeps).
std::map<std::tuple<int, int, int>, int> g_pairs;

norm_status_t check_shape(int64_t M, int64_t K, int64_t Nout) {
  if (M < 1 || M > int64_t(65535) * kBM) return NORM_ERR_SHAPE;
  if (K < kBK || K > NORM_MAX_N_FUSED || K % kBK != 0) return NORM_ERR_SHAPE;
  if (Nout < 32 || Nout > (int64_t(1) << 20) || Nout % 32 != 0) return NORM_ERR_SHAPE;
  return NORM_OK;
}

}  // namespace

const void *norm_gemm_kernel_ptr(int mode, int form) {
  const bool rms = mode == kRMS;
  switch (form) {
    case kFormPair:
      return rms ? reinterpret_cast<const void *>(&norm_gemm_kernel<kRMS, kFormPair>)
                 : reinterpret_cast<const void *>(&norm_gemm_kernel<kLayer, kFormPair>);
    default:
      return rms ? reinterpret_cast<const void *>(&norm_gemm_kernel<kRMS, kFormSingle>)
                 : reinterpret_cast<const void *>(&norm_gemm_kernel<kLayer, kFormSingle>);
  }
}

}  // namespace gbn

using namespace gbn;

extern "C" {

norm_status_t norm_gemm_prepare(const void *w, const void *gamma, const void *beta, int64_t K,
                                int64_t Nout, norm_mode_t mode, void *wg, float *u, float *v,
                                norm_stream_t stream) {
  if (mode != NORM_RMS && mode != NORM_LAYER) return NORM_ERR_MODE;
  if (!w || !gamma || !wg) return NORM_ERR_NULL;
  if (mode == NORM_RMS && beta) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && (!u || !v)) return NORM_ERR_MODE;
  norm_status_t st = check_shape(1, K, Nout);
  if (st != NORM_OK) return st;
  const void *ptrs[] = {w, gamma, beta, wg, u, v};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return NORM_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  norm_gemm_prepare_kernel<<<unsigned((Nout + 7) / 8), 256, 0, s>>>(
      static_cast<const uint16_t *>(w), static_cast<const uint16_t *>(gamma),
      static_cast<const uint16_t *>(beta), int(K), int(Nout), static_cast<uint16_t *>(wg), u,
      v);
  if (cudaGetLastError() != cudaSuccess) return NORM_ERR_CUDA;
  return NORM_OK;
}

norm_status_t norm_gemm_fwd(const void *x, const void *wg, const float *u, const float *v,
                            int64_t M, int64_t K, int64_t Nout, float eps, norm_mode_t mode,
                            void *out, float *rstd, float *mean, norm_stream_t stream) {
  if (mode != NORM_RMS && mode != NORM_LAYER) return NORM_ERR_MODE;
  if (!x || !wg || !out || !rstd) return NORM_ERR_NULL;
  if (mode == NORM_RMS && mean) return NORM_ERR_MODE;
  if (mode == NORM_LAYER && (!mean || !u || !v)) return NORM_ERR_MODE;
  norm_status_t st = check_shape(M, K, Nout);
  if (st != NORM_OK) return st;
  if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
  const void *ptrs[] = {x, wg, u, v, out, rstd, mean};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return NORM_ERR_ALIGN;

  int dev = 0, sms = 0, optin = 0;
  unsigned *err = nullptr;
  unsigned long long ctx = 0;
  if ((st = device_context(&dev, &sms, &optin, &err, &ctx)) != NORM_OK) return st;
  const void *moved[] = {x, wg, out};
  for (const void *p : moved)
    if ((st = check_device_memory(p, dev)) != NORM_OK) return st;
  const int form = gemm_form();
  const bool cluster = form != kFormSingle;
  const uint32_t smem = form_smem(form);
  if (optin < int(smem)) return NORM_ERR_UNSUPPORTED;
  const void *fn = norm_gemm_kernel_ptr(mode, form);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_attr_done.count({ctx, fn})) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
          cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
      }
      g_attr_done.insert({ctx, fn});
    }
  }
  // Boxes no taller than the tensor: a tile's rows beyond M (or Nout) are
  // then left as they were in shared memory; they only reach accumulator
  // rows (columns) that are never stored.  Per K block: the single CTA
  // expects its x box and its 256-row W' box; rank 0 of a pair the x and
  // W' boxes of both CTAs.
  const int ctas = cluster ? 2 : 1;
  const int brows = cluster ? kBN / 2 : kBN;
  const uint32_t box_x = uint32_t(M < kBM ? M : kBM);
  const uint32_t box_w = uint32_t(Nout < brows ? Nout : brows);
  uint32_t tx = form == kFormPair ? 2 * (box_x + box_w) * kBK * 2 : (box_x + box_w) * kBK * 2;
  CUtensorMap tm_x, tm_w, tm_o;
  if ((st = make_map(&tm_x, x, M, K, box_x)) != NORM_OK) return st;
  if ((st = make_map(&tm_w, wg, Nout, K, box_w)) != NORM_OK) return st;
  if ((st = make_map(&tm_o, out, M, Nout, box_x)) != NORM_OK) return st;

  const int64_t m_blocks = (M + int64_t(kBM) * ctas - 1) / (int64_t(kBM) * ctas);
  const int64_t n_tiles = (Nout + kBN - 1) / kBN;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  int pairs = 0;  // co-resident 2-CTA clusters (cluster forms)
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  if (cluster) {
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      auto it = g_pairs.find({dev, int(mode), form});
      if (it != g_pairs.end()) pairs = it->second;
    }
    if (const char *ov = std::getenv("GBNORM_GEMM_PAIRS")) pairs = std::atoi(ov);
    if (pairs == 0) {
      cfg.gridDim = dim3(unsigned(sms - sms % 2));
      if (cudaOccupancyMaxActiveClusters(&pairs, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return NORM_ERR_CUDA;
      }
      if (pairs < 1) return NORM_ERR_UNSUPPORTED;
      std::lock_guard<std::mutex> lk(g_mu);
      g_pairs[{dev, int(mode), form}] = pairs;
    }
  }
  // Column tiles per unit (statistics computed once per unit): the largest
  // of 8, 5, 4, 2 that divides the column tiles and adds at most 5 % to the
  // most tiles any CTA (pair) runs.  CTA pairs, TF/s at K = Nout = 2048 /
  // 3072 / 4096 / 5120 / 8192, RMSNorm: one tile per unit 1605 / 1590 /
  // 1611 / 1536 / 1526, two 1678 / 1614 / 1618 / 1578 / 1573; on another
  // box at 5120 four 1637, five 1675, at 8192 four 1614, eight 1644;
  // LayerNorm at 5120 four 1546, five 1590, ten 1449 (10 % more tiles on
  // the busiest pair), at 8192 four 1504, eight 1550.
  // GBNORM_GEMM_GROUP=r forces r (for sweeps; r must divide the column tiles).
  const int64_t slots = cluster ? pairs : sms;
  auto most = [&](int64_t r) {  // tiles of the busiest CTA (pair)
    const int64_t u = m_blocks * (n_tiles / r);
    return ((u + slots - 1) / slots) * r;
  };
  int rgrp = 1;
  for (int r : {8, 5, 4, 2})
    if (n_tiles % r == 0 && most(r) * 100 <= most(1) * 105) {
      rgrp = r;
      break;
    }
  if (const char *ov = std::getenv("GBNORM_GEMM_GROUP")) {
    const int r = std::atoi(ov);
    if (r >= 1 && n_tiles % r == 0) rgrp = r;
  }
  const int64_t units = m_blocks * (n_tiles / rgrp);
  if (cluster)
    cfg.gridDim = dim3(unsigned(2 * (units < pairs ? units : pairs)));
  else
    cfg.gridDim = dim3(unsigned(units < sms ? units : sms));
  int Mi = int(M), Ki = int(K), Ni = int(Nout);
  int gm = kGroupRows / (kBM * ctas);
  void *args[] = {&tm_x, &tm_w, &tm_o, &u,  &v,  &rstd, &mean,
                  &Mi,   &Ki,   &Ni,   &eps, &tx, &rgrp, &gm, &err};
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return NORM_ERR_CUDA;
  }
  return NORM_OK;
}

}  // extern "C"
