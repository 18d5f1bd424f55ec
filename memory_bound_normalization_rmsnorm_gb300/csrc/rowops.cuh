// rowops.cuh -- per-row building blocks shared by the forward and backward
// kernels: bf16 <-> packed fp32 pairs, packed-FP32 arithmetic, fixed-order
// (hence bitwise reproducible) sums within a row group, across the warps of
// a group and across the CTAs of a cluster, and the shared-memory ring
// refill hand-off.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gbn {

// ------------------------------------------------------- bf16 <-> fp32
// Two bf16 packed in a 32-bit word -> the two exact fp32 values (the
// element at the lower address is .x).
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// Round two fp32 to bf16 (nearest even) and pack, .x at the lower address.
__device__ __forceinline__ uint32_t f2_to_bf2(float2 v) {
  __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ void chunk_to_f2(const uint4 &c, float2 (&v)[4]) {
  v[0] = bf2_to_f2(c.x);
  v[1] = bf2_to_f2(c.y);
  v[2] = bf2_to_f2(c.z);
  v[3] = bf2_to_f2(c.w);
}
__device__ __forceinline__ uint4 f2_to_chunk(const float2 (&v)[4]) {
  return make_uint4(f2_to_bf2(v[0]), f2_to_bf2(v[1]), f2_to_bf2(v[2]), f2_to_bf2(v[3]));
}

// ------------------------------------------ packed FP32 (two lanes per op)
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  return __ffma2_rn(a, b, c);
}
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// ------------------------------------------------------- group sums
// Sum of NV values over the `tpr` threads of a row group, returned to every
// thread of the group.  Butterfly within the warp (IEEE addition commutes,
// so both partners of an exchange get the same bits), then for tpr > 32 the
// per-warp totals are added in warp order from shared memory behind a named
// barrier of the group's warps.  `red` is the CTA's [2][G][W][4] scratch and
// `rpar` the buffer parity (flipped on return).  All threads of a group must
// make the same calls.
// WIDE: the caller guarantees tpr >= 32 (all five butterfly levels).
template <int NV, bool WIDE>
__device__ __forceinline__ void group_sum(float (&v)[NV], int tpr, int g, int G, int t,
                                          float *red, int &rpar) {
  const int width = WIDE ? 32 : (tpr < 32 ? tpr : 32);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (WIDE || o < width) {
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    }
  }
  if (tpr > 32) {
    const int W = tpr >> 5;
    float *slot = red + (static_cast<size_t>(rpar * G + g) * W) * 4;
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
      for (int i = 0; i < NV; ++i) slot[(t >> 5) * 4 + i] = v[i];
    }
    named_bar_sync(1 + g, tpr);
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = slot[i];
#pragma unroll 4
    for (int w = 1; w < W; ++w) {
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] += slot[w * 4 + i];
    }
    rpar ^= 1;
  }
}

// Maximum of one non-negative value over the row group (same structure
// and calling rule as group_sum).  max is exact, so the order is free.
template <bool WIDE>
__device__ __forceinline__ float group_max(float v, int tpr, int g, int G, int t, float *red,
                                           int &rpar) {
  const int width = WIDE ? 32 : (tpr < 32 ? tpr : 32);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    if (WIDE || o < width) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (tpr > 32) {
    const int W = tpr >> 5;
    float *slot = red + (static_cast<size_t>(rpar * G + g) * W) * 4;
    if ((threadIdx.x & 31) == 0) slot[(t >> 5) * 4] = v;
    named_bar_sync(1 + g, tpr);
    v = slot[0];
#pragma unroll 4
    for (int w = 1; w < W; ++w) v = fmaxf(v, slot[w * 4]);
    rpar ^= 1;
  }
  return v;
}

// ------------------------------------------- (mean, M2) of equal counts
// Parallel variance merge of two partials that cover the same number of
// elements n_each: mean = (ma + mb) / 2, M2 = M2a + M2b + (mb - ma)^2 *
// n_each / 2.  Symmetric in its operands (both exchange partners compute the
// same bits: negation and IEEE addition commute exactly).
__device__ __forceinline__ void ms_merge_equal(float &m, float &q, float mo, float qo,
                                               float half_n_each) {
  const float d = mo - m;
  q = (q + qo) + d * d * half_n_each;
  m = 0.5f * (m + mo);
}
// Merge of a partial over n_a elements with one over n_b elements, given
// wb = n_b / (n_a + n_b) and the product n_a * n_b / (n_a + n_b).
__device__ __forceinline__ void ms_merge(float &m, float &q, float mo, float qo, float wb,
                                         float nab) {
  const float d = mo - m;
  q = (q + qo) + d * d * nab;
  m = fmaf(d, wb, m);
}

// Pairwise tree over W (mean, M2) partials of nw elements each, stored as
// float2 at stride 4 floats: ((0,1),(2,3)),... in a fixed order.
template <int W>
__device__ __forceinline__ void tree_fold(const float *slot, float nw, float &m, float &q) {
  float2 v[W];
#pragma unroll
  for (int w = 0; w < W; ++w) v[w] = *reinterpret_cast<const float2 *>(slot + w * 4);
  float h = 0.5f * nw;
#pragma unroll
  for (int span = 1; span < W; span <<= 1) {
#pragma unroll
    for (int w = 0; w + span < W; w += 2 * span)
      ms_merge_equal(v[w].x, v[w].y, v[w + span].x, v[w + span].y, h);
    h *= 2.f;
  }
  m = v[0].x;
  q = v[0].y;
}

// (mean, M2) over the tpr >= 32 threads of a row group, every thread
// holding a partial over n_t elements.  Butterfly of equal-count merges,
// then for tpr > 32 a fold of the per-warp partials in warp order (warp w's
// running partial covers w warps, the next one warp).
__device__ __forceinline__ void group_meanvar(float &m, float &q, float n_t, int tpr, int g,
                                              int G, int t, float *red, int &rpar) {
  float h = 0.5f * n_t;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, o);
    const float qo = __shfl_xor_sync(0xffffffffu, q, o);
    ms_merge_equal(m, q, mo, qo, h);
    h *= 2.f;
  }
  if (tpr > 32) {
    const int W = tpr >> 5;
    float *slot = red + (static_cast<size_t>(rpar * G + g) * W) * 4;
    if ((threadIdx.x & 31) == 0)
      *reinterpret_cast<float2 *>(slot + (t >> 5) * 4) = make_float2(m, q);
    named_bar_sync(1 + g, tpr);
    const float nw = 32.f * n_t;  // elements per warp
    if (W == 2 || W == 4 || W == 8 || W == 16) {
      // Power-of-two warp count: pairwise tree of equal-count merges in a
      // fixed order, no division.
      switch (W) {
        case 2: tree_fold<2>(slot, nw, m, q); break;
        case 4: tree_fold<4>(slot, nw, m, q); break;
        case 8: tree_fold<8>(slot, nw, m, q); break;
        default: tree_fold<16>(slot, nw, m, q); break;
      }
    } else {
      // Running partial over w warps merged with warp w, in warp order
      // (unrolled, so 1 / (w + 1) is a compile-time constant).
      float2 f = *reinterpret_cast<const float2 *>(slot);
      m = f.x;
      q = f.y;
#pragma unroll
      for (int w = 1; w < 16; ++w) {
        if (w < W) {
          f = *reinterpret_cast<const float2 *>(slot + w * 4);
          const float wb = 1.0f / static_cast<float>(w + 1);
          ms_merge(m, q, f.x, f.y, wb, nw * static_cast<float>(w) * wb);
        }
      }
    }
    rpar ^= 1;
  }
}

// Cross-CTA exchange state of a cluster kernel.  kXchBuffers buffers, used by
// successive rounds in turn, each holding [RT][C] float4 slots and one
// mbarrier; bit b of `phase` is the parity of buffer b's current round.
struct ClusterXch {
  float *slots;    // [kXchBuffers][RT][C][4]
  uint64_t *bars;  // [kXchBuffers]
  int RT;
  int C;
  int crank;
  int push_buf;    // buffer of the next round to push
  int wait_buf;    // buffer of the oldest round not yet consumed
  uint32_t phase;
};

__device__ __forceinline__ uint64_t *xch_bars(unsigned char *smem, const SmemLayout &L, int RT,
                                              int C) {
  return reinterpret_cast<uint64_t *>(smem + L.xch_off +
                                      static_cast<uint32_t>(kXchBuffers * RT * C * 4) * 4u);
}

__device__ __forceinline__ ClusterXch make_xch(unsigned char *smem, const SmemLayout &L,
                                               int RT, int C, int crank) {
  ClusterXch x;
  x.slots = reinterpret_cast<float *>(smem + L.xch_off);
  x.bars = xch_bars(smem, L, RT, C);
  x.RT = RT;
  x.C = C;
  x.crank = crank;
  x.push_buf = 0;
  x.wait_buf = 0;
  x.phase = 0;
  return x;
}

// Cross-CTA reductions for row slot `r` of the tile, in CTA-rank order, so
// every CTA gets the same bits.  A round: thread 0 of the CTA posts the bytes
// the round expects (RT rows x C ranks x 16 bytes) on the round's local
// mbarrier; thread t == 0 of every row group pushes its group partial into
// slot [r][crank] of EVERY CTA of the cluster (itself included) with
// asynchronous stores that complete on the receiver's mbarrier; every thread
// later waits on the local mbarrier and folds the C slots of its row.  No
// cluster barrier and no memory fence: nothing orders the threads' global
// stores.  Every thread of the CTA makes the same sequence of push and wait
// calls, and a CTA pushes round k+1 at the earliest before it waits for
// round k.  Then four buffers suffice: a CTA pushes round k+1 only after its
// wait for round k-1 has seen every CTA's round k-1 push, and each CTA folds
// round k-3 (same buffer as k+1) before it pushes round k-1.
__device__ __forceinline__ void cluster_push(float a, float b, float c, int r, int t,
                                             ClusterXch &x, float d = 0.f) {
  const int bsel = x.push_buf;
  float *base = x.slots + static_cast<size_t>(bsel) * x.RT * x.C * 4;
  uint64_t *bar = x.bars + bsel;
  if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(x.RT * x.C * 16));
  if (t == 0) {
    const float4 val = make_float4(a, b, c, d);
    const float *mine = base + (static_cast<size_t>(r) * x.C + x.crank) * 4;
    for (int q = 0; q < x.C; ++q)
      st_async_f32x4(mapa_shared(mine, q), val, mapa_shared(bar, q));
  }
  x.push_buf = (bsel + 1) % kXchBuffers;
}

// Waits for the oldest pushed round; returns this CTA's view of row r's C
// slots (rank order).
__device__ __forceinline__ const float *cluster_wait_row(int r, ClusterXch &x, unsigned *err,
                                                         volatile int *abort) {
  const int bsel = x.wait_buf;
  mbar_wait(x.bars + bsel, (x.phase >> bsel) & 1u, err, abort);
  x.phase ^= 1u << bsel;
  x.wait_buf = (bsel + 1) % kXchBuffers;
  return x.slots + (static_cast<size_t>(bsel) * x.RT + r) * x.C * 4;
}

__device__ __forceinline__ const float *cluster_exchange(float a, float b, float c, int r,
                                                         int t, ClusterXch &x, unsigned *err,
                                                         volatile int *abort) {
  cluster_push(a, b, c, r, t, x);
  return cluster_wait_row(r, x, err, abort);
}

// Rank-order sums of the first NV floats of the C slots of a row.
template <int NV>
__device__ __forceinline__ void fold_sum(const float *row, int C, float (&v)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float acc = row[i];
    for (int q = 1; q < C; ++q) acc += row[q * 4 + i];
    v[i] = acc;
  }
}

// Sum of NV <= 3 values over the C CTAs, added in rank order.
template <int NV>
__device__ __forceinline__ void cluster_sum(float (&v)[NV], int r, int t, ClusterXch &x,
                                            unsigned *err, volatile int *abort) {
  const float *row = cluster_exchange(v[0], NV > 1 ? v[NV > 1 ? 1 : 0] : 0.f,
                                      NV > 2 ? v[NV > 2 ? 2 : 0] : 0.f, r, t, x, err, abort);
  fold_sum<NV>(row, x.C, v);
}

// (mean, M2) of C <= 16 partials of n_cta elements each (row[4k], row[4k+1]),
// the running partial over k CTAs merged with CTA k in rank order.  Unrolled,
// so every 1 / (k + 1) is a compile-time constant, not a division per row.
__device__ __forceinline__ void rank_fold_meanvar(const float *row, int C, float n_cta, float &m,
                                                  float &q) {
  m = row[0];
  q = row[1];
#pragma unroll
  for (int k = 1; k < 16; ++k) {
    if (k < C) {
      const float wb = 1.0f / static_cast<float>(k + 1);
      ms_merge(m, q, row[k * 4 + 0], row[k * 4 + 1], wb, n_cta * static_cast<float>(k) * wb);
    }
  }
}

// (mean, M2) over the C CTAs, each partial covering n_cta elements, merged
// in rank order.
__device__ __forceinline__ void cluster_meanvar(float &m, float &q, float n_cta, int r, int t,
                                                ClusterXch &x, unsigned *err,
                                                volatile int *abort) {
  const float *row = cluster_exchange(m, q, 0.f, r, t, x, err, abort);
  rank_fold_meanvar(row, x.C, n_cta, m, q);
}

// ------------------------------------ (count, mean, M2) of any counts
// Chan's pairwise merge of (n, mean, M2) partials; `lo` is the partial of
// the lower-indexed participant so that both partners of a butterfly
// exchange compute the same bits.  Empty partials (n = 0) are neutral.
__device__ __forceinline__ void nms_merge(float &n, float &m, float &q, float n2, float m2,
                                          float q2) {
  if (n2 == 0.f) return;
  if (n == 0.f) {
    n = n2;
    m = m2;
    q = q2;
    return;
  }
  const float nt = n + n2;
  const float wb = n2 / nt;
  const float d = m2 - m;
  q = (q + q2) + d * d * (n * wb);
  m = fmaf(d, wb, m);
  n = nt;
}

// (n, mean, M2) over the tpr threads of a row group (any tpr, any counts).
__device__ __forceinline__ void group_nmeanvar(float &n, float &m, float &q, int tpr, int g,
                                               int G, int t, float *red, int &rpar) {
  const int lane = threadIdx.x & 31;
  const int width = tpr < 32 ? tpr : 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (o < width) {
      const float no = __shfl_xor_sync(0xffffffffu, n, o);
      const float mo = __shfl_xor_sync(0xffffffffu, m, o);
      const float qo = __shfl_xor_sync(0xffffffffu, q, o);
      if (lane & o) {  // the partner is the lower participant
        float n0 = no, m0 = mo, q0 = qo;
        nms_merge(n0, m0, q0, n, m, q);
        n = n0;
        m = m0;
        q = q0;
      } else {
        nms_merge(n, m, q, no, mo, qo);
      }
    }
  }
  if (tpr > 32) {
    const int W = tpr >> 5;
    float *slot = red + (static_cast<size_t>(rpar * G + g) * W) * 4;
    if (lane == 0) {
      slot[(t >> 5) * 4 + 0] = n;
      slot[(t >> 5) * 4 + 1] = m;
      slot[(t >> 5) * 4 + 2] = q;
    }
    named_bar_sync(1 + g, tpr);
    n = slot[0];
    m = slot[1];
    q = slot[2];
    for (int w = 1; w < W; ++w) nms_merge(n, m, q, slot[w * 4 + 0], slot[w * 4 + 1], slot[w * 4 + 2]);
    rpar ^= 1;
  }
}

// Rank-order (n, mean, M2) merge of a row's C slots.
__device__ __forceinline__ void fold_nmeanvar(const float *row, int C, float &n, float &m,
                                              float &q) {
  m = row[0];
  q = row[1];
  n = row[2];
  for (int k = 1; k < C; ++k) nms_merge(n, m, q, row[k * 4 + 2], row[k * 4 + 0], row[k * 4 + 1]);
}

// ---------------------------------------------------- ring hand-off
// Called by every warp of the CTA once it has finished reading stage `s`
// (all of its loads from the stage have completed: their values were used).
// Returns true in exactly one warp per use of the stage -- the last to
// finish -- which then refills the stage.  No warp waits for another.
__device__ __forceinline__ bool last_warp_done(int *cnt, int s, int nwarps) {
  __syncwarp();
  int last = 0;
  if ((threadIdx.x & 31) == 0) {
    __threadfence_block();
    const int old = atomicAdd(cnt + s, 1);
    last = (old == nwarps - 1);
    if (last) {
      cnt[s] = 0;
      __threadfence_block();
    }
  }
  return __shfl_sync(0xffffffffu, last, 0) != 0;
}

}  // namespace gbn
