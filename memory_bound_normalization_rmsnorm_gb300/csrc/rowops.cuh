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
    if ((threadIdx.x & 31) == 0) {
      slot[(t >> 5) * 4 + 0] = m;
      slot[(t >> 5) * 4 + 1] = q;
    }
    named_bar_sync(1 + g, tpr);
    const float nw = 32.f * n_t;  // elements per warp
    m = slot[0];
    q = slot[1];
    for (int w = 1; w < W; ++w) {
      const float wb = 1.0f / static_cast<float>(w + 1);
      ms_merge(m, q, slot[w * 4 + 0], slot[w * 4 + 1], wb, nw * static_cast<float>(w) * wb);
    }
    rpar ^= 1;
  }
}

// Cross-CTA exchange state of a cluster kernel.  Buffer b (two of them,
// used alternately by successive rounds) holds [RT][C] float4 slots and has
// one mbarrier; `phase` bit b is the parity of buffer b's current round.
struct ClusterXch {
  float *slots;    // [2][RT][C][4]
  uint64_t *bars;  // [2]
  int RT;
  int C;
  int crank;
  int buf;
  uint32_t phase;
};

__device__ __forceinline__ ClusterXch make_xch(unsigned char *smem, const SmemLayout &L,
                                               int RT, int C, int crank) {
  ClusterXch x;
  x.slots = reinterpret_cast<float *>(smem + L.xch_off);
  x.bars = reinterpret_cast<uint64_t *>(smem + L.xch_off + static_cast<uint32_t>(2 * RT * C * 4) * 4u);
  x.RT = RT;
  x.C = C;
  x.crank = crank;
  x.buf = 0;
  x.phase = 0;
  return x;
}

// Cross-CTA reductions for row slot `r` of the tile, in CTA-rank order, so
// every CTA gets the same bits.  One round: thread 0 of the CTA posts the bytes the round expects (RT rows x C ranks
// x 16 bytes) on the local buffer mbarrier; thread t == 0 of every row
// group pushes its group total into slot [r][crank] of EVERY CTA of the
// cluster (itself included) with asynchronous stores that complete on the
// receiver's mbarrier; every thread then waits for the local mbarrier and
// folds the C slots of its row.  No cluster barrier and no memory fence:
// nothing orders the threads' global stores.  Every thread of the CTA must
// make the same sequence of calls.  Two buffers suffice: a CTA can only send
// round k+2 after receiving every CTA's round k+1, which each sends only
// after all of its groups finished reading round k.
//
// One exchange round: pushes (a, b, c) of row slot r to every CTA of the
// cluster and returns this CTA's local view of the row's C slots, in rank
// order, once all have arrived.
__device__ __forceinline__ const float *cluster_exchange(float a, float b, float c, int r,
                                                         int t, ClusterXch &x, unsigned *err,
                                                         volatile int *abort) {
  const int bsel = x.buf;
  float *base = x.slots + static_cast<size_t>(bsel) * x.RT * x.C * 4;
  uint64_t *bar = x.bars + bsel;
  if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(x.RT * x.C * 16));
  if (t == 0) {
    const float4 val = make_float4(a, b, c, 0.f);
    const float *mine = base + (static_cast<size_t>(r) * x.C + x.crank) * 4;
    for (int q = 0; q < x.C; ++q)
      st_async_f32x4(mapa_shared(mine, q), val, mapa_shared(bar, q));
  }
  mbar_wait(bar, (x.phase >> bsel) & 1u, err, abort);
  x.phase ^= 1u << bsel;
  x.buf ^= 1;
  return base + static_cast<size_t>(r) * x.C * 4;
}

// Sum of NV <= 3 values over the C CTAs, added in rank order.
template <int NV>
__device__ __forceinline__ void cluster_sum(float (&v)[NV], int r, int t, ClusterXch &x,
                                            unsigned *err, volatile int *abort) {
  const float *row = cluster_exchange(v[0], NV > 1 ? v[NV > 1 ? 1 : 0] : 0.f,
                                      NV > 2 ? v[NV > 2 ? 2 : 0] : 0.f, r, t, x, err, abort);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float acc = row[i];
    for (int q = 1; q < x.C; ++q) acc += row[q * 4 + i];
    v[i] = acc;
  }
}

// (mean, M2) over the C CTAs, each partial covering n_cta elements, merged
// in rank order.
__device__ __forceinline__ void cluster_meanvar(float &m, float &q, float n_cta, int r, int t,
                                                ClusterXch &x, unsigned *err,
                                                volatile int *abort) {
  const float *row = cluster_exchange(m, q, 0.f, r, t, x, err, abort);
  m = row[0];
  q = row[1];
  for (int k = 1; k < x.C; ++k) {
    const float wb = 1.0f / static_cast<float>(k + 1);
    ms_merge(m, q, row[k * 4 + 0], row[k * 4 + 1], wb, n_cta * static_cast<float>(k) * wb);
  }
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
