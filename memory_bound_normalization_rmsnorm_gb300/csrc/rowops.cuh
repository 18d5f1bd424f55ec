// rowops.cuh -- per-row building blocks shared by the forward and backward
// kernels: bf16 packing, and fixed-order (hence bitwise reproducible)
// reductions within a row group, across the warps of a group and across
// the CTAs of a cluster.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gbn {

// --------------------------------------------------------------- bf16
__device__ __forceinline__ float bf_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf_hi(uint32_t w) {
  return __uint_as_float(w & 0xffff0000u);
}
// Element e (0..7) of a 16-byte chunk of 8 bf16.
__device__ __forceinline__ float bf_elem(const uint4 &v, int e) {
  const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
  return (e & 1) ? bf_hi(w) : bf_lo(w);
}
// Round two floats to bf16 (nearest even) and pack: `lo` is the element at
// the lower address.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// --------------------------------------------------------- partials
// A reduction payload of up to 3 floats, combined either by summation or
// by Chan's pairwise merge of (count, mean, sum of squared deviations).
struct Part {
  float a, b, c;
};

__device__ __forceinline__ Part part_sum(const Part &lo, const Part &hi) {
  return Part{lo.a + hi.a, lo.b + hi.b, lo.c + hi.c};
}

// (n, mean, M2) merge.  `lo` is always the partial of the lower-indexed
// participant, so every participant computes bit-identical results.
__device__ __forceinline__ Part part_chan(const Part &lo, const Part &hi) {
  if (hi.a == 0.f) return lo;
  if (lo.a == 0.f) return hi;
  const float n = lo.a + hi.a;
  const float d = hi.b - lo.b;
  const float wh = hi.a / n;
  Part r;
  r.a = n;
  r.b = fmaf(d, wh, lo.b);
  r.c = lo.c + hi.c + d * d * lo.a * wh;
  return r;
}

template <bool CHAN>
__device__ __forceinline__ Part part_op(const Part &lo, const Part &hi) {
  return CHAN ? part_chan(lo, hi) : part_sum(lo, hi);
}

__device__ __forceinline__ Part shfl_xor_part(const Part &p, int o) {
  return Part{__shfl_xor_sync(0xffffffffu, p.a, o),
              __shfl_xor_sync(0xffffffffu, p.b, o),
              __shfl_xor_sync(0xffffffffu, p.c, o)};
}
__device__ __forceinline__ Part shfl_part(const Part &p, int src) {
  return Part{__shfl_sync(0xffffffffu, p.a, src),
              __shfl_sync(0xffffffffu, p.b, src),
              __shfl_sync(0xffffffffu, p.c, src)};
}

// All-reduce over the `tpr` threads of a row group.  Butterfly within the
// warp (lanes of one group when tpr <= 32), then, for tpr > 32, a fold of
// the per-warp results in warp order through shared memory behind a named
// barrier.  `red` is this CTA's [2][G][W][4] scratch, `rpar` the parity of
// the buffer to use (flipped on return).  Every thread of the CTA must call
// this the same number of times.
template <bool CHAN>
__device__ __forceinline__ Part group_allreduce(Part v, int tpr, int g, int G,
                                                int t, float *red, int &rpar) {
  const int lane = threadIdx.x & 31;
  const int width = tpr < 32 ? tpr : 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (o < width) {
      const Part other = shfl_xor_part(v, o);
      v = ((lane & o) == 0) ? part_op<CHAN>(v, other) : part_op<CHAN>(other, v);
    }
  }
  if (tpr > 32) {
    const int W = tpr >> 5;
    float *slot = red + (static_cast<size_t>(rpar * G + g) * W) * 4;
    if (lane == 0) {
      const int w = t >> 5;
      *reinterpret_cast<float4 *>(slot + w * 4) = make_float4(v.a, v.b, v.c, 0.f);
    }
    named_bar_sync(1 + g, tpr);
    float4 f = *reinterpret_cast<const float4 *>(slot);
    v = Part{f.x, f.y, f.z};
    for (int w = 1; w < W; ++w) {
      f = *reinterpret_cast<const float4 *>(slot + w * 4);
      v = part_op<CHAN>(v, Part{f.x, f.y, f.z});
    }
    rpar ^= 1;
  }
  return v;
}

// Combines the group partials of the C CTAs of a cluster for row slot `r`
// of the tile, in CTA-rank order, so every CTA gets the same bits.  Also a
// cluster-wide barrier: on return every thread of every CTA in the cluster
// has passed the point of its call.  `xch` is this CTA's [2][RT][4] scratch.
template <bool CHAN>
__device__ __forceinline__ Part cluster_allreduce(Part v, int r, int RT, int t,
                                                  float *xch, int &xpar) {
  float *slot = xch + (static_cast<size_t>(xpar) * RT + r) * 4;
  if (t == 0) *reinterpret_cast<float4 *>(slot) = make_float4(v.a, v.b, v.c, 0.f);
  cluster_arrive_release();
  cluster_wait_acquire();
  const int C = static_cast<int>(cluster_nctarank());
  const int lane = threadIdx.x & 31;
  float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane < C) f = ld_dsmem_f32x4(slot, static_cast<uint32_t>(lane));
  const Part mine{f.x, f.y, f.z};
  Part acc = shfl_part(mine, 0);
  for (int q = 1; q < C; ++q) acc = part_op<CHAN>(acc, shfl_part(mine, q));
  xpar ^= 1;
  return acc;
}

}  // namespace gbn
