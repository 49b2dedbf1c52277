// Direct-load star sweep for small grids.
//
// The staged kernel (star_kernels.cuh) pays, per launch, for its ring set-up, descriptor
// fetch and the R + 1 planes each z-chunk loads before its first output; on a grid of a
// few million points, which L2 holds whole, that latency is most of the sweep.  This
// kernel has none of it: one thread computes four consecutive x points of one interior
// row, reading every operand straight from global memory with 128-bit loads (the centre
// float4, its left and right neighbours for the x terms, and one float4 per y and z
// neighbour), and stores the four results.  No shared memory, no barrier, no wait.
//
// Same operation as the staged sweep (the plain star-stencil definition of "Accelerating
// High-Order Stencils on GPUs", the problem statement, and the 7-point update of the PMPP
// stencil chapter): out = c0 u + sum_r c_r (six neighbours at distance r), on the points
// at least R from every face; the shell is never written.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace libstencil {

struct DirectParams {
  const float* in;
  float* out;
  int nx, ny;        // row length (a multiple of 4) and rows per plane
  int z0;            // first output plane
  int q0, nq;        // first float4 column holding an interior point; columns per row
  int nyi;           // interior rows per plane, ny - 2R
  int64_t total;     // threads with work: nq * nyi * output planes
  float c[5];        // c[0] centre, c[r] per neighbour at distance r
};

template <int R>
__global__ void __launch_bounds__(256) star_direct_kernel(const DirectParams p) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= p.total) return;
  const int q = p.q0 + (int)(t % p.nq);
  const int64_t row = t / p.nq;
  const int y = R + (int)(row % p.nyi);
  const int z = p.z0 + (int)(row / p.nyi);
  const int64_t sy = p.nx;
  const int64_t sz = (int64_t)p.nx * p.ny;
  const int64_t base = (int64_t)z * sz + (int64_t)y * sy + 4 * (int64_t)q;
  const int x0 = 4 * q;

  // x neighbours: a column's interior points reach at most R <= 4 points to each side, so
  // the float4 columns left and right of it cover them (read only where they exist; an
  // interior point never needs the missing side).
  const float4 cen = __ldg(reinterpret_cast<const float4*>(p.in + base));
  float4 lft = make_float4(0.f, 0.f, 0.f, 0.f), rgt = lft;
  if (q > 0) lft = __ldg(reinterpret_cast<const float4*>(p.in + base - 4));
  if (x0 + 4 < p.nx) rgt = __ldg(reinterpret_cast<const float4*>(p.in + base + 4));
  const float v[12] = {lft.x, lft.y, lft.z, lft.w, cen.x, cen.y, cen.z, cen.w,
                       rgt.x, rgt.y, rgt.z, rgt.w};

  float acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = p.c[0] * v[4 + i];
#pragma unroll
  for (int r = 1; r <= R; ++r) {
    const float4 ym = __ldg(reinterpret_cast<const float4*>(p.in + base - r * sy));
    const float4 yp = __ldg(reinterpret_cast<const float4*>(p.in + base + r * sy));
    const float4 zm = __ldg(reinterpret_cast<const float4*>(p.in + base - r * sz));
    const float4 zp = __ldg(reinterpret_cast<const float4*>(p.in + base + r * sz));
    const float cr = p.c[r];
    acc[0] = fmaf(cr, (v[4 - r] + v[4 + r]) + (ym.x + yp.x) + (zm.x + zp.x), acc[0]);
    acc[1] = fmaf(cr, (v[5 - r] + v[5 + r]) + (ym.y + yp.y) + (zm.y + zp.y), acc[1]);
    acc[2] = fmaf(cr, (v[6 - r] + v[6 + r]) + (ym.z + yp.z) + (zm.z + zp.z), acc[2]);
    acc[3] = fmaf(cr, (v[7 - r] + v[7 + r]) + (ym.w + yp.w) + (zm.w + zp.w), acc[3]);
  }

  float* o = p.out + base;
  if (x0 >= R && x0 + 3 < p.nx - R) {
    *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  } else {  // a column at an x face: only its interior points
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (x0 + i >= R && x0 + i < p.nx - R) o[i] = acc[i];
  }
}

}  // namespace libstencil
