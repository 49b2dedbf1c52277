// Stencil-sweep kernel instantiations, radius 1..4.  Only the lead plane is read from
// shared memory, so the ring holds the landed plane plus the planes in flight.
//
// Radii 1-3: 64 x 32 tiles, 256 threads (4 x 2 outputs per thread); ring slots released
// warp by warp (DRIFT; at 512^3 2-6 % faster than a CTA barrier per plane).
//
// Radius 4: 128 threads per CTA, three CTAs per SM, output tiles stored by TMA; a thread
// owns 4 x TYT outputs, so each of its shared-memory loads of a row feeds more outputs
// (TYT = 4: 20 float4 loads per 16 outputs and plane, against 14 per 8 with TYT = 2) at
// 155-166 registers.  Two shapes, chosen by the size of an x-y plane (GB300, against the
// former 64 x 32 tile of 4 x 2 outputs on 256 threads, two CTAs per SM):
//  * planes below 2^20 points: 64 x 32 tiles of 4 x 4 per thread, a 4-slot ring, a CTA
//    barrier per plane: 512^3 0.186 against 0.201 ms, 384^3 -6 %, 640^3 -4 %,
//    768 x 768 x 384 -6 %, 1536 x 512 x 512 -8 %, 136 x 1000 x 200 -14 %;
//  * larger planes: 64 x 24 tiles of 4 x 3 per thread, a 5-slot ring, a barrier per two
//    planes: 1536 x 1536 x 256 0.834 against 0.887 ms, 2048 x 512 x 512 -9 %, 1024^3 -1 %,
//    1152 x 1152 x 256 -11 %.  (The first shape on these grids measured 11-24 % slower
//    than the old tile, whatever the z-chunk count or store staging depth: at
//    1536 x 1536 x 256 it read 3.56 GB from DRAM per sweep against 2.65 GB for this shape
//    and 2.42 GB compulsory, i.e. its boxes' halo rows no longer met in L2.)
#include "kernel_table.h"

namespace libstencil {

constexpr int64_t kWidePlanePoints = int64_t(1) << 20;

KernelDesc apply_kernel_desc(int radius, int64_t nx, int64_t ny) {
  switch (radius) {
    case 1: return make_desc<1, 2, 16, 5, 1, false, 1, 1, false, false, true>();
    case 2: return make_desc<2, 2, 16, 6, 1, false, 1, 1, false, false, true>();
    case 3: return make_desc<3, 2, 16, 7, 1, false, 1, 1, false, false, true>();
    default:
      if (nx * ny < kWidePlanePoints) return make_desc<4, 4, 8, 4, 1, false, 3, 1, false, false, false, 2>();
      return make_desc<4, 3, 8, 5, 1, false, 3, 2, false, false, false, 2>();
  }
}

// Two radius-1 sweeps per pass: 64 x 30 output tiles, a 5-slot ring, 4 rows per thread on
// 128 threads (165 registers, three CTAs per SM).  Against 2 rows per thread on 256
// threads (96 registers, two CTAs per SM), on GB300: 512^3 0.261 against 0.290 ms per
// pass, 1536 x 1536 x 256 1.122 against 1.275, 640^3 0.511 against 0.539; the same
// results bit for bit.  A 4-slot ring: the same; 6 slots drop to two CTAs per SM (-25 %).
KernelDesc apply2_kernel_desc(int radius) {
  if (radius == 1) return make_desc2<5, 2, 4>();
  KernelDesc none{};
  return none;
}

// Semi-stencil sweeps: the ring also keeps the R planes behind the lead (the left half of
// the z stencil is read from them), so it holds 2R + 1 slots or more.
KernelDesc semi_kernel_desc(int radius) {
  switch (radius) {
    case 1: return make_desc<1, 2, 16, 6, 1, false, 1, 1, false, true>();
    case 2: return make_desc<2, 2, 16, 7, 1, false, 1, 1, false, true>();
    case 3: return make_desc<3, 2, 16, 8, 1, false, 1, 1, false, true>();
    default: return make_desc<4, 2, 16, 9, 1, false, 2, 1, false, true>();
  }
}

// Direct-load sweeps (small grids).
const void* direct_kernel_fn(int radius) {
  switch (radius) {
    case 1: return (const void*)star_direct_kernel<1>;
    case 2: return (const void*)star_direct_kernel<2>;
    case 3: return (const void*)star_direct_kernel<3>;
    default: return (const void*)star_direct_kernel<4>;
  }
}

cudaError_t launch_direct(int radius, dim3 grid, cudaStream_t stream, const DirectParams& p) {
  switch (radius) {
    case 1: star_direct_kernel<1><<<grid, kDirectThreads, 0, stream>>>(p); break;
    case 2: star_direct_kernel<2><<<grid, kDirectThreads, 0, stream>>>(p); break;
    case 3: star_direct_kernel<3><<<grid, kDirectThreads, 0, stream>>>(p); break;
    default: star_direct_kernel<4><<<grid, kDirectThreads, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace libstencil
