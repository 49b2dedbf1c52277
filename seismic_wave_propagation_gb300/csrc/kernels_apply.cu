// Stencil-sweep kernel instantiations, radius 1..4.
// Tile 64 x 32 outputs, 256 threads (4 x 2 outputs per thread).  Only the lead plane is
// read from shared memory, so the ring is the landed plane plus R+3 in flight (radius 4:
// a 5-slot ring and one CTA barrier per 2 planes, 1-3 % faster than a barrier per plane on
// eight of nine grid shapes from 384^3 to 2048 x 512 x 512; 7 or 8 slots are slower).
// Radii 1-3 release ring slots warp by warp (DRIFT; at 512^3 2-6 % faster than a CTA
// barrier per plane), radius 4 keeps the barrier (1-2 % faster there).
#include "kernel_table.h"

namespace libstencil {

KernelDesc apply_kernel_desc(int radius) {
  switch (radius) {
    case 1: return make_desc<1, 2, 16, 5, 1, false, 1, 1, false, false, true>();
    case 2: return make_desc<2, 2, 16, 6, 1, false, 1, 1, false, false, true>();
    case 3: return make_desc<3, 2, 16, 7, 1, false, 1, 1, false, false, true>();
    default: return make_desc<4, 2, 16, 5, 1, false, 2, 2, false, false, false, true>();
  }
}

// Two radius-1 sweeps per pass: 64 x 30 output tiles, 256 threads, a 5-slot ring.
KernelDesc apply2_kernel_desc(int radius) {
  if (radius == 1) return make_desc2<5, 2>();
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
