// Fused wave-step kernel instantiations, radius 1..4.
// Tile 64 x 16 outputs, 256 threads (4 x 1 outputs per thread), two CTAs per SM; a ring
// of R+4 u planes (R kept behind the lead for u at the output plane, three in flight)
// and three stages of (u_prev, v2dt2, eta) tiles (four for R = 4: 1 % faster at 640^3;
// two stages are 9 % slower).
#include "kernel_table.h"

namespace libstencil {

KernelDesc wave_kernel_desc(int radius, bool noeta) {
  if (noeta) {
    switch (radius) {
      case 1: return make_desc<1, 1, 16, 5, 3, true, 2, 1, true>();
      case 2: return make_desc<2, 1, 16, 6, 3, true, 2, 1, true>();
      case 3: return make_desc<3, 1, 16, 7, 3, true, 2, 1, true>();
      default: return make_desc<4, 1, 16, 8, 4, true, 2, 1, true>();
    }
  }
  switch (radius) {
    case 1: return make_desc<1, 1, 16, 5, 3, true, 2>();
    case 2: return make_desc<2, 1, 16, 6, 3, true, 2>();
    case 3: return make_desc<3, 1, 16, 7, 3, true, 2>();
    default: return make_desc<4, 1, 16, 8, 4, true, 2>();
  }
}

}  // namespace libstencil
