// Fused wave-step kernel instantiations, radius 1..4.
// Radii 1-3: tile 64 x 16 outputs, 256 threads (4 x 1 outputs per thread), two CTAs per
// SM; a ring of R+4 u planes (R kept behind the lead for u at the output plane, three in
// flight) and three stages of (u_prev, v2dt2, eta) tiles.
// Radius 4: tile 64 x 16 outputs on 128 threads (4 x 2 outputs per thread, so each
// shared-memory row load feeds two outputs), three CTAs per SM, a ring of 6 u planes
// (R kept, one in flight) and two aux stages, which is what fits three CTAs: on GB300
// 640^3 0.775 against 0.803 ms for 4 x 1 outputs on 256 threads at two CTAs per SM with
// 8 u slots and 4 aux stages, 512^3 -7 %, 384^3 -8 %; the no-eta kernel of the inner
// region likewise (640^3 with no band 0.654 against 0.755 ms, the 1024^3 step with a
// 16-point band 2.87 against 3.18 ms).  7 u slots: the same; 9 z-chunks at 640^3 (the
// planner's choice) the fastest of 2-12.
#include "kernel_table.h"

namespace libstencil {

KernelDesc wave_kernel_desc(int radius, bool noeta) {
  if (noeta) {
    switch (radius) {
      case 1: return make_desc<1, 1, 16, 5, 3, true, 2, 1, true>();
      case 2: return make_desc<2, 1, 16, 6, 3, true, 2, 1, true>();
      case 3: return make_desc<3, 1, 16, 7, 3, true, 2, 1, true>();
      default: return make_desc<4, 2, 8, 6, 2, true, 3, 1, true>();
    }
  }
  switch (radius) {
    case 1: return make_desc<1, 1, 16, 5, 3, true, 2>();
    case 2: return make_desc<2, 1, 16, 6, 3, true, 2>();
    case 3: return make_desc<3, 1, 16, 7, 3, true, 2>();
    default: return make_desc<4, 2, 8, 6, 2, true, 3>();
  }
}

}  // namespace libstencil
