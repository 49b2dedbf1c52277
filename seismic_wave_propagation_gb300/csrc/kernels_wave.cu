// Fused wave-step kernel instantiations, radius 1..4: tile 64 x 16 outputs on 128 threads
// (4 x 2 outputs per thread, so each shared-memory row load feeds two outputs), a ring of
// R + 3 u planes (R kept behind the lead for u at the output plane, two in flight; R + 2
// for radius 4, which then fits three CTAs per SM) and two stages of (u_prev, v2dt2, eta)
// tiles.  Against 4 x 1 outputs on 256 threads at two CTAs per SM with R + 4 u slots and 3-4
// aux stages, on GB300: radius 4 640^3 0.775 against 0.803 ms, 512^3 -7 %, 384^3 -8 %;
// radius 1, 2, 3 at 512^3 -7 %, -9 %, -7 %.  The no-eta kernel of the inner region
// likewise (radius 4: 640^3 with no band 0.654 against 0.755 ms, the 1024^3 step with a
// 16-point band 2.87 against 3.18 ms).  Radius 4 with 7 u slots: the same; 9 z-chunks at
// 640^3 (the planner's choice) the fastest of 2-12.
#include "kernel_table.h"

namespace libstencil {

KernelDesc wave_kernel_desc(int radius, bool noeta) {
  if (noeta) {
    switch (radius) {
      case 1: return make_desc<1, 2, 8, 4, 2, true, 3, 1, true>();
      case 2: return make_desc<2, 2, 8, 5, 2, true, 3, 1, true>();
      case 3: return make_desc<3, 2, 8, 6, 2, true, 3, 1, true>();
      default: return make_desc<4, 2, 8, 6, 2, true, 3, 1, true>();
    }
  }
  switch (radius) {
    case 1: return make_desc<1, 2, 8, 4, 2, true, 3>();
    case 2: return make_desc<2, 2, 8, 5, 2, true, 3>();
    case 3: return make_desc<3, 2, 8, 6, 2, true, 3>();
    default: return make_desc<4, 2, 8, 6, 2, true, 3>();
  }
}

}  // namespace libstencil
