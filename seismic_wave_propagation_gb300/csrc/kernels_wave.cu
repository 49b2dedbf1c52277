// Fused wave-step kernel instantiations, radius 1..4.
// Tile 64 x 16 outputs, 128 threads (4 x 2 outputs per thread), ring of R+4 u planes and
// three stages of (u_prev, v2dt2, eta) tiles.
#include "kernel_table.h"

namespace libstencil {

KernelDesc wave_kernel_desc(int radius) {
  switch (radius) {
    case 1: return make_desc<1, 2, 8, 5, 3, true, 1>();
    case 2: return make_desc<2, 2, 8, 6, 3, true, 1>();
    case 3: return make_desc<3, 2, 8, 7, 3, true, 1>();
    default: return make_desc<4, 2, 8, 8, 3, true, 1>();
  }
}

}  // namespace libstencil
