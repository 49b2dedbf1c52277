// Launch descriptors of the compiled sweep kernels (one per radius and kind).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "star_kernels.cuh"

namespace libstencil {

using LaunchFn = cudaError_t (*)(dim3 grid, cudaStream_t stream, const CUtensorMap& u,
                                 const CUtensorMap& uprev, const CUtensorMap& v2dt2,
                                 const CUtensorMap& eta, const StarParams& p);

struct KernelDesc {
  const void* fn;   // kernel entry (for attributes and occupancy)
  int threads;      // threads per CTA
  int smem;         // dynamic shared bytes
  int tile_y;       // output tile height (width is kTX)
  int stages;       // u ring slots
  int box_w, box_h; // u box (floats)
  LaunchFn launch;
};

template <int R, int TYT, int NWY, int STAGES, int ASTAGES, bool WAVE, int MINB, int KB = 1,
          bool PML = false, bool SEMI = false, bool DRIFT = false>
cudaError_t launch_star(dim3 grid, cudaStream_t stream, const CUtensorMap& u,
                        const CUtensorMap& uprev, const CUtensorMap& v2dt2, const CUtensorMap& eta,
                        const StarParams& p) {
  using C = StarCfg<R, TYT, NWY, STAGES, ASTAGES, WAVE, SEMI>;
  star_sweep_kernel<R, TYT, NWY, STAGES, ASTAGES, WAVE, MINB, KB, PML, SEMI, DRIFT>
      <<<grid, C::kThreads, C::kSmemBytes, stream>>>(u, uprev, v2dt2, eta, p);
  return cudaGetLastError();
}

template <int R, int TYT, int NWY, int STAGES, int ASTAGES, bool WAVE, int MINB, int KB = 1,
          bool PML = false, bool SEMI = false, bool DRIFT = false>
KernelDesc make_desc() {
  using C = StarCfg<R, TYT, NWY, STAGES, ASTAGES, WAVE, SEMI>;
  return KernelDesc{(const void*)star_sweep_kernel<R, TYT, NWY, STAGES, ASTAGES, WAVE, MINB, KB, PML, SEMI, DRIFT>,
                    C::kThreads,
                    C::kSmemBytes,
                    C::TY,
                    STAGES,
                    C::BW,
                    C::BH,
                    &launch_star<R, TYT, NWY, STAGES, ASTAGES, WAVE, MINB, KB, PML, SEMI, DRIFT>};
}

// Defined in kernels_apply.cu / kernels_wave.cu; radius in [1, 4].  `pml`: the wave step
// that reads eta only in a band along the faces (wave_step_pml).  `semi`: the sweep with
// the z stencil split into halves (stencil_apply_semi).
KernelDesc apply_kernel_desc(int radius);
KernelDesc semi_kernel_desc(int radius);
KernelDesc wave_kernel_desc(int radius, bool pml);

}  // namespace libstencil
