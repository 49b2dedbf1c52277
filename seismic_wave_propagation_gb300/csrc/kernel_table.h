// Launch descriptors of the compiled sweep kernels (one per radius and kind).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "direct_kernels.cuh"
#include "star2_kernels.cuh"
#include "star_kernels.cuh"

namespace libstencil {

using LaunchFn = cudaError_t (*)(dim3 grid, cudaStream_t stream, const CUtensorMap& u,
                                 const CUtensorMap& uprev, const CUtensorMap& v2dt2,
                                 const CUtensorMap& eta, const CUtensorMap& out, const StarParams& p);

struct KernelDesc {
  const void* fn;   // kernel entry (for attributes and occupancy)
  int threads;      // threads per CTA
  int smem;         // dynamic shared bytes
  int tile_y;       // output tile height (width is kTX)
  int stages;       // u ring slots
  int box_w, box_h; // u box (floats)
  bool tstore;      // output stored by TMA through a map of the interior (tiles start at x = R)
  LaunchFn launch;
};

template <int R, int TYT, int NWY, int STAGES, int ASTAGES, bool WAVE, int MINB, int KB = 1,
          bool NOETA = false, bool SEMI = false, bool DRIFT = false, int TSTORE = 0>
cudaError_t launch_star(dim3 grid, cudaStream_t stream, const CUtensorMap& u,
                        const CUtensorMap& uprev, const CUtensorMap& v2dt2, const CUtensorMap& eta,
                        const CUtensorMap& out, const StarParams& p) {
  using C = StarCfg<R, TYT, NWY, STAGES, ASTAGES, WAVE, SEMI, TSTORE, KB>;
  star_sweep_kernel<R, TYT, NWY, STAGES, ASTAGES, WAVE, MINB, KB, NOETA, SEMI, DRIFT, TSTORE>
      <<<grid, C::kThreads, C::kSmemBytes, stream>>>(u, uprev, v2dt2, eta, out, p);
  return cudaGetLastError();
}

template <int R, int TYT, int NWY, int STAGES, int ASTAGES, bool WAVE, int MINB, int KB = 1,
          bool NOETA = false, bool SEMI = false, bool DRIFT = false, int TSTORE = 0>
KernelDesc make_desc() {
  using C = StarCfg<R, TYT, NWY, STAGES, ASTAGES, WAVE, SEMI, TSTORE, KB>;
  return KernelDesc{
      (const void*)star_sweep_kernel<R, TYT, NWY, STAGES, ASTAGES, WAVE, MINB, KB, NOETA, SEMI, DRIFT, TSTORE>,
      C::kThreads,
      C::kSmemBytes,
      C::TY,
      STAGES,
      C::BW,
      C::BH,
      TSTORE != 0,
      &launch_star<R, TYT, NWY, STAGES, ASTAGES, WAVE, MINB, KB, NOETA, SEMI, DRIFT, TSTORE>};
}

// Two radius-1 sweeps in one pass (star2_kernels.cuh).
template <int STAGES, int MINB, int NR>
cudaError_t launch_star2(dim3 grid, cudaStream_t stream, const CUtensorMap& u, const CUtensorMap& uprev,
                         const CUtensorMap& v2dt2, const CUtensorMap& eta, const CUtensorMap& out,
                         const StarParams& p) {
  using C = Star2Cfg<STAGES, NR>;
  star2_sweep_kernel<STAGES, MINB, NR><<<grid, C::kThreads, C::kSmemBytes, stream>>>(u, uprev, v2dt2, eta, out, p);
  return cudaGetLastError();
}

template <int STAGES, int MINB, int NR = 2>
KernelDesc make_desc2() {
  using C = Star2Cfg<STAGES, NR>;
  return KernelDesc{(const void*)star2_sweep_kernel<STAGES, MINB, NR>, C::kThreads, C::kSmemBytes, C::TY, STAGES,
                    C::BW, C::BH, false, &launch_star2<STAGES, MINB, NR>};
}

// Defined in kernels_apply.cu / kernels_wave.cu; radius in [1, 4].  The sweep's
// configuration also depends on the grid's x-y plane (radius 4).  `noeta`: the wave step
// of a region where eta is zero (no eta staged, no divide; the inner region of
// wave_step_pml).  `semi`: the sweep with
// the z stencil split into halves (stencil_apply_semi).
KernelDesc apply_kernel_desc(int radius, int64_t nx, int64_t ny);  // tile shape by plane size
// Two sweeps in one pass: built for radius 1 (fn is null for other radii).
KernelDesc apply2_kernel_desc(int radius);
KernelDesc semi_kernel_desc(int radius);
KernelDesc wave_kernel_desc(int radius, bool noeta);
// The direct-load sweep for small grids (direct_kernels.cuh), radius 1..4: its entry (for
// attributes and occupancy) and its launch with 256 threads per block.
const void* direct_kernel_fn(int radius);
cudaError_t launch_direct(int radius, dim3 grid, cudaStream_t stream, const DirectParams& p);
constexpr int kDirectThreads = 256;

}  // namespace libstencil
