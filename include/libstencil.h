/*
 * libstencil: 3D star-stencil sweeps and the fused acoustic wave step on NVIDIA GB300.
 *
 * Problem statement followed by every entry point:
 *  - Fields are flat 1D fp32 arrays with x innermost: point (x, y, z) lives at
 *    i = x + nx*(y + ny*z) (64-bit arithmetic).  "Accelerating High-Order Stencils on
 *    GPUs", 3D blocking with global memory: the grid is a flat 1D array and X, the
 *    innermost dimension, is the coalescing axis.
 *  - The star stencil of radius R computes, at every point at least R away from every
 *    face,
 *        out = coeffs[0]*u + sum_{r=1..R} coeffs[r] * (u at the six points at distance r
 *                                                       along +-x, +-y, +-z).
 *    coeffs[0] is the TOTAL centre weight (the three axes summed); coeffs[r] weighs each
 *    of the six neighbours at distance r.  Same page (the 25-point stencil reads four
 *    neighbours per direction per axis) and "Thread Coarsening 與 Register Tiling",
 *    Fig 8.10 (seven-point case; boundary points are not written).
 *  - Points closer than R to any face (the "shell") are NEVER written by any call.
 *
 * Memory ownership: the caller owns every field (device memory of the plan's device,
 * allocated by any allocator, e.g. PyTorch).  A plan owns a small device status block,
 * a cache of TMA descriptors and, only for the *_host entry points, a device workspace
 * allocated on their first call.  A plan must not be used by two host threads at once.
 *
 * Asynchrony: stencil_apply and wave_step only enqueue work on `stream` (a cudaStream_t;
 * NULL = the legacy default stream) and return.  STENCIL_OK means "enqueued".  A device
 * side failure (a bounded wait that ran out) is reported by stencil_plan_status.
 *
 * Errors: every int-returning call returns STENCIL_OK (0) or a negative code below;
 * stencil_last_error() then holds a message for the calling host thread.
 */
#ifndef LIBSTENCIL_H
#define LIBSTENCIL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define STENCIL_OK 0
#define STENCIL_ERR_ARG (-1)       /* null pointer, bad radius/size/count, wrong device */
#define STENCIL_ERR_ALIGNMENT (-2) /* pointer not 16-byte aligned, or nx not a multiple of 4 */
#define STENCIL_ERR_ALIAS (-3)     /* forbidden overlap between an input and the output */
#define STENCIL_ERR_CUDA (-4)      /* CUDA runtime or driver error (launch, copy, alloc) */
#define STENCIL_ERR_TIMEOUT (-5)   /* a kernel's bounded wait ran out (from stencil_plan_status) */

#define STENCIL_MAX_RADIUS 4

/* Sweep paths (stencil_plan_set_sweep_path). */
#define STENCIL_PATH_AUTO 0   /* chosen by grid size (the default) */
#define STENCIL_PATH_STAGED 1 /* the 2.5D kernel: TMA-staged planes, z window in registers */
#define STENCIL_PATH_DIRECT 2 /* the direct-load kernel: operands read straight from memory */

typedef struct stencil_plan stencil_plan; /* opaque */

/*
 * Create a plan for an nx x ny x nz grid and a star stencil of the given radius.
 *  nx, ny, nz  >= 1; nx must be a multiple of 4 (TMA row pitch is a multiple of 16 B).
 *              A grid with any dimension < 2*radius+1 has an empty interior: valid,
 *              and every sweep is then a no-op.
 *  radius      in [1, STENCIL_MAX_RADIUS].
 *  coeffs      radius+1 host floats (see the stencil definition above); copied.
 * The plan binds to the CUDA device current at creation.  Returns NULL on failure
 * (stencil_last_error() says why).
 */
stencil_plan* stencil_plan_create(int64_t nx, int64_t ny, int64_t nz, int radius,
                                  const float* coeffs);

/* Release the plan and everything it owns.  NULL is a no-op.  Synchronises nothing:
 * the caller must ensure no work that uses the plan is still running. */
void stencil_plan_destroy(stencil_plan* plan);

/*
 * One stencil sweep: out = stencil(in) on the interior; the shell of `out` is untouched.
 * Callers wanting the shell copied (a "fixed boundary") pre-copy `in` into `out` once;
 * ping-pong sweeps that start from two copies of the same field keep it fixed.
 *  in, out   device pointers to nx*ny*nz floats, 16-byte aligned, must not overlap.
 * The sweep runs on the plan's sweep path (stencil_plan_set_sweep_path).
 * Errors: STENCIL_ERR_ARG, _ALIGNMENT, _ALIAS, _CUDA.
 */
int stencil_apply(stencil_plan* plan, const float* in, float* out, void* stream);

/*
 * Which kernel computes the plan's sweeps (stencil_apply, the sweep loops and host-buffer
 * sweeps, the slabs of stencil_slabs_apply; not stencil_apply_semi or stencil_apply2):
 *  STENCIL_PATH_STAGED  the 2.5D kernel: each x-y tile plus its halo staged plane by plane
 *                       in shared memory by TMA, the z window held in registers; reads
 *                       each point from DRAM about once; the fast path on large grids.
 *  STENCIL_PATH_DIRECT  one thread per four x points of an interior row, every operand a
 *                       128-bit load from global memory; no staging and no waits.  On
 *                       small grids its launch-to-finish time is well below the staged
 *                       kernel's (GB300, one sweep launched after another: 64^3 radius 1
 *                       4.1 against 6.2 us, radius 4 4.1 against 8.2 us).
 *  STENCIL_PATH_AUTO    (the default) single sweeps on the direct kernel up to 100, 12, 5
 *                       and 3.5 million grid points for radius 1, 2, 3 and 4, on the
 *                       staged one above.
 * Both compute the same sweep up to fp32 rounding order.  Radius-1 loops (stencil_sweeps,
 * stencil_apply_host with nsweeps > 1) run most sweeps as two-sweep passes
 * (stencil_apply2) on the staged path, and on the automatic path from 8 million points,
 * where a pass beats two direct sweeps; their other sweeps run on the plan's sweep path,
 * and the direct path runs none as passes.  stencil_debug_inject affects only the staged
 * kernels.  Returns STENCIL_OK, or STENCIL_ERR_ARG for a NULL plan or a path outside
 * [0, 2].
 */
int stencil_plan_set_sweep_path(stencil_plan* plan, int path);

/*
 * Two sweeps in one pass: out = S(S(in)) for the plan's stencil S (temporal blocking of
 * the ping-pong loop), with the shell of every level held at in's values, i.e. exactly
 * what two stencil_apply calls in -> tmp -> out compute when out and tmp start with in's
 * shell.  The intermediate level stays in shared memory, so the pass reads and writes the
 * grid once for two sweeps.  Built for radius 1 (the 7-point stencil); other radii return
 * STENCIL_ERR_ARG.  Same arguments, layout, aliasing rules and errors as stencil_apply;
 * the shell of `out` is untouched.  stencil_sweeps and stencil_apply_host use it for most
 * of a radius-1 loop.
 */
int stencil_apply2(stencil_plan* plan, const float* in, float* out, void* stream);

/*
 * The same sweep computed in semi-stencil form ("Accelerating High-Order Stencils on
 * GPUs", the semi-stencil strategy: a stencil along one axis is split into a forward and
 * a backward half, so the centre and one half are read together and the other half is
 * carried as a partial result).  Along z, the centre and the R planes below each output
 * plane are read from shared memory (the ring keeps them), and the R planes above
 * finish a running partial sum held in registers, R partial sums per point instead of
 * 2R.  Same result up to fp32 rounding order, same arguments, layout, aliasing rules and
 * errors as stencil_apply.  An alternative kernel for comparison: stencil_apply is the
 * faster one on GB300.
 */
int stencil_apply_semi(stencil_plan* plan, const float* in, float* out, void* stream);

/*
 * One time step of the acoustic isotropic wave equation with a sponge layer, fused
 * into a single pass (the stencil of the plan is the Laplacian, h = 1):
 *   u_next = (2*u - (1 - eta)*u_prev + v2dt2 * lap(u)) / (1 + eta)
 * on the interior; the shell of u_next is untouched.  "Accelerating High-Order Stencils
 * on GPUs" names the acoustic isotropic model, its fields u and eta and the PML region;
 * the update above is the second-order leapfrog with a pointwise damping term.
 *  All six pointers: device, nx*ny*nz floats, 16-byte aligned.
 *  u_next must not overlap u, v2dt2 or eta.  u_next == u_prev exactly is allowed (each
 *  point reads u_prev only where it writes u_next), which permits two-buffer stepping;
 *  any partial overlap is STENCIL_ERR_ALIAS.
 * Errors: STENCIL_ERR_ARG, _ALIGNMENT, _ALIAS, _CUDA.
 */
int wave_step(stencil_plan* plan, const float* u_prev, const float* u, float* u_next,
              const float* v2dt2, const float* eta, void* stream);

/*
 * The same wave step for a model whose damping lives in a band of `pml_width` points
 * along the six faces, run as the pages run it: one launch per data region ("Accelerating
 * High-Order Stencils on GPUs" launches the inner region and the PML region separately).
 * Precondition: eta = 0 at every point at least pml_width away from all faces.  The inner
 * region (every 64 x tile-height output tile lying wholly at least pml_width from the x
 * and y faces, over the output planes at least pml_width from the z faces) runs a kernel
 * that stages no eta and never divides, the plain leapfrog
 * u_next = 2u - u_prev + v2dt2*lap(u) (16 instead of 20 bytes per point); the band around
 * it (at most six boxes, one launch) runs the full update on an internal stream beside
 * it, and `stream` waits for both.  If the precondition does not hold, points of the inner
 * region are computed with eta taken as 0.  Same fields, layout, aliasing rules and errors
 * as wave_step; pml_width >= 0.
 */
int wave_step_pml(stencil_plan* plan, const float* u_prev, const float* u, float* u_next,
                  const float* v2dt2, const float* eta, int64_t pml_width, void* stream);

/*
 * Damping field of a PML whose computation reads eta through a 7-point stencil
 * ("Accelerating High-Order Stencils on GPUs": in the PML region the computations on eta
 * use a low-order 7-point stencil, halo one; the page prints no formula).  Reading: the
 * damping at a point is the radius-1 star stencil of eta,
 *   eta_eff = e0*eta + e1*(eta at the six face neighbours),
 * written at every point at least one away from every face (the points on the faces are
 * left as they were: no step reads them).  eta does not change in time, so this runs once per model: every later
 * wave_step / wave_step_pml / wave_steps with eta_eff in place of eta is the step with the
 * 7-point damping, at the cost of the pointwise step.  With e0 + 6*e1 = 1 a constant eta
 * is left unchanged.  eta, eta_eff: device, nx*ny*nz floats, 16-byte aligned, must not
 * overlap.  The first call creates a radius-1 plan of the grid inside the plan.
 * Errors: STENCIL_ERR_ARG, _ALIGNMENT, _ALIAS, _CUDA.
 */
int wave_eta_stencil(stencil_plan* plan, const float* eta, float* eta_eff, float e0, float e1,
                     void* stream);

/*
 * Time loops on device buffers (hot-path loop row: sweeps and steps back to back on one
 * stream, as the benchmark workloads run them).
 *
 * stencil_sweeps: `nsweeps` ping-pong sweeps a -> b -> a -> ...; after an even count the
 *   result is in a, after an odd count in b.  For radius 1, 2*floor(nsweeps/4) passes of
 *   stencil_apply2 carry most of them (each pass two sweeps), the rest are single sweeps.  Both buffers keep their shells (start them
 *   as two copies of the same field for a fixed boundary).  a and b must not overlap.
 * wave_steps: `nsteps` wave steps with three-buffer rotation: each step computes the next
 *   level into the buffer of the oldest one, so after n steps the newest level is in
 *   (u_prev, u, u_tmp)[(n + 1) % 3] and the one before it in [n % 3].  pml_width < 0 uses
 *   wave_step, pml_width >= 0 wave_step_pml.  The three levels must not overlap each other,
 *   v2dt2 or eta.
 * use_graph != 0 records the launches once into a CUDA graph (cached in the plan for the
 *   same buffers and count) and replays it, which removes the per-launch host cost.  The
 *   first call with a new key captures on a private stream; do not call it while `stream`
 *   itself is being captured.  Errors as for stencil_apply / wave_step.
 */
int stencil_sweeps(stencil_plan* plan, float* a, float* b, int nsweeps, int use_graph, void* stream);
int wave_steps(stencil_plan* plan, float* u_prev, float* u, float* u_tmp, const float* v2dt2,
               const float* eta, int nsteps, int64_t pml_width, int use_graph, void* stream);

/*
 * Synchronise `stream`, then report device-side failures of this plan's kernels since
 * the previous call: STENCIL_ERR_TIMEOUT if a kernel's bounded wait for staged data ran
 * out (its outputs are then undefined), STENCIL_ERR_CUDA on a CUDA error, else STENCIL_OK.
 * Reading the status clears it.
 */
int stencil_plan_status(stencil_plan* plan, void* stream);

/* Message describing the last error of the calling host thread ("" if none). */
const char* stencil_last_error(void);

/*
 * Host-buffer convenience entry points.  They copy host arrays to a device workspace
 * owned by the plan (allocated on first use, 2 or 4 fields), run on `stream`, copy the
 * result back and synchronise the stream.  Host memory may be pageable or pinned
 * (pinned overlaps better).  Return STENCIL_OK or an error code; a device timeout is
 * reported as STENCIL_ERR_TIMEOUT.
 *
 * stencil_apply_host: out_host = `nsweeps` ping-pong sweeps of in_host with a fixed
 *   shell (the shell of out_host equals that of in_host).  nsweeps >= 0.  A single sweep
 *   is pipelined over z-slabs on three internal streams (copy in, sweep, copy out), so
 *   both copy directions and the sweep overlap; use pinned host memory to benefit.
 * wave_run_host: `nsteps` wave steps from (u_prev_host, u_host); on return
 *   u_prev_host and u_host hold the last two time levels (u_host the newest).
 */
int stencil_apply_host(stencil_plan* plan, const float* in_host, float* out_host,
                       int nsweeps, void* stream);
int wave_run_host(stencil_plan* plan, float* u_prev_host, float* u_host,
                  const float* v2dt2_host, const float* eta_host, int nsteps, void* stream);

/*
 * Launch geometry the plan chose for `kind` (0 = stencil_apply, 1 = wave_step,
 * 2 = the no-eta kernel of wave_step_pml's inner region, over the whole grid,
 * 3 = stencil_apply_semi, 4 = stencil_apply2 (radius 1 only)), written
 * to info[0..n): grid CTAs, threads per CTA, dynamic shared bytes, CTAs resident per
 * SM, x-y tiles, z-chunks, tile width, tile height, pipeline stages, SM count, and the
 * sweep path (STENCIL_PATH_STAGED or _DIRECT; kind 0 on a direct plan reports its blocks,
 * 256 threads, no shared memory, blocks per SM, 0 tiles and chunks, a 4 x 1 "tile" and 0
 * stages).  At most 11 values.  Returns the number of values written, or a negative error
 * code.
 */
int stencil_plan_launch_info(const stencil_plan* plan, int kind, int64_t* info, int n);

/*
 * Where the time of the plan's last pipelined host-buffer sweep (stencil_apply_host with
 * nsweeps == 1) went, from CUDA events on its three streams, in milliseconds since the
 * call's start: ms[0] the whole call (last copy out done), ms[1] the first slab landed on
 * the device, ms[2] the last slab landed (copies in done), ms[3] the last slab swept;
 * ms[4] is the number of slabs.  Valid after that call returned; n values at most 5 are
 * written.  Returns the number written, or STENCIL_ERR_ARG if no such call has run.
 */
int stencil_plan_host_phases(const stencil_plan* plan, float* ms, int n);

/*
 * The z-chunk schedule stencil_plan_create would choose for `kind` (as for
 * stencil_plan_launch_info) on a GPU with `num_sms` SMs that holds `ctas_per_sm` CTAs of
 * that kernel per SM.  Host-only: makes no CUDA call, so it also runs without a GPU
 * (capacity planning, tests).  Its cost does not grow with nz.  Writes to info[0..n):
 * grid CTAs, x-y tiles, z-chunks per tile column, work items, tile width, tile height,
 * x of the first tile column (0, or R where the kernel stores whole tiles through a map of
 * the interior) (all 0 but the tile sizes and origin when the interior is empty).  Returns the number of values
 * written, or STENCIL_ERR_ARG for a grid or radius stencil_plan_create would reject, a
 * kind outside [0, 3], num_sms or ctas_per_sm < 1.
 */
int stencil_schedule_query(int64_t nx, int64_t ny, int64_t nz, int radius, int kind,
                           int num_sms, int ctas_per_sm, int64_t* info, int n);

/*
 * Test hook for the device watchdog: mode 1 makes every CTA of the plan's next launches
 * skip one of its staged loads, so the bounded wait for it runs out and
 * stencil_plan_status returns STENCIL_ERR_TIMEOUT; mode 0 restores normal operation.
 * The wait limit is about two seconds.  Returns STENCIL_OK or STENCIL_ERR_ARG.
 */
int stencil_debug_inject(stencil_plan* plan, int mode);

/*
 * Allocation-free stencil sweep.  No counterpart in the paper: it serves callers that
 * cannot call cudaMalloc when they need a sweep (for example code running inside another
 * framework's memory pool that owns the free device memory, or a process whose device
 * memory footprint is fixed at start-up).  It computes exactly what
 * stencil_plan_create + stencil_apply compute (on the automatic sweep path), with the same
 * arguments, restrictions and error codes, and allocates nothing: no cudaMalloc/cudaFree,
 * no heap, no plan.
 *
 * Scratch: the kernel's 16-byte status block lives in a file-scope device array of 256
 * bytes that every GPU which loads the library holds until the process exits.  The need
 * does not grow with the grid; grids beyond the library's maximum (each dimension
 * <= 2^30, at most 2^40 points) are rejected with STENCIL_ERR_ARG.  Every call looks up
 * the array's address in the current device's context (cudaGetSymbolAddress, which
 * allocates nothing); the first lookup in a context may load the library's device code
 * there, so make the first call on a device before any stream capture.  The call clears
 * the status words, enqueues the sweep on `stream`, then synchronises `stream` so that it
 * can report a device-side timeout (STENCIL_ERR_TIMEOUT); it must therefore not be made
 * from a CUDA stream callback or host function, where CUDA forbids those calls.  Every
 * call shares the one array per device: calls that overlap on the GPU (other host
 * threads, other streams) race on it.
 */
int stencil_apply_noalloc(int64_t nx, int64_t ny, int64_t nz, int radius, const float* coeffs,
                          const float* in, float* out, void* stream);

/*
 * z-slab decomposition.  The grid is cut along z into `nslabs` slabs; slab k owns the
 * global planes [o_k, o_k+1), o_k = floor(k * nz / nslabs), and is stored as a separate
 * nx x ny x (e_k - s_k) device array holding the global planes [s_k, e_k) =
 * [max(0, o_k - R), min(nz, o_k+1 + R)): its owned planes plus up to R ghost planes on
 * each side (plane z of the grid is plane z - s_k of the slab array, x innermost as
 * everywhere).  Every slab must own at least R planes.  Each slab array has the layout,
 * alignment and shell rules of a field of stencil_apply; the ghost planes are slab-local
 * shell, which no sweep writes.
 *
 * The path shards this way along z, one ghost exchange of R planes each way per cut and
 * per sweep or step.  Here every slab lives on the device current at creation; the calls
 * copy ghost planes between slab arrays with device-to-device copies on an internal
 * stream, which then also computes the output planes next to the cuts, while `stream`
 * computes the planes that read no ghost plane; `stream` waits for both.
 *
 * stencil_slabs_create:   plans for every slab (coeffs and radius as stencil_plan_create);
 *                         NULL on failure (stencil_last_error says why).
 * stencil_slabs_extent:   info[0..n) = s_k, e_k, o_k, o_k+1 (global planes) of slab k.
 * stencil_slabs_exchange: fill every ghost plane of the field's slabs from its owner.
 * stencil_slabs_apply:    one sweep of the whole grid: exchange ghost planes of `in`, then
 *                         stencil_apply on every slab; out[k] gets slab k's owned interior
 *                         planes (its shell and ghost planes are untouched).
 * stencil_slabs_wave_step: one wave step of the whole grid (ghosts of `u` exchanged; the
 *                         other fields are read only at the output points).  u_next[k] ==
 *                         u_prev[k] for every slab is allowed (two-buffer stepping).
 * stencil_slabs_status:   stencil_plan_status of every slab's plan.
 * Fields are host arrays of nslabs device pointers; no two slab arrays may overlap
 * (STENCIL_ERR_ALIAS).  Errors as for stencil_apply / wave_step.
 */
typedef struct stencil_slabs stencil_slabs; /* opaque */
stencil_slabs* stencil_slabs_create(int64_t nx, int64_t ny, int64_t nz, int radius, const float* coeffs,
                                    int nslabs);
void stencil_slabs_destroy(stencil_slabs* slabs);
int stencil_slabs_extent(const stencil_slabs* slabs, int k, int64_t* info, int n);
int stencil_slabs_exchange(stencil_slabs* slabs, float* const* fields, void* stream);
int stencil_slabs_apply(stencil_slabs* slabs, float* const* in, float* const* out, void* stream);
int stencil_slabs_wave_step(stencil_slabs* slabs, float* const* u_prev, float* const* u,
                            float* const* u_next, float* const* v2dt2, float* const* eta, void* stream);
int stencil_slabs_status(stencil_slabs* slabs, void* stream);

/* Library version string. */
const char* stencil_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBSTENCIL_H */
