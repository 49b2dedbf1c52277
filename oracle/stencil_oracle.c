/*
 * CPU oracle for the 3D star stencil and the fused acoustic wave step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library under test calls, links or
 * includes this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or constant with the CUDA
 * path: it is a plain, slow, obviously correct restatement of what the pages define.
 *
 * Grid layout (all entry points): a flat 1D array with x innermost,
 * i = x + nx*(y + ny*z), 64-bit indices.  Source: "Accelerating High-Order Stencils on
 * GPUs", 3D blocking with global memory (gmem_{Dx}_{Dy}_{Dz}): the 3D grid is stored as
 * a flat 1D array and X is the innermost dimension.
 *
 * Star stencil of radius R (apply):
 *   out[i] = c[0]*in[i] + sum_{r=1..R} c[r] * ( in[i-r] + in[i+r]
 *                                             + in[i-r*nx] + in[i+r*nx]
 *                                             + in[i-r*nx*ny] + in[i+r*nx*ny] )
 * for every point at least R away from every face; every other output element is left
 * untouched.  Sources: "Accelerating High-Order Stencils on GPUs", 3D blocking with
 * global memory (the 25-point stencil fetches the point itself and four neighbours in
 * each direction of each axis); "Thread Coarsening 與 Register Tiling", Fig 8.10 body
 * (centre plus six face neighbours; threads on the boundary write nothing).
 * c[0] is the TOTAL centre weight (all three axes summed); c[r] weights each of the six
 * neighbours at distance r.
 *
 * Wave step (the acoustic isotropic update with a pointwise sponge):
 *   u_next[i] = ( 2*u[i] - (1 - eta[i])*u_prev[i] + v2dt2[i]*lap(u)[i] ) / (1 + eta[i])
 * on the same interior, lap = the star stencil above.  The pages name the acoustic
 * isotropic model, the fields u and eta, the 25-point inner stencil and the PML region
 * ("Accelerating High-Order Stencils on GPUs", smem_eta kernels) but print no update
 * equation; this is the plainest second-order leapfrog with a sponge that fits them.
 *
 * Arithmetic: every input value and coefficient is converted to double, the whole
 * expression is evaluated in double in the order written above, and the fp32 entry
 * points round once to fp32 at the end.  Build with -ffp-contract=off so that x86 and
 * Arm give identical bits.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Star stencil at linear index i, double inputs. */
static double star_f64(const double* u, int64_t i, int64_t sx, int64_t sy, int64_t sz,
                       int R, const double* c) {
    double acc = c[0] * u[i];
    for (int r = 1; r <= R; ++r) {
        double s = u[i - r * sx] + u[i + r * sx]
                 + u[i - r * sy] + u[i + r * sy]
                 + u[i - r * sz] + u[i + r * sz];
        acc += c[r] * s;
    }
    return acc;
}

/* Same expression on fp32 inputs, each converted to double before use. */
static double star_f32(const float* u, int64_t i, int64_t sx, int64_t sy, int64_t sz,
                       int R, const double* c) {
    double acc = c[0] * (double)u[i];
    for (int r = 1; r <= R; ++r) {
        double s = (double)u[i - r * sx] + (double)u[i + r * sx]
                 + (double)u[i - r * sy] + (double)u[i + r * sy]
                 + (double)u[i - r * sz] + (double)u[i + r * sz];
        acc += c[r] * s;
    }
    return acc;
}

static int interior_empty(int64_t nx, int64_t ny, int64_t nz, int R) {
    return nx < 2 * R + 1 || ny < 2 * R + 1 || nz < 2 * R + 1;
}

static int is_interior(int64_t nx, int64_t ny, int64_t nz, int R, int64_t i) {
    int64_t x = i % nx, y = (i / nx) % ny, z = i / (nx * ny);
    return x >= R && x < nx - R && y >= R && y < ny - R && z >= R && z < nz - R;
}

/* ---- apply ---------------------------------------------------------------------- */

void oracle_apply_f64(int64_t nx, int64_t ny, int64_t nz, int R, const double* c,
                      const double* in, double* out) {
    if (interior_empty(nx, ny, nz, R)) return;
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t z = R; z < nz - R; ++z)
        for (int64_t y = R; y < ny - R; ++y)
            for (int64_t x = R; x < nx - R; ++x) {
                int64_t i = x + sy * y + sz * z;
                out[i] = star_f64(in, i, 1, sy, sz, R, c);
            }
}

void oracle_apply_f32(int64_t nx, int64_t ny, int64_t nz, int R, const float* cf,
                      const float* in, float* out) {
    if (interior_empty(nx, ny, nz, R)) return;
    double c[8];
    for (int r = 0; r <= R; ++r) c[r] = (double)cf[r];
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t z = R; z < nz - R; ++z)
        for (int64_t y = R; y < ny - R; ++y)
            for (int64_t x = R; x < nx - R; ++x) {
                int64_t i = x + sy * y + sz * z;
                out[i] = (float)star_f32(in, i, 1, sy, sz, R, c);
            }
}

/* Apply at an explicit list of linear indices (for sampled checks of large grids).
 * Indices outside the interior give NaN. */
void oracle_apply_points_f32(int64_t nx, int64_t ny, int64_t nz, int R, const float* cf,
                             const float* in, int64_t npts, const int64_t* idx, float* vals) {
    double c[8];
    for (int r = 0; r <= R; ++r) c[r] = (double)cf[r];
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < npts; ++k) {
        int64_t i = idx[k];
        if (i < 0 || i >= nx * ny * nz || !is_interior(nx, ny, nz, R, i)) {
            vals[k] = NAN;
            continue;
        }
        vals[k] = (float)star_f32(in, i, 1, sy, sz, R, c);
    }
}

/* ---- wave step ------------------------------------------------------------------ */

void oracle_wave_step_f64(int64_t nx, int64_t ny, int64_t nz, int R, const double* c,
                          const double* u_prev, const double* u, double* u_next,
                          const double* v2dt2, const double* eta) {
    if (interior_empty(nx, ny, nz, R)) return;
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t z = R; z < nz - R; ++z)
        for (int64_t y = R; y < ny - R; ++y)
            for (int64_t x = R; x < nx - R; ++x) {
                int64_t i = x + sy * y + sz * z;
                double lap = star_f64(u, i, 1, sy, sz, R, c);
                double t = 2.0 * u[i] - (1.0 - eta[i]) * u_prev[i] + v2dt2[i] * lap;
                u_next[i] = t / (1.0 + eta[i]);
            }
}

static float wave_point_f32(const float* u_prev, const float* u, const float* v2dt2,
                            const float* eta, int64_t i, int64_t sy, int64_t sz, int R,
                            const double* c) {
    double lap = star_f32(u, i, 1, sy, sz, R, c);
    double e = (double)eta[i];
    double t = 2.0 * (double)u[i] - (1.0 - e) * (double)u_prev[i] + (double)v2dt2[i] * lap;
    return (float)(t / (1.0 + e));
}

/* u_next may be the same array as u_prev (each point reads u_prev only where it
 * writes u_next); it must not overlap u. */
void oracle_wave_step_f32(int64_t nx, int64_t ny, int64_t nz, int R, const float* cf,
                          const float* u_prev, const float* u, float* u_next,
                          const float* v2dt2, const float* eta) {
    if (interior_empty(nx, ny, nz, R)) return;
    double c[8];
    for (int r = 0; r <= R; ++r) c[r] = (double)cf[r];
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t z = R; z < nz - R; ++z)
        for (int64_t y = R; y < ny - R; ++y)
            for (int64_t x = R; x < nx - R; ++x) {
                int64_t i = x + sy * y + sz * z;
                u_next[i] = wave_point_f32(u_prev, u, v2dt2, eta, i, sy, sz, R, c);
            }
}

void oracle_wave_points_f32(int64_t nx, int64_t ny, int64_t nz, int R, const float* cf,
                            const float* u_prev, const float* u, const float* v2dt2,
                            const float* eta, int64_t npts, const int64_t* idx, float* vals) {
    double c[8];
    for (int r = 0; r <= R; ++r) c[r] = (double)cf[r];
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < npts; ++k) {
        int64_t i = idx[k];
        if (i < 0 || i >= nx * ny * nz || !is_interior(nx, ny, nz, R, i)) {
            vals[k] = NAN;
            continue;
        }
        vals[k] = wave_point_f32(u_prev, u, v2dt2, eta, i, sy, sz, R, c);
    }
}

/* ---- wave step with the damping read through a 7-point stencil of eta ------------ */

/* "Accelerating High-Order Stencils on GPUs" says the computation on eta in the PML
 * region is a low-order 7-point stencil (halo of eta: one point) but prints no formula.
 * Reading: the damping at an interior point is the radius-1 star stencil of eta,
 *   eff = e0*eta[i] + e1*(eta[i-1] + eta[i+1] + eta[i-nx] + eta[i+nx] + eta[i-nx*ny] + eta[i+nx*ny]),
 * used in place of eta[i] in the update above.  With e0 + 6*e1 = 1 a constant eta gives
 * back the pointwise update. */
static double eta7_f64(const double* eta, int64_t i, int64_t sy, int64_t sz, double e0, double e1) {
    double s = eta[i - 1] + eta[i + 1] + eta[i - sy] + eta[i + sy] + eta[i - sz] + eta[i + sz];
    return e0 * eta[i] + e1 * s;
}

void oracle_wave_step_eta7_f64(int64_t nx, int64_t ny, int64_t nz, int R, const double* c,
                               double e0, double e1, const double* u_prev, const double* u,
                               double* u_next, const double* v2dt2, const double* eta) {
    if (interior_empty(nx, ny, nz, R)) return;
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t z = R; z < nz - R; ++z)
        for (int64_t y = R; y < ny - R; ++y)
            for (int64_t x = R; x < nx - R; ++x) {
                int64_t i = x + sy * y + sz * z;
                double lap = star_f64(u, i, 1, sy, sz, R, c);
                double e = eta7_f64(eta, i, sy, sz, e0, e1);
                double t = 2.0 * u[i] - (1.0 - e) * u_prev[i] + v2dt2[i] * lap;
                u_next[i] = t / (1.0 + e);
            }
}

void oracle_wave_step_eta7_f32(int64_t nx, int64_t ny, int64_t nz, int R, const float* cf,
                               float e0f, float e1f, const float* u_prev, const float* u,
                               float* u_next, const float* v2dt2, const float* eta) {
    if (interior_empty(nx, ny, nz, R)) return;
    double c[8];
    for (int r = 0; r <= R; ++r) c[r] = (double)cf[r];
    const double e0 = (double)e0f, e1 = (double)e1f;
    const int64_t sy = nx, sz = nx * ny;
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t z = R; z < nz - R; ++z)
        for (int64_t y = R; y < ny - R; ++y)
            for (int64_t x = R; x < nx - R; ++x) {
                int64_t i = x + sy * y + sz * z;
                double lap = star_f32(u, i, 1, sy, sz, R, c);
                double s = (double)eta[i - 1] + (double)eta[i + 1] + (double)eta[i - sy] +
                           (double)eta[i + sy] + (double)eta[i - sz] + (double)eta[i + sz];
                double e = e0 * (double)eta[i] + e1 * s;
                double t = 2.0 * (double)u[i] - (1.0 - e) * (double)u_prev[i] + (double)v2dt2[i] * lap;
                u_next[i] = (float)(t / (1.0 + e));
            }
}
