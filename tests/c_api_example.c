/*
 * A plain C caller of libstencil: the 25-point (radius 4) 8th-order Laplacian of a field
 * read from a file, once through device buffers (stencil_apply) and once through the
 * host-buffer call (stencil_apply_host); both results are written out.  It uses only
 * include/libstencil.h and the CUDA runtime API.
 *
 *   c_api_example NX NY NZ IN OUT_DEVICE OUT_HOST
 *
 * IN holds NX*NY*NZ float32 values, x innermost.  The output files hold the same shape;
 * their shell (points closer than 4 to a face) is a copy of the input.  Exit status 0 on
 * success; on failure the message of stencil_last_error() goes to stderr.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "libstencil.h"

static int read_file(const char* path, float* dst, size_t n) {
  FILE* f = fopen(path, "rb");
  if (!f) return -1;
  const size_t got = fread(dst, sizeof(float), n, f);
  fclose(f);
  return got == n ? 0 : -1;
}

static int write_file(const char* path, const float* src, size_t n) {
  FILE* f = fopen(path, "wb");
  if (!f) return -1;
  const size_t put = fwrite(src, sizeof(float), n, f);
  fclose(f);
  return put == n ? 0 : -1;
}

static int fail_stencil(const char* what, int rc) {
  fprintf(stderr, "%s failed (%d): %s\n", what, rc, stencil_last_error());
  return 1;
}

static int fail_cuda(const char* what, cudaError_t e) {
  fprintf(stderr, "%s failed: %s\n", what, cudaGetErrorString(e));
  return 1;
}

int main(int argc, char** argv) {
  if (argc != 7) {
    fprintf(stderr, "usage: %s NX NY NZ IN OUT_DEVICE OUT_HOST\n", argv[0]);
    return 2;
  }
  const int64_t nx = atoll(argv[1]), ny = atoll(argv[2]), nz = atoll(argv[3]);
  const size_t n = (size_t)(nx * ny * nz);
  /* Per-axis 8th-order weights -205/72, 8/5, -1/5, 8/315, -1/560; the centre weight is the
     three axes summed. */
  const float coeffs[5] = {(float)(3.0 * -205.0 / 72.0), 8.0f / 5.0f, -1.0f / 5.0f,
                           8.0f / 315.0f, -1.0f / 560.0f};

  float* host_in = (float*)malloc(n * sizeof(float));
  float* host_out = (float*)malloc(n * sizeof(float));
  if (!host_in || !host_out || read_file(argv[4], host_in, n)) {
    fprintf(stderr, "cannot read %s\n", argv[4]);
    return 1;
  }

  stencil_plan* plan = stencil_plan_create(nx, ny, nz, 4, coeffs);
  if (!plan) return fail_stencil("stencil_plan_create", 0);

  /* Device buffers: the caller owns them; the output starts as a copy of the input so its
     shell holds the input's values (the library never writes the shell). */
  float *d_in = NULL, *d_out = NULL;
  cudaError_t e = cudaMalloc((void**)&d_in, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc((void**)&d_out, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMemcpy(d_in, host_in, n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(d_out, d_in, n * sizeof(float), cudaMemcpyDeviceToDevice);
  if (e != cudaSuccess) return fail_cuda("device setup", e);

  cudaStream_t stream;
  e = cudaStreamCreate(&stream);
  if (e != cudaSuccess) return fail_cuda("cudaStreamCreate", e);
  int rc = stencil_apply(plan, d_in, d_out, stream);
  if (rc != STENCIL_OK) return fail_stencil("stencil_apply", rc);
  rc = stencil_plan_status(plan, stream); /* synchronises the stream */
  if (rc != STENCIL_OK) return fail_stencil("stencil_plan_status", rc);
  e = cudaMemcpy(host_out, d_out, n * sizeof(float), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda("copy out", e);
  if (write_file(argv[5], host_out, n)) {
    fprintf(stderr, "cannot write %s\n", argv[5]);
    return 1;
  }

  /* The same sweep from host buffers; the call copies, sweeps and synchronises itself. */
  rc = stencil_apply_host(plan, host_in, host_out, 1, stream);
  if (rc != STENCIL_OK) return fail_stencil("stencil_apply_host", rc);
  if (write_file(argv[6], host_out, n)) {
    fprintf(stderr, "cannot write %s\n", argv[6]);
    return 1;
  }

  /* An error path: in and out may not alias. */
  rc = stencil_apply(plan, d_in, d_in, stream);
  if (rc != STENCIL_ERR_ALIAS) {
    fprintf(stderr, "aliasing was not rejected (%d)\n", rc);
    return 1;
  }

  stencil_plan_destroy(plan);
  cudaStreamDestroy(stream);
  cudaFree(d_in);
  cudaFree(d_out);
  free(host_in);
  free(host_out);
  printf("ok %s\n", stencil_version());
  return 0;
}
