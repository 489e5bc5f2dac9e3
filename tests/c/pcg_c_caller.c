/* A plain C99 caller of the library: only include/pcg.h and the host-buffer
 * entry points, no CUDA runtime of its own.  Reads the grid, the
 * coefficients and b from a binary input file, solves A x = b to a relative
 * residual of 1e-10 with pcg_solve_host, then again with new coefficients
 * through pcg_update_solve_host, and writes both iteration counts, statuses
 * and solutions to the output file.
 *
 * Input  (doubles unless noted): int32 nx, ny, nz; a_v; mass; a_h field
 *        (nx*ny); dz (nz); b (nx*ny*nz); scale of the second field.
 * Output: int32 iters1, status1; x1 (n); int32 iters2, status2; x2 (n).
 * Exit code: 0, or 10 + the status of a failed pcg_create, or 20 + the
 * status of a failed solve. */
#include <stdio.h>
#include <stdlib.h>

#include "pcg.h"

static int read_all(FILE* f, void* p, size_t size, size_t count) {
  return fread(p, size, count, f) == count;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s input output\n", argv[0]);
    return 2;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 3;
  int dims[3];
  double a_v, mass, scale;
  if (!read_all(in, dims, sizeof(int), 3) || !read_all(in, &a_v, sizeof(double), 1) ||
      !read_all(in, &mass, sizeof(double), 1))
    return 4;
  const int nx = dims[0], ny = dims[1], nz = dims[2];
  const size_t ncols = (size_t)nx * ny, n = ncols * nz;
  double* ah = malloc(sizeof(double) * ncols);
  double* ah2 = malloc(sizeof(double) * ncols);
  double* dz = malloc(sizeof(double) * nz);
  double* b = malloc(sizeof(double) * n);
  double* x = calloc(n, sizeof(double));
  double* hist = malloc(sizeof(double) * 501);
  if (!ah || !ah2 || !dz || !b || !x || !hist) return 5;
  if (!read_all(in, ah, sizeof(double), ncols) || !read_all(in, dz, sizeof(double), nz) ||
      !read_all(in, b, sizeof(double), n) || !read_all(in, &scale, sizeof(double), 1))
    return 4;
  fclose(in);

  pcg_coeffs c = {1.0, ah, a_v, mass, dz};
  pcg_ctx* ctx = NULL;
  int st = pcg_create(nx, ny, nz, &c, &ctx);
  if (st != PCG_OK) {
    fprintf(stderr, "pcg_create: %s\n", pcg_last_error(NULL));
    return 10 + st;
  }
  FILE* out = fopen(argv[2], "wb");
  if (!out) return 3;
  int res[2];
  /* x holds the initial guess (zero) and receives the solution */
  st = pcg_solve_host(ctx, b, x, 1e-10, 500, &res[0], hist);
  res[1] = st;
  fwrite(res, sizeof(int), 2, out);
  fwrite(x, sizeof(double), n, out);
  if (st != PCG_OK) {
    fprintf(stderr, "pcg_solve_host: %s\n", pcg_last_error(ctx));
    pcg_destroy(ctx);
    fclose(out);
    return 20 + st;
  }
  /* new coefficients and a zero initial guess in one call */
  for (size_t i = 0; i < ncols; ++i) ah2[i] = ah[i] * scale;
  pcg_coeffs c2 = {1.0, ah2, a_v, mass, dz};
  st = pcg_update_solve_host(ctx, &c2, b, NULL, x, 1e-10, 500, &res[0], NULL);
  res[1] = st;
  fwrite(res, sizeof(int), 2, out);
  fwrite(x, sizeof(double), n, out);
  fclose(out);
  pcg_destroy(ctx);
  free(ah);
  free(ah2);
  free(dz);
  free(b);
  free(x);
  free(hist);
  return st == PCG_OK ? 0 : 20 + st;
}
