/*
 * A plain C consumer of libosm: no C++ and no Python, only osm.h, the CUDA
 * runtime and libosm.so.  It allocates its own device buffers, runs the
 * attention forward and the row softmax through the C ABI, and checks the
 * results against direct double-precision sums of the definitions (small
 * sizes, so a double loop is enough).  Exit status 0 = every check passed.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "osm.h"

static uint32_t lcg_state = 12345u;
static float uniform_pm1(void) { /* deterministic, in [-1, 1) */
  lcg_state = lcg_state * 1664525u + 1013904223u;
  return (float)(lcg_state >> 8) / 8388608.0f - 1.0f;
}

static uint16_t to_bf16(float f) { /* round to nearest even (finite inputs) */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

#define CHECK_CUDA(x)                                                       \
  do {                                                                      \
    cudaError_t e_ = (x);                                                   \
    if (e_ != cudaSuccess) {                                                \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));              \
      return 2;                                                             \
    }                                                                       \
  } while (0)

static int attention_check(void) {
  const int B = 1, H = 2, Nq = 100, Nk = 150, d = 64, causal = 1;
  const float scale = 0.125f;
  const size_t nq = (size_t)B * H * Nq * d, nk = (size_t)B * H * Nk * d;
  uint16_t *hq = malloc(nq * 2), *hk = malloc(nk * 2), *hv = malloc(nk * 2), *ho = malloc(nq * 2);
  float *hl = malloc((size_t)B * H * Nq * 4);
  void *dq, *dk, *dv, *dout;
  float *dl;
  int bad = 0;
  for (size_t i = 0; i < nq; ++i) hq[i] = to_bf16(2.0f * uniform_pm1());
  for (size_t i = 0; i < nk; ++i) hk[i] = to_bf16(2.0f * uniform_pm1());
  for (size_t i = 0; i < nk; ++i) hv[i] = to_bf16(uniform_pm1());
  CHECK_CUDA(cudaMalloc(&dq, nq * 2));
  CHECK_CUDA(cudaMalloc(&dk, nk * 2));
  CHECK_CUDA(cudaMalloc(&dv, nk * 2));
  CHECK_CUDA(cudaMalloc(&dout, nq * 2));
  CHECK_CUDA(cudaMalloc((void **)&dl, (size_t)B * H * Nq * 4));
  CHECK_CUDA(cudaMemcpy(dq, hq, nq * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dk, hk, nk * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dv, hv, nk * 2, cudaMemcpyHostToDevice));

  if (osm_attn_fwd(dq, dk, dv, dout, dl, B, H, Nq, Nk, 96, scale, causal, NULL, NULL) !=
      OSM_ERR_UNSUPPORTED) {
    fprintf(stderr, "d = 96 was not refused\n");
    bad = 1;
  }
  osm_status st = osm_attn_fwd(dq, dk, dv, dout, dl, B, H, Nq, Nk, d, scale, causal, NULL, NULL);
  if (st != OSM_OK) {
    fprintf(stderr, "osm_attn_fwd: %s\n", osm_status_string(st));
    return 1;
  }
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(ho, dout, nq * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hl, dl, (size_t)B * H * Nq * 4, cudaMemcpyDeviceToHost));

  double worst_o = 0.0, worst_l = 0.0;
  double *s = malloc((size_t)Nk * sizeof(double));
  for (int h = 0; h < H; ++h) {
    for (int i = 0; i < Nq; ++i) {
      const uint16_t *q = hq + ((size_t)h * Nq + i) * d;
      const int last = i + (Nk - Nq); /* bottom-right causal alignment */
      double m = -INFINITY, l = 0.0;
      for (int j = 0; j <= last && j < Nk; ++j) {
        const uint16_t *k = hk + ((size_t)h * Nk + j) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += from_bf16(q[c]) * from_bf16(k[c]);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
      }
      for (int j = 0; j <= last && j < Nk; ++j) l += exp(s[j] - m);
      for (int c = 0; c < d; ++c) {
        double o = 0.0;
        for (int j = 0; j <= last && j < Nk; ++j)
          o += exp(s[j] - m) / l * from_bf16(hv[((size_t)h * Nk + j) * d + c]);
        const double got = from_bf16(ho[((size_t)h * Nq + i) * d + c]);
        const double err = fabs(got - o) - ldexp(fabs(o), -8);
        if (err > worst_o) worst_o = err;
      }
      const double lse = m + log(l);
      const double errl = fabs((double)hl[(size_t)h * Nq + i] - lse);
      if (errl > worst_l) worst_l = errl;
    }
  }
  printf("attention: max |O - ref| - 2^-8 |ref| = %.3g, max |lse - ref| = %.3g\n", worst_o, worst_l);
  if (!(worst_o <= 1e-2) || !(worst_l <= 1e-3)) bad = 1;
  free(s);
  free(hq);
  free(hk);
  free(hv);
  free(ho);
  free(hl);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(dout);
  cudaFree(dl);
  return bad;
}

static int softmax_check(void) {
  const int64_t rows = 3, cols = 1000;
  const size_t n = (size_t)(rows * cols);
  float *hx = malloc(n * 4), *hy = malloc(n * 4);
  float *dx, *dy;
  int bad = 0;
  for (size_t i = 0; i < n; ++i) hx[i] = 4.0f * uniform_pm1();
  hx[5] = 40.0f; /* a large entry in row 0 */
  CHECK_CUDA(cudaMalloc((void **)&dx, n * 4));
  CHECK_CUDA(cudaMalloc((void **)&dy, n * 4));
  CHECK_CUDA(cudaMemcpy(dx, hx, n * 4, cudaMemcpyHostToDevice));
  osm_status st = osm_softmax_rows(dx, dy, rows, cols, NULL);
  if (st != OSM_OK) {
    fprintf(stderr, "osm_softmax_rows: %s\n", osm_status_string(st));
    return 1;
  }
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(hy, dy, n * 4, cudaMemcpyDeviceToHost));
  double worst = 0.0;
  for (int64_t r = 0; r < rows; ++r) {
    double m = -INFINITY, l = 0.0;
    for (int64_t c = 0; c < cols; ++c)
      if (hx[r * cols + c] > m) m = hx[r * cols + c];
    for (int64_t c = 0; c < cols; ++c) l += exp((double)hx[r * cols + c] - m);
    for (int64_t c = 0; c < cols; ++c) {
      const double ref = exp((double)hx[r * cols + c] - m) / l;
      const double err = fabs((double)hy[r * cols + c] - ref) / (ref > 1e-30 ? ref : 1e-30);
      if (ref > 1e-30 && err > worst) worst = err;
    }
  }
  printf("softmax: max relative error = %.3g\n", worst);
  if (!(worst <= 1e-5)) bad = 1;
  free(hx);
  free(hy);
  cudaFree(dx);
  cudaFree(dy);
  return bad;
}

int main(void) {
  int bad = 0;
  if (osm_abi_version() <= 0) {
    fprintf(stderr, "bad ABI version\n");
    return 1;
  }
  bad |= attention_check();
  bad |= softmax_check();
  uint32_t word = 0;
  if (osm_device_status(NULL, &word) != OSM_OK || word != 0) {
    fprintf(stderr, "device status word %u\n", word);
    bad = 1;
  }
  printf(bad ? "FAILED\n" : "OK\n");
  return bad;
}
