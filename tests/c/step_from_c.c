/* An owner step from plain C with the CUDA runtime: device buffers from
 * cudaMalloc, one call of mfsdp_muon_owner_step and one of the no-workspace
 * entry point on the default stream, no other framework.  Checks both device
 * status words, that every update element is finite and that each matrix's update
 * has the Frobenius norm Newton-Schulz gives a full-rank input (its singular
 * values lie in [0.68, 1.14], so ||O||_F / sqrt(s) does too), and that the two
 * entry points agree bit for bit.  Prints "ok" and returns 0, or names the
 * first failed check. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "mfsdp.h"

#define CHECK(cond)                                          \
  do {                                                       \
    if (!(cond)) {                                           \
      printf("failed: %s (line %d)\n", #cond, __LINE__);     \
      return 1;                                              \
    }                                                        \
  } while (0)

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint16_t float_to_bf16(float f) {   /* round to nearest even; inputs are finite */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

int main(void) {
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    printf("no device\n");
    return 2;
  }
  const mfsdp_param params[2] = {{256, 512, MFSDP_KIND_MATRIX, 0}, {640, 384, MFSDP_KIND_MATRIX, 0}};
  mfsdp_matrix_shard m[2];
  int32_t n_m = 0, n_t = 0;
  int64_t mat_elems[1], tail_elems[1];
  CHECK(mfsdp_plan_owners(params, 2, 1, 5, 128, m, &n_m, NULL, &n_t, mat_elems, tail_elems) == MFSDP_OK);
  CHECK(n_m == 2 && n_t == 0);
  const int64_t n = mat_elems[0];
  const size_t ws_bytes = mfsdp_muon_workspace_bytes(m, n_m);
  CHECK(ws_bytes > 0);

  uint16_t* g_host = (uint16_t*)calloc((size_t)n, sizeof(uint16_t));
  uint16_t* u_host = (uint16_t*)calloc((size_t)n, sizeof(uint16_t));
  uint16_t* u2_host = (uint16_t*)calloc((size_t)n, sizeof(uint16_t));
  CHECK(g_host && u_host && u2_host);
  uint32_t state = 12345u;   /* a fixed linear congruential sequence, values in (-1e-2, 1e-2) */
  for (int64_t i = 0; i < n; ++i) {
    state = state * 1664525u + 1013904223u;
    g_host[i] = float_to_bf16(((float)(state >> 8) / 16777216.0f - 0.5f) * 2e-2f);
  }
  void *g = NULL, *u = NULL, *u2 = NULL, *ws = NULL;
  float *mom = NULL, *mom2 = NULL;
  CHECK(cudaMalloc(&g, (size_t)n * 2) == cudaSuccess);
  CHECK(cudaMalloc(&u, (size_t)n * 2) == cudaSuccess);
  CHECK(cudaMalloc(&u2, (size_t)n * 2) == cudaSuccess);
  CHECK(cudaMalloc((void**)&mom, (size_t)n * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&mom2, (size_t)n * 4) == cudaSuccess);
  CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess);
  CHECK(cudaMemcpy(g, g_host, (size_t)n * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemset(mom, 0, (size_t)n * 4) == cudaSuccess);
  CHECK(cudaMemset(mom2, 0, (size_t)n * 4) == cudaSuccess);

  CHECK(mfsdp_muon_owner_step(m, n_m, g, MFSDP_DTYPE_BF16, mom, u, MFSDP_DTYPE_BF16, n, 0.95, 0, 5, 3.4445, -4.7750,
                              2.0315, 1e-7, ws, ws_bytes, NULL) == MFSDP_OK);
  int32_t detail = -1;
  CHECK(mfsdp_muon_device_status(ws, NULL, &detail) == MFSDP_OK);
  CHECK(mfsdp_muon_owner_step_static_scratch(m, n_m, g, MFSDP_DTYPE_BF16, mom2, u2, MFSDP_DTYPE_BF16, n, 0.95, 0, 5,
                                             3.4445, -4.7750, 2.0315, 1e-7, NULL) == MFSDP_OK);
  CHECK(mfsdp_muon_static_scratch_status(NULL, &detail) == MFSDP_OK);
  CHECK(cudaDeviceSynchronize() == cudaSuccess);
  CHECK(cudaMemcpy(u_host, u, (size_t)n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(u2_host, u2, (size_t)n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);

  for (int k = 0; k < n_m; ++k) {
    const int64_t cnt = m[k].rows * m[k].cols;
    const int64_t s = m[k].rows < m[k].cols ? m[k].rows : m[k].cols;
    double ss = 0.0;
    for (int64_t i = 0; i < cnt; ++i) {
      const float v = bf16_to_float(u_host[m[k].offset + i]);
      CHECK(isfinite(v));
      ss += (double)v * v;
    }
    const double r = sqrt(ss / (double)s);
    printf("matrix %d (%lld x %lld): ||O||_F / sqrt(s) = %.4f\n", k, (long long)m[k].rows, (long long)m[k].cols, r);
    CHECK(r >= 0.68 && r <= 1.14);
    CHECK(memcmp(u_host + m[k].offset, u2_host + m[k].offset, (size_t)cnt * 2) == 0);
  }
  cudaFree(g); cudaFree(u); cudaFree(u2); cudaFree(mom); cudaFree(mom2); cudaFree(ws);
  free(g_host); free(u_host); free(u2_host);
  printf("ok\n");
  return 0;
}
