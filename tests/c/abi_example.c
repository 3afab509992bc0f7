/*
 * A plain C99 caller of the library: device buffers from the CUDA runtime,
 * one b2g_sgemm call on small-integer operands (every product and sum exact
 * in FP32, so the result must equal the integer reference bit for bit), the
 * same call through b2g_sgemm_host on host buffers, and an error code for a
 * bad leading dimension.  Prints "ok" and returns 0 on success.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "b2g_sgemm.h"

#define M 300
#define N 260
#define K 170

static int fail(const char* what, int rc) {
  fprintf(stderr, "%s: %d %s\n", what, rc, b2g_strerror(rc));
  return 1;
}

static int cuda_fail(const char* what, cudaError_t e) {
  fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
  return 1;
}

int main(void) {
  static float A[M * K], B[K * N], C[M * N], out[M * N], ref[M * N];
  for (int i = 0; i < M * K; ++i) A[i] = (float)((i * 7) % 13 - 6);
  for (int i = 0; i < K * N; ++i) B[i] = (float)((i * 5) % 11 - 5);
  for (int i = 0; i < M * N; ++i) C[i] = (float)(i % 9 - 4);
  for (int i = 0; i < M; ++i)
    for (int j = 0; j < N; ++j) {
      long long s = 0;
      for (int k = 0; k < K; ++k) s += (long long)A[i * K + k] * (long long)B[k * N + j];
      ref[i * N + j] = (float)(2 * s - (long long)C[i * N + j]);
    }

  float *dA = NULL, *dB = NULL, *dC = NULL;
  cudaError_t e = cudaMalloc((void**)&dA, sizeof A);
  if (e == cudaSuccess) e = cudaMalloc((void**)&dB, sizeof B);
  if (e == cudaSuccess) e = cudaMalloc((void**)&dC, sizeof C);
  if (e != cudaSuccess) return cuda_fail("cudaMalloc", e);
  cudaMemcpy(dA, A, sizeof A, cudaMemcpyHostToDevice);
  cudaMemcpy(dB, B, sizeof B, cudaMemcpyHostToDevice);
  cudaMemcpy(dC, C, sizeof C, cudaMemcpyHostToDevice);

  int rc = b2g_sgemm(M, N, K, 2.0f, dA, K, dB, N, -1.0f, dC, N, NULL);
  if (rc) return fail("b2g_sgemm", rc);
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail("cudaDeviceSynchronize", e);
  cudaMemcpy(out, dC, sizeof out, cudaMemcpyDeviceToHost);
  if (memcmp(out, ref, sizeof out) != 0) {
    fprintf(stderr, "b2g_sgemm result differs from the integer reference\n");
    return 1;
  }

  memcpy(out, C, sizeof out);  /* host operands, same call */
  rc = b2g_sgemm_host(M, N, K, 2.0f, A, K, B, N, -1.0f, out, N, NULL);
  if (rc) return fail("b2g_sgemm_host", rc);
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail("cudaDeviceSynchronize", e);
  if (memcmp(out, ref, sizeof out) != 0) {
    fprintf(stderr, "b2g_sgemm_host result differs from the integer reference\n");
    return 1;
  }

  rc = b2g_sgemm(M, N, K, 1.0f, dA, K - 1, dB, N, 0.0f, dC, N, NULL);
  if (rc != B2G_ERR_INVALID_LD) return fail("lda < K not refused", rc);

  cudaFree(dA);
  cudaFree(dB);
  cudaFree(dC);
  printf("ok %s\n", b2g_version());
  return 0;
}
