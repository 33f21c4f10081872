/*
 * Plain-C use of the boundary (include/attn.h), no Python or torch: device
 * buffers from the CUDA runtime, bf16 inputs built on the host, then
 * attn_fwd / attn_bwd and two properties that hold exactly in exact
 * arithmetic (softmax rows sum to one):
 *   - V with every row equal to the same vector c gives O = c;
 *   - dO = 0 gives dQ = dK = dV = 0.
 * Exit status 0 when both hold (O within 1e-2, gradients exactly zero).
 * Built and run by tests/test_gpu_c_abi.py.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "attn.h"

static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest even */
  return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t lcg(uint32_t* s) {
  *s = *s * 1664525u + 1013904223u;
  return *s;
}

#define CHECK(x)                                                    \
  do {                                                              \
    if (!(x)) {                                                     \
      fprintf(stderr, "failed: %s (line %d)\n", #x, __LINE__);     \
      return 1;                                                     \
    }                                                               \
  } while (0)

int main(void) {
  const int B = 1, H = 2, N = 200, d = 64;
  const size_t n = (size_t)B * H * N * d, bytes = n * 2, lbytes = (size_t)B * H * N * 4;
  uint16_t *hq = malloc(bytes), *hk = malloc(bytes), *hv = malloc(bytes), *hz = calloc(n, 2), *ho = malloc(bytes);
  float* hl = malloc(lbytes);
  CHECK(hq && hk && hv && hz && ho && hl);
  uint32_t seed = 12345u;
  for (size_t i = 0; i < n; ++i) {
    hq[i] = to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 4.0f);
    hk[i] = to_bf16(((float)(lcg(&seed) >> 8) / 16777216.0f - 0.5f) * 4.0f);
    hv[i] = to_bf16(0.01f * (float)(i % d) - 0.3f); /* every row of V is the same vector c */
  }
  void *q, *k, *v, *o, *z, *dq, *dk, *dv;
  float* lse;
  CHECK(cudaMalloc(&q, bytes) == cudaSuccess && cudaMalloc(&k, bytes) == cudaSuccess &&
        cudaMalloc(&v, bytes) == cudaSuccess && cudaMalloc(&o, bytes) == cudaSuccess &&
        cudaMalloc(&z, bytes) == cudaSuccess && cudaMalloc(&dq, bytes) == cudaSuccess &&
        cudaMalloc(&dk, bytes) == cudaSuccess && cudaMalloc(&dv, bytes) == cudaSuccess &&
        cudaMalloc((void**)&lse, lbytes) == cudaSuccess);
  CHECK(cudaMemcpy(q, hq, bytes, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(k, hk, bytes, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(v, hv, bytes, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(z, hz, bytes, cudaMemcpyHostToDevice) == cudaSuccess);
  for (int causal = 0; causal < 2; ++causal) {
    CHECK(attn_fwd(q, k, v, o, lse, B, H, N, d, 0.125f, causal, NULL) == ATTN_OK);
    CHECK(attn_bwd(q, k, v, o, z, lse, dq, dk, dv, B, H, N, d, 0.125f, causal, NULL) == ATTN_OK);
    CHECK(attn_sync_status(NULL) == ATTN_OK);
    CHECK(cudaMemcpy(ho, o, bytes, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(hl, lse, lbytes, cudaMemcpyDeviceToHost) == cudaSuccess);
    double worst = 0.0;
    for (size_t i = 0; i < n; ++i) {
      const double e = fabs((double)from_bf16(ho[i]) - (double)from_bf16(hv[i]));
      if (e > worst) worst = e;
    }
    for (size_t r = 0; r < (size_t)B * H * N; ++r) CHECK(isfinite(hl[r]));
    printf("causal=%d max|O - c| = %g\n", causal, worst);
    CHECK(worst <= 1e-2);
    void* grads[3] = {dq, dk, dv};
    for (int g = 0; g < 3; ++g) {
      CHECK(cudaMemcpy(ho, grads[g], bytes, cudaMemcpyDeviceToHost) == cudaSuccess);
      for (size_t i = 0; i < n; ++i) CHECK(from_bf16(ho[i]) == 0.0f);
    }
  }
  CHECK(attn_fwd(q, k, v, o, lse, B, H, N, 48, 0.125f, 0, NULL) == ATTN_ERR_UNSUPPORTED);
  printf("ok\n");
  return 0;
}
