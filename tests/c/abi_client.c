/*
 * A plain C client of the library: includes the public header, links
 * libfa.so, and checks the host-side contract (version, status names,
 * workspace sizes, argument errors). With the argument "gpu" it also runs one
 * forward pass through fa_forward_ex on device buffers it allocates with the
 * CUDA runtime, and prints one output value and one LSE value, which the
 * calling test compares with the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fa.h"

/* CUDA runtime entry points used by the GPU part (declared here so that the
 * client needs no CUDA headers). */
extern int cudaMalloc(void **ptr, size_t size);
extern int cudaFree(void *ptr);
extern int cudaMemcpy(void *dst, const void *src, size_t count, int kind);
extern int cudaDeviceSynchronize(void);

#define CHECK(cond)                                             \
  do {                                                          \
    if (!(cond)) {                                              \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      return 1;                                                 \
    }                                                           \
  } while (0)

static uint16_t to_bf16(float x) { /* round to nearest even; inputs are finite */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

int main(int argc, char **argv) {
  CHECK(fa_abi_version() == 2);
  CHECK(strcmp(fa_status_string(FA_ERR_MISALIGNED), "FA_ERR_MISALIGNED") == 0);
  /* row statistics (2 x fp32 per padded row) + the one-pass form's fp32 dQ accumulator
     (the default form for d <= 128); statistics only at d = 256 (two-kernel form) */
  CHECK(fa_backward_workspace_bytes(2, 3, 200, 64) ==
        2 * (size_t)(2 * 3 * 256 * 4) + (size_t)(2 * 3 * 256 * 64 * 4));
  CHECK(fa_backward_min_workspace_bytes(2, 3, 200, 64) == 2 * (size_t)(2 * 3 * 256 * 4));
  CHECK(fa_backward_one_pass_workspace_bytes(2, 3, 200, 128) ==
        2 * (size_t)(2 * 3 * 256 * 4) + (size_t)(2 * 3 * 256 * 128 * 4));
  CHECK(fa_backward_workspace_bytes(2, 3, 200, 256) == 2 * (size_t)(2 * 3 * 256 * 4));
  CHECK(fa_forward(NULL, NULL, NULL, NULL, NULL, 1, 1, 0, 64, 0, 0.125f, NULL, NULL) == FA_OK);
  CHECK(fa_forward((void *)16, (void *)16, (void *)16, (void *)16, (float *)16, 1, 1, 128, 80,
                   0, 0.125f, NULL, NULL) == FA_ERR_UNSUPPORTED);
  fa_tensor t = {(void *)16, 0, 0, 60, FA_BF16, 0}; /* row stride of 120 bytes */
  fa_tensor good = {(void *)16, 0, 0, 64, FA_BF16, 0};
  CHECK(fa_forward_ex(&t, &good, &good, &good, (float *)16, 1, 1, 128, 128, 64, 0, 0.125f, NULL,
                      NULL) == FA_ERR_MISALIGNED);
  CHECK(fa_num_kernels() >= 4 && strcmp(fa_kernel_name(0), "fa_fwd_kernel") == 0);
  if (argc < 2 || strcmp(argv[1], "gpu") != 0) {
    printf("host checks passed\n");
    return 0;
  }

  /* one head, N = 130 (a partial second tile), d = 64, causal; Q, K, V are a
   * fixed pattern the test re-creates in Python */
  enum { N = 130, D = 64 };
  static uint16_t q[N * D], k[N * D], v[N * D], o[N * D];
  static float lse[N];
  for (int i = 0; i < N * D; ++i) {
    q[i] = to_bf16(0.01f * (float)((i * 7) % 23 - 11));
    k[i] = to_bf16(0.02f * (float)((i * 5) % 19 - 9));
    v[i] = to_bf16(0.05f * (float)((i * 3) % 17 - 8));
  }
  void *dq = NULL, *dk = NULL, *dv = NULL, *dout = NULL, *dlse = NULL;
  CHECK(cudaMalloc(&dq, sizeof q) == 0 && cudaMalloc(&dk, sizeof k) == 0 &&
        cudaMalloc(&dv, sizeof v) == 0 && cudaMalloc(&dout, sizeof o) == 0 &&
        cudaMalloc(&dlse, sizeof lse) == 0);
  CHECK(cudaMemcpy(dq, q, sizeof q, 1) == 0 && cudaMemcpy(dk, k, sizeof k, 1) == 0 &&
        cudaMemcpy(dv, v, sizeof v, 1) == 0);
  fa_tensor tq = {dq, 0, 0, D, FA_BF16, 0}, tk = {dk, 0, 0, D, FA_BF16, 0};
  fa_tensor tv = {dv, 0, 0, D, FA_BF16, 0}, to = {dout, 0, 0, D, FA_BF16, 0};
  const fa_status s = fa_forward_ex(&tq, &tk, &tv, &to, (float *)dlse, 1, 1, N, N, D, 1,
                                    0.125f, NULL, NULL);
  CHECK(s == FA_OK);
  CHECK(cudaDeviceSynchronize() == 0);
  unsigned int code = 1;
  CHECK(fa_device_status(NULL, &code) == FA_OK && code == 0);
  CHECK(cudaMemcpy(o, dout, sizeof o, 2) == 0 && cudaMemcpy(lse, dlse, sizeof lse, 2) == 0);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(dout);
  cudaFree(dlse);
  /* row 129 (the partial tile), column 5, and its LSE */
  printf("%.8e %.8e %.8e\n", from_bf16(o[129 * D + 5]), lse[129], lse[0]);
  return 0;
}
