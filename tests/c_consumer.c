/* A plain C consumer of include/mla.h: no Python, no PyTorch.  Built and run
 * by tests/test_c_consumer.py.
 *
 *   c_consumer host   host-side calls only (no GPU needed): version, status
 *                     strings, dimension checks, workspace sizes, argument
 *                     validation
 *   c_consumer gpu    one decode step through cudaMalloc'd buffers: append a
 *                     single token (no RoPE) and decode it.  With one cached
 *                     token the softmax weight is 1, so out_h = W^UV_h c_0
 *                     ("Beyond the Attention Bottleneck", "Down-Projection
 *                     and Up-Projection Mechanics": the value is the latent's
 *                     up-projection), checked against a double-precision sum
 *                     here.
 * Prints "OK" and exits 0 on success. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "mla.h"

#define CHECK(c)                                                         \
  do {                                                                   \
    if (!(c)) {                                                          \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c);    \
      return 1;                                                          \
    }                                                                    \
  } while (0)

static uint16_t to_bf16(float f) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static float lcg(uint32_t* s) { /* uniform in [-1, 1) */
  *s = *s * 1664525u + 1013904223u;
  return (float)((*s >> 8) & 0xFFFFFF) / 8388608.0f - 1.0f;
}

static int host_checks(void) {
  mla_dims d = {16, 512, 64, 128, 128, 64, MLA_CACHE_BF16};
  CHECK(mla_version() >= 100);
  CHECK(strcmp(mla_status_string(MLA_OK), "ok") == 0);
  CHECK(mla_check_dims(&d) == MLA_OK);
  mla_dims bad = d;
  bad.kv_lora_rank = 256;
  CHECK(mla_check_dims(&bad) == MLA_ERR_UNSUPPORTED);
  CHECK(mla_check_dims(NULL) == MLA_ERR_INVALID_ARG);
  CHECK(mla_decode_workspace_size(&d, 32, 76) > (size_t)(76 + 32) * 16 * 512 * 4);
  CHECK(mla_decode_multi_workspace_size(&d, 32, 2, 76) > mla_decode_workspace_size(&d, 32, 76));
  CHECK(mla_decode_sparse_workspace_size(&d, 32, 2048, 76) > (size_t)32 * 2048 * 1152);
  /* rejected on the host before anything runs: null queries */
  CHECK(mla_decode(&d, NULL, NULL, NULL, NULL, 1, NULL, 1, NULL, 1, NULL, NULL, 0.1f, 4, NULL, 0, NULL, NULL,
                   NULL) == MLA_ERR_INVALID_ARG);
  /* FP8 caches and prefill chunks through the same header */
  mla_dims d8 = d;
  d8.cache_dtype = MLA_CACHE_FP8;
  CHECK(mla_check_dims(&d8) == MLA_OK);
  CHECK(mla_prefill_workspace_size(&d, 4, 512, 3) > mla_decode_workspace_size(&d, 4, 3));
  CHECK(mla_prefill_workspace_size(&d, 4, MLA_MAX_PREFILL_CHUNK + 1, 3) == 0);
  CHECK(mla_prefill(&d8, NULL, NULL, 1, NULL, 1, NULL, 1, 8, NULL, NULL, 1e4, NULL, NULL, NULL, NULL, 0.1f, 3,
                    NULL, 0, NULL, NULL, NULL) == MLA_ERR_INVALID_ARG);
  return 0;
}

static int gpu_decode(void) {
  enum { H = 16, P = 64, NPG = 2 };
  mla_dims d = {H, 512, 64, 128, 128, P, MLA_CACHE_BF16};
  const size_t row = 576, nW = (size_t)H * 128 * 512;
  uint32_t seed = 12345;
  uint16_t *c_kv = malloc(512 * 2), *k_pe = malloc(64 * 2), *q_nope = malloc(H * 128 * 2), *q_pe = malloc(H * 64 * 2);
  uint16_t *wuk = malloc(nW * 2), *wuv = malloc(nW * 2), *out = malloc(H * 128 * 2);
  for (int i = 0; i < 512; ++i) c_kv[i] = to_bf16(lcg(&seed));
  for (int i = 0; i < 64; ++i) k_pe[i] = to_bf16(lcg(&seed));
  for (int i = 0; i < H * 128; ++i) q_nope[i] = to_bf16(lcg(&seed));
  for (int i = 0; i < H * 64; ++i) q_pe[i] = to_bf16(lcg(&seed));
  for (size_t i = 0; i < nW; ++i) wuk[i] = to_bf16(0.05f * lcg(&seed));
  for (size_t i = 0; i < nW; ++i) wuv[i] = to_bf16(0.05f * lcg(&seed));
  const int32_t table[NPG] = {1, 0}, lens[1] = {1}, ids[1] = {0}, pos[1] = {0};

  void *d_cache, *d_c, *d_k, *d_qn, *d_qp, *d_wuk, *d_wuv, *d_out, *d_ws;
  int32_t *d_table, *d_lens, *d_ids, *d_pos;
  const size_t ws_bytes = mla_decode_workspace_size(&d, 1, 4);
  CHECK(ws_bytes > 0);
  CHECK(cudaMalloc(&d_cache, (size_t)NPG * P * row * 2) == 0);
  CHECK(cudaMemset(d_cache, 0, (size_t)NPG * P * row * 2) == 0);
  CHECK(cudaMalloc(&d_c, 512 * 2) == 0 && cudaMalloc(&d_k, 64 * 2) == 0);
  CHECK(cudaMalloc(&d_qn, H * 128 * 2) == 0 && cudaMalloc(&d_qp, H * 64 * 2) == 0);
  CHECK(cudaMalloc(&d_wuk, nW * 2) == 0 && cudaMalloc(&d_wuv, nW * 2) == 0);
  CHECK(cudaMalloc(&d_out, H * 128 * 2) == 0 && cudaMalloc(&d_ws, ws_bytes) == 0);
  CHECK(cudaMalloc((void**)&d_table, sizeof table) == 0 && cudaMalloc((void**)&d_lens, 4) == 0);
  CHECK(cudaMalloc((void**)&d_ids, 4) == 0 && cudaMalloc((void**)&d_pos, 4) == 0);
  CHECK(cudaMemcpy(d_c, c_kv, 512 * 2, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_k, k_pe, 64 * 2, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_qn, q_nope, H * 128 * 2, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_qp, q_pe, H * 64 * 2, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_wuk, wuk, nW * 2, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_wuv, wuv, nW * 2, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_table, table, sizeof table, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_lens, lens, 4, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_ids, ids, 4, cudaMemcpyHostToDevice) == 0);
  CHECK(cudaMemcpy(d_pos, pos, 4, cudaMemcpyHostToDevice) == 0);

  CHECK(mla_cache_append(&d, d_cache, NULL, NPG, d_table, 1, NPG, d_ids, d_pos, 1, d_c, d_k, 0.0, NULL, NULL) ==
        MLA_OK);
  CHECK(mla_decode(&d, d_qn, d_qp, d_cache, NULL, NPG, d_table, NPG, d_lens, 1, d_wuk, d_wuv, 0.0721f, 4, d_ws,
                   ws_bytes, d_out, NULL, NULL) == MLA_OK);
  int32_t status = -99;
  CHECK(mla_read_device_status(d_ws, &status, NULL) == MLA_OK && status == MLA_OK);
  CHECK(cudaMemcpy(out, d_out, H * 128 * 2, cudaMemcpyDeviceToHost) == 0);
  double worst = 0.0;
  for (int h = 0; h < H; ++h) {
    double ref_max = 0.0, err_max = 0.0;
    for (int j = 0; j < 128; ++j) {
      double ref = 0.0;
      for (int m = 0; m < 512; ++m) ref += from_bf16(wuv[((size_t)h * 128 + j) * 512 + m]) * from_bf16(c_kv[m]);
      const double err = fabs(from_bf16(out[h * 128 + j]) - ref);
      if (fabs(ref) > ref_max) ref_max = fabs(ref);
      if (err > err_max) err_max = err;
    }
    CHECK(err_max <= 2e-2 && err_max <= 1e-2 * ref_max);
    if (err_max > worst) worst = err_max;
  }
  printf("max abs error %.3g\n", worst);
  return 0;
}

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  int rc = host_checks();
  if (rc == 0 && strcmp(argv[1], "gpu") == 0) rc = gpu_decode();
  if (rc == 0) printf("OK\n");
  return rc;
}
