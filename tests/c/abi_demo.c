/*
 * The C ABI used from plain C (no Python, no torch): test infrastructure.
 *   abi_demo host  - host-only calls: layout of the tiny MLP unit, the 7B/8-GPU
 *                    accountant example, status strings, a rejected argument.
 *   abi_demo gpu   - a fused shard step (W = 4, all ranks, 3 steps) on buffers
 *                    from cudaMalloc, then a fourth step through the one-launch
 *                    unfused calls (every rank's reduce-scatter, every shard's
 *                    Adam), each checked bit for bit against the C oracle.
 * Exit status 0 on success.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fsdp.h"

/* the oracle's entry points (oracle/fsdp_oracle.c) */
int ora_shard_step(const uint16_t *const *grads, int32_t world_size, int32_t shard_factor,
                   int64_t padded_numel, int32_t rank_begin, int32_t rank_end, float *const *master,
                   float *const *exp_avg, float *const *exp_avg_sq, const uint16_t *const *other_shards,
                   uint16_t *const *full_out, double lr, double beta1, double beta2, double eps, int64_t step);
int ora_reduce_scatter(const uint16_t *const *grads, int32_t world_size, int32_t shard_factor, int64_t padded_numel,
                       int32_t rank, float *out);
void ora_adam(float *param, float *exp_avg, float *exp_avg_sq, const float *grad, int64_t n, double lr, double beta1,
              double beta2, double eps, int64_t step, uint16_t *bf16_out);

#define CHECK(c, msg)                                   \
  do {                                                  \
    if (!(c)) {                                         \
      fprintf(stderr, "abi_demo: %s (line %d)\n", msg, __LINE__); \
      return 1;                                         \
    }                                                   \
  } while (0)

static int host_checks(void) {
  const int64_t numels[4] = {64 * 32, 32, 32 * 16, 16};
  int64_t offs[5];
  fsdp_layout_t lay;
  CHECK(fsdp_flatten_layout(numels, 4, 4, 4, offs, &lay) == FSDP_OK, "layout");
  CHECK(offs[1] == 2048 && offs[2] == 2080 && offs[3] == 2592 && offs[4] == 2608, "offsets");
  CHECK(lay.padded_numel == 2608 && lay.shard_numel == 652, "padded / shard");
  fsdp_account_t a;
  CHECK(fsdp_account(7e9, 0.22e9, 8, 8, 1, &a) == FSDP_OK, "account");
  CHECK(a.persistent_bytes == 14e9 && a.ddp_persistent_bytes == 112e9, "persistent");
  CHECK(a.comm_bytes == 42e9 && a.ddp_comm_bytes == 28e9, "communication");
  CHECK(fsdp_flatten_layout(numels, 4, 8, 3, offs, &lay) == FSDP_EINVAL, "W=8 F=3 rejected");
  CHECK(strcmp(fsdp_status_string(FSDP_OK), "ok") == 0, "status string");
  return 0;
}

static uint32_t lcg(uint32_t *s) {
  *s = *s * 1664525u + 1013904223u;
  return *s;
}

static float uniform_pm(uint32_t *s, float scale) { /* in [-scale, scale) */
  return ((float)(lcg(s) >> 8) * (1.0f / 16777216.0f) * 2.0f - 1.0f) * scale;
}

static uint16_t bf16_trunc(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  return (uint16_t)(u >> 16);
}

static int gpu_checks(void) {
  enum { W = 4 };
  const int64_t numels[4] = {64 * 32, 32, 32 * 16, 16};
  int64_t offs[5];
  fsdp_layout_t lay;
  CHECK(fsdp_flatten_layout(numels, 4, W, W, offs, &lay) == FSDP_OK, "layout");
  const int64_t P = lay.padded_numel, S = lay.shard_numel;
  uint32_t seed = 12345u;
  uint16_t *hg[W];
  float *hm[W], *he[W], *hv[W];
  uint16_t *hfull = calloc((size_t)P, 2), *dev_full_copy = calloc((size_t)P, 2);
  for (int r = 0; r < W; ++r) {
    hg[r] = malloc((size_t)P * 2);
    hm[r] = malloc((size_t)S * 4);
    he[r] = calloc((size_t)S, 4);
    hv[r] = calloc((size_t)S, 4);
    for (int64_t j = 0; j < S; ++j) hm[r][j] = uniform_pm(&seed, 0.05f);
  }
  uint16_t *dg[W], *dfull;
  float *dm[W], *de[W], *dv[W];
  CHECK(cudaMalloc((void **)&dfull, (size_t)P * 2) == cudaSuccess, "cudaMalloc");
  for (int r = 0; r < W; ++r) {
    CHECK(cudaMalloc((void **)&dg[r], (size_t)P * 2) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void **)&dm[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void **)&de[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void **)&dv[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    cudaMemcpy(dm[r], hm[r], (size_t)S * 4, cudaMemcpyHostToDevice);
    cudaMemset(de[r], 0, (size_t)S * 4);
    cudaMemset(dv[r], 0, (size_t)S * 4);
  }
  fsdp_adam_t adam = {1e-3, 0.9, 0.999, 1e-8, 0.0, 1};
  for (int64_t t = 1; t <= 3; ++t) {
    for (int r = 0; r < W; ++r) {
      for (int64_t j = 0; j < P; ++j) hg[r][j] = bf16_trunc(uniform_pm(&seed, 1e-2f));
      cudaMemcpy(dg[r], hg[r], (size_t)P * 2, cudaMemcpyHostToDevice);
    }
    adam.step = t;
    const uint16_t *const *grads = (const uint16_t *const *)dg;
    CHECK(fsdp_shard_step(grads, &lay, 0, W, dm, de, dv, NULL, &dfull, &adam, 0) == FSDP_OK, "shard step");
    CHECK(ora_shard_step((const uint16_t *const *)hg, W, W, P, 0, W, hm, he, hv, NULL, &hfull, 1e-3, 0.9,
                         0.999, 1e-8, t) == 0, "oracle step");
  }
  CHECK(cudaDeviceSynchronize() == cudaSuccess, "device sync");
  float *tmp = malloc((size_t)S * 4);
  for (int r = 0; r < W; ++r) {
    cudaMemcpy(tmp, dm[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(tmp, hm[r], (size_t)S * 4) == 0, "master differs from the oracle");
    cudaMemcpy(tmp, de[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(tmp, he[r], (size_t)S * 4) == 0, "exp_avg differs from the oracle");
    cudaMemcpy(tmp, dv[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(tmp, hv[r], (size_t)S * 4) == 0, "exp_avg_sq differs from the oracle");
  }
  cudaMemcpy(dev_full_copy, dfull, (size_t)P * 2, cudaMemcpyDeviceToHost);
  CHECK(memcmp(dev_full_copy, hfull, (size_t)P * 2) == 0, "full bf16 differs from the oracle");

  /* step 4 through the unfused calls: one launch reduces every rank's slice, one launch
     updates every rank's shard (with its bf16 cast) */
  float *dgs[W], *hgs = malloc((size_t)S * 4);
  uint16_t *dbf[W], *hbf = malloc((size_t)S * 2), *obf = malloc((size_t)S * 2);
  for (int r = 0; r < W; ++r) {
    CHECK(cudaMalloc((void **)&dgs[r], (size_t)S * 4) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc((void **)&dbf[r], (size_t)S * 2) == cudaSuccess, "cudaMalloc");
    for (int64_t j = 0; j < P; ++j) hg[r][j] = bf16_trunc(uniform_pm(&seed, 1e-2f));
    cudaMemcpy(dg[r], hg[r], (size_t)P * 2, cudaMemcpyHostToDevice);
  }
  adam.step = 4;
  CHECK(fsdp_reduce_scatter_ranks((const uint16_t *const *)dg, &lay, 0, W, dgs, 0) == FSDP_OK, "reduce-scatter ranks");
  fsdp_adam_shard_t shards[W];
  for (int r = 0; r < W; ++r) {
    shards[r].master = dm[r];
    shards[r].exp_avg = de[r];
    shards[r].exp_avg_sq = dv[r];
    shards[r].grad_shard = dgs[r];
    shards[r].bf16_shard_out = dbf[r];
    shards[r].n = S;
  }
  CHECK(fsdp_adam_shard_step_grouped(shards, W, &adam, 0) == FSDP_OK, "grouped Adam");
  CHECK(cudaDeviceSynchronize() == cudaSuccess, "device sync");
  for (int r = 0; r < W; ++r) {
    CHECK(ora_reduce_scatter((const uint16_t *const *)hg, W, W, P, r, hgs) == 0, "oracle reduce-scatter");
    cudaMemcpy(tmp, dgs[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(tmp, hgs, (size_t)S * 4) == 0, "reduce-scatter of a rank differs from the oracle");
    ora_adam(hm[r], he[r], hv[r], hgs, S, 1e-3, 0.9, 0.999, 1e-8, 4, obf);
    cudaMemcpy(tmp, dm[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(tmp, hm[r], (size_t)S * 4) == 0, "grouped Adam master differs from the oracle");
    cudaMemcpy(tmp, de[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(tmp, he[r], (size_t)S * 4) == 0, "grouped Adam exp_avg differs from the oracle");
    cudaMemcpy(tmp, dv[r], (size_t)S * 4, cudaMemcpyDeviceToHost);
    CHECK(memcmp(tmp, hv[r], (size_t)S * 4) == 0, "grouped Adam exp_avg_sq differs from the oracle");
    cudaMemcpy(hbf, dbf[r], (size_t)S * 2, cudaMemcpyDeviceToHost);
    CHECK(memcmp(hbf, obf, (size_t)S * 2) == 0, "grouped Adam bf16 differs from the oracle");
  }
  printf("abi_demo: 3 fused steps and 1 unfused step from C match the oracle bit for bit\n");
  return 0;
}

int main(int argc, char **argv) {
  if (argc < 2) return 2;
  if (strcmp(argv[1], "host") == 0) return host_checks();
  if (strcmp(argv[1], "gpu") == 0) return host_checks() || gpu_checks();
  return 2;
}
