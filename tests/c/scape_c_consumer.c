/*
 * A plain C99 user of libscape: it includes only include/scape.h, links only
 * libscape.so and passes host pointers, so the C ABI is exercised without
 * Python, ctypes or torch in between.
 *
 *   scape_c_consumer args
 *       argument errors come back as SCAPE_EINVAL with a message, before any
 *       CUDA work (runs without a GPU);
 *   scape_c_consumer run N W chunk density steps dir
 *       reads dir/theta.bin (N fp32) and dir/grads.bin (steps x W x N bf16),
 *       takes the steps through scape_step_host on a new handle (step 0
 *       builds the first mask), checks that every chunk of M_t carries
 *       exactly floor(density * len) bits and that the compact coordinate
 *       list is strictly increasing, and writes dir/out_theta.bin,
 *       dir/out_mask.bin and dir/out_bbar.bin.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include "scape.h"

static int fails = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    fprintf(stderr, "FAILED: %s\n", what);
    fails++;
  }
}

static int run_args(void) {
  uint64_t numel[1] = {1024};
  scape_layout lay = {1, numel, 1024};
  scape_handle* h = (scape_handle*)1;
  expect(scape_create(&lay, 0, 0.1, 0.9f, 0.95f, 1e-3f, 0.1f, 1e-8f, &h) == SCAPE_EINVAL, "W = 0");
  expect(h == NULL, "handle cleared on failure");
  expect(strstr(scape_last_error(NULL), "W=") != NULL, "message names W");
  expect(scape_create(&lay, 2, 1.5, 0.9f, 0.95f, 1e-3f, 0.1f, 1e-8f, &h) == SCAPE_EINVAL,
         "density above 1");
  lay.chunk = 48;
  expect(scape_create(&lay, 2, 0.1, 0.9f, 0.95f, 1e-3f, 0.1f, 1e-8f, &h) == SCAPE_EINVAL,
         "chunk not a multiple of 32");
  expect(scape_step(NULL, NULL, NULL) == SCAPE_EINVAL, "step on NULL handle");
  scape_destroy(NULL);
  if (!fails) printf("args ok\n");
  return fails ? 1 : 0;
}

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* p = malloc(bytes);
  size_t got = p ? fread(p, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static int write_file(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return -1;
  size_t put = fwrite(p, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : -1;
}

static int popcount32(uint32_t x) {
  int n = 0;
  while (x) {
    x &= x - 1u;
    n++;
  }
  return n;
}

static int run_steps(uint64_t N, int W, uint32_t C, double density, int steps, const char* dir) {
  float* theta = (float*)read_file(dir, "theta.bin", N * sizeof(float));
  uint16_t* grads = (uint16_t*)read_file(dir, "grads.bin", (size_t)steps * W * N * 2);
  if (!theta || !grads) {
    fprintf(stderr, "missing inputs in %s\n", dir);
    return 2;
  }
  uint64_t numel[1] = {N};
  scape_layout lay = {1, numel, C};
  scape_handle* h = NULL;
  if (scape_create(&lay, W, density, 0.9f, 0.95f, 1e-3f, 0.1f, 1e-8f, &h) != SCAPE_OK) {
    fprintf(stderr, "scape_create: %s\n", scape_last_error(NULL));
    return 2;
  }
  expect(scape_load_state(h, SCAPE_THETA, 0, theta, 0, N) == SCAPE_OK, "load theta");
  const void** gp = (const void**)malloc(sizeof(void*) * (size_t)W);
  for (int t = 0; t < steps; t++) {
    for (int w = 0; w < W; w++) gp[w] = grads + ((size_t)t * W + w) * N;
    if (scape_step_host(h, gp, NULL) != SCAPE_OK) {
      fprintf(stderr, "scape_step_host: %s\n", scape_last_error(h));
      return 2;
    }
  }
  scape_info_t inf;
  expect(scape_info(h, &inf) == SCAPE_OK, "info");
  expect(inf.step == steps, "step count");
  uint32_t* mask = (uint32_t*)calloc(inf.mask_words, 4);
  expect(scape_mask(h, mask) == SCAPE_OK, "mask");
  for (uint64_t c = 0; c < inf.n_chunks; c++) {  /* exactly k_c bits per chunk */
    const uint64_t c0 = c * C, len = (N - c0) < C ? (N - c0) : C;
    const uint64_t k = (uint64_t)floor(density * (double)len);
    uint64_t bits = 0;
    for (uint64_t j = c0 / 32; j < (c0 + len + 31) / 32; j++) bits += (uint64_t)popcount32(mask[j]);
    expect(bits == k, "k_c bits in a chunk");
  }
  float* out = (float*)malloc(N * sizeof(float));
  expect(scape_read_state(h, SCAPE_THETA, 0, out, 0, N) == SCAPE_OK, "read theta");
  uint64_t K = 0;
  expect(scape_read_sparse(h, -1, NULL, NULL, 0, 0, &K) == SCAPE_OK, "sparse total");
  expect(K == inf.K, "K");
  uint32_t* idx = (uint32_t*)malloc(K * 4 + 4);
  float* bbar = (float*)malloc(K * 4 + 4);
  expect(scape_read_sparse(h, -1, idx, bbar, 0, K, NULL) == SCAPE_OK, "sparse");
  for (uint64_t r = 1; r < K; r++) expect(idx[r] > idx[r - 1], "coordinates ascending");
  expect(write_file(dir, "out_theta.bin", out, N * sizeof(float)) == 0, "write theta");
  expect(write_file(dir, "out_mask.bin", mask, inf.mask_words * 4) == 0, "write mask");
  expect(write_file(dir, "out_bbar.bin", bbar, K * 4) == 0, "write bbar");
  scape_destroy(h);
  free(theta); free(grads); free(gp); free(mask); free(out); free(idx); free(bbar);
  if (!fails) printf("run ok: N=%llu W=%d K=%llu steps=%d\n", (unsigned long long)N, W,
                     (unsigned long long)K, steps);
  return fails ? 1 : 0;
}

int main(int argc, char** argv) {
  if (argc >= 2 && strcmp(argv[1], "args") == 0) return run_args();
  if (argc == 8 && strcmp(argv[1], "run") == 0)
    return run_steps(strtoull(argv[2], NULL, 10), atoi(argv[3]), (uint32_t)strtoul(argv[4], NULL, 10),
                     atof(argv[5]), atoi(argv[6]), argv[7]);
  fprintf(stderr, "usage: %s args | run N W chunk density steps dir\n", argv[0]);
  return 2;
}
