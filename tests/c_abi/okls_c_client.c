/*
 * A client of libokls.so written in plain C: no Python, no PyTorch.  It owns
 * its device memory through the CUDA runtime, drives the C ABI declared in
 * okls.h, and writes the parameters after `steps` steps to a file.
 *
 *   okls_c_client METHOD B M N STEPS G.bin W.out
 *
 * METHOD is an okls_method value (0 OKLS, 1 Shampoo, 2 SOAP); G.bin holds
 * STEPS x B x M x N fp32 gradients (one batch per step), W starts at zero.
 * Exit status 0 on success; every failing call prints okls_last_error().
 */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "okls.h"

static int check(okls_status s, const char* what) {
  if (s != OKLS_OK) {
    fprintf(stderr, "%s failed (%d): %s\n", what, (int)s, okls_last_error());
    return 1;
  }
  return 0;
}

static int check_cuda(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "%s failed: %s\n", what, cudaGetErrorString(e));
    return 1;
  }
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: %s METHOD B M N STEPS G.bin W.out\n", argv[0]);
    return 2;
  }
  const int method = atoi(argv[1]);
  const long long B = atoll(argv[2]), M = atoll(argv[3]), N = atoll(argv[4]);
  const int steps = atoi(argv[5]);
  const size_t elems = (size_t)(B * M * N);
  if (okls_abi_version() != OKLS_ABI_VERSION) {
    fprintf(stderr, "ABI version %d, header %d\n", okls_abi_version(), OKLS_ABI_VERSION);
    return 1;
  }
  float* hostG = (float*)malloc(elems * sizeof(float) * (size_t)steps);
  float* hostW = (float*)malloc(elems * sizeof(float));
  FILE* f = fopen(argv[6], "rb");
  if (!hostG || !hostW || !f || fread(hostG, sizeof(float), elems * (size_t)steps, f) != elems * (size_t)steps) {
    fprintf(stderr, "cannot read %s\n", argv[6]);
    return 1;
  }
  fclose(f);

  okls_config cfg;
  if (check(okls_config_default(&cfg, B, M, N), "okls_config_default")) return 1;
  cfg.method = method;
  if (method == OKLS_METHOD_SOAP) {
    cfg.beta1 = 0.95f;
    cfg.beta2 = 0.95f;
    cfg.eps = 1e-8f;
    cfg.weight_decay = 0.0f;
    cfg.root_every = 2;
  }
  size_t state_bytes = 0, ws_bytes = 0;
  if (check(okls_state_bytes(&cfg, &state_bytes, &ws_bytes), "okls_state_bytes")) return 1;
  void *state = NULL, *ws = NULL, *W = NULL, *G = NULL;
  cudaStream_t st;
  if (check_cuda(cudaStreamCreate(&st), "cudaStreamCreate") || check_cuda(cudaMalloc(&state, state_bytes), "state") ||
      check_cuda(cudaMalloc(&ws, ws_bytes), "workspace") || check_cuda(cudaMalloc(&W, elems * 4), "W") ||
      check_cuda(cudaMalloc(&G, elems * 4), "G") || check_cuda(cudaMemset(W, 0, elems * 4), "memset W"))
    return 1;
  okls_handle h = NULL;
  if (check(okls_create(&cfg, state, state_bytes, ws, ws_bytes, &h), "okls_create")) return 1;
  if (check(okls_reset_state(h, st), "okls_reset_state")) return 1;
  for (int t = 0; t < steps; ++t) {
    if (check_cuda(cudaMemcpyAsync(G, hostG + (size_t)t * elems, elems * 4, cudaMemcpyHostToDevice, st), "copy G"))
      return 1;
    if (check(okls_step(h, W, G, cfg.lr_peak, st), "okls_step")) return 1;
  }
  uint32_t dev = 0;
  if (check(okls_query_status(h, st, &dev), "okls_query_status")) return 1;
  int64_t t_done = 0;
  if (check(okls_get_step(h, &t_done), "okls_get_step") || t_done != steps) return 1;
  if (check_cuda(cudaMemcpy(hostW, W, elems * 4, cudaMemcpyDeviceToHost), "copy W")) return 1;
  if (check(okls_destroy(h), "okls_destroy")) return 1;
  cudaFree(G);
  cudaFree(W);
  cudaFree(ws);
  cudaFree(state);
  cudaStreamDestroy(st);
  f = fopen(argv[7], "wb");
  if (!f || fwrite(hostW, sizeof(float), elems, f) != elems) {
    fprintf(stderr, "cannot write %s\n", argv[7]);
    return 1;
  }
  fclose(f);
  free(hostG);
  free(hostW);
  printf("ok %d steps, status 0x%x\n", steps, dev);
  return 0;
}
