/*
 * A plain-C client of the library: no Python, no PyTorch.  It draws
 * deterministic bf16 inputs, runs dualkv_fwd and dualkv_bwd (deterministic
 * mode) through include/dualkv.h with cudaMalloc'd buffers, and writes the
 * inputs and every output to <dir>/<name>.bin so that a test can compare them
 * with the Python binding's results on the same inputs.
 *
 * usage: abi_client <dir>
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "dualkv.h"

static uint32_t rng_state = 12345u;

/* xorshift32, then a value in [-2, 2) rounded to bf16 by truncation of an exact float */
static uint16_t next_bf16(void) {
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 17;
  rng_state ^= rng_state << 5;
  float f = ((float)(rng_state >> 8) / 16777216.0f) * 4.0f - 2.0f;
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return (uint16_t)(bits >> 16);
}

static int write_file(const char* dir, const char* name, const void* p, size_t n) {
  char path[1024];
  snprintf(path, sizeof(path), "%s/%s.bin", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  size_t w = fwrite(p, 1, n, f);
  fclose(f);
  return w != n;
}

#define CK(x)                                                        \
  do {                                                               \
    cudaError_t e_ = (x);                                            \
    if (e_ != cudaSuccess) {                                         \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));       \
      return 2;                                                      \
    }                                                                \
  } while (0)

int main(int argc, char** argv) {
  if (argc < 2) return 1;
  const char* dir = argv[1];
  const int64_t P = 200;
  const int32_t N = 3, R[3] = {150, 0, 131}, Hq = 4, Hkv = 2, d = 128;
  const int64_t T = P + R[0] + R[1] + R[2];
  const float scale = 0.08838834764831845f; /* 1/sqrt(128) */
  const size_t nq = (size_t)T * Hq * d, nk = (size_t)T * Hkv * d;

  uint16_t *hq = malloc(nq * 2), *hk = malloc(nk * 2), *hv = malloc(nk * 2), *hdo = malloc(nq * 2);
  uint16_t *hout = malloc(nq * 2), *hdq = malloc(nq * 2), *hdk = malloc(nk * 2), *hdv = malloc(nk * 2);
  float* hlse = malloc((size_t)Hq * T * 4);
  if (!hq || !hk || !hv || !hdo || !hout || !hdq || !hdk || !hdv || !hlse) return 1;
  for (size_t i = 0; i < nq; ++i) hq[i] = next_bf16();
  for (size_t i = 0; i < nk; ++i) hk[i] = next_bf16();
  for (size_t i = 0; i < nk; ++i) hv[i] = next_bf16();
  for (size_t i = 0; i < nq; ++i) hdo[i] = next_bf16();

  void *q, *k, *v, *dout, *out, *dq, *dk, *dv, *ws;
  float* lse;
  CK(cudaMalloc(&q, nq * 2));
  CK(cudaMalloc(&k, nk * 2));
  CK(cudaMalloc(&v, nk * 2));
  CK(cudaMalloc(&dout, nq * 2));
  CK(cudaMalloc(&out, nq * 2));
  CK(cudaMalloc(&dq, nq * 2));
  CK(cudaMalloc(&dk, nk * 2));
  CK(cudaMalloc(&dv, nk * 2));
  CK(cudaMalloc((void**)&lse, (size_t)Hq * T * 4));
  const size_t ws_bytes = dualkv_bwd_workspace_bytes(P, N, R, Hq, Hkv, d, 1, 2);
  if (ws_bytes == 0) return 3;
  CK(cudaMalloc(&ws, ws_bytes));
  CK(cudaMemcpy(q, hq, nq * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(k, hk, nk * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(v, hv, nk * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dout, hdo, nq * 2, cudaMemcpyHostToDevice));

  int st = dualkv_fwd(q, k, v, P, N, R, Hq, Hkv, d, scale, out, lse, NULL);
  if (st != DUALKV_OK) {
    fprintf(stderr, "dualkv_fwd: %s\n", dualkv_status_string(st));
    return 4;
  }
  st = dualkv_bwd(q, k, v, out, dout, lse, P, N, R, Hq, Hkv, d, scale, 1, 2, ws, ws_bytes, dq, dk, dv, NULL);
  if (st != DUALKV_OK) {
    fprintf(stderr, "dualkv_bwd: %s\n", dualkv_status_string(st));
    return 5;
  }
  int32_t site = 0;
  st = dualkv_last_device_error(NULL, &site);
  if (st != DUALKV_OK) {
    fprintf(stderr, "device error %d at site %d\n", st, site);
    return 6;
  }
  CK(cudaMemcpy(hout, out, nq * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hlse, lse, (size_t)Hq * T * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hdq, dq, nq * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hdk, dk, nk * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hdv, dv, nk * 2, cudaMemcpyDeviceToHost));

  int bad = 0;
  bad |= write_file(dir, "q", hq, nq * 2) | write_file(dir, "k", hk, nk * 2) | write_file(dir, "v", hv, nk * 2);
  bad |= write_file(dir, "dout", hdo, nq * 2) | write_file(dir, "out", hout, nq * 2);
  bad |= write_file(dir, "lse", hlse, (size_t)Hq * T * 4) | write_file(dir, "dq", hdq, nq * 2);
  bad |= write_file(dir, "dk", hdk, nk * 2) | write_file(dir, "dv", hdv, nk * 2);
  printf("abi_client ok T=%lld version=%d\n", (long long)T, dualkv_version());
  return bad ? 7 : 0;
}
