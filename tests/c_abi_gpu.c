/* A plain C user of the library on the GPU: reads bf16 H [T, Hd], bf16 W [V, Hd]
 * and int64 targets [T] from raw files, runs flce_forward (mean) and
 * flce_backward (dloss = 1) through the C ABI with cudaMalloc'd buffers, and
 * writes lse [T] fp32, logp [T] fp32, loss fp32, dH [T, Hd] bf16 and
 * dW [V, Hd] fp32 to raw files.
 * usage: c_abi_gpu DIR T Hd V */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "flce.h"

#define CK(x)                                                                 \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                \
      return 2;                                                               \
    }                                                                         \
  } while (0)
#define FL(x)                                                                 \
  do {                                                                        \
    flce_status s_ = (x);                                                     \
    if (s_ != FLCE_OK) {                                                      \
      fprintf(stderr, "%s: %s %s\n", #x, flce_status_string(s_), flce_last_error()); \
      return 3;                                                               \
    }                                                                         \
  } while (0)

static void* slurp(const char* dir, const char* name, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* p = malloc(bytes ? bytes : 1);
  size_t got = fread(p, 1, bytes, f);
  fclose(f);
  if (got != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static int spill(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(p, 1, bytes, f);
  fclose(f);
  return put != bytes;
}

int main(int argc, char** argv) {
  if (argc != 5) return 1;
  const char* dir = argv[1];
  const int64_t T = atoll(argv[2]), Hd = atoll(argv[3]), V = atoll(argv[4]);
  const size_t hb = (size_t)(T * Hd * 2), wb = (size_t)(V * Hd * 2), yb = (size_t)(T * 8);
  void* H_h = slurp(dir, "H.bin", hb);
  void* W_h = slurp(dir, "W.bin", wb);
  void* y_h = slurp(dir, "y.bin", yb);
  if (!H_h || !W_h || !y_h) return 4;
  void *H, *W, *y, *lse, *logp, *loss, *nv, *dH, *dW, *dl, *fws, *bws;
  const size_t fwsb = flce_forward_workspace_size(T, Hd, V), bwsb = flce_backward_workspace_size(T, Hd, V);
  CK(cudaMalloc(&H, hb));
  CK(cudaMalloc(&W, wb));
  CK(cudaMalloc(&y, yb));
  CK(cudaMalloc(&lse, (size_t)T * 4));
  CK(cudaMalloc(&logp, (size_t)T * 4));
  CK(cudaMalloc(&loss, 4));
  CK(cudaMalloc(&nv, 8));
  CK(cudaMalloc(&dH, hb));
  CK(cudaMalloc(&dW, (size_t)(V * Hd * 4)));
  CK(cudaMalloc(&dl, 4));
  CK(cudaMalloc(&fws, fwsb));
  CK(cudaMalloc(&bws, bwsb));
  CK(cudaMemcpy(H, H_h, hb, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(W, W_h, wb, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(y, y_h, yb, cudaMemcpyHostToDevice));
  const float one = 1.0f;
  CK(cudaMemcpy(dl, &one, 4, cudaMemcpyHostToDevice));
  FL(flce_forward(H, W, (const int64_t*)y, T, Hd, V, -100, FLCE_REDUCTION_MEAN, (float*)loss, (float*)lse,
                  (float*)logp, (int64_t*)nv, fws, fwsb, NULL));
  FL(flce_backward((const float*)dl, H, W, (const int64_t*)y, (const float*)lse, T, Hd, V, -100,
                   FLCE_REDUCTION_MEAN, dH, (float*)dW, bws, bwsb, NULL));
  int32_t st = -1;
  FL(flce_read_device_status(fws, NULL, &st));
  if (st != 0) return 5;
  FL(flce_read_device_status(bws, NULL, &st));
  if (st != 0) return 6;
  float* out_f = (float*)malloc((size_t)(V * Hd * 4) > hb ? (size_t)(V * Hd * 4) : hb);
  CK(cudaMemcpy(out_f, lse, (size_t)T * 4, cudaMemcpyDeviceToHost));
  if (spill(dir, "lse.bin", out_f, (size_t)T * 4)) return 7;
  CK(cudaMemcpy(out_f, logp, (size_t)T * 4, cudaMemcpyDeviceToHost));
  if (spill(dir, "logp.bin", out_f, (size_t)T * 4)) return 7;
  CK(cudaMemcpy(out_f, loss, 4, cudaMemcpyDeviceToHost));
  if (spill(dir, "loss.bin", out_f, 4)) return 7;
  CK(cudaMemcpy(out_f, dH, hb, cudaMemcpyDeviceToHost));
  if (spill(dir, "dH.bin", out_f, hb)) return 7;
  CK(cudaMemcpy(out_f, dW, (size_t)(V * Hd * 4), cudaMemcpyDeviceToHost));
  if (spill(dir, "dW.bin", out_f, (size_t)(V * Hd * 4))) return 7;
  printf("ok\n");
  return 0;
}
