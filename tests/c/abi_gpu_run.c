/* A plain C99 program that runs the forward and backward through the C ABI on
 * the GPU, with the CUDA runtime for memory: reads X (bf16 bits), W (bf16
 * bits) and labels (int64) from files, writes loss, lse, n_valid, dX and dW
 * (bf16 bits) to files.  Usage:
 *   abi_gpu_run N H V seq_len shift reduction(0 mean, 1 sum) in_dir out_dir
 * Exits 0 on success; prints the failing call otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "flce.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
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

static int write_file(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(p, 1, bytes, f);
  fclose(f);
  return put != bytes;
}

#define CHECK_CUDA(x)                                 \
  do {                                                \
    if ((x) != cudaSuccess) {                         \
      printf("CUDA call failed: %s\n", #x);           \
      return 1;                                       \
    }                                                 \
  } while (0)

#define CHECK_FLCE(x)                                                  \
  do {                                                                 \
    flce_status st_ = (x);                                             \
    if (st_ != FLCE_OK) {                                              \
      printf("%s returned %s\n", #x, flce_status_string(st_));         \
      return 1;                                                        \
    }                                                                  \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 9) {
    printf("usage: abi_gpu_run N H V seq_len shift reduction in_dir out_dir\n");
    return 2;
  }
  const int64_t N = atoll(argv[1]), H = atoll(argv[2]), V = atoll(argv[3]);
  const int64_t seq_len = atoll(argv[4]);
  const int shift = atoi(argv[5]);
  const flce_reduction red = atoi(argv[6]) ? FLCE_REDUCTION_SUM : FLCE_REDUCTION_MEAN;
  const char* in_dir = argv[7];
  const char* out_dir = argv[8];
  const size_t xb = (size_t)N * H * 2, wb = (size_t)V * H * 2, lb = (size_t)N * 8;
  void* hx = read_file(in_dir, "X.bin", xb);
  void* hw = read_file(in_dir, "W.bin", wb);
  void* hl = read_file(in_dir, "labels.bin", lb);
  if (!hx || !hw || !hl) {
    printf("cannot read the inputs\n");
    return 1;
  }
  const size_t ws_bytes = flce_workspace_size(N, H, V);
  if (ws_bytes == 0) {
    printf("flce_workspace_size rejected the sizes\n");
    return 1;
  }
  void *dx_in, *dw_in, *dl, *ws, *dX, *dW;
  float *loss, *lse, *g;
  int64_t* nv;
  CHECK_CUDA(cudaMalloc(&dx_in, xb));
  CHECK_CUDA(cudaMalloc(&dw_in, wb));
  CHECK_CUDA(cudaMalloc(&dl, lb));
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMalloc(&dX, xb));
  CHECK_CUDA(cudaMalloc(&dW, wb));
  CHECK_CUDA(cudaMalloc((void**)&loss, 4));
  CHECK_CUDA(cudaMalloc((void**)&lse, (size_t)N * 4));
  CHECK_CUDA(cudaMalloc((void**)&g, 4));
  CHECK_CUDA(cudaMalloc((void**)&nv, 8));
  CHECK_CUDA(cudaMemcpy(dx_in, hx, xb, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dw_in, hw, wb, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dl, hl, lb, cudaMemcpyHostToDevice));
  const float one = 1.0f;
  CHECK_CUDA(cudaMemcpy(g, &one, 4, cudaMemcpyHostToDevice));
  cudaStream_t s;
  CHECK_CUDA(cudaStreamCreate(&s));
  flce_stream_t fs = (flce_stream_t)s;
  CHECK_FLCE(flce_forward(dx_in, dw_in, (const int64_t*)dl, N, H, V, seq_len, -100, shift, red,
                          loss, lse, nv, ws, ws_bytes, fs));
  CHECK_FLCE(flce_backward(dx_in, dw_in, (const int64_t*)dl, N, H, V, seq_len, -100, shift, red,
                           lse, nv, g, dX, dW, ws, ws_bytes, fs));
  CHECK_FLCE(flce_get_error(ws, fs));
  float h_loss;
  int64_t h_nv;
  float* h_lse = (float*)malloc((size_t)N * 4);
  void* h_dX = malloc(xb);
  void* h_dW = malloc(wb);
  CHECK_CUDA(cudaMemcpy(&h_loss, loss, 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(&h_nv, nv, 8, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_lse, lse, (size_t)N * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_dX, dX, xb, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_dW, dW, wb, cudaMemcpyDeviceToHost));
  if (write_file(out_dir, "loss.bin", &h_loss, 4) || write_file(out_dir, "n_valid.bin", &h_nv, 8) ||
      write_file(out_dir, "lse.bin", h_lse, (size_t)N * 4) ||
      write_file(out_dir, "dX.bin", h_dX, xb) || write_file(out_dir, "dW.bin", h_dW, wb)) {
    printf("cannot write the outputs\n");
    return 1;
  }
  cudaStreamDestroy(s);
  cudaFree(dx_in);
  cudaFree(dw_in);
  cudaFree(dl);
  cudaFree(ws);
  cudaFree(dX);
  cudaFree(dW);
  cudaFree(loss);
  cudaFree(lse);
  cudaFree(g);
  cudaFree(nv);
  printf("ok\n");
  return 0;
}
