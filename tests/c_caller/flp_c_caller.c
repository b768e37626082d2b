/*
 * A plain C caller of libfusedlogp: no Python, no torch.  Reads inputs from
 * raw files, scores them through the C ABI on the default stream, and
 * writes the outputs as raw float32 files for the test to compare with the
 * float64 oracle.
 *
 *   flp_c_caller DIR T H V N
 *
 * DIR holds h.bin (T x H bf16 bits), W.bin (V x H), ht.bin, Wt.bin (the
 * teacher's), targets.bin (T int64), rows.bin (N int64), g1.bin, g2.bin
 * (N float32).  Writes logp.bin, ent.bin, kl.bin, klmx.bin (N float32; the
 * last with the teacher on the block-scaled tensor cores), logpmx.bin and
 * entmx.bin (N float32: h scored against the teacher's head, in MXFP4, on the
 * block-scaled tensor cores), dh.bin (T x H bf16 bits) and dW.bin (V x H
 * float32).  Exit status 0 on success,
 * 2 on a library or CUDA error (the reason is printed).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "fusedlogp.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) return NULL;
  void *buf = malloc(bytes ? bytes : 1);
  size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static int write_file(const char *dir, const char *name, const void *buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f) return -1;
  size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : -1;
}

#define CUDA_OK(x)                                                       \
  do {                                                                   \
    cudaError_t e_ = (x);                                                \
    if (e_ != cudaSuccess) {                                             \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));           \
      return 2;                                                          \
    }                                                                    \
  } while (0)

#define FLP_OK_(x)                                                       \
  do {                                                                   \
    flp_status s_ = (x);                                                 \
    if (s_ != FLP_OK) {                                                  \
      fprintf(stderr, "%s: %s (%s)\n", #x, flp_status_string(s_),        \
              flp_last_error());                                         \
      return 2;                                                          \
    }                                                                    \
  } while (0)

static void *to_device(const void *host, size_t bytes) {
  void *d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char **argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s DIR T H V N\n", argv[0]);
    return 1;
  }
  const char *dir = argv[1];
  const int64_t T = atoll(argv[2]), H = atoll(argv[3]), V = atoll(argv[4]), N = atoll(argv[5]);
  const size_t hb = (size_t)(T * H * 2), wb = (size_t)(V * H * 2);
  void *h = read_file(dir, "h.bin", hb), *W = read_file(dir, "W.bin", wb);
  void *ht = read_file(dir, "ht.bin", hb), *Wt = read_file(dir, "Wt.bin", wb);
  void *tg = read_file(dir, "targets.bin", (size_t)T * 8), *rows = read_file(dir, "rows.bin", (size_t)N * 8);
  void *g1 = read_file(dir, "g1.bin", (size_t)N * 4), *g2 = read_file(dir, "g2.bin", (size_t)N * 4);
  if (!h || !W || !ht || !Wt || !tg || !rows || !g1 || !g2) {
    fprintf(stderr, "missing or short input file\n");
    return 1;
  }

  flp_shape s;
  memset(&s, 0, sizeof s);
  s.T = T;
  s.H = H;
  s.V = V;
  s.n_rows = N;
  s.dtype = FLP_BF16;
  s.ld_h = H;
  s.ld_w = H;

  void *d_h = to_device(h, hb), *d_W = to_device(W, wb), *d_ht = to_device(ht, hb);
  void *d_Wt = to_device(Wt, wb), *d_tg = to_device(tg, (size_t)T * 8);
  void *d_rows = to_device(rows, (size_t)N * 8), *d_g1 = to_device(g1, (size_t)N * 4);
  void *d_g2 = to_device(g2, (size_t)N * 4);
  if (!d_h || !d_W || !d_ht || !d_Wt || !d_tg || !d_rows || !d_g1 || !d_g2) {
    fprintf(stderr, "device allocation or copy failed\n");
    return 2;
  }
  size_t ws_bytes = flp_workspace_size(&s, FLP_OP_LOGPROB_ENTROPY);
  const size_t ws_kl = flp_workspace_size(&s, FLP_OP_KL), ws_bw = flp_workspace_size(&s, FLP_OP_BACKWARD);
  const size_t ws_klmx = flp_workspace_size(&s, FLP_OP_KL_MX);
  const size_t ws_fmx = flp_workspace_size(&s, FLP_OP_LOGPROB_ENTROPY_MX);
  if (ws_fmx > ws_bytes) ws_bytes = ws_fmx;
  if (ws_kl > ws_bytes) ws_bytes = ws_kl;
  if (ws_bw > ws_bytes) ws_bytes = ws_bw;
  if (ws_klmx > ws_bytes) ws_bytes = ws_klmx;
  const size_t head_bytes = flp_mx_head_bytes(V, H);
  if (ws_klmx == 0 || head_bytes == 0) {
    fprintf(stderr, "H must be a multiple of 128 for the block-scaled teacher\n");
    return 2;
  }
  if (ws_bytes == 0) {
    fprintf(stderr, "flp_workspace_size rejected the shape\n");
    return 2;
  }
  void *ws = NULL, *d_logp = NULL, *d_ent = NULL, *d_kl = NULL, *d_dh = NULL, *d_dW = NULL;
  void *d_head = NULL, *d_klmx = NULL, *d_lpmx = NULL, *d_enmx = NULL;
  CUDA_OK(cudaMalloc(&ws, ws_bytes));
  CUDA_OK(cudaMalloc(&d_head, head_bytes));
  CUDA_OK(cudaMalloc(&d_klmx, (size_t)N * 4 + 16));
  CUDA_OK(cudaMalloc(&d_lpmx, (size_t)N * 4 + 16));
  CUDA_OK(cudaMalloc(&d_enmx, (size_t)N * 4 + 16));
  CUDA_OK(cudaMalloc(&d_logp, (size_t)N * 4 + 16));
  CUDA_OK(cudaMalloc(&d_ent, (size_t)N * 4 + 16));
  CUDA_OK(cudaMalloc(&d_kl, (size_t)N * 4 + 16));
  CUDA_OK(cudaMalloc(&d_dh, hb));
  CUDA_OK(cudaMalloc(&d_dW, (size_t)V * H * 4));

  const float tau = 0.7f;
  FLP_OK_(flp_logprob_entropy(&s, d_h, d_W, (const int64_t *)d_tg, (const int64_t *)d_rows, tau,
                              (float *)d_logp, (float *)d_ent, NULL, NULL, ws, ws_bytes, NULL));
  flp_device_status st;
  FLP_OK_(flp_read_device_status(ws, &st, NULL));
  FLP_OK_(flp_kl(&s, d_h, d_W, d_ht, d_Wt, (const int64_t *)d_rows, (float *)d_kl, ws, ws_bytes, NULL));
  FLP_OK_(flp_read_device_status(ws, &st, NULL));
  FLP_OK_(flp_mx_head_quantize(d_Wt, FLP_BF16, V, H, H, d_head, NULL));
  FLP_OK_(flp_kl_mx(&s, d_h, d_W, d_ht, d_head, (const int64_t *)d_rows, (float *)d_klmx, ws, ws_bytes,
                    NULL));
  FLP_OK_(flp_read_device_status(ws, &st, NULL));
  FLP_OK_(flp_logprob_entropy_mx(&s, d_h, d_head, (const int64_t *)d_tg, (const int64_t *)d_rows, tau,
                                 (float *)d_lpmx, (float *)d_enmx, NULL, NULL, ws, ws_bytes, NULL));
  FLP_OK_(flp_read_device_status(ws, &st, NULL));
  FLP_OK_(flp_backward(&s, d_h, d_W, (const int64_t *)d_tg, (const int64_t *)d_rows, tau,
                       (const float *)d_g1, (const float *)d_g2, NULL, NULL, d_dh, (float *)d_dW, ws,
                       ws_bytes, NULL));
  FLP_OK_(flp_read_device_status(ws, &st, NULL));
  /* a call the library must reject on the host, with a reason */
  if (flp_logprob_entropy(&s, d_h, d_W, (const int64_t *)d_tg, (const int64_t *)d_rows, -1.0f,
                          (float *)d_logp, (float *)d_ent, NULL, NULL, ws, ws_bytes, NULL) !=
          FLP_ERR_INVALID_ARG ||
      strlen(flp_last_error()) == 0) {
    fprintf(stderr, "a negative temperature was not rejected\n");
    return 2;
  }
  CUDA_OK(cudaDeviceSynchronize());

  float *logp = malloc((size_t)N * 4 + 4), *ent = malloc((size_t)N * 4 + 4), *kl = malloc((size_t)N * 4 + 4);
  float *klmx = malloc((size_t)N * 4 + 4), *lpmx = malloc((size_t)N * 4 + 4);
  float *enmx = malloc((size_t)N * 4 + 4);
  void *dh = malloc(hb);
  float *dW = malloc((size_t)V * H * 4);
  if (!logp || !ent || !kl || !klmx || !lpmx || !enmx || !dh || !dW) return 2;
  CUDA_OK(cudaMemcpy(klmx, d_klmx, (size_t)N * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(lpmx, d_lpmx, (size_t)N * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(enmx, d_enmx, (size_t)N * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(logp, d_logp, (size_t)N * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(ent, d_ent, (size_t)N * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(kl, d_kl, (size_t)N * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(dh, d_dh, hb, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(dW, d_dW, (size_t)V * H * 4, cudaMemcpyDeviceToHost));
  if (write_file(dir, "logp.bin", logp, (size_t)N * 4) || write_file(dir, "ent.bin", ent, (size_t)N * 4) ||
      write_file(dir, "kl.bin", kl, (size_t)N * 4) || write_file(dir, "klmx.bin", klmx, (size_t)N * 4) ||
      write_file(dir, "logpmx.bin", lpmx, (size_t)N * 4) ||
      write_file(dir, "entmx.bin", enmx, (size_t)N * 4) ||
      write_file(dir, "dh.bin", dh, hb) ||
      write_file(dir, "dW.bin", dW, (size_t)V * H * 4)) {
    fprintf(stderr, "writing the outputs failed\n");
    return 1;
  }
  printf("ok: workspace %zu bytes\n", ws_bytes);
  return 0;
}
