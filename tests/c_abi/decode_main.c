/*
 * A C caller of the library: no Python and no PyTorch in the process, only
 * include/mla_decode.h and the CUDA runtime.  Reads one bf16 decode request
 * from raw little-endian files in <dir>, runs the split-KV schedule and the
 * decode on the legacy default stream, and writes the results back:
 *
 *   <dir>/request.txt   "B T H num_pages max_pages softmax_scale"
 *   <dir>/q.bin         bf16 [B][T][H][576]
 *   <dir>/kv.bin        bf16 [num_pages][64][576]
 *   <dir>/block_table.bin  int32 [B][max_pages]
 *   <dir>/seqlens.bin   int32 [B]
 *   -> <dir>/out.bin    bf16 [B][T][H][512]
 *   -> <dir>/lse.bin    fp32 [B][H][T]
 *
 * Exit status 0 on success; any library or CUDA error is printed with
 * mla_last_error_string() and gives exit status 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "mla_decode.h"

#define LIB(call)                                                                 \
  do {                                                                            \
    int rc_ = (call);                                                             \
    if (rc_ < 0) {                                                                \
      fprintf(stderr, "%s -> %d: %s\n", #call, rc_, mla_last_error_string());     \
      return 1;                                                                   \
    }                                                                             \
  } while (0)

#define CUDA(call)                                                                \
  do {                                                                            \
    cudaError_t e_ = (call);                                                      \
    if (e_ != cudaSuccess) {                                                      \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                 \
      return 1;                                                                   \
    }                                                                             \
  } while (0)

static void *read_file(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) return NULL;
  void *p = malloc(bytes ? bytes : 1);
  size_t got = p ? fread(p, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static int write_file(const char *dir, const char *name, const void *p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f) return 0;
  size_t put = fwrite(p, 1, bytes, f);
  fclose(f);
  return put == bytes;
}

int main(int argc, char **argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s <request dir>\n", argv[0]);
    return 2;
  }
  const char *dir = argv[1];
  char path[4096];
  snprintf(path, sizeof path, "%s/request.txt", dir);
  FILE *rf = fopen(path, "r");
  int B, T, H, num_pages, max_pages;
  float scale;
  if (!rf || fscanf(rf, "%d %d %d %d %d %f", &B, &T, &H, &num_pages, &max_pages, &scale) != 6) {
    fprintf(stderr, "cannot read %s\n", path);
    return 2;
  }
  fclose(rf);

  const size_t q_bytes = (size_t)B * T * H * 576 * 2;
  const size_t kv_bytes = (size_t)num_pages * 64 * 576 * 2;
  const size_t bt_bytes = (size_t)B * max_pages * 4;
  const size_t sk_bytes = (size_t)B * 4;
  const size_t out_bytes = (size_t)B * T * H * 512 * 2;
  const size_t lse_bytes = (size_t)B * H * T * 4;
  void *h_q = read_file(dir, "q.bin", q_bytes);
  void *h_kv = read_file(dir, "kv.bin", kv_bytes);
  void *h_bt = read_file(dir, "block_table.bin", bt_bytes);
  void *h_sk = read_file(dir, "seqlens.bin", sk_bytes);
  void *h_out = malloc(out_bytes);
  void *h_lse = malloc(lse_bytes);
  if (!h_q || !h_kv || !h_bt || !h_sk || !h_out || !h_lse) {
    fprintf(stderr, "cannot read the request files\n");
    return 2;
  }

  void *q, *kv, *out, *workspace;
  int32_t *bt, *sk, *tile_md, *num_splits;
  float *lse;
  CUDA(cudaMalloc(&q, q_bytes));
  CUDA(cudaMalloc(&kv, kv_bytes));
  CUDA(cudaMalloc((void **)&bt, bt_bytes));
  CUDA(cudaMalloc((void **)&sk, sk_bytes));
  CUDA(cudaMalloc(&out, out_bytes));
  CUDA(cudaMalloc((void **)&lse, lse_bytes));
  CUDA(cudaMemcpy(q, h_q, q_bytes, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(kv, h_kv, kv_bytes, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(bt, h_bt, bt_bytes, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(sk, h_sk, sk_bytes, cudaMemcpyHostToDevice));

  int device = 0;
  CUDA(cudaGetDevice(&device));
  const int parts = mla_default_num_parts(device);
  LIB(parts);
  size_t md_elems = 0, ns_elems = 0;
  LIB(mla_decode_metadata_sizes(B, H, T, 0, parts, &md_elems, &ns_elems));
  CUDA(cudaMalloc((void **)&tile_md, md_elems * sizeof(int32_t)));
  CUDA(cudaMalloc((void **)&num_splits, ns_elems * sizeof(int32_t)));
  const size_t ws_bytes = mla_decode_workspace_bytes(B, H, T, 0, parts);
  if (ws_bytes == 0) {
    fprintf(stderr, "mla_decode_workspace_bytes refused the request\n");
    return 1;
  }
  CUDA(cudaMalloc(&workspace, ws_bytes));  /* cudaMalloc memory is 256-byte aligned */

  LIB(mla_decode_metadata(sk, B, H, T, 0, 0, parts, tile_md, num_splits, NULL));
  LIB(mla_decode(q, kv, MLA_KV_BF16, num_pages, MLA_PAGE_SIZE, bt, max_pages, sk, NULL, 0, NULL, NULL,
                 scale, 0, tile_md, num_splits, parts, workspace, ws_bytes, out, lse, B, T, H, NULL));
  CUDA(cudaDeviceSynchronize());
  uint32_t status = 0;
  LIB(mla_device_status(&status));
  if (status != 0) {
    fprintf(stderr, "device status 0x%x\n", status);
    return 1;
  }
  CUDA(cudaMemcpy(h_out, out, out_bytes, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(h_lse, lse, lse_bytes, cudaMemcpyDeviceToHost));
  if (!write_file(dir, "out.bin", h_out, out_bytes) || !write_file(dir, "lse.bin", h_lse, lse_bytes)) {
    fprintf(stderr, "cannot write the results\n");
    return 1;
  }
  cudaFree(q);
  cudaFree(kv);
  cudaFree(bt);
  cudaFree(sk);
  cudaFree(out);
  cudaFree(lse);
  cudaFree(tile_md);
  cudaFree(num_splits);
  cudaFree(workspace);
  free(h_q);
  free(h_kv);
  free(h_bt);
  free(h_sk);
  free(h_out);
  free(h_lse);
  printf("ok\n");
  return 0;
}
