/*
 * A plain C99 caller of libdsa_cb.so: no Python, no PyTorch, only the
 * declarations of include/dsa_cb.h and the CUDA runtime API.
 *
 *   c_abi_consumer <input> <output>
 *
 * <input> holds a selection problem: six int64 values (rows, width,
 * block_size, topk_blocks, row_repeat, pin_newest), then rows * width fp32
 * logits (row-major), then ceil(rows / row_repeat) int32 window ends and as
 * many int32 window starts. The program copies them into device memory it
 * allocates itself, runs dsa_select_candidate_blocks on a stream it creates
 * (with a workspace of dsa_select_workspace_bytes, zero-filled once, and
 * calls it twice to reuse it), and writes the rows * topk_blocks int32 ids
 * to <output>. It exits non-zero, with a message, on any error.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "dsa_cb.h"

static int fail(const char *what) {
  fprintf(stderr, "c_abi_consumer: %s\n", what);
  return 1;
}

#define CUDA_OK(call) \
  do { if ((call) != cudaSuccess) return fail(#call); } while (0)

static void *read_all(const char *path, size_t *size) {
  FILE *f = fopen(path, "rb");
  if (!f) return NULL;
  fseek(f, 0, SEEK_END);
  long n = ftell(f);
  fseek(f, 0, SEEK_SET);
  void *buf = n > 0 ? malloc((size_t)n) : NULL;
  if (buf && fread(buf, 1, (size_t)n, f) != (size_t)n) {
    free(buf);
    buf = NULL;
  }
  fclose(f);
  *size = buf ? (size_t)n : 0;
  return buf;
}

int main(int argc, char **argv) {
  if (argc != 3) return fail("usage: c_abi_consumer <input> <output>");
  size_t size = 0;
  unsigned char *in = read_all(argv[1], &size);
  if (!in || size < 6 * sizeof(int64_t)) return fail("cannot read the input");
  const int64_t *hdr = (const int64_t *)in;
  const int64_t rows = hdr[0], width = hdr[1];
  const int32_t block_size = (int32_t)hdr[2], topk = (int32_t)hdr[3];
  const int32_t row_repeat = (int32_t)hdr[4], pin = (int32_t)hdr[5];
  if (rows < 1 || width < 1 || row_repeat < 1 || topk < 1) return fail("bad header");
  const int64_t groups = (rows + row_repeat - 1) / row_repeat;
  const size_t n_logits = (size_t)(rows * width), n_ids = (size_t)(rows * topk);
  if (size != 6 * sizeof(int64_t) + n_logits * sizeof(float) + 2 * (size_t)groups * 4)
    return fail("input size does not match its header");
  const float *logits = (const float *)(hdr + 6);
  const int32_t *ke = (const int32_t *)(logits + n_logits);
  const int32_t *ks = ke + groups;

  float *d_logits = NULL;
  int32_t *d_ke = NULL, *d_ks = NULL, *d_out = NULL;
  void *d_ws = NULL;
  const int64_t nb = (width + block_size - 1) / block_size;
  const size_t ws_bytes = dsa_select_workspace_bytes(rows, nb);
  cudaStream_t stream = NULL;
  CUDA_OK(cudaStreamCreate(&stream));
  CUDA_OK(cudaMalloc((void **)&d_logits, n_logits * sizeof(float)));
  CUDA_OK(cudaMalloc((void **)&d_ke, (size_t)groups * 4));
  CUDA_OK(cudaMalloc((void **)&d_ks, (size_t)groups * 4));
  CUDA_OK(cudaMalloc((void **)&d_out, n_ids * 4));
  CUDA_OK(cudaMalloc(&d_ws, ws_bytes));
  CUDA_OK(cudaMemset(d_ws, 0, ws_bytes));
  CUDA_OK(cudaMemcpy(d_logits, logits, n_logits * sizeof(float), cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(d_ke, ke, (size_t)groups * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(d_ks, ks, (size_t)groups * 4, cudaMemcpyHostToDevice));

  for (int call = 0; call < 2; ++call) {
    CUDA_OK(cudaMemsetAsync(d_out, 0x7f, n_ids * 4, stream));
    const dsa_status st = dsa_select_candidate_blocks(
        d_logits, rows, width, width, d_ks, d_ke, topk, block_size, row_repeat, pin, d_out,
        topk, NULL, 0, d_ws, ws_bytes, (void *)stream);
    if (st != DSA_OK) return fail(dsa_status_string(st));
  }
  CUDA_OK(cudaStreamSynchronize(stream));

  int32_t *ids = (int32_t *)malloc(n_ids * 4);
  if (!ids) return fail("out of host memory");
  CUDA_OK(cudaMemcpy(ids, d_out, n_ids * 4, cudaMemcpyDeviceToHost));
  FILE *f = fopen(argv[2], "wb");
  if (!f || fwrite(ids, 4, n_ids, f) != n_ids) return fail("cannot write the output");
  fclose(f);

  /* The invalid-argument path: nothing is launched, the status says why. */
  if (dsa_select_candidate_blocks(d_logits, rows, width, width - 1, d_ks, d_ke, topk,
                                  block_size, row_repeat, pin, d_out, topk, NULL, 0, NULL, 0,
                                  (void *)stream) != DSA_EINVAL)
    return fail("ld_logits < width was not refused");

  free(ids);
  free(in);
  CUDA_OK(cudaFree(d_ws));
  CUDA_OK(cudaFree(d_out));
  CUDA_OK(cudaFree(d_ks));
  CUDA_OK(cudaFree(d_ke));
  CUDA_OK(cudaFree(d_logits));
  CUDA_OK(cudaStreamDestroy(stream));
  return 0;
}
