/*
 * A plain C consumer of libspecverify (no Python, no torch): reads one
 * batch of chain-verify inputs from a file, runs spec_verify_bf16 and the
 * tree verify through the C ABI on a stream of its own, and writes the
 * outputs to a file.  Used by tests/test_gpu_c_abi.py.
 *
 * Input file (little endian): int32 B, K, V, N; float tau; uint64 seed;
 * then target bf16 [B, K+1, V], draft bf16 [B, K, V], tokens int32 [B, K],
 * tree target bf16 [B, N+1, V], tree tokens int32 [B, N], parents int32
 * [B, N].  Output file: int32 tokens [B, K+1], n [B], path [B, N+1],
 * len [B], mask uint32 [B, N, ceil(N/32)], then uint32 status flags.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "specverify.h"

#define CHECK_CUDA(x)                                                                     \
  do {                                                                                    \
    cudaError_t e_ = (x);                                                                 \
    if (e_ != cudaSuccess) {                                                              \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x, cudaGetErrorString(e_)); \
      return 2;                                                                           \
    }                                                                                     \
  } while (0)
#define CHECK_SPEC(x)                                                                   \
  do {                                                                                  \
    int r_ = (x);                                                                       \
    if (r_ != SPEC_OK) {                                                                \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x, spec_status_string(r_)); \
      return 3;                                                                         \
    }                                                                                   \
  } while (0)

static void *read_block(FILE *f, size_t bytes) {
  void *p = malloc(bytes ? bytes : 1);
  if (p && bytes && fread(p, 1, bytes, f) != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static int to_device(void **dst, const void *src, size_t bytes, cudaStream_t s) {
  if (cudaMalloc(dst, bytes ? bytes : 16) != cudaSuccess) return 1;
  return bytes && cudaMemcpyAsync(*dst, src, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess;
}

int main(int argc, char **argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s input output\n", argv[0]);
    return 1;
  }
  FILE *f = fopen(argv[1], "rb");
  if (!f) return 1;
  int32_t dims[4];
  float tau;
  uint64_t seed;
  if (fread(dims, 4, 4, f) != 4 || fread(&tau, 4, 1, f) != 1 || fread(&seed, 8, 1, f) != 1) return 1;
  const int B = dims[0], K = dims[1], V = dims[2], N = dims[3];
  const int W = (N + 31) / 32;
  const size_t nt = (size_t)B * (K + 1) * V, nd = (size_t)B * K * V, ntt = (size_t)B * (N + 1) * V;
  void *h_t = read_block(f, nt * 2), *h_d = read_block(f, nd * 2), *h_x = read_block(f, (size_t)B * K * 4);
  void *h_tt = read_block(f, ntt * 2), *h_tok = read_block(f, (size_t)B * N * 4);
  void *h_par = read_block(f, (size_t)B * N * 4);
  fclose(f);
  if (!h_t || !h_d || !h_x || !h_tt || !h_tok || !h_par) return 1;

  cudaStream_t s;
  CHECK_CUDA(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
  void *d_t, *d_d, *d_x, *d_tt, *d_tok, *d_par, *d_out, *d_n, *d_path, *d_len, *d_mask;
  if (to_device(&d_t, h_t, nt * 2, s) || to_device(&d_d, h_d, nd * 2, s) ||
      to_device(&d_x, h_x, (size_t)B * K * 4, s) || to_device(&d_tt, h_tt, ntt * 2, s) ||
      to_device(&d_tok, h_tok, (size_t)B * N * 4, s) || to_device(&d_par, h_par, (size_t)B * N * 4, s))
    return 2;
  CHECK_CUDA(cudaMalloc(&d_out, (size_t)B * (K + 1) * 4));
  CHECK_CUDA(cudaMalloc(&d_n, (size_t)B * 4));
  CHECK_CUDA(cudaMalloc(&d_path, (size_t)B * (N + 1) * 4));
  CHECK_CUDA(cudaMalloc(&d_len, (size_t)B * 4));
  CHECK_CUDA(cudaMalloc(&d_mask, (size_t)B * N * W * 4 + 4));

  CHECK_SPEC(spec_verify_bf16((const uint16_t *)d_t, (const uint16_t *)d_d, (const int32_t *)d_x, B, K, V,
                              tau, seed, (int32_t *)d_out, (int32_t *)d_n, s));
  CHECK_SPEC(spec_tree_verify_greedy_bf16((const uint16_t *)d_tt, (const int32_t *)d_tok,
                                          (const int32_t *)d_par, B, N, V, (int32_t *)d_path,
                                          (int32_t *)d_len, (uint32_t *)d_mask, s));
  uint32_t flags = 0;
  CHECK_SPEC(spec_get_status(s, &flags));

  const size_t o1 = (size_t)B * (K + 1) * 4, o2 = (size_t)B * 4, o3 = (size_t)B * (N + 1) * 4,
               o4 = (size_t)B * 4, o5 = (size_t)B * N * W * 4;
  char *h_o = (char *)malloc(o1 + o2 + o3 + o4 + o5 + 4);
  if (!h_o) return 1;
  CHECK_CUDA(cudaMemcpy(h_o, d_out, o1, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_o + o1, d_n, o2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_o + o1 + o2, d_path, o3, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_o + o1 + o2 + o3, d_len, o4, cudaMemcpyDeviceToHost));
  if (o5) CHECK_CUDA(cudaMemcpy(h_o + o1 + o2 + o3 + o4, d_mask, o5, cudaMemcpyDeviceToHost));
  *(uint32_t *)(h_o + o1 + o2 + o3 + o4 + o5) = flags;
  FILE *g = fopen(argv[2], "wb");
  if (!g || fwrite(h_o, 1, o1 + o2 + o3 + o4 + o5 + 4, g) != o1 + o2 + o3 + o4 + o5 + 4) return 1;
  fclose(g);
  CHECK_CUDA(cudaStreamDestroy(s));
  return 0;
}
