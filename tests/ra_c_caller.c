/*
 * A plain C caller of libra.so through include/ra.h: no Python, no torch.
 * It checks the boundary the way a C user meets it.
 *
 * Host part (no GPU needed): chunk bounds of the tirogla.com "Ring all-reduce"
 * self-test shape (section "Code": N = 5, L = 1003 gives chunks of 200, 201,
 * 200, 201 and 201 elements), and argument errors caught before any launch.
 *
 * Device part: x_r[i] = r*L + i on N = 5 ranks, whose ring sum is 5*i + 10030
 * on every rank, exact in fp32 (the same page's self-test). The all-reduce,
 * the reduce-scatter (shard c = chunk c of that sum) and the all-gather of the
 * shards must give exactly that; an average on a created stream must give
 * the fp32 product of the sum and 1.0f/5.
 *
 * Usage: ra_c_caller [--host-only]; prints "C ABI HOST OK" / "C ABI OK".
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ra.h"

#define N 5
#define L 1003

static int fail(const char* what) {
  fprintf(stderr, "FAIL: %s\n", what);
  return 1;
}

static int host_checks(void) {
  const size_t bounds[N + 1] = {0, 200, 401, 601, 802, 1003};
  for (int c = 0; c < N; ++c) {
    size_t b = 0, e = 0;
    if (ra_chunk_range(L, N, c, &b, &e) != RA_SUCCESS) return fail("ra_chunk_range status");
    if (b != bounds[c] || e != bounds[c + 1]) return fail("chunk bounds");
  }
  const void* sends[1] = {NULL};
  void* recvs[1] = {NULL};
  if (ra_allreduce(sends, recvs, 16, RA_FLOAT32, RA_SUM, 0, NULL) != RA_ERR_INVALID_ARG)
    return fail("nranks 0 accepted");
  if (ra_allreduce(sends, recvs, 16, RA_FLOAT32, RA_SUM, RA_MAX_RANKS + 1, NULL) != RA_ERR_INVALID_ARG)
    return fail("nranks above RA_MAX_RANKS accepted");
  if (ra_allreduce(NULL, recvs, 16, RA_FLOAT32, RA_SUM, 1, NULL) != RA_ERR_INVALID_ARG)
    return fail("null send array accepted");
  if (ra_allreduce(sends, recvs, 16, (ra_dtype_t)9, RA_SUM, 1, NULL) != RA_ERR_INVALID_ARG)
    return fail("bad dtype accepted");
  if (ra_allreduce(sends, recvs, 16, RA_FLOAT32, RA_SUM, 1, NULL) != RA_ERR_INVALID_ARG)
    return fail("null buffers accepted");
  if (ra_allreduce(sends, recvs, 0, RA_FLOAT32, RA_SUM, 1, NULL) != RA_SUCCESS)
    return fail("count 0 not a no-op");
  const char* s = ra_status_string(RA_ERR_ALIAS);
  if (s == NULL || s[0] == '\0') return fail("ra_status_string");
  if (ra_vector_bytes() < 16) return fail("ra_vector_bytes");
  return 0;
}

static int cuda_ok(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return 1;
  fprintf(stderr, "FAIL: %s: %s\n", what, cudaGetErrorString(e));
  return 0;
}

static int device_checks(void) {
  float* host = (float*)malloc(sizeof(float) * L);
  float* send[N] = {0};
  float* recv[N] = {0};
  float* shard[N] = {0};
  float* gathered[N] = {0};
  size_t b[N], e[N];
  int rc = 1;
  for (int r = 0; r < N; ++r) {
    for (int i = 0; i < L; ++i) host[i] = (float)(r * L + i);
    if (ra_chunk_range(L, N, r, &b[r], &e[r]) != RA_SUCCESS) goto out;
    if (!cuda_ok(cudaMalloc((void**)&send[r], sizeof(float) * L), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&recv[r], sizeof(float) * L), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&shard[r], sizeof(float) * (e[r] - b[r])), "cudaMalloc") ||
        !cuda_ok(cudaMalloc((void**)&gathered[r], sizeof(float) * L), "cudaMalloc") ||
        !cuda_ok(cudaMemcpy(send[r], host, sizeof(float) * L, cudaMemcpyHostToDevice), "copy in"))
      goto out;
  }
  const void* const* sends = (const void* const*)send;
  if (ra_allreduce(sends, (void* const*)recv, L, RA_FLOAT32, RA_SUM, N, NULL) != RA_SUCCESS ||
      ra_reduce_scatter(sends, (void* const*)shard, L, RA_FLOAT32, RA_SUM, N, NULL) != RA_SUCCESS ||
      ra_allgather((const void* const*)shard, (void* const*)gathered, L, RA_FLOAT32, RA_SUM, N, NULL) != RA_SUCCESS) {
    fail("a collective returned an error");
    goto out;
  }
  if (!cuda_ok(cudaDeviceSynchronize(), "synchronize")) goto out;
  for (int r = 0; r < N; ++r) {
    if (!cuda_ok(cudaMemcpy(host, recv[r], sizeof(float) * L, cudaMemcpyDeviceToHost), "copy out")) goto out;
    for (int i = 0; i < L; ++i)
      if (host[i] != (float)(5 * i + 10030)) { fail("all-reduce value"); goto out; }
    if (!cuda_ok(cudaMemcpy(host, gathered[r], sizeof(float) * L, cudaMemcpyDeviceToHost), "copy out")) goto out;
    for (int i = 0; i < L; ++i)
      if (host[i] != (float)(5 * i + 10030)) { fail("all-gather of the shards"); goto out; }
    const size_t len = e[r] - b[r];
    if (!cuda_ok(cudaMemcpy(host, shard[r], sizeof(float) * len, cudaMemcpyDeviceToHost), "copy out")) goto out;
    for (size_t j = 0; j < len; ++j)
      if (host[j] != (float)(5 * (int)(b[r] + j) + 10030)) { fail("reduce-scatter shard"); goto out; }
  }
  cudaStream_t stream;
  if (!cuda_ok(cudaStreamCreate(&stream), "stream")) goto out;
  if (ra_allreduce(sends, (void* const*)recv, L, RA_FLOAT32, RA_AVG, N, (void*)stream) != RA_SUCCESS) {
    fail("average returned an error");
    cudaStreamDestroy(stream);
    goto out;
  }
  if (!cuda_ok(cudaStreamSynchronize(stream), "stream synchronize")) goto out;
  cudaStreamDestroy(stream);
  const float inv_n = 1.0f / 5.0f;
  for (int r = 0; r < N; ++r) {
    if (!cuda_ok(cudaMemcpy(host, recv[r], sizeof(float) * L, cudaMemcpyDeviceToHost), "copy out")) goto out;
    for (int i = 0; i < L; ++i) {
      const float want = (float)(5 * i + 10030) * inv_n;
      if (host[i] != want) { fail("average value"); goto out; }
    }
  }
  rc = 0;
out:
  for (int r = 0; r < N; ++r) {
    cudaFree(send[r]);
    cudaFree(recv[r]);
    cudaFree(shard[r]);
    cudaFree(gathered[r]);
  }
  free(host);
  return rc;
}

int main(int argc, char** argv) {
  if (host_checks() != 0) return 1;
  if (argc > 1 && strcmp(argv[1], "--host-only") == 0) {
    printf("C ABI HOST OK\n");
    return 0;
  }
  if (device_checks() != 0) return 1;
  printf("C ABI OK\n");
  return 0;
}
