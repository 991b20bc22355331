/*
 * A plain C client of the vcoll C ABI (include/vcoll.h), built by
 * tests/test_c_client.py.  Mode "host": argument checks and the host-only
 * helpers, no GPU needed.  Mode "gpu": integer-valued fp32 buffers on the
 * device through reduce-scatter / allgather / allreduce, the user-ring
 * reduce-scatter and the fusion-buffer pipeline; every output element is
 * printed as its bits for the test to check against the oracle.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "vcoll.h"

#define W 4
#define N 1003

static int host_mode(void) {
  int64_t off, len;
  for (int j = 0; j < W; ++j) {
    if (vcoll_segment(N, W, j, &off, &len) != VCOLL_OK) return 1;
    printf("segment %d %lld %lld\n", j, (long long)off, (long long)len);
  }
  int64_t counts[5] = {10, 10, 10, 30, 2};
  int begin[6], nb = 0;
  if (vcoll_fuse_plan(counts, 5, VCOLL_F32, 100, begin, &nb) != VCOLL_OK) return 1;
  printf("plan");
  for (int b = 0; b <= nb; ++b) printf(" %d", begin[b]);
  printf("\n");
  const void* in[W] = {(void*)0x100000, (void*)0x200000, (void*)0x300000, (void*)0x400000};
  void* out[W] = {(void*)0x1100000, (void*)0x1200000, (void*)0x1300000, (void*)0x1400000};
  printf("bad_op %d\n", vcoll_allreduce(in, out, W, N, VCOLL_F32, 42, 0, NULL));
  printf("bad_type %d\n", vcoll_allreduce(in, out, W, N, 42, VCOLL_SUM, 0, NULL));
  printf("bad_w %d\n", vcoll_allreduce(in, out, 0, N, VCOLL_F32, VCOLL_SUM, 0, NULL));
  printf("empty %d\n", vcoll_allreduce(in, out, W, 0, VCOLL_F32, VCOLL_SUM, 0, NULL));
  printf("status %s\n", vcoll_status_string(VCOLL_ERR_INVALID_OP));
  return 0;
}

static void print_bits(const char* tag, int u, const float* d, int n) {
  float* h = (float*)malloc(sizeof(float) * (n > 0 ? n : 1));
  cudaMemcpy(h, d, sizeof(float) * n, cudaMemcpyDeviceToHost);
  for (int i = 0; i < n; ++i) {
    unsigned bits;
    memcpy(&bits, &h[i], 4);
    printf("%s %d %d %08x\n", tag, u, i, bits);
  }
  free(h);
}

/* Integer-valued inputs through reduce-scatter + allgather, allreduce, the
 * user-ring reduce-scatter and the fusion-buffer pipeline; every output
 * element is printed as its bits for the test to compare with the oracle. */
static int gpu_mode(void) {
  float* h = (float*)malloc(sizeof(float) * N);
  float* d_in[W];
  float* d_out[W];
  float* d_seg[W];
  for (int u = 0; u < W; ++u) {
    for (int i = 0; i < N; ++i) h[i] = (float)((i * 7 + u * 13) % 41 - 20);
    if (cudaMalloc((void**)&d_in[u], sizeof(float) * N) != cudaSuccess) return 1;
    if (cudaMalloc((void**)&d_out[u], sizeof(float) * N) != cudaSuccess) return 1;
    if (cudaMalloc((void**)&d_seg[u], sizeof(float) * N) != cudaSuccess) return 1;
    cudaMemcpy(d_in[u], h, sizeof(float) * N, cudaMemcpyHostToDevice);
  }
  const void* const* in = (const void* const*)d_in;
  int rc = vcoll_reduce_scatter(in, (void* const*)d_seg, W, N, VCOLL_F32, VCOLL_SUM,
                                VCOLL_FLAG_RING_ORDER, NULL);
  if (rc) { printf("rs %d %s\n", rc, vcoll_last_error()); return 1; }
  rc = vcoll_allgather((const void* const*)d_seg, (void* const*)d_out, W, N, VCOLL_F32, VCOLL_SUM,
                       0, NULL);
  if (rc) { printf("ag %d %s\n", rc, vcoll_last_error()); return 1; }
  cudaDeviceSynchronize();
  for (int u = 0; u < W; ++u) print_bits("ag", u, d_out[u], N);
  rc = vcoll_allreduce(in, (void* const*)d_out, W, N, VCOLL_F32, VCOLL_SUM, 0, NULL);
  if (rc) { printf("ar %d %s\n", rc, vcoll_last_error()); return 1; }
  cudaDeviceSynchronize();
  for (int u = 0; u < W; ++u) print_bits("ar", u, d_out[u], N);
  /* avg over the ring {1, 2, 0, 3}: segment j ends at rank j */
  const int ring[W] = {1, 2, 0, 3};
  rc = vcoll_reduce_scatter_ring(in, (void* const*)d_seg, W, N, VCOLL_F32, VCOLL_AVG, ring, NULL);
  if (rc) { printf("rsr %d %s\n", rc, vcoll_last_error()); return 1; }
  cudaDeviceSynchronize();
  for (int j = 0; j < W; ++j) {
    int64_t off, len;
    vcoll_segment(N, W, j, &off, &len);
    print_bits("rsr", j, d_seg[j], (int)len);
  }
  /* fusion buffers: three tensors per rank (the first N - 353, then 3, then
   * 350 elements of d_in[u]) through d_seg[u], in place into d_out[u] */
  const int64_t counts[3] = {N - 353, 3, 350};
  const void* tin[W * 3];
  void* tout[W * 3];
  for (int u = 0; u < W; ++u) {
    cudaMemcpy(d_out[u], d_in[u], sizeof(float) * N, cudaMemcpyDeviceToDevice);
    int64_t o = 0;
    for (int t = 0; t < 3; ++t) {
      tin[u * 3 + t] = d_out[u] + o;
      tout[u * 3 + t] = d_out[u] + o;
      o += counts[t];
    }
  }
  int nb = 0;
  rc = vcoll_fusion_allreduce_buffered(tin, tout, counts, 3, (void* const*)d_seg,
                                       (int64_t)sizeof(float) * N, W, VCOLL_F32, VCOLL_SUM, 0,
                                       (int64_t)1 << 20, &nb, NULL);
  if (rc) { printf("fb %d %s\n", rc, vcoll_last_error()); return 1; }
  cudaDeviceSynchronize();
  printf("fb_batches %d\n", nb);
  for (int u = 0; u < W; ++u) print_bits("fb", u, d_out[u], N);
  for (int u = 0; u < W; ++u) {
    cudaFree(d_in[u]);
    cudaFree(d_out[u]);
    cudaFree(d_seg[u]);
  }
  free(h);
  return 0;
}

int main(int argc, char** argv) {
  if (argc > 1 && strcmp(argv[1], "gpu") == 0) return gpu_mode();
  return host_mode();
}
