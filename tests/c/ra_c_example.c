/* A C caller of the ring AllReduce library, for the test suite: plain C99,
 * only include/ra.h and the CUDA runtime.  R ranks of n fp32 elements hold
 * x_r[i] = 1000 r + (i mod 997); every output must hold the closed form
 * S[i] = 1000 R(R-1)/2 + R (i mod 997) exactly (small integers: exact in fp32
 * whatever the order).  Runs every variant (the pipelined one with each message
 * protocol too), the compact forms and the
 * host-buffer entry point, checks the chunk plan and the placement of the
 * 4-rank example, and exits non-zero on the first mismatch. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ra.h"

#define CHECK_RA(call)                                                              \
  do {                                                                              \
    ra_status s_ = (call);                                                          \
    if (s_ != RA_OK) {                                                              \
      fprintf(stderr, "%s failed: %s (%s)\n", #call, ra_status_string(s_), ra_last_error()); \
      return 1;                                                                     \
    }                                                                               \
  } while (0)

#define CHECK_CUDA(call)                                                            \
  do {                                                                              \
    cudaError_t e_ = (call);                                                        \
    if (e_ != cudaSuccess) {                                                        \
      fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));            \
      return 1;                                                                     \
    }                                                                               \
  } while (0)

/* protocol: the pipelined variant's RA_OPT_PROTOCOL, or -1 to leave it */
static int run(int R, size_t n, int variant, int protocol) {
  float* host = (float*)malloc(n * sizeof(float));
  void* in[32];
  void* out[32];
  ra_handle h = NULL;
  size_t i;
  int r;
  if (!host) return 1;
  for (r = 0; r < R; ++r) {
    CHECK_CUDA(cudaMalloc(&in[r], n * sizeof(float)));
    CHECK_CUDA(cudaMalloc(&out[r], n * sizeof(float)));
    for (i = 0; i < n; ++i) host[i] = (float)(1000 * r + (int)(i % 997));
    CHECK_CUDA(cudaMemcpy(in[r], host, n * sizeof(float), cudaMemcpyHostToDevice));
  }
  CHECK_RA(ra_create(R, n, RA_F32, RA_SUM, &h));
  CHECK_RA(ra_set_option(h, RA_OPT_VARIANT, variant));
  if (protocol >= 0) CHECK_RA(ra_set_option(h, RA_OPT_PROTOCOL, protocol));
  CHECK_RA(ra_allreduce(h, (const void* const*)in, (void* const*)out, NULL));
  CHECK_RA(ra_get_device_status(h, NULL, NULL));
  for (r = 0; r < R; ++r) {
    CHECK_CUDA(cudaMemcpy(host, out[r], n * sizeof(float), cudaMemcpyDeviceToHost));
    for (i = 0; i < n; ++i) {
      const float want = (float)(1000 * R * (R - 1) / 2 + R * (int)(i % 997));
      if (host[i] != want) {
        fprintf(stderr, "variant %d protocol %d R=%d n=%zu rank %d element %zu: %f != %f\n", variant, protocol, R,
                n, r, i, host[i], want);
        return 1;
      }
    }
  }
  if (variant == RA_VARIANT_AUTO) {
    /* compact ReduceScatter then compact AllGather give the same */
    void* chunk[32];
    for (r = 0; r < R; ++r) {
      size_t off, len;
      CHECK_RA(ra_owned_chunk(h, r, &off, &len));
      CHECK_CUDA(cudaMalloc(&chunk[r], (len ? len : 1) * sizeof(float)));
      CHECK_CUDA(cudaMemset(out[r], 0, n * sizeof(float)));
    }
    CHECK_RA(ra_reduce_scatter_compact(h, (const void* const*)in, (void* const*)chunk, NULL));
    CHECK_RA(ra_all_gather_compact(h, (const void* const*)chunk, (void* const*)out, NULL));
    CHECK_RA(ra_get_device_status(h, NULL, NULL));
    for (r = 0; r < R; ++r) {
      CHECK_CUDA(cudaMemcpy(host, out[r], n * sizeof(float), cudaMemcpyDeviceToHost));
      for (i = 0; i < n; ++i)
        if (host[i] != (float)(1000 * R * (R - 1) / 2 + R * (int)(i % 997))) {
          fprintf(stderr, "compact R=%d rank %d element %zu wrong\n", R, r, i);
          return 1;
        }
      CHECK_CUDA(cudaFree(chunk[r]));
    }
    /* the same AllReduce from host buffers (plain malloc: pageable) */
    {
      float* hin[32];
      float* hout[32];
      for (r = 0; r < R; ++r) {
        hin[r] = (float*)malloc(n * sizeof(float));
        hout[r] = (float*)malloc(n * sizeof(float));
        if (!hin[r] || !hout[r]) return 1;
        for (i = 0; i < n; ++i) hin[r][i] = (float)(1000 * r + (int)(i % 997));
      }
      CHECK_RA(ra_allreduce_host(h, (const void* const*)hin, (void* const*)hout, NULL));
      CHECK_CUDA(cudaStreamSynchronize(NULL));
      for (r = 0; r < R; ++r) {
        for (i = 0; i < n; ++i)
          if (hout[r][i] != (float)(1000 * R * (R - 1) / 2 + R * (int)(i % 997))) {
            fprintf(stderr, "host buffers R=%d rank %d element %zu wrong\n", R, r, i);
            return 1;
          }
        free(hin[r]);
        free(hout[r]);
      }
    }
  }
  CHECK_RA(ra_destroy(h));
  for (r = 0; r < R; ++r) {
    CHECK_CUDA(cudaFree(in[r]));
    CHECK_CUDA(cudaFree(out[r]));
  }
  free(host);
  return 0;
}

int main(void) {
  static const int variants[] = {RA_VARIANT_AUTO, RA_VARIANT_DIRECT, RA_VARIANT_RING, RA_VARIANT_PERSISTENT,
                                 RA_VARIANT_PIPELINED, RA_VARIANT_LOCAL};
  static const int ranks[] = {2, 4, 7, 16};
  static const size_t sizes[] = {1, 4096, 100003};
  size_t off[4], len[4];
  unsigned v, a, b;
  int k;
  /* the 4-rank example: chunks of 1024, rank r owns chunk (r+1) mod 4 */
  CHECK_RA(ra_chunk_plan(4, 4096, off, len));
  for (k = 0; k < 4; ++k)
    if (off[k] != (size_t)k * 1024 || len[k] != 1024) return 1;
  for (v = 0; v < sizeof(variants) / sizeof(variants[0]); ++v)
    for (a = 0; a < sizeof(ranks) / sizeof(ranks[0]); ++a)
      for (b = 0; b < sizeof(sizes) / sizeof(sizes[0]); ++b)
        if (run(ranks[a], sizes[b], variants[v], -1)) return 1;
  /* the pipelined variant's flag-in-data protocols */
  for (k = RA_PROTOCOL_LL; k <= RA_PROTOCOL_LL_CLUSTER; ++k)
    for (a = 0; a < sizeof(ranks) / sizeof(ranks[0]); ++a)
      for (b = 0; b < sizeof(sizes) / sizeof(sizes[0]); ++b)
        if (run(ranks[a], sizes[b], RA_VARIANT_PIPELINED, k)) return 1;
  printf("c example: ok\n");
  return 0;
}
