// ra_ll.h -- the pipelined variant's flag-in-data messages for small chunks
// (RA_OPT_PROTOCOL = RA_PROTOCOL_LL, RA_PROTOCOL_LL_CLUSTER): shared by the
// host runtime and ra_ll.cu.  Nothing here is part of the public C ABI.
#pragma once

#include "ra_internal.h"

namespace ra {

// A message word: 32 bits of data below a 32-bit flag.  Elements of 1 to 4
// bytes take one word each; 8-byte elements two (low half, then high half).
constexpr int kLLThreads = 256;   // most threads per CTA
constexpr int kLLMaxE = 4;        // most positions a thread carries per round
constexpr int kLLClusterMaxSmem = 200 * 1024;   // most shared memory of a cluster CTA's rows

// R*G CTAs of `threads` threads; CTA (g, r) = blockIdx.x g*R + r carries
// positions g*threads*E + k*threads + tid (k < E) of every chunk it works on.
// LL: one cooperative launch; position pos of a message is word pos*wpe
// (+1) of the receiving rank's inbox row.  LL_CLUSTER: one cluster of R CTAs
// per channel; local position k*threads + tid is word (k*threads + tid)*wpe
// (+1) of the receiving CTA's row in its shared memory.
struct LLArgs {
  Ptrs p;
  Plan plan;
  int R;
  int G;
  int E;
  int mode;
  int elem_bytes;
  int rounds;           // ring rounds this call runs; messages 0 .. rounds-2
  uint64_t* inbox;      // LL: [message][receiving rank][plan.C * wpe] words
  uint32_t flag_base;   // LL: message t of this call carries flag flag_base + t (no wrap within a call)
  uint64_t* bases;      // LL: each CTA's copy of the flag its next call starts at, [nbases >= R*G]
  int nbases;
  int from_memory;      // LL: take the flag base from the CTA's copy (a launch a CUDA graph replays)
  int64_t timeout_ns;
  ra_device_error* err;
  int skip_rank;        // failure injection: this rank sends nothing from round skip_round on
  int skip_round;
};

// Message words per element.
inline int ll_words_per_element(int elem_bytes) { return elem_bytes == 8 ? 2 : 1; }

cudaError_t launch_ll(int dtype, int op, const LLArgs& a, int threads, cudaStream_t st);
cudaError_t ll_blocks_per_sm(int dtype, int op, int threads, int* blocks);

// LL_CLUSTER: shared memory of one CTA's rows, the per-device set-up (cluster
// sizes up to 16, the shared-memory opt-in), clusters that fit at once.
size_t ll_cluster_smem_bytes(const LLArgs& a, int threads, int elem_bytes);
cudaError_t prepare_ll_cluster();
cudaError_t ll_cluster_capacity(int dtype, int op, const LLArgs& a, int threads, size_t smem, int* clusters);
cudaError_t launch_ll_cluster(int dtype, int op, const LLArgs& a, int threads, size_t smem, cudaStream_t st);

}  // namespace ra
