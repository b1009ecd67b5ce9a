// ra_ll.h -- the pipelined variant's message protocol for small chunks
// (RA_OPT_PROTOCOL = RA_PROTOCOL_LL): shared by the host runtime and
// ra_ll.cu.  Nothing here is part of the public C ABI.
#pragma once

#include "ra_internal.h"

namespace ra {

// A message word: 32 bits of data below a 32-bit flag.  Elements of 1 to 4
// bytes take one word each; 8-byte elements two (low half, then high half).
constexpr int kLLThreads = 256;   // most threads per CTA
constexpr int kLLMaxE = 4;        // most positions a thread carries per round

// One cooperative launch of R*G CTAs of `threads` threads; CTA g of rank r
// carries positions g*threads*E + k*threads + tid (k < E) of every chunk it
// works on, and position pos of a message is word pos*wpe (+1) of the
// receiving rank's row.
struct LLArgs {
  Ptrs p;
  Plan plan;
  int R;
  int G;
  int E;
  int mode;
  int rounds;           // ring rounds this call runs; messages 0 .. rounds-2
  uint64_t* inbox;      // [message][receiving rank][plan.C * wpe] words
  uint32_t flag_base;   // message t of this call carries flag flag_base + t (no wrap within a call)
  int64_t timeout_ns;
  ra_device_error* err;
  int skip_rank;        // failure injection: this rank sends nothing from round skip_round on
  int skip_round;
};

// Message words per element.
inline int ll_words_per_element(int elem_bytes) { return elem_bytes == 8 ? 2 : 1; }

cudaError_t launch_ll(int dtype, int op, const LLArgs& a, int threads, cudaStream_t st);
cudaError_t ll_blocks_per_sm(int dtype, int op, int threads, int* blocks);

}  // namespace ra
