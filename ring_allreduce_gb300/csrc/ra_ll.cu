// ra_ll.cu -- the pipelined variant with flag-in-data messages
// (RA_OPT_PROTOCOL = RA_PROTOCOL_LL), for chunks small enough that a ring
// round is a chain of memory latencies rather than a stream of bytes.
//
// "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce",
// sections 4 to 8: in every round a rank receives one chunk's partial from
// its predecessor, folds its own piece into it (incoming (+) local) and
// sends the result on; the last reduce round leaves the complete chunk with
// its owner, and R-1 copy rounds carry the complete chunks round the ring.
// The schedule, the chunks and the fold order are those of the other
// variants, so the results are bitwise the same.
//
// What differs is how a message travels.  The other variants write a
// partial into the sender's output buffer and then publish it (a release
// fence and a signal the receiver polls), so every hop costs a store, a
// fence that waits for the store to be acknowledged, the signal's trip and
// the receiver's poll, then a load of the data.  Here each message word
// carries 32 bits of data together with a 32-bit flag naming the call and
// the round, written by one 8-byte store (single-copy atomic): the receiver
// polls the data words themselves, and a word whose flag is the expected
// one holds the expected data.  A hop is then one store and the poll that
// sees it, with no fence, no separate signal and no CTA barrier: thread k
// of a receiving CTA depends only on thread k of the sending CTA, which
// carries the same positions of the same chunk.  This is the low-latency
// message form of NCCL's ring (flags inside the data), which the pages do
// not describe.  The price is twice the bytes per element (four times for
// 16-bit elements), so it is for small chunks only.
//
// Messages live in an inbox of the handle, one row per (message, receiving
// rank), each row written once per call, so no word is overwritten while
// someone may still read it.  Flags grow by one per message and by the
// call's rounds per call (the host restarts them, zeroing the inbox, before
// they would wrap), so a word left from any earlier call or round never
// carries the flag being waited for.  Outputs are written only with complete
// values (the owner's chunk after the last reduce round, every chunk in the
// copy rounds), and each is written by the thread that read the same
// element of the same rank's input earlier, or (a rank's chunk r read by its
// successor in the first round) at the end of a chain of messages each of
// which carries a value computed from that read: in place calls are safe.
//
// Waits are bounded (timeout_ns, two clocks); one that runs out records code
// 5 (round, rank, channel, predecessor, flag seen, flag expected) and the
// thread returns; every other waiter returns once it sees the record.
#include "ra_device.cuh"
#include "ra_ll.h"

namespace ra {
namespace {

template <class T>
__device__ __forceinline__ uint64_t raw_bits(T v) {
  uint64_t b = 0;
  memcpy(&b, &v, sizeof(T));
  return b;
}

template <class T>
__device__ __forceinline__ T from_raw(uint64_t b) {
  T v;
  memcpy(&v, &b, sizeof(T));
  return v;
}

__device__ __forceinline__ uint32_t word_flag(uint64_t w) { return (uint32_t)(w >> 32); }

// Poll the words of this thread's positions in `box` until each carries
// `flag`; the data into val[].  False when the thread must stop.
template <class T, int WPE>
__device__ __forceinline__ bool ll_receive(const LLArgs& a, const uint64_t* box, int64_t pos0, int64_t len,
                                           uint32_t flag, T* val, int t, int r, int g, int p) {
  uint64_t w[kLLMaxE * WPE];
  uint32_t pending = 0;
#pragma unroll
  for (int k = 0; k < kLLMaxE; ++k) {
    const int64_t pos = pos0 + (int64_t)k * blockDim.x;
    if (k < a.E && pos < len) {
#pragma unroll
      for (int h = 0; h < WPE; ++h) {
        w[k * WPE + h] = signal_load_relaxed(box + pos * WPE + h);
        if (word_flag(w[k * WPE + h]) != flag) pending |= 1u << (k * WPE + h);
      }
    }
  }
  if (pending) {
    const Deadline limit(a.timeout_ns);
    for (uint32_t it = 0;; ++it) {
      if (it >= 64) __nanosleep(64);
#pragma unroll
      for (int i = 0; i < kLLMaxE * WPE; ++i) {
        if (pending & (1u << i)) {
          const int64_t pos = pos0 + (int64_t)(i / WPE) * blockDim.x;
          w[i] = signal_load_relaxed(box + pos * WPE + (i % WPE));
          if (word_flag(w[i]) == flag) pending &= ~(1u << i);
        }
      }
      if (!pending) break;
      if ((it & 7u) == 7u && load_relaxed_u32(&a.err->code) != 0u) return false;
      if (limit.passed()) {
        uint32_t seen = 0;
#pragma unroll
        for (int i = kLLMaxE * WPE - 1; i >= 0; --i)
          if (pending & (1u << i)) seen = word_flag(w[i]);
        record_wait_error(a.err, 5u, t, r, g, p, seen, flag);
        return false;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kLLMaxE; ++k) {
    const int64_t pos = pos0 + (int64_t)k * blockDim.x;
    if (k < a.E && pos < len) {
      uint64_t b = (uint32_t)w[k * WPE];
      if (WPE == 2) b |= (uint64_t)(uint32_t)w[k * WPE + WPE - 1] << 32;
      val[k] = from_raw<T>(b);
    }
  }
  return true;
}

template <class D, int OP>
__global__ void __launch_bounds__(kLLThreads, 4) ll_kernel(const LLArgs a) {
  using T = typename D::T;
  constexpr int WPE = sizeof(T) == 8 ? 2 : 1;
  const int R = a.R, E = a.E;
  const int r = blockIdx.x % R;
  const int g = blockIdx.x / R;
  const int p = (r == 0) ? R - 1 : r - 1;
  const int q = (r == R - 1) ? 0 : r + 1;
  const int64_t row = a.plan.C * WPE;
  const int64_t pos0 = (int64_t)g * blockDim.x * E + threadIdx.x;
  const T* in_r = static_cast<const T*>(a.p.in[r]);
  T* out_r = static_cast<T*>(a.p.out[r]);
  for (int t = 0; t < a.rounds; ++t) {
    bool reduce;
    int s;
    if (a.mode == kModeAllGather) {
      reduce = false;
      s = t + 1;
    } else if (t < R - 1) {
      reduce = true;
      s = t + 1;
    } else {
      reduce = false;
      s = t - (R - 1) + 1;
    }
    int c = reduce ? (r - s) : (r + 1 - s);
    c %= R;
    if (c < 0) c += R;
    const int64_t off = min((int64_t)c * a.plan.C, a.plan.n);
    const int64_t len = min(off + a.plan.C, a.plan.n) - off;
    T own[kLLMaxE];
    T val[kLLMaxE];
    // the local piece first: it does not wait for the predecessor
    if (reduce) {
#pragma unroll
      for (int k = 0; k < kLLMaxE; ++k) {
        const int64_t pos = pos0 + (int64_t)k * blockDim.x;
        if (k < E && pos < len) own[k] = ld_l2_scalar(in_r + off + pos);
      }
    }
    if (t == 0) {
      // round 1 reads the predecessor's input (its owned chunk in AllGather)
      const T* src = static_cast<const T*>(reduce ? a.p.in[p] : a.p.out[p]);
#pragma unroll
      for (int k = 0; k < kLLMaxE; ++k) {
        const int64_t pos = pos0 + (int64_t)k * blockDim.x;
        if (k < E && pos < len) val[k] = ld_l2_scalar(src + off + pos);
      }
    } else {
      const uint64_t* box = a.inbox + ((int64_t)(t - 1) * R + r) * row;
      if (!ll_receive<T, WPE>(a, box, pos0, len, a.flag_base + (uint32_t)(t - 1), val, t, r, g, p)) return;
    }
    if (reduce) {
#pragma unroll
      for (int k = 0; k < kLLMaxE; ++k) {
        const int64_t pos = pos0 + (int64_t)k * blockDim.x;
        if (k < E && pos < len) val[k] = Op<D, OP>::apply(val[k], own[k]);
      }
    }
    // send before writing the output: the successor is waiting for it.
    // Failure injection: a rank that is to fall silent sends nothing from
    // round skip_round on.
    if (t + 1 < a.rounds && !(r == a.skip_rank && t >= a.skip_round)) {
      uint64_t* box = a.inbox + ((int64_t)t * R + q) * row;
      const uint64_t f = (uint64_t)(a.flag_base + (uint32_t)t) << 32;
#pragma unroll
      for (int k = 0; k < kLLMaxE; ++k) {
        const int64_t pos = pos0 + (int64_t)k * blockDim.x;
        if (k < E && pos < len) {
          const uint64_t b = raw_bits(val[k]);
          signal_store_relaxed(box + pos * WPE, f | (b & 0xFFFFFFFFull));
          if (WPE == 2) signal_store_relaxed(box + pos * WPE + WPE - 1, f | (b >> 32));
        }
      }
    }
    // complete values: the owner's chunk after the last reduce round, every
    // chunk of the copy rounds
    if (!reduce || s == R - 1) {
#pragma unroll
      for (int k = 0; k < kLLMaxE; ++k) {
        const int64_t pos = pos0 + (int64_t)k * blockDim.x;
        if (k < E && pos < len) st_g(out_r + off + pos, val[k]);
      }
    }
  }
}

const void* ll_select(int dtype, int op) {
  const void* fn = nullptr;
  with_dtype_op(dtype, op, [&](auto d, auto o) {
    fn = reinterpret_cast<const void*>(&ll_kernel<decltype(d), decltype(o)::value>);
    return cudaSuccess;
  });
  return fn;
}

}  // namespace

cudaError_t ll_blocks_per_sm(int dtype, int op, int threads, int* blocks) {
  const void* fn = ll_select(dtype, op);
  if (!fn) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, threads, 0);
}

cudaError_t launch_ll(int dtype, int op, const LLArgs& a, int threads, cudaStream_t st) {
  const void* fn = ll_select(dtype, op);
  if (!fn || a.R < 2 || a.R > kMaxRanks || a.G < 1 || a.E < 1 || a.E > kLLMaxE || threads < 32 ||
      threads > kLLThreads || threads % 32 != 0 || a.rounds < 1 || !a.inbox || !a.err ||
      (int64_t)a.G * threads * a.E < a.plan.C)
    return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<LLArgs*>(&a)};
  return cudaLaunchCooperativeKernel(fn, dim3(a.R * a.G), dim3(threads), args, 0, st);
}

}  // namespace ra
