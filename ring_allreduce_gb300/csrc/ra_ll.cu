// ra_ll.cu -- the pipelined variant with flag-in-data messages
// (RA_OPT_PROTOCOL = RA_PROTOCOL_LL or RA_PROTOCOL_LL_CLUSTER), for chunks
// small enough that a ring round is a chain of memory latencies rather than
// a stream of bytes.
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
// carries 32 bits of data together with a 32-bit flag naming the message,
// written by one 8-byte store (single-copy atomic): the receiver polls the
// data words themselves, and a word whose flag is the expected one holds the
// expected data.  A hop is then one store and the poll that sees it, with no
// fence, no separate signal and no CTA barrier: thread k of a receiving CTA
// depends only on thread k of the sending CTA, which carries the same
// positions of the same chunk.  This is the low-latency message form of
// NCCL's ring (flags inside the data), which the pages do not describe.  The
// price is twice the bytes per element (four times for 16-bit elements), so
// it is for small chunks only.
//
// Two transports:
//  * LL: rows of an inbox in device memory, one per (message, receiving
//    rank), each written once per call, so no word is overwritten while
//    someone may still read it.  Flags grow by one per message and by the
//    call's rounds per call (the host restarts them, zeroing the inbox,
//    before they would wrap), so a word left from any earlier call or round
//    never carries the flag being waited for.  One cooperative launch (every
//    channel's CTAs wait on each other's messages).
//  * LL_CLUSTER: the R CTAs of a channel form one thread-block cluster, and
//    a message word is stored straight into the successor's shared memory
//    (distributed shared memory, st.relaxed.cluster), which the successor
//    polls locally: the hop stays inside one GPC instead of going through
//    L2.  Each CTA zeroes its rows and the cluster meets once before any
//    message is sent, so message m carries flag m + 1 in every launch and
//    nothing is kept between calls (a CUDA graph may replay the launch); the
//    cluster meets again before any CTA exits, so no store reaches the
//    shared memory of a CTA that has left.  Channels are independent
//    clusters: no cooperative launch.
//
// Outputs are written only with complete values (the owner's chunk after
// the last reduce round, every chunk in the copy rounds), and each is
// written by the thread that read the same element of the same rank's input
// earlier, or (a rank's chunk r read by its successor in the first round) at
// the end of a chain of messages each of which carries a value computed from
// that read: in place calls are safe.
//
// Waits are bounded (timeout_ns, two clocks); one that runs out records code
// 5 (round, rank, channel, predecessor, flag seen, flag expected) and the
// thread stops; every other waiter stops once it sees the record.  A
// replayed LL launch whose flags would wrap records code 6 and does nothing.
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

// ------------------------------------------------------------ transports
// A transport gives the row a rank receives message m in (already at this
// channel's first position) and stores a word into the successor's row.

struct GlobalInbox {
  uint64_t* inbox;
  int64_t row;        // words of one (message, rank) row: C * wpe
  int64_t chan;       // this channel's first word in a row
  int R, r, q;
  uint32_t flag_base;
  __device__ __forceinline__ const uint64_t* recv_row(int m) const {
    return inbox + ((int64_t)m * R + r) * row + chan;
  }
  __device__ __forceinline__ uint64_t load(const uint64_t* w) const { return signal_load_relaxed(w); }
  __device__ __forceinline__ void store(int m, int64_t word, uint64_t v) const {
    signal_store_relaxed(inbox + ((int64_t)m * R + q) * row + chan + word, v);
  }
  __device__ __forceinline__ uint32_t flag(int m) const { return flag_base + (uint32_t)m; }
  // polls between looks at the clocks and the error record; polls after
  // which each one sleeps (a poll is a round trip through L2)
  static constexpr uint32_t kCheckEvery = 8;
  static constexpr uint32_t kSleepAfter = 64;
};

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(v));
  return v;
}

// Every thread of the cluster; not .aligned: threads may arrive from
// different points of a loop they left early.
__device__ __forceinline__ void cluster_meet() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

struct ClusterInbox {
  uint64_t* box;      // this CTA's rows in shared memory: [message][P * wpe]
  int64_t row;        // words of one row
  uint32_t q;         // the successor's rank in the cluster
  uint32_t remote;    // the successor's rows, as a shared::cluster address
  __device__ __forceinline__ const uint64_t* recv_row(int m) const { return box + (int64_t)m * row; }
  __device__ __forceinline__ uint64_t load(const uint64_t* w) const {
    uint64_t v;
    asm volatile("ld.relaxed.cluster.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(smem_addr(w)) : "memory");
    return v;
  }
  // the same word of the successor's rows (every CTA lays its rows out
  // alike, and a CTA's shared memory maps linearly into the cluster window)
  __device__ __forceinline__ void store(int m, int64_t word, uint64_t v) const {
    const uint32_t at = remote + (uint32_t)(((int64_t)m * row + word) * sizeof(uint64_t));
    asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" ::"r"(at), "l"(v) : "memory");
  }
  __device__ __forceinline__ uint32_t flag(int m) const { return (uint32_t)m + 1u; }
  // a poll of shared memory is short next to a look at the clocks or a load
  // of the error record, and occupies nothing but this SM: no sleeping
  static constexpr uint32_t kCheckEvery = 32;
  static constexpr uint32_t kSleepAfter = 0;
};

// Positions a thread carries: local k*blockDim.x + tid for k < EM (a
// compile-time bound, 1 or kLLMaxE) and k < a.E, valid below `lim` (at most
// EM*blockDim.x, so 32 bits hold every local position).
template <int EM>
__device__ __forceinline__ bool carries(const LLArgs& a, int k, int lim) {
  return (EM == 1 || k < a.E) && k * (int)blockDim.x + (int)threadIdx.x < lim;
}

// Poll the words of this thread's positions in `row` until each carries
// `flag`; the data into val[].  False when the thread must stop.
template <class T, int WPE, int EM, class Tr>
__device__ __forceinline__ bool ll_receive(const LLArgs& a, const Tr& tr, const uint64_t* row, int lim,
                                           uint32_t flag, T* val, int t, int r, int g, int p) {
  uint64_t w[EM * WPE];
  uint32_t pending = 0;
#pragma unroll
  for (int k = 0; k < EM; ++k) {
    if (carries<EM>(a, k, lim)) {
      const int loc = k * (int)blockDim.x + (int)threadIdx.x;
#pragma unroll
      for (int h = 0; h < WPE; ++h) {
        w[k * WPE + h] = tr.load(row + loc * WPE + h);
        if (word_flag(w[k * WPE + h]) != flag) pending |= 1u << (k * WPE + h);
      }
    }
  }
  if (pending) {
    // Off the fast path: the clocks start at the first look, not the first
    // poll, and the error record is loaded one look ahead of its test, so
    // its trip overlaps polls.  The bound is the limit plus one look.
    uint64_t t0 = 0, c0 = 0;
    uint32_t stop = 0;
    for (uint32_t it = 0;; ++it) {
      if (Tr::kSleepAfter && it >= Tr::kSleepAfter) __nanosleep(64);
#pragma unroll
      for (int i = 0; i < EM * WPE; ++i) {
        if (pending & (1u << i)) {
          const int loc = (i / WPE) * (int)blockDim.x + (int)threadIdx.x;
          w[i] = tr.load(row + loc * WPE + (i % WPE));
          if (word_flag(w[i]) == flag) pending &= ~(1u << i);
        }
      }
      if (!pending) break;
      if (it % Tr::kCheckEvery != Tr::kCheckEvery - 1) continue;
      if (stop != 0u) return false;
      stop = load_relaxed_u32(&a.err->code);
      if (it == Tr::kCheckEvery - 1) {
        t0 = globaltimer_ns();
        c0 = sm_cycles();
        continue;
      }
      const int64_t cycles = a.timeout_ns > ((int64_t)1 << 60) ? ((int64_t)1 << 62) : 3 * a.timeout_ns;
      if ((int64_t)(globaltimer_ns() - t0) > a.timeout_ns || (int64_t)(sm_cycles() - c0) > cycles) {
        uint32_t seen = 0;
#pragma unroll
        for (int i = EM * WPE - 1; i >= 0; --i)
          if (pending & (1u << i)) seen = word_flag(w[i]);
        record_wait_error(a.err, 5u, t, r, g, p, seen, flag);
        return false;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < EM; ++k) {
    if (carries<EM>(a, k, lim)) {
      uint64_t b = (uint32_t)w[k * WPE];
      if (WPE == 2) b |= (uint64_t)(uint32_t)w[k * WPE + WPE - 1] << 32;
      val[k] = from_raw<T>(b);
    }
  }
  return true;
}

// Every ring round of rank r, channel g, over this thread's positions
// chan0 + k*blockDim.x + tid of each chunk; false if a wait gave up.
template <class D, int OP, int EM, class Tr>
__device__ __forceinline__ bool ll_rounds(const LLArgs& a, const Tr& tr, int r, int g) {
  using T = typename D::T;
  constexpr int WPE = sizeof(T) == 8 ? 2 : 1;
  const int R = a.R;
  const int p = (r == 0) ? R - 1 : r - 1;
  const int span = EM == 1 ? (int)blockDim.x : a.E * (int)blockDim.x;   // positions of a channel
  const int64_t chan0 = (int64_t)g * span;
  const int64_t C = a.plan.C, n = a.plan.n;
  const T* in_r = static_cast<const T*>(a.p.in[r]);
  T* out_r = static_cast<T*>(a.p.out[r]);
  const bool gather = a.mode == kModeAllGather;
  // The chunk of round t steps back round the ring by one every round:
  // ReduceScatter round s = t + 1 takes chunk r - s and the copy rounds that
  // follow it chunk r + 1 - s' (s' = t - R + 2), i.e. r - 1 - t throughout;
  // an AllGather on its own (s = t + 1) takes r - t.  Kept by one decrement
  // a round, as is the channel's first element in it: the time between a
  // send and the next poll is on the ring's critical path.
  int c = gather ? r : (r == 0 ? R - 1 : r - 1);
  int64_t first = (int64_t)c * C + chan0;
  for (int t = 0; t < a.rounds; ++t) {
    const bool reduce = !gather && t < R - 1;
    const bool complete = !reduce || t == R - 2;   // the owner's chunk after the last reduce round
    // positions of this channel in chunk c: local < lim (chunk end - first,
    // clamped to the channel's span)
    const int64_t left = min((int64_t)(c + 1) * C, n) - first;
    const int lim = left <= 0 ? 0 : (left < span ? (int)left : span);
    T own[EM];
    T val[EM];
    // the local piece first: it does not wait for the predecessor
    if (reduce) {
      const T* src = in_r + first;
#pragma unroll
      for (int k = 0; k < EM; ++k)
        if (carries<EM>(a, k, lim)) own[k] = ld_l2_scalar(src + k * (int)blockDim.x + (int)threadIdx.x);
    }
    if (t == 0) {
      // round 1 reads the predecessor's input (its owned chunk in AllGather)
      const T* src = static_cast<const T*>(reduce ? a.p.in[p] : a.p.out[p]) + first;
#pragma unroll
      for (int k = 0; k < EM; ++k)
        if (carries<EM>(a, k, lim)) val[k] = ld_l2_scalar(src + k * (int)blockDim.x + (int)threadIdx.x);
    } else if (!ll_receive<T, WPE, EM>(a, tr, tr.recv_row(t - 1), lim, tr.flag(t - 1), val, t, r, g, p)) {
      return false;
    }
    if (reduce) {
#pragma unroll
      for (int k = 0; k < EM; ++k)
        if (carries<EM>(a, k, lim)) val[k] = Op<D, OP>::apply(val[k], own[k]);
    }
    // send before writing the output: the successor is waiting for it.
    // Failure injection: a rank that is to fall silent sends nothing from
    // round skip_round on.
    if (t + 1 < a.rounds && !(r == a.skip_rank && t >= a.skip_round)) {
      const uint64_t f = (uint64_t)tr.flag(t) << 32;
#pragma unroll
      for (int k = 0; k < EM; ++k) {
        if (carries<EM>(a, k, lim)) {
          const int loc = k * (int)blockDim.x + (int)threadIdx.x;
          const uint64_t b = raw_bits(val[k]);
          tr.store(t, (int64_t)loc * WPE, f | (b & 0xFFFFFFFFull));
          if (WPE == 2) tr.store(t, (int64_t)loc * WPE + WPE - 1, f | (b >> 32));
        }
      }
    }
    // complete values: the owner's chunk after the last reduce round, every
    // chunk of the copy rounds
    if (complete) {
      T* dst = out_r + first;
#pragma unroll
      for (int k = 0; k < EM; ++k)
        if (carries<EM>(a, k, lim)) st_g(dst + k * (int)blockDim.x + (int)threadIdx.x, val[k]);
    }
    if (c == 0) {
      c = R - 1;
      first += (int64_t)(R - 1) * C;
    } else {
      --c;
      first -= C;
    }
  }
  return true;
}

template <class D, int OP, int EM>
__global__ void __launch_bounds__(kLLThreads, 3) ll_kernel(const LLArgs a) {
  constexpr int WPE = sizeof(typename D::T) == 8 ? 2 : 1;
  const int r = blockIdx.x % a.R;
  const int g = blockIdx.x / a.R;
  // The flag base.  Each CTA keeps its own copy of the flag its next call
  // starts at, in device memory, and moves it on itself (no other CTA reads
  // it): a launch from the host is handed the base and writes the next one
  // down; a launch a CUDA graph replays (from_memory) takes its base from
  // there -- 0, never written, is 1 on the inbox zeroed when it was made --
  // and gives up with code 6, touching nothing, when its flags would pass
  // 2^32 - 1 (every CTA holds the same value, so every CTA gives up).
  uint32_t base = a.flag_base;
  if (a.from_memory) {
    __shared__ uint32_t s_base;
    if (threadIdx.x == 0) {
      uint64_t next = (uint64_t)ld_l2_scalar(reinterpret_cast<const int64_t*>(a.bases + blockIdx.x));
      if (next == 0) next = 1;
      if (next + (uint64_t)a.rounds > 0xFFFFFFFFull) {
        record_wait_error(a.err, 6u, 0, r, g, -1, next, 0xFFFFFFFFull);
        next = 0;
      }
      s_base = (uint32_t)next;
    }
    __syncthreads();
    base = s_base;
    if (base == 0) return;
  }
  {
    // the next base: this CTA's copy; a launch from the host also sets the
    // copies of the CTAs beyond its grid (CTA 0's threads), so that every
    // copy agrees whatever grid a later launch has
    const unsigned long long nb = (unsigned long long)base + (unsigned long long)a.rounds;
    auto put = [&](int i) {
      if (RA_ACCESS_OK(a.bases + i, 8u, 2u)) __stcg(reinterpret_cast<unsigned long long*>(a.bases + i), nb);
    };
    if (threadIdx.x == 0) put((int)blockIdx.x);
    if (!a.from_memory && blockIdx.x == 0)
      for (int i = (int)gridDim.x + (int)threadIdx.x; i < a.nbases; i += (int)blockDim.x) put(i);
  }
  GlobalInbox tr;
  tr.inbox = a.inbox;
  tr.row = a.plan.C * WPE;
  tr.chan = (int64_t)g * blockDim.x * (EM == 1 ? 1 : a.E) * WPE;
  tr.R = a.R;
  tr.r = r;
  tr.q = (r == a.R - 1) ? 0 : r + 1;
  tr.flag_base = base;
  ll_rounds<D, OP, EM>(a, tr, r, g);
}

template <class D, int OP, int EM>
__global__ void __launch_bounds__(kLLThreads, 1) ll_cluster_kernel(const LLArgs a) {
  constexpr int WPE = sizeof(typename D::T) == 8 ? 2 : 1;
  extern __shared__ __align__(16) uint64_t ll_box[];
  const int r = (int)cluster_cta_rank();   // blockIdx.x = g R + r
  const int g = blockIdx.x / a.R;
  ClusterInbox tr;
  tr.box = ll_box;
  tr.row = (int64_t)blockDim.x * (EM == 1 ? 1 : a.E) * WPE;
  tr.q = (uint32_t)((r == a.R - 1) ? 0 : r + 1);
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(tr.remote) : "r"(smem_addr(ll_box)), "r"(tr.q));
  // zero this CTA's rows, then meet: no peer stores into them before
  const int64_t words = (int64_t)(a.rounds - 1) * tr.row;
  for (int64_t i = threadIdx.x; i < words; i += blockDim.x) ll_box[i] = 0;
  cluster_meet();
  ll_rounds<D, OP, EM>(a, tr, r, g);
  // nobody leaves while a peer may still store into its rows
  cluster_meet();
}

// The instantiation for E positions per thread: one position (the usual
// small call) has code of its own, without the loops over positions.
const void* ll_fn(int dtype, int op, int E) {
  const void* fn = nullptr;
  with_dtype_op(dtype, op, [&](auto d, auto o) {
    using D = decltype(d);
    constexpr int OP = decltype(o)::value;
    fn = E == 1 ? reinterpret_cast<const void*>(&ll_kernel<D, OP, 1>)
                : reinterpret_cast<const void*>(&ll_kernel<D, OP, kLLMaxE>);
    return cudaSuccess;
  });
  return fn;
}

const void* ll_cluster_fn(int dtype, int op, int E) {
  const void* fn = nullptr;
  with_dtype_op(dtype, op, [&](auto d, auto o) {
    using D = decltype(d);
    constexpr int OP = decltype(o)::value;
    fn = E == 1 ? reinterpret_cast<const void*>(&ll_cluster_kernel<D, OP, 1>)
                : reinterpret_cast<const void*>(&ll_cluster_kernel<D, OP, kLLMaxE>);
    return cudaSuccess;
  });
  return fn;
}

bool ll_shape_ok(const LLArgs& a, int threads) {
  return a.R >= 2 && a.R <= kMaxRanks && a.G >= 1 && a.E >= 1 && a.E <= kLLMaxE && threads >= 32 &&
         threads <= kLLThreads && threads % 32 == 0 && a.rounds >= 1 && a.err &&
         (int64_t)a.G * threads * a.E >= a.plan.C;
}

cudaLaunchConfig_t ll_cluster_config(const LLArgs& a, int threads, size_t smem, cudaStream_t st,
                                     cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.R * a.G);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.R;   // CTA (r, g) = blockIdx.x = g R + r: rank r of cluster g
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t ll_blocks_per_sm(int dtype, int op, int threads, int* blocks) {
  const void* fn = ll_fn(dtype, op, kLLMaxE);   // the larger register count of the two
  if (!fn) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, threads, 0);
}

cudaError_t launch_ll(int dtype, int op, const LLArgs& a, int threads, cudaStream_t st) {
  const void* fn = ll_fn(dtype, op, a.E);
  if (!fn || !ll_shape_ok(a, threads) || !a.inbox || !a.bases || a.R * a.G > a.nbases) return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<LLArgs*>(&a)};
  return cudaLaunchCooperativeKernel(fn, dim3(a.R * a.G), dim3(threads), args, 0, st);
}

size_t ll_cluster_smem_bytes(const LLArgs& a, int threads, int elem_bytes) {
  const size_t rows = a.rounds > 1 ? (size_t)(a.rounds - 1) : 1;
  return rows * (size_t)threads * (size_t)a.E * (size_t)ll_words_per_element(elem_bytes) * sizeof(uint64_t);
}

cudaError_t prepare_ll_cluster() {
  cudaError_t err = cudaSuccess;
  for (int dt = RA_F32; dt <= RA_I64 && err == cudaSuccess; ++dt)
    for (int op = RA_SUM; op <= RA_MAX && err == cudaSuccess; ++op)
      for (int E : {1, kLLMaxE}) {
        const void* fn = ll_cluster_fn(dt, op, E);
        if (err == cudaSuccess) err = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err == cudaSuccess)
          err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kLLClusterMaxSmem);
      }
  return err;
}

cudaError_t ll_cluster_capacity(int dtype, int op, const LLArgs& a, int threads, size_t smem, int* clusters) {
  const void* fn = ll_cluster_fn(dtype, op, a.E);
  if (!fn || a.R < 2 || a.R > 16) return cudaErrorInvalidValue;
  LLArgs one = a;
  one.G = 1;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = ll_cluster_config(one, threads, smem, 0, attr);
  return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

cudaError_t launch_ll_cluster(int dtype, int op, const LLArgs& a, int threads, size_t smem, cudaStream_t st) {
  const void* fn = ll_cluster_fn(dtype, op, a.E);
  if (!fn || !ll_shape_ok(a, threads) || a.R > 16 || smem > (size_t)kLLClusterMaxSmem ||
      smem < ll_cluster_smem_bytes(a, threads, a.elem_bytes))
    return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = ll_cluster_config(a, threads, smem, st, attr);
  void* args[] = {const_cast<LLArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace ra
