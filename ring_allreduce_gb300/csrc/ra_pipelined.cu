// ra_pipelined.cu -- the pipelined variant: every ring round in one
// cooperative launch, and no barrier -- each rank waits only for its
// predecessor, one sub-slice at a time.
//
// "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce",
// section 4: a rank receives only from its predecessor.  So instead of
// stopping every rank at a barrier after each round, rank r starts round T on
// a piece of its chunk as soon as rank r-1 has finished round T-1 on the
// same piece.  The pieces: CTA g of each rank (channel g) owns the g-th slice
// of the round's chunk, cut into J sub-slices; each (channel, rank, sub-slice)
// has a progress flag holding how many rounds that rank has finished on it.
// Different sub-slices of one rank can be in different rounds, so rounds
// overlap along the ring, as NCCL pipelines a ring by slices.
//
// Order of the work: the sub-slices are taken W at a time (a window), and a
// rank runs every round on a window before it starts the next one.  The
// partial a rank writes for its successor in round t is then read a window's
// round later instead of a whole slice's round later -- while it is still in
// L2 -- and the place it is later overwritten with the complete value is
// written again within 2(R-1) window rounds.  Within a window, the wait for
// one sub-slice overlaps the work on the others.  W = J is the round-by-round
// order.  The order changes nothing in the protocol below: every wait is on
// one sub-slice and one round, whatever was done before it.
//
// Why waiting on the predecessor alone is safe.  A rank's output buffer is
// the "message" its successor reads, and one place of it is written twice:
// chunk (r - t) holds the partial of ReduceScatter round t and, R rounds
// later (AllGather round t + 1), the complete value.  Rank r can start round
// T only once rank r-1 has finished round T-1, which needed rank r-2 to have
// finished T-2, and so on round the ring to rank r+1 having finished
// T-(R-1).  For T = R + t that is round t + 1, in which r+1 read the partial:
// the overwrite can never overtake the read it would spoil.  Reads of inputs
// in round 1 need no wait at all.
//
// Flags are signals of the signal layer (ra_signal.cuh): a rank publishes a
// finished round with SignalAdd(1) on its flag of the sub-slice.  The waiter
// keeps a shadow of each predecessor flag it waits on -- in a register during
// the launch, in device memory between calls -- moved forward by 1 per round
// (increaseSignalShadow), and waits for the flag to meet it
// (waitSignalMeetShadow), in rolling order on the low RA_OPT_SIGNAL_BITS
// bits.  After every call shadow == flag == its start value + calls x rounds,
// and nothing is cleared between calls.  Waits are bounded; one that runs out
// records (round, rank, channel, predecessor, observed, expected) and the CTA
// returns, and every other waiter returns at its next poll.  Data another CTA
// wrote is read through L2.
#include "ra_signal.cuh"

namespace ra {

// Thread 0 waits until the predecessor's flag of the sub-slice meets its
// shadow of it, which stands `t` rounds past where it started the call
// (moved forward by one per round: increaseSignalShadow); false when the
// CTA must stop.
__device__ __forceinline__ bool wait_flag(const PersistArgs& a, const uint64_t* flag, sig::Shadow start, int t, int r,
                                          int g, int pred, int* s_abort) {
  if (threadIdx.x == 0) {
    sig::Shadow shadow = start;
    sig::increase_shadow(shadow, (uint64_t)t);
    uint64_t seen = 0;
    const sig::Wait w = sig::wait_meet_shadow(flag, shadow, a.bits, a.timeout_ns, &a.err->code, &seen);
    if (w == sig::kTimedOut) record_wait_error(a.err, 4u, t, r, g, pred, seen, sig::low_bits(shadow.v, a.bits));
    *s_abort = w != sig::kReached;
  }
  __syncthreads();
  return *s_abort == 0;
}

// All threads' stores of the sub-slice are done; thread 0 publishes the
// finished round (SignalAdd of 1).
__device__ __forceinline__ void publish_flag(uint64_t* flag, bool withhold) {
  __syncthreads();
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();   // release
    if (!withhold) sig::add(flag, 1);
  }
}

// `dead_inc`: the incoming data is the predecessor's partial, which nobody
// reads again before the complete value overwrites it in AllGather; its L2
// lines are dropped once read instead of being written back to DRAM.
template <class D, int OP>
__device__ __forceinline__ void reduce_range(const typename D::T* inc, const typename D::T* loc, typename D::T* dst,
                                             int64_t qb, int64_t qe, const Span<D::kVec>& sp, bool scalars,
                                             bool dead_inc) {
  const uint4* inc4 = reinterpret_cast<const uint4*>(inc);
  const int lane = threadIdx.x & 31;
  for (int64_t w = qb + (threadIdx.x - lane); w < qe; w += blockDim.x) {
    const int64_t v = w + lane;
    if (v < qe) {
      const uint4 x = ld_l2(inc4 + v);
      const uint4 y = ld_l2(reinterpret_cast<const uint4*>(loc) + v);
      st_l2(reinterpret_cast<uint4*>(dst) + v, combine_vec<D, OP>(x, y));
    }
    if (dead_inc) discard_read_lines(inc4 + w, qe - w < 32 ? qe - w : 32);
  }
  if (scalars) {
    const int64_t ns = sp.scalar_count();
    for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
      const int64_t i = sp.scalar_at(t);
      st_g(dst + i, Op<D, OP>::apply(ld_l2_scalar(inc + i), ld_l2_scalar(loc + i)));
    }
  }
}

template <class D>
__device__ __forceinline__ void copy_range(const typename D::T* src, typename D::T* dst, int64_t qb, int64_t qe,
                                           const Span<D::kVec>& sp, bool scalars) {
  for (int64_t v = qb + threadIdx.x; v < qe; v += blockDim.x)
    st_l2(reinterpret_cast<uint4*>(dst) + v, ld_l2(reinterpret_cast<const uint4*>(src) + v));
  if (scalars) {
    const int64_t ns = sp.scalar_count();
    for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
      const int64_t i = sp.scalar_at(t);
      st_g(dst + i, ld_l2_scalar(src + i));
    }
  }
}

// FROM_MEMORY: the instantiation for launches a CUDA graph replays, which
// read the shadow start back from device memory; launches from the host run
// the other one, whose code does not carry that path at all.  The channels
// are sized from the host instantiation's co-resident CTAs; the other is
// held to 4 CTAs of 512 threads per SM (32 registers), at least as many as
// the host one allows for any element type, so the same grid fits both.
template <class D, int OP, bool FROM_MEMORY>
__global__ void __launch_bounds__(kPipeThreads, FROM_MEMORY ? 4 : 3)
pipelined_kernel(const PersistArgs a) {
  using T = typename D::T;
  constexpr int V = D::kVec;
  __shared__ int s_abort;
  const int R = a.R, G = a.G, J = a.J;
  const int r = blockIdx.x % R;
  const int g = blockIdx.x / R;
  const int p = (r == 0) ? R - 1 : r - 1;
  uint64_t* mine = a.slots + ((int64_t)g * R + r) * J;
  const uint64_t* pred = a.slots + ((int64_t)g * R + p) * J;
  // Waiter r's shadows of the predecessor's J flags.  They start every call
  // equal -- reset or seeded together, each moved by the call's rounds -- at
  // a value the host keeps with the flags and passes in (a.shadow_base), so
  // the waiter holds its shadow in a register for the launch (reading it
  // back from device memory here measured 5-12 % slower calls on GB300; a
  // launch a CUDA graph replays does read it back: from_memory).
  // Thread j keeps the copy of sub-slice j in device memory where it stands
  // after the call -- moved past every round's publication, the last one
  // too, which nobody waits on -- since nothing reads it during the launch.
  sig::Shadow start{a.shadow_base};
  if (FROM_MEMORY) {
    // a launch a CUDA graph replays: the start is where this waiter's own
    // shadows stand (all J alike; only this CTA writes them)
    __shared__ uint64_t s_start;
    if (threadIdx.x == 0) s_start = sig::load_shadow(a.shadows + ((int64_t)g * R + r) * J).v;
    __syncthreads();
    start = sig::Shadow{s_start};
  }
  if (threadIdx.x < J) {
    sig::Shadow s = start;
    sig::increase_shadow(s, (uint64_t)a.rounds);
    sig::store_shadow(a.shadows + ((int64_t)g * R + r) * J + threadIdx.x, s);
  }
  for (int w0 = 0; w0 < J; w0 += a.W) {
    const int w1 = min(J, w0 + a.W);
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
      const int64_t end = min(off + a.plan.C, a.plan.n);
      const Span<V> sp(off, end);
      // failure injection: a flag counts finished rounds, so a rank that is
      // to fall silent withholds every publication from that round on
      const bool withhold = (r == a.skip_rank && t >= a.skip_round);
      for (int j = w0; j < w1; ++j) {
        // sub-slice j of channel g: slice g J + j of the chunk cut in G J
        int64_t qb, qe;
        split_vectors(sp.vb, sp.ve, g * J + j, G * J, &qb, &qe);
        // round 0 reads inputs only; every later round reads what the
        // predecessor wrote in its previous round on this sub-slice
        if (t > 0 && !wait_flag(a, pred + j, start, t, r, g, p, &s_abort)) return;
        const bool scalars = (g == 0 && j == 0);
        if (off < end) {
          if (reduce) {
            const T* inc = static_cast<const T*>(s == 1 ? a.p.in[p] : a.p.out[p]);
            reduce_range<D, OP>(inc, static_cast<const T*>(a.p.in[r]), static_cast<T*>(a.p.out[r]), qb, qe, sp,
                                scalars, s != 1);
          } else {
            copy_range<D>(static_cast<const T*>(a.p.out[p]), static_cast<T*>(a.p.out[r]), qb, qe, sp, scalars);
          }
        }
        publish_flag(mine + j, withhold);
      }
    }
  }
}

static const void* pipelined_select(int dtype, int op, bool from_memory) {
  const void* fn = nullptr;
  with_dtype_op(dtype, op, [&](auto d, auto o) {
    using D = decltype(d);
    constexpr int OP = decltype(o)::value;
    fn = from_memory ? reinterpret_cast<const void*>(&pipelined_kernel<D, OP, true>)
                     : reinterpret_cast<const void*>(&pipelined_kernel<D, OP, false>);
    return cudaSuccess;
  });
  return fn;
}

// Co-resident CTAs of the host instantiation (the replay one fits as many).
cudaError_t pipelined_blocks_per_sm(int dtype, int op, int threads, int* blocks) {
  const void* fn = pipelined_select(dtype, op, false);
  if (!fn) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, threads, 0);
}

cudaError_t launch_pipelined(int dtype, int op, const PersistArgs& a, int threads, cudaStream_t st) {
  const void* fn = pipelined_select(dtype, op, a.from_memory != 0);
  if (!fn || a.R < 2 || a.R > kMaxRanks || a.G < 1 || a.J < 1 || a.J > kPipeMaxSlices || a.W < 1 || a.rounds < 1 ||
      !a.shadows)
    return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<PersistArgs*>(&a)};
  return cudaLaunchCooperativeKernel(fn, dim3(a.R * a.G), dim3(threads), args, 0, st);
}

}  // namespace ra
