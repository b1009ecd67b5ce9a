// ra_persistent.cu -- the persistent variant: every ring round in one
// cooperative launch, simulated ranks meeting at a counting barrier
// between rounds.
//
// Rounds ("Why AllReduce = ReduceScatter + AllGather -- NCCL Ring
// AllReduce", sections 5 and 6): ReduceScatter round s computes, on every
// rank r, P_r[c] = P_{r-1}[c] (+) x_r[c] with c = (r - s) mod R; AllGather
// round s copies chunk (r + 1 - s) mod R from rank r-1.  The partial a rank
// passes on is what it stored in its output buffer.
//
// Ranks and channels: the launch has R x G CTAs.  CTA (r, g) is rank r's
// channel g: in every round it handles the g-th slice of its rank's chunk.
// Slices are cut from the chunk alone, so channel g of rank r only ever
// reads what channel g of rank r-1 wrote: each channel is a ring of its own,
// as NCCL runs several rings side by side.
//
// Barrier between rounds ("comm: lift the GIN scale-out ceiling by making
// the rail barrier a counting barrier", section "Fix"): after a round each
// CTA adds 1 to one signal of every peer of its channel (release, so its
// round's stores are visible with the count), then polls its own signal
// (acquire) until the shadow target is reached, and a __syncthreads lets
// the rest of the CTA on.  The page's section "Scoped to the rail team,
// deliberately" explains that a single counter reused across rounds lets a
// peer a round ahead stand in for a late one; here every (channel, round,
// waiter) has its own 64-bit slot, so a count comes only from its round.
// Release takes the fence form (one fence.acq_rel.gpu before the R-1
// relaxed adds); the poll uses acquire loads.
// Signals and shadows are never cleared between calls: each waiter's shadow
// moves by R-1 per call and the signal is compared with it in 64-bit rolling
// order (NCCL Device API GIN article, signals and counters; the signal layer
// is ra_signal.cuh).
//
// With RA_BARRIER_CLUSTER the R CTAs of a channel are launched as one
// thread-block cluster and meet at the hardware cluster barrier instead
// (R <= 16; no cooperative launch needed, as no cluster waits on another).
//
// Passes: a channel's slice may be cut into J sub-slices that each go
// through every round, with its own barrier rounds, before the next one
// starts (J = 1: every round over the whole slice).  The partial a rank
// writes in a round is then still in L2 when its successor reads it in the
// next.  The passes touch disjoint elements, so no barrier separates them;
// each (channel, pass, round) has its own slots.
//
// No wait is unbounded: a poll that passes the time limit records
// (round, rank, channel, observed, expected) in the handle's error record and
// the CTA returns; every other CTA sees the record at its next poll and
// returns as well.  Data produced by another CTA of the launch is read
// through L2 (ld.global.cg), never from a possibly stale L1 line.
#include "ra_signal.cuh"

namespace ra {

// Signal row of one (virtual channel, round): R slots, one per waiting rank.
// Virtual channel g J + j is pass j of channel g, so the rows are laid out
// [channel][pass][round].
__device__ __forceinline__ int64_t counting_row(const PersistArgs& a, int gv, int t) {
  return ((int64_t)gv * (a.rounds - 1) + t) * a.R;
}

// One counting-barrier round, on the signal layer (ra_signal.cuh): each
// peer adds 1 to the waiter's signal of this (channel, round); the waiter
// moves its shadow forward by R-1 and waits for the signal to meet it.
// `shadow` is thread 0's shadow for this round, read from device memory when
// the round began (sig::shadow_ahead), so that read is off the barrier's
// path.  Returns false when this CTA must stop.
__device__ __forceinline__ bool counting_barrier(const PersistArgs& a, int g, int t, int r, sig::Shadow shadow,
                                                 int* s_abort) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t row = counting_row(a, g, t);
    uint64_t* sigs = a.slots + row;
    fence_acq_rel_gpu();   // release: this round's stores of the whole CTA
    if (!(r == a.skip_rank && t == a.skip_round)) {
      for (int q = 0; q < a.R; ++q)
        if (q != r) sig::add(sigs + q, 1);
    }
    const uint64_t target = sig::increase_shadow(shadow, (uint64_t)(a.R - 1));
    sig::store_shadow(a.shadows + row + r, shadow);
    uint64_t seen = 0;
    const sig::Wait w = sig::wait_meet_shadow(sigs + r, shadow, a.bits, a.timeout_ns, &a.err->code, &seen);
    // one counting slot cannot say which peer is late: peer = -1; values in
    // the compared width (the low `bits` bits)
    if (w == sig::kTimedOut) record_wait_error(a.err, 1u, t, r, g, -1, seen, sig::low_bits(target, a.bits));
    *s_abort = w != sig::kReached;
  }
  __syncthreads();
  return *s_abort == 0;
}

// Per-peer barrier round, the design the counting barrier replaced ("comm:
// lift the GIN scale-out ceiling ...", section "Problem" and the comparison in
// section "Performance"): every waiter has one signal per peer; a peer adds 1
// to its own signal of each waiter (SignalAdd), so after the k-th call on the
// slots every one holds k (the call's epoch), and the waiter reads all R-1
// (readSignal, one lane of warp 0 per peer) until each has reached the epoch.
// A wait that runs out can name the peer that did not arrive.
__device__ __forceinline__ bool per_peer_barrier(const PersistArgs& a, const uint64_t* s_epoch, int g, int t,
                                                 int r, int* s_abort) {
  __syncthreads();
  const int R = a.R;
  uint64_t* round_slots = a.slots + ((int64_t)g * (a.rounds - 1) + t) * R * R;   // [waiter][peer]
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();   // release: this round's stores of the whole CTA
    if (!(r == a.skip_rank && t == a.skip_round)) {
      for (int q = 0; q < R; ++q)
        if (q != r) sig::add(round_slots + (int64_t)q * R + r, 1);
    }
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const uint64_t epoch = *s_epoch;
    const uint64_t* mine = round_slots + (int64_t)r * R;
    const bool active = lane < R && lane != r;
    const Deadline limit(a.timeout_ns);
    int abort = 0;
    for (uint64_t it = 0;; ++it) {
      bool ok = true;
      uint64_t v = 0;
      if (active) {
        v = sig::read(mine + lane, a.bits);   // acquire, by the lane that observes the slot
        ok = sig::reached(v, epoch, a.bits);
      }
      const unsigned missing = __ballot_sync(0xffffffffu, !ok);
      if (missing == 0u) break;
      int stop = 0;
      if (lane == 0) {
        // the error record's stop word, on every 8th poll (read by every waiter)
        if ((it & 7u) == 7u && load_relaxed_u32(&a.err->code) != 0u)
          stop = 1;
        else if (limit.passed())
          stop = 2;
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      if (stop) {
        if (stop == 2 && lane == 0)
          record_wait_error(a.err, 3u, t, r, g, __ffs(missing) - 1, (uint64_t)(R - 1 - __popc(missing)),
                            (uint64_t)(R - 1));
        abort = 1;
        break;
      }
      if (it > 32) __nanosleep(100);
    }
    if (lane == 0) *s_abort = abort;
  }
  __syncthreads();
  return *s_abort == 0;
}

// Round boundary when the R CTAs of a channel form one thread-block cluster:
// the hardware cluster barrier, release on arrival and acquire on the wait, at
// cluster scope -- the scope that holds every CTA this one exchanges data with.
// All threads of all R CTAs take it, the same number of times, and clusters
// are scheduled whole, so no CTA can wait on one that is not running.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// g, G: the (virtual) channel and the channel count -- pass j of channel c
// is virtual channel c J + j of G J, the (c J + j)-th slice of the chunk.
// `dead_inc`: the incoming data is a partial of the ring that nobody reads
// again (its place is overwritten by the complete value in AllGather), so
// its L2 lines are dropped once read instead of being written back to DRAM.
template <class D, int OP>
__device__ __forceinline__ void reduce_slice(const typename D::T* inc, const typename D::T* loc,
                                             typename D::T* dst, int64_t off, int64_t end, int g, int G,
                                             bool dead_inc) {
  constexpr int V = D::kVec;
  const Span<V> sp(off, end);
  int64_t pb, pe;
  split_vectors(sp.vb, sp.ve, g, G, &pb, &pe);
  const uint4* inc4 = reinterpret_cast<const uint4*>(inc);
  // a warp takes 32 consecutive vectors per step (all lanes loop the same
  // number of times, so the warp can drop the lines it has read together)
  const int lane = threadIdx.x & 31;
  for (int64_t w = pb + (threadIdx.x - lane); w < pe; w += blockDim.x) {
    const int64_t v = w + lane;
    if (v < pe) {
      const uint4 x = ld_l2(inc4 + v);
      const uint4 y = ld_l2(reinterpret_cast<const uint4*>(loc) + v);
      st_l2(reinterpret_cast<uint4*>(dst) + v, combine_vec<D, OP>(x, y));
    }
    if (dead_inc) discard_read_lines(inc4 + w, pe - w < 32 ? pe - w : 32);
  }
  if (g == 0) {
    const int64_t ns = sp.scalar_count();
    for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
      const int64_t i = sp.scalar_at(t);
      st_g(dst + i, Op<D, OP>::apply(ld_l2_scalar(inc + i), ld_l2_scalar(loc + i)));
    }
  }
}

template <class D>
__device__ __forceinline__ void copy_slice(const typename D::T* src, typename D::T* dst, int64_t off,
                                           int64_t end, int g, int G) {
  constexpr int V = D::kVec;
  const Span<V> sp(off, end);
  int64_t pb, pe;
  split_vectors(sp.vb, sp.ve, g, G, &pb, &pe);
  const uint4* src4 = reinterpret_cast<const uint4*>(src);
  uint4* dst4 = reinterpret_cast<uint4*>(dst);
  const int64_t step = blockDim.x;
  // two vectors a CTA's width apart per iteration: two loads in flight
  for (int64_t v = pb + threadIdx.x; v < pe; v += 2 * step) {
    const uint4 a0 = ld_l2(src4 + v);
    uint4 a1;
    if (v + step < pe) a1 = ld_l2(src4 + v + step);
    st_l2(dst4 + v, a0);
    if (v + step < pe) st_l2(dst4 + v + step, a1);
  }
  if (g == 0) {
    const int64_t ns = sp.scalar_count();
    for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
      const int64_t i = sp.scalar_at(t);
      st_g(dst + i, ld_l2_scalar(src + i));
    }
  }
}

template <class D, int OP>
__global__ void __launch_bounds__(kPersistThreads, 6)
persistent_kernel(const PersistArgs a) {
  using T = typename D::T;
  __shared__ int s_abort;
  const int R = a.R, GV = a.G * a.J;
  const int r = blockIdx.x % R;
  const int p = (r == 0) ? R - 1 : r - 1;
  // The per-peer barrier's epoch: every slot of a waiter holds the number of
  // calls it took part in.  Each CTA keeps its own copy of that count in
  // device memory and moves it on itself (no other CTA reads it), so a launch
  // a CUDA graph replays takes its epoch from there (from_memory); a launch
  // from the host is handed the count and writes it down.
  __shared__ uint64_t s_epoch;
  if (a.sync == kSyncPerPeer && a.rounds > 1) {
    uint64_t* mine = a.shadows + blockIdx.x;
    if (threadIdx.x == 0) {
      const uint64_t e = a.from_memory ? sig::load_shadow(mine).v + 1 : a.epoch;
      sig::store_shadow(mine, sig::Shadow{e});
      s_epoch = e;
    }
    __syncthreads();
  }
  // pass j of channel c is virtual channel c J + j of G J (one pass: c)
  for (int g = blockIdx.x / R * a.J, gend = g + a.J; g < gend; ++g) {
    for (int t = 0; t < a.rounds; ++t) {
      // the counting barrier's waiter reads its shadow now; the value is used
      // after the round's data work
      sig::Shadow shadow{0};
      if (a.sync == kSyncCounting && threadIdx.x == 0 && t + 1 < a.rounds)
        shadow = sig::shadow_ahead(a.shadows + counting_row(a, g, t) + r);
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
      if (off < end) {
        if (reduce) {
          const T* inc = static_cast<const T*>(s == 1 ? a.p.in[p] : a.p.out[p]);
          // from round 2 on the incoming data is the predecessor's partial
          reduce_slice<D, OP>(inc, static_cast<const T*>(a.p.in[r]), static_cast<T*>(a.p.out[r]), off, end, g, GV,
                              s != 1);
        } else {
          copy_slice<D>(static_cast<const T*>(a.p.out[p]), static_cast<T*>(a.p.out[r]), off, end, g, GV);
        }
      }
      if (t + 1 < a.rounds) {
        if (a.sync == kSyncCluster) {
          cluster_barrier();
          continue;
        }
        const bool go = a.sync == kSyncPerPeer ? per_peer_barrier(a, &s_epoch, g, t, r, &s_abort)
                                                : counting_barrier(a, g, t, r, shadow, &s_abort);
        if (!go) return;
      }
    }
  }
}

static const void* persistent_select(int dtype, int op) {
  const void* fn = nullptr;
  with_dtype_op(dtype, op, [&](auto d, auto o) {
    fn = reinterpret_cast<const void*>(&persistent_kernel<decltype(d), decltype(o)::value>);
    return cudaSuccess;
  });
  return fn;
}

cudaError_t persistent_blocks_per_sm(int dtype, int op, int threads, int* blocks) {
  const void* fn = persistent_select(dtype, op);
  if (!fn) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, threads, 0);
}

cudaError_t prepare_persistent_cluster() {
  cudaError_t err = cudaSuccess;
  for (int dt = RA_F32; dt <= RA_I64 && err == cudaSuccess; ++dt)
    for (int op = RA_SUM; op <= RA_MAX && err == cudaSuccess; ++op)
      err = cudaFuncSetAttribute(persistent_select(dt, op), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return err;
}

static cudaLaunchConfig_t cluster_config(const PersistArgs& a, int threads, cudaStream_t st,
                                         cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.R * a.G);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.R;   // CTA (r, g) = blockIdx.x = g*R + r: rank r of cluster g
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t persistent_cluster_capacity(int dtype, int op, int R, int threads, int* clusters) {
  const void* fn = persistent_select(dtype, op);
  if (!fn || R < 2 || R > 16) return cudaErrorInvalidValue;
  PersistArgs a;
  a.R = R;
  a.G = 1;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(a, threads, 0, attr);
  return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

cudaError_t launch_persistent_cluster(int dtype, int op, const PersistArgs& a, int threads, cudaStream_t st) {
  const void* fn = persistent_select(dtype, op);
  if (!fn || a.R < 2 || a.R > 16 || a.G < 1 || a.J < 1 || a.rounds < 1 || a.sync != kSyncCluster)
    return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(a, threads, st, attr);
  void* args[] = {const_cast<PersistArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_persistent(int dtype, int op, const PersistArgs& a, int threads, cudaStream_t st) {
  const void* fn = persistent_select(dtype, op);
  if (!fn || a.R < 2 || a.R > kMaxRanks || a.G < 1 || a.J < 1 || a.rounds < 1 || (a.sync == kSyncPerPeer && a.J != 1))
    return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<PersistArgs*>(&a)};
  return cudaLaunchCooperativeKernel(fn, dim3(a.R * a.G), dim3(threads), args, 0, st);
}

// ------------------------------------------------ signal maintenance
// The handle's signals and shadows between calls, on the signal layer: no
// kernel of the handle runs meanwhile (the calls are ordered on the stream),
// so a reset cannot race an update.
//   kSigReset  resetSignal on every signal; shadows to 0
//   kSigSeed   resetSignal, then SignalAdd(value) on every signal; shadows
//              to 0, then moved forward by the shadow value
//   kSigRead   readSignal(bits) of every signal into out[]
__global__ void signal_io_kernel(const SignalIoArgs a) {
  const size_t step = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.count; i += step) {
    if (a.op == kSigRead) {
      const uint64_t v = sig::read(a.signals + i, a.bits);
      if (RA_ACCESS_OK(a.out + i, 8u, 2u)) a.out[i] = v;
      continue;
    }
    sig::reset(a.signals + i);
    if (a.op == kSigSeed) sig::add(a.signals + i, a.signal_value);
    if (a.shadows) {
      sig::Shadow s{0};
      if (a.op == kSigSeed) sig::increase_shadow(s, a.shadow_value);
      sig::store_shadow(a.shadows + i, s);
    }
  }
}

cudaError_t launch_signal_io(const SignalIoArgs& a, cudaStream_t st) {
  if (!a.signals || (a.op == kSigRead && !a.out) || a.bits < 1 || a.bits > 64) return cudaErrorInvalidValue;
  if (a.count == 0) return cudaSuccess;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  const size_t blocks = (a.count + 255) / 256;
  signal_io_kernel<<<(unsigned)(blocks > 1024 ? 1024 : blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace ra
