// ra_round.cu -- the ring variant: one launch per ring round.
//
// "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce":
//   section 5, ReduceScatter round s (1..R-1): every rank r at once receives
//     from r-1 the partial of chunk c = (r - s) mod R and adds its own copy:
//       P_r[c] = P_{r-1}[c] (+) x_r[c],   P_{r-1}[c] = x_{r-1}[c] when s = 1.
//     The partial a rank "sends" is what it stored in its output buffer; its
//     successor reads it there in the next round.  After round R-1, chunk
//     (r+1) mod R of out[r] is complete -- the final reduce of section 9's
//     recvReduceCopySend already lands in the rank's output, and the
//     AllGather's first send reads it from there, so no copy pass is needed.
//   section 6, AllGather round s (1..R-1): rank r copies chunk
//     c = (r + 1 - s) mod R from out[r-1] into out[r]: receive + copy, no
//     reduce.  The copy runs on the Tensor Memory Accelerator: 16-byte
//     aligned tiles go global -> shared -> global with cp.async.bulk, a few
//     tiles in flight per CTA; the unaligned head and tail bytes of a chunk
//     are copied by the CTA's threads.
// One launch covers all R ranks of a round (grid.y = rank); the stream
// order between launches is the round order of the ring.  At large n the
// chunks go through the rounds in J passes: pass j launches every round on
// the j-th of J parts of each chunk, before pass j+1 starts, so the partial
// a round writes is read back by the next round while it is still in L2
// (the element-wise head and tail of a chunk belong to pass 0).  Rounds are
// launched with programmatic dependent launch: a round's CTAs may be
// scheduled while the previous round drains and wait (griddepcontrol.wait)
// for its completion before they read.
#include "ra_device.cuh"

namespace ra {

// ------------------------------------------------------------ reduce round

// Ask the bulk-copy unit to bring the 16-byte vectors [v0, v0 + nv) into L2
// ahead of their reads (cp.async.bulk.prefetch.L2: asynchronous; nothing in
// the SM waits for it or receives data, and L2 stays coherent, so it cannot
// change what a later load returns).  Requests of at most 64 KB each.
__device__ __forceinline__ void prefetch_l2(const uint4* v0, int64_t nv) {
  const char* p = reinterpret_cast<const char*>(v0);
  for (int64_t left = nv * 16; left > 0;) {
    const uint32_t piece = left > 65536 ? 65536u : (uint32_t)left;
    if (RA_ACCESS_OK(p, piece, 1u))
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(piece) : "memory");
    p += piece;
    left -= piece;
  }
}

template <class D, int OP>
__global__ void __launch_bounds__(kRoundThreads)
rs_round_kernel(const RoundArgs a) {
  using T = typename D::T;
  constexpr int V = D::kVec;
  griddep_launch_dependents();   // the next round may be scheduled ...
  const int R = a.R, s = a.s, r = blockIdx.y;
  int c = r - s;
  if (c < 0) c += R;
  const int p = (r == 0) ? R - 1 : r - 1;
  const int64_t off = min((int64_t)c * a.plan.C, a.plan.n);
  const int64_t end = min(off + a.plan.C, a.plan.n);
  const T* inc = static_cast<const T*>(s == 1 ? a.p.in[p] : a.p.out[p]);
  const T* loc = static_cast<const T*>(a.p.in[r]);
  T* dst = static_cast<T*>(a.p.out[r]);
  const Span<V> sp(off, end);
  int64_t qb = 0, qe = 0;
  if (off < end) split_vectors(sp.vb, sp.ve, a.j, a.J, &qb, &qe);
  // The inputs do not depend on the previous round (the own input never; the
  // predecessor's in round 1): each CTA starts the DRAM reads of its share of
  // them into L2 before the wait, so they overlap the previous round's drain.
  if (threadIdx.x == 0 && qe > qb) {
    int64_t cb, ce;
    split_vectors(qb, qe, blockIdx.x, gridDim.x, &cb, &ce);
    if (ce > cb) {
      prefetch_l2(reinterpret_cast<const uint4*>(loc) + cb, ce - cb);
      if (s == 1) prefetch_l2(reinterpret_cast<const uint4*>(inc) + cb, ce - cb);
    }
  }
  griddep_wait();                // ... but this one reads what the previous round wrote
  if (off >= end) return;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const uint4* inc4 = reinterpret_cast<const uint4*>(inc);
  // from round 2 on the incoming data is the predecessor's partial, which
  // nobody reads again before AllGather overwrites it with the complete
  // value: its L2 lines are dropped once read, not written back to DRAM
  const bool dead_inc = s != 1;
  const int lane = threadIdx.x & 31;
  const uint4* loc4 = reinterpret_cast<const uint4*>(loc);
  uint4* dst4 = reinterpret_cast<uint4*>(dst);
  // two steps of the grid (a grid's width apart) per iteration: four loads
  // in flight per thread
  for (int64_t w = qb + (int64_t)blockIdx.x * blockDim.x + (threadIdx.x - lane); w < qe; w += 2 * stride) {
    const int64_t v0 = w + lane, v1 = v0 + stride;
    uint4 x0, y0, x1, y1;
    if (v0 < qe) {
      x0 = ld_g(inc4 + v0);
      y0 = ld_stream(loc4 + v0);
    }
    if (v1 < qe) {
      x1 = ld_g(inc4 + v1);
      y1 = ld_stream(loc4 + v1);
    }
    // plain stores: the next round reads this partial, possibly from L2
    if (v0 < qe) st_g(dst4 + v0, combine_vec<D, OP>(x0, y0));
    if (v1 < qe) st_g(dst4 + v1, combine_vec<D, OP>(x1, y1));
    if (dead_inc) {
      discard_read_lines(inc4 + w, qe - w < 32 ? qe - w : 32);
      if (w + stride < qe) discard_read_lines(inc4 + w + stride, qe - w - stride < 32 ? qe - w - stride : 32);
    }
  }
  if (blockIdx.x == 0 && a.j == 0) {
    const int64_t ns = sp.scalar_count();
    for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
      const int64_t i = sp.scalar_at(t);
      st_g(dst + i, Op<D, OP>::apply(ld_g(inc + i), ld_g(loc + i)));
    }
  }
}

// Launch with programmatic stream serialisation: the kernel may be
// scheduled while the previous one in the stream drains, and waits for it
// in griddep_wait().
template <class K, class A>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const A& args) {
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

cudaError_t launch_rs_round(int dtype, int op, const RoundArgs& a, int ctas_per_rank, cudaStream_t st) {
  if (a.R < 2 || a.R > kMaxRanks || a.s < 1 || a.s >= a.R || a.J < 1 || a.j < 0 || a.j >= a.J || ctas_per_rank < 1)
    return cudaErrorInvalidValue;
  dim3 grid(ctas_per_rank, a.R);
  return with_dtype_op(dtype, op, [&](auto d, auto o) {
    return launch_pdl(rs_round_kernel<decltype(d), decltype(o)::value>, grid, dim3(kRoundThreads), 0, st, a);
  });
}

// ---------------------------------------------------- AllGather round, TMA

// 8 stages of 8 KB in flight per CTA (64 KB): on GB300 1-2 % faster at R = 8 than 4 x 16 KB and
// as fast at R = 2-32; 2 x 32 KB and 6 x 16 KB were 2-5 % slower, 16 x 4 KB 4 % slower at R = 16-32
constexpr int kTileBytes = 8192;
constexpr int kStages = 8;
constexpr int kCopySmem = kTileBytes * kStages;

// Bounded wait for a bulk load: gives up after timeout_ns of the global
// timer (or of the SM's cycle counter, should that timer stand still: see
// Deadline); false when it gave up.
__device__ __forceinline__ bool wait_tile(uint64_t* bar, uint32_t parity, int64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const Deadline limit(timeout_ns);
  while (!mbar_try_wait(bar, parity)) {
    if (limit.passed()) return false;
  }
  return true;
}

__global__ void __launch_bounds__(kCopyThreads)
ag_round_kernel(const CopyArgs a) {
  extern __shared__ __align__(128) uint8_t tiles[];
  __shared__ __align__(8) uint64_t bars[kStages];
  griddep_launch_dependents();
  griddep_wait();
  const int R = a.R, s = a.s, r = blockIdx.y;
  int c = (r + 1 - s) % R;
  if (c < 0) c += R;
  const int p = (r == 0) ? R - 1 : r - 1;
  const int64_t eb = a.elem_bytes;
  const int64_t b0 = min((int64_t)c * a.plan.C, a.plan.n) * eb;
  const int64_t b1 = min((int64_t)c * a.plan.C + a.plan.C, a.plan.n) * eb;
  if (b0 >= b1) return;
  const uint8_t* src = static_cast<const uint8_t*>(a.buf[p]);
  uint8_t* dst = static_cast<uint8_t*>(a.buf[r]);

  // 16-byte aligned body [c0, c1); the rest is copied byte by byte (pass 0)
  int64_t c0 = (b0 + 15) & ~int64_t(15);
  int64_t c1 = b1 & ~int64_t(15);
  if (c0 >= c1) { c0 = b1; c1 = b1; }
  if (blockIdx.x == 0 && a.j == 0) {
    for (int64_t i = b0 + threadIdx.x; i < c0; i += blockDim.x) st_g(dst + i, ld_g(src + i));
    for (int64_t i = max(c1, c0) + threadIdx.x; i < b1; i += blockDim.x) st_g(dst + i, ld_g(src + i));
  }
  // this pass's part of the body, in whole 16-byte units: [a0, a1)
  int64_t u0, u1;
  split_vectors(0, (c1 - c0) / 16, a.j, a.J, &u0, &u1);
  const int64_t a0 = c0 + 16 * u0;
  const int64_t a1 = c0 + 16 * u1;
  const int64_t body = a1 - a0;
  const int64_t ntiles = (body + kTileBytes - 1) / kTileBytes;
  if ((int64_t)blockIdx.x >= ntiles || threadIdx.x != 0) return;
  const int count = (int)((ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x);
  auto tile_of = [&](int i) -> int64_t { return blockIdx.x + (int64_t)i * gridDim.x; };
  auto bytes_of = [&](int64_t t) -> uint32_t {
    int64_t b = body - t * kTileBytes;
    return (uint32_t)(b < kTileBytes ? b : kTileBytes);
  };
  auto issue_load = [&](int i) {
    const int st = i % kStages;
    const int64_t t = tile_of(i);
    const uint32_t nb = bytes_of(t);
    mbar_arrive_expect_tx(&bars[st], nb);
    bulk_load(tiles + st * kTileBytes, src + a0 + t * kTileBytes, nb, &bars[st]);
  };

  for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
  fence_mbar_init();
  const int pro = count < kStages ? count : kStages;
  for (int i = 0; i < pro; ++i) issue_load(i);
  int issued = pro;   // loads issued so far
  bool ok = true;
  for (int i = 0; i < count; ++i) {
    const int st = i % kStages;
    if (!wait_tile(&bars[st], (uint32_t)((i / kStages) & 1), a.timeout_ns)) {
      record_wait_error(a.err, 2u, s, r, blockIdx.x, -1, (uint64_t)i, (uint64_t)count);
      ok = false;
      break;
    }
    fence_proxy_async_smem();
    const int64_t t = tile_of(i);
    bulk_store(dst + a0 + t * kTileBytes, tiles + st * kTileBytes, bytes_of(t));
    bulk_commit();
    // refill the stage of tile i-1 once its store has read shared memory
    if (i >= 1 && issued < count) {
      bulk_wait_read<1>();
      issue_load(issued);
      ++issued;
    }
  }
  if (!ok) {
    // drain: give every load that may still be in flight one more bounded wait
    for (int i = 0; i < issued; ++i) {
      const int st = i % kStages;
      wait_tile(&bars[st], (uint32_t)((i / kStages) & 1), a.timeout_ns);
    }
  }
  bulk_wait_all();
}

cudaError_t prepare_ag_round() {
  return cudaFuncSetAttribute(ag_round_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCopySmem);
}

cudaError_t launch_ag_round(const CopyArgs& a, int ctas_per_rank, cudaStream_t st) {
  if (a.R < 2 || a.R > kMaxRanks || a.s < 1 || a.s >= a.R || a.J < 1 || a.j < 0 || a.j >= a.J || ctas_per_rank < 1)
    return cudaErrorInvalidValue;
  dim3 grid(ctas_per_rank, a.R);
  return launch_pdl(ag_round_kernel, grid, dim3(kCopyThreads), kCopySmem, st, a);
}

}  // namespace ra
