// ra_direct.cu -- the direct variant: every element's ring fold in one
// launch.
//
// "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce",
// section 5: chunk k starts at rank k (round 1, rank r sends its chunk r)
// and every rank on the way adds its own chunk, so the complete S_k is
//     ((x_k (+) x_{k+1}) (+) x_{k+2}) ... (+) x_{k-1}
// and ends on rank k-1.  Section 6: AllGather then copies S_k, unchanged,
// to every other rank.  This kernel computes exactly that fold for every
// element, in registers, reading each rank's element once and writing the
// result once to every output -- the 2*R*n*b bytes no AllReduce of R
// separate buffers can avoid -- instead of moving partials through HBM
// round by round.  The fold order, and with it every rounding, is the
// ring's, so the result is bitwise the ring's.
//
// Modes: AllReduce writes S_k to all R outputs; ReduceScatter writes it to
// the owner's output only (rank k-1, section 5's placement); AllGather
// reads chunk k from its owner's buffer and writes it to the other R-1.
//
// Grid: (CTAs per chunk, R chunks); each thread takes 16-byte vectors of its
// chunk in a grid-stride loop; the unaligned head and tail of a chunk (a
// ragged chunk plan puts chunk starts off 16 bytes) are done element by
// element by the first CTA of the chunk.
#include "ra_device.cuh"

namespace ra {

template <class D, int OP, int MAXR, int MODE>
__global__ void __launch_bounds__(kDirectThreads)
direct_kernel(const DirectArgs a) {
  using T = typename D::T;
  constexpr int V = D::kVec;
  const int R = a.R;
  const int k = blockIdx.y;
  const int64_t off = min((int64_t)k * a.plan.C, a.plan.n);
  const int64_t end = min(off + a.plan.C, a.plan.n);
  if (off >= end) return;
  const Span<V> sp(off, end);
  const int owner = (k == 0) ? R - 1 : k - 1;   // rank holding S_k after ReduceScatter

  // rank feeding fold position j of chunk k
  auto src_rank = [&](int j) { int q = k + j; return q >= R ? q - R : q; };

  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = sp.vb + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < sp.ve; v += stride) {
    if (MODE == kModeAllGather) {
      const uint4 s = ld_stream(static_cast<const uint4*>(a.p.in[owner]) + v);
#pragma unroll
      for (int j = 0; j < MAXR; ++j)
        if (j < R && j != owner) st_stream(static_cast<uint4*>(a.p.out[j]) + v, s);
    } else {
      uint4 x[MAXR];
#pragma unroll
      for (int j = 0; j < MAXR; ++j)
        if (j < R) x[j] = ld_stream(static_cast<const uint4*>(a.p.in[src_rank(j)]) + v);
      uint4 acc = x[0];
#pragma unroll
      for (int j = 1; j < MAXR; ++j)
        if (j < R) acc = combine_vec<D, OP>(acc, x[j]);
      if (MODE == kModeAllReduce) {
#pragma unroll
        for (int j = 0; j < MAXR; ++j)
          if (j < R) st_stream(static_cast<uint4*>(a.p.out[j]) + v, acc);
      } else {
        st_stream(static_cast<uint4*>(a.p.out[owner]) + v, acc);
      }
    }
  }

  if (blockIdx.x == 0) {
    const int64_t ns = sp.scalar_count();
    for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
      const int64_t i = sp.scalar_at(t);
      if (MODE == kModeAllGather) {
        const T s = static_cast<const T*>(a.p.in[owner])[i];
        for (int j = 0; j < R; ++j)
          if (j != owner) static_cast<T*>(a.p.out[j])[i] = s;
      } else {
        T acc = static_cast<const T*>(a.p.in[src_rank(0)])[i];
        for (int j = 1; j < R; ++j) acc = Op<D, OP>::apply(acc, static_cast<const T*>(a.p.in[src_rank(j)])[i]);
        if (MODE == kModeAllReduce) {
          for (int j = 0; j < R; ++j) static_cast<T*>(a.p.out[j])[i] = acc;
        } else {
          static_cast<T*>(a.p.out[owner])[i] = acc;
        }
      }
    }
  }
}

template <class D, int OP, int MAXR>
static cudaError_t launch_direct_r(const DirectArgs& a, dim3 grid, cudaStream_t st) {
  if (a.mode == kModeAllReduce)
    direct_kernel<D, OP, MAXR, kModeAllReduce><<<grid, kDirectThreads, 0, st>>>(a);
  else if (a.mode == kModeReduceScatter)
    direct_kernel<D, OP, MAXR, kModeReduceScatter><<<grid, kDirectThreads, 0, st>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

template <class D, int OP>
static cudaError_t launch_direct_d(const DirectArgs& a, dim3 grid, cudaStream_t st) {
  if (a.R <= 4) return launch_direct_r<D, OP, 4>(a, grid, st);
  if (a.R <= 8) return launch_direct_r<D, OP, 8>(a, grid, st);
  if (a.R <= 16) return launch_direct_r<D, OP, 16>(a, grid, st);
  return launch_direct_r<D, OP, 32>(a, grid, st);
}

// AllGather moves bits only: one instantiation per element width.
template <class D>
static cudaError_t launch_direct_ag(const DirectArgs& a, dim3 grid, cudaStream_t st) {
  if (a.R <= 8)
    direct_kernel<D, kOpSum, 8, kModeAllGather><<<grid, kDirectThreads, 0, st>>>(a);
  else
    direct_kernel<D, kOpSum, kMaxRanks, kModeAllGather><<<grid, kDirectThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_direct(int dtype, int op, const DirectArgs& a, int ctas_per_chunk, cudaStream_t st) {
  if (a.R < 1 || a.R > kMaxRanks || ctas_per_chunk < 1) return cudaErrorInvalidValue;
  dim3 grid(ctas_per_chunk, a.R);
  if (a.mode == kModeAllGather)
    return dtype == RA_BF16 ? launch_direct_ag<DBF16>(a, grid, st) : launch_direct_ag<DI32>(a, grid, st);
  switch (dtype * 2 + op) {
    case RA_F32 * 2 + RA_SUM: return launch_direct_d<DF32, kOpSum>(a, grid, st);
    case RA_F32 * 2 + RA_MAX: return launch_direct_d<DF32, kOpMax>(a, grid, st);
    case RA_BF16 * 2 + RA_SUM: return launch_direct_d<DBF16, kOpSum>(a, grid, st);
    case RA_BF16 * 2 + RA_MAX: return launch_direct_d<DBF16, kOpMax>(a, grid, st);
    case RA_I32 * 2 + RA_SUM: return launch_direct_d<DI32, kOpSum>(a, grid, st);
    case RA_I32 * 2 + RA_MAX: return launch_direct_d<DI32, kOpMax>(a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ra
