// ra_direct.cuh -- the direct variant: every element's ring fold in one
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
// reads chunk k from its owner's buffer and writes it to the other R-1 (to
// all R when the owner's input is a separate, compact buffer).
//
// A launch may cover only a window [lo, hi) of the elements: each chunk's
// part of it, with the chunk's own fold order.
//
// Grid: (CTAs per chunk, R chunks).  By default a thread takes U 16-byte
// vectors of its chunk (U = 4, 2, 1 for R <= 2, <= 4, more) and the grid has
// as many CTAs as that needs: many short CTAs that the hardware schedules as
// SMs free up beat one resident wave looping over the chunk (measured on
// GB300: 6.68 vs 6.22 TB/s at R = 8, 2^24 fp32).  Past 65535 CTAs per chunk
// the loop takes over.  The unaligned head and tail of a chunk (a ragged
// chunk plan puts chunk starts off 16 bytes) are done element by element by
// the first CTA of the chunk.
#pragma once

#include "ra_device.cuh"

namespace ra {

template <class D, int OP, int MAXR, int MODE, int U>
__global__ void __launch_bounds__(kDirectThreads)
direct_kernel(const DirectArgs a) {
  using T = typename D::T;
  constexpr int V = D::kVec;
  const int R = a.R;
  const int k = blockIdx.y;
  const int64_t chunk_off = min((int64_t)k * a.plan.C, a.plan.n);
  const int64_t off = max(chunk_off, a.lo);
  const int64_t end = min(min(chunk_off + a.plan.C, a.plan.n), a.hi);
  if (off >= end) return;
  const Span<V> sp(off, end);
  const int owner = (k == 0) ? R - 1 : k - 1;   // rank holding S_k after ReduceScatter

  // rank feeding fold position j of chunk k
  auto src_rank = [&](int j) { int q = k + j; return q >= R ? q - R : q; };

  // A CTA takes U x blockDim.x consecutive vectors per step; slice u of a
  // step is contiguous across the CTA, so every warp access is coalesced.
  const int64_t per_step = (int64_t)U * blockDim.x;
  for (int64_t base = sp.vb + (int64_t)blockIdx.x * per_step; base < sp.ve;
       base += (int64_t)gridDim.x * per_step) {
    if (MODE == kModeAllGather) {
      uint4 s[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = base + u * blockDim.x + threadIdx.x;
        if (v < sp.ve) s[u] = ld_stream(static_cast<const uint4*>(a.p.in[owner]) + v);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = base + u * blockDim.x + threadIdx.x;
        if (v < sp.ve) {
#pragma unroll
          for (int j = 0; j < MAXR; ++j)
            if (j < R && (j != owner || a.write_owner)) st_stream(static_cast<uint4*>(a.p.out[j]) + v, s[u]);
        }
      }
    } else {
      uint4 x[U][MAXR];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = base + u * blockDim.x + threadIdx.x;
        if (v < sp.ve) {
#pragma unroll
          for (int j = 0; j < MAXR; ++j)
            if (j < R) x[u][j] = ld_stream(static_cast<const uint4*>(a.p.in[src_rank(j)]) + v);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = base + u * blockDim.x + threadIdx.x;
        if (v < sp.ve) {
          uint4 acc = x[u][0];
#pragma unroll
          for (int j = 1; j < MAXR; ++j)
            if (j < R) acc = combine_vec<D, OP>(acc, x[u][j]);
          if (MODE == kModeAllReduce) {
#pragma unroll
            for (int j = 0; j < MAXR; ++j)
              if (j < R) st_stream(static_cast<uint4*>(a.p.out[j]) + v, acc);
          } else {
            st_stream(static_cast<uint4*>(a.p.out[owner]) + v, acc);
          }
        }
      }
    }
  }

  if (blockIdx.x == 0) {
    const int64_t ns = sp.scalar_count();
    for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
      const int64_t i = sp.scalar_at(t);
      if (MODE == kModeAllGather) {
        const T s = ld_g(static_cast<const T*>(a.p.in[owner]) + i);
        for (int j = 0; j < R; ++j)
          if (j != owner || a.write_owner) st_g(static_cast<T*>(a.p.out[j]) + i, s);
      } else {
        T acc = ld_g(static_cast<const T*>(a.p.in[src_rank(0)]) + i);
        for (int j = 1; j < R; ++j) acc = Op<D, OP>::apply(acc, ld_g(static_cast<const T*>(a.p.in[src_rank(j)]) + i));
        if (MODE == kModeAllReduce) {
          for (int j = 0; j < R; ++j) st_g(static_cast<T*>(a.p.out[j]) + i, acc);
        } else {
          st_g(static_cast<T*>(a.p.out[owner]) + i, acc);
        }
      }
    }
  }
}

// Vectors per thread and step: small R has few loads per vector, so it
// takes several vectors at once to keep enough bytes in flight.
template <int MAXR> struct Unroll { static constexpr int value = MAXR <= 2 ? 4 : (MAXR <= 4 ? 2 : 1); };
constexpr int kGatherUnroll = 4;

template <class D, int OP, int MAXR>
inline cudaError_t launch_direct_r(const DirectArgs& a, dim3 grid, cudaStream_t st) {
  constexpr int U = Unroll<MAXR>::value;
  if (a.mode == kModeAllReduce)
    direct_kernel<D, OP, MAXR, kModeAllReduce, U><<<grid, kDirectThreads, 0, st>>>(a);
  else if (a.mode == kModeReduceScatter)
    direct_kernel<D, OP, MAXR, kModeReduceScatter, U><<<grid, kDirectThreads, 0, st>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

template <class D, int OP>
inline cudaError_t launch_direct_d(const DirectArgs& a, dim3 grid, cudaStream_t st) {
  if (a.R <= 2) return launch_direct_r<D, OP, 2>(a, grid, st);
  if (a.R <= 4) return launch_direct_r<D, OP, 4>(a, grid, st);
  if (a.R <= 8) return launch_direct_r<D, OP, 8>(a, grid, st);
  if (a.R <= 16) return launch_direct_r<D, OP, 16>(a, grid, st);
  return launch_direct_r<D, OP, 32>(a, grid, st);
}

// One (dtype) instantiation set per object: ra_direct_inst.cu is compiled
// once per dtype, with RA_INST_DTYPE naming it.
template <int DT>
cudaError_t launch_direct_dt(int op, const DirectArgs& a, dim3 grid, cudaStream_t st);

}  // namespace ra
