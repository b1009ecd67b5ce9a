// ra_compact.cu -- ReduceScatter into compact outputs and AllGather from
// compact inputs when chunk starts are not 16-byte aligned.
//
// Compact buffers hold one chunk per rank: rank r's is chunk (r+1) mod R,
// the chunk it owns after ReduceScatter ("Why AllReduce = ReduceScatter +
// AllGather -- NCCL Ring AllReduce", sections 2 and 5: GPU0 holds S1, ...,
// GPU3 holds S0).  Element i of chunk k sits at i - k*C in the compact buffer
// and at i in a full one.  When C * sizeof(element) is a multiple of 16 the
// host runs the direct kernel with per-rank shifted pointers instead; here a
// full-buffer element and its compact copy fall on different 16-byte
// phases, so every access is one element wide (still coalesced: the
// threads of a warp take consecutive elements).  The fold of chunk k is the
// ring's, x_k, x_{k+1}, ..., x_{k-1}, as in the direct kernel.
#include "ra_device.cuh"

namespace ra {

template <class D, int OP>
__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(const CompactArgs a) {
  using T = typename D::T;
  const int R = a.R;
  const int k = blockIdx.y;
  const int64_t off = min((int64_t)k * a.plan.C, a.plan.n);
  const int64_t len = min(off + a.plan.C, a.plan.n) - off;
  if (len <= 0) return;
  const int owner = (k == 0) ? R - 1 : k - 1;
  const int64_t per_step = (int64_t)blockDim.x * kCompactPerThread;
  for (int64_t base = (int64_t)blockIdx.x * per_step; base < len; base += (int64_t)gridDim.x * per_step) {
    if (a.mode == kModeReduceScatter) {
      T acc[kCompactPerThread];
#pragma unroll
      for (int e = 0; e < kCompactPerThread; ++e) {
        const int64_t c = base + e * blockDim.x + threadIdx.x;
        if (c < len) acc[e] = ld_stream_scalar(static_cast<const T*>(a.p.in[k]) + off + c);
      }
      for (int j = 1; j < R; ++j) {
        const int q = (k + j >= R) ? k + j - R : k + j;
        const T* src = static_cast<const T*>(a.p.in[q]) + off;
#pragma unroll
        for (int e = 0; e < kCompactPerThread; ++e) {
          const int64_t c = base + e * blockDim.x + threadIdx.x;
          if (c < len) acc[e] = Op<D, OP>::apply(acc[e], ld_stream_scalar(src + c));
        }
      }
#pragma unroll
      for (int e = 0; e < kCompactPerThread; ++e) {
        const int64_t c = base + e * blockDim.x + threadIdx.x;
        if (c < len) static_cast<T*>(a.p.out[owner])[c] = acc[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < kCompactPerThread; ++e) {
        const int64_t c = base + e * blockDim.x + threadIdx.x;
        if (c < len) {
          const T v = ld_stream_scalar(static_cast<const T*>(a.p.in[owner]) + c);
          for (int j = 0; j < R; ++j) static_cast<T*>(a.p.out[j])[off + c] = v;
        }
      }
    }
  }
}

cudaError_t launch_compact(int dtype, int op, const CompactArgs& a, int ctas_per_chunk, cudaStream_t st) {
  if (a.R < 1 || a.R > kMaxRanks || ctas_per_chunk < 1) return cudaErrorInvalidValue;
  if (a.mode != kModeReduceScatter && a.mode != kModeAllGather) return cudaErrorInvalidValue;
  dim3 grid(ctas_per_chunk, a.R);
  return with_dtype_op(dtype, op, [&](auto d, auto o) {
    compact_kernel<decltype(d), decltype(o)::value><<<grid, kCompactThreads, 0, st>>>(a);
    return cudaGetLastError();
  });
}

}  // namespace ra
