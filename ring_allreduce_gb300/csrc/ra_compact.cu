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
// phases.  Each thread still writes one aligned 16-byte vector: it reads the
// two aligned vectors around the unaligned one it needs and funnel-shifts
// the bytes into place.  Vectors that would reach past a buffer, and the
// chunk's head and tail, go element by element.  The fold of chunk k is the
// ring's, x_k, x_{k+1}, ..., x_{k-1}, as in the direct kernel.
#include <type_traits>

#include "ra_device.cuh"

namespace ra {

// Bytes [s, s + 16) of the 32 bytes A:B (0 <= s < 16): the 16-byte vector
// that starts s bytes into A.  Little-endian words; q = whole words to skip,
// sh = bits to shift within a word (funnel shift of two neighbouring words).
__device__ __forceinline__ uint4 shift_bytes(uint4 A, uint4 B, int s) {
  const uint32_t W[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
  const int q = s >> 2;
  const uint32_t sh = (uint32_t)(s & 3) * 8u;
  uint32_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = q == 0 ? W[j] : q == 1 ? W[j + 1] : q == 2 ? W[j + 2] : W[j + 3];
    const uint32_t hi = q == 0 ? W[j + 1] : q == 1 ? W[j + 2] : q == 2 ? W[j + 3] : W[j + 4];
    r[j] = __funnelshift_r(lo, hi, sh);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// The 16-byte vector starting `e` elements into `base` (any element phase),
// read as the two aligned vectors around it; both must lie inside the buffer.
// Read-only, non-overlapping buffers: the second load mostly hits L1.
template <class T>
__device__ __forceinline__ uint4 load_at(const T* base, int64_t e) {
  constexpr int V = 16 / sizeof(T);
  const uint4* v = reinterpret_cast<const uint4*>(base) + e / V;
  const int s = (int)(e % V) * (int)sizeof(T);
  const uint4 A = ld_ro(v);
  if (s == 0) return A;
  return shift_bytes(A, ld_ro(v + 1), s);
}

// Whole 16-byte vectors a thread may read starting at element e of a buffer
// of n elements (the second aligned vector included when the phase is not 0).
template <int V>
__device__ __forceinline__ bool readable(int64_t e, int64_t n) {
  const int64_t last = (e % V == 0) ? e / V + 1 : e / V + 2;   // one past the last aligned vector touched
  return last * V <= n;
}

// B: how many of a vector's R operand loads ReduceScatter issues before
// folding them (all R when R <= B, as the direct kernel does; batches of B
// otherwise, which keeps the registers of R = 32 to a few CTAs per SM).
// B = 1: one load at a time, each folded as it arrives.  The AllGather
// branch does not use B, but it shares the kernel's register allocation,
// which B sets; it runs in the B = 1 instantiation.
template <class D, int OP, int B>
__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(const CompactArgs a) {
  using T = typename D::T;
  constexpr int V = D::kVec;
  const int R = a.R;
  const int k = blockIdx.y;
  const int64_t n = a.plan.n;
  const int64_t off = min((int64_t)k * a.plan.C, n);
  const int64_t len = min(off + a.plan.C, n) - off;
  if (len <= 0) return;
  const int owner = (k == 0) ? R - 1 : k - 1;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;

  if (a.mode == kModeReduceScatter) {
    // Compact output vector u = chunk elements [uV, uV + V) = full-buffer
    // elements from e = off + uV, phase s = (off mod V) bytes.  All R inputs
    // share that phase, so the fold runs on aligned vectors (g = e / V) and
    // only the folded result is shifted: lane l folds vector g, takes lane
    // l+1's folded vector g+1 by shuffle (lane 31 folds its own), and writes
    // the shifted pair.  The loop is warp-uniform so every lane shuffles.
    const int s = (int)(off % V) * (int)sizeof(T);
    int64_t nu = len / V;
    while (nu > 0 && !readable<V>(off + (nu - 1) * V, n)) --nu;
    T* dst = static_cast<T*>(a.p.out[owner]);
    // B loads of the vector in flight at once, then their fold in ring
    // order (x_k first), then the next B
    auto load = [&](int j, int64_t g) {
      const int q = (k + j >= R) ? k + j - R : k + j;
      return ld_ro(reinterpret_cast<const uint4*>(a.p.in[q]) + g);
    };
    auto fold = [&](int64_t g) {
      if constexpr (B == 1) {
        uint4 acc = ld_ro(reinterpret_cast<const uint4*>(a.p.in[k]) + g);
        for (int j = 1; j < R; ++j) {
          const int q = (k + j >= R) ? k + j - R : k + j;
          acc = combine_vec<D, OP>(acc, ld_ro(reinterpret_cast<const uint4*>(a.p.in[q]) + g));
        }
        return acc;
      } else {
        uint4 x[B];
#pragma unroll
        for (int j = 0; j < B; ++j)
          if (j < R) x[j] = load(j, g);
        uint4 acc = x[0];
#pragma unroll
        for (int j = 1; j < B; ++j)
          if (j < R) acc = combine_vec<D, OP>(acc, x[j]);
        for (int j0 = B; j0 < R; j0 += B) {
#pragma unroll
          for (int t = 0; t < B; ++t)
            if (j0 + t < R) x[t] = load(j0 + t, g);
#pragma unroll
          for (int t = 0; t < B; ++t)
            if (j0 + t < R) acc = combine_vec<D, OP>(acc, x[t]);
        }
        return acc;
      }
    };
    // A warp folds 32 consecutive vectors and writes the 31 outputs whose
    // both halves it holds: ~3 % extra loads, no lane folding twice.
    const int lane = threadIdx.x & 31;
    const int64_t g0 = off / V;
    const int64_t warp = tid >> 5, warps = stride >> 5;
    for (int64_t ub = warp * 31; ub < nu; ub += warps * 31) {
      const int64_t u = ub + lane;
      const int64_t g = g0 + u;
      uint4 acc = make_uint4(0, 0, 0, 0);
      if (u <= nu && (g + 1) * V <= n) acc = fold(g);       // vector g is whole inside the buffer
      uint4 nxt;
      nxt.x = __shfl_down_sync(0xffffffffu, acc.x, 1);
      nxt.y = __shfl_down_sync(0xffffffffu, acc.y, 1);
      nxt.z = __shfl_down_sync(0xffffffffu, acc.z, 1);
      nxt.w = __shfl_down_sync(0xffffffffu, acc.w, 1);
      // for u < nu, readable() put vector g+1 inside the buffer, and lane+1 folded it
      if (lane < 31 && u < nu)
        st_stream(reinterpret_cast<uint4*>(dst) + u, s == 0 ? acc : shift_bytes(acc, nxt, s));
    }
    if (blockIdx.x == 0) {
      for (int64_t c = nu * V + threadIdx.x; c < len; c += blockDim.x) {
        T acc = ld_stream_scalar(static_cast<const T*>(a.p.in[k]) + off + c);
        for (int j = 1; j < R; ++j) {
          const int q = (k + j >= R) ? k + j - R : k + j;
          acc = Op<D, OP>::apply(acc, ld_stream_scalar(static_cast<const T*>(a.p.in[q]) + off + c));
        }
        st_g(dst + c, acc);
      }
    }
  } else {
    // full output vector g = elements [gV, gV + V), read from the owner's
    // compact chunk at element gV - off (any phase), written aligned to all R
    const T* src = static_cast<const T*>(a.p.in[owner]);
    const int64_t gb = (off + V - 1) / V;
    int64_t ge = (off + len) / V;
    while (ge > gb && !readable<V>((ge - 1) * V - off, len)) --ge;
    if (ge < gb) ge = gb;
    for (int64_t g = gb + tid; g < ge; g += stride) {
      const uint4 v = load_at(src, g * V - off);
      for (int j = 0; j < R; ++j) st_stream(static_cast<uint4*>(a.p.out[j]) + g, v);
    }
    if (blockIdx.x == 0) {
      const int64_t head = gb * V - off;             // elements before the first whole output vector
      const int64_t vec_end = ge * V - off;          // compact index where the vector part ends
      const int64_t head_n = head < len ? head : len;
      const int64_t tail_b = ge > gb ? vec_end : head_n;
      const int64_t ns = head_n + (len - tail_b);
      for (int64_t t = threadIdx.x; t < ns; t += blockDim.x) {
        const int64_t c = t < head_n ? t : tail_b + (t - head_n);
        const T v = ld_stream_scalar(src + c);
        for (int j = 0; j < R; ++j) st_g(static_cast<T*>(a.p.out[j]) + off + c, v);
      }
    }
  }
}

cudaError_t launch_compact(int dtype, int op, const CompactArgs& a, int ctas_per_chunk, cudaStream_t st) {
  if (a.R < 1 || a.R > kMaxRanks || ctas_per_chunk < 1) return cudaErrorInvalidValue;
  if (a.mode != kModeReduceScatter && a.mode != kModeAllGather) return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  dim3 grid(ctas_per_chunk, a.R);
  return with_dtype_op(dtype, op, [&](auto d, auto o) {
    using D = decltype(d);
    constexpr int OP = decltype(o)::value;
    // AllGather runs in the B = 1 instantiation: in the B = 2 one (fewer
    // registers, more CTAs per SM) the ragged bf16 AllGather measured 6 %
    // slower, in the B = 8 one the 4-rank fp64 one 8 % slower.  fp64 additions are a scarce unit on this GPU: an 8-rank ragged
    // fp64 sum keeps them busy most of the time, and there folding each
    // operand as it arrives (B = 1) measured 3-6 % faster than batched loads.
    constexpr bool fp64_sum = std::is_same<D, DF64>::value && OP == kOpSum;
    if (a.mode == kModeAllGather || fp64_sum) {
      compact_kernel<D, OP, 1><<<grid, kCompactThreads, 0, st>>>(a);
    } else if constexpr (!fp64_sum) {
      if (a.R <= 2)
        compact_kernel<D, OP, 2><<<grid, kCompactThreads, 0, st>>>(a);
      else if (a.R <= 4)
        compact_kernel<D, OP, 4><<<grid, kCompactThreads, 0, st>>>(a);
      else
        compact_kernel<D, OP, 8><<<grid, kCompactThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
  });
}

}  // namespace ra
