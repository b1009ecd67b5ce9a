// ra_direct.cu -- dispatch of the direct variant (kernel in ra_direct.cuh;
// its reduce instantiations in ra_direct_inst.cu, one object per dtype).
#include "ra_direct.cuh"

namespace ra {

// AllGather moves bits only: one instantiation per element width.
template <class D>
static cudaError_t launch_direct_ag(const DirectArgs& a, dim3 grid, cudaStream_t st) {
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  if (a.R <= 8)
    direct_kernel<D, kOpSum, 8, kModeAllGather, kGatherUnroll><<<grid, kDirectThreads, 0, st>>>(a);
  else
    direct_kernel<D, kOpSum, kMaxRanks, kModeAllGather, kGatherUnroll><<<grid, kDirectThreads, 0, st>>>(a);
  return cudaGetLastError();
}

int direct_vectors_per_thread(int R, int mode) {
  if (mode == kModeAllGather) return kGatherUnroll;
  if (R <= 2) return Unroll<2>::value;
  if (R <= 4) return Unroll<4>::value;
  return 1;
}

cudaError_t launch_direct(int dtype, int op, const DirectArgs& a, int ctas_per_chunk, cudaStream_t st) {
  if (a.R < 1 || a.R > kMaxRanks || ctas_per_chunk < 1) return cudaErrorInvalidValue;
  dim3 grid(ctas_per_chunk, a.R);
  if (a.mode == kModeAllGather) {
    switch (dtype) {
      case RA_BF16: case RA_F16: return launch_direct_ag<DBF16>(a, grid, st);
      case RA_F32: case RA_I32: return launch_direct_ag<DI32>(a, grid, st);
      case RA_F64: case RA_I64: return launch_direct_ag<DI64>(a, grid, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (dtype) {
    case RA_F32: return launch_direct_dt<RA_F32>(op, a, grid, st);
    case RA_BF16: return launch_direct_dt<RA_BF16>(op, a, grid, st);
    case RA_I32: return launch_direct_dt<RA_I32>(op, a, grid, st);
    case RA_F16: return launch_direct_dt<RA_F16>(op, a, grid, st);
    case RA_F64: return launch_direct_dt<RA_F64>(op, a, grid, st);
    case RA_I64: return launch_direct_dt<RA_I64>(op, a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ra
