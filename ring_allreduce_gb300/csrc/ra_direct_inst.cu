// ra_direct_inst.cu -- the direct kernel's AllReduce / ReduceScatter
// instantiations for one dtype, named by RA_INST_DTYPE at compile time (the
// build compiles this file once per dtype, in parallel).
#include "ra_direct.cuh"

#ifndef RA_INST_DTYPE
#error "compile with -DRA_INST_DTYPE=<one of the ra_dtype names>"
#endif

namespace ra {

template <>
cudaError_t launch_direct_dt<RA_INST_DTYPE>(int op, const DirectArgs& a, dim3 grid, cudaStream_t st) {
  using D = typename DTypeOf<RA_INST_DTYPE>::type;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  if (op == RA_SUM) return launch_direct_d<D, kOpSum>(a, grid, st);
  if (op == RA_MAX) return launch_direct_d<D, kOpMax>(a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace ra
