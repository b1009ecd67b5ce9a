// ra_bcast.cu -- AllGather as a broadcast through shared memory with the
// Tensor Memory Accelerator: every 16-byte-aligned tile of a chunk is
// loaded once from its owner (cp.async.bulk global -> shared, mbarrier
// completion) and stored from that one copy to every other rank
// (cp.async.bulk shared -> global, R-1 stores per tile).
//
// "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce",
// section 6: AllGather copies the complete chunk S_k, unchanged, from the
// rank that holds it (k-1, section 5) to every other rank.  The bytes are
// read once and written R-1 times (R times when the owner's chunk comes
// from a separate compact buffer).  One elected thread per CTA drives a
// ring of kStages tiles; the unaligned head and tail bytes of a chunk are
// copied by the CTA's threads.  Every mbarrier wait is bounded.
#include "ra_device.cuh"

namespace ra {

namespace {

constexpr int kTile = 16384;
constexpr int kStages = 4;
constexpr int kSmem = kTile * kStages;

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

}  // namespace

__global__ void __launch_bounds__(32)
bcast_kernel(const BcastArgs a) {
  extern __shared__ __align__(128) uint8_t tiles[];
  __shared__ __align__(8) uint64_t bars[kStages];
  const int R = a.R;
  const int k = blockIdx.y;
  const int owner = (k == 0) ? R - 1 : k - 1;
  const int64_t eb = a.elem_bytes;
  const int64_t b0 = min((int64_t)k * a.plan.C, a.plan.n) * eb;      // chunk bytes in full-buffer coordinates
  const int64_t b1 = min((int64_t)k * a.plan.C + a.plan.C, a.plan.n) * eb;
  if (b0 >= b1) return;
  // src + x addresses byte x of the chunk in full-buffer coordinates
  const uint8_t* src = static_cast<const uint8_t*>(a.src[owner]) - (a.src_compact ? b0 : 0);

  int64_t a0 = (b0 + 15) & ~int64_t(15);
  int64_t a1 = b1 & ~int64_t(15);
  if (a0 >= a1) { a0 = b1; a1 = b1; }
  if (blockIdx.x == 0) {
    for (int j = 0; j < R; ++j) {
      if (j == owner && !a.write_owner) continue;
      uint8_t* dst = static_cast<uint8_t*>(a.dst[j]);
      for (int64_t i = b0 + threadIdx.x; i < a0; i += blockDim.x) st_g(dst + i, ld_g(src + i));
      for (int64_t i = max(a1, a0) + threadIdx.x; i < b1; i += blockDim.x) st_g(dst + i, ld_g(src + i));
    }
  }
  const int64_t body = a1 - a0;
  const int64_t ntiles = (body + kTile - 1) / kTile;
  if ((int64_t)blockIdx.x >= ntiles || threadIdx.x != 0) return;
  const int count = (int)((ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x);
  auto tile_of = [&](int i) -> int64_t { return blockIdx.x + (int64_t)i * gridDim.x; };
  auto bytes_of = [&](int64_t t) -> uint32_t {
    const int64_t b = body - t * kTile;
    return (uint32_t)(b < kTile ? b : kTile);
  };
  auto issue_load = [&](int i) {
    const int st = i % kStages;
    const int64_t t = tile_of(i);
    const uint32_t nb = bytes_of(t);
    mbar_arrive_expect_tx(&bars[st], nb);
    bulk_load(tiles + st * kTile, src + a0 + t * kTile, nb, &bars[st]);
  };
  for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
  fence_mbar_init();
  const int pro = count < kStages ? count : kStages;
  for (int i = 0; i < pro; ++i) issue_load(i);
  int issued = pro;
  bool ok = true;
  for (int i = 0; i < count; ++i) {
    const int st = i % kStages;
    if (!wait_tile(&bars[st], (uint32_t)((i / kStages) & 1), a.timeout_ns)) {
      record_wait_error(a.err, 2u, 0, owner, blockIdx.x, -1, (uint64_t)i, (uint64_t)count);
      ok = false;
      break;
    }
    fence_proxy_async_smem();
    const int64_t t = tile_of(i);
    const uint32_t nb = bytes_of(t);
    for (int j = 0; j < R; ++j) {
      if (j == owner && !a.write_owner) continue;
      bulk_store(static_cast<uint8_t*>(a.dst[j]) + a0 + t * kTile, tiles + st * kTile, nb);
    }
    bulk_commit();
    // refill the stage of tile i-1 once its stores have read shared memory
    if (i >= 1 && issued < count) {
      bulk_wait_read<1>();
      issue_load(issued);
      ++issued;
    }
  }
  if (!ok) {
    for (int i = 0; i < issued; ++i) wait_tile(&bars[i % kStages], (uint32_t)((i / kStages) & 1), a.timeout_ns);
  }
  bulk_wait_all();
}

cudaError_t prepare_bcast() {
  return cudaFuncSetAttribute(bcast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

int bcast_tile_bytes() { return kTile; }

cudaError_t launch_bcast(const BcastArgs& a, int ctas_per_chunk, cudaStream_t st) {
  if (a.R < 1 || a.R > kMaxRanks || ctas_per_chunk < 1) return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  dim3 grid(ctas_per_chunk, a.R);
  bcast_kernel<<<grid, 32, kSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace ra
