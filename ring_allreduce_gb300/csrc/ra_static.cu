// ra_static.cu -- ra_allreduce_noalloc: the persistent AllReduce with its
// scratch in a fixed device array instead of memory the library allocates.
//
// Who needs this: callers that must not allocate device memory themselves
// or through the library -- code whose device memory is owned by another
// allocator (a framework's caching allocator, or a host process that gives
// plug-ins a fixed memory budget) and so may not call cudaMalloc, and code on
// a path where the device-wide synchronisation of cudaFree is not
// acceptable.  ra_create allocates the persistent variant's signal slots and
// error record with cudaMalloc; this entry point needs no handle and takes
// both from the array below, which the CUDA module holds from the moment the
// library is loaded on a device until the process exits.
//
// The kernel is the persistent kernel of ra_persistent.cu, unchanged; only
// where its signal slots and error record live differs.
#include <cuda_runtime.h>

#include <mutex>

#include "ra.h"
#include "ra_internal.h"

namespace ra {

// 64-bit words of scratch: the error record in the first 256 bytes, then the
// counting barrier's signals followed by the waiters' shadows.  256 KiB +
// 256 bytes per device.
constexpr size_t kStaticErrWords = 32;
constexpr size_t kStaticSlotWords = 32768;

static __device__ __align__(256) uint64_t g_noalloc_scratch[kStaticErrWords + kStaticSlotWords];

// Implemented in ra_host.cpp: records the text ra_last_error() returns.
ra_status record_error(ra_status s, const char* fmt, ...);

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
uint64_t* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (set-up once per
// device: in host code the array's name is only a host-side stand-in).
ra_status scratch_address(int dev, uint64_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return record_error(RA_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return record_error(RA_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    }
    g_scratch_addr[dev] = static_cast<uint64_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return RA_OK;
}

bool overlaps(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + bytes && y < x + bytes;
}

// A buffer the kernel may be given: device or managed memory that the
// current device can use.  cudaPointerGetAttributes allocates nothing; host
// memory, an address CUDA does not know and another device's memory are
// turned into RA_ERR_INVALID here instead of a memory fault in the kernel.
ra_status check_pointer(const void* p, const char* name, int r, int dev) {
  cudaPointerAttributes at;
  const cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return record_error(RA_ERR_INVALID, "%s[%d]=%p: not a CUDA pointer (%s)", name, r, p, cudaGetErrorName(e));
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
    return record_error(RA_ERR_INVALID, "%s[%d]=%p: not device memory", name, r, p);
  if (at.type == cudaMemoryTypeDevice && at.device != dev)
    return record_error(RA_ERR_INVALID, "%s[%d]=%p: memory of device %d, the current device is %d", name, r, p,
                        at.device, dev);
  return RA_OK;
}

}  // namespace
}  // namespace ra

extern "C" ra_status ra_allreduce_noalloc(int R, size_t n, ra_dtype dtype, ra_op op, const void* const* in,
                                          void* const* out, void* stream) {
  using namespace ra;
  if (R < 2 || R > kMaxRanks) return record_error(RA_ERR_INVALID, "R=%d outside [2, %d]", R, kMaxRanks);
  if (dtype < RA_F32 || dtype > RA_I64) return record_error(RA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (op != RA_SUM && op != RA_MAX) return record_error(RA_ERR_INVALID, "unknown op %d", (int)op);
  if (!in || !out) return record_error(RA_ERR_INVALID, "NULL pointer array");
  if (n == 0) return RA_OK;
  if (n > ((size_t)1 << 40)) return record_error(RA_ERR_INVALID, "n=%zu above 2^40 elements", n);
  const size_t esize = (dtype == RA_BF16 || dtype == RA_F16) ? 2 : ((dtype == RA_F64 || dtype == RA_I64) ? 8 : 4);
  const size_t bytes = n * esize;
  for (int r = 0; r < R; ++r) {
    if (!in[r] || !out[r]) return record_error(RA_ERR_INVALID, "NULL buffer for rank %d", r);
    if (((uintptr_t)in[r] | (uintptr_t)out[r]) & 15u)
      return record_error(RA_ERR_INVALID, "buffers of rank %d are not 16-byte aligned", r);
  }
  for (int r = 0; r < R; ++r)
    for (int q = 0; q < R; ++q) {
      if (q != r && overlaps(out[r], out[q], bytes))
        return record_error(RA_ERR_INVALID, "output buffers %d and %d overlap", r, q);
      if (!(q == r && in[q] == out[r]) && overlaps(out[r], in[q], bytes))
        return record_error(RA_ERR_INVALID, "out[%d] overlaps in[%d] (only out[r] == in[r] is allowed)", r, q);
    }

  int dev = -1, sms = 0, coop = 0, bps = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e == cudaSuccess) e = persistent_blocks_per_sm(dtype, op, kPersistThreads, &bps);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return record_error(RA_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  }
  if (!coop || bps < 1) return record_error(RA_ERR_UNSUPPORTED, "device has no cooperative launch");
  for (int r = 0; r < R; ++r) {
    ra_status ps = in[r] == out[r] ? RA_OK : check_pointer(in[r], "in", r, dev);
    if (ps == RA_OK) ps = check_pointer(out[r], "out", r, dev);
    if (ps != RA_OK) return ps;
  }
  uint64_t* scratch = nullptr;
  ra_status s = scratch_address(dev, &scratch);
  if (s != RA_OK) return s;

  // channels: as many as are co-resident and useful, within the array
  const int64_t C = (int64_t)((n + (size_t)R - 1) / (size_t)R);
  const int64_t per_vec = (int64_t)(16 / esize);
  const int64_t vecs = (C + per_vec - 1) / per_vec + 1;
  int64_t G = (vecs + (int64_t)kPersistThreads * 4 - 1) / ((int64_t)kPersistThreads * 4);
  const int64_t co_resident = (int64_t)bps * sms / R;
  if (G > co_resident) G = co_resident;
  // barrier rounds x waiters, for the signals and again for the waiters' shadows
  const int64_t per_channel = (int64_t)(2 * R - 3) * R;
  if (G > (int64_t)kStaticSlotWords / (2 * per_channel)) G = (int64_t)kStaticSlotWords / (2 * per_channel);
  if (G < 1)
    return record_error(RA_ERR_INVALID, "R=%d needs %lld signal slots, the static scratch holds %zu", R,
                        (long long)per_channel, kStaticSlotWords);

  // every call starts from zeroed slots and a clear error record (epoch 1)
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t used = (kStaticErrWords + 2 * (size_t)(G * per_channel)) * sizeof(uint64_t);
  e = cudaMemsetAsync(scratch, 0, used, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return record_error(RA_ERR_CUDA, "clearing the static scratch: %s", cudaGetErrorString(e));
  }
  PersistArgs a;
  a.from_memory = 0;
  for (int r = 0; r < kMaxRanks; ++r) {
    a.p.in[r] = r < R ? in[r] : nullptr;
    a.p.out[r] = r < R ? out[r] : nullptr;
  }
  a.plan.n = (int64_t)n;
  a.plan.C = C;
  a.R = R;
  a.G = (int)G;
  a.mode = kModeAllReduce;
  a.sync = kSyncCounting;
  a.J = 1;
  a.rounds = 2 * (R - 1);
  a.slots = scratch + kStaticErrWords;
  a.shadows = a.slots + G * per_channel;
  a.epoch = 1;
  a.shadow_base = 0;
  a.bits = 64;
  a.timeout_ns = 1000000000LL;
  a.err = reinterpret_cast<ra_device_error*>(scratch);
  a.skip_rank = -1;
  a.skip_round = -1;
#ifdef RA_DEBUG_BOUNDS
  {   // bounds-checked builds: the call's buffers and the part of the scratch it uses
    DebugTable& t = debug_table();
    t.count = 0;
    t.report = debug_report();
    auto add = [&](const void* p, size_t bytes) {
      if (t.count < kDebugRanges) t.r[t.count++] = {(uint64_t)p, (uint64_t)p + bytes};
    };
    for (int r = 0; r < R; ++r) {
      add(in[r], n * esize);
      add(out[r], n * esize);
    }
    add(scratch, used);
  }
#endif
  e = launch_persistent(dtype, op, a, kPersistThreads, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return record_error(e == cudaErrorCooperativeLaunchTooLarge ? RA_ERR_UNSUPPORTED : RA_ERR_CUDA,
                        "persistent kernel launch: %s", cudaGetErrorString(e));
  }
  return RA_OK;
}
