// ra_device.cuh -- device building blocks shared by the ring kernels:
// the reduction applied at a ring hop, 16-byte vector I/O, the counting
// barrier's signal operations, and the TMA bulk-copy / mbarrier primitives.
//
// The reduction follows "Why AllReduce = ReduceScatter + AllGather -- NCCL
// Ring AllReduce", sections 5 and 7: the receiver computes
// new_partial = incoming_partial (+) local_chunk, elementwise.
//   fp32 SUM  one binary32 addition, __fadd_rn (never contracted, no FTZ);
//   bf16 SUM  both operands widened to binary32 exactly, one binary32
//             addition, then round-to-nearest-even to bf16: the partial is
//             kept in bf16 at every hop, as a ring shipping bf16 would;
//   int32 SUM two's-complement wrap;
//   MAX       local if local > incoming, else incoming.
//
// The signal operations follow the counting barrier of "comm: lift the GIN
// scale-out ceiling by making the rail barrier a counting barrier" (section
// "Fix": every peer adds 1, the waiter moves its shadow by R-1 and polls)
// with the 64-bit rolling comparison of the NCCL Device API GIN article
// (section on signals and counters).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ra_internal.h"

namespace ra {

enum : int { kOpSum = 0, kOpMax = 1 };

// Element storage types.  kVec elements make one 16-byte vector.
struct DF32 { using T = float;    static constexpr int kVec = 4; };
struct DBF16 { using T = uint16_t; static constexpr int kVec = 8; };
struct DI32 { using T = int32_t;  static constexpr int kVec = 4; };
struct DF16 { using T = uint16_t; static constexpr int kVec = 8; };
struct DF64 { using T = double;   static constexpr int kVec = 2; };
struct DI64 { using T = int64_t;  static constexpr int kVec = 2; };

template <int V> struct IntC { static constexpr int value = V; };

template <int DT> struct DTypeOf;
template <> struct DTypeOf<RA_F32> { using type = DF32; };
template <> struct DTypeOf<RA_BF16> { using type = DBF16; };
template <> struct DTypeOf<RA_I32> { using type = DI32; };
template <> struct DTypeOf<RA_F16> { using type = DF16; };
template <> struct DTypeOf<RA_F64> { using type = DF64; };
template <> struct DTypeOf<RA_I64> { using type = DI64; };

// Call f(D{}, IntC<OP>{}) for the (dtype, op) pair; cudaErrorInvalidValue
// for an unknown one.  One place lists every supported combination.
template <class F>
cudaError_t with_dtype_op(int dtype, int op, F&& f) {
  const bool mx = op == RA_MAX;
  if (op != RA_SUM && op != RA_MAX) return cudaErrorInvalidValue;
  switch (dtype) {
    case RA_F32: return mx ? f(DF32{}, IntC<kOpMax>{}) : f(DF32{}, IntC<kOpSum>{});
    case RA_BF16: return mx ? f(DBF16{}, IntC<kOpMax>{}) : f(DBF16{}, IntC<kOpSum>{});
    case RA_I32: return mx ? f(DI32{}, IntC<kOpMax>{}) : f(DI32{}, IntC<kOpSum>{});
    case RA_F16: return mx ? f(DF16{}, IntC<kOpMax>{}) : f(DF16{}, IntC<kOpSum>{});
    case RA_F64: return mx ? f(DF64{}, IntC<kOpMax>{}) : f(DF64{}, IntC<kOpSum>{});
    case RA_I64: return mx ? f(DI64{}, IntC<kOpMax>{}) : f(DI64{}, IntC<kOpSum>{});
    default: return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------ reduction

__device__ __forceinline__ float bf16_widen(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint16_t bf16_round(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <class D, int OP> struct Op;

template <> struct Op<DF32, kOpSum> {
  static __device__ __forceinline__ float apply(float inc, float loc) { return __fadd_rn(inc, loc); }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) {
    return __float_as_uint(__fadd_rn(__uint_as_float(inc), __uint_as_float(loc)));
  }
};

template <> struct Op<DF32, kOpMax> {
  static __device__ __forceinline__ float apply(float inc, float loc) { return loc > inc ? loc : inc; }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) {
    return __uint_as_float(loc) > __uint_as_float(inc) ? loc : inc;
  }
};

template <> struct Op<DI32, kOpSum> {
  static __device__ __forceinline__ int32_t apply(int32_t inc, int32_t loc) {
    return (int32_t)((uint32_t)inc + (uint32_t)loc);
  }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) { return inc + loc; }
};

template <> struct Op<DI32, kOpMax> {
  static __device__ __forceinline__ int32_t apply(int32_t inc, int32_t loc) { return loc > inc ? loc : inc; }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) {
    return (int32_t)loc > (int32_t)inc ? loc : inc;
  }
};

// bf16: one 32-bit word holds elements 2j (low half) and 2j+1 (high half).
template <> struct Op<DBF16, kOpSum> {
  static __device__ __forceinline__ uint16_t apply(uint16_t inc, uint16_t loc) {
    return bf16_round(__fadd_rn(bf16_widen(inc), bf16_widen(loc)));
  }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) {
    float lo = __fadd_rn(__uint_as_float(inc << 16), __uint_as_float(loc << 16));
    float hi = __fadd_rn(__uint_as_float(inc & 0xFFFF0000u), __uint_as_float(loc & 0xFFFF0000u));
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);   // .x = lo (low half), .y = hi
    return *reinterpret_cast<uint32_t*>(&p);
  }
};

template <> struct Op<DBF16, kOpMax> {
  static __device__ __forceinline__ uint16_t apply(uint16_t inc, uint16_t loc) {
    return bf16_widen(loc) > bf16_widen(inc) ? loc : inc;
  }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) {
    uint32_t lo = __uint_as_float(loc << 16) > __uint_as_float(inc << 16) ? (loc & 0xFFFFu) : (inc & 0xFFFFu);
    uint32_t hi = __uint_as_float(loc & 0xFFFF0000u) > __uint_as_float(inc & 0xFFFF0000u)
                      ? (loc & 0xFFFF0000u) : (inc & 0xFFFF0000u);
    return lo | hi;
  }
};

// fp16: as bf16, widened exactly to binary32, one addition, rounded to
// nearest-even fp16 (24 >= 2*11+2, so the double rounding is innocuous).
template <> struct Op<DF16, kOpSum> {
  static __device__ __forceinline__ float widen(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)bits16));
  }
  static __device__ __forceinline__ uint16_t apply(uint16_t inc, uint16_t loc) {
    return __half_as_ushort(__float2half_rn(__fadd_rn(widen(inc), widen(loc))));
  }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) {
    return (uint32_t)apply((uint16_t)(inc & 0xFFFFu), (uint16_t)(loc & 0xFFFFu)) |
           ((uint32_t)apply((uint16_t)(inc >> 16), (uint16_t)(loc >> 16)) << 16);
  }
};

template <> struct Op<DF16, kOpMax> {
  static __device__ __forceinline__ uint16_t apply(uint16_t inc, uint16_t loc) {
    return Op<DF16, kOpSum>::widen(loc) > Op<DF16, kOpSum>::widen(inc) ? loc : inc;
  }
  static __device__ __forceinline__ uint32_t word(uint32_t inc, uint32_t loc) {
    return (uint32_t)apply((uint16_t)(inc & 0xFFFFu), (uint16_t)(loc & 0xFFFFu)) |
           ((uint32_t)apply((uint16_t)(inc >> 16), (uint16_t)(loc >> 16)) << 16);
  }
};

// 64-bit types: a 16-byte vector holds two elements.
template <> struct Op<DF64, kOpSum> {
  static __device__ __forceinline__ double apply(double inc, double loc) { return __dadd_rn(inc, loc); }
  static __device__ __forceinline__ uint64_t lane(uint64_t inc, uint64_t loc) {
    return (uint64_t)__double_as_longlong(__dadd_rn(__longlong_as_double((long long)inc),
                                                    __longlong_as_double((long long)loc)));
  }
};

template <> struct Op<DF64, kOpMax> {
  static __device__ __forceinline__ double apply(double inc, double loc) { return loc > inc ? loc : inc; }
  static __device__ __forceinline__ uint64_t lane(uint64_t inc, uint64_t loc) {
    return __longlong_as_double((long long)loc) > __longlong_as_double((long long)inc) ? loc : inc;
  }
};

template <> struct Op<DI64, kOpSum> {
  static __device__ __forceinline__ int64_t apply(int64_t inc, int64_t loc) {
    return (int64_t)((uint64_t)inc + (uint64_t)loc);
  }
  static __device__ __forceinline__ uint64_t lane(uint64_t inc, uint64_t loc) { return inc + loc; }
};

template <> struct Op<DI64, kOpMax> {
  static __device__ __forceinline__ int64_t apply(int64_t inc, int64_t loc) { return loc > inc ? loc : inc; }
  static __device__ __forceinline__ uint64_t lane(uint64_t inc, uint64_t loc) {
    return (int64_t)loc > (int64_t)inc ? loc : inc;
  }
};

template <class D> struct Is64 { static constexpr bool value = false; };
template <> struct Is64<DF64> { static constexpr bool value = true; };
template <> struct Is64<DI64> { static constexpr bool value = true; };

template <class D, int OP, bool W64 = Is64<D>::value>
struct VecOp {
  static __device__ __forceinline__ uint4 apply(uint4 inc, uint4 loc) {
    uint4 r;
    r.x = Op<D, OP>::word(inc.x, loc.x);
    r.y = Op<D, OP>::word(inc.y, loc.y);
    r.z = Op<D, OP>::word(inc.z, loc.z);
    r.w = Op<D, OP>::word(inc.w, loc.w);
    return r;
  }
};

template <class D, int OP>
struct VecOp<D, OP, true> {
  static __device__ __forceinline__ uint4 apply(uint4 inc, uint4 loc) {
    const uint64_t a0 = ((uint64_t)inc.y << 32) | inc.x, a1 = ((uint64_t)inc.w << 32) | inc.z;
    const uint64_t b0 = ((uint64_t)loc.y << 32) | loc.x, b1 = ((uint64_t)loc.w << 32) | loc.z;
    const uint64_t r0 = Op<D, OP>::lane(a0, b0), r1 = Op<D, OP>::lane(a1, b1);
    return make_uint4((uint32_t)r0, (uint32_t)(r0 >> 32), (uint32_t)r1, (uint32_t)(r1 >> 32));
  }
};

template <class D, int OP>
__device__ __forceinline__ uint4 combine_vec(uint4 inc, uint4 loc) {
  return VecOp<D, OP>::apply(inc, loc);
}

// --------------------------------------------- bounds checks (debug builds)
// Built with -DRA_DEBUG_BOUNDS, every global access below is first checked
// against the byte ranges registered for the launch; one outside all of them
// is counted, the first one noted, and skipped (a load reads zero), so the
// kernel runs on without touching memory it does not own.  This stands in
// for a memory checker.  Without the flag the checks are compiled out and
// every helper is the plain access.

#ifdef RA_DEBUG_BOUNDS
static __constant__ DebugTable g_debug_ranges;   // one per translation unit

static __device__ __noinline__ bool debug_access_ok(const void* p, unsigned bytes, unsigned kind) {
  const uint64_t a = reinterpret_cast<uint64_t>(p);
  for (int i = 0; i < g_debug_ranges.count; ++i)
    if (a >= g_debug_ranges.r[i].lo && a + bytes <= g_debug_ranges.r[i].hi) return true;
  DebugReport* rep = g_debug_ranges.report;
  if (rep && atomicAdd(&rep->count, 1ull) == 0ull) {
    rep->first_addr = a;
    rep->first_bytes = bytes;
    rep->first_kind = kind;
  }
  return false;
}
#define RA_ACCESS_OK(p, bytes, kind) (::ra::debug_access_ok((p), (bytes), (kind)))

// Launch functions call this first: the kernels of this translation unit
// check against the table the host filled for the call.
inline cudaError_t debug_upload(cudaStream_t st) {
  return cudaMemcpyToSymbolAsync(g_debug_ranges, &debug_table(), sizeof(DebugTable), 0, cudaMemcpyHostToDevice,
                                 st);
}
#else
#define RA_ACCESS_OK(p, bytes, kind) true
inline cudaError_t debug_upload(cudaStream_t) { return cudaSuccess; }
#endif

// One element of global memory, plain access.
template <class T> __device__ __forceinline__ T ld_g(const T* p) {
  if (!RA_ACCESS_OK(p, sizeof(T), 1u)) return T();
  return *p;
}
template <class T> __device__ __forceinline__ void st_g(T* p, T v) {
  if (RA_ACCESS_OK(p, sizeof(T), 2u)) *p = v;
}

// ------------------------------------------------------------ vector I/O
// Streaming loads/stores for data touched once per launch (evict-first in
// L2), and L2-only (.cg) accesses for data another CTA of the same launch
// wrote or will read (the persistent kernel), which must not come from a
// stale L1 line.

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  if (!RA_ACCESS_OK(p, 16u, 1u)) return make_uint4(0u, 0u, 0u, 0u);
  return __ldcs(p);
}
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  if (RA_ACCESS_OK(p, 16u, 2u)) __stcs(p, v);
}
// Read-only data (the non-coherent path): buffers no CTA of the launch writes.
__device__ __forceinline__ uint4 ld_ro(const uint4* p) {
  if (!RA_ACCESS_OK(p, 16u, 1u)) return make_uint4(0u, 0u, 0u, 0u);
  return __ldg(p);
}
__device__ __forceinline__ uint4 ld_l2(const uint4* p) {
  if (!RA_ACCESS_OK(p, 16u, 1u)) return make_uint4(0u, 0u, 0u, 0u);
  return __ldcg(p);
}
__device__ __forceinline__ void st_l2(uint4* p, uint4 v) {
  if (RA_ACCESS_OK(p, 16u, 2u)) __stcg(p, v);
}

// Drop dead data from L2 without writing it back.  After a warp has read
// the 32 consecutive 16-byte vectors [v0, v0 + nv) of a partial that nobody
// reads again before it is overwritten, the 128-byte lines lying wholly
// inside that range are invalidated in L2 (discard.global.L2: a dirty line
// is dropped instead of written to DRAM; the memory reads as undefined until
// it is written again).  Lines the range only partly covers are left alone:
// their other bytes may belong to another warp, CTA or chunk.  Every lane of
// the warp calls this, after its own read of the range has completed.
__device__ __forceinline__ void discard_read_lines(const uint4* v0, int64_t nv) {
  __syncwarp();   // every lane's load of the range has returned
  const uintptr_t a = reinterpret_cast<uintptr_t>(v0);
  const uintptr_t lo = (a + 127u) & ~uintptr_t(127);
  const uintptr_t hi = (a + 16u * (uintptr_t)nv) & ~uintptr_t(127);
  const uintptr_t line = lo + 128u * (threadIdx.x & 31u);
  if (line < hi && RA_ACCESS_OK(reinterpret_cast<const void*>(line), 128u, 2u))
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
}

// One element, read once (evict-first), through the coherent path.
template <class T> __device__ __forceinline__ T ld_stream_scalar(const T* p) {
  if (!RA_ACCESS_OK(p, sizeof(T), 1u)) return T();
  return __ldcs(p);
}
template <> __device__ __forceinline__ uint16_t ld_stream_scalar<uint16_t>(const uint16_t* p) {
  if (!RA_ACCESS_OK(p, 2u, 1u)) return 0;
  return __ldcs(reinterpret_cast<const unsigned short*>(p));
}
template <> __device__ __forceinline__ int64_t ld_stream_scalar<int64_t>(const int64_t* p) {
  if (!RA_ACCESS_OK(p, 8u, 1u)) return 0;
  return (int64_t)__ldcs(reinterpret_cast<const long long*>(p));
}

template <class T> __device__ __forceinline__ T ld_l2_scalar_raw(const T* p);
template <> __device__ __forceinline__ float ld_l2_scalar_raw<float>(const float* p) { return __ldcg(p); }
template <> __device__ __forceinline__ int32_t ld_l2_scalar_raw<int32_t>(const int32_t* p) { return __ldcg(p); }
template <> __device__ __forceinline__ uint16_t ld_l2_scalar_raw<uint16_t>(const uint16_t* p) {
  return __ldcg(reinterpret_cast<const unsigned short*>(p));
}
template <> __device__ __forceinline__ double ld_l2_scalar_raw<double>(const double* p) { return __ldcg(p); }
template <> __device__ __forceinline__ int64_t ld_l2_scalar_raw<int64_t>(const int64_t* p) {
  return (int64_t)__ldcg(reinterpret_cast<const long long*>(p));
}
template <class T> __device__ __forceinline__ T ld_l2_scalar(const T* p) {
  if (!RA_ACCESS_OK(p, sizeof(T), 1u)) return T();
  return ld_l2_scalar_raw(p);
}

// Split [off, end) (element indices, buffers 16-byte aligned) into a scalar
// head, whole 16-byte vectors [vb, ve) (vector indices) and a scalar tail.
template <int V>
struct Span {
  int64_t off, end, vb, ve;
  __device__ __forceinline__ Span(int64_t o, int64_t e) : off(o), end(e) {
    vb = (o + V - 1) / V;
    ve = e / V;
    if (vb > ve) { vb = ve = 0; }   // no whole vector: all scalar
  }
  __device__ __forceinline__ bool has_vectors() const { return ve > vb; }
  // scalar elements: [off, head_end) and [tail_begin, end)
  __device__ __forceinline__ int64_t head_end() const { return has_vectors() ? vb * V : end; }
  __device__ __forceinline__ int64_t tail_begin() const { return has_vectors() ? ve * V : end; }
  __device__ __forceinline__ int64_t scalar_count() const {
    return (head_end() - off) + (end - tail_begin());
  }
  // i-th scalar element (i < scalar_count())
  __device__ __forceinline__ int64_t scalar_at(int64_t i) const {
    int64_t h = head_end() - off;
    return i < h ? off + i : tail_begin() + (i - h);
  }
};

// Part `part` of `parts` of a vector range [vb, ve): contiguous, whole vectors.
__device__ __forceinline__ void split_vectors(int64_t vb, int64_t ve, int part, int parts,
                                              int64_t* pb, int64_t* pe) {
  int64_t nv = ve - vb;
  int64_t per = (nv + parts - 1) / parts;
  int64_t b = vb + per * part;
  int64_t e = b + per;
  if (b > ve) b = ve;
  if (e > ve) e = ve;
  *pb = b;
  *pe = e;
}

// ----------------------------------------------------- signals / barrier

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// The end of a bounded wait, kept on two clocks: the global timer, and the
// SM's own cycle counter in case that timer stands still.  The cycle budget
// is 3 cycles per nanosecond of the limit (saturating): at GB300's highest
// SM clock (2.07 GHz) it runs out at 1.45 x the limit, at 1 GHz at 3 x, so a
// wait never outlasts a small multiple of its limit whatever the poll costs.
__device__ __forceinline__ uint64_t sm_cycles() {
  uint64_t c;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
  return c;
}

struct Deadline {
  uint64_t t0, c0;
  int64_t ns, cycles;
  __device__ __forceinline__ explicit Deadline(int64_t timeout_ns) {
    t0 = globaltimer_ns();
    c0 = sm_cycles();
    ns = timeout_ns;
    cycles = timeout_ns > ((int64_t)1 << 60) ? ((int64_t)1 << 62) : 3 * timeout_ns;
  }
  __device__ __forceinline__ bool passed() const {
    return (int64_t)(globaltimer_ns() - t0) > ns || (int64_t)(sm_cycles() - c0) > cycles;
  }
};

// Release / acquire in the fence form: one fence.acq_rel.gpu before a
// batch of relaxed SignalAdds makes everything ordered before the fence
// (this thread's writes and those of the CTA it synchronised with) visible
// to whoever observes any of the adds and then runs the acquire fence.
// One fence for the R-1 adds of a barrier round instead of a release per add.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void signal_add_relaxed(uint64_t* p, uint64_t v) {
  if (!RA_ACCESS_OK(p, 8u, 2u)) return;
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Acquire load: polling with it orders everything after the poll that sees
// the target behind the peers' release, with no separate fence (measured
// on GB300: 14 % cheaper barrier rounds than relaxed polls plus a fence).
__device__ __forceinline__ uint64_t signal_load_acquire(const uint64_t* p) {
  if (!RA_ACCESS_OK(p, 8u, 1u)) return 0;
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t signal_load_relaxed(const uint64_t* p) {
  if (!RA_ACCESS_OK(p, 8u, 1u)) return 0;
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void signal_store_relaxed(uint64_t* p, uint64_t v) {
  if (!RA_ACCESS_OK(p, 8u, 2u)) return;
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t load_relaxed_u32(const uint32_t* p) {
  if (!RA_ACCESS_OK(p, 4u, 1u)) return 0;
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The first wait that gives up fills the error record; later ones leave it.
__device__ __forceinline__ void record_wait_error(ra_device_error* err, uint32_t code, int round, int rank,
                                                  int channel, int peer, uint64_t observed, uint64_t expected) {
  if (!RA_ACCESS_OK(err, sizeof(ra_device_error), 2u)) return;
  if (atomicCAS(&err->code, 0u, code) == 0u) {
    err->round = round;
    err->rank = rank;
    err->channel = channel;
    err->peer = peer;
    err->observed = observed;
    err->expected = expected;
    __threadfence();
  }
}

// ------------------------------------------ programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start while
// the kernel before it in the stream is still running; it must wait for that
// kernel (and the visibility of its memory) before touching data it wrote.
// Letting dependents launch early only lets their CTAs be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------- TMA bulk copy, mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// global -> shared (this CTA), completion counted on `bar` in bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
// (A debug build that skips a copy leaves its bytes unannounced: the wait on
// `bar` then runs out, bounded, and reports.)
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  if (!RA_ACCESS_OK(gmem_src, bytes, 3u)) return;
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared (this CTA) -> global, tracked by bulk async-groups.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  if (!RA_ACCESS_OK(gmem_dst, bytes, 4u)) return;
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(gmem_dst), "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group has completed (writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace ra
