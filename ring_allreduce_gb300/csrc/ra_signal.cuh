// ra_signal.cuh -- signals and shadows over device memory, after the GIN
// signal API of NCCL's Device API (the GIN article, section "信号（Signals）与
// 计数器（Counters）"), for simulated ranks that are CTAs of one GPU.
//
// What the article describes, and how it is kept here:
//   * a signal is a 64-bit value that remote actions add to; SignalInc may not
//     be mixed with other operations without a reset, so only Add is offered
//     (`add`);
//   * readSignal returns the low `bits` bits, with acquire ordering (`read`);
//   * waitSignal waits until the low `bits` bits reach a value, compared in
//     rolling order so that x < x + 1 holds across wrap-around (`wait`);
//   * resetSignal sets the value to 0 and must not race other updates
//     (`reset`);
//   * each signal has a shadow its owner moves at will; increaseSignalShadow
//     and waitSignalMeetShadow wait for the value to catch up with it
//     (`increase_shadow`, `wait_meet_shadow`).
// Who uses what: the counting barrier of the persistent kernel (add, wait,
// and its shadows in device memory through shadow_ahead /
// increase_shadow_from), the per-peer barrier (add, read), the pipelined
// kernel's progress flags (add; each waiter keeps its shadows of the flags it
// waits on in shared memory for the launch: increase_shadow,
// wait_meet_shadow), and the handle's signal maintenance kernel (reset, add,
// read, increase_shadow; ra_persistent.cu).  The comparison width `bits`
// (RA_OPT_SIGNAL_BITS) is 64 unless a call asks for fewer, as a counter of
// 56 bits would.
// Release is the caller's: one fence.acq_rel.gpu before a batch of adds
// publishes everything the CTA wrote before it (the counting barrier issues
// R-1 adds after one fence); the waits poll with acquire loads.  Every wait is
// bounded: it gives up after `timeout_ns` (global timer, with the SM's cycle
// counter as a second clock, see Deadline), or when a stop word (the error
// record's code) says another waiter has already given up.  The stop word is
// read on every 8th poll only: every waiter of a launch reads the same word,
// and reading it on each poll (serially, or issued alongside the signal's
// load) measured slower on GB300 than this.
#pragma once

#include "ra_device.cuh"

namespace ra {
namespace sig {

enum Wait : int { kReached = 0, kAborted = 1, kTimedOut = 2 };

__device__ __forceinline__ uint64_t low_bits(uint64_t v, int bits) {
  return bits >= 64 ? v : (v & ((1ull << bits) - 1ull));
}

// Rolling comparison on the low `bits` bits: has `value` reached `least`?
__device__ __forceinline__ bool reached(uint64_t value, uint64_t least, int bits = 64) {
  if (bits >= 64) return (int64_t)(value - least) >= 0;
  const uint64_t d = low_bits(value - least, bits);
  return d < (1ull << (bits - 1));
}

// SignalAdd.
__device__ __forceinline__ void add(uint64_t* sig, uint64_t delta) { signal_add_relaxed(sig, delta); }

// readSignal: the low `bits` bits, acquire.
__device__ __forceinline__ uint64_t read(const uint64_t* sig, int bits = 64) {
  return low_bits(signal_load_acquire(sig), bits);
}

// resetSignal: 0; no other update of the signal may race it.
__device__ __forceinline__ void reset(uint64_t* sig) { signal_store_relaxed(sig, 0); }

// Shadows belong to one waiter (one thread), so plain accesses do, in
// device memory (where they persist across launches, read and written
// through L2) or in shared memory (for the length of a launch).
__device__ __forceinline__ uint64_t shadow(const uint64_t* sh) {
  if (__isShared(sh)) return *sh;
  return (uint64_t)ld_l2_scalar(reinterpret_cast<const int64_t*>(sh));
}

// increaseSignalShadow: move the shadow forward by `delta`; returns it.
__device__ __forceinline__ uint64_t increase_shadow(uint64_t* sh, uint64_t delta) {
  const uint64_t v = shadow(sh) + delta;
  if (__isShared(sh)) {
    *sh = v;
  } else if (RA_ACCESS_OK(sh, 8u, 2u)) {
    __stcg(reinterpret_cast<unsigned long long*>(sh), (unsigned long long)v);
  }
  return v;
}

// The same in two steps, for a waiter that knows early which shadow in
// device memory it will move: `shadow_ahead` issues the read (an ordered
// load, so the compiler keeps it where it is written and its latency
// overlaps whatever comes next); `increase_shadow_from` stores the moved
// value and returns it.
__device__ __forceinline__ uint64_t shadow_ahead(const uint64_t* sh) { return signal_load_relaxed(sh); }

__device__ __forceinline__ uint64_t increase_shadow_from(uint64_t* sh, uint64_t read, uint64_t delta) {
  const uint64_t v = read + delta;
  if (RA_ACCESS_OK(sh, 8u, 2u)) __stcg(reinterpret_cast<unsigned long long*>(sh), (unsigned long long)v);
  return v;
}

// waitSignal: wait until the signal reaches `least` (rolling, low `bits`
// bits), polling with acquire loads: on kReached the load that saw it
// ordered what follows; *seen holds the low `bits` bits of the last value
// read.  Gives up (kAborted) once *stop is nonzero, or (kTimedOut) after
// timeout_ns.
__device__ __forceinline__ Wait wait(const uint64_t* sig, uint64_t least, int bits, int64_t timeout_ns,
                                     const uint32_t* stop, uint64_t* seen) {
  uint64_t v = signal_load_acquire(sig);
  if (!reached(v, least, bits)) {
    const Deadline limit(timeout_ns);
    for (uint64_t it = 0;; ++it) {
      if (it > 32) __nanosleep(100);
      v = signal_load_acquire(sig);
      if (reached(v, least, bits)) break;
      if ((it & 7u) == 7u && load_relaxed_u32(stop) != 0u) {
        *seen = low_bits(v, bits);
        return kAborted;
      }
      if (limit.passed()) {
        *seen = low_bits(v, bits);
        return kTimedOut;
      }
    }
  }
  *seen = low_bits(v, bits);
  return kReached;
}

// waitSignalMeetShadow: wait until the signal reaches its shadow.
__device__ __forceinline__ Wait wait_meet_shadow(const uint64_t* sig, const uint64_t* sh, int bits,
                                                 int64_t timeout_ns, const uint32_t* stop, uint64_t* seen) {
  return wait(sig, shadow(sh), bits, timeout_ns, stop, seen);
}

}  // namespace sig
}  // namespace ra
