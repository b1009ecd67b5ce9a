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
// Who uses what: the counting barrier of the persistent kernel (add; each
// waiter's shadow read ahead from device memory, increase_shadow by R-1,
// store_shadow, wait_meet_shadow), the per-peer barrier (add, read; each
// CTA's copy of its epoch kept with load_shadow / store_shadow), the
// pipelined kernel's progress flags (add; the waiter's shadow of its
// predecessor's flag, held in a register for the launch: increase_shadow,
// wait_meet_shadow; its start read back with load_shadow by launches a CUDA
// graph replays), and the handle's signal maintenance kernel (reset, add,
// read, increase_shadow, store_shadow; ra_persistent.cu).  The comparison width `bits`
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

// The low `bits` bits (1 <= bits <= 64).
__device__ __forceinline__ uint64_t low_bits(uint64_t v, int bits) { return v & (~0ull >> (64 - bits)); }

// Rolling comparison on the low `bits` bits (1 <= bits <= 64): has `value`
// reached `least`?  The difference, modulo 2^bits, lies in the lower half;
// shifted up to the top of 64 bits, that is its sign bit being clear.
__device__ __forceinline__ bool reached(uint64_t value, uint64_t least, int bits = 64) {
  return (int64_t)((value - least) << (64 - bits)) >= 0;
}

// SignalAdd.
__device__ __forceinline__ void add(uint64_t* sig, uint64_t delta) { signal_add_relaxed(sig, delta); }

// readSignal: the low `bits` bits, acquire.
__device__ __forceinline__ uint64_t read(const uint64_t* sig, int bits = 64) {
  return low_bits(signal_load_acquire(sig), bits);
}

// resetSignal: 0; no other update of the signal may race it.
__device__ __forceinline__ void reset(uint64_t* sig) { signal_store_relaxed(sig, 0); }

// A waiter's shadow of a signal: a value its owner (one thread) moves at
// will and waits for the signal to meet.  The owner holds it in a register
// while it runs; where it persists between launches (device memory) is the
// owner's business: load_shadow / shadow_ahead / store_shadow.
struct Shadow {
  uint64_t v;
};

// The shadow kept in device memory, read through L2.
__device__ __forceinline__ Shadow load_shadow(const uint64_t* sh) {
  return Shadow{(uint64_t)ld_l2_scalar(reinterpret_cast<const int64_t*>(sh))};
}

// The same read issued early, as an ordered load, for a waiter that knows
// which shadow it will move next: the compiler keeps the load where it is
// written, so its latency overlaps whatever comes next.
__device__ __forceinline__ Shadow shadow_ahead(const uint64_t* sh) { return Shadow{signal_load_relaxed(sh)}; }

__device__ __forceinline__ void store_shadow(uint64_t* sh, Shadow s) {
  if (RA_ACCESS_OK(sh, 8u, 2u)) __stcg(reinterpret_cast<unsigned long long*>(sh), (unsigned long long)s.v);
}

// increaseSignalShadow: move the shadow forward by `delta`; returns its value.
__device__ __forceinline__ uint64_t increase_shadow(Shadow& s, uint64_t delta) {
  s.v += delta;
  return s.v;
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
__device__ __forceinline__ Wait wait_meet_shadow(const uint64_t* sig, const Shadow& s, int bits, int64_t timeout_ns,
                                                 const uint32_t* stop, uint64_t* seen) {
  return wait(sig, s.v, bits, timeout_ns, stop, seen);
}

}  // namespace sig
}  // namespace ra
