// ra_internal.h -- what the host runtime (ra_host.cpp) and the kernel
// translation units share: kernel argument blocks and launch functions.
// Nothing here is part of the public C ABI (include/ra.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ra.h"

namespace ra {

constexpr int kMaxRanks = 32;

// Bounds checks of debug builds (-DRA_DEBUG_BOUNDS): the byte ranges a
// launch may touch -- the call's buffers and the handle's device memory --
// and where violations are counted.  The host fills the table before every
// launch (debug_table(), per host thread); each kernel translation unit
// uploads it to its own constant copy in its launch functions.
struct DebugRange {
  uint64_t lo, hi;     // [lo, hi)
};
struct DebugReport {
  unsigned long long count;        // accesses outside every range (skipped)
  unsigned long long first_addr;   // the first one
  unsigned int first_bytes;
  unsigned int first_kind;         // 1 load, 2 store, 3 bulk copy source, 4 bulk copy destination
};
constexpr int kDebugRanges = 96;
struct DebugTable {
  int count;
  DebugReport* report;
  DebugRange r[kDebugRanges];
};
#ifdef RA_DEBUG_BOUNDS
DebugTable& debug_table();     // ra_host.cpp: this host thread's table
DebugReport* debug_report();   // ra_host.cpp: the process's report (device memory)
#endif

// Which collective a launch carries out.
enum Mode : int { kModeAllReduce = 0, kModeReduceScatter = 1, kModeAllGather = 2 };

// Rank buffers, copied by value into the kernel parameters.
struct Ptrs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
};

// Chunk k of a rank buffer is [k*C, min((k+1)*C, n)).
struct Plan {
  int64_t n;
  int64_t C;
};

// Direct variant: one launch, grid.y = chunk.
struct DirectArgs {
  Ptrs p;
  Plan plan;
  int64_t lo, hi;       // only elements [lo, hi) are processed (0, n: all)
  int R;
  int mode;
  int write_owner;      // AllGather: also write the owner's output (compact input)
};

// AllGather as a TMA broadcast: chunk k read once from its owner (rank k-1)
// and stored to every other rank (and to the owner too with write_owner).
// src_compact: the owner's src buffer holds only its chunk.
struct BcastArgs {
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  Plan plan;
  int R;
  int elem_bytes;
  int write_owner;
  int src_compact;
  int64_t timeout_ns;
  ra_device_error* err;
};

// Compact ReduceScatter / AllGather where chunk starts are not 16-byte
// aligned: one 16-byte output vector per thread and step, grid.y = chunk.  in / out hold
// full buffers on the full side and compact ones (rank r: its chunk
// (r+1) mod R only) on the compact side.
struct CompactArgs {
  Ptrs p;
  Plan plan;
  int R;
  int mode;             // kModeReduceScatter or kModeAllGather
};

// Ring variant, one reduce round s (1..R-1), grid.y = rank.
struct RoundArgs {
  Ptrs p;
  Plan plan;
  int R;
  int s;
  int j, J;             // pass j of J: the j-th of J parts of each chunk's whole vectors
};

// Ring variant, one AllGather round s (1..R-1) on out[]; grid.y = rank.
struct CopyArgs {
  void* buf[kMaxRanks];
  Plan plan;
  int R;
  int s;
  int j, J;             // pass j of J: the j-th of J parts of each chunk's 16-byte body
  int elem_bytes;
  int64_t timeout_ns;
  ra_device_error* err;
};

// Local variant: one CTA runs every ring round for slice g of every chunk
// (SV 16-byte vectors per chunk), g = blockIdx.x, blockIdx.x + gridDim.x, ...
struct LocalArgs {
  Ptrs p;
  Plan plan;
  int R;
  int mode;
  int SV;               // 16-byte vectors of each chunk per slice, 1..local_slice_vectors(R)
  int64_t slices;       // slices per chunk: ceil(most whole vectors in a chunk / SV)
  int64_t timeout_ns;   // bound of every mbarrier wait
  ra_device_error* err;
};

// How the ranks of a channel synchronise between rounds.
enum Sync : int {
  kSyncCounting = 0,   // one slot per (channel, round, waiter); each peer adds 1
  kSyncPerPeer = 1,    // one slot per (channel, round, waiter, peer); each peer stores the epoch
  kSyncFlags = 2,      // pipelined variant: one progress flag per (channel, rank, sub-slice)
  kSyncCluster = 3     // the R CTAs of a channel form one thread-block cluster: hardware barrier
};

// Persistent and pipelined variants: one cooperative launch of R*G CTAs
// (G channels).
struct PersistArgs {
  Ptrs p;
  Plan plan;
  int R;
  int G;
  int J;                // sub-slices per channel slice (pipelined variant)
  int W;                // sub-slices per window: every round runs on a window before the next (pipelined)
  int mode;
  int sync;             // Sync
  int rounds;           // ring rounds this call runs
  uint64_t* slots;      // counting: [G][rounds-1][R]; per-peer: [G][rounds-1][R][R];
                        // flags: [G][R][J]
  uint64_t* shadows;    // counting: each waiter's shadow, laid out as slots; flags: rank r's
                        // shadows of its predecessor's flags, [G][R][J] by waiter; per-peer:
                        // each CTA's copy of the epoch of its last call, [G][R]
  uint64_t epoch;       // calls on this slot array since it was zeroed, this one included
  uint64_t shadow_base; // flags: the value every waiter's shadow starts this call at
  int from_memory;      // per-peer and flags: take the call's epoch / shadow start from the
                        // CTA's own copy in device memory (moved on by every launch) instead
                        // of epoch / shadow_base -- for launches a CUDA graph replays
  int bits;             // width of the signal comparisons (rolling order on the low bits), <= 64
  int64_t timeout_ns;
  ra_device_error* err;
  int skip_rank;        // failure injection: rank withholding one arrival, -1 = none
  int skip_round;
};

// Signal maintenance on the signal layer (ra_persistent.cu): reset, seed or
// read every signal of an array (and its shadows, when given).
enum SigOp : int { kSigReset = 0, kSigSeed = 1, kSigRead = 2 };
struct SignalIoArgs {
  uint64_t* signals;
  uint64_t* shadows;      // may be null
  uint64_t* out;          // kSigRead: the values read
  size_t count;
  int op;
  int bits;               // kSigRead: low bits returned
  uint64_t signal_value;  // kSigSeed
  uint64_t shadow_value;
};
cudaError_t launch_signal_io(const SignalIoArgs& a, cudaStream_t st);

cudaError_t launch_direct(int dtype, int op, const DirectArgs& a, int ctas_per_chunk, cudaStream_t st);
// 16-byte vectors a thread of the direct kernel takes per step.
int direct_vectors_per_thread(int R, int mode);
cudaError_t launch_compact(int dtype, int op, const CompactArgs& a, int ctas_per_chunk, cudaStream_t st);
cudaError_t launch_bcast(const BcastArgs& a, int ctas_per_chunk, cudaStream_t st);
cudaError_t prepare_bcast();   // per-device shared-memory opt-in, as prepare_ag_round
int bcast_tile_bytes();
constexpr int kCompactThreads = 256;
cudaError_t launch_rs_round(int dtype, int op, const RoundArgs& a, int ctas_per_rank, cudaStream_t st);
cudaError_t launch_ag_round(const CopyArgs& a, int ctas_per_rank, cudaStream_t st);
// Per-device set-up of the AllGather kernel (its shared-memory opt-in);
// call with the device current before its first launch there.
cudaError_t prepare_ag_round();
cudaError_t launch_persistent(int dtype, int op, const PersistArgs& a, int threads, cudaStream_t st);
// Cluster launch (one cluster of R CTAs per channel, no cooperative launch);
// prepare once per device: allows clusters of up to 16 CTAs.
cudaError_t launch_persistent_cluster(int dtype, int op, const PersistArgs& a, int threads, cudaStream_t st);
cudaError_t prepare_persistent_cluster();
// Clusters of R CTAs of `threads` threads that can be resident at once (0: none fit).
cudaError_t persistent_cluster_capacity(int dtype, int op, int R, int threads, int* clusters);
// Co-resident CTAs per SM of the persistent kernel for `threads` threads.
cudaError_t persistent_blocks_per_sm(int dtype, int op, int threads, int* blocks);
cudaError_t launch_pipelined(int dtype, int op, const PersistArgs& a, int threads, cudaStream_t st);
cudaError_t pipelined_blocks_per_sm(int dtype, int op, int threads, int* blocks);

cudaError_t launch_local(int dtype, int op, const LocalArgs& a, int ctas, cudaStream_t st);
cudaError_t prepare_local();   // per-device shared-memory opt-in
cudaError_t local_blocks_per_sm(int dtype, int op, int R, int* blocks);
int local_slice_vectors(int R);
size_t local_smem_bytes(int R);

constexpr int kDirectThreads = 256;
constexpr int kRoundThreads = 256;
constexpr int kCopyThreads = 32;
// Persistent kernel: CTAs of 256 threads, 6 per SM (one channel each; a
// channel's barrier wait then overlaps five other channels' work on the SM).
// Pipelined kernel: 512 threads, 3 per SM.  Measured on GB300 at R = 8, 2^24
// fp32: persistent with the cluster barrier 286 -> 253 us at 256 threads,
// counting barrier unchanged there, R = 16 605 -> 570 us, one-channel calls
// 8-11 % faster; the pipelined kernel was 2-5 % slower at 256 or 128 threads.
constexpr int kPersistThreads = 256;
constexpr int kPipeThreads = 512;
constexpr int kPipeMaxSlices = 64;   // sub-slices of a pipelined channel slice

}  // namespace ra
