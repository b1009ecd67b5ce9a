/*
 * ra.h -- ring AllReduce, ReduceScatter and AllGather over R ranks that are
 * held as R buffers in the HBM of one GPU (GB300, sm_103a).
 *
 * What the calls compute follows the web page "Why AllReduce =
 * ReduceScatter + AllGather -- NCCL Ring AllReduce":
 *
 *   section 1   every rank r holds x_r[0..n); afterwards every rank holds
 *               S[i] = x_0[i] (+) x_1[i] (+) ... (+) x_{R-1}[i] for all i;
 *   section 12  the n elements are cut into R chunks; here chunk k is
 *               [k*C, min((k+1)*C, n)) with C = ceil(n/R), so the last
 *               chunks are the short ones and may be empty;
 *   section 4   the ring is rank 0 -> 1 -> ... -> R-1 -> 0;
 *   section 5   ReduceScatter: in round 1 rank r sends its chunk r to r+1,
 *               which adds its own chunk; the partial travels on, and after
 *               R-1 rounds rank r holds the complete S of chunk (r+1) mod R
 *               (GPU0:S1, GPU1:S2, GPU2:S3, GPU3:S0 for R=4).  Chunk k is
 *               therefore folded in ring order x_k, x_{k+1}, ..., x_{k-1},
 *               each hop computing  incoming (+) local;
 *   section 6   AllGather: the complete chunks travel on for R-1 more
 *               rounds, copied, never reduced;
 *   sections 8, 9  the boundary step recvReduceCopySend: the last reduction
 *               of a chunk writes it to the rank's output and is the first
 *               AllGather send.
 *
 * Results are bitwise the ones of that ring for every dtype: the fold order
 * of each element is fixed; bf16 and fp16 partials are rounded
 * (round-to-nearest-even) to their format at every hop, as a ring carrying
 * such messages would store them, each hop being one binary32 addition of
 * the exactly widened operands; fp32 and fp64 additions are single IEEE
 * additions with no contraction and no flush to zero; integer sums wrap.
 * MAX keeps the incoming partial unless the local value is strictly greater.
 *
 * Buffers and ownership
 *   - The caller owns every buffer.  in[r] and out[r] (r = 0..R-1) are
 *     device pointers to n elements, in memory of the device that was
 *     current at ra_create, each 16-byte aligned.  The pointer arrays
 *     themselves are host arrays of R entries, read during the call only.
 *   - out[r] == in[r] (in place) is allowed.  Any other overlap between the
 *     2R ranges, or between two outputs, is RA_ERR_INVALID.
 *   - The handle owns only what it allocates: at ra_create the counting
 *     barrier's signal slots, a device error record and a private stream (for
 *     capturing the ring variant's graph); on the first call that needs them,
 *     the per-peer barrier's slots, the pipelined variant's flags, and for
 *     ra_allreduce_host its device copies of the buffers, two copy streams
 *     and their events.
 *
 * Asynchrony and errors
 *   - Every compute call is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns once enqueued.  Host-side argument
 *     errors return a status and enqueue nothing.
 *   - No device wait is unbounded: the persistent and pipelined kernels'
 *     polls and the copy waits of the AllGather round and local kernels give
 *     up after RA_OPT_TIMEOUT_NS, note what they waited for in the handle's
 *     error record and return (the cluster barrier is the hardware's own).
 *     That record is read by ra_get_device_status.  No kernel traps.
 *   - ra_last_error() gives a text for the calling thread's last failure.
 *   - A handle is used by one host thread at a time.  Its device calls must
 *     be ordered (one stream, or synchronised by the caller): the persistent
 *     variant's signal slots are per handle.  ra_allreduce_host is the
 *     exception: its calls may alternate between streams (see there).
 *
 * Edge cases: n == 0 is a no-op returning RA_OK (the buffer pointers are not
 * looked at, NULL included).  R == 1 copies in[0] to
 * out[0].  R outside [1, 32], a NULL or misaligned pointer, an unknown dtype
 * or op return RA_ERR_INVALID.  Every dtype supports RA_SUM and RA_MAX.
 */
#ifndef RING_ALLREDUCE_GB300_RA_H
#define RING_ALLREDUCE_GB300_RA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ra_status {
  RA_OK = 0,
  RA_ERR_INVALID = 1,      /* bad argument; nothing was enqueued */
  RA_ERR_CUDA = 2,         /* a CUDA runtime call failed (no device, launch error, ...) */
  RA_ERR_OOM = 3,          /* device allocation of the handle's state failed */
  RA_ERR_UNSUPPORTED = 4,  /* e.g. the persistent grid cannot be co-resident */
  RA_ERR_TIMEOUT = 5       /* a device-side wait gave up (see ra_get_device_status) */
} ra_status;

typedef enum ra_dtype {
  RA_F32 = 0,   /* IEEE binary32 */
  RA_BF16 = 1,  /* bfloat16 (16-bit patterns) */
  RA_I32 = 2,   /* int32, sums wrap */
  RA_F16 = 3,   /* IEEE binary16 */
  RA_F64 = 4,   /* IEEE binary64 */
  RA_I64 = 5    /* int64, sums wrap */
} ra_dtype;
typedef enum ra_op { RA_SUM = 0, RA_MAX = 1 } ra_op;

/* Which kernels carry out a call.  All give bitwise the same result. */
typedef enum ra_variant {
  RA_VARIANT_AUTO = 0,        /* currently DIRECT */
  RA_VARIANT_DIRECT = 1,      /* one launch: every element's ring fold done in
                                 registers; reads each input once, writes each
                                 output once */
  RA_VARIANT_RING = 2,        /* one launch per ring round: R-1 reduce rounds
                                 (recvReduceSend ... recvReduceCopySend), then
                                 R-1 AllGather rounds done with TMA bulk copies;
                                 at large n the chunks go through the rounds
                                 in passes (RA_OPT_SLICES) */
  RA_VARIANT_PERSISTENT = 3,  /* one cooperative launch running every round;
                                 simulated ranks meet at a barrier between
                                 rounds (RA_OPT_BARRIER: counting, the
                                 default, per-peer or cluster); at large n
                                 each channel's slice goes through the rounds
                                 in passes (RA_OPT_SLICES) */
  RA_VARIANT_PIPELINED = 4,   /* one cooperative launch running every round
                                 with no barrier: a rank starts a round on a
                                 sub-slice as soon as its predecessor has
                                 finished the previous round on it
                                 (per-predecessor progress flags; rounds of
                                 different sub-slices overlap; RA_OPT_PROTOCOL
                                 chooses how the messages travel).  Each call
                                 is handed where its flags start; every CTA
                                 also keeps that in device memory, and a call
                                 made while its stream is being captured into
                                 a CUDA graph -- and every call after it
                                 until ra_get_device_status resets the handle
                                 -- takes it from there, so replays continue
                                 the count (a few percent slower at large n) */
  RA_VARIANT_LOCAL = 5        /* one launch, each CTA running every ring round
                                 for one slice of every chunk: the ranks'
                                 messages pass through shared memory, the
                                 operands arrive by TMA bulk copies ahead of
                                 the rounds; reads each input once, writes
                                 each output once, no waits between CTAs */
} ra_variant;

/* Barrier of the persistent variant (RA_OPT_BARRIER). */
typedef enum ra_barrier {
  RA_BARRIER_COUNTING = 0,    /* one 64-bit signal per (channel, round, waiter);
                                 each of the R-1 peers adds 1 ("comm: lift the
                                 GIN scale-out ceiling by making the rail
                                 barrier a counting barrier", section "Fix") */
  RA_BARRIER_PER_PEER = 1,    /* one signal per (channel, round, waiter, peer),
                                 the design that page replaced; a wait that runs
                                 out can name the missing peer.  Each call is
                                 handed its epoch; every CTA also keeps it in
                                 device memory, and calls captured into a
                                 CUDA graph (and the calls after them, until
                                 a reset) take it from there */
  RA_BARRIER_CLUSTER = 2      /* the R CTAs of a channel form one thread-block
                                 cluster and meet at the hardware cluster
                                 barrier (R <= 16, else RA_ERR_UNSUPPORTED);
                                 no signal memory, no cooperative launch */
} ra_barrier;

/* How the pipelined variant's messages travel (RA_OPT_PROTOCOL). */
typedef enum ra_protocol {
  RA_PROTOCOL_SIMPLE = 0,     /* a rank's partial goes to its output buffer,
                                 then a progress flag is published (a release
                                 fence and a SignalAdd) that the successor
                                 polls before reading the partial */
  RA_PROTOCOL_LL = 1,         /* flag-in-data messages for small chunks: each
                                 8-byte word carries 32 bits of data and a
                                 32-bit flag naming the call and the round,
                                 written by one store into the successor's row
                                 of an inbox the handle allocates on first use
                                 ((2R-3) x R x C x w words of 8 bytes, w = 2
                                 for 8-byte elements, else 1; at most 64 MiB,
                                 else RA_ERR_UNSUPPORTED); the successor polls
                                 the words themselves, so a ring hop is one
                                 store and one poll, with no fence and no
                                 separate flag.  Twice the bytes per element
                                 (four times for 16-bit elements).  Every CTA
                                 keeps the flag its next call starts at in
                                 device memory; calls captured into a CUDA
                                 graph (and the calls after them, until a
                                 reset) start from there, and a replayed call
                                 whose flags would pass 2^32 - 1 does nothing
                                 and reports error code 6 (the status call
                                 zeroes the inbox). */
  RA_PROTOCOL_LL_CLUSTER = 2  /* the same words, stored straight into the
                                 successor's shared memory: the R CTAs of a
                                 channel form one thread-block cluster (R <=
                                 16, else RA_ERR_UNSUPPORTED) and each polls
                                 its own shared memory, so a hop stays inside
                                 one GPC.  No inbox and no state kept between
                                 calls (capturable into a CUDA graph); a
                                 CTA's rows take (2R-3) x 8 x w bytes per
                                 position it carries, at most 200 KiB. */
} ra_protocol;

typedef enum ra_option {
  RA_OPT_VARIANT = 1,        /* ra_variant, default RA_VARIANT_AUTO */
  RA_OPT_TIMEOUT_NS = 2,     /* limit of every device-side wait in ns, 1e3
                                (1 us) to 6e10 (60 s), default 1e9 */
  RA_OPT_CTAS = 3,           /* CTAs per rank (ring, persistent) or per chunk
                                (direct), or in all (local); 0 = chosen
                                from the SM count */
  RA_OPT_CHECK_POINTERS = 4, /* 1 (default): a call checks with
                                cudaPointerGetAttributes that every buffer is
                                device memory of the handle's device; a call
                                with the same pointers as the last call that
                                passed is not checked again */
  RA_OPT_SKIP_ARRIVAL = 5,   /* failure injection for tests: (rank << 16) |
                                round names a rank that withholds, in every
                                channel, its arrival at that barrier round
                                (persistent variant) or every progress flag
                                from that ring round on (pipelined variant);
                                -1 (default) = off.  The waits of the ranks
                                that depend on it then run out after
                                RA_OPT_TIMEOUT_NS and the call reports
                                RA_ERR_TIMEOUT through ra_get_device_status. */
  RA_OPT_GRAPHS = 6,         /* 1 (default): the ring variant captures its
                                2(R-1) launches in a CUDA graph the first time
                                it meets a set of buffers and replays the graph
                                on later calls with the same buffers (one host
                                launch instead of 2(R-1)); when the caller's
                                stream is itself being captured it launches
                                directly.  0: always launch directly.  Any
                                ra_set_option drops the cached graph. */
  RA_OPT_BARRIER = 7,        /* ra_barrier of the persistent variant */
  RA_OPT_SLICES = 8,         /* sub-slices per channel slice of the pipelined
                                variant, 1..64, and passes of the persistent
                                variant with the counting or cluster barrier
                                and of the ring variant (each pass takes one
                                part of every slice or chunk through every
                                round), at most 8 there; 0 (default) = the
                                fewest that keep n * b / J within 32 MiB, at
                                most 8 (1 up to 32 MiB per rank).  The
                                per-peer barrier always runs one pass. */
  RA_OPT_GATHER = 9,         /* kernel of the direct AllGather (and of the compact
                                AllGather when chunk starts are 16-byte
                                aligned): 0 (default) = chosen by the library,
                                1 = 16-byte vector loads and stores, 2 = TMA
                                broadcast (each tile loaded once into shared
                                memory, bulk-stored to every other rank) */
  RA_OPT_HOST_WINDOWS = 10,  /* windows of ra_allreduce_host: 0 (default) =
                                chosen by the library, 1..8 = that many (fewer
                                when a window would hold less than one 16-byte
                                vector per rank) */
  RA_OPT_WINDOW = 12,        /* sub-slices per window of the pipelined
                                variant: each rank runs every ring round on a
                                window of this many sub-slices before it
                                starts the next window, so a round's partials
                                are read back soon after they are written.
                                0 (default) = 1 (every round on one sub-slice
                                before the next); values at or above the
                                sub-slice count mean all of them (every round
                                over the whole slice) */
  RA_OPT_SIGNAL_BITS = 14,   /* width, 16..64 (default 64), of the signal
                                comparisons of the persistent variant's
                                barriers and the pipelined variant's flags:
                                a wait compares the low bits in rolling order
                                (x < x + 1 across wrap-around), as the GIN
                                article's waitSignal(..., bits) does; a device
                                whose signals are 56-bit counters would use 56.
                                ra_read_signals returns the low bits too. */
  RA_OPT_PROTOCOL = 15,      /* ra_protocol of the pipelined variant, default
                                RA_PROTOCOL_SIMPLE.  With RA_PROTOCOL_LL and
                                RA_PROTOCOL_LL_CLUSTER, RA_OPT_CTAS is the
                                channels per rank (0: chosen),
                                RA_OPT_SKIP_ARRIVAL names a rank that sends
                                nothing from that round on, and
                                RA_OPT_SLICES, RA_OPT_WINDOW and
                                RA_OPT_SIGNAL_BITS do not apply. */
  RA_OPT_LL_FLAG = 16,       /* the flag the next RA_PROTOCOL_LL call's first
                                message carries, 1..2^32-1 (1 after creation).
                                Each call moves it on by its ring rounds; a
                                call whose flags would pass 2^32-1 first
                                zeroes the inbox and starts again at 1, so no
                                word left in the inbox ever carries a flag
                                being waited for.  Setting it is for tests of
                                that restart.  It governs calls from the host;
                                once a call has been captured into a CUDA
                                graph the CTAs' own copies do, until
                                ra_get_device_status resets the handle. */
  RA_OPT_DEBUG_SHRINK = 11   /* bounds-checked builds only (see
                                ra_debug_bounds_report): register each of the
                                call's buffers this many bytes shorter than it
                                is, so that the accesses to its last bytes are
                                reported and skipped -- a test of the checks.
                                RA_ERR_UNSUPPORTED in other builds. */
} ra_option;

/* Device error record, filled by the first wait that gives up. */
typedef struct ra_device_error {
  uint32_t code;      /* 0 = none; 1 = counting-barrier wait ran out; 2 = bulk-copy wait
                         ran out; 3 = per-peer barrier wait ran out; 4 = pipelined
                         flag wait ran out; 5 = RA_PROTOCOL_LL message wait ran
                         out; 6 = a replayed RA_PROTOCOL_LL call ran out of flags */
  int32_t round;      /* barrier round (0-based), ring round (codes 4, 5) or AllGather round (code 2) */
  int32_t rank;       /* waiting rank */
  int32_t channel;    /* channel: the CTA index within its rank */
  int32_t peer;       /* rank that did not arrive when it can be named (codes 3, 4, 5), else -1 */
  int32_t reserved;
  uint64_t observed;  /* arrivals (codes 1, 3), progress (code 4) or a message word's flag
                         (code 5) seen last */
  uint64_t expected;  /* what was waited for (codes 1-4: expected - observed were missing;
                         code 5: the flag of the awaited message) */
} ra_device_error;

typedef struct ra_ctx* ra_handle;

/* Create a handle for R ranks of n elements of `dtype`, reduced with `op`,
 * on the current CUDA device.  Allocates the barrier signal slots (zeroed)
 * and the error record.  *out is set only on RA_OK. */
ra_status ra_create(int R, size_t n, ra_dtype dtype, ra_op op, ra_handle* out);

/* Free the handle's device state after synchronising the device.  NULL is
 * a no-op. */
ra_status ra_destroy(ra_handle h);

/* Ring ReduceScatter (section 5 of the ring page).  On completion chunk
 * (r+1) mod R of out[r] holds the complete S of that chunk; the other chunks
 * of out[r] hold unspecified values (partials of the ring, or, where the
 * round-by-round variants dropped a partial from L2 once its successor had
 * read it, whatever memory then returns). */
ra_status ra_reduce_scatter(ra_handle h, const void* const* in, void* const* out, void* stream);

/* Ring AllGather (section 6), in place: buf[r] must hold in its chunk
 * (r+1) mod R the complete value of that chunk (the layout ra_reduce_scatter
 * leaves); afterwards every buf[r] holds all R chunks. */
ra_status ra_all_gather(ra_handle h, void* const* buf, void* stream);

/* ReduceScatter into compact outputs (the layout of NCCL's ReduceScatter):
 * in[r] holds n elements; out[r] holds only rank r's chunk, (r+1) mod R,
 * len elements as ra_owned_chunk reports (a rank whose chunk is empty gets
 * no write and its out[r] is not looked at).  Buffers must not overlap, except
 * inputs with each other.  Runs the direct kernel whatever RA_OPT_VARIANT
 * says; when the chunk starts are not 16-byte aligned (ragged plans),
 * element-wide accesses are used. */
ra_status ra_reduce_scatter_compact(ra_handle h, const void* const* in, void* const* out, void* stream);

/* AllGather from compact inputs: in[r] holds rank r's chunk, (r+1) mod R
 * (len elements as ra_owned_chunk reports); out[r] gets all n elements.
 * Buffers must not overlap, except inputs with each other.  Direct kernel,
 * as ra_reduce_scatter_compact. */
ra_status ra_all_gather_compact(ra_handle h, const void* const* in, void* const* out, void* stream);

/* Ring AllReduce (sections 4-9): out[r] = S for every r. */
ra_status ra_allreduce(ra_handle h, const void* const* in, void* const* out, void* stream);

/* Ring AllReduce (sections 4-9) of R buffers in HOST memory: host_out[r] =
 * S for every r, computed by the direct kernel on device copies.  host_in and
 * host_out are R host pointers to n elements each (any alignment; in place,
 * host_in[r] == host_out[r], allowed; other overlaps are RA_ERR_INVALID, and
 * device or managed memory is RA_ERR_INVALID -- use ra_allreduce).  Page-
 * locked memory (cudaHostAlloc, cudaHostRegister) lets the copies run
 * asynchronously and overlap; pageable memory works, with the CUDA runtime's
 * synchronous copies.  The handle owns two sets of device copies, used by
 * alternate calls (4 R n b bytes, allocated on the first call, RA_ERR_OOM if
 * that fails, freed by ra_destroy).  The elements are processed in up to 8
 * windows (RA_OPT_HOST_WINDOWS; by default at least 32 MiB per rank each,
 * boundaries on 2 MiB multiples of the buffers): window j's inputs are copied
 * in on one internal stream, folded on `stream`, and copied out on another,
 * so window j+1 comes in while window j is folded and window j-1 goes out (a
 * window moves in R copies per direction).  A call's copies in start after everything before it on
 * `stream`, the previous call on that stream included; calls issued on two
 * streams overlap, the second one's copies in running alongside the first
 * one's copies out (each set of device copies passes from a call to the call
 * after next, window by window, in order).
 * Asynchronous on `stream` like ra_allreduce: work
 * already on `stream` comes first, later work on `stream` sees host_out
 * complete; host_in must not change and host_out must not be read before
 * that.  Not capturable into a CUDA graph (RA_ERR_UNSUPPORTED while `stream`
 * captures).  RA_OPT_VARIANT does not apply. */
ra_status ra_allreduce_host(ra_handle h, const void* const* host_in, void* const* host_out, void* stream);

/* Host only, needs no device: the chunk plan of section 12 as read here.
 * off[k], len[k] for k < R (arrays of R entries owned by the caller). */
ra_status ra_chunk_plan(int R, size_t n, size_t* off, size_t* len);

/* The chunk rank r holds complete after ReduceScatter: (r+1) mod R. */
ra_status ra_owned_chunk(ra_handle h, int r, size_t* off, size_t* len);

ra_status ra_set_option(ra_handle h, int key, long long value);
ra_status ra_get_option(ra_handle h, int key, long long* value);

/* Synchronise `stream`, then read the device error record into *err (may
 * be NULL).  Returns RA_ERR_TIMEOUT when a wait gave up since the last
 * read; the record and the handle's signal slots are then reset, so the
 * handle can be used again. */
ra_status ra_get_device_status(ra_handle h, void* stream, ra_device_error* err);

/* Synchronise the device and read the signal array of the last persistent
 * or pipelined launch (its kind and scheme) into dst (host array of cap
 * entries): readSignal on the device, so each entry is the low
 * RA_OPT_SIGNAL_BITS bits of its signal (all 64 by default).  With dst ==
 * NULL only the sizes are returned.  *count gets the
 * entries, *channels the channel count G, *calls how many calls of that kind
 * and scheme ran since the array was last zeroed, *rounds:
 *   counting barrier  [G][rounds][R] (rounds = barrier rounds of a call:
 *                     passes x (2R-3) for AllReduce, passes x (R-2) for
 *                     ReduceScatter or AllGather, passes ordered before the
 *                     rounds of a pass); every entry equals calls * (R - 1),
 *                     as does every shadow (ra_read_shadows)
 *   per-peer barrier  [G][rounds][R waiters][R peers]; every entry equals
 *                     calls, except waiter == peer, which stays 0
 *   pipelined flags   [G][R][J] (rounds = ring rounds, J = count / (G R));
 *                     every entry equals calls * rounds (SignalAdd of 1 per
 *                     finished round), as does every waiter's shadow of its
 *                     predecessor's flag (ra_read_shadows, laid out by
 *                     waiter) */
ra_status ra_read_signals(ra_handle h, uint64_t* dst, size_t cap, size_t* count,
                          int* channels, int* rounds, long long* calls);

/* AllReduce that allocates nothing.  The pages have no counterpart: this
 * is a library convenience, not a step of the ring.
 *
 * For callers that may not allocate device memory: code whose device memory
 * belongs to another allocator (a framework's caching allocator, a host
 * process that gives plug-ins a fixed memory budget) and may not call
 * cudaMalloc, and code that cannot accept the device-wide synchronisation of
 * cudaFree.  ra_create allocates the persistent variant's scratch (signal
 * slots, error record); this call needs no handle and takes that scratch from
 * a fixed array inside the library instead: 256 KiB of signal slots plus a
 * 256-byte error record, held on every GPU that loads the library until the
 * process exits.  It runs the persistent variant (one cooperative launch,
 * counting barrier between rounds) with results bitwise equal to
 * ra_allreduce's.
 *
 * Arguments as for ra_allreduce, with R in [2, 32] and n <= 2^40; the
 * scratch a call needs, (2R-3) * R slots per channel, always fits for one
 * channel, and the channel count is limited to what fits (every co-resident
 * channel up to R = 10, 8 channels at R = 32).  Every buffer must be device
 * (or managed) memory of the current device: each is checked with
 * cudaPointerGetAttributes, which allocates nothing.  Host-side argument
 * errors (including host memory, unknown addresses and another device's
 * memory) return RA_ERR_INVALID and enqueue nothing.  No cudaMalloc,
 * cudaFree or other allocating call is made.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and keeps it for the life of the
 * process; make that first call before any stream capture, and do not use
 * this entry point on a device after cudaDeviceReset (the module, and with
 * it the array, may then be loaded at another address).  Every call clears the part of the array it uses (an async memset
 * on `stream`) before its kernel, so nothing carries over from the previous
 * call.  All calls share the one array: calls that overlap on the GPU (other
 * streams, other threads) race on it and give wrong results.  A barrier wait
 * that runs out (1 s) ends the kernel early, records the fact in the array's
 * error record and leaves the outputs undefined; this entry point does not
 * report it -- callers that need that report use a handle and
 * ra_get_device_status. */
ra_status ra_allreduce_noalloc(int R, size_t n, ra_dtype dtype, ra_op op, const void* const* in,
                               void* const* out, void* stream);

/* The waiters' shadows after the last persistent call with the counting
 * barrier or the last pipelined call, laid out as the signals: each waiter
 * moves its own shadow forward by R-1 per call (counting barrier) or by 1 per
 * round (a pipelined rank's shadow of its predecessor's flag) and waits for
 * the signal to meet it ("comm: lift the GIN scale-out ceiling ...", section
 * "Fix"; the GIN article's increaseSignalShadow / waitSignalMeetShadow), so
 * after a successful call every shadow equals its signal.  The raw 64-bit
 * values.  With dst == NULL only *count is set. */
ra_status ra_read_shadows(ra_handle h, uint64_t* dst, size_t cap, size_t* count);

/* Set every signal of the counting barrier and of the pipelined flags that
 * the handle holds to `signal_value` (resetSignal, then SignalAdd of the
 * value) and every shadow to `shadow_value`, on the device, and synchronise.
 * For tests of wrap-around and of the comparison width (RA_OPT_SIGNAL_BITS):
 * the barrier and the flags compare each signal with its waiter's shadow,
 * never with a count from 0, so any start value works as long as signal and
 * shadow agree on the compared bits.  The slots keep the channel and pass
 * layout of the last call; a call with another layout zeroes them again.
 * The per-peer barrier's slots, which count calls, are left alone.  Do not
 * call it while a call of the handle may be running. */
ra_status ra_seed_signals(ra_handle h, uint64_t signal_value, uint64_t shadow_value);

/* Builds with bounds checks (libra_gb300_debug.so, compiled with
 * -DRA_DEBUG_BOUNDS) only.  There every global access of every kernel is first
 * checked against the byte ranges of the call's buffers and of the handle's
 * device memory; an access outside all of them is counted and skipped (a load
 * reads zero), so a wrong index shows up here instead of as a memory fault.
 * This call synchronises the device and returns how many such accesses there
 * were since the last reset (*count) and the address of the first one
 * (*first_address, 0 if none); a non-zero `reset` clears both.  Such builds
 * launch the ring variant directly (no CUDA graphs) and are not capturable.
 * RA_ERR_UNSUPPORTED in other builds. */
ra_status ra_debug_bounds_report(unsigned long long* count, unsigned long long* first_address, int reset);

/* Text of the calling thread's last error ("" if none). */
const char* ra_last_error(void);

/* Name of a status code. */
const char* ra_status_string(ra_status s);

#ifdef __cplusplus
}
#endif

#endif /* RING_ALLREDUCE_GB300_RA_H */
