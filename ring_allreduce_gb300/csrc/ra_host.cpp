// ra_host.cpp -- host runtime behind the C ABI of include/ra.h: handles,
// argument checks, the chunk plan, variant selection, launches and errors.
//
// The chunk plan is the ring page's section 12 ("Why AllReduce =
// ReduceScatter + AllGather -- NCCL Ring AllReduce": N elements cut into k
// chunks of about N/k), read as C = ceil(n/R), chunk k = [kC, min((k+1)C, n)).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "ra.h"
#include "ra_internal.h"
#include "ra_ll.h"

namespace {

thread_local std::string g_last_error;

ra_status fail(ra_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

ra_status cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();  // clear a non-sticky error so the next call starts clean
  ra_status s = RA_ERR_CUDA;
  if (e == cudaErrorMemoryAllocation) s = RA_ERR_OOM;
  if (e == cudaErrorCooperativeLaunchTooLarge) s = RA_ERR_UNSUPPORTED;
  return fail(s, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t elem_bytes(ra_dtype d) {
  switch (d) {
    case RA_BF16: case RA_F16: return 2;
    case RA_F64: case RA_I64: return 8;
    default: return 4;
  }
}

// Switch to the handle's device for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Signal slots of one synchronisation scheme (counting barrier, per-peer
// barrier, pipelined flags) and one kind of call (AllReduce, ReduceScatter,
// AllGather).
struct SlotRegion {
  uint64_t* d = nullptr;
  uint64_t* shadows = nullptr;   // counting barrier: the waiters' shadows, cap entries after d
  size_t cap = 0;       // entries (signals; the shadows take as many again)
  bool owned = false;   // allocated on its own (the counting slots share one allocation)
  int G = 0;            // channel count the slots were last used with
  int J = 0;            // sub-slices (pipelined flags)
  int rounds = 0;       // ring rounds of this kind
  long long calls = 0;  // completed-or-enqueued calls since the last reset
  // pipelined flags: the value every waiter's shadow starts the next call at
  // (0 after a reset, the seeded value after ra_seed_signals, moved by the
  // ring rounds with every call)
  uint64_t shadow_base = 0;
  // per-peer and flags: a launch of this region was captured into a CUDA
  // graph, so the host's epoch / shadow start no longer follow the device:
  // every launch takes them from the CTAs' own copies until the next reset
  bool from_memory = false;
};

enum Kind { kKindAllReduce = 0, kKindReduceScatter = 1, kKindAllGather = 2 };
constexpr int kMaxSlices = 64;
constexpr int kMaxPasses = 8;   // passes of the persistent variant (counting or cluster barrier)

}  // namespace

constexpr int kHostWindows = 8;   // ra_allreduce_host pipeline depth
constexpr size_t kHostWindowBytes = (size_t)32 << 20;   // least bytes per rank and window
constexpr size_t kHostWindowAlign = (size_t)2 << 20;    // window boundaries, in bytes

struct ra_ctx {
  int R = 0;
  size_t n = 0;
  ra_dtype dtype = RA_F32;
  ra_op op = RA_SUM;
  int device = 0;
  int num_sms = 0;
  int persist_blocks_per_sm = 0;
  int pipe_blocks_per_sm = 0;
  int local_blocks_per_sm = 0;
  int barrier = RA_BARRIER_COUNTING;
  int slices = 0;
  int window = 0;   // RA_OPT_WINDOW
  int gather = 0;   // RA_OPT_GATHER
  int variant = RA_VARIANT_AUTO;
  long long timeout_ns = 1000000000LL;
  int signal_bits = 64;   // RA_OPT_SIGNAL_BITS
  int protocol = RA_PROTOCOL_SIMPLE;   // RA_OPT_PROTOCOL
  int ll_blocks_per_sm = 0;
  // RA_PROTOCOL_LL: the inbox (allocated on first use) and the flag the next
  // call's first message carries
  uint64_t* ll_inbox = nullptr;
  size_t ll_inbox_words = 0;   // the inbox's words, then one flag-base word per co-resident CTA
  size_t ll_alloc_words = 0;
  uint64_t ll_flag = 1;
  bool ll_from_memory = false;   // an LL launch was captured: bases come from the CTAs' copies
  int ctas = 0;
  int check_pointers = 1;
  long long skip = -1;
  uint64_t* d_slots = nullptr;
  ra_device_error* d_err = nullptr;
  SlotRegion region[3][3];   // [ra::Sync][Kind]
  int last_sync = -1;
  int last_kind = -1;
  // the last pointer set that passed the device-memory check: a call on the
  // same buffers does not query their attributes again
  bool checked_valid = false;
  bool checked_has_in = false;
  const void* checked_in[ra::kMaxRanks] = {};
  void* checked_out[ra::kMaxRanks] = {};
  // the ring variant's 2(R-1) launches, captured once per buffer set and
  // replayed as one CUDA graph
  int use_graphs = 1;
  cudaStream_t capture_stream = nullptr;
  cudaGraphExec_t ring_exec = nullptr;
  int ring_kind = -1;
  const void* ring_in[ra::kMaxRanks] = {};
  void* ring_out[ra::kMaxRanks] = {};
  // ra_allreduce_host: two sets of device copies of the R inputs and R
  // outputs, used by alternate calls (set s: inputs then outputs, rank r at
  // element r * host_n_pad of each), two copy streams and one event per set,
  // stage and window; allocated on first use
  char* host_dev = nullptr;
  size_t host_n_pad = 0;
  cudaStream_t host_s_in = nullptr, host_s_out = nullptr;
  cudaEvent_t host_start = nullptr;
  cudaEvent_t host_ev[2][3][kHostWindows] = {};   // [set][in, fold, out][window]
  int host_set = 0;                               // the set the next call uses
  int64_t host_step = 0;                          // window size of the last call (elements)
  bool host_ready = false;                        // every staging resource exists
  int host_windows = 0;   // RA_OPT_HOST_WINDOWS
  long long debug_shrink = 0;   // RA_OPT_DEBUG_SHRINK (debug builds)
};

#ifdef RA_DEBUG_BOUNDS
namespace ra {

DebugTable& debug_table() {
  static thread_local DebugTable t;
  return t;
}

DebugReport* debug_report() {
  static DebugReport* rep = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!rep) {
    if (cudaMalloc(&rep, sizeof(DebugReport)) != cudaSuccess || cudaMemset(rep, 0, sizeof(*rep)) != cudaSuccess) {
      cudaGetLastError();
      rep = nullptr;
    }
  }
  return rep;
}

}  // namespace ra
#endif

namespace {

void debug_add(const void* p, size_t bytes);   // bounds checks of debug builds, below


bool valid_dtype(int d) { return d >= RA_F32 && d <= RA_I64; }
bool valid_op(int o) { return o == RA_SUM || o == RA_MAX; }

ra::Plan make_plan(int R, size_t n) {
  ra::Plan p;
  p.n = (int64_t)n;
  p.C = (int64_t)((n + (size_t)R - 1) / (size_t)R);
  return p;
}

bool overlap(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + bytes && y < x + bytes;
}

ra_status check_device_pointer(const ra_ctx* h, const void* p, const char* name, int r) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RA_ERR_INVALID, "%s[%d]=%p: not a CUDA pointer (%s)", name, r, p, cudaGetErrorName(e));
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
    return fail(RA_ERR_INVALID, "%s[%d]=%p: not device memory", name, r, p);
  if (at.type == cudaMemoryTypeDevice && at.device != h->device)
    return fail(RA_ERR_INVALID, "%s[%d]=%p: memory of device %d, handle is on device %d", name, r, p,
                at.device, h->device);
  return RA_OK;
}

// in may equal out (then only `out` is checked); in == nullptr means an
// in-place AllGather over out.
bool same_as_checked(const ra_ctx* h, const void* const* in, void* const* out) {
  if (!h->checked_valid || h->checked_has_in != (in != nullptr)) return false;
  for (int r = 0; r < h->R; ++r) {
    if (out[r] != h->checked_out[r]) return false;
    if (in && in[r] != h->checked_in[r]) return false;
  }
  return true;
}

ra_status check_buffers(ra_ctx* h, const void* const* in, void* const* out) {
  const int R = h->R;
  const size_t bytes = h->n * elem_bytes(h->dtype);
  if (!out) return fail(RA_ERR_INVALID, "NULL pointer array");
  if (bytes == 0) return RA_OK;  // nothing is accessed: any pointers do
  for (int r = 0; r < R; ++r) {
    if (in && !in[r]) return fail(RA_ERR_INVALID, "in[%d] is NULL", r);
    if (!out[r]) return fail(RA_ERR_INVALID, "%s[%d] is NULL", in ? "out" : "buf", r);
    if (in && ((uintptr_t)in[r] & 15u)) return fail(RA_ERR_INVALID, "in[%d]=%p is not 16-byte aligned", r, in[r]);
    if ((uintptr_t)out[r] & 15u)
      return fail(RA_ERR_INVALID, "%s[%d]=%p is not 16-byte aligned", in ? "out" : "buf", r, out[r]);
  }
  for (int r = 0; r < R; ++r) {
    for (int q = 0; q < R; ++q) {
      if (q != r && overlap(out[r], out[q], bytes))
        return fail(RA_ERR_INVALID, "output buffers %d and %d overlap", r, q);
      if (in) {
        const bool same = (q == r) && (in[q] == out[r]);
        if (!same && overlap(out[r], in[q], bytes))
          return fail(RA_ERR_INVALID, "out[%d] overlaps in[%d] (only out[r] == in[r] is allowed)", r, q);
      }
    }
  }
  if (h->check_pointers && !same_as_checked(h, in, out)) {
    h->checked_valid = false;
    for (int r = 0; r < R; ++r) {
      if (in && in[r] != out[r]) {
        ra_status s = check_device_pointer(h, in[r], "in", r);
        if (s != RA_OK) return s;
      }
      ra_status s = check_device_pointer(h, out[r], in ? "out" : "buf", r);
      if (s != RA_OK) return s;
    }
    for (int r = 0; r < R; ++r) {
      h->checked_in[r] = in ? in[r] : nullptr;
      h->checked_out[r] = out[r];
    }
    h->checked_has_in = in != nullptr;
    h->checked_valid = true;
  }
  return RA_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int vec_elems(ra_dtype d) { return (int)(16 / elem_bytes(d)); }

// Enough CTAs for every thread to take its vectors once (see ra_direct.cu).
int direct_ctas_per_chunk(const ra_ctx* h, const ra::Plan& pl, int mode) {
  if (h->ctas > 0) return h->ctas;
  const int64_t vecs = ceil_div(pl.C, vec_elems(h->dtype)) + 1;
  const int64_t per_cta = (int64_t)ra::kDirectThreads * ra::direct_vectors_per_thread(h->R, mode);
  int64_t c = ceil_div(vecs, per_cta);
  if (c > 65535) c = 65535;
  return (int)(c < 1 ? 1 : c);
}

int round_ctas_per_rank(const ra_ctx* h, const ra::Plan& pl) {
  if (h->ctas > 0) return h->ctas;
  const int64_t vecs = ceil_div(pl.C, vec_elems(h->dtype)) + 1;
  const int64_t need = ceil_div(vecs, ra::kRoundThreads);
  const int64_t target = ceil_div((int64_t)h->num_sms * 8, h->R);
  int64_t c = need < target ? need : target;
  return (int)(c < 1 ? 1 : c);
}

// AllGather round: at most one CTA per 16 KB of a chunk, and up to 3 CTAs
// (64 KB of staging each) per SM over the R ranks.
int copy_ctas_per_rank(const ra_ctx* h, const ra::Plan& pl) {
  if (h->ctas > 0) return h->ctas;
  const int64_t tiles = ceil_div(pl.C * (int64_t)elem_bytes(h->dtype), 16384) + 1;
  const int64_t target = ceil_div((int64_t)h->num_sms * 3, h->R);
  int64_t c = tiles < target ? tiles : target;
  return (int)(c < 1 ? 1 : c);
}

// Channels of the persistent and pipelined variants when RA_OPT_CTAS is 0:
// one per 128 vectors of a chunk up to 16 -- a round's latency falls as its
// slice shrinks (measured at R = 8: 53.6 -> 36.9 us per call at 2^18 fp32 per
// rank), while tiny chunks gain nothing from more CTAs -- then enough for 4
// vectors per thread (`threads` per CTA), up to `most` (one wave).
int64_t default_channels(const ra_ctx* h, const ra::Plan& pl, int64_t most, int threads) {
  const int64_t vecs = ceil_div(pl.C, vec_elems(h->dtype)) + 1;
  int64_t G = std::max<int64_t>(std::min<int64_t>(16, ceil_div(vecs, 128)),
                                ceil_div(vecs, (int64_t)threads * 4));
  if (G > most) G = most;
  return G < 1 ? 1 : G;
}

int persistent_channels(const ra_ctx* h, const ra::Plan& pl) {
  const int cap = h->persist_blocks_per_sm * h->num_sms / h->R;
  const int G = h->ctas > 0 ? h->ctas : (int)default_channels(h, pl, cap, ra::kPersistThreads);
  return G < 1 ? 1 : G;
}

ra::Ptrs make_ptrs(const ra_ctx* h, const void* const* in, void* const* out) {
  ra::Ptrs p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < h->R; ++r) {
    p.in[r] = in ? in[r] : out[r];
    p.out[r] = out[r];
  }
  return p;
}

// The AllGather kernel RA_OPT_GATHER picks (0 = the library's choice).
bool use_bcast(const ra_ctx* h) { return h->gather == 2; }

ra_status run_bcast(ra_ctx* h, const void* const* src, void* const* dst, bool compact_src, cudaStream_t st) {
  ra::BcastArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < h->R; ++r) {
    a.src[r] = src[r];
    a.dst[r] = dst[r];
  }
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.elem_bytes = (int)elem_bytes(h->dtype);
  a.write_owner = compact_src ? 1 : 0;
  a.src_compact = compact_src ? 1 : 0;
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  int64_t ctas = h->ctas;
  if (ctas <= 0) {
    const int64_t tiles = ceil_div(a.plan.C * (int64_t)a.elem_bytes, ra::bcast_tile_bytes()) + 1;
    const int64_t target = ceil_div((int64_t)h->num_sms * 3, h->R);
    ctas = tiles < target ? tiles : target;
  }
  if (ctas > 65535) ctas = 65535;
  if (ctas < 1) ctas = 1;
  cudaError_t e = ra::launch_bcast(a, (int)ctas, st);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "broadcast kernel launch");
}

ra_status run_direct(ra_ctx* h, int mode, const void* const* in, void* const* out, cudaStream_t st) {
  if (mode == ra::kModeAllGather && use_bcast(h)) return run_bcast(h, out, out, false, st);
  ra::DirectArgs a;
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.lo = 0;
  a.hi = a.plan.n;
  a.R = h->R;
  a.mode = mode;
  a.write_owner = 0;
  cudaError_t e = ra::launch_direct(h->dtype, h->op, a, direct_ctas_per_chunk(h, a.plan, mode), st);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "direct kernel launch");
}

// Local variant: slices of SV whole 16-byte vectors per chunk, one CTA per
// slice at a time (grid-stride over slices); RA_OPT_CTAS sets the grid.
ra_status run_local(ra_ctx* h, int mode, const void* const* in, void* const* out, cudaStream_t st) {
  ra::LocalArgs a;
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.mode = mode;
  a.SV = ra::local_slice_vectors(h->R);
  const int64_t V = 16 / (int64_t)elem_bytes(h->dtype);
  int64_t most = 0;
  for (int k = 0; k < h->R; ++k) {
    const int64_t off = std::min((int64_t)k * a.plan.C, a.plan.n);
    const int64_t end = std::min(off + a.plan.C, a.plan.n);
    const int64_t vb = (off + V - 1) / V, ve = end / V;
    if (ve > vb) most = std::max(most, ve - vb);
  }
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  // narrow the slices so that every CTA gets the same number of them (within one)
  int64_t ctas = h->ctas > 0 ? h->ctas : (int64_t)h->num_sms * std::max(1, h->local_blocks_per_sm);
  const int64_t per_cta = std::max<int64_t>(1, ceil_div(ceil_div(most, a.SV), ctas));
  a.SV = (int)std::max<int64_t>(1, std::min<int64_t>(a.SV, ceil_div(most, per_cta * ctas)));
  a.slices = std::max<int64_t>(1, ceil_div(most, a.SV));
  ctas = std::min(ctas, a.slices);
  if (ctas > 0x7fffffff) ctas = 0x7fffffff;
  cudaError_t e = ra::launch_local(h->dtype, h->op, a, (int)ctas, st);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "local kernel launch");
}

// Compact ReduceScatter (compact_out) or AllGather (compact_in): the
// compact side holds rank r's chunk (r+1) mod R only.
ra_status check_compact(ra_ctx* h, const void* const* full, const void* const* compact, bool full_is_input) {
  const int R = h->R;
  const size_t b = elem_bytes(h->dtype);
  size_t off[ra::kMaxRanks], len[ra::kMaxRanks];
  ra_chunk_plan(R, h->n, off, len);
  const char* fname = full_is_input ? "in" : "out";
  const char* cname = full_is_input ? "out" : "in";
  struct Range { const void* p; size_t bytes; const char* name; int r; bool input; };
  Range rs[2 * ra::kMaxRanks];
  int nr = 0;
  for (int r = 0; r < R; ++r) {
    const size_t cb = len[(r + 1) % R] * b;
    if (!full[r]) return fail(RA_ERR_INVALID, "%s[%d] is NULL", fname, r);
    if ((uintptr_t)full[r] & 15u) return fail(RA_ERR_INVALID, "%s[%d]=%p is not 16-byte aligned", fname, r, full[r]);
    rs[nr++] = {full[r], h->n * b, fname, r, full_is_input};
    if (cb == 0) continue;   // an empty chunk: the compact buffer is not accessed
    if (!compact[r]) return fail(RA_ERR_INVALID, "%s[%d] is NULL", cname, r);
    if ((uintptr_t)compact[r] & 15u)
      return fail(RA_ERR_INVALID, "%s[%d]=%p is not 16-byte aligned", cname, r, compact[r]);
    rs[nr++] = {compact[r], cb, cname, r, !full_is_input};
  }
  for (int i = 0; i < nr; ++i)
    for (int j = i + 1; j < nr; ++j) {
      if (rs[i].input && rs[j].input) continue;   // inputs may overlap each other
      const uintptr_t x = (uintptr_t)rs[i].p, y = (uintptr_t)rs[j].p;
      if (x < y + rs[j].bytes && y < x + rs[i].bytes)
        return fail(RA_ERR_INVALID, "%s[%d] overlaps %s[%d]", rs[i].name, rs[i].r, rs[j].name, rs[j].r);
    }
  if (h->check_pointers)
    for (int i = 0; i < nr; ++i) {
      ra_status s = check_device_pointer(h, rs[i].p, rs[i].name, rs[i].r);
      if (s != RA_OK) return s;
    }
  return RA_OK;
}

ra_status run_compact(ra_ctx* h, int mode, const void* const* in, void* const* out, cudaStream_t st) {
  const int R = h->R;
  const size_t b = elem_bytes(h->dtype);
  const ra::Plan pl = make_plan(R, h->n);
  size_t off[ra::kMaxRanks], len[ra::kMaxRanks];
  ra_chunk_plan(R, h->n, off, len);
  if ((pl.C * (int64_t)b) % 16 == 0 && mode == ra::kModeAllGather && use_bcast(h))
    return run_bcast(h, in, out, true, st);
  if ((pl.C * (int64_t)b) % 16 == 0) {
    // every chunk starts on a 16-byte boundary: the direct kernel, with each
    // compact buffer addressed as if it began at its chunk's offset
    ra::DirectArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int r = 0; r < R; ++r) {
      const size_t shift = off[(r + 1) % R] * b;
      if (mode == ra::kModeReduceScatter) {
        a.p.in[r] = in[r];
        a.p.out[r] = static_cast<char*>(out[r]) - shift;
      } else {
        a.p.in[r] = static_cast<const char*>(in[r]) - shift;
        a.p.out[r] = out[r];
      }
    }
    a.plan = pl;
    a.lo = 0;
    a.hi = pl.n;
    a.R = R;
    a.mode = mode;
    a.write_owner = 1;
    cudaError_t e = ra::launch_direct(h->dtype, h->op, a, direct_ctas_per_chunk(h, pl, mode), st);
    return e == cudaSuccess ? RA_OK : cuda_fail(e, "direct kernel launch");
  }
  ra::CompactArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < R; ++r) {
    a.p.in[r] = in[r];
    a.p.out[r] = out[r];
  }
  a.plan = pl;
  a.R = R;
  a.mode = mode;
  int64_t ctas = h->ctas > 0 ? h->ctas : ceil_div(ceil_div(pl.C, vec_elems(h->dtype)) + 1, (int64_t)ra::kCompactThreads);
  if (ctas > 65535) ctas = 65535;
  if (ctas < 1) ctas = 1;
  cudaError_t e = ra::launch_compact(h->dtype, h->op, a, (int)ctas, st);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "compact kernel launch");
}

// Sub-slices of a channel's slice when RA_OPT_SLICES is 0 (pipelined
// variant), and passes of the persistent variant: the fewest that keep the
// partials one round writes over all ranks -- n b / J bytes -- within 32 MiB,
// a quarter of L2, so the successor reads them back from L2; at most 8.
// Each sub-slice or pass adds a wait (pipelined) or barrier (persistent) per
// round, so more of them cost more than they save.  Measured on GB300, fp32,
// every J from 1 to 8, three runs each: R = 8 at 2^23 per rank (32 MiB per
// round): J = 1 best for the persistent variant; 2^24: J = 2-3 (persistent,
// counting barrier, 384 -> 324 us; pipelined 383 -> 339); 2^25: J = 4-6
// (747 -> 631-651); 2^26: J = 8 (1472 -> 1291); R = 2, 16, 32 at 2^24: J = 2-3.
int pipeline_slices(const ra_ctx* h, const ra::Plan& pl) {
  if (h->slices > 0) return h->slices;
  const int64_t round_bytes = pl.n * (int64_t)elem_bytes(h->dtype);
  int64_t J = ceil_div(round_bytes, (int64_t)32 << 20);
  if (J > 8) J = 8;
  return (int)(J < 1 ? 1 : J);
}

// Passes of the persistent variant (counting or cluster barrier) and of the
// ring variant: as the pipelined variant's sub-slices, at most kMaxPasses;
// each pass takes one part of every channel slice (ring variant: of every
// chunk) through every round before the next pass starts.
int persistent_passes(const ra_ctx* h, const ra::Plan& pl) {
  return std::min(pipeline_slices(h, pl), kMaxPasses);
}

// The ReduceScatter rounds of pass j of J.
ra_status run_ring_reduce(ra_ctx* h, const void* const* in, void* const* out, int j, int J, cudaStream_t st) {
  ra::RoundArgs a;
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.j = j;
  a.J = J;
  const int ctas = round_ctas_per_rank(h, a.plan);
  for (int s = 1; s < h->R; ++s) {
    a.s = s;
    cudaError_t e = ra::launch_rs_round(h->dtype, h->op, a, ctas, st);
    if (e != cudaSuccess) return cuda_fail(e, "reduce round launch");
  }
  return RA_OK;
}

// The AllGather rounds of pass j of J.
ra_status run_ring_gather(ra_ctx* h, void* const* buf, int j, int J, cudaStream_t st) {
  ra::CopyArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < h->R; ++r) a.buf[r] = buf[r];
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.j = j;
  a.J = J;
  a.elem_bytes = (int)elem_bytes(h->dtype);
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  const int ctas = copy_ctas_per_rank(h, a.plan);
  for (int s = 1; s < h->R; ++s) {
    a.s = s;
    cudaError_t e = ra::launch_ag_round(a, ctas, st);
    if (e != cudaSuccess) return cuda_fail(e, "AllGather round launch");
  }
  return RA_OK;
}

void drop_ring_graph(ra_ctx* h) {
  if (h->ring_exec) cudaGraphExecDestroy(h->ring_exec);
  h->ring_exec = nullptr;
  h->ring_kind = -1;
}

// Every round of every pass, pass after pass (a pass runs all its rounds
// before the next starts).
ra_status run_ring_launches(ra_ctx* h, int kind, const void* const* in, void* const* out, cudaStream_t st) {
  const int J = persistent_passes(h, make_plan(h->R, h->n));
  for (int j = 0; j < J; ++j) {
    ra_status s = RA_OK;
    if (kind != kKindAllGather) s = run_ring_reduce(h, in, out, j, J, st);
    if (s == RA_OK && kind != kKindReduceScatter) s = run_ring_gather(h, out, j, J, st);
    if (s != RA_OK) return s;
  }
  return RA_OK;
}

// Ring variant: replay the cached graph of this call's launches when the
// buffers are those it was captured with; otherwise capture it first.  When
// the caller's own stream is being captured, or graphs are off, launch
// directly (the launches then join the caller's graph).
ra_status run_ring(ra_ctx* h, int kind, const void* const* in, void* const* out, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (!h->use_graphs || !h->capture_stream || cudaStreamIsCapturing(st, &cs) != cudaSuccess ||
      cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return run_ring_launches(h, kind, in, out, st);
  }
  bool same = h->ring_exec && h->ring_kind == kind;
  for (int r = 0; same && r < h->R; ++r)
    same = h->ring_out[r] == out[r] && h->ring_in[r] == (in ? in[r] : nullptr);
  if (!same) {
    drop_ring_graph(h);
    cudaError_t e = cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "ring graph capture");
    ra_status s = run_ring_launches(h, kind, in, out, h->capture_stream);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(h->capture_stream, &g);
    if (s != RA_OK) {
      if (g) cudaGraphDestroy(g);
      return s;
    }
    if (e != cudaSuccess) return cuda_fail(e, "ring graph capture");
    e = cudaGraphInstantiate(&h->ring_exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      h->ring_exec = nullptr;
      return cuda_fail(e, "ring graph instantiation");
    }
    h->ring_kind = kind;
    for (int r = 0; r < h->R; ++r) {
      h->ring_in[r] = in ? in[r] : nullptr;
      h->ring_out[r] = out[r];
    }
  }
  cudaError_t e = cudaGraphLaunch(h->ring_exec, st);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "ring graph launch");
}

int gmax_channels(const ra_ctx* h, int blocks_per_sm) {
  return (blocks_per_sm > 0 ? blocks_per_sm : 1) * h->num_sms / h->R + 1;
}

// Entries of a slot array: counting [G][J passes][barrier rounds][R];
// per-peer [G][barrier rounds][R][R] (always one pass); flags [G][R][J].
size_t region_entries(const ra_ctx* h, int sync, int rounds, int G, int J) {
  const size_t R = (size_t)h->R;
  const size_t br = (size_t)(rounds > 1 ? rounds - 1 : 0);
  if (sync == ra::kSyncCounting) return (size_t)G * (size_t)J * br * R;
  if (sync == ra::kSyncPerPeer) return (size_t)G * br * R * R;
  return (size_t)G * R * (size_t)J;
}

// Words of a region: its signals, and as many shadows after them when it has any.
size_t region_words(const SlotRegion& reg) { return reg.shadows ? 2 * reg.cap : reg.cap; }

// The slot array of (sync, kind), allocated on first use for the per-peer
// barrier and the pipelined flags (the counting slots come with ra_create).
ra_status ensure_region(ra_ctx* h, int sync, int kind, SlotRegion** out) {
  SlotRegion& reg = h->region[sync][kind];
  if (!reg.d) {
    const int bps = sync == ra::kSyncFlags ? h->pipe_blocks_per_sm : h->persist_blocks_per_sm;
    const size_t cap = region_entries(h, sync, reg.rounds, gmax_channels(h, bps), kMaxSlices);
    // the pipelined flags come with their waiters' shadows, laid out as the
    // flags; the per-peer slots with each CTA's copy of its epoch ([G][R],
    // well within cap words)
    const size_t words = 2 * cap;
    if (cap > 0) {
      cudaError_t e = cudaMalloc(&reg.d, words * sizeof(uint64_t));
      if (e == cudaSuccess) e = cudaMemset(reg.d, 0, words * sizeof(uint64_t));
      if (e != cudaSuccess) {
        if (reg.d) cudaFree(reg.d);
        reg.d = nullptr;
        return cuda_fail(e, "signal slot allocation");
      }
      reg.shadows = reg.d + cap;
    }
    reg.cap = cap;
    reg.owned = true;
    reg.G = 0;
    reg.calls = 0;
    debug_add(reg.d, region_words(reg) * sizeof(uint64_t));
  }
  *out = &reg;
  return RA_OK;
}

// Zero a region when the launch shape it was counted with changes.

// ---------------------------------------------------------------- bounds checks
// Debug builds (-DRA_DEBUG_BOUNDS): the byte ranges one call may touch, put in
// this host thread's table (ra::debug_table()) before its launches -- the
// call's buffers and every piece of the handle's device memory; memory the
// call allocates on the way is added when it is allocated.  Release builds:
// nothing.
#ifdef RA_DEBUG_BOUNDS
using ra::debug_report;

void debug_add(const void* p, size_t bytes) {
  ra::DebugTable& t = ra::debug_table();
  if (!p || bytes == 0 || t.count >= ra::kDebugRanges) return;
  t.r[t.count].lo = reinterpret_cast<uint64_t>(p);
  t.r[t.count].hi = reinterpret_cast<uint64_t>(p) + bytes;
  ++t.count;
}

void debug_begin(const ra_ctx* h) {
  ra::DebugTable& t = ra::debug_table();
  t.count = 0;
  t.report = debug_report();
  if (!h) return;
  for (auto& row : h->region)
    for (auto& reg : row)
      if (reg.d) debug_add(reg.d, region_words(reg) * sizeof(uint64_t));
  debug_add(h->d_err, sizeof(ra_device_error));
  if (h->ll_inbox) debug_add(h->ll_inbox, h->ll_alloc_words * sizeof(uint64_t));
  if (h->host_dev) debug_add(h->host_dev, 4 * (size_t)h->R * h->host_n_pad * elem_bytes(h->dtype));
}

// one of the call's own buffers, RA_OPT_DEBUG_SHRINK bytes shorter than it
// is (a test of the checks: the accesses to its last bytes are then reported
// and skipped)
void debug_user(const ra_ctx* h, const void* p, size_t bytes) {
  const size_t cut = (size_t)std::max<long long>(0, h->debug_shrink);
  debug_add(p, bytes > cut ? bytes - cut : 0);
}
#else
void debug_add(const void*, size_t) {}
void debug_begin(const ra_ctx*) {}
void debug_user(const ra_ctx*, const void*, size_t) {}
#endif

void debug_buffers(const ra_ctx* h, const void* const* p, size_t bytes) {
  for (int r = 0; r < h->R; ++r) debug_user(h, p[r], bytes);
}

// Compact calls: the full side n elements per rank, the compact side rank r's
// chunk (r+1) mod R only.
void debug_compact(const ra_ctx* h, const void* const* full, const void* const* compact) {
  size_t off[ra::kMaxRanks], len[ra::kMaxRanks];
  ra_chunk_plan(h->R, h->n, off, len);
  const size_t b = elem_bytes(h->dtype);
  debug_buffers(h, full, h->n * b);
  for (int r = 0; r < h->R; ++r) debug_user(h, compact[r], len[(r + 1) % h->R] * b);
}

// resetSignal on every signal of a region (and its shadows to 0), on the stream.
cudaError_t reset_region(const SlotRegion& reg, cudaStream_t st) {
  if (!reg.d || !reg.cap) return cudaSuccess;
  ra::SignalIoArgs a;
  std::memset(&a, 0, sizeof(a));
  a.signals = reg.d;
  a.shadows = reg.shadows;
  a.count = reg.cap;
  a.op = ra::kSigReset;
  a.bits = 64;
  return ra::launch_signal_io(a, st);
}

ra_status prepare_region(SlotRegion& reg, int G, int J, cudaStream_t st) {
  if (reg.G != G || reg.J != J) {
    cudaError_t e = reset_region(reg, st);
    if (e != cudaSuccess) return cuda_fail(e, "signal slot reset");
    reg.shadow_base = 0;
    reg.from_memory = false;
    reg.G = G;
    reg.J = J;
    reg.calls = 0;
  }
  return RA_OK;
}

// Persistent variant with the R CTAs of each channel in one thread-block
// cluster: no signal memory, no co-residency across channels.
ra_status run_persistent_cluster(ra_ctx* h, int kind, int mode, const void* const* in, void* const* out,
                                 cudaStream_t st) {
  if (h->R > 16) return fail(RA_ERR_UNSUPPORTED, "cluster barrier needs R <= 16 (R=%d)", h->R);
  int clusters = 0;
  cudaError_t e = ra::persistent_cluster_capacity(h->dtype, h->op, h->R, ra::kPersistThreads, &clusters);
  if (e != cudaSuccess) return cuda_fail(e, "cluster occupancy query");
  if (clusters < 1) return fail(RA_ERR_UNSUPPORTED, "a cluster of %d CTAs does not fit", h->R);
  ra::PersistArgs a;
  std::memset(&a, 0, sizeof(a));
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.mode = mode;
  a.sync = ra::kSyncCluster;
  a.rounds = h->region[ra::kSyncCounting][kind].rounds;
  if (h->ctas > 0) {
    a.G = h->ctas;
  } else {
    a.G = (int)default_channels(h, a.plan, clusters, ra::kPersistThreads);   // one wave of clusters
  }
  a.J = persistent_passes(h, a.plan);
  if ((int64_t)a.G * h->R > 2147483647LL) return fail(RA_ERR_UNSUPPORTED, "too many clusters");
  a.epoch = 1;
  a.bits = h->signal_bits;
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  a.skip_rank = -1;
  a.skip_round = -1;
  e = ra::launch_persistent_cluster(h->dtype, h->op, a, ra::kPersistThreads, st);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "cluster kernel launch");
}

// Launches whose per-call state the host passes in as a kernel parameter
// (the per-peer barrier's epoch, the pipelined variant's shadow start and
// LL flag base) would replay that value unchanged from a CUDA graph.  Their
// CTAs also keep that state in device memory, each its own copy; a launch
// made on a stream that is being captured -- and every launch of the same
// state after it, until a reset -- takes it from there instead.
ra_status stream_capturing(cudaStream_t st, bool* capturing) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "stream capture status");
  *capturing = cs != cudaStreamCaptureStatusNone;
  return RA_OK;
}

ra_status run_persistent(ra_ctx* h, int kind, int mode, const void* const* in, void* const* out,
                         cudaStream_t st) {
  if (h->barrier == RA_BARRIER_CLUSTER) return run_persistent_cluster(h, kind, mode, in, out, st);
  const int sync = h->barrier == RA_BARRIER_PER_PEER ? ra::kSyncPerPeer : ra::kSyncCounting;
  bool capturing = false;
  ra_status s = sync == ra::kSyncPerPeer ? stream_capturing(st, &capturing) : RA_OK;
  if (s != RA_OK) return s;
  SlotRegion* reg = nullptr;
  s = ensure_region(h, sync, kind, &reg);
  if (s != RA_OK) return s;
  ra::PersistArgs a;
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.mode = mode;
  a.sync = sync;
  a.rounds = reg->rounds;
  a.G = persistent_channels(h, a.plan);
  a.J = sync == ra::kSyncCounting ? persistent_passes(h, a.plan) : 1;
  const int cap = h->persist_blocks_per_sm * h->num_sms;
  if ((long long)a.G * h->R > cap)
    return fail(RA_ERR_UNSUPPORTED, "persistent grid of %d x %d CTAs cannot be co-resident (%d fit)", h->R, a.G, cap);
  if (region_entries(h, sync, a.rounds, a.G, a.J) > reg->cap)
    return fail(RA_ERR_UNSUPPORTED, "too many channels for the signal slots");
  s = prepare_region(*reg, a.G, a.J, st);
  if (s != RA_OK) return s;
  a.slots = reg->d;
  a.shadows = reg->shadows;
  a.epoch = (uint64_t)(reg->calls + 1);
  a.shadow_base = 0;
  if (capturing) reg->from_memory = true;
  a.from_memory = reg->from_memory ? 1 : 0;
  a.bits = h->signal_bits;
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  a.skip_rank = h->skip >= 0 ? (int)(h->skip >> 16) : -1;
  a.skip_round = h->skip >= 0 ? (int)(h->skip & 0xFFFF) : -1;
  cudaError_t e = ra::launch_persistent(h->dtype, h->op, a, ra::kPersistThreads, st);
  if (e != cudaSuccess) return cuda_fail(e, "persistent kernel launch");
  reg->calls += 1;
  h->last_sync = sync;
  h->last_kind = kind;
  return RA_OK;
}

// Sub-slices per window: the rounds run over W sub-slices before the next W.
// Default 1: every round on one sub-slice, then the next (measured fastest
// for every J from 2 to 8; at J = 4, R = 8, 2^24 fp32 per rank: W = 1 342 us,
// 2 381 us, 4 408 us).
int pipeline_window(const ra_ctx* h, int J) {
  if (h->window > 0) return std::min(h->window, J);
  return 1;
}

constexpr size_t kLLInboxBytes = (size_t)64 << 20;   // most bytes of the RA_PROTOCOL_LL inbox
constexpr long long kMaxTimeoutNs = 60LL * 1000 * 1000 * 1000;   // RA_OPT_TIMEOUT_NS at most (60 s)

// The pipelined variant with flag-in-data messages (ra_ll.cu).
ra_status run_pipelined_ll(ra_ctx* h, int kind, int mode, const void* const* in, void* const* out,
                           bool capturing, cudaStream_t st) {
  ra::LLArgs a;
  std::memset(&a, 0, sizeof(a));
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.mode = mode;
  a.elem_bytes = (int)elem_bytes(h->dtype);
  a.rounds = h->region[ra::kSyncFlags][kind].rounds;
  const int64_t C = a.plan.C;
  const int wpe = ra::ll_words_per_element(a.elem_bytes);
  // rows: the most messages a call sends (AllReduce: 2R-3) x receiving ranks
  const size_t words = (size_t)(2 * h->R - 3) * (size_t)h->R * (size_t)C * (size_t)wpe;
  if (words > kLLInboxBytes / sizeof(uint64_t))
    return fail(RA_ERR_UNSUPPORTED, "LL protocol: chunks of %lld elements need a %zu-byte inbox (at most %zu)",
                (long long)C, words * sizeof(uint64_t), kLLInboxBytes);
  // threads per CTA, positions per thread (E) and channels (G): one position
  // per thread while the channels can be co-resident
  const int threads = (int)std::min<int64_t>(ra::kLLThreads, std::max<int64_t>(32, (C + 31) / 32 * 32));
  const int cap = h->ll_blocks_per_sm * h->num_sms;
  if (h->ctas > 0) {
    a.G = h->ctas;
    a.E = (int)std::max<int64_t>(1, (C + (int64_t)a.G * threads - 1) / ((int64_t)a.G * threads));
  } else {
    const int64_t gmax = std::max(1, cap / h->R);
    a.E = (int)std::max<int64_t>(1, (C + gmax * threads - 1) / (gmax * threads));
    a.G = (int)std::max<int64_t>(1, (C + (int64_t)threads * a.E - 1) / ((int64_t)threads * a.E));
  }
  if (a.E > ra::kLLMaxE)
    return fail(RA_ERR_UNSUPPORTED, "LL protocol: %d channels of %d threads cannot carry %lld-element chunks", a.G,
                threads, (long long)C);
  if ((long long)a.G * h->R > cap)
    return fail(RA_ERR_UNSUPPORTED, "LL grid of %d x %d CTAs cannot be co-resident (%d fit)", h->R, a.G, cap);
  if (!h->ll_inbox) {
    // the inbox, then each co-resident CTA's copy of its next flag base
    const size_t all = words + (size_t)std::max(cap, 1);
    cudaError_t e = cudaMalloc(&h->ll_inbox, all * sizeof(uint64_t));
    if (e == cudaSuccess) e = cudaMemset(h->ll_inbox, 0, all * sizeof(uint64_t));
    if (e != cudaSuccess) {
      if (h->ll_inbox) cudaFree(h->ll_inbox);
      h->ll_inbox = nullptr;
      return cuda_fail(e, "LL inbox allocation");
    }
    h->ll_inbox_words = words;
    h->ll_alloc_words = all;
    h->ll_from_memory = false;   // any flag (1 by default, or as RA_OPT_LL_FLAG set it) suits a zeroed inbox
    debug_add(h->ll_inbox, all * sizeof(uint64_t));
  }
  if (capturing) h->ll_from_memory = true;
  // flags never wrap: a call from the host whose flags would pass 2^32 - 1
  // starts again at 1 on a zeroed inbox (0 marks a word never written); a
  // replayed call whose flags would wrap gives up (code 6) and the status
  // call that reports it zeroes the inbox
  if (!h->ll_from_memory && h->ll_flag + (uint64_t)a.rounds > 0xFFFFFFFFull) {
    const cudaError_t e = cudaMemsetAsync(h->ll_inbox, 0, h->ll_alloc_words * sizeof(uint64_t), st);
    if (e != cudaSuccess) return cuda_fail(e, "LL inbox reset");
    h->ll_flag = 1;
  }
  a.inbox = h->ll_inbox;
  a.bases = h->ll_inbox + h->ll_inbox_words;
  a.nbases = (int)(h->ll_alloc_words - h->ll_inbox_words);
  a.from_memory = h->ll_from_memory ? 1 : 0;
  a.flag_base = (uint32_t)h->ll_flag;
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  a.skip_rank = h->skip >= 0 ? (int)(h->skip >> 16) : -1;
  a.skip_round = h->skip >= 0 ? (int)(h->skip & 0xFFFF) : -1;
  const cudaError_t e = ra::launch_ll(h->dtype, h->op, a, threads, st);
  if (e != cudaSuccess) return cuda_fail(e, "LL kernel launch");
  h->ll_flag += (uint64_t)a.rounds;
  return RA_OK;
}

// The pipelined variant with flag-in-data messages through distributed
// shared memory (ra_ll.cu): one cluster of R CTAs per channel.
ra_status run_pipelined_ll_cluster(ra_ctx* h, int kind, int mode, const void* const* in, void* const* out,
                                   cudaStream_t st) {
  if (h->R > 16) return fail(RA_ERR_UNSUPPORTED, "LL_CLUSTER protocol needs R <= 16 (R=%d)", h->R);
  ra::LLArgs a;
  std::memset(&a, 0, sizeof(a));
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.mode = mode;
  a.elem_bytes = (int)elem_bytes(h->dtype);
  a.rounds = h->region[ra::kSyncFlags][kind].rounds;
  const int64_t C = a.plan.C;
  const int threads = (int)std::min<int64_t>(ra::kLLThreads, std::max<int64_t>(32, (C + 31) / 32 * 32));
  if (h->ctas > 0) {
    a.G = h->ctas;
    a.E = (int)std::max<int64_t>(1, (C + (int64_t)a.G * threads - 1) / ((int64_t)a.G * threads));
  } else {
    // one position per thread; channels are independent clusters, so any
    // number of them may run one wave after another
    a.E = 1;
    a.G = (int)std::max<int64_t>(1, (C + threads - 1) / threads);
  }
  if (a.E > ra::kLLMaxE)
    return fail(RA_ERR_UNSUPPORTED, "LL_CLUSTER protocol: %d channels of %d threads cannot carry %lld-element chunks",
                a.G, threads, (long long)C);
  if ((int64_t)a.G * h->R > 2147483647LL) return fail(RA_ERR_UNSUPPORTED, "too many clusters");
  const size_t smem = ra::ll_cluster_smem_bytes(a, threads, a.elem_bytes);
  if (smem > (size_t)ra::kLLClusterMaxSmem)
    return fail(RA_ERR_UNSUPPORTED, "LL_CLUSTER protocol: %zu bytes of rows per CTA (at most %d)", smem,
                ra::kLLClusterMaxSmem);
  int clusters = 0;
  cudaError_t e = ra::ll_cluster_capacity(h->dtype, h->op, a, threads, smem, &clusters);
  if (e != cudaSuccess) return cuda_fail(e, "cluster occupancy query");
  if (clusters < 1) return fail(RA_ERR_UNSUPPORTED, "a cluster of %d CTAs with %zu bytes each does not fit", h->R, smem);
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  a.skip_rank = h->skip >= 0 ? (int)(h->skip >> 16) : -1;
  a.skip_round = h->skip >= 0 ? (int)(h->skip & 0xFFFF) : -1;
  e = ra::launch_ll_cluster(h->dtype, h->op, a, threads, smem, st);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "LL_CLUSTER kernel launch");
}

ra_status run_pipelined(ra_ctx* h, int kind, int mode, const void* const* in, void* const* out,
                        cudaStream_t st) {
  // nothing of the cluster form is kept between calls: a graph may replay it
  if (h->protocol == RA_PROTOCOL_LL_CLUSTER) return run_pipelined_ll_cluster(h, kind, mode, in, out, st);
  bool capturing = false;
  ra_status s = stream_capturing(st, &capturing);
  if (s != RA_OK) return s;
  if (h->protocol == RA_PROTOCOL_LL) return run_pipelined_ll(h, kind, mode, in, out, capturing, st);
  SlotRegion* reg = nullptr;
  s = ensure_region(h, ra::kSyncFlags, kind, &reg);
  if (s != RA_OK) return s;
  ra::PersistArgs a;
  a.p = make_ptrs(h, in, out);
  a.plan = make_plan(h->R, h->n);
  a.R = h->R;
  a.mode = mode;
  a.sync = ra::kSyncFlags;
  a.rounds = reg->rounds;
  const int cap = h->pipe_blocks_per_sm * h->num_sms;
  if (h->ctas > 0) {
    a.G = h->ctas;
  } else {
    a.G = (int)default_channels(h, a.plan, cap / h->R, ra::kPipeThreads);
  }
  if ((long long)a.G * h->R > cap)
    return fail(RA_ERR_UNSUPPORTED, "pipelined grid of %d x %d CTAs cannot be co-resident (%d fit)", h->R, a.G, cap);
  a.J = pipeline_slices(h, a.plan);
  a.W = pipeline_window(h, a.J);
  if (region_entries(h, ra::kSyncFlags, a.rounds, a.G, a.J) > reg->cap)
    return fail(RA_ERR_UNSUPPORTED, "too many channels or sub-slices for the progress flags");
  s = prepare_region(*reg, a.G, a.J, st);
  if (s != RA_OK) return s;
  a.slots = reg->d;
  a.shadows = reg->shadows;
  a.epoch = (uint64_t)(reg->calls + 1);
  a.shadow_base = 0;
  a.bits = h->signal_bits;
  a.timeout_ns = h->timeout_ns;
  a.err = h->d_err;
  a.skip_rank = h->skip >= 0 ? (int)(h->skip >> 16) : -1;
  a.skip_round = h->skip >= 0 ? (int)(h->skip & 0xFFFF) : -1;
  a.shadow_base = reg->shadow_base;
  if (capturing) reg->from_memory = true;
  a.from_memory = reg->from_memory ? 1 : 0;
  cudaError_t e = ra::launch_pipelined(h->dtype, h->op, a, ra::kPipeThreads, st);
  if (e != cudaSuccess) return cuda_fail(e, "pipelined kernel launch");
  reg->calls += 1;
  reg->shadow_base += (uint64_t)a.rounds;
  h->last_sync = ra::kSyncFlags;
  h->last_kind = kind;
  return RA_OK;
}

ra_status reset_device_state(ra_ctx* h, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(h->d_err, 0, sizeof(ra_device_error), st);
  debug_begin(h);
  for (auto& row : h->region)
    for (auto& reg : row)
      if (e == cudaSuccess) e = reset_region(reg, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "device state reset");
  for (auto& row : h->region)
    for (auto& reg : row) {
      reg.calls = 0;
      reg.shadow_base = 0;
      reg.from_memory = false;
    }
  if (h->ll_inbox) {
    // the LL inbox and the CTAs' flag bases start again too (after a
    // replayed call ran out of flags, the only way back)
    e = cudaMemset(h->ll_inbox, 0, h->ll_alloc_words * sizeof(uint64_t));
    if (e != cudaSuccess) return cuda_fail(e, "LL inbox reset");
    h->ll_flag = 1;
    h->ll_from_memory = false;
  }
  return RA_OK;
}

}  // namespace

namespace ra {

// Error text for entry points defined in other translation units.
ra_status record_error(ra_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

}  // namespace ra

extern "C" {

ra_status ra_chunk_plan(int R, size_t n, size_t* off, size_t* len) {
  if (R < 1 || R > ra::kMaxRanks) return fail(RA_ERR_INVALID, "R=%d outside [1, %d]", R, ra::kMaxRanks);
  if (!off || !len) return fail(RA_ERR_INVALID, "NULL output array");
  const size_t C = (n + (size_t)R - 1) / (size_t)R;
  for (int k = 0; k < R; ++k) {
    size_t lo = (size_t)k * C;
    size_t hi = lo + C;
    if (lo > n) lo = n;
    if (hi > n) hi = n;
    off[k] = lo;
    len[k] = hi - lo;
  }
  return RA_OK;
}

ra_status ra_create(int R, size_t n, ra_dtype dtype, ra_op op, ra_handle* out) {
  if (!out) return fail(RA_ERR_INVALID, "NULL handle pointer");
  if (R < 1 || R > ra::kMaxRanks) return fail(RA_ERR_INVALID, "R=%d outside [1, %d]", R, ra::kMaxRanks);
  if (!valid_dtype(dtype)) return fail(RA_ERR_INVALID, "unknown dtype %d", (int)dtype);
  if (!valid_op(op)) return fail(RA_ERR_INVALID, "unknown op %d", (int)op);
  if (n > ((size_t)1 << 40)) return fail(RA_ERR_INVALID, "n=%zu too large", n);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  int coop = 0;
  e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  int bps = 0, pbps = 0, llbps = 0;
  e = ra::persistent_blocks_per_sm(dtype, op, ra::kPersistThreads, &bps);
  if (e == cudaSuccess) e = ra::pipelined_blocks_per_sm(dtype, op, ra::kPipeThreads, &pbps);
  if (e == cudaSuccess) e = ra::ll_blocks_per_sm(dtype, op, ra::kLLThreads, &llbps);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  e = ra::prepare_ag_round();
  if (e == cudaSuccess) e = ra::prepare_bcast();
  if (e == cudaSuccess) e = ra::prepare_persistent_cluster();
  if (e == cudaSuccess) e = ra::prepare_local();
  if (e == cudaSuccess) e = ra::prepare_ll_cluster();
  if (e != cudaSuccess) return cuda_fail(e, "kernel set-up");
  int lbps = 0;
  if (R >= 2) {
    e = ra::local_blocks_per_sm(dtype, op, R, &lbps);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  }

  ra_ctx* h = new (std::nothrow) ra_ctx();
  if (!h) return fail(RA_ERR_OOM, "host allocation failed");
  h->R = R;
  h->n = n;
  h->dtype = dtype;
  h->op = op;
  h->device = dev;
  h->num_sms = sms;
  h->persist_blocks_per_sm = coop ? bps : 0;
#ifdef RA_DEBUG_BOUNDS
  h->use_graphs = 0;   // the bounds table is uploaded before every launch
#endif
  h->pipe_blocks_per_sm = coop ? pbps : 0;
  h->ll_blocks_per_sm = coop ? llbps : 0;
  h->local_blocks_per_sm = lbps;

  // counting-barrier slots: per kind, the most channels that can be
  // co-resident x the most passes x barrier rounds x waiters (the other
  // schemes allocate theirs on first use)
  const int gmax = gmax_channels(h, bps);
  const int rounds[3] = {2 * (R - 1), R - 1, R - 1};
  size_t total = 0;
  for (int k = 0; k < 3; ++k) {
    for (int sy = 0; sy < 3; ++sy) h->region[sy][k].rounds = rounds[k];
    h->region[ra::kSyncCounting][k].cap = region_entries(h, ra::kSyncCounting, rounds[k], gmax, kMaxPasses);
    total += 2 * h->region[ra::kSyncCounting][k].cap;   // signals and shadows
  }
  if (total > 0) {
    e = cudaMalloc(&h->d_slots, total * sizeof(uint64_t));
    if (e != cudaSuccess) {
      delete h;
      return cuda_fail(e, "signal slot allocation");
    }
    e = cudaMemset(h->d_slots, 0, total * sizeof(uint64_t));
    if (e != cudaSuccess) {
      cudaFree(h->d_slots);
      delete h;
      return cuda_fail(e, "signal slot init");
    }
    size_t o = 0;
    for (auto& r : h->region[ra::kSyncCounting]) {
      r.d = h->d_slots + o;
      r.shadows = r.d + r.cap;
      o += 2 * r.cap;
    }
  }
  e = cudaMalloc(&h->d_err, sizeof(ra_device_error));
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(ra_device_error));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    if (h->d_slots) cudaFree(h->d_slots);
    if (h->d_err) cudaFree(h->d_err);
    delete h;
    return cuda_fail(e, "handle set-up");
  }
  *out = h;
  return RA_OK;
}

ra_status ra_destroy(ra_handle h) {
  if (!h) return RA_OK;
  DeviceGuard g(h->device);
  ra_status s = RA_OK;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) s = cuda_fail(e, "synchronise before destroy");
  drop_ring_graph(h);
  if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
  for (auto& row : h->region)
    for (auto& reg : row)
      if (reg.owned && reg.d) cudaFree(reg.d);
  if (h->d_slots) cudaFree(h->d_slots);
  if (h->d_err) cudaFree(h->d_err);
  if (h->ll_inbox) cudaFree(h->ll_inbox);
  if (h->host_dev) cudaFree(h->host_dev);
  if (h->host_s_in) cudaStreamDestroy(h->host_s_in);
  if (h->host_s_out) cudaStreamDestroy(h->host_s_out);
  if (h->host_start) cudaEventDestroy(h->host_start);
  for (auto& set : h->host_ev)
    for (auto& row : set)
      for (auto& ev : row)
        if (ev) cudaEventDestroy(ev);
  delete h;
  return s;
}

namespace {

ra_status prepare_host_pipe(ra_ctx* h) {
  if (h->host_ready) return RA_OK;
  const size_t b = elem_bytes(h->dtype);
  const size_t n_pad = (h->n + 63) / 64 * 64;   // every rank's copy starts 128-byte aligned
  cudaError_t e = cudaSuccess;
  if (!h->host_dev) {
    e = cudaMalloc(&h->host_dev, 4 * (size_t)h->R * n_pad * b);
    if (e != cudaSuccess) {
      h->host_dev = nullptr;
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? fail(RA_ERR_OOM, "staging for host buffers: %zu bytes",
                                                   4 * (size_t)h->R * n_pad * b)
                                            : cuda_fail(e, "staging allocation");
    }
  }
  h->host_n_pad = n_pad;
  if (!h->host_s_in) e = cudaStreamCreateWithFlags(&h->host_s_in, cudaStreamNonBlocking);
  if (e == cudaSuccess && !h->host_s_out) e = cudaStreamCreateWithFlags(&h->host_s_out, cudaStreamNonBlocking);
  if (e == cudaSuccess && !h->host_start) e = cudaEventCreateWithFlags(&h->host_start, cudaEventDisableTiming);
  for (auto& set : h->host_ev)
    for (auto& row : set)
      for (auto& ev : row)
        if (e == cudaSuccess && !ev) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(e, "staging streams and events");
  debug_add(h->host_dev, 4 * (size_t)h->R * n_pad * b);
  h->host_ready = true;
  return RA_OK;
}

// Host buffers only: device (or managed) memory belongs to ra_allreduce.
ra_status check_host_buffers(ra_ctx* h, const void* const* in, void* const* out) {
  const size_t bytes = h->n * elem_bytes(h->dtype);
  for (int r = 0; r < h->R; ++r) {
    if (!in[r]) return fail(RA_ERR_INVALID, "host_in[%d] is NULL", r);
    if (!out[r]) return fail(RA_ERR_INVALID, "host_out[%d] is NULL", r);
    for (int q = 0; q < h->R; ++q) {
      if (q != r && overlap(out[r], out[q], bytes))
        return fail(RA_ERR_INVALID, "host_out[%d] overlaps host_out[%d]", r, q);
      if (in[q] != out[r] && overlap(in[q], out[r], bytes))
        return fail(RA_ERR_INVALID, "host_in[%d] overlaps host_out[%d]", q, r);
    }
    if (h->check_pointers) {
      for (int side = 0; side < 2; ++side) {
        const void* p = side ? static_cast<const void*>(out[r]) : in[r];
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
          cudaGetLastError();
          continue;   // not known to CUDA: pageable host memory
        }
        if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
          return fail(RA_ERR_INVALID, "%s[%d]=%p is device memory: use ra_allreduce", side ? "host_out" : "host_in",
                      r, p);
      }
    }
  }
  return RA_OK;
}

}  // namespace

ra_status ra_allreduce_host(ra_handle h, const void* const* host_in, void* const* host_out, void* stream) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  if (!host_in || !host_out) return fail(RA_ERR_INVALID, "NULL pointer array");
  DeviceGuard g(h->device);
  if (!g.ok) return fail(RA_ERR_CUDA, "cannot switch to device %d", h->device);
  if (h->n == 0) return RA_OK;
  ra_status s = check_host_buffers(h, host_in, host_out);
  if (s != RA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "stream query");
  if (cap != cudaStreamCaptureStatusNone) return fail(RA_ERR_UNSUPPORTED, "ra_allreduce_host cannot be captured");
  debug_begin(h);
  s = prepare_host_pipe(h);
  if (s != RA_OK) return s;

  const int R = h->R;
  const size_t b = elem_bytes(h->dtype);
  const int64_t n = (int64_t)h->n;
  // windows of whole 16-byte vectors (the last one takes the rest)
  const int64_t vec = 16 / (int64_t)b;
  int W = h->host_windows > 0
              ? h->host_windows
              : (int)std::min<int64_t>(kHostWindows, std::max<int64_t>(1, (int64_t)(h->n * b / kHostWindowBytes)));
  // window boundaries on 2 MiB multiples of each buffer (whole 16-byte vectors
  // when a window is smaller than that)
  const int64_t align = std::max<int64_t>(vec, (int64_t)(kHostWindowAlign / b));
  const int64_t want = ceil_div(n, W);
  const int64_t step = want >= align ? ceil_div(want, align) * align : ceil_div(want, vec) * vec;
  W = (int)ceil_div(n, step);
  const int set = h->host_set;
  char* d_in = h->host_dev + (size_t)(2 * set) * R * h->host_n_pad * b;
  char* d_out = d_in + (size_t)R * h->host_n_pad * b;
  const void* dev_in[ra::kMaxRanks];
  void* dev_out[ra::kMaxRanks];
  for (int r = 0; r < R; ++r) {
    dev_in[r] = d_in + (size_t)r * h->host_n_pad * b;
    dev_out[r] = d_out + (size_t)r * h->host_n_pad * b;
  }
  ra::DirectArgs a;
  a.p = make_ptrs(h, dev_in, dev_out);
  a.plan = make_plan(R, h->n);
  a.R = R;
  a.mode = ra::kModeAllReduce;
  a.write_owner = 0;
  const int ctas = direct_ctas_per_chunk(h, a.plan, ra::kModeAllReduce);

  // everything before the call on `stream` happens first
  e = cudaEventRecord(h->host_start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->host_s_in, h->host_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->host_s_out, h->host_start, 0);
  // windows of another size than the last call's: the per-window events no
  // longer cover the same elements, so wait for every earlier use of both sets
  if (h->host_step != 0 && h->host_step != step)
    for (auto& set_ev : h->host_ev)
      for (auto& row : set_ev)
        for (cudaEvent_t ev : row) {
          if (e == cudaSuccess) e = cudaStreamWaitEvent(h->host_s_in, ev, 0);
          if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev, 0);
        }
  h->host_step = step;
  for (int j = 0; j < W && e == cudaSuccess; ++j) {
    const int64_t lo = j * step, hi = std::min(n, lo + step);
    const size_t off = (size_t)lo * b, len = (size_t)(hi - lo) * b;
    cudaEvent_t ev_in = h->host_ev[set][0][j], ev_fold = h->host_ev[set][1][j], ev_out = h->host_ev[set][2][j];
    // window j of this set is free once the call before last has folded it
    // (inputs) and copied it out (outputs); events never recorded yet are
    // complete
    e = cudaStreamWaitEvent(h->host_s_in, ev_fold, 0);
    for (int r = 0; r < R && e == cudaSuccess; ++r)
      e = cudaMemcpyAsync(static_cast<char*>(const_cast<void*>(dev_in[r])) + off,
                          static_cast<const char*>(host_in[r]) + off, len, cudaMemcpyHostToDevice, h->host_s_in);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in, h->host_s_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_out, 0);
    if (e == cudaSuccess) {
      a.lo = lo;
      a.hi = hi;
      e = ra::launch_direct(h->dtype, h->op, a, ctas, st);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_fold, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->host_s_out, ev_fold, 0);
    for (int r = 0; r < R && e == cudaSuccess; ++r)
      e = cudaMemcpyAsync(static_cast<char*>(host_out[r]) + off, static_cast<char*>(dev_out[r]) + off, len,
                          cudaMemcpyDeviceToHost, h->host_s_out);
    if (e == cudaSuccess) e = cudaEventRecord(ev_out, h->host_s_out);
  }
  // the caller's stream continues once the last window is back on the host
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->host_ev[set][2][W - 1], 0);
  if (e != cudaSuccess) return cuda_fail(e, "host pipeline");
  h->host_set = 1 - set;
  return RA_OK;
}

ra_status ra_allreduce(ra_handle h, const void* const* in, void* const* out, void* stream) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  if (!in || !out) return fail(RA_ERR_INVALID, "NULL pointer array");
  DeviceGuard g(h->device);
  if (!g.ok) return fail(RA_ERR_CUDA, "cannot switch to device %d", h->device);
  ra_status s = check_buffers(h, in, out);
  if (s != RA_OK) return s;
  debug_begin(h);
  debug_buffers(h, in, h->n * elem_bytes(h->dtype));
  debug_buffers(h, out, h->n * elem_bytes(h->dtype));
  if (h->n == 0) return RA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->R == 1) {
    if (in[0] == out[0]) return RA_OK;
    return run_direct(h, ra::kModeAllReduce, in, out, st);
  }
  switch (h->variant) {
    case RA_VARIANT_RING:
      return run_ring(h, kKindAllReduce, in, out, st);
    case RA_VARIANT_PERSISTENT:
      return run_persistent(h, kKindAllReduce, ra::kModeAllReduce, in, out, st);
    case RA_VARIANT_PIPELINED:
      return run_pipelined(h, kKindAllReduce, ra::kModeAllReduce, in, out, st);
    case RA_VARIANT_LOCAL:
      return run_local(h, ra::kModeAllReduce, in, out, st);
    default:
      return run_direct(h, ra::kModeAllReduce, in, out, st);
  }
}

ra_status ra_reduce_scatter(ra_handle h, const void* const* in, void* const* out, void* stream) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  if (!in || !out) return fail(RA_ERR_INVALID, "NULL pointer array");
  DeviceGuard g(h->device);
  if (!g.ok) return fail(RA_ERR_CUDA, "cannot switch to device %d", h->device);
  ra_status s = check_buffers(h, in, out);
  if (s != RA_OK) return s;
  debug_begin(h);
  debug_buffers(h, in, h->n * elem_bytes(h->dtype));
  debug_buffers(h, out, h->n * elem_bytes(h->dtype));
  if (h->n == 0) return RA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->R == 1) {
    if (in[0] == out[0]) return RA_OK;
    return run_direct(h, ra::kModeAllReduce, in, out, st);
  }
  switch (h->variant) {
    case RA_VARIANT_RING:
      return run_ring(h, kKindReduceScatter, in, out, st);
    case RA_VARIANT_PERSISTENT:
      return run_persistent(h, kKindReduceScatter, ra::kModeReduceScatter, in, out, st);
    case RA_VARIANT_PIPELINED:
      return run_pipelined(h, kKindReduceScatter, ra::kModeReduceScatter, in, out, st);
    case RA_VARIANT_LOCAL:
      return run_local(h, ra::kModeReduceScatter, in, out, st);
    default:
      return run_direct(h, ra::kModeReduceScatter, in, out, st);
  }
}

ra_status ra_all_gather(ra_handle h, void* const* buf, void* stream) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  if (!buf) return fail(RA_ERR_INVALID, "NULL pointer array");
  DeviceGuard g(h->device);
  if (!g.ok) return fail(RA_ERR_CUDA, "cannot switch to device %d", h->device);
  ra_status s = check_buffers(h, nullptr, buf);
  if (s != RA_OK) return s;
  debug_begin(h);
  debug_buffers(h, buf, h->n * elem_bytes(h->dtype));
  if (h->n == 0 || h->R == 1) return RA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (h->variant) {
    case RA_VARIANT_RING:
      return run_ring(h, kKindAllGather, nullptr, buf, st);
    case RA_VARIANT_PERSISTENT:
      return run_persistent(h, kKindAllGather, ra::kModeAllGather, buf, buf, st);
    case RA_VARIANT_PIPELINED:
      return run_pipelined(h, kKindAllGather, ra::kModeAllGather, buf, buf, st);
    case RA_VARIANT_LOCAL:
      return run_local(h, ra::kModeAllGather, buf, buf, st);
    default:
      return run_direct(h, ra::kModeAllGather, buf, buf, st);
  }
}

ra_status ra_reduce_scatter_compact(ra_handle h, const void* const* in, void* const* out, void* stream) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  if (!in || !out) return fail(RA_ERR_INVALID, "NULL pointer array");
  DeviceGuard g(h->device);
  if (!g.ok) return fail(RA_ERR_CUDA, "cannot switch to device %d", h->device);
  if (h->n == 0) return RA_OK;
  ra_status s = check_compact(h, in, out, true);
  if (s != RA_OK) return s;
  debug_begin(h);
  debug_compact(h, in, out);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->R == 1) return run_direct(h, ra::kModeAllReduce, in, out, st);
  return run_compact(h, ra::kModeReduceScatter, in, out, st);
}

ra_status ra_all_gather_compact(ra_handle h, const void* const* in, void* const* out, void* stream) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  if (!in || !out) return fail(RA_ERR_INVALID, "NULL pointer array");
  DeviceGuard g(h->device);
  if (!g.ok) return fail(RA_ERR_CUDA, "cannot switch to device %d", h->device);
  if (h->n == 0) return RA_OK;
  ra_status s = check_compact(h, out, in, false);
  if (s != RA_OK) return s;
  debug_begin(h);
  debug_compact(h, out, in);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->R == 1) return run_direct(h, ra::kModeAllReduce, in, out, st);
  return run_compact(h, ra::kModeAllGather, in, out, st);
}

ra_status ra_owned_chunk(ra_handle h, int r, size_t* off, size_t* len) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  if (r < 0 || r >= h->R) return fail(RA_ERR_INVALID, "rank %d outside [0, %d)", r, h->R);
  if (!off || !len) return fail(RA_ERR_INVALID, "NULL output pointer");
  size_t o[ra::kMaxRanks], l[ra::kMaxRanks];
  ra_chunk_plan(h->R, h->n, o, l);
  const int k = (r + 1) % h->R;
  *off = o[k];
  *len = l[k];
  return RA_OK;
}

ra_status ra_set_option(ra_handle h, int key, long long value) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  {
    // launch shapes and limits are baked into a captured ring graph
    DeviceGuard g(h->device);
    drop_ring_graph(h);
  }
  switch (key) {
    case RA_OPT_GRAPHS:
#ifdef RA_DEBUG_BOUNDS
      if (value != 0) return fail(RA_ERR_UNSUPPORTED, "bounds-checked builds launch the ring variant directly");
#endif
      h->use_graphs = value != 0;
      return RA_OK;
    case RA_OPT_DEBUG_SHRINK:
#ifdef RA_DEBUG_BOUNDS
      if (value < 0) return fail(RA_ERR_INVALID, "shrink %lld below 0", value);
      h->debug_shrink = value;
      return RA_OK;
#else
      return fail(RA_ERR_UNSUPPORTED, "built without bounds checks");
#endif
    case RA_OPT_VARIANT:
      if (value < RA_VARIANT_AUTO || value > RA_VARIANT_LOCAL)
        return fail(RA_ERR_INVALID, "unknown variant %lld", value);
      if ((value == RA_VARIANT_PERSISTENT && h->persist_blocks_per_sm == 0) ||
          (value == RA_VARIANT_PIPELINED && h->pipe_blocks_per_sm == 0))
        return fail(RA_ERR_UNSUPPORTED, "device has no cooperative launch");
      h->variant = (int)value;
      return RA_OK;
    case RA_OPT_BARRIER:
      if (value != RA_BARRIER_COUNTING && value != RA_BARRIER_PER_PEER && value != RA_BARRIER_CLUSTER)
        return fail(RA_ERR_INVALID, "unknown barrier %lld", value);
      h->barrier = (int)value;
      return RA_OK;
    case RA_OPT_SLICES:
      if (value < 0 || value > kMaxSlices) return fail(RA_ERR_INVALID, "slices %lld outside [0, %d]", value, kMaxSlices);
      h->slices = (int)value;
      return RA_OK;
    case RA_OPT_WINDOW:
      if (value < 0 || value > kMaxSlices) return fail(RA_ERR_INVALID, "window %lld outside [0, %d]", value, kMaxSlices);
      h->window = (int)value;
      return RA_OK;
    case RA_OPT_PROTOCOL:
      if (value != RA_PROTOCOL_SIMPLE && value != RA_PROTOCOL_LL && value != RA_PROTOCOL_LL_CLUSTER)
        return fail(RA_ERR_INVALID, "unknown protocol %lld", value);
      if (value == RA_PROTOCOL_LL && h->ll_blocks_per_sm == 0)
        return fail(RA_ERR_UNSUPPORTED, "device has no cooperative launch");
      h->protocol = (int)value;
      return RA_OK;
    case RA_OPT_LL_FLAG:
      if (value < 1 || value > 0xFFFFFFFFLL) return fail(RA_ERR_INVALID, "LL flag %lld outside [1, 2^32-1]", value);
      h->ll_flag = (uint64_t)value;
      return RA_OK;
    case RA_OPT_SIGNAL_BITS:
      if (value < 16 || value > 64) return fail(RA_ERR_INVALID, "signal bits %lld outside [16, 64]", value);
      h->signal_bits = (int)value;
      return RA_OK;
    case RA_OPT_GATHER:
      if (value < 0 || value > 2) return fail(RA_ERR_INVALID, "gather kernel %lld outside [0, 2]", value);
      h->gather = (int)value;
      return RA_OK;
    case RA_OPT_HOST_WINDOWS:
      if (value < 0 || value > kHostWindows)
        return fail(RA_ERR_INVALID, "host windows %lld outside [0, %d]", value, kHostWindows);
      h->host_windows = (int)value;
      return RA_OK;
    case RA_OPT_TIMEOUT_NS:
      // at most a minute: a wait that cannot end (a withheld arrival) must
      // not hold a GPU for longer
      if (value < 1000 || value > kMaxTimeoutNs)
        return fail(RA_ERR_INVALID, "timeout %lld ns outside [1 us, 60 s]", value);
      h->timeout_ns = value;
      return RA_OK;
    case RA_OPT_CTAS:
      if (value < 0 || value > 65535) return fail(RA_ERR_INVALID, "CTA count %lld outside [0, 65535]", value);
      h->ctas = (int)value;
      return RA_OK;
    case RA_OPT_CHECK_POINTERS:
      h->check_pointers = value != 0;
      return RA_OK;
    case RA_OPT_SKIP_ARRIVAL:
      if (value < -1 || (value >= 0 && ((value >> 16) >= h->R))) return fail(RA_ERR_INVALID, "bad skip %lld", value);
      h->skip = value;
      return RA_OK;
    default:
      return fail(RA_ERR_INVALID, "unknown option %d", key);
  }
}

ra_status ra_get_option(ra_handle h, int key, long long* value) {
  if (!h || !value) return fail(RA_ERR_INVALID, "NULL argument");
  switch (key) {
    case RA_OPT_VARIANT: *value = h->variant; return RA_OK;
    case RA_OPT_TIMEOUT_NS: *value = h->timeout_ns; return RA_OK;
    case RA_OPT_CTAS: *value = h->ctas; return RA_OK;
    case RA_OPT_CHECK_POINTERS: *value = h->check_pointers; return RA_OK;
    case RA_OPT_SKIP_ARRIVAL: *value = h->skip; return RA_OK;
    case RA_OPT_GRAPHS: *value = h->use_graphs; return RA_OK;
    case RA_OPT_BARRIER: *value = h->barrier; return RA_OK;
    case RA_OPT_SLICES: *value = h->slices; return RA_OK;
    case RA_OPT_WINDOW: *value = h->window; return RA_OK;
    case RA_OPT_SIGNAL_BITS: *value = h->signal_bits; return RA_OK;
    case RA_OPT_PROTOCOL: *value = h->protocol; return RA_OK;
    case RA_OPT_LL_FLAG: *value = (long long)h->ll_flag; return RA_OK;
    case RA_OPT_GATHER: *value = h->gather; return RA_OK;
    case RA_OPT_HOST_WINDOWS: *value = h->host_windows; return RA_OK;
    case RA_OPT_DEBUG_SHRINK: *value = h->debug_shrink; return RA_OK;
    default: return fail(RA_ERR_INVALID, "unknown option %d", key);
  }
}

ra_status ra_debug_bounds_report(unsigned long long* count, unsigned long long* first_address, int reset) {
#ifdef RA_DEBUG_BOUNDS
  if (!count || !first_address) return fail(RA_ERR_INVALID, "NULL output pointer");
  ra::DebugReport* rep = debug_report();
  if (!rep) return fail(RA_ERR_CUDA, "no bounds report on this device");
  cudaError_t e = cudaDeviceSynchronize();
  ra::DebugReport host;
  if (e == cudaSuccess) e = cudaMemcpy(&host, rep, sizeof(host), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && reset) e = cudaMemset(rep, 0, sizeof(*rep));
  if (e != cudaSuccess) return cuda_fail(e, "bounds report");
  *count = host.count;
  *first_address = host.count ? host.first_addr : 0;
  return RA_OK;
#else
  (void)count;
  (void)first_address;
  (void)reset;
  return fail(RA_ERR_UNSUPPORTED, "built without bounds checks (build with debug=True)");
#endif
}

ra_status ra_get_device_status(ra_handle h, void* stream, ra_device_error* err) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  DeviceGuard g(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
  ra_device_error rec;
  e = cudaMemcpy(&rec, h->d_err, sizeof(rec), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "error record read");
  if (err) *err = rec;
  if (rec.code == 0) return RA_OK;
  ra_status s = reset_device_state(h, st);
  if (s != RA_OK) return s;
  if (rec.code == 6)
    return fail(RA_ERR_TIMEOUT,
                "LL flags exhausted in a call replayed from a CUDA graph (rank %d, channel %d, next flag %llu): "
                "the inbox is zeroed and the flags start again at 1",
                rec.rank, rec.channel, (unsigned long long)rec.observed);
  if (rec.code == 5)
    return fail(RA_ERR_TIMEOUT,
                "device wait gave up: LL message, round %d, rank %d, channel %d, peer %d, flag observed %llu, "
                "expected %llu",
                rec.round, rec.rank, rec.channel, rec.peer, (unsigned long long)rec.observed,
                (unsigned long long)rec.expected);
  const char* what = rec.code == 1 ? "counting barrier"
                     : rec.code == 2 ? "bulk copy"
                     : rec.code == 3 ? "per-peer barrier"
                     : "predecessor flag";
  return fail(RA_ERR_TIMEOUT,
              "device wait gave up: %s, round %d, rank %d, channel %d, peer %d, observed %llu of %llu "
              "(%llu missing)",
              what, rec.round, rec.rank, rec.channel, rec.peer, (unsigned long long)rec.observed,
              (unsigned long long)rec.expected,
              (unsigned long long)((rec.expected - rec.observed) &
                                   (h->signal_bits >= 64 ? ~0ull : ((1ull << h->signal_bits) - 1ull))));
}

ra_status ra_read_signals(ra_handle h, uint64_t* dst, size_t cap, size_t* count, int* channels, int* rounds,
                          long long* calls) {
  if (!h || !count) return fail(RA_ERR_INVALID, "NULL argument");
  DeviceGuard g(h->device);
  if (h->last_kind < 0) {
    *count = 0;
    if (channels) *channels = 0;
    if (rounds) *rounds = 0;
    if (calls) *calls = 0;
    return RA_OK;
  }
  const SlotRegion& reg = h->region[h->last_sync][h->last_kind];
  const size_t need = region_entries(h, h->last_sync, reg.rounds, reg.G, reg.J);
  *count = need;
  if (channels) *channels = reg.G;
  if (rounds) {
    const int br = reg.rounds > 1 ? reg.rounds - 1 : 0;
    *rounds = h->last_sync == ra::kSyncFlags ? reg.rounds : (h->last_sync == ra::kSyncCounting ? br * reg.J : br);
  }
  if (calls) *calls = reg.calls;
  if (!dst || need == 0) return RA_OK;  // sizes only
  if (cap < need) return fail(RA_ERR_INVALID, "need %zu entries, got %zu", need, cap);
  // readSignal on the device: the low RA_OPT_SIGNAL_BITS bits of each
  uint64_t* d_out = nullptr;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMalloc(&d_out, need * sizeof(uint64_t));
  if (e == cudaSuccess) {
    ra::SignalIoArgs a;
    std::memset(&a, 0, sizeof(a));
    a.signals = reg.d;
    a.out = d_out;
    a.count = need;
    a.op = ra::kSigRead;
    a.bits = h->signal_bits;
    debug_begin(h);
    debug_add(d_out, need * sizeof(uint64_t));
    e = ra::launch_signal_io(a, 0);
  }
  if (e == cudaSuccess) e = cudaMemcpy(dst, d_out, need * sizeof(uint64_t), cudaMemcpyDeviceToHost);
  if (d_out) cudaFree(d_out);
  if (e != cudaSuccess) return cuda_fail(e, "signal read");
  return RA_OK;
}

ra_status ra_seed_signals(ra_handle h, uint64_t signal_value, uint64_t shadow_value) {
  if (!h) return fail(RA_ERR_INVALID, "NULL handle");
  DeviceGuard g(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  debug_begin(h);
  for (int sync : {(int)ra::kSyncCounting, (int)ra::kSyncFlags})
    for (auto& reg : h->region[sync]) {
      if (e != cudaSuccess || !reg.d || !reg.cap) continue;
      ra::SignalIoArgs a;
      std::memset(&a, 0, sizeof(a));
      a.signals = reg.d;
      a.shadows = reg.shadows;
      a.count = reg.cap;
      a.op = ra::kSigSeed;
      a.bits = 64;
      a.signal_value = signal_value;
      a.shadow_value = shadow_value;
      e = ra::launch_signal_io(a, 0);
      reg.shadow_base = shadow_value;
    }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "signal seed");
  return RA_OK;
}

ra_status ra_read_shadows(ra_handle h, uint64_t* dst, size_t cap, size_t* count) {
  if (!h || !count) return fail(RA_ERR_INVALID, "NULL argument");
  DeviceGuard g(h->device);
  *count = 0;
  if (h->last_kind < 0 || h->last_sync == ra::kSyncPerPeer || h->last_sync == ra::kSyncCluster) return RA_OK;
  const SlotRegion& reg = h->region[h->last_sync][h->last_kind];
  if (!reg.shadows) return RA_OK;
  const size_t need = region_entries(h, h->last_sync, reg.rounds, reg.G, reg.J);
  *count = need;
  if (!dst || need == 0) return RA_OK;
  if (cap < need) return fail(RA_ERR_INVALID, "need %zu entries, got %zu", need, cap);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(dst, reg.shadows, need * sizeof(uint64_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "shadow read");
  return RA_OK;
}

const char* ra_last_error(void) { return g_last_error.c_str(); }

const char* ra_status_string(ra_status s) {
  switch (s) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID: return "RA_ERR_INVALID";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_OOM: return "RA_ERR_OOM";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT";
    default: return "RA_ERR_UNKNOWN";
  }
}

}  // extern "C"
