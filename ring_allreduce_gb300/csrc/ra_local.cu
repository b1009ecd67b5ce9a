// ra_local.cu -- the local variant: one CTA runs the whole ring, round by
// round, for one slice of every chunk; the messages the R simulated ranks
// pass to their successors live in the CTA's shared memory.
//
// "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce",
// sections 5 and 6, on slice g (SV 16-byte vectors of every chunk):
//   ReduceScatter round s = 1..R-1: every rank r at once forms
//     m_r = m_{r-1} (+) x_r[c],  c = (r - s) mod R,
//   where m_{r-1} is what rank r-1 made in round s-1 (x_{r-1}[c] itself in
//   round 1), and a barrier of the folding warps ends the round.  In round
//   R-1, m_r is S_{(r+1) mod R}: rank r stores it to its own output (the
//   recvReduceCopySend of section 9) and keeps it.
//   AllGather round s = 1..R-1: rank r copies chunk (r+1-s) mod R -- the
//   S kept by rank r-s -- to its output.
// Every x_r[c] is read once and every output vector written once: the
// compulsory 2 R n b bytes, with no synchronisation between CTAs.
//
// Loads never stall a round.  Warp 0 streams the operands into a ring of
// kStages shared-memory stages with TMA bulk copies (cp.async.bulk, one
// mbarrier per stage counting the bytes; lane r copies rank r's part), in
// load steps that run ahead of the rounds and across slice boundaries: step
// 0 of a slice holds x_r[r] for every r (round 1's incoming messages), step
// s holds x_r[(r - s) mod R].  Round s writes m_r over x_r[c] in step s's
// stage, so that stage is round s+1's incoming messages and no other buffer
// is needed.  The folding warps release a step's stage once the round after
// it is done (the last step's, once its results are stored) by arriving on
// the stage's second mbarrier; warp 0 waits on that before refilling it and
// takes no part in the rounds' barriers, so its copies overlap the folds.
// Every wait is bounded; a wait that runs out records error code 2, the
// folding warps tell warp 0 to stop, and the CTA leaves once its copies in
// flight have landed.  The unaligned head and tail elements of the chunks
// are folded element by element, in the same ring order, by CTA 0.
#include "ra_device.cuh"

namespace ra {

namespace {

constexpr int kLocalThreads = 512;   // one CTA per SM: warp 0 issues the bulk copies, 15 warps fold
constexpr int kStages = 6;           // load steps in flight or in use per CTA
constexpr int kSliceItems = 1920;    // R * SV <= 1920 16-byte vectors per stage (30 KiB)
constexpr int kFolders = kLocalThreads - 32;
constexpr int kItems = kSliceItems / kFolders;       // (rank, vector) positions per folding thread
static_assert(kItems * kFolders == kSliceItems, "slice items must split evenly over the folding threads");

struct LocalShared {
  uint64_t full[kStages];     // the stage holds its step's operands
  uint64_t empty[kStages];    // the folding warps are done with the stage's step
  int64_t issued;             // steps warp 0 issued (read on abort)
  int abort;                  // the folding warps gave up: warp 0 stops
  int64_t cvb[kMaxRanks];     // chunk c's whole vectors: [cvb, cve)
  int64_t cve[kMaxRanks];
  int64_t base[2][kMaxRanks]; // slice j (index j & 1): first vector of chunk c's part
  int len[2][kMaxRanks];      // slice j (index j & 1): vectors of chunk c's part
};

// Bounded wait on a stage's mbarrier: gives up after timeout_ns of the
// global timer (or of the SM's cycle counter, should that timer stand still:
// see Deadline), or once *abort is set; false when it gave up.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, int64_t timeout_ns,
                                             const volatile int* abort = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const Deadline limit(timeout_ns);
  while (!mbar_try_wait(bar, parity)) {
    if (limit.passed() || (abort && *abort)) return false;
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Named barrier 1: the folding warps only (warp 0 never waits on it).
__device__ __forceinline__ void folders_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kFolders) : "memory"); }

__device__ __forceinline__ bool folders_all(bool pred) {
  uint32_t all;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(all)
      : "r"((uint32_t)pred), "n"(kFolders)
      : "memory");
  return all != 0;
}

// vectors of chunk c in slice g, starting at *off
__device__ __forceinline__ int slice_part(const LocalShared& sh, int c, int64_t g, int SV, int64_t* off) {
  const int64_t o = sh.cvb[c] + g * SV;
  *off = o;
  const int64_t left = sh.cve[c] - o;
  return left <= 0 ? 0 : (left < SV ? (int)left : SV);
}

}  // namespace

template <class D, int OP>
__global__ void __launch_bounds__(kLocalThreads, 1)
local_kernel(const LocalArgs a) {
  using T = typename D::T;
  constexpr int V = D::kVec;
  extern __shared__ __align__(128) uint4 smem[];   // stage[kStages][R][SV]
  __shared__ LocalShared sh;
  const int R = a.R, SV = a.SV;
  const int items = R * SV;
  const int64_t n = a.plan.n, C = a.plan.C;
  uint4* const stage0 = smem;
  const bool reduce = a.mode != kModeAllGather;
  const int T_ = reduce ? R : 1;                          // load steps per slice
  const int64_t G = a.slices;
  const int64_t J = G > blockIdx.x ? (G - 1 - blockIdx.x) / gridDim.x + 1 : 0;   // slices of this CTA
  const int64_t steps = J * T_;
  const bool producer = threadIdx.x < 32;   // warp 0 issues the copies

  if (threadIdx.x < R) {
    const int64_t off = min((int64_t)threadIdx.x * C, n);
    const Span<V> sp(off, min(off + C, n));
    sh.cvb[threadIdx.x] = sp.vb;
    sh.cve[threadIdx.x] = sp.ve;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.full[i], 1);    // one arrival: lane 0's expect_tx
      mbar_init(&sh.empty[i], 1);   // one arrival: the releasing folding thread
    }
    sh.abort = 0;
    sh.issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  auto next = [](int st) { return st + 1 == kStages ? 0 : st + 1; };
  bool ok = true;

  if (producer) {
    // Warp 0 issues load steps in order, each once its stage is free.  Step
    // u: slice u / T_, s = u % T_, stage u % kStages.  Rank r's operand:
    // x_r[(r - s) mod R] (step 0: x_r[r], round 1's incoming message);
    // AllGather alone: x_r[(r + 1) mod R].  Lane r copies rank r's part;
    // lane 0 announces the step's bytes first.
    const int lane = threadIdx.x;
    const uint4* const lane_in = lane < R ? static_cast<const uint4*>(a.p.in[lane]) : nullptr;
    int64_t slice = 0;
    int s = 0, st = 0;
    uint32_t eparity = 0;   // bit i: parity of stage i's next release
    int64_t u = 0;
    for (; u < steps; ++u) {
      if (u >= kStages) {   // the stage's previous step must be released
        const bool freed = wait_bounded(&sh.empty[st], (eparity >> st) & 1u, a.timeout_ns, &sh.abort);
        eparity ^= 1u << st;
        if (!freed) {
          if (lane == 0 && !sh.abort)
            record_wait_error(a.err, 2u, s, -1, blockIdx.x, -1, (uint64_t)u, (uint64_t)steps);
          break;
        }
      }
      const int64_t g = blockIdx.x + slice * gridDim.x;
      int c = reduce ? lane - s : lane + 1;
      c = c < 0 ? c + R : (c >= R ? c - R : c);
      int64_t off = 0;
      const int len = lane < R ? slice_part(sh, c, g, SV, &off) : 0;
      const uint32_t bytes = __reduce_add_sync(0xffffffffu, (uint32_t)len * 16u);
      if (lane == 0) mbar_arrive_expect_tx(&sh.full[st], bytes);
      __syncwarp();
      if (len > 0) bulk_load(stage0 + st * items + lane * SV, lane_in + off, (uint32_t)len * 16u, &sh.full[st]);
      if (++s == T_) {
        s = 0;
        ++slice;
      }
      st = next(st);
    }
    if (lane == 0) sh.issued = u;
  } else {
    // Folding warps.  Positions fixed for the whole launch: rank rk, vector
    // own - rk*SV of the slice.
    const int ft = threadIdx.x - 32;
    int rk[kItems], own[kItems], pred[kItems];
    uint4* outp[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int i = ft + k * kFolders;
      const bool on = i < items;
      const int r = on ? i / SV : 0;
      const int v = i - r * SV;
      rk[k] = on ? r : -1;
      own[k] = on ? i : 0;                                      // r*SV + v
      pred[k] = on ? ((r == 0 ? R - 1 : r - 1) * SV + v) : 0;   // the predecessor's slot
      outp[k] = on ? static_cast<uint4*>(a.p.out[r]) + v : nullptr;
    }
    int cst = 0;              // stage of the next step to consume
    uint32_t parity = 0;      // bit i: parity of stage i's next fill
    auto wait_stage = [&](int st) {
      const bool got = wait_bounded(&sh.full[st], (parity >> st) & 1u, a.timeout_ns);
      parity ^= 1u << st;
      return got;
    };
    // steps are released in order, by one thread, once every folding warp is past them
    auto release = [&](int st) {
      if (ft == 0) mbar_arrive(&sh.empty[st]);
    };
    int held = -1;   // stage of the previous slice's last step, until its stores are done

    for (int64_t j = 0; j < J && ok; ++j) {
      const int64_t g = blockIdx.x + j * gridDim.x;
      const int tb = (int)(j & 1);
      const int* len = sh.len[tb];
      const int64_t* base = sh.base[tb];
      if (ft < R) {
        // slice j-1 reads the other table; slice j-2, the last reader of this one, is past a barrier
        sh.len[tb][ft] = slice_part(sh, ft, g, SV, &sh.base[tb][ft]);
      }
      folders_sync();   // the slice table; and slice j-1's stores have read its last stage
      if (held >= 0) {
        release(held);
        held = -1;
      }
      const uint4* fin;   // rank q's slot: S_{(q+1) mod R}
      if (reduce) {
        bool got = wait_stage(cst);   // step 0: x_p[p]
        int pst = cst;
        cst = next(cst);
        for (int s = 1; s < R; ++s) {
          const uint4* prev = stage0 + pst * items;
          uint4* cur = stage0 + cst * items;
          got = wait_stage(cst) && got;
          if (got) {
            uint4 pv[kItems], cv[kItems];
            bool on[kItems];
            int64_t at[kItems];
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
              int c = rk[k] - s;
              c = c < 0 ? c + R : c;
              on[k] = rk[k] >= 0 && own[k] - rk[k] * SV < len[c];
              at[k] = base[c];
              if (on[k]) {
                pv[k] = prev[pred[k]];
                cv[k] = cur[own[k]];
              }
            }
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
              if (!on[k]) continue;
              // m_r = m_{r-1} (+) x_r[c], kept in place of x_r[c]: round s+1's incoming message
              const uint4 m = combine_vec<D, OP>(pv[k], cv[k]);
              cur[own[k]] = m;
              if (s == R - 1) st_stream(outp[k] + at[k], m);
            }
          } else {
            record_wait_error(a.err, 2u, s, -1, blockIdx.x, -1, (uint64_t)(j * T_ + s), (uint64_t)steps);
          }
          fence_proxy_async_smem();   // these shared-memory accesses precede later bulk copies into the stages
          if (!folders_all(got)) {
            ok = false;
            break;
          }
          release(pst);   // round s's incoming messages
          pst = cst;
          cst = next(cst);
        }
        if (!ok) break;
        fin = stage0 + pst * items;
        if (a.mode == kModeReduceScatter) release(pst);
        else held = pst;
      } else {
        const bool got = wait_stage(cst);
        if (!got) record_wait_error(a.err, 2u, 0, -1, blockIdx.x, -1, (uint64_t)j, (uint64_t)steps);
        if (!folders_all(got)) {
          ok = false;
          break;
        }
        fin = stage0 + cst * items;   // rank q's slot: x_q[q+1], which is S_{q+1}
        held = cst;
        cst = next(cst);
      }

      if (a.mode != kModeReduceScatter) {
        for (int s = 1; s < R; ++s) {
          uint4 val[kItems];
          bool on[kItems];
          int64_t at[kItems];
#pragma unroll
          for (int k = 0; k < kItems; ++k) {
            int q = rk[k] - s;                           // holder of chunk q+1
            q = q < 0 ? q + R : q;
            const int c = (q + 1 == R) ? 0 : q + 1;
            const int v = own[k] - rk[k] * SV;
            on[k] = rk[k] >= 0 && v < len[c];
            at[k] = base[c];
            if (on[k]) val[k] = fin[q * SV + v];
          }
#pragma unroll
          for (int k = 0; k < kItems; ++k)
            if (on[k]) st_stream(outp[k] + at[k], val[k]);
        }
      }
    }
    if (!ok && ft == 0) *(volatile int*)&sh.abort = 1;
  }

  __syncthreads();   // warp 0 has issued its last step (or stopped)
  if (!__syncthreads_and(ok)) {
    // leave only once every copy in flight has landed: only the last step
    // of each stage can still be in flight
    if (threadIdx.x == 0) {
      const int64_t issued = sh.issued;
      for (int64_t u = issued > kStages ? issued - kStages : 0; u < issued; ++u)
        wait_bounded(&sh.full[u % kStages], (uint32_t)((u / kStages) & 1), a.timeout_ns);
    }
    return;
  }

  // chunk heads and tails off the 16-byte grid: element by element, same ring order
  if (blockIdx.x == 0) {
    for (int k = 0; k < R; ++k) {
      const int64_t off = min((int64_t)k * C, n);
      const Span<V> sp(off, min(off + C, n));
      const int64_t ns = sp.scalar_count();
      const int owner = (k == 0) ? R - 1 : k - 1;
      for (int64_t e = threadIdx.x; e < ns; e += blockDim.x) {
        const int64_t i = sp.scalar_at(e);
        T acc;
        if (!reduce) {
          acc = ld_g(static_cast<const T*>(a.p.in[owner]) + i);
        } else {
          acc = ld_g(static_cast<const T*>(a.p.in[k]) + i);
          for (int jr = 1; jr < R; ++jr) {
            const int q = (k + jr >= R) ? k + jr - R : k + jr;
            acc = Op<D, OP>::apply(acc, ld_g(static_cast<const T*>(a.p.in[q]) + i));
          }
        }
        if (a.mode == kModeReduceScatter) {
          st_g(static_cast<T*>(a.p.out[owner]) + i, acc);
        } else {
          for (int jr = 0; jr < R; ++jr)
            if (a.mode == kModeAllReduce || jr != owner) st_g(static_cast<T*>(a.p.out[jr]) + i, acc);
        }
      }
    }
  }
}

namespace {

const void* local_select(int dtype, int op) {
  const void* fn = nullptr;
  with_dtype_op(dtype, op, [&](auto d, auto o) {
    fn = reinterpret_cast<const void*>(local_kernel<decltype(d), decltype(o)::value>);
    return cudaSuccess;
  });
  return fn;
}

}  // namespace

int local_slice_vectors(int R) { return R < 1 ? 0 : kSliceItems / R; }

size_t local_smem_bytes(int R) { return (size_t)kStages * R * local_slice_vectors(R) * sizeof(uint4); }

cudaError_t prepare_local() {
  cudaError_t err = cudaSuccess;
  for (int dt = RA_F32; dt <= RA_I64 && err == cudaSuccess; ++dt)
    for (int op = RA_SUM; op <= RA_MAX && err == cudaSuccess; ++op)
      err = cudaFuncSetAttribute(local_select(dt, op), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)local_smem_bytes(1));
  return err;
}

cudaError_t local_blocks_per_sm(int dtype, int op, int R, int* blocks) {
  const void* fn = local_select(dtype, op);
  if (!fn || R < 2 || R > kMaxRanks) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, kLocalThreads, local_smem_bytes(R));
}

cudaError_t launch_local(int dtype, int op, const LocalArgs& a, int ctas, cudaStream_t st) {
  if (a.R < 2 || a.R > kMaxRanks || a.SV < 1 || a.SV > local_slice_vectors(a.R) || ctas < 1 || a.slices < 1)
    return cudaErrorInvalidValue;
  const cudaError_t e = debug_upload(st);
  if (e != cudaSuccess) return e;
  return with_dtype_op(dtype, op, [&](auto d, auto o) {
    const size_t smem = (size_t)kStages * a.R * a.SV * sizeof(uint4);
    local_kernel<decltype(d), decltype(o)::value><<<ctas, kLocalThreads, smem, st>>>(a);
    return cudaGetLastError();
  });
}

}  // namespace ra
