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
// Loads never stall a round.  The first P warps stream the operands into a
// ring of shared-memory stages with TMA bulk copies (cp.async.bulk, one
// mbarrier per stage counting the bytes; warp w copies the parts of ranks
// w, w + P, ...), in load steps that run ahead of the rounds and across
// slice boundaries: step 0 of a slice holds x_r[r] for every r (round 1's
// incoming messages), step s holds x_r[(r - s) mod R].  Round s writes m_r over x_r[c] in step s's
// stage, so that stage is round s+1's incoming messages and no other buffer
// is needed.  The folding warps release a step's stage once the round after
// it is done (the last step's, once its results are stored) by arriving on
// the stage's second mbarrier; warp 0 waits on that before refilling it and
// the copying warps take no part in the rounds' barriers, so their copies
// overlap the folds.  One warp's lanes issue their bulk copies one after
// another (~40 ns each on GB300, whatever the size): 32 parts of 960 bytes
// a step took 1.25 us from one warp and 0.66 us spread over four.  So P is
// 1 up to 8 ranks and 4 above (the other warps fold, so more copying warps
// mean smaller stages: 2 or 4 of them cost R = 8 3-6 %).
// Every wait is bounded; a wait that runs out records error code 2, the
// folding warps tell warp 0 to stop, and the CTA leaves once its copies in
// flight have landed.  The unaligned head and tail elements of the chunks
// are folded element by element, in the same ring order, by CTA 0.
#include "ra_device.cuh"

namespace ra {

namespace {

constexpr int kLocalThreads = 512;   // one CTA per SM: P warps issue the bulk copies, the others fold
constexpr int kMaxStages = 8;        // load steps in flight or in use per CTA
constexpr int kItems = 4;            // (rank, vector) positions per folding thread
constexpr int kStageBudget = 200 * 1024;   // shared memory of the stages, at most

// Warps issuing the bulk copies, 16-byte vectors a stage holds (kItems per
// folding thread) and stages, for R ranks.
__host__ __device__ constexpr int copy_warps(int R) { return R <= 8 ? 1 : 4; }
__host__ __device__ constexpr int stage_items(int R) { return kItems * (kLocalThreads - 32 * copy_warps(R)); }
__host__ __device__ constexpr int stage_count(int R) {
  return kStageBudget / (stage_items(R) * 16) < kMaxStages ? kStageBudget / (stage_items(R) * 16) : kMaxStages;
}
static_assert(stage_count(2) >= 2 && stage_count(kMaxRanks) >= 2, "at least two stages");
static_assert(32 * copy_warps(kMaxRanks) >= kMaxRanks, "a copying lane for every rank");

struct LocalShared {
  uint64_t full[kMaxStages];  // the stage holds its step's operands
  uint64_t empty[kMaxStages]; // the folding warps are done with the stage's step
  int64_t issued;             // steps the copying warps issued (read on abort)
  int abort;                  // the folding warps gave up: the copying warps stop
  int go[2];                  // warp 0 to the other copying warps: step u goes ahead (slot u & 1)
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

// Named barrier 1: the nf folding threads only (the copying warps never
// wait on it); named barrier 2: the copying warps only.
__device__ __forceinline__ void folders_sync(int nf) { asm volatile("bar.sync 1, %0;" ::"r"(nf) : "memory"); }
__device__ __forceinline__ void producers_sync(int np) { asm volatile("bar.sync 2, %0;" ::"r"(np) : "memory"); }

__device__ __forceinline__ bool folders_all(bool pred, int nf) {
  uint32_t all;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(all)
      : "r"((uint32_t)pred), "r"(nf)
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
  extern __shared__ __align__(128) uint4 smem[];   // stage[NS][R][SV]
  __shared__ LocalShared sh;
  const int R = a.R, SV = a.SV, P = copy_warps(a.R), NS = stage_count(a.R);
  const int nf = kLocalThreads - 32 * P;   // folding threads
  const int items = R * SV;
  const int64_t n = a.plan.n, C = a.plan.C;
  uint4* const stage0 = smem;
  const bool reduce = a.mode != kModeAllGather;
  const int T_ = reduce ? R : 1;                          // load steps per slice
  const int64_t G = a.slices;
  const int64_t J = G > blockIdx.x ? (G - 1 - blockIdx.x) / gridDim.x + 1 : 0;   // slices of this CTA
  const int64_t steps = J * T_;
  const bool producer = threadIdx.x < 32 * P;   // warps 0 .. P-1 issue the copies

  if (threadIdx.x < R) {
    const int64_t off = min((int64_t)threadIdx.x * C, n);
    const Span<V> sp(off, min(off + C, n));
    sh.cvb[threadIdx.x] = sp.vb;
    sh.cve[threadIdx.x] = sp.ve;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sh.full[i], 1);    // one arrival: lane 0's expect_tx
      mbar_init(&sh.empty[i], 1);   // one arrival: the releasing folding thread
    }
    sh.abort = 0;
    sh.issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  auto next = [NS](int st) { return st + 1 == NS ? 0 : st + 1; };
  bool ok = true;

  if (producer) {
    // The copying warps issue load steps in order, each once its stage is
    // free.  Step u: slice u / T_, s = u % T_, stage u % NS.  Rank r's
    // operand: x_r[(r - s) mod R] (step 0: x_r[r], round 1's incoming
    // message); AllGather alone: x_r[(r + 1) mod R].  Warp 0 alone waits
    // for the stage and announces the step's bytes (lane r: rank r's part),
    // then tells the other copying warps whether the step goes ahead, so
    // every warp issues the same steps; warp w copies ranks w + P j (lane j).
    const int pw = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = pw + P * lane;
    const uint4* const rank_in = rank < R ? static_cast<const uint4*>(a.p.in[rank]) : nullptr;
    auto chunk_of = [&](int r, int s) {
      int c = reduce ? r - s : r + 1;
      return c < 0 ? c + R : (c >= R ? c - R : c);
    };
    int64_t slice = 0;
    int s = 0, st = 0;
    uint32_t eparity = 0;   // bit i: parity of stage i's next release (warp 0)
    int64_t u = 0;
    for (; u < steps; ++u) {
      const int64_t g = blockIdx.x + slice * gridDim.x;
      bool go = true;
      if (pw == 0) {
        if (u >= NS) {   // the stage's previous step must be released
          go = wait_bounded(&sh.empty[st], (eparity >> st) & 1u, a.timeout_ns, &sh.abort);
          // one answer for the warp: a lane that saw the release just before
          // another saw the folding warps give up must not copy alone
          go = __all_sync(0xffffffffu, go);
          eparity ^= 1u << st;
          if (!go && lane == 0 && !sh.abort)
            record_wait_error(a.err, 2u, s, -1, blockIdx.x, -1, (uint64_t)u, (uint64_t)steps);
        }
        if (go) {
          int64_t off = 0;
          const int len = lane < R ? slice_part(sh, chunk_of(lane, s), g, SV, &off) : 0;
          const uint32_t bytes = __reduce_add_sync(0xffffffffu, (uint32_t)len * 16u);
          if (lane == 0) mbar_arrive_expect_tx(&sh.full[st], bytes);
        }
        if (P > 1 && lane == 0) sh.go[u & 1] = go ? 1 : 0;
      }
      if (P > 1) {
        producers_sync(32 * P);   // the bytes are announced before any of the step's copies
        go = sh.go[u & 1] != 0;
      }
      if (!go) break;
      if (rank < R) {
        int64_t off = 0;
        const int len = slice_part(sh, chunk_of(rank, s), g, SV, &off);
        if (len > 0) bulk_load(stage0 + st * items + rank * SV, rank_in + off, (uint32_t)len * 16u, &sh.full[st]);
      }
      if (++s == T_) {
        s = 0;
        ++slice;
      }
      st = next(st);
    }
    if (threadIdx.x == 0) sh.issued = u;
  } else {
    // Folding warps.  Positions fixed for the whole launch: rank rk, vector
    // own - rk*SV of the slice.
    const int ft = threadIdx.x - 32 * P;
    int rk[kItems], own[kItems], pred[kItems];
    uint4* outp[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int i = ft + k * nf;
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
      folders_sync(nf);   // the slice table; and slice j-1's stores have read its last stage
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
          if (!folders_all(got, nf)) {
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
        if (!folders_all(got, nf)) {
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
      for (int64_t u = issued > NS ? issued - NS : 0; u < issued; ++u)
        wait_bounded(&sh.full[u % NS], (uint32_t)((u / NS) & 1), a.timeout_ns);
    }
    return;
  }

  // Chunk heads and tails off the 16-byte grid: element by element, in the
  // same ring order, every chunk's at once -- CTA 0's threads 2V k .. 2V k +
  // 2V-1 take chunk k (a chunk with a whole vector has at most 2(V-1) such
  // elements) -- and an element's R loads issued together before the fold.
  // Taken one chunk after another, each load after the previous fold, they
  // held R = 24 x 2^24 fp32 back by tens of microseconds: the words around a
  // chunk boundary are in no bulk copy, so every one of those loads came
  // from DRAM.
  if (blockIdx.x == 0) {
    constexpr int S = 2 * V;
    static_assert(S * kMaxRanks <= kLocalThreads, "a thread group for every chunk");
    const int k = (int)threadIdx.x / S;
    if (k < R) {
      const int64_t off = min((int64_t)k * C, n);
      const Span<V> sp(off, min(off + C, n));
      const int64_t ns = sp.scalar_count();
      const int owner = (k == 0) ? R - 1 : k - 1;
      for (int64_t e = threadIdx.x % S; e < ns; e += S) {
        const int64_t i = sp.scalar_at(e);
        T acc;
        if (!reduce) {
          acc = ld_g(static_cast<const T*>(a.p.in[owner]) + i);
        } else {
          T x[kMaxRanks];   // x[j]: rank (k + j) mod R's element
#pragma unroll
          for (int j = 0; j < kMaxRanks; ++j)
            if (j < R) x[j] = ld_g(static_cast<const T*>(a.p.in[k + j >= R ? k + j - R : k + j]) + i);
          acc = x[0];
#pragma unroll
          for (int j = 1; j < kMaxRanks; ++j)
            if (j < R) acc = Op<D, OP>::apply(acc, x[j]);
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

int local_slice_vectors(int R) { return R < 1 ? 0 : stage_items(R) / R; }

size_t local_smem_bytes(int R) { return R < 1 ? 0 : (size_t)stage_count(R) * R * local_slice_vectors(R) * sizeof(uint4); }

cudaError_t prepare_local() {
  size_t most = 0;
  for (int R = 2; R <= kMaxRanks; ++R) most = std::max(most, local_smem_bytes(R));
  cudaError_t err = cudaSuccess;
  for (int dt = RA_F32; dt <= RA_I64 && err == cudaSuccess; ++dt)
    for (int op = RA_SUM; op <= RA_MAX && err == cudaSuccess; ++op)
      err = cudaFuncSetAttribute(local_select(dt, op), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
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
    const size_t smem = (size_t)stage_count(a.R) * a.R * a.SV * sizeof(uint4);
    local_kernel<decltype(d), decltype(o)::value><<<ctas, kLocalThreads, smem, st>>>(a);
    return cudaGetLastError();
  });
}

}  // namespace ra
