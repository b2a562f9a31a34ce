// Persistent, warp-specialised BF16 TN GEMM on tcgen05 (sm_103a).
//
//   D[M,N] = alpha * A[M,K] * B[N,K]^T + beta * C[M,N]     (fp32 accumulate)
//
// Structure (one CTA per SM, 6 warps):
//   warp 0 lane 0   TMA producer: fills a ring of shared-memory stages with
//                   128x64 A tiles and (BN/CG)x64 B tiles (128-byte swizzle),
//                   each stage guarded by a FULL / EMPTY mbarrier pair — the
//                   per-stage ownership state machine of the Ampere-to-Hopper
//                   page (section "a stage maintains two kinds of ownership")
//                   and the transaction-count completion of its section
//                   "Transaction Barrier".
//   warp 1          allocates Tensor Memory; lane 0 issues tcgen05.mma for
//                   the whole CTA (or CTA pair) into one of two TMEM
//                   accumulators and releases stages with tcgen05.commit —
//                   the single-thread MMA issue, TMEM accumulator and 2-SM
//                   pair MMA of the SemiAnalysis Blackwell page ("Blackwell
//                   architecture features", "5th-generation tensor core MMA").
//   warps 2..5      epilogue: tcgen05.ld 32 columns at a time, alpha/beta,
//                   bf16 rounding, swizzled staging in shared memory and a TMA
//                   store that clips rows/columns outside D (the hardware
//                   out-of-bounds handling of the Ampere-to-Hopper page's TMA
//                   section).  Two TMEM accumulators let the epilogue of tile
//                   i overlap the mainloop of tile i+1.
//
// CG = 2 runs the pair form: cluster of two CTAs on one TPC, MMA M = 256,
// each CTA loads its own 128 rows of A and half of the B tile, the leader
// CTA issues the MMA for both and the accumulator rows stay in each CTA's
// own TMEM.  No TMA multicast is used; each CTA loads its own tiles.
//
// Tile schedule: either a persistent grid with a fixed stride (CTA c takes
// tiles c, c + G, ...), or one CTA (pair) per tile with cluster launch
// control: at the start of each tile the producer asks the hardware to cancel
// a cluster that has not launched yet; the 16-byte answer lands in a small
// ring in shared memory (in both CTAs of a pair) and every role reads it to
// learn its next tile, or that there is none.
//
// Every mbarrier wait is bounded by %globaltimer.  A wait that gives up sets
// a CTA abort flag and the device status word; all roles then leave their
// loops, drain what they issued and free TMEM, so the kernel always returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace gtn {

namespace {

constexpr int kStageK = 128;      // bytes of K per operand row per stage (one 128-byte swizzle atom)
constexpr int kMmaPerStage = 4;   // tcgen05.mma instructions per stage, 32 bytes of K each

// K elements per stage: 64 bf16 or 128 fp8.
template <int KIND>
constexpr int stage_k_elems() { return KIND == kKindF16 ? 64 : 128; }
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kErrTimeout = -5;   // GEMM_ERR_TIMEOUT

template <int CG, bool OUT_F32>
struct Cfg {
  static constexpr int BN = 256;                      // tile N (MMA N)
  static constexpr int TILE_M = 128 * CG;             // rows per (pair) tile = MMA M
  static constexpr int B_ROWS = BN / CG;              // B rows loaded per CTA
  static constexpr int A_BYTES = 128 * kStageK;       // 16 KiB
  static constexpr int B_BYTES = B_ROWS * kStageK;
  static constexpr int STAGES = (CG == 1) ? 4 : 6;
  static constexpr uint32_t STAGE_TX = (A_BYTES + B_BYTES) * CG;
  static constexpr int OUT_BYTES = OUT_F32 ? 4 : 2;
  static constexpr int EPI_COLS = 32;
  static constexpr int EPI_BYTES = 32 * EPI_COLS * OUT_BYTES;   // one 32x32 box
  static constexpr int TMEM_COLS = 2 * BN;            // two accumulators
  static constexpr int CLC_SLOTS = 4;                 // cluster-launch-control answers in flight
  // readers of each answer, all arriving on the leader CTA's CLC_EMPTY:
  // producer + 4 epilogue warps per CTA, and the leader's MMA thread
  static constexpr int CLC_READERS = CG * (1 + kEpiWarps) + 1;
  // + two barriers per epilogue warp for the k-split partials (see the epilogue)
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * kEpiWarps + 1 + 2 * CLC_SLOTS + 2 * kEpiWarps;
  // k-split: each epilogue warp stages two chunks of up to three partials
  // (4 KiB each) in the operand ring, which is idle by then
  static constexpr int PART_SLOT = 32 * 32 * 4;
  static_assert(kEpiWarps * 2 * 3 * PART_SLOT <= STAGES * (A_BYTES + B_BYTES), "partial staging fits the ring");
  static constexpr int RING_BYTES = STAGES * (A_BYTES + B_BYTES);
  static constexpr int EPI_TOTAL = kEpiWarps * 2 * EPI_BYTES;
  static constexpr int CLC_BYTES = CLC_SLOTS * 16;
  static constexpr int SMEM = 1024 + RING_BYTES + EPI_TOTAL + CLC_BYTES + NUM_BARS * 8 + 16;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TMEM_COLS <= 512, "TMEM columns");
};

struct Abort {
  volatile uint32_t* flag;
  uint64_t timeout_ns;
  int* status;
  int role;
};

template <bool CLUSTER>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  if constexpr (CLUSTER) return mbar_try_wait_cluster(bar, parity);
  else return mbar_try_wait(bar, parity);
}

// Slow path of a bounded wait: spin on the phase with a %globaltimer limit.
template <bool CLUSTER>
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile uint32_t* flag,
                                           uint64_t timeout_ns, int* status, int role) {
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (try_wait<CLUSTER>(bar, parity)) return true;
    if (flag && *flag) return false;
    if (globaltimer() - t0 > timeout_ns) {
      if (flag) *flag = 1;
      if (atomicCAS(status, 0, kErrTimeout) == 0) atomicExch(status + 1, (role << 24) | (int)blockIdx.x);
      return false;
    }
  }
}

// Bounded wait on an mbarrier phase.  Returns false if this CTA is aborting.
template <bool CLUSTER>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Abort& ab) {
  if (try_wait<CLUSTER>(bar, parity)) return true;
  return wait_bar_slow<CLUSTER>(bar, parity, ab.flag, ab.timeout_ns, ab.status, ab.role);
}

// Spin for `ns` nanoseconds (lets copies already in flight land before exit).
__device__ __noinline__ void settle(uint64_t ns) {
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < ns) __nanosleep(1000);
}

// Warp-wide bounded wait until `expected` parts of a split tile have been
// counted at `arrivals` (lane 0 polls with acquire; the warp barrier passes
// the acquire on to the other lanes), then clears the counter for the next
// call.  False if the CTA is aborting or the limit expired (status recorded).
__device__ __noinline__ bool wait_parts(int* arrivals, int expected, const Abort& ab) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    if (ld_acquire_gpu(arrivals) != expected) {
      const uint64_t t0 = globaltimer();
      while (ld_acquire_gpu(arrivals) != expected) {
        if (*ab.flag || globaltimer() - t0 > ab.timeout_ns) {
          if (!*ab.flag) {
            *ab.flag = 1;
            if (atomicCAS(ab.status, 0, kErrTimeout) == 0)
              atomicExch(ab.status + 1, (kRoleFixup << 24) | (int)blockIdx.x);
          }
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    if (ok) *arrivals = 0;
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// k-blocks [kb0, kb1) of part `part` of a tile split into `parts`.
__device__ __forceinline__ void part_range(int num_kb, int parts, int part, int& kb0, int& kb1) {
  kb0 = (int)((long long)part * num_kb / parts);
  kb1 = (int)((long long)(part + 1) * num_kb / parts);
}

__device__ __forceinline__ void tile_coords(int t, int raster_group, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int per_group = raster_group * tiles_n;
  const int g = t / per_group;
  const int first_m = g * raster_group;
  const int gm = min(raster_group, tiles_m - first_m);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

template <int MODE>
using GroupArg = typename std::conditional<MODE == kModeList, GroupList, NoGroup>::type;

// B with boxes of a slice's rows, for a launch whose last round is cut into slices.
struct SliceArg {
  CUtensorMap b;
};

// The kernel's last parameter: the problem list, the slice map, or nothing.
template <int MODE, bool SLICE>
using KernelArg = typename std::conditional<SLICE, SliceArg, GroupArg<MODE>>::type;

// Everything a role needs to know about tile t: its position, the sizes of
// its problem and that problem's tensor maps (z = batch index for a strided
// batch, else 0).
struct TileRef {
  int tm, tn, z;
  int M, N, num_kb;
  const CUtensorMap *a, *b, *c, *d;
};

template <int MODE>
__device__ __forceinline__ TileRef resolve(int t, const TileParams& p, const GroupArg<MODE>& ga, const CUtensorMap* tA,
                                           const CUtensorMap* tB, const CUtensorMap* tC, const CUtensorMap* tD) {
  TileRef r;
  if constexpr (MODE == kModeList) {
    // last problem whose first tile is <= t (tile_begin ascends)
    int g = 0, hi = ga.count - 1;
    while (g < hi) {
      const int mid = (g + hi + 1) >> 1;
      if (ga.prob[mid].tile_begin <= t) g = mid;
      else hi = mid - 1;
    }
    const GroupProblem& q = ga.prob[g];
    tile_coords(t - q.tile_begin, q.raster_group, q.tiles_m, q.tiles_n, r.tm, r.tn);
    r.z = 0;
    r.M = q.M;
    r.N = q.N;
    r.num_kb = q.num_kb;
    r.a = &ga.a[g];
    r.b = &ga.b[g];
    r.c = &ga.c[g];
    r.d = &ga.d[g];
  } else {
    int local = t;
    r.z = 0;
    if constexpr (MODE == kModeStrided) {
      const int per = p.tiles_m * p.tiles_n;
      r.z = t / per;
      local = t - r.z * per;
    }
    tile_coords(local, p.raster_group, p.tiles_m, p.tiles_n, r.tm, r.tn);
    r.M = p.M;
    r.N = p.N;
    r.num_kb = p.num_kb;
    r.a = tA;
    r.b = tB;
    r.c = tC;
    r.d = tD;
  }
  return r;
}

// TMA through 2D maps, or 3D maps with the batch index for a strided batch.
template <int MODE>
__device__ __forceinline__ void tload(uint32_t dst, const CUtensorMap* m, int x, int y, int z, uint32_t bar) {
  if constexpr (MODE == kModeStrided) tma_load_3d(dst, m, x, y, z, bar);
  else tma_load_2d(dst, m, x, y, bar);
}
template <int MODE>
__device__ __forceinline__ void tload_pair(uint32_t dst, const CUtensorMap* m, int x, int y, int z, uint32_t bar) {
  if constexpr (MODE == kModeStrided) tma_load_3d_pair(dst, m, x, y, z, bar);
  else tma_load_2d_pair(dst, m, x, y, bar);
}
template <int MODE>
__device__ __forceinline__ void tstore(const CUtensorMap* m, int x, int y, int z, uint32_t src) {
  if constexpr (MODE == kModeStrided) tma_store_3d(m, x, y, z, src);
  else tma_store_2d(m, x, y, src);
}

// Position of one role in the cluster-launch-control answer ring.
struct ClcCursor {
  int slot = 0;
  uint32_t phase = 0;
  __device__ void advance(int slots) {
    if (++slot == slots) {
      slot = 0;
      phase ^= 1;
    }
  }
};

// Next tile of a role after tile t.  Static schedule: t + stride.  Cluster
// launch control: wait for the answer in the cursor's slot, read it, hand
// the slot back (arrive on the leader's CLC_EMPTY; `arrive` is false for the
// lanes of a warp other than lane 0) and return the cancelled cluster's tile,
// or num_tiles if no cluster was left.  Returns -1 if the wait gave up.
template <bool CLUSTER, int CG, int SLOTS, bool WARP>
__device__ __forceinline__ int next_tile(int t, int stride, const TileParams& p, ClcCursor& cur, uint32_t full0,
                                         uint32_t empty0_leader, uint32_t resp0, bool arrive, const Abort& ab) {
  if (!p.clc) return t + stride;
  if (!wait_bar<CLUSTER>(full0 + 8u * cur.slot, cur.phase, ab)) return -1;
  uint32_t first_x;
  const bool got = clc_query(resp0 + 16u * cur.slot, first_x);
  if constexpr (WARP) __syncwarp();  // every lane has read the answer before lane 0 frees the slot
  if (arrive) {  // the answer is in registers already: a relaxed arrive suffices
    if constexpr (CLUSTER) mbar_arrive_relaxed_cluster(empty0_leader + 8u * cur.slot);
    else mbar_arrive_relaxed(empty0_leader + 8u * cur.slot);
  }
  cur.advance(SLOTS);
  return got ? (int)(first_x / CG) : p.num_units;
}

// SLICE: the launch's last round is cut into column slices (single problems,
// static schedule, no split); a separate instantiation, so that the code of
// every other launch stays as it is.
template <int CG, bool OUT_F32, int KIND, int MODE, bool SPLIT, bool SLICE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tn_tiled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                         const TileParams p, const __grid_constant__ KernelArg<MODE, SLICE> karg) {
  static_assert(!SLICE || (MODE == kModeSingle && !SPLIT), "slices: single problems without a split");
  const GroupArg<MODE>& ga = *reinterpret_cast<const GroupArg<MODE>*>(&karg);
  using C_ = Cfg<CG, OUT_F32>;
  constexpr bool kCluster = (CG == 2);
  constexpr int kBK = stage_k_elems<KIND>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + C_::STAGES * C_::A_BYTES;
  const uint32_t sE = sA + C_::RING_BYTES;
  const uint32_t sClc = sE + C_::EPI_TOTAL;           // CLC answers, 16 bytes each
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C_::RING_BYTES + C_::EPI_TOTAL + C_::CLC_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C_::STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * C_::STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * C_::STAGES + 2 + b); };
  auto c_bar = [&](int w, int b) { return bar0 + 8u * (2 * C_::STAGES + 4 + 2 * w + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C_::STAGES + 4 + 2 * kEpiWarps);
  const uint32_t clcf0 = drain_bar + 8u;                          // CLC_FULL[slot]
  const uint32_t clce0 = clcf0 + 8u * C_::CLC_SLOTS;              // CLC_EMPTY[slot] (used in the leader)
  const uint32_t pbar0 = clce0 + 8u * C_::CLC_SLOTS;              // PART[epilogue warp][buffer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C_::NUM_BARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A pair is two CTAs whose cluster ranks differ in bit 0.  The launch may
  // group pairs into larger clusters (a preferred cluster size): the pair's
  // leader is then the CTA of rank pair_base, and its barriers are addressed
  // and its commits multicast by that rank.
  const uint32_t crank = kCluster ? cluster_ctarank() : 0;
  const uint32_t rank = crank & 1u;
  const uint32_t pair_base = crank & ~1u;
  const uint16_t pair_mask = (uint16_t)(0x3u << pair_base);
  const bool leader = (rank == 0);
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;
  // Unit u -> tile and k-part.  Only a split launch (SPLIT, one unit per
  // cluster) has more units than tiles; the finishing part 0 takes the
  // highest units, so every part it waits for has a lower cluster id.
  const int ks = SPLIT ? p.ksplit : 1;
  auto unit_tile = [&](int u) {
    if (SPLIT) return u % p.num_tiles;
    if (SLICE && u >= p.sub_begin) return p.sub_begin + ((u - p.sub_begin) >> p.sub_shift);
    return u;
  };
  auto unit_part = [&](int u) { return SPLIT ? ks - 1 - u / p.num_tiles : 0; };
  // Slice of a unit of the last round (-1: the whole tile).  A slice is
  // BN >> sub_shift columns of its tile, with an MMA of that width.
  auto unit_slice = [&](int u) {
    if (!SLICE || u < p.sub_begin) return -1;
    return (u - p.sub_begin) & ((1 << p.sub_shift) - 1);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C_::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpiWarps * CG);
    }
    for (int w = 0; w < kEpiWarps; ++w)
      for (int b = 0; b < 2; ++b) mbar_init(c_bar(w, b), 1);
    mbar_init(drain_bar, 1);
    for (int s = 0; s < C_::CLC_SLOTS; ++s) {
      mbar_init(clcf0 + 8u * s, 1);
      mbar_init(clce0 + 8u * s, C_::CLC_READERS);
    }
    for (int b = 0; b < 2 * kEpiWarps; ++b) mbar_init(pbar0 + 8u * b, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    // the first tile's tensor maps (kernel parameters: valid before the
    // previous kernel on the stream has finished)
    const TileRef r0 = resolve<MODE>(cluster_id < p.num_units ? unit_tile(cluster_id) : 0, p, ga, &tmA, &tmB,
                                     &tmC, &tmD);
    if (r0.num_kb > 0) {
      tma_prefetch_desc(r0.a);
      tma_prefetch_desc(r0.b);
      if constexpr (SLICE) tma_prefetch_desc(&karg.b);
    }
    if (p.has_c) tma_prefetch_desc(r0.c);
    tma_prefetch_desc(r0.d);
  }
  if (warp == 1) tmem_alloc<CG>(smem_u32(tmem_slot), C_::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  if constexpr (kCluster) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Inputs may come from the previous kernel on the stream: no global memory
  // access before this point (the set-up above overlaps that kernel's tail).
  // Exception: a later launch of one grouped call.  It starts only after every
  // CTA of the launch before it has passed this point, so the inputs are ready;
  // its problems do not touch that launch's, so it runs alongside it and
  // waits at its end instead, which keeps completion in stream order.
  if (!p.defer_wait) griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Abort ab{abort_flag, p.timeout_ns, p.status, kRoleProducer};
      bool ok = true;
      bool skip_once = (p.fault & kFaultSkipTmaOnce) && blockIdx.x == 0;
      int stage = 0;
      uint32_t phase = 0;
      ClcCursor req, rd;  // slot of the next request, slot of the next answer to read
      const uint32_t clce_leader = kCluster ? mapa_shared(clce0, pair_base) : clce0;
      // L2 priorities (single problems): A rows are re-read by every tile of
      // their raster strip, B columns only by the strip's few concurrent tiles
      const bool hint_a = MODE == kModeSingle && (p.l2_hints & kL2HintAEvictLast);
      const bool hint_b = MODE == kModeSingle && (p.l2_hints & kL2HintBEvictFirst);
      const uint64_t pol_a = l2_policy_evict_last(), pol_b = l2_policy_evict_first();
      int t = cluster_id;
      while (t < p.num_units && ok) {
        if (p.clc) {
          // ask for the tile after this one now; the answer is read once this tile's loads are issued
          if (leader && !wait_bar<kCluster>(clce0 + 8u * req.slot, req.phase ^ 1, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(clcf0 + 8u * req.slot, 16);
          if (leader) {
            if constexpr (CG == 2) clc_try_cancel_multicast(sClc + 16u * req.slot, clcf0 + 8u * req.slot);
            else clc_try_cancel(sClc + 16u * req.slot, clcf0 + 8u * req.slot);
          }
          req.advance(C_::CLC_SLOTS);
        }
        const TileRef r = resolve<MODE>(unit_tile(t), p, ga, &tmA, &tmB, &tmC, &tmD);
        int kb0, kb1;
        part_range(r.num_kb, ks, unit_part(t), kb0, kb1);
        if constexpr (MODE == kModeList) {
          // a list's next tile is usually another problem: fetch its maps early
          const int tn_next = t + num_clusters;
          if (!p.clc && tn_next < p.num_tiles) {
            const TileRef rn = resolve<MODE>(tn_next, p, ga, &tmA, &tmB, &tmC, &tmD);
            if (rn.num_kb > 0) {
              tma_prefetch_desc(rn.a);
              tma_prefetch_desc(rn.b);
            }
            if (p.has_c) tma_prefetch_desc(rn.c);
            tma_prefetch_desc(rn.d);
          }
        }
        const int a_row = r.tm * C_::TILE_M + (int)rank * 128;
        const CUtensorMap* bmap = r.b;
        int b_row = r.tn * C_::BN + (int)rank * C_::B_ROWS;
        uint32_t stage_tx = C_::STAGE_TX;
        if constexpr (SLICE) {
          const int slice = unit_slice(t);
          if (slice >= 0) {
            // this CTA's rows of the slice, through the map with slice-high boxes
            const int cols = C_::BN >> p.sub_shift;
            bmap = &karg.b;
            b_row = r.tn * C_::BN + slice * cols + (int)rank * (cols / CG);
            stage_tx = (uint32_t)((C_::A_BYTES + (C_::B_BYTES >> p.sub_shift)) * CG);
          }
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar<kCluster>(empty_bar(stage), phase ^ 1, ab)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          if (leader) mbar_arrive_expect_tx(fb, stage_tx);
          if (skip_once) {
            skip_once = false;  // test-only: leave this stage's bytes missing
          } else if constexpr (CG == 1) {
            if (hint_a) tma_load_2d_hint(sA + stage * C_::A_BYTES, r.a, kb * kBK, a_row, fb, pol_a);
            else tload<MODE>(sA + stage * C_::A_BYTES, r.a, kb * kBK, a_row, r.z, fb);
            if (hint_b) tma_load_2d_hint(sB + stage * C_::B_BYTES, bmap, kb * kBK, b_row, fb, pol_b);
            else tload<MODE>(sB + stage * C_::B_BYTES, bmap, kb * kBK, b_row, r.z, fb);
          } else {
            const uint32_t fb_leader = mapa_shared(fb, pair_base);
            if (hint_a) tma_load_2d_pair_hint(sA + stage * C_::A_BYTES, r.a, kb * kBK, a_row, fb_leader, pol_a);
            else tload_pair<MODE>(sA + stage * C_::A_BYTES, r.a, kb * kBK, a_row, r.z, fb_leader);
            if (hint_b) tma_load_2d_pair_hint(sB + stage * C_::B_BYTES, bmap, kb * kBK, b_row, fb_leader, pol_b);
            else tload_pair<MODE>(sB + stage * C_::B_BYTES, bmap, kb * kBK, b_row, r.z, fb_leader);
          }
          if (++stage == C_::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        t = next_tile<kCluster, CG, C_::CLC_SLOTS, false>(t, num_clusters, p, rd, clcf0, clce_leader, sClc, true, ab);
        if (t < 0) ok = false;
      }
      if (!ok) settle(2000000);  // copies (and a CLC answer) already issued land before teardown
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      Abort ab{abort_flag, p.timeout_ns, p.status, kRoleMma};
      const uint32_t idesc = KIND == kKindF16 ? instr_desc_bf16_f32(C_::TILE_M, C_::BN)
                                              : instr_desc_f32acc(C_::TILE_M, C_::BN, p.a_fmt, p.b_fmt);
      const uint32_t slice_n = (uint32_t)(C_::BN >> p.sub_shift);
      const uint32_t idesc_slice = KIND == kKindF16 ? instr_desc_bf16_f32(C_::TILE_M, slice_n)
                                                    : instr_desc_f32acc(C_::TILE_M, slice_n, p.a_fmt, p.b_fmt);
      bool ok = true;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      ClcCursor rd;
      const uint32_t clce_leader = kCluster ? mapa_shared(clce0, pair_base) : clce0;
      int t = cluster_id;
      while (t < p.num_units && ok) {
        if (!wait_bar<kCluster>(acce_bar(acc), acc_phase ^ 1, ab)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C_::BN);
        const uint32_t id = (SLICE && unit_slice(t) >= 0) ? idesc_slice : idesc;
        int kb0, kb1;
        part_range(resolve<MODE>(unit_tile(t), p, ga, &tmA, &tmB, &tmC, &tmD).num_kb, ks, unit_part(t), kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar<kCluster>(full_bar(stage), phase, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a0 = smem_desc_sw128(sA + stage * C_::A_BYTES);
          const uint64_t b0 = smem_desc_sw128(sB + stage * C_::B_BYTES);
#pragma unroll
          for (int k = 0; k < kMmaPerStage; ++k) {
            // +32 bytes along K inside the swizzle atom = +2 in the encoded address
            mma_issue<CG, KIND>(d_tmem, a0 + 2 * k, b0 + 2 * k, id, (kb != kb0 || k != 0) ? 1u : 0u);
          }
          if constexpr (CG == 1) mma_commit(empty_bar(stage));
          else mma_commit_pair(empty_bar(stage), pair_mask);
          if (++stage == C_::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (CG == 1) mma_commit(accf_bar(acc));
        else mma_commit_pair(accf_bar(acc), pair_mask);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        t = next_tile<kCluster, CG, C_::CLC_SLOTS, false>(t, num_clusters, p, rd, clcf0, clce_leader, sClc, true, ab);
        if (t < 0) break;
      }
      // All MMAs issued by this thread complete before TMEM is released.
      if constexpr (CG == 1) mma_commit(drain_bar);
      else mma_commit_pair(drain_bar, (uint16_t)(0x1u << pair_base));
      Abort ab_drain{nullptr, p.timeout_ns, p.status, kRoleMma};
      wait_bar<kCluster>(drain_bar, 0, ab_drain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;          // staging slot 0..3
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    Abort ab{abort_flag, p.timeout_ns, p.status, kRoleEpilogue};
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t cphase0 = 0, cphase1 = 0;
    int buf = 0;
    const uint32_t acce_target = kCluster ? mapa_shared(acce_bar(0), pair_base) : acce_bar(0);
    ClcCursor rd;
    const uint32_t clce_leader = kCluster ? mapa_shared(clce0, pair_base) : clce0;
    int t = cluster_id;
    while (t < p.num_units) {
      const int tile = unit_tile(t);
      const int part = unit_part(t);
      const TileRef tr = resolve<MODE>(tile, p, ga, &tmA, &tmB, &tmC, &tmD);
      const int slice = SLICE ? unit_slice(t) : -1;
      const int cols = slice >= 0 ? (C_::BN >> p.sub_shift) : C_::BN;   // this unit's columns
      const int col_base = tr.tn * C_::BN + (slice >= 0 ? slice * cols : 0);
      const int chunks = cols / C_::EPI_COLS;
      const int row0 = tr.tm * C_::TILE_M + (int)rank * 128 + q * 32;
      // Split tile: parts > 0 publish this warp's 32 rows x 256 columns of
      // raw fp32 accumulators and count them; part 0 waits for the count and
      // adds the parts in order before the epilogue proper.
      int* arrivals = ks > 1 ? p.counters + ((long long)tile * CG + rank) * 4 + q : nullptr;
      // this warp's 32 x 32 block of part pt, chunk c (4 KiB, contiguous).
      // Inside it, float4 j of lane l (columns 4j..4j+3 of row l) sits at
      // float4 index j * 32 + l: a warp's stores of one j cover 512
      // contiguous bytes, and the staged copy is read without bank conflicts.
      // (With each lane's 32 values contiguous instead, publishing and adding
      // the partials took 5 us and 2.2 us per chunk at 256 x 2048 x 8192.)
      auto partial_at = [&](int pt, int c) {
        return p.partials + ((((long long)tile * (ks - 1) + (pt - 1)) * CG + rank) * (C_::BN / 32) + c) *
                                (128 * 32) +
               q * 32 * 32;
      };
      // Part 0 stages the other parts' chunks in the operand ring, two chunks
      // ahead, with bulk copies: a split launch runs one unit per cluster, so
      // once the accumulator is complete no MMA or load touches the ring.
      const bool fix = SPLIT && ks > 1 && part == 0;
      const uint32_t pstage = sA + (uint32_t)(ew * 2 * 3 * C_::PART_SLOT);
      auto fetch = [&](int c) {
        const uint32_t bar = pbar0 + 8u * (uint32_t)(ew * 2 + (c & 1));
        mbar_arrive_expect_tx(bar, (uint32_t)((ks - 1) * C_::PART_SLOT));
        for (int pt = 1; pt < ks; ++pt)
          bulk_load_1d(pstage + (uint32_t)(((c & 1) * 3 + pt - 1) * C_::PART_SLOT), partial_at(pt, c),
                       C_::PART_SLOT, bar);
      };
      if (!wait_bar<kCluster>(accf_bar(acc), acc_phase, ab)) break;
      tc_fence_after();
      if (fix) {
        Abort abf{abort_flag, p.timeout_ns, p.status, kRoleFixup};
        if (!wait_parts(arrivals, ks - 1, abf)) break;
        if (lane == 0) {
          fence_proxy_async_global();  // the acquired partials, then the bulk copies that read them
          fetch(0);
          fetch(1);
        }
      }
#pragma unroll 1
      for (int c = 0; c < chunks; ++c) {
        const int col0 = col_base + c * C_::EPI_COLS;
        uint32_t r[32];
        if (tr.num_kb > 0) {
          tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C_::BN + c * 32), r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0;
        }
        if (c == chunks - 1) {
          // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kCluster) mbar_arrive_cluster(acce_target + 8u * acc);
            else mbar_arrive(acce_bar(acc));
          }
        }
        if (part > 0) {
          float4* dst = reinterpret_cast<float4*>(partial_at(part, c)) + lane;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j * 32] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                      __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          continue;
        }
        if (fix) {
          // parts in order: (0 + part 0) + part 1 + ...; the chunk's barrier
          // is consumed even for a box outside D, so the phases stay in step
          const int b = c & 1;
          if (!wait_bar<false>(pbar0 + 8u * (uint32_t)(ew * 2 + b), (uint32_t)((c >> 1) & 1), ab)) break;
          float a[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = 0.0f + __uint_as_float(r[j]);
          for (int pt = 1; pt < ks; ++pt) {
            const uint32_t src = pstage + (uint32_t)((b * 3 + pt - 1) * C_::PART_SLOT) + (uint32_t)lane * 16u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t x0, x1, x2, x3;
              ld_shared_v4(src + 512u * j, x0, x1, x2, x3);
              a[4 * j] += __uint_as_float(x0);
              a[4 * j + 1] += __uint_as_float(x1);
              a[4 * j + 2] += __uint_as_float(x2);
              a[4 * j + 3] += __uint_as_float(x3);
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(a[j]);
          __syncwarp();  // every lane has read buffer b
          if (lane == 0 && c + 2 < C_::BN / C_::EPI_COLS) fetch(c + 2);
        }
        if (row0 >= tr.M || col0 >= tr.N) continue;  // box entirely outside D
        const uint32_t sbuf = sE + (uint32_t)((ew * 2 + buf) * C_::EPI_BYTES);
        if (lane == 0) bulk_wait_read<1>();       // buffer's previous store has read it
        __syncwarp();
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[j]);
        if (p.has_c) {
          const uint32_t cb = c_bar(ew, buf);
          if (lane == 0) {
            mbar_arrive_expect_tx(cb, C_::EPI_BYTES);
            tload<MODE>(sbuf, tr.c, col0, row0, tr.z, cb);
          }
          const uint32_t par = buf ? cphase1 : cphase0;
          if (!wait_bar<false>(cb, par, ab)) break;
          if (buf) cphase1 ^= 1; else cphase0 ^= 1;
          if constexpr (OUT_F32) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t x0, x1, x2, x3;
              ld_shared_v4(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4), x0, x1, x2, x3);
              v[4 * j + 0] = fmaf(p.beta, __uint_as_float(x0), v[4 * j + 0]);
              v[4 * j + 1] = fmaf(p.beta, __uint_as_float(x1), v[4 * j + 1]);
              v[4 * j + 2] = fmaf(p.beta, __uint_as_float(x2), v[4 * j + 2]);
              v[4 * j + 3] = fmaf(p.beta, __uint_as_float(x3), v[4 * j + 3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t x[4];
              ld_shared_v4(sbuf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), x[0], x[1], x[2], x[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[8 * j + 2 * e + 0] = fmaf(p.beta, __uint_as_float(x[e] << 16), v[8 * j + 2 * e + 0]);
                v[8 * j + 2 * e + 1] = fmaf(p.beta, __uint_as_float(x[e] & 0xFFFF0000u), v[8 * j + 2 * e + 1]);
              }
            }
          }
        }
        // bias and activation, on the finisher's sums in a split launch (the
        // host splits fused calls only into four long parts, where the split
        // pays for the epilogue sitting after the hand-off)
        if (p.epi.bias || p.epi.act) {
          // bias is per column: lane l fetches column col0 + l, every lane
          // then takes the 32 values by shuffle
          if (p.epi.bias) {
            const float bl = col0 + lane < p.N ? load_bias(p.epi, col0 + lane) : 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xffffffffu, bl, j);
          }
          activate_chunk(v, p.epi.act);
        }
        if constexpr (OUT_F32) {
          // 128-byte rows, 128-byte swizzle: 16-byte chunk j sits at j ^ (row % 8)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4), __float_as_uint(v[4 * j]),
                         __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                         __float_as_uint(v[4 * j + 3]));
        } else {
          // 64-byte rows, 64-byte swizzle: 16-byte chunk j sits at j ^ ((row / 2) % 4)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_shared_v4(sbuf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), pack_bf16x2(v[8 * j], v[8 * j + 1]),
                         pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                         pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // D is written once and not read again by this kernel
          if (MODE == kModeSingle && (p.l2_hints & kL2HintDEvictFirst))
            tma_store_2d_hint(tr.d, col0, row0, sbuf, l2_policy_evict_first());
          else tstore<MODE>(tr.d, col0, row0, tr.z, sbuf);
          bulk_commit();
        }
        buf ^= 1;
      }
      if (part > 0) {
        // every lane's partial is written before lane 0 counts it
        __syncwarp();
        if (lane == 0) red_add_release_gpu(arrivals, 1);
      }
      if (*abort_flag) break;
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
      t = next_tile<kCluster, CG, C_::CLC_SLOTS, true>(t, num_clusters, p, rd, clcf0, clce_leader, sClc, lane == 0,
                                                       ab);
      if (t < 0) break;
    }
    if (lane == 0) bulk_wait<0>();
    // an aborted k-split fix-up may leave bulk copies of partials in flight
    if (SPLIT && ks > 1 && *abort_flag && lane == 0) settle(1000000);
  }

  __syncthreads();
  if constexpr (kCluster) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, C_::TMEM_COLS);
  }
  if (p.defer_wait) griddep_wait();
}

template <int CG, bool OUT_F32, int KIND, int MODE, bool SPLIT, bool SLICE = false>
cudaError_t launch_impl(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const CUtensorMap& tmD, const TileParams& p_in, const KernelArg<MODE, SLICE>& ga,
                        int grid_override, bool pdl, cudaStream_t stream, LaunchInfo* info) {
  TileParams p = p_in;
  if (!SPLIT || MODE != kModeSingle || p.clc || p.ksplit < 1 || !p.partials || !p.counters) p.ksplit = 1;
  using C_ = Cfg<CG, OUT_F32>;
  static_assert(sizeof(KernelArg<MODE, SLICE>) + 4 * sizeof(CUtensorMap) + sizeof(TileParams) < 32000,
                "kernel parameters must stay within 32 KB");
  auto kern = gemm_tn_tiled_kernel<CG, OUT_F32, KIND, MODE, SPLIT, SLICE>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::SMEM);
    if (e != cudaSuccess) return e;
    if (CG == 2) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      (void)e;
    }
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C_::SMEM;
  cfg.stream = stream;
  int num_attrs = 0;
  if (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    num_attrs = 1;
  }
  const int n_occupancy_attrs = num_attrs;
  if (pdl) {
    attr[num_attrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[num_attrs].val.programmaticStreamSerializationAllowed = 1;
    ++num_attrs;
  }
  cfg.attrs = attr;
  cfg.numAttrs = num_attrs;

  // Persistent grid: as many CTAs (pairs) as can be co-resident, never more
  // than there are tiles.
  int max_units = 0;
  if (CG == 2) {
    cfg.gridDim = dim3(2, 1, 1);
    cfg.numAttrs = n_occupancy_attrs;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    cfg.numAttrs = num_attrs;
    if (e != cudaSuccess) return e;
    max_units = clusters;
  } else {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    max_units = sms;
  }
  if (max_units < 1) return cudaErrorInvalidConfiguration;
  // A split tile's part 0 waits for its other parts: every unit must have
  // its own co-resident cluster, so the split shrinks to what fits.
  while (p.ksplit > 1 && (long long)p.num_tiles * p.ksplit > max_units) --p.ksplit;
  p.num_units = p.num_tiles * p.ksplit;
  // slices of the last round: static single-problem launches without a split
  if (SLICE && p.ksplit == 1 && !p.clc && grid_override <= 0 && p.sub_shift > 0 && p.sub_shift <= 2 &&
      p.sub_begin >= 0 && p.sub_begin < p.num_tiles) {
    p.num_units = p.sub_begin + ((p.num_tiles - p.sub_begin) << p.sub_shift);
  } else {
    p.sub_begin = p.num_units;
    p.sub_shift = 0;
  }
  int units = p.num_units < max_units ? p.num_units : max_units;
  if (grid_override > 0 && p.ksplit == 1) units = grid_override / CG;
  // cluster launch control: one cluster per tile; the ones that find their
  // tile already taken over are cancelled before they start
  if (p.clc) units = p.num_tiles;
  if (units < 1) units = 1;
  cfg.gridDim = dim3(units * CG, 1, 1);
  // Preferred cluster size (pairs grouped into clusters of 4 or 8 CTAs where
  // the GPU's clusters of SMs have room, single pairs elsewhere): a static
  // single-problem pair launch whose grid it divides.
  int pref = 0;
  if (CG == 2 && MODE == kModeSingle && !p.clc && (p.cluster_pref == 4 || p.cluster_pref == 8) &&
      (units * CG) % p.cluster_pref == 0) {
    pref = p.cluster_pref;
    attr[num_attrs].id = cudaLaunchAttributePreferredClusterDimension;
    attr[num_attrs].val.preferredClusterDim.x = (unsigned)pref;
    attr[num_attrs].val.preferredClusterDim.y = 1;
    attr[num_attrs].val.preferredClusterDim.z = 1;
    ++num_attrs;
    cfg.numAttrs = num_attrs;
  }
  if (info) {
    info->path = CG;
    info->scheduler = p.clc ? 2 : 1;
    info->k_parts = p.ksplit;
    info->grid = units * CG;
    info->cluster = CG;
    info->cluster_pref = pref;
    info->tail_slices = 1 << p.sub_shift;
    info->block = kThreads;
    info->tile_m = C_::TILE_M;
    info->tile_n = C_::BN;
    info->stages = C_::STAGES;
    info->smem_bytes = C_::SMEM;
    static const char* names[2][2][2] = {
        {{"gemm_tn_tiled_kernel<1,bf16>", "gemm_tn_tiled_kernel<1,f32>"},
         {"gemm_tn_tiled_kernel<2,bf16>", "gemm_tn_tiled_kernel<2,f32>"}},
        {{"gemm_tn_tiled_kernel<1,bf16,fp8 in>", "gemm_tn_tiled_kernel<1,f32,fp8 in>"},
         {"gemm_tn_tiled_kernel<2,bf16,fp8 in>", "gemm_tn_tiled_kernel<2,f32,fp8 in>"}}};
    static const char* group_names[2][2][2] = {
        {{"gemm_tn_tiled_kernel<1,bf16,list>", "gemm_tn_tiled_kernel<1,f32,list>"},
         {"gemm_tn_tiled_kernel<2,bf16,list>", "gemm_tn_tiled_kernel<2,f32,list>"}},
        {{"gemm_tn_tiled_kernel<1,bf16,strided>", "gemm_tn_tiled_kernel<1,f32,strided>"},
         {"gemm_tn_tiled_kernel<2,bf16,strided>", "gemm_tn_tiled_kernel<2,f32,strided>"}}};
    static const char* split_names[2][2][2] = {
        {{"gemm_tn_tiled_kernel<1,bf16,split>", "gemm_tn_tiled_kernel<1,f32,split>"},
         {"gemm_tn_tiled_kernel<2,bf16,split>", "gemm_tn_tiled_kernel<2,f32,split>"}},
        {{"gemm_tn_tiled_kernel<1,bf16,fp8 in,split>", "gemm_tn_tiled_kernel<1,f32,fp8 in,split>"},
         {"gemm_tn_tiled_kernel<2,bf16,fp8 in,split>", "gemm_tn_tiled_kernel<2,f32,fp8 in,split>"}}};
    static const char* slice_names[2][2][2] = {
        {{"gemm_tn_tiled_kernel<1,bf16,slices>", "gemm_tn_tiled_kernel<1,f32,slices>"},
         {"gemm_tn_tiled_kernel<2,bf16,slices>", "gemm_tn_tiled_kernel<2,f32,slices>"}},
        {{"gemm_tn_tiled_kernel<1,bf16,fp8 in,slices>", "gemm_tn_tiled_kernel<1,f32,fp8 in,slices>"},
         {"gemm_tn_tiled_kernel<2,bf16,fp8 in,slices>", "gemm_tn_tiled_kernel<2,f32,fp8 in,slices>"}}};
    info->kernel = MODE != kModeSingle ? group_names[MODE == kModeStrided][CG - 1][OUT_F32 ? 1 : 0]
                   : p.ksplit > 1  ? split_names[KIND][CG - 1][OUT_F32 ? 1 : 0]
                   : SLICE         ? slice_names[KIND][CG - 1][OUT_F32 ? 1 : 0]
                                   : names[KIND][CG - 1][OUT_F32 ? 1 : 0];
  }
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, tmD, p, ga);
}

}  // namespace

void tiled_shape(int cta_group, int out_f32, int* tile_m, int* tile_n, int* b_rows_per_cta, int* epi_rows,
                 int* epi_cols) {
  (void)out_f32;
  *tile_m = 128 * cta_group;
  *tile_n = 256;
  *b_rows_per_cta = 256 / cta_group;
  *epi_rows = 32;
  *epi_cols = 32;
}

cudaError_t launch_tiled(int cta_group, int out_f32, int kind, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const CUtensorMap& tmC, const CUtensorMap& tmD, const CUtensorMap& tmBs, TileParams p,
                         int grid_override, bool pdl, cudaStream_t stream, LaunchInfo* info) {
  const NoGroup none{0};
  SliceArg sl;
  sl.b = tmBs;
  const bool slices = p.ksplit <= 1 && p.sub_shift > 0;
#define GTN_LAUNCH(CGV, OF, KV)                                                                                    \
  (p.ksplit > 1 ? launch_impl<CGV, OF, KV, kModeSingle, true>(tmA, tmB, tmC, tmD, p, none, grid_override, pdl,      \
                                                               stream, info)                                      \
   : slices     ? launch_impl<CGV, OF, KV, kModeSingle, false, true>(tmA, tmB, tmC, tmD, p, sl, grid_override, pdl, \
                                                                      stream, info)                               \
                : launch_impl<CGV, OF, KV, kModeSingle, false>(tmA, tmB, tmC, tmD, p, none, grid_override, pdl,     \
                                                                stream, info))
  if (kind == kKindF8F6F4) {
    if (cta_group == 2) return out_f32 ? GTN_LAUNCH(2, true, kKindF8F6F4) : GTN_LAUNCH(2, false, kKindF8F6F4);
    return out_f32 ? GTN_LAUNCH(1, true, kKindF8F6F4) : GTN_LAUNCH(1, false, kKindF8F6F4);
  }
  if (cta_group == 2) return out_f32 ? GTN_LAUNCH(2, true, kKindF16) : GTN_LAUNCH(2, false, kKindF16);
  return out_f32 ? GTN_LAUNCH(1, true, kKindF16) : GTN_LAUNCH(1, false, kKindF16);
#undef GTN_LAUNCH
}

cudaError_t launch_tiled_group(int cta_group, int out_f32, int mode, const CUtensorMap& tmA, const CUtensorMap& tmB,
                               const CUtensorMap& tmC, const CUtensorMap& tmD, const GroupList* list, TileParams p,
                               bool pdl, cudaStream_t stream, LaunchInfo* info) {
  if (mode == kModeList) {
#define GTN_LAUNCH(CGV, OF) \
  launch_impl<CGV, OF, kKindF16, kModeList, false>(tmA, tmB, tmC, tmD, p, *list, 0, pdl, stream, info)
    if (cta_group == 2) return out_f32 ? GTN_LAUNCH(2, true) : GTN_LAUNCH(2, false);
    return out_f32 ? GTN_LAUNCH(1, true) : GTN_LAUNCH(1, false);
#undef GTN_LAUNCH
  }
  const NoGroup none{0};
#define GTN_LAUNCH(CGV, OF) \
  launch_impl<CGV, OF, kKindF16, kModeStrided, false>(tmA, tmB, tmC, tmD, p, none, 0, pdl, stream, info)
  if (cta_group == 2) return out_f32 ? GTN_LAUNCH(2, true) : GTN_LAUNCH(2, false);
  return out_f32 ? GTN_LAUNCH(1, true) : GTN_LAUNCH(1, false);
#undef GTN_LAUNCH
}

}  // namespace gtn
