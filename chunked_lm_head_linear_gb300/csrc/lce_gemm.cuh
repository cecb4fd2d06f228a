// Persistent, warp-specialised tcgen05 GEMM core shared by the three
// contractions of the fused LM-head cross-entropy:
//
//   logits   z_c  = H_c W^T        A = H_c   [C, d] K-major,  B = W   [V, d] K-major
//   input    dH_c = G_c W          A = G_c   [C, V] K-major,  B = W   [V, d] MN-major
//   weight   dW  += G_c^T H_c      A = G_c^T (G_c MN-major), B = H_c [C, d] MN-major
//
// ("XTuner on Ascend 910C: Qwen3.5-2B training optimisation", section 3.1.4:
// the logits chunk, and the backward's d_input / d_weight.)
//
// The kernel runs on clusters of two CTAs (the two SMs of one TPC) and computes 256 x 256
// output tiles with tcgen05.mma.cta_group::2. Each CTA has 256 threads:
//   warp 0      TMA producer (one thread): its CTA's half of the A/B k-blocks
//   warp 1      MMA issuer (one thread, even CTA of the pair)
//   warp 2      TMEM allocator (512 columns = two 128x256 fp32 accumulators)
//   warps 4-7   epilogue: warp w reads TMEM lanes 32*(w%4).. (the hardware
//               lane quarter of its sub-partition) of its CTA's 128 rows, all
//               256 columns in two halves, does the per-tile arithmetic and
//               writes results through its own 4 KiB shared-memory staging
//               tile with TMA stores (or reduce-adds). One epilogue warp per
//               sub-partition: with two, the producer and MMA issuer (which
//               share sub-partitions 0 and 1 with them) lost issue slots
//               (measured 1.9% slower).
// The two accumulators alternate so the epilogue of tile t overlaps the main
// loop of tile t+1. What is multiplied, how operands are loaded and what the
// epilogue does come from a problem type (see lce_kernels.cu): one GEMM, or
// the dH and dW GEMMs of the backward in one launch.
#pragma once

#include "lce_internal.h"
#include "sm100_ptx.cuh"

namespace lce {

constexpr int BM = 128;             // rows of an output tile (TMEM lanes)
constexpr int BN = 256;             // columns of an output tile (TMEM columns)
constexpr int BK = 64;              // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int MN_SLAB_BYTES = 64 * BK * 2;   // one 64-wide MN slab of a k-block: 8 KiB
constexpr int EPI_WARP0 = 4;
constexpr int EPI_WARPS = 4;             // one per TMEM lane quarter (see the role list above)
constexpr int EPI_COLS = BN / 2;             // columns of the tile one epilogue warp owns
constexpr int NUM_THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr int STAGE_TILE_BYTES = 4096;       // 32 rows x 128 bytes, 128-byte swizzled
constexpr int TMEM_COLS = 2 * BN;

// ============================================================================
// The CTA-pair kernel: tcgen05.mma.cta_group::2, 256 x 256 output tile per
// pair. CTA rank r of the pair loads rows [128 r, 128 r + 128) of the A tile
// and columns [128 r, 128 r + 128) of the B tile into its own shared memory;
// the even CTA's MMA thread multiplies across both, and accumulator rows
// 128 r.. live in CTA r's TMEM. Per SM and 64-deep k-block this moves 32 KiB,
// and the ring is 6 deep.
//   full[s]   (even CTA only) : its own arrive.expect_tx of the pair's bytes +
//                               the byte counts of both CTAs' loads
//   empty[s]  (both CTAs)     : multicast commit from the even CTA's MMAs
//   tfull[a]  (both CTAs)     : multicast commit after a tile's last k-block
//   tempty[a] (even CTA only) : one arrival per epilogue warp of both CTAs
// ============================================================================
constexpr int P_STAGES = 6;
constexpr int P_A_BYTES = 128 * BK * 2;   // 16 KiB: this CTA's 128 rows of A
constexpr int P_B_BYTES = 128 * BK * 2;   // 16 KiB: this CTA's 128 columns of B
constexpr int P_TILE_M = 256;

struct PairSmemLayout {
  static constexpr int kTiles = P_STAGES * (P_A_BYTES + P_B_BYTES);
  static constexpr int kStaging = kTiles;
  static constexpr int kBars = kStaging + EPI_WARPS * STAGE_TILE_BYTES;
  static constexpr int kNumBars = 2 * P_STAGES + 4 + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kDynamicBytes = kTotal + 1024;
};
static_assert(PairSmemLayout::kDynamicBytes <= 232448, "shared memory budget (pair kernel)");

// A tile of work: which GEMM of the problem (kind), its 256-row block, its
// 256-column block, its number of k-blocks, the first of them (k-block kb0 of
// the operands' K extent) and, for a reduction cut into parts, which part.
struct TileJob {
  int kind, mb, nb, k_blocks, kb0, part;
};

// What an epilogue warp needs besides its tile: its staging tile, the store
// map and where its 32 rows start.
struct EpiCtx {
  uint8_t* stage;            // this warp's staging tile (1 KiB aligned)
  const CUtensorMap* out;    // TMA store / reduce map of the epilogue's output
  int lane;
  int row0;                  // first tile row of this warp (tile-relative)
  int* flags;                // device status word (bounds bit of the checked build)
};

// Byte offset of 16-byte chunk j of row r in a 128-byte-swizzled staging tile.
__device__ __forceinline__ uint32_t stage_off(int r, int j) {
  return static_cast<uint32_t>(r * 128 + ((j ^ (r & 7)) << 4));
}

// Before rewriting the staging tile: the previous TMA store must have read it.
__device__ __forceinline__ void stage_acquire(const EpiCtx& c) {
  if (c.lane == 0) bulk_wait_read_all();
  __syncwarp();
}

// Hand the staging tile to TMA: store (or add) it at element (x, y) of the output.
__device__ __forceinline__ void stage_release(const EpiCtx& c, int x, int y, bool reduce_add) {
  fence_proxy_async_smem();
  __syncwarp();
  if (c.lane == 0) {
    // checked build: a store box starts at a non-negative, 16-byte aligned element (x % 8 == 0
    // covers both bf16 and fp32 outputs); otherwise the store is skipped
    bool ok = true;
    if constexpr (kChecks)
      ok = in_bounds(x, 1ll << 31, c.flags) && in_bounds(y, 1ll << 31, c.flags) && in_bounds(x % 8, 1, c.flags);
    if (!ok) {
    } else if (reduce_add)
      tma_reduce_add_2d(c.out, c.stage, x, y);
    else
      tma_store_2d(c.out, c.stage, x, y);
    bulk_commit();
  }
}

__device__ __forceinline__ void report_timeout(volatile int* abort, int* flags) {
  *abort = 1;
  atomicOr(flags, kFlagTimeout);
}

// Shared-memory descriptors of one 16-deep K step (k = 0..3 within a 64-wide
// k-block) of a 128-row (or 128-column) operand half in 128-byte swizzle:
// K-major: the next 16 elements are 32 bytes further along each row;
// MN-major: two 64-wide slabs 8 KiB apart, the next 16 K rows 2 KiB further.
__device__ __forceinline__ uint64_t desc_k_major(uint32_t addr, int k) {
  return smem_desc_sw128(addr + k * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mn_major(uint32_t addr, int k) {
  return smem_desc_sw128(addr + k * 2048, MN_SLAB_BYTES, 1024);
}

__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort, int lane) {
  int ok = 0;
  if (lane == 0) ok = mbar_wait_cluster(bar, parity, abort) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded pause (used only when leaving after a timeout, so that copies the
// CTA issued have landed before the pair is released).
__device__ __forceinline__ void pause_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

// Problem interface (Prob):
//   Params                      kernel parameters (tensor maps, shapes, epilogue params)
//   State                       per-epilogue-thread constants
//   skip(p)                     conditional launch: true = do nothing
//   no_loads(p)                 timeout test: the producer issues no loads
//   flags(p)                    device status word
//   num_jobs(p, cluster, P)     number of tiles of this cluster (P clusters in the grid)
//   job(p, cluster, P, j)       its j-th tile
//   job_ok(p, job)              the tile lies inside the problem (checked build only)
//   load(p, kind, a, b, bar, m0, n0, k0)  this CTA's half of the k-block (TMA, pair form)
//   a_desc / b_desc(kind, addr, k), idesc(kind)   MMA descriptors
//   init(p, st), epilogue(p, st, job, ctx, m0, col0, taddr)
template <class Prob>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ typename Prob::Params p) {
  grid_dep_wait();    // everything below reads or writes what earlier kernels of the stream touch
  grid_dep_launch();
  if (Prob::skip(p)) return;  // same value in both CTAs of the pair (one global word)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sA = smem;
  uint8_t* sB = smem + P_STAGES * P_A_BYTES;
  uint8_t* staging = smem + PairSmemLayout::kStaging;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PairSmemLayout::kBars);
  uint64_t* full = bars;
  uint64_t* empty = bars + P_STAGES;
  uint64_t* tfull = bars + 2 * P_STAGES;
  uint64_t* tempty = bars + 2 * P_STAGES + 2;
  uint64_t* drain = bars + 2 * P_STAGES + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + PairSmemLayout::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + PairSmemLayout::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);
  const int njobs = Prob::num_jobs(p, cluster, nclusters);
  int* flags = Prob::flags(p);

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before anything signals them
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;
    bool ok = !Prob::no_loads(p);  // (timeout test: issue nothing)
    for (int j = 0; j < njobs && ok; ++j) {
      const TileJob tj = Prob::job(p, cluster, nclusters, j);
      if (kChecks && !Prob::job_ok(p, tj)) {  // checked build: every role skips a bad tile
        atomicOr(flags, kFlagBounds);
        continue;
      }
      const int m0 = tj.mb * P_TILE_M + static_cast<int>(rank) * 128;  // this CTA's A rows
      const int nh = tj.nb * BN + static_cast<int>(rank) * 128;         // this CTA's B columns
      for (int kb = 0; kb < tj.k_blocks; ++kb) {
        if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, abort)) {
          report_timeout(abort, flags);
          ok = false;
          break;
        }
        const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (P_A_BYTES + P_B_BYTES));
        Prob::load(p, tj.kind, sA + stage * P_A_BYTES, sB + stage * P_B_BYTES, fbar, m0, nh, (tj.kb0 + kb) * BK);
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if ((!ok && !Prob::no_loads(p)) || *abort) {
      if (rank == 0)
        for (int s = 0; s < P_STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(&full[s], (armed_parity >> s) & 1u, 100000000ull);
      pause_ns(200000);  // let copies this CTA issued land before the pair is released
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (even CTA) ----------------
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    bool issued = false;
    for (int j = 0; j < njobs && ok; ++j) {
      const TileJob tj = Prob::job(p, cluster, nclusters, j);
      if (kChecks && !Prob::job_ok(p, tj)) continue;
      const uint32_t idesc = Prob::idesc(tj.kind);
      if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort)) {
        report_timeout(abort, flags);
        break;
      }
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < tj.k_blocks; ++kb) {
        if (!mbar_wait_cluster(&full[stage], phase, abort)) {
          report_timeout(abort, flags);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(sA + stage * P_A_BYTES);
        const uint32_t b_addr = smem_u32(sB + stage * P_B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          umma_bf16_pair(d_tmem, Prob::a_desc(tj.kind, a_addr, k), Prob::b_desc(tj.kind, b_addr, k), idesc,
                         (kb | k) != 0 ? 1u : 0u);
        issued = true;
        umma_commit_pair(&empty[stage], 0x3);
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit_pair(&tfull[acc], 0x3);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (*abort && issued) {
      umma_commit_pair(drain, 0x1);
      mbar_wait_drain(drain, 0, 100000000ull);
    }
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue (both CTAs) ----------------
    const int e = warp - EPI_WARP0;
    const int q = warp & 3;
    const int half = e >> 2;
    EpiCtx ctx{staging + e * STAGE_TILE_BYTES, nullptr, lane, q * 32, flags};
    int acc = 0;
    uint32_t acc_phase = 0;
    typename Prob::State st;
    Prob::init(p, st);
    for (int j = 0; j < njobs; ++j) {
      if (kChecks && !Prob::job_ok(p, Prob::job(p, cluster, nclusters, j))) continue;
      if (!warp_wait_cluster(&tfull[acc], acc_phase, abort, lane)) {
        if (lane == 0) report_timeout(abort, flags);
        break;
      }
      tc_fence_after_sync();
      const TileJob tj = Prob::job(p, cluster, nclusters, j);
      for (int h = half; h < 2; h += EPI_WARPS / 4) {  // the 128-column halves this warp owns
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(acc * BN + h * EPI_COLS);
        Prob::epilogue(p, st, tj, ctx, tj.mb * P_TILE_M + static_cast<int>(rank) * 128, tj.nb * BN + h * EPI_COLS,
                       taddr);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncwarp();        // the cluster barrier below is warp-aligned
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still signal it
  tc_fence_after_sync();
  if (warp == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace lce
