// Kernels of the fused LM-head linear + cross-entropy: the three tcgen05
// GEMM instantiations with their epilogues, and the small per-row kernels.
//
// Where the arithmetic comes from:
//   * token-level cross-entropy over the vocabulary of H W^T, its d_input and
//     d_weight ("XTuner on Ascend 910C: Qwen3.5-2B training optimisation",
//     section 3.1.4, Fig. 12: the fused backward emits d_weight / d_input and
//     never stores the full d_logits);
//   * the streaming max / sum-exp over vocabulary tiles ("MindSpeed fusion
//     optimisation: principles and practice", section 3.2: blockwise softmax
//     without materialising the full score matrix), applied here along the
//     vocabulary instead of the attention keys.
#include <math.h>

#include "lce_gemm.cuh"
#include "lce_internal.h"

namespace lce {

constexpr float kLog2e = 1.4426950408889634f;

// ----------------------------------------------------------------------------
// Logits epilogue. An epilogue warp owns 32 rows x 128 columns of the 128 x 256
// tile (one thread = one row); results leave through the warp's swizzled
// staging tile as TMA stores of 32 rows x 64 bf16.
//   FWD_STATS:   per (row, 128-column half tile) max m and sum of exp(z - m)
//                over the in-vocabulary columns, plus the label's logit.
//   FWD_STATS_P: the exp tile P = bf16(exp(z - ref_row)) for the backward,
//                where ref_row is the row's maximum over the first 128 words,
//                and per (row, half tile) the pair (ref_row, sum of those
//                exps), plus the label's logit; sets the chunk's guard word if
//                a 32-column sum exceeds kRefGuardSum (range protection: the
//                chunk's statistics and gradient tile are then recomputed
//                exactly by conditional launches).
//   FWD_STATS_PX: FWD_STATS's exact partials and FWD_STATS_P's exp tile (two
//                exps per element), guard as FWD_STATS_P but on the tile only:
//                the statistics stay exact (vocabulary shards exchange them
//                before the tile's scale is known).
//   FWD_REF:     ref_row (launched for the first tile only; the warps holding
//                columns 128..255 do nothing).
//   FWD_GRAD:    the gradient tile exp(z - lse) - [v = y] in bf16 for valid
//                rows, zeros for ignored rows.
// Columns past the vocabulary are masked to -inf (zero logits are not neutral
// in a softmax); stores past the vocabulary are dropped by TMA.
// ----------------------------------------------------------------------------
// The label's logit if it lies in these 32 columns (yo = its column within
// them). The branch is taken for about one group in 4700, so the unrolled
// compares cost almost nothing.
__device__ __forceinline__ void take_label(const float (&v)[32], int yo, float& zt, bool& have_t) {
  if (yo >= 0 && yo < 32) {
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (c == yo) {
        zt = v[c];
        have_t = true;
      }
  }
}

struct FwdEpi {
  using Params = FwdParams;
  struct State {};
  static __device__ __forceinline__ bool skip(const Params& p) { return p.only_if != nullptr && *p.only_if == 0; }
  static __device__ __forceinline__ void init(const Params&, State&) {}

  static __device__ __forceinline__ void tile(const Params& p, State&, const EpiCtx& ctx, int m0, int col0,
                                              uint32_t taddr) {
    const int lane = ctx.lane;
    const int r = m0 + ctx.row0 + lane;
    const bool live = r < p.rows;
    const long long yr = live ? static_cast<long long>(p.y[r]) : p.ignore_index;
    const bool valid = live && yr != p.ignore_index && yr >= 0 && yr < p.V_total;
    // column of the label in this half tile (outside [0, 128) when the label is elsewhere)
    const long long yc = valid ? yr - p.y_offset - col0 : -1;
    const int ycol = (yc >= 0 && yc < EPI_COLS) ? static_cast<int>(yc) : -1;
    const int vlim = p.V - col0;  // columns >= vlim are past the vocabulary (warp-uniform)
    const int part = col0 / EPI_COLS;

    if (p.mode == FWD_REF && col0 >= EPI_COLS) return;
    if (vlim <= 0) {  // this half tile lies entirely past the vocabulary
      if (live && p.mode != FWD_REF && p.mode != FWD_GRAD && in_bounds(part, p.nparts, p.flags))
        p.partials[static_cast<long long>(r) * p.nparts + part] = make_float2(-INFINITY, 0.f);
      return;
    }
    const bool grad = p.mode == FWD_GRAD;
    const bool stats = p.mode == FWD_STATS || p.mode == FWD_STATS_P || p.mode == FWD_STATS_PX;
    const bool store = p.mode == FWD_STATS_P || p.mode == FWD_STATS_PX || grad;
    const bool by_ref = p.mode == FWD_STATS_P || p.mode == FWD_STATS_PX;  // the tile is exp(z - ref)
    const float refv = !live ? 0.f : (grad ? p.lse[r] : (by_ref ? p.ref[r] : 0.f));
    const float rb = refv * kLog2e;
    const float gmask = (grad && !valid) ? 0.f : 1.f;   // gradient rows of ignored tokens are zero

    // A store box never starts past the output's extent (rows or vocabulary).
    const bool rows_in = m0 + ctx.row0 < p.rows;
    float m = -INFINITY, s = 0.f, zt = 0.f;
    bool have_t = false, over = false;
#pragma unroll 1
    for (int u = 0; u < EPI_COLS / 64; ++u) {
      if (u * 64 >= vlim) break;  // the rest of this half tile is past the vocabulary
      if (store) stage_acquire(ctx);
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int c0 = u * 64 + hh * 32;
        float v[32];
        tmem_ld_32x32b_x32(taddr + c0, v);
        if (vlim < c0 + 32) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c0 + c >= vlim) v[c] = -INFINITY;
        }
        if (p.mode == FWD_STATS_P) {
          // One exp per element: the exp tile's values exp(z - ref) also give the row's sum
          // (partials against ref instead of the tile maximum). A 32-column sum above
          // kRefGuardSum sets the guard (the chunk is then redone exactly).
          float s2 = 0.f;
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float e0 = ex2_approx(fmaf(v[c], kLog2e, -rb));
            const float e1 = ex2_approx(fmaf(v[c + 1], kLog2e, -rb));
            s2 += e0;
            s2 += e1;
            pk[c / 2] = pack_bf16x2(e0, e1);
          }
          s += s2;
          m = refv;
          over |= !(s2 <= kRefGuardSum);
          take_label(v, ycol - c0, zt, have_t);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(ctx.stage + stage_off(lane, hh * 4 + q)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          continue;
        }
        if (stats || p.mode == FWD_REF) {
          float cm = v[0];
#pragma unroll
          for (int c = 1; c < 32; ++c) cm = fmaxf(cm, v[c]);
          if (p.mode == FWD_REF) {
            m = fmaxf(m, cm);
          } else {
            if (cm > m) {
              s *= ex2_approx((m - cm) * kLog2e);
              m = cm;
            }
            const float mb = m * kLog2e;
            float s2 = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) s2 += ex2_approx(fmaf(v[c], kLog2e, -mb));
            s += s2;
            take_label(v, ycol - c0, zt, have_t);
          }
        }
        if (store) {
          uint32_t pk[16];
          float s3 = 0.f;
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float e0 = ex2_approx(fmaf(v[c], kLog2e, -rb));
            float e1 = ex2_approx(fmaf(v[c + 1], kLog2e, -rb));
            if (grad) {
              e0 = (e0 - (c0 + c == ycol ? 1.f : 0.f)) * gmask;
              e1 = (e1 - (c0 + c + 1 == ycol ? 1.f : 0.f)) * gmask;
            }
            s3 += e0;
            s3 += e1;
            pk[c / 2] = pack_bf16x2(e0, e1);
          }
          if (p.mode == FWD_STATS_PX) over |= !(s3 <= kRefGuardSum);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(ctx.stage + stage_off(lane, hh * 4 + q)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (store && rows_in) stage_release(ctx, col0 + u * 64, m0 + ctx.row0, false);
    }
    if (!live) return;
    if (p.mode == FWD_REF) {
      p.ref[r] = m;
      return;
    }
    if (stats && in_bounds(part, p.nparts, p.flags)) {
      p.partials[static_cast<long long>(r) * p.nparts + part] = make_float2(m, s);
      if (have_t) p.ztgt[r] = zt;
      if (by_ref && over) *p.guard = 1;
    }
  }
};

// dH tile: bf16(acc * g/n [* per-row factor]), stored by TMA into the chunk's dH
// rows (fp32 instead when the result is a partial sum over vocabulary shards).
struct DhEpi {
  using Params = DhParams;
  struct State {
    float g;
  };
  static __device__ __forceinline__ bool skip(const Params&) { return false; }
  static __device__ __forceinline__ void init(const Params& p, State& st) { st.g = p.st->gscale; }

  // One 128-column half (col0) of a part tile: store this warp's fp32 sums of
  // the part (32 rows x 128 columns, lane-contiguous: slot[group][lane]). After
  // the second half the warp counts its arrival; the warp that brings the count
  // to `parts` adds the parts' sums in part order and writes the 256 columns of
  // the tile (so the order of the additions never depends on which part ends
  // last). No warp waits for another.
  // When a block's parts run back to back on one cluster (block_major), the
  // same thread handles every part of its rows, in part order: the last part is
  // known in advance, keeps its own sum in TMEM (no store) and needs no count,
  // and the earlier parts' sums are this thread's own earlier stores. The
  // additions are the same, in the same order.
  static __device__ __forceinline__ void part_half(const Params& p, const EpiCtx& ctx, int m0, int col0,
                                                   uint32_t taddr, int part, int tile, float f) {
    const int lane = ctx.lane;
    const int rank = (m0 % P_TILE_M) / 128;
    const int q = ctx.row0 / 32;
    const int h = (col0 % BN) / EPI_COLS;
    const long long slice = (static_cast<long long>(tile) * 2 + rank) * 4 + q;  // this warp's 32 rows of the tile
    if (!in_bounds(slice, p.part_slices, ctx.flags) || !in_bounds(part, p.parts, ctx.flags)) return;
    auto slot = [&](int s) { return p.part_buf + ((slice * p.parts + s) * 64) * 32; };
    const bool last_in_order = p.block_major && part == p.parts - 1;
    if (!last_in_order) {
      float4* mine = slot(part);
#pragma unroll 1
      for (int u = 0; u < EPI_COLS / 32; ++u) {
        float v[32];
        tmem_ld_32x32b_x32(taddr + u * 32, v);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mine[(h * 32 + u * 8 + j) * 32 + lane] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
    }
    if (h == 0) return;
    if (p.block_major) {
      if (!last_in_order) return;
    } else {
      // all 256 columns of this part are stored: count the arrival (release), and
      // the last of the parts finishes the tile (acquire)
      __threadfence();
      __syncwarp();
      int prior = 0;
      if (lane == 0) {
        __threadfence();
        prior = atomicAdd(p.part_cnt + slice, 1);
      }
      prior = __shfl_sync(0xffffffffu, prior, 0);
      if (prior != p.parts - 1) return;
      __threadfence();
    }
    const int tcol0 = col0 - EPI_COLS;                              // first column of the tile
    const uint32_t ttile = taddr - static_cast<uint32_t>(EPI_COLS);  // its TMEM columns
    const int from_mem = last_in_order ? p.parts - 1 : p.parts;     // parts whose sums are in memory
    const int groups = p.f32_out ? BN / 32 : BN / 64;
#pragma unroll 1
    for (int u = 0; u < groups; ++u) {
      const int width = p.f32_out ? 32 : 64;
      if (tcol0 + u * width >= p.N) break;
      stage_acquire(ctx);
#pragma unroll 1
      for (int hh = 0; hh < width / 32; ++hh) {
        const int g0 = (u * width + hh * 32) / 4;  // first 4-column group of these 32 columns
        float v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 a = __ldcg(slot(0) + (g0 + j) * 32 + lane);
          v[4 * j] = a.x;
          v[4 * j + 1] = a.y;
          v[4 * j + 2] = a.z;
          v[4 * j + 3] = a.w;
        }
#pragma unroll 1
        for (int s = 1; s < from_mem; ++s) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 a = __ldcg(slot(s) + (g0 + j) * 32 + lane);
            v[4 * j] += a.x;
            v[4 * j + 1] += a.y;
            v[4 * j + 2] += a.z;
            v[4 * j + 3] += a.w;
          }
        }
        if (last_in_order) {  // the last part's own sum, still in TMEM, added last
          float w[32];
          tmem_ld_32x32b_x32(ttile + static_cast<uint32_t>(u * width + hh * 32), w);
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] += w[c];
        }
        if (p.f32_out) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            *reinterpret_cast<float4*>(ctx.stage + stage_off(lane, q4)) =
                make_float4(v[4 * q4] * f, v[4 * q4 + 1] * f, v[4 * q4 + 2] * f, v[4 * q4 + 3] * f);
        } else {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(v[8 * q4 + 0] * f, v[8 * q4 + 1] * f);
            w.y = pack_bf16x2(v[8 * q4 + 2] * f, v[8 * q4 + 3] * f);
            w.z = pack_bf16x2(v[8 * q4 + 4] * f, v[8 * q4 + 5] * f);
            w.w = pack_bf16x2(v[8 * q4 + 6] * f, v[8 * q4 + 7] * f);
            *reinterpret_cast<uint4*>(ctx.stage + stage_off(lane, hh * 4 + q4)) = w;
          }
        }
      }
      stage_release(ctx, tcol0 + u * width, m0 + ctx.row0, false);
    }
    if (!p.block_major && lane == 0) p.part_cnt[slice] = 0;  // ready for the next launch
  }

  static __device__ __forceinline__ void tile(const Params& p, State& st, const EpiCtx& ctx, int m0, int col0,
                                              uint32_t taddr, int part, int tile_index) {
    const int r = m0 + ctx.row0 + ctx.lane;
    if (m0 + ctx.row0 >= p.rows) return;  // all 32 rows of this warp are past the chunk
    float f = st.g;
    if (r < p.rows && p.rowscale != nullptr) f *= p.rowscale[r];
    if (p.parts > 1) {
      part_half(p, ctx, m0, col0, taddr, part, tile_index, f);
      return;
    }
    if (p.f32_out) {  // fp32 tiles of 32 columns, like the dW epilogue
#pragma unroll 1
      for (int u = 0; u < EPI_COLS / 32; ++u) {
        if (col0 + u * 32 >= p.N) break;
        stage_acquire(ctx);
        float v[32];
        tmem_ld_32x32b_x32(taddr + u * 32, v);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(ctx.stage + stage_off(ctx.lane, q)) =
              make_float4(v[4 * q] * f, v[4 * q + 1] * f, v[4 * q + 2] * f, v[4 * q + 3] * f);
        stage_release(ctx, col0 + u * 32, m0 + ctx.row0, false);
      }
      return;
    }
#pragma unroll 1
    for (int u = 0; u < EPI_COLS / 64; ++u) {
      if (col0 + u * 64 >= p.N) break;
      stage_acquire(ctx);
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        tmem_ld_32x32b_x32(taddr + u * 64 + hh * 32, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16x2(v[8 * q + 0] * f, v[8 * q + 1] * f);
          w.y = pack_bf16x2(v[8 * q + 2] * f, v[8 * q + 3] * f);
          w.z = pack_bf16x2(v[8 * q + 4] * f, v[8 * q + 5] * f);
          w.w = pack_bf16x2(v[8 * q + 6] * f, v[8 * q + 7] * f);
          *reinterpret_cast<uint4*>(ctx.stage + stage_off(ctx.lane, hh * 4 + q)) = w;
        }
      }
      stage_release(ctx, col0 + u * 64, m0 + ctx.row0, false);
    }
  }
};

// dW tile: fp32 acc * g/n, stored (first chunk) or added (TMA reduce-add in L2)
// into the vocabulary rows of dW.
struct DwEpi {
  using Params = DwParams;
  struct State {
    float g;
  };
  static __device__ __forceinline__ bool skip(const Params&) { return false; }
  static __device__ __forceinline__ void init(const Params& p, State& st) { st.g = p.st->gscale; }

  static __device__ __forceinline__ void tile(const Params& p, State& st, const EpiCtx& ctx, int m0, int col0,
                                              uint32_t taddr) {
    const float f = st.g;
    if (m0 + ctx.row0 >= p.rows) return;  // all 32 rows of this warp are past the vocabulary
#pragma unroll 1
    for (int u = 0; u < EPI_COLS / 32; ++u) {
      if (col0 + u * 32 >= p.N) break;
      stage_acquire(ctx);
      float v[32];
      tmem_ld_32x32b_x32(taddr + u * 32, v);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(ctx.stage + stage_off(ctx.lane, q)) =
            make_float4(v[4 * q] * f, v[4 * q + 1] * f, v[4 * q + 2] * f, v[4 * q + 3] * f);
      stage_release(ctx, col0 + u * 32, m0 + ctx.row0, p.accumulate != 0);
    }
  }
};

// ----------------------------------------------------------------------------
// Label scan: n = number of labels in [0, V) that are not ignore_index, the
// range-error bit, and the scales g/n and 1/n. One block, fixed-order sums.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_prepare(const int64_t* __restrict__ y, long long N, int V,
                                                  long long ignore_index, int reduction, long long n_override,
                                                  const float* grad_loss, DevStatus* st, int* guards, int nguards,
                                                  int* part_cnt, int ncnt) {
  grid_dep_wait();
  grid_dep_launch();
  for (int i = threadIdx.x; i < nguards; i += blockDim.x) guards[i] = 0;
  for (int i = threadIdx.x; i < ncnt; i += blockDim.x) part_cnt[i] = 0;
  __shared__ long long s_cnt[32];
  __shared__ int s_bad[32];
  long long cnt = 0;
  int bad = 0;
  for (long long i = threadIdx.x; i < N; i += blockDim.x) {
    const long long v = y[i];
    if (v != ignore_index) {
      if (v >= 0 && v < V)
        ++cnt;
      else
        bad = 1;
    }
  }
  for (int off = 16; off > 0; off >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    bad |= __shfl_xor_sync(0xffffffffu, bad, off);
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_cnt[w] = cnt;
    s_bad[w] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long total = 0;
    int anybad = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) {
      total += s_cnt[i];
      anybad |= s_bad[i];
    }
    const long long n = n_override >= 0 ? n_override : total;
    const float g = grad_loss != nullptr ? *grad_loss : 1.f;
    st->flags = anybad ? kFlagLabelRange : 0;
    st->n_counted = total;
    st->n_valid = n;
    if (reduction == 0) {
      st->gscale = n > 0 ? g / static_cast<float>(n) : 0.f;
      st->lscale = n > 0 ? 1.0 / static_cast<double>(n) : 0.0;
    } else {
      st->gscale = g;
      st->lscale = 1.0;
    }
  }
}

// Merge two (max, sum-exp) pairs: m' = max, s' = s1 e^{m1-m'} + s2 e^{m2-m'}.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  const float e1 = (m == M) ? 1.f : exp2f((m - M) * kLog2e);
  const float e2 = (m2 == M) ? 1.f : exp2f((m2 - M) * kLog2e);
  s = s * e1 + s2 * e2;
  m = M;
}

// A lane's running (max, sum-exp) over its row's partials t = lane, lane + 32,
// lane + 64, ... in that order. Eight loads are issued before their merges, so
// a warp waits for memory once per eight partials instead of once per partial;
// entries past T merge as (-inf, 0), which leaves (m, s) exactly unchanged, so
// the result is that of the plain one-at-a-time loop bit for bit.
__device__ __forceinline__ void lane_partials(const float2* __restrict__ pr, int T, int lane, float& m, float& s) {
  constexpr int kBatch = 8;
  for (int t0 = lane; t0 < T; t0 += 32 * kBatch) {
    float2 q[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int t = t0 + 32 * k;
      q[k] = t < T ? pr[t] : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) merge_ms(m, s, q[k].x, q[k].y);
  }
}

// One warp per row: combine the row's vocabulary-tile partials in a fixed
// order, lse = m + log s, loss_i = lse - z_y for valid rows (else 0).
__global__ void __launch_bounds__(256) k_combine(const float2* __restrict__ partials, int T, int rows,
                                                 const float* __restrict__ ztgt, const int64_t* __restrict__ y,
                                                 int V, long long ignore_index, float* __restrict__ lse,
                                                 float* __restrict__ loss_i) {
  grid_dep_wait();
  grid_dep_launch();
  const int r = static_cast<int>((blockIdx.x * static_cast<unsigned>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float m = -INFINITY, s = 0.f;
  const float2* pr = partials + static_cast<long long>(r) * T;
  lane_partials(pr, T, lane, m, s);
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    merge_ms(m, s, m2, s2);
  }
  if (lane == 0) {
    const float l = m + logf(s);
    lse[r] = l;
    const long long yr = y[r];
    const bool valid = yr != ignore_index && yr >= 0 && yr < V;
    loss_i[r] = valid ? l - ztgt[r] : 0.f;
  }
}

// k_combine, plus what the backward needs from the exp tile P = exp(z - ref):
// alpha_i = exp(ref_i - lse_i) for valid rows (so that alpha_i P_iv is the
// softmax) and the label entry rewritten as exp(z_y - ref) - exp(lse - ref)
// (so that alpha_i P_iy = p_iy - 1). Ignored rows get alpha = 0. If the
// chunk's guard tripped, the exact gradient tile replaces P and alpha is 1.
__global__ void __launch_bounds__(256) k_combine_exp(const float2* __restrict__ partials, int T, int rows,
                                                     const float* __restrict__ ztgt, const int64_t* __restrict__ y,
                                                     int V, long long ignore_index, const float* __restrict__ ref,
                                                     const int* __restrict__ guard, float* __restrict__ lse,
                                                     float* __restrict__ loss_i, float* __restrict__ alpha,
                                                     __nv_bfloat16* __restrict__ P, long long ldp,
                                                     const uint4* __restrict__ H, int groups_per_row,
                                                     uint4* __restrict__ Ht, const int* __restrict__ only_if,
                                                     int* flags) {
  grid_dep_wait();
  grid_dep_launch();
  if (only_if != nullptr && *only_if == 0) return;  // conditional launch whose condition is false
  const int r = static_cast<int>((blockIdx.x * static_cast<unsigned>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  // the row's scalars, loaded before the partials so that their latency overlaps the merge
  const long long yr = y[r];
  const float zt = ztgt[r], rf = ref[r];
  const int gd = *guard;
  float m = -INFINITY, s = 0.f;
  const float2* pr = partials + static_cast<long long>(r) * T;
  lane_partials(pr, T, lane, m, s);
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    merge_ms(m, s, m2, s2);
  }
  float a = 0.f;  // alpha_i, decided by lane 0
  if (lane == 0) {
    const float l = m + logf(s);
    lse[r] = l;
    const bool valid = yr != ignore_index && yr >= 0 && yr < V;
    loss_i[r] = valid ? l - zt : 0.f;
    if (valid) {
      if (gd != 0) {
        a = 1.f;
      } else {
        a = exp2f((rf - l) * kLog2e);
        const float py = exp2f((zt - rf) * kLog2e) - exp2f((l - rf) * kLog2e);
        if (in_bounds(yr, ldp, flags)) P[static_cast<long long>(r) * ldp + yr] = __float2bfloat16_rn(py);
      }
    }
    alpha[r] = a;
  }
  // Ht_i = bf16(alpha_i H_i): the B operand of the dW GEMM (the whole warp, 16 bytes per lane)
  a = __shfl_sync(0xffffffffu, a, 0);
  const uint4* hr = H + static_cast<long long>(r) * groups_per_row;
  uint4* tr = Ht + static_cast<long long>(r) * groups_per_row;
#pragma unroll 4
  for (int g = lane; g < groups_per_row; g += 32) {
    const uint4 h = hr[g];
    const uint32_t w[4] = {h.x, h.y, h.z, h.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = pack_bf16x2(__uint_as_float(w[q] << 16) * a, __uint_as_float(w[q] & 0xffff0000u) * a);
    tr[g] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Ht_r = bf16(alpha_r * H_r): the per-row softmax scale moved onto the dW
// GEMM's B operand (dW = P^T Ht). Eight bf16 per thread; d % 8 == 0.

// One warp per row: this vocabulary shard's (max, sum-exp) over its columns,
// its logit of the label if the label lies in the shard, and whether it does.
__global__ void __launch_bounds__(256) k_shard_stats(const float2* __restrict__ partials, int T, int rows,
                                                     const float* __restrict__ ztgt, const int64_t* __restrict__ y,
                                                     long long y_offset, int V_shard, int V_total,
                                                     long long ignore_index, float4* __restrict__ stats) {
  grid_dep_wait();
  grid_dep_launch();
  const int r = static_cast<int>((blockIdx.x * static_cast<unsigned>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float m = -INFINITY, s = 0.f;
  const float2* pr = partials + static_cast<long long>(r) * T;
  lane_partials(pr, T, lane, m, s);
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    merge_ms(m, s, m2, s2);
  }
  if (lane == 0) {
    const long long yr = y[r];
    const bool valid = yr != ignore_index && yr >= 0 && yr < V_total;
    const long long col = yr - y_offset;
    const bool here = valid && col >= 0 && col < V_shard;
    stats[r] = make_float4(m, s, here ? ztgt[r] : 0.f, here ? 1.f : 0.f);
  }
}

// Merge R shards' row statistics in shard order: M = max_r m_r,
// S = sum_r s_r e^{m_r - M}, lse = M + log S, z_y from the shard that holds
// the label; loss_i = lse - z_y for valid rows. One thread per row.
__global__ void __launch_bounds__(256) k_shard_merge(const float4* __restrict__ stats, int R, long long N,
                                                     const int64_t* __restrict__ y, int V_total,
                                                     long long ignore_index, float* __restrict__ lse,
                                                     float* __restrict__ loss_i) {
  grid_dep_wait();
  grid_dep_launch();
  const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (i >= N) return;
  float M = -INFINITY;
  for (int r = 0; r < R; ++r) M = fmaxf(M, stats[r * N + i].x);
  float S = 0.f, zt = 0.f;
  for (int r = 0; r < R; ++r) {
    const float4 q = stats[r * N + i];
    if (q.y > 0.f) S += q.y * exp2f((q.x - M) * kLog2e);
    zt += q.w > 0.f ? q.z : 0.f;
  }
  const float l = M + logf(S);
  lse[i] = l;
  const long long yr = y[i];
  const bool valid = yr != ignore_index && yr >= 0 && yr < V_total;
  loss_i[i] = valid ? l - zt : 0.f;
}

// Stored-tile vocabulary-parallel backward, first pass, one thread per chunk
// row: the merge of k_shard_merge over the R shards' statistics (stats
// [R, rows, 4]) -> lse. A valid row whose label lies in this shard and whose
// lse exceeds the shard's row reference by more than kRefGuardLogit sets the
// chunk's guard: its label entry exp(z_y - ref) - exp(lse - ref) would leave
// the fp32 range (and alpha = exp(ref - lse) underflow), so the chunk takes
// the exact gradient tile instead.
__global__ void __launch_bounds__(256) k_vshard_lse(const float4* __restrict__ stats, int R, int rows,
                                                    const int64_t* __restrict__ y, long long y_offset, int V_shard,
                                                    int V_total, long long ignore_index, const float* __restrict__ ref,
                                                    int* __restrict__ guard, float* __restrict__ lse) {
  grid_dep_wait();
  grid_dep_launch();
  const int r = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
  if (r >= rows) return;
  float M = -INFINITY;
  for (int k = 0; k < R; ++k) M = fmaxf(M, stats[static_cast<long long>(k) * rows + r].x);
  float S = 0.f;
  for (int k = 0; k < R; ++k) {
    const float4 q = stats[static_cast<long long>(k) * rows + r];
    if (q.y > 0.f) S += q.y * exp2f((q.x - M) * kLog2e);
  }
  const float l = M + logf(S);
  lse[r] = l;
  const long long yr = y[r];
  const bool valid = yr != ignore_index && yr >= 0 && yr < V_total;
  const long long col = yr - y_offset;
  if (valid && col >= 0 && col < V_shard && !(l - ref[r] <= kRefGuardLogit)) *guard = 1;
}

// Second pass, one warp per chunk row: alpha_i = exp(ref_i - lse_i) scales
// this shard's exp tile exp(z - ref) into softmax probabilities (1 if the
// chunk's guard is set, the tile then being the exact gradient; 0 for ignored
// rows); the label's entry of the tile becomes exp(z_y - ref) - exp(lse - ref)
// when the label lies in this shard, so that alpha P is softmax - onehot
// there; Ht_i = bf16(alpha_i H_i).
__global__ void __launch_bounds__(256) k_vshard_scale(const float4* __restrict__ stats, int R, int rows,
                                                      const int64_t* __restrict__ y, long long y_offset, int V_shard,
                                                      int V_total, long long ignore_index, const float* __restrict__ ref,
                                                      const int* __restrict__ guard, const float* __restrict__ lse,
                                                      float* __restrict__ alpha, __nv_bfloat16* __restrict__ P,
                                                      long long ldp, const uint4* __restrict__ H, int groups_per_row,
                                                      uint4* __restrict__ Ht, int* flags) {
  grid_dep_wait();
  grid_dep_launch();
  const int r = static_cast<int>((blockIdx.x * static_cast<unsigned>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float a = 0.f;
  if (lane == 0) {
    const long long yr = y[r];
    const bool valid = yr != ignore_index && yr >= 0 && yr < V_total;
    if (valid) {
      if (*guard != 0) {
        a = 1.f;
      } else {
        const float l = lse[r], rf = ref[r];
        a = exp2f((rf - l) * kLog2e);
        const long long col = yr - y_offset;
        if (col >= 0 && col < V_shard && in_bounds(col, ldp, flags)) {
          float zt = 0.f;  // the label's logit, from the shard that holds it (this one)
          for (int k = 0; k < R; ++k) {
            const float4 q = stats[static_cast<long long>(k) * rows + r];
            zt += q.w > 0.f ? q.z : 0.f;
          }
          P[static_cast<long long>(r) * ldp + col] =
              __float2bfloat16_rn(exp2f((zt - rf) * kLog2e) - exp2f((l - rf) * kLog2e));
        }
      }
    }
    alpha[r] = a;
  }
  a = __shfl_sync(0xffffffffu, a, 0);
  const uint4* hr = H + static_cast<long long>(r) * groups_per_row;
  uint4* tr = Ht + static_cast<long long>(r) * groups_per_row;
#pragma unroll 4
  for (int g = lane; g < groups_per_row; g += 32) {
    const uint4 h = hr[g];
    const uint32_t w[4] = {h.x, h.y, h.z, h.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = pack_bf16x2(__uint_as_float(w[q] << 16) * a, __uint_as_float(w[q] & 0xffff0000u) * a);
    tr[g] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// x *= g in place for bf16 (8 per thread) and fp32 (4 per thread) arrays;
// nothing is read or written when g == 1.
__global__ void __launch_bounds__(256) k_scale(uint4* __restrict__ bf, long long nbf8, float4* __restrict__ f32,
                                               long long nf4, const float* __restrict__ gptr) {
  grid_dep_wait();
  grid_dep_launch();
  const float g = *gptr;
  if (g == 1.f) return;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nbf8; i += stride) {
    const uint4 v = bf[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = pack_bf16x2(__uint_as_float(w[q] << 16) * g, __uint_as_float(w[q] & 0xffff0000u) * g);
    bf[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nf4; i += stride) {
    float4 v = f32[i];
    v.x *= g;
    v.y *= g;
    v.z *= g;
    v.w *= g;
    f32[i] = v;
  }
}

// loss = (sum_i loss_i) * lscale, fp64 accumulation in a fixed order.
__global__ void __launch_bounds__(1024) k_finalize(const float* __restrict__ loss_i, long long N,
                                                   const DevStatus* st, float* loss) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ double red[1024];
  double acc = 0.0;
  for (long long i = threadIdx.x; i < N; i += blockDim.x) acc += static_cast<double>(loss_i[i]);
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = static_cast<float>(red[0] * st->lscale);
}

// ----------------------------------------------------------------------------
// Launch wrappers
// ----------------------------------------------------------------------------

// ----------------------------------------------------------------------------
// Problems for the pair kernel
// ----------------------------------------------------------------------------
enum : int { KIND_LOGITS = 0, KIND_DH = 1, KIND_DW = 2 };

// This CTA's half of a k-block: 128 rows of a K-major operand (one box), or
// 128 columns of an MN-major operand (two 64-wide boxes).
__device__ __forceinline__ void load_k_major(uint8_t* dst, const CUtensorMap* m, uint32_t bar, int row0, int k0) {
  tma_load_2d_pair(dst, m, bar, k0, row0);
}
__device__ __forceinline__ void load_mn_major(uint8_t* dst, const CUtensorMap* m, uint32_t bar, int mn0, int k0) {
  tma_load_2d_pair(dst, m, bar, mn0, k0);
  tma_load_2d_pair(dst + MN_SLAB_BYTES, m, bar, mn0 + 64, k0);
}

// Logits of a chunk: z = H_c W^T (both operands K-major) with the FwdEpi
// epilogue. Tiles walk M first, so the pairs running at once share W tiles.
struct LogitsProb {
  struct Params {
    CUtensorMap a, b, c;
    int m_tiles, n_tiles, k_blocks;
    int no_loads;   // timeout test only
    int* flags;
    FwdParams ep;
  };
  using State = FwdEpi::State;
  static __device__ __forceinline__ bool skip(const Params& p) { return FwdEpi::skip(p.ep); }
  static __device__ __forceinline__ bool no_loads(const Params& p) { return p.no_loads != 0; }
  static __device__ __forceinline__ int* flags(const Params& p) { return p.flags; }
  static __device__ __forceinline__ int num_jobs(const Params& p, int c, int P) {
    const int tiles = p.m_tiles * p.n_tiles;
    return c < tiles ? (tiles - 1 - c) / P + 1 : 0;
  }
  static __device__ __forceinline__ TileJob job(const Params& p, int c, int P, int j) {
    const int t = c + j * P;
    return TileJob{KIND_LOGITS, t % p.m_tiles, t / p.m_tiles, p.k_blocks, 0, 0};
  }
  static __device__ __forceinline__ bool job_ok(const Params& p, const TileJob& tj) {
    return tj.kind == KIND_LOGITS && tj.mb >= 0 && tj.mb < p.m_tiles && tj.nb >= 0 && tj.nb < p.n_tiles &&
           tj.kb0 == 0 && tj.k_blocks == p.k_blocks && tj.k_blocks > 0;
  }
  static __device__ __forceinline__ void load(const Params& p, int, uint8_t* a, uint8_t* b, uint32_t bar, int m0,
                                              int n0, int k0) {
    load_k_major(a, &p.a, bar, m0, k0);
    load_k_major(b, &p.b, bar, n0, k0);
  }
  static __device__ __forceinline__ uint64_t a_desc(int, uint32_t addr, int k) { return desc_k_major(addr, k); }
  static __device__ __forceinline__ uint64_t b_desc(int, uint32_t addr, int k) { return desc_k_major(addr, k); }
  static __device__ __forceinline__ uint32_t idesc(int) { return idesc_bf16_f32(P_TILE_M, BN, false, false); }
  static __device__ __forceinline__ void init(const Params& p, State& st) { FwdEpi::init(p.ep, st); }
  static __device__ __forceinline__ void epilogue(const Params& p, State& st, const TileJob&, EpiCtx ctx, int m0,
                                                  int col0, uint32_t taddr) {
    ctx.out = &p.c;
    FwdEpi::tile(p.ep, st, ctx, m0, col0, taddr);
  }
};

// The backward of a chunk in one launch: dH tiles (dH_c = G_c W: A = G_c
// K-major, B = W N-major) and dW tiles (dW += G_c^T B: A = G_c read M-major,
// B = Ht or H_c N-major). dH tiles are few and long (K = V), dW tiles many and
// short (K = C). The static schedule gives every cluster, in this order:
//   1. w_phase1 / P dW tiles dealt round-robin to all clusters,
//   2. its dH tiles, dealt round-robin,
//   3. the remaining dW tiles, dealt round-robin to the clusters that hold
//      one dH tile fewer,
// so every cluster ends with about the same number of k-blocks, and the tiles
// running at the same time are neighbours in their lists (they share operand
// rows in L2): all clusters start phase 1 together, and the clusters of phase
// 3 all enter it after the same number of dH tiles. Tiles walk N first, so the
// pairs running at once share the A rows.
struct BwdProb {
  struct Params {
    CUtensorMap ah, bh, ch, aw, bw, cw;
    int h_m, h_n, h_k;   // dH: 256-row blocks of the chunk, 256-column blocks of d, k-blocks of V
    int h_parts, h_kpart;  // dH tiles per (row block, column block): vocabulary parts of h_kpart k-blocks
    int w_m, w_n, w_k;   // dW: 256-row blocks of V, 256-column blocks of d, k-blocks of the chunk
    int w_t0, w_tiles;   // this launch's dW tiles: [w_t0, w_t0 + w_tiles) in (row block, column block) order
    int w_phase1;        // dW tiles dealt round-robin to every cluster (a multiple of the cluster count)
    int dh_mfast;        // dH tiles walk row blocks first (when W is larger than the chunk's exp tile)
    int odd_dh_first;    // odd clusters take their dH tiles before their first-phase dW tiles
    int h_group;         // dH part tiles dealt together: 1 (each part on its own), or h_parts (the
                         // parts of one 256 x 256 block back to back on one cluster)
    int* flags;
    DhParams h;
    DwParams w;
  };
  struct State {
    DhEpi::State h;
    DwEpi::State w;
  };
  struct Sched {
    int hcount, q1, li, nlight, count2;
  };
  // Position of cluster c in the dealing order. Normally c itself; when odd clusters take their
  // dH tiles first, the even clusters come first and then the odd ones, so that the tiles dealt
  // next to each other (which share operand blocks: the dH tiles of one W block, the dW tiles of
  // one exp-tile block) go to clusters of the same parity and so run at the same time.
  static __device__ __forceinline__ int deal_rank(const Params& p, int c, int P) {
    if (!p.odd_dh_first) return c;
    return (c & 1) ? (P + 1) / 2 + c / 2 : c / 2;
  }
  static __device__ __forceinline__ Sched sched(const Params& p, int c, int P) {
    Sched s;
    c = deal_rank(p, c, P);
    const int nH = p.h_m * p.h_n * p.h_parts / p.h_group, nW = p.w_tiles;  // dH units dealt
    s.hcount = (c < nH ? (nH - 1 - c) / P + 1 : 0) * p.h_group;
    const int r = nH % P;  // clusters c < r hold one dH unit more
    s.q1 = p.w_phase1 / P;
    s.nlight = r == 0 ? P : P - r;
    s.li = r == 0 ? c : c - r;
    const int rem = nW - p.w_phase1;
    s.count2 = (s.li >= 0 && s.li < rem) ? (rem - 1 - s.li) / s.nlight + 1 : 0;
    return s;
  }
  static __device__ __forceinline__ bool skip(const Params&) { return false; }
  static __device__ __forceinline__ bool no_loads(const Params&) { return false; }
  static __device__ __forceinline__ int* flags(const Params& p) { return p.flags; }
  static __device__ __forceinline__ int num_jobs(const Params& p, int c, int P) {
    const Sched s = sched(p, c, P);
    return s.hcount + s.q1 + s.count2;
  }
  // dW tile t of the launch's range [w_t0, w_t0 + w_tiles), in groups of up to kDwGroup column
  // blocks of d: a group runs through every vocabulary block of the range before the next group
  // starts, so the part of Ht that the running tiles read (kDwGroup x C x 256 bf16) stays small
  // enough for L2; each exp-tile column block is then read once per group. With d <= 2048 there
  // is one group and the order is vocabulary block, then column block of d.
  static constexpr int kDwGroup = 8;
  static __device__ __forceinline__ TileJob dw_job(const Params& p, int t) {
    const int vb0 = p.w_t0 / p.w_n, nmb = p.w_tiles / p.w_n;
    const int G = p.w_n < kDwGroup ? p.w_n : kDwGroup;
    const int tl = t - p.w_t0;
    const int g = tl / (nmb * G);
    const int gc = p.w_n - g * G < G ? p.w_n - g * G : G;
    const int r = tl - g * nmb * G;
    return TileJob{KIND_DW, vb0 + r / gc, g * G + r % gc, p.w_k, 0, 0};
  }
  static __device__ __forceinline__ TileJob job(const Params& p, int c, int P, int j) {
    const Sched s = sched(p, c, P);
    const int k = deal_rank(p, c, P);
    if (p.odd_dh_first && (c & 1)) {  // this cluster: dH tiles, then its first-phase dW tiles
      if (j < s.hcount) return dh_job(p, k, P, j);
      j -= s.hcount;
      if (j < s.q1) return dw_job(p, p.w_t0 + k + j * P);
      j -= s.q1;
      return dw_job(p, p.w_t0 + p.w_phase1 + s.li + j * s.nlight);
    }
    if (j < s.q1) return dw_job(p, p.w_t0 + k + j * P);
    j -= s.q1;
    if (j < s.hcount) return dh_job(p, k, P, j);
    j -= s.hcount;
    return dw_job(p, p.w_t0 + p.w_phase1 + s.li + j * s.nlight);
  }
  static __device__ __forceinline__ bool job_ok(const Params& p, const TileJob& tj) {
    if (tj.kind == KIND_DH)
      return tj.mb >= 0 && tj.mb < p.h_m && tj.nb >= 0 && tj.nb < p.h_n && tj.part >= 0 && tj.part < p.h_parts &&
             tj.kb0 == tj.part * p.h_kpart && tj.k_blocks > 0 && tj.kb0 + tj.k_blocks <= p.h_k;
    const int vb0 = p.w_t0 / p.w_n;
    return tj.kind == KIND_DW && tj.mb >= vb0 && tj.mb < vb0 + p.w_tiles / p.w_n && tj.mb < p.w_m && tj.nb >= 0 &&
           tj.nb < p.w_n && tj.kb0 == 0 && tj.k_blocks == p.w_k && tj.k_blocks > 0;
  }
  // The j-th dH tile of the cluster at dealing position k. Dealt one part at a time, unit
  // u = k + j P is part u / (h_m h_n) (parts slowest, so the tiles running at once share operand
  // rows of one part) of block u mod (h_m h_n); dealt a block at a time, unit u = k + (j / parts) P
  // is block u and the cluster runs its parts in order.
  static __device__ __forceinline__ TileJob dh_job(const Params& p, int k, int P, int j) {
    const int u = k + (j / p.h_group) * P;
    const int per = p.h_m * p.h_n;
    const int part = p.h_group == 1 ? u / per : j % p.h_group;
    const int t = p.h_group == 1 ? u - part * per : u;
    const int kb0 = part * p.h_kpart;
    const int kb = p.h_k - kb0 < p.h_kpart ? p.h_k - kb0 : p.h_kpart;
    return p.dh_mfast ? TileJob{KIND_DH, t % p.h_m, t / p.h_m, kb, kb0, part}
                      : TileJob{KIND_DH, t / p.h_n, t % p.h_n, kb, kb0, part};
  }
  static __device__ __forceinline__ void load(const Params& p, int kind, uint8_t* a, uint8_t* b, uint32_t bar,
                                              int m0, int n0, int k0) {
    if (kind == KIND_DH) {
      load_k_major(a, &p.ah, bar, m0, k0);
      load_mn_major(b, &p.bh, bar, n0, k0);
    } else {
      load_mn_major(a, &p.aw, bar, m0, k0);
      load_mn_major(b, &p.bw, bar, n0, k0);
    }
  }
  static __device__ __forceinline__ uint64_t a_desc(int kind, uint32_t addr, int k) {
    return kind == KIND_DH ? desc_k_major(addr, k) : desc_mn_major(addr, k);
  }
  static __device__ __forceinline__ uint64_t b_desc(int, uint32_t addr, int k) { return desc_mn_major(addr, k); }
  static __device__ __forceinline__ uint32_t idesc(int kind) {
    return kind == KIND_DH ? idesc_bf16_f32(P_TILE_M, BN, false, true) : idesc_bf16_f32(P_TILE_M, BN, true, true);
  }
  static __device__ __forceinline__ void init(const Params& p, State& st) {
    DhEpi::init(p.h, st.h);
    DwEpi::init(p.w, st.w);
  }
  static __device__ __forceinline__ void epilogue(const Params& p, State& st, const TileJob& tj, EpiCtx ctx, int m0,
                                                  int col0, uint32_t taddr) {
    if (tj.kind == KIND_DH) {
      ctx.out = &p.ch;
      DhEpi::tile(p.h, st.h, ctx, m0, col0, taddr, tj.part, tj.mb * p.h_n + tj.nb);
    } else {
      ctx.out = &p.cw;
      DwEpi::tile(p.w, st.w, ctx, m0, col0, taddr);
    }
  }
};

template <class Prob>
static cudaError_t launch_pair(const typename Prob::Params& p, int clusters, cudaStream_t s) {
  if (clusters <= 0) return cudaSuccess;
  auto kern = gemm_pair_kernel<Prob>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PairSmemLayout::kDynamicBytes);
  if (e != cudaSuccess) return e;
  return launch_k(kern, 2 * clusters, NUM_THREADS, PairSmemLayout::kDynamicBytes, s, p);
}

static int ceil_div_i(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

cudaError_t launch_logits(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, long long M, long long N,
                          long long K, const FwdParams& ep, int no_loads, int num_sms, cudaStream_t s) {
  LogitsProb::Params p;
  p.no_loads = no_loads;
  p.a = a;
  p.b = b;
  p.c = c;
  p.m_tiles = ceil_div_i(M, P_TILE_M);
  p.n_tiles = ceil_div_i(N, BN);
  p.k_blocks = ceil_div_i(K, BK);
  p.flags = ep.flags;
  p.ep = ep;
  const long long tiles = static_cast<long long>(p.m_tiles) * p.n_tiles;
  const int clusters = static_cast<int>(tiles < num_sms / 2 ? tiles : num_sms / 2);
  return launch_pair<LogitsProb>(p, clusters, s);
}

constexpr int kOddDhFirstMaxK = 16;  // k-blocks of a dW tile (chunks of up to 1024 rows)
constexpr double kDhBlockMaxShare = 1.25;

cudaError_t launch_backward(const CUtensorMap& ah, const CUtensorMap& bh, const CUtensorMap& ch, const CUtensorMap& aw,
                            const CUtensorMap& bw, const CUtensorMap& cw, long long rows, long long V, long long d,
                            const DhParams& h, const DwParams& w, int* flags, int num_sms, cudaStream_t s,
                            long long v_begin, long long v_end, bool with_dh) {
  BwdProb::Params p;
  p.ah = ah;
  p.bh = bh;
  p.ch = ch;
  p.aw = aw;
  p.bw = bw;
  p.cw = cw;
  p.h_m = with_dh ? ceil_div_i(rows, P_TILE_M) : 0;
  p.h_n = ceil_div_i(d, BN);
  p.h_k = ceil_div_i(V, BK);
  p.h_kpart = dh_kblocks_per_part(V);
  p.h_parts = dh_parts_for(V);
  p.w_m = ceil_div_i(V, P_TILE_M);
  p.w_n = ceil_div_i(d, BN);
  p.w_k = ceil_div_i(rows, BK);
  // dW tiles of the vocabulary rows [v_begin, v_end) (v_begin a multiple of the tile height)
  if (v_end < 0 || v_end > V) v_end = V;
  if (v_begin < 0) v_begin = 0;
  const int vb0 = static_cast<int>(v_begin / P_TILE_M);
  const int vb1 = v_end > v_begin ? ceil_div_i(v_end, P_TILE_M) : vb0;
  p.w_t0 = vb0 * p.w_n;
  p.w_tiles = (vb1 - vb0) * p.w_n;
  // The dH tiles running at once (about P of them) share an operand only if they read the same
  // rows of P (row block) or the same columns of W (column block of d); whichever the round does
  // not share is streamed again each round, so let that be the smaller one: P [rows, V] (walk
  // column blocks first) or W [V, d] (walk row blocks first). On the d = 7168 head this cut the
  // dH part's DRAM reads from 24 to 15 GB per chunk.
  p.dh_mfast = d > rows ? 1 : 0;
  // Short dW tiles (K = the chunk's rows) are dominated by their fp32 reduce-add into dW; when all
  // clusters run them at once the launch waits on DRAM. With odd clusters taking their dH tiles
  // first, half of the clusters run dW tiles at any time.
  p.odd_dh_first = p.w_k <= kOddDhFirstMaxK ? 1 : 0;
  p.flags = flags;
  p.h = h;
  p.h.parts = p.h_parts;
  p.h.tiles_n = p.h_n;
  p.h.block_major = 0;  // set below with the dealing
  p.w = w;
  const long long nParts = static_cast<long long>(p.h_m) * p.h_n * p.h_parts, nW = p.w_tiles;
  const int P = static_cast<int>(nParts + nW < num_sms / 2 ? nParts + nW : num_sms / 2);
  if (P <= 0) return cudaSuccess;
  // Balance: every cluster should end with the same share of the launch's time. A dH k-block (A
  // K-major, B N-major) runs in ~0.98 of a dW k-block's time (both N-major): 584 vs 594 SM cycles
  // per 64-deep k-block, measured on the Qwen3.5-2B-like head with cycle counters in the MMA issuer.
  constexpr double kDhKblockCost = 0.98;
  const double w_cost = p.w_k;
  // The parts of a dH block go to one cluster back to back when the whole block is no longer than
  // kDhBlockMaxShare of a cluster's fair share: the blocks then run side by side on some clusters,
  // each W and exp-tile block read by all the tiles that need it at once, while the other clusters
  // stream the dW tiles (A/B on one box, Qwen3.5-2B-like head: 784K vs 755K tokens/s at 1024-token
  // chunks, equal at 2048 and 4096). Otherwise the parts are dealt one by one, which balances the
  // clusters when the blocks are fewer than them (540K vs 470K tokens/s at 512-token chunks).
  const double fair = (static_cast<double>(nParts) * kDhKblockCost * p.h_kpart + static_cast<double>(nW) * w_cost) / P;
  p.h_group = (p.h_parts > 1 && kDhKblockCost * p.h_k <= kDhBlockMaxShare * fair) ? p.h_parts : 1;
  p.h.block_major = p.h_group > 1 ? 1 : 0;
  const long long nH = nParts / p.h_group;
  const double h_cost = kDhKblockCost * (p.h_group == 1 ? p.h_kpart : p.h_k);
  const double target = (static_cast<double>(nH) * h_cost + static_cast<double>(nW) * w_cost) / P;
  const long long hmax = (nH + P - 1) / P;
  const long long r = nH % P, nlight = r == 0 ? P : P - r;
  // Longest cluster for q dW tiles each in the first phase: the clusters holding hmax dH tiles, or
  // those holding one fewer that take the second phase's tiles round-robin.
  auto longest = [&](long long q) {
    const long long rem = nW - q * P;
    const long long c2 = rem > 0 ? (rem + nlight - 1) / nlight : 0;
    const double light = static_cast<double>(r == 0 ? hmax : hmax - 1) * h_cost + static_cast<double>(q + c2) * w_cost;
    const double heavy = static_cast<double>(hmax) * h_cost + static_cast<double>(q) * w_cost;
    return r == 0 ? light : (heavy > light ? heavy : light);
  };
  long long q0 = static_cast<long long>((target - static_cast<double>(hmax) * h_cost) / w_cost);
  if (q0 < 0) q0 = 0;
  if (q0 > nW / P) q0 = nW / P;
  long long q1 = q0;
  for (long long q = q0 > 0 ? q0 - 1 : 0; q <= q0 + 1 && q <= nW / P; ++q)
    if (longest(q) < longest(q1)) q1 = q;
  p.w_phase1 = static_cast<int>(q1 * P);
  return launch_pair<BwdProb>(p, P, s);
}

cudaError_t launch_prepare(const int64_t* y, long long N, int V, long long ignore_index, int reduction,
                           long long n_override, const float* grad_loss, DevStatus* st, int* guards, int nguards,
                           int* cnt, int ncnt, cudaStream_t s) {
  return launch_k(k_prepare, 1, 1024, 0, s, y, N, V, ignore_index, reduction, n_override, grad_loss, st, guards,
                  nguards, cnt, ncnt);
}

cudaError_t launch_combine(const float2* partials, int nparts, int rows, const float* ztgt, const int64_t* y,
                           int V, long long ignore_index, float* lse, float* loss_i, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int grid = (rows + warps_per_block - 1) / warps_per_block;
  return launch_k(k_combine, grid, 32 * warps_per_block, 0, s, partials, nparts, rows, ztgt, y, V, ignore_index, lse,
                  loss_i);
}

cudaError_t launch_combine_exp(const float2* partials, int nparts, int rows, const float* ztgt, const int64_t* y,
                               int V, long long ignore_index, const float* ref, const int* guard, float* lse,
                               float* loss_i, float* alpha, __nv_bfloat16* P, long long ldp,
                               const __nv_bfloat16* H, int d, __nv_bfloat16* Ht, const int* only_if, int* flags,
                               cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int grid = (rows + warps_per_block - 1) / warps_per_block;
  return launch_k(k_combine_exp, grid, 32 * warps_per_block, 0, s, partials, nparts, rows, ztgt, y, V, ignore_index,
                  ref, guard, lse, loss_i, alpha, P, ldp, reinterpret_cast<const uint4*>(H), d / 8,
                  reinterpret_cast<uint4*>(Ht), only_if, flags);
}

cudaError_t launch_shard_stats(const float2* partials, int nparts, int rows, const float* ztgt, const int64_t* y,
                               long long y_offset, int V_shard, int V_total, long long ignore_index, float4* stats,
                               cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + 7) / 8;
  return launch_k(k_shard_stats, grid, 256, 0, s, partials, nparts, rows, ztgt, y, y_offset, V_shard, V_total,
                  ignore_index, stats);
}

cudaError_t launch_shard_merge(const float4* stats, int R, long long N, const int64_t* y, int V_total,
                               long long ignore_index, float* lse, float* loss_i, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  const long long grid = (N + 255) / 256;
  return launch_k(k_shard_merge, static_cast<unsigned>(grid), 256, 0, s, stats, R, N, y, V_total, ignore_index, lse,
                  loss_i);
}

cudaError_t launch_vshard_scale(const float4* stats, int R, int rows, const int64_t* y, long long y_offset,
                                int V_shard, int V_total, long long ignore_index, const float* ref, int* guard,
                                float* lse, float* alpha, __nv_bfloat16* P, long long ldp, const __nv_bfloat16* H,
                                int d, __nv_bfloat16* Ht, int* flags, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const cudaError_t e = launch_k(k_vshard_lse, (rows + 255) / 256, 256, 0, s, stats, R, rows, y, y_offset, V_shard,
                                 V_total, ignore_index, ref, guard, lse);
  if (e != cudaSuccess) return e;
  return launch_k(k_vshard_scale, (rows + 7) / 8, 256, 0, s, stats, R, rows, y, y_offset, V_shard, V_total,
                  ignore_index, ref, guard, lse, alpha, P, ldp, reinterpret_cast<const uint4*>(H), d / 8,
                  reinterpret_cast<uint4*>(Ht), flags);
}

cudaError_t launch_scale(void* bf16, long long n_bf16, float* f32, long long n_f32, const float* g, int num_sms,
                         cudaStream_t s) {
  if (n_bf16 <= 0 && n_f32 <= 0) return cudaSuccess;
  return launch_k(k_scale, num_sms * 4, 256, 0, s, static_cast<uint4*>(bf16), n_bf16 / 8,
                  reinterpret_cast<float4*>(f32), n_f32 / 4, g);
}

cudaError_t launch_finalize(const float* loss_i, long long N, const DevStatus* st, float* loss, cudaStream_t s) {
  return launch_k(k_finalize, 1, 1024, 0, s, loss_i, N, st, loss);
}

}  // namespace lce
