// Internal interface between the C-ABI layer (lce_api.cu) and the kernels
// (lce_kernels.cu). Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace lce {

// Programmatic dependent launch. Every kernel of the library starts with
// grid_dep_wait(): it returns once the grids it depends on (the previous
// kernel of the stream) have completed and their writes are visible, at once
// when the launch did not ask for programmatic serialization. grid_dep_launch()
// then lets the next kernel of the stream be scheduled; that kernel's own wait
// still holds its work back until this one has completed.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Every kernel of the library goes out with programmatic stream serialization,
// so that its launch and the scheduling of its blocks overlap the end of the
// kernel before it in the stream (its grid_dep_wait keeps the order).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Device status bits (the workspace's flag word; the first two equal the
// public LCE_DEVICE_* bits).
constexpr int kFlagLabelRange = 1;
constexpr int kFlagTimeout = 2;
constexpr int kFlagBounds = 4;

// Bounds-checking debug build (compiled with -DLCE_CHECKS): every index a
// kernel computes into a plain global buffer, and every tile coordinate it
// hands to TMA, is checked before use; a bad one sets kFlagBounds in the
// device status word and the access is skipped (nothing traps). In the normal
// build the checks compile to nothing.
#if defined(LCE_CHECKS)
constexpr bool kChecks = true;
#else
constexpr bool kChecks = false;
#endif

// True if 0 <= i < n (always true without LCE_CHECKS).
__device__ __forceinline__ bool in_bounds(long long i, long long n, int* flags) {
  if constexpr (!kChecks) {
    return true;
  } else {
    if (i >= 0 && i < n) return true;
    if (flags != nullptr) atomicOr(flags, kFlagBounds);
    return false;
  }
}

// Device-side status block at the start of the workspace.
struct DevStatus {
  int flags;              // kFlag* bits
  int pad0;
  long long n_valid;      // denominator n actually used (count or override)
  long long n_counted;    // valid labels counted in this call
  float gscale;           // g / n (mean), g (sum); 0 when n == 0 under mean
  float pad1;
  double lscale;          // 1 / n (mean), 1 (sum); 0 when n == 0 under mean
};

enum FwdMode : int {
  FWD_STATS = 0,    // per-(row, vocab tile) max / sum-exp partials + target logit
  FWD_STATS_P = 1,  // FWD_STATS + exp-tile P = bf16(exp(z - ref_row)) stored for the backward
  FWD_GRAD = 2,     // gradient tile exp(z - lse) - onehot (valid rows), from a known lse
  FWD_REF = 3,      // row maximum over the first 128 words (one launch over the first tile)
  FWD_STATS_PX = 4, // exact FWD_STATS partials + the exp tile P = bf16(exp(z - ref_row)) (vocabulary shards:
                    // the statistics are exchanged before the tile's scale is known)
};

// An exp-tile entry may exceed the row reference by at most this many nats;
// beyond it the chunk falls back to the exact gradient tile (FWD_GRAD).
constexpr float kRefGuardSum = 1.0e26f;  // ~e^60: bound on a 32-column sum of exp(z - ref)
constexpr float kRefGuardLogit = 60.f;   // the same bound in nats, on lse - ref (vocabulary shards)

struct FwdParams {
  int mode;
  int rows;              // rows of this chunk
  int V;                 // vocabulary columns of this GEMM (a shard's size under vocabulary parallelism)
  int V_total;           // label range: labels in [0, V_total) are valid
  long long y_offset;    // label y sits in column y - y_offset (0 unless W is a vocabulary shard)
  int nparts;            // partials per row: two per 256-column vocabulary tile
  long long ignore_index;
  const int64_t* y;      // labels of this chunk
  float2* partials;      // [rows, nparts] (max, sum-exp) per 128-column half tile
  float* ztgt;           // [rows] logit of the label
  float* ref;            // [rows] row reference (FWD_REF output, FWD_STATS_P / FWD_STATS_PX input)
  const float* lse;      // [rows] (FWD_GRAD input)
  __nv_bfloat16* P;      // [rows, ldp] exp tile (FWD_STATS_P) or gradient tile (FWD_GRAD)
  long long ldp;
  int* flags;
  int* guard;            // FWD_STATS_P(X): set to 1 if some logit exceeds its row reference + guard
  const int* only_if;    // if non-null, the launch does nothing unless *only_if != 0
};

struct DhParams {
  int rows;              // rows of this chunk
  int N;                 // d
  int f32_out;           // 1: fp32 output (a partial dH to be summed across vocabulary shards)
  __nv_bfloat16* out;    // dH of this chunk, [rows, ld] (bf16, or fp32 when f32_out)
  long long ld;
  const float* rowscale; // optional per-row factor (nullptr: none)
  const DevStatus* st;   // gscale
  // The K = V reduction of a dH tile runs as `parts` tiles over fixed vocabulary
  // parts (dh_parts_for(V)); each stores its fp32 sum, and the last of them to
  // arrive adds the parts in part order and writes the tile.
  int parts;             // 1: one tile over the whole vocabulary
  int tiles_n;           // 256-column blocks of d (tile index = row block * tiles_n + column block)
  float4* part_buf;      // [tiles, parts, 2 CTAs, 4 warps, 64 column groups, 32 lanes] fp32 part sums
  int* part_cnt;         // [tiles, 2, 4] arrivals per warp slice; zero before and after each launch
  long long part_slices; // counters (warp slices) the workspace holds (checked build)
  int block_major;       // the parts of each block run back to back on one cluster, in part order
};

// dH parts: the vocabulary's k-blocks (64 words each) are cut into at most
// kDhParts parts of ceil(kblocks / kDhParts) k-blocks. A function of V alone,
// so that every chunk size sums dH in the same order (dH is bitwise the same
// for every chunk size).
constexpr int kDhParts = 4;
inline int dh_kblocks_per_part(long long V) {
  const long long kb = (V + 63) / 64;
  return static_cast<int>((kb + kDhParts - 1) / kDhParts);
}
inline int dh_parts_for(long long V) {
  const long long kb = (V + 63) / 64;
  const long long per = dh_kblocks_per_part(V);
  return per > 0 ? static_cast<int>((kb + per - 1) / per) : 1;
}

struct DwParams {
  int rows;              // V
  int N;                 // d
  float* out;            // dW [V, ld]
  long long ld;
  int accumulate;        // 1: out += result
  const DevStatus* st;   // gscale
};

// Kernel launches (return cudaGetLastError()).
// Also zeroes guards[0, nguards) and cnt[0, ncnt) (the dH part counters).
cudaError_t launch_prepare(const int64_t* y, long long N, int V, long long ignore_index, int reduction,
                           long long n_override, const float* grad_loss, DevStatus* st, int* guards, int nguards,
                           int* cnt, int ncnt, cudaStream_t s);
// Logits GEMM of a chunk: z [M, N] = A [M, K] B [N, K]^T with the FwdEpi
// epilogue; a, b: K-major operand maps, c: the epilogue's store map (any valid
// map if the mode stores nothing).
// no_loads = 1 only for the timeout test (LCE_TEST_FORCE_TIMEOUT): no operand
// loads are issued, so the MMA issuer's bounded wait runs out.
cudaError_t launch_logits(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, long long M, long long N,
                          long long K, const FwdParams& ep, int no_loads, int num_sms, cudaStream_t s);
// Backward GEMMs of a chunk in one launch: dH_c = G W (ah: G K-major, bh: W
// N-major, ch: dH store) and dW (+)= G^T B (aw: G M-major, bw: B N-major, cw:
// dW store / reduce-add). Only the dW rows [v_begin, v_end) are computed
// (v_end < 0: to V; v_begin a multiple of 256), and the dH tiles only if
// with_dh; every tile computed is the same as in the whole launch.
cudaError_t launch_backward(const CUtensorMap& ah, const CUtensorMap& bh, const CUtensorMap& ch, const CUtensorMap& aw,
                            const CUtensorMap& bw, const CUtensorMap& cw, long long rows, long long V, long long d,
                            const DhParams& h, const DwParams& w, int* flags, int num_sms, cudaStream_t s,
                            long long v_begin = 0, long long v_end = -1, bool with_dh = true);
cudaError_t launch_combine(const float2* partials, int nparts, int rows, const float* ztgt, const int64_t* y,
                           int V, long long ignore_index, float* lse, float* loss_i, cudaStream_t s);
// Per row of a chunk: lse, loss_i, alpha_i = exp(ref_i - lse_i) (1 if the chunk's guard is set,
// 0 for ignored rows), the label entry of the exp tile P, and Ht_i = bf16(alpha_i H_i) for the
// chunk's rows of H [rows, d] (the B operand of the dW GEMM). With only_if, the launch does
// nothing unless *only_if != 0.
cudaError_t launch_combine_exp(const float2* partials, int nparts, int rows, const float* ztgt, const int64_t* y,
                               int V, long long ignore_index, const float* ref, const int* guard, float* lse,
                               float* loss_i, float* alpha, __nv_bfloat16* P, long long ldp,
                               const __nv_bfloat16* H, int d, __nv_bfloat16* Ht, const int* only_if, int* flags,
                               cudaStream_t s);
// Vocabulary shards: per-row partial (max, sum-exp, target logit, has-target)
// of this shard, and the fixed-order merge of R shards' partials.
cudaError_t launch_shard_stats(const float2* partials, int nparts, int rows, const float* ztgt, const int64_t* y,
                               long long y_offset, int V_shard, int V_total, long long ignore_index, float4* stats,
                               cudaStream_t s);
cudaError_t launch_shard_merge(const float4* stats, int R, long long N, const int64_t* y, int V_total,
                               long long ignore_index, float* lse, float* loss_i, cudaStream_t s);
// Chunk rows of the stored-tile vocabulary-parallel backward (two launches):
// the merge of launch_shard_merge on stats [R, rows, 4] -> lse, setting *guard
// for a row whose label lies in the shard and whose lse exceeds its reference
// by more than kRefGuardLogit; then alpha_i = exp(ref_i - lse_i) (1 if *guard:
// the tile is then the exact gradient; 0 for ignored rows), the label entry of
// this shard's exp tile P when the label lies in the shard, and
// Ht_i = bf16(alpha_i H_i) for H [rows, d].
cudaError_t launch_vshard_scale(const float4* stats, int R, int rows, const int64_t* y, long long y_offset,
                                int V_shard, int V_total, long long ignore_index, const float* ref, int* guard,
                                float* lse, float* alpha, __nv_bfloat16* P, long long ldp, const __nv_bfloat16* H,
                                int d, __nv_bfloat16* Ht, int* flags, cudaStream_t s);
// Final zero-centred RMSNorm (lce_rmsnorm.cu). rmsnorm_bwd_blocks(N) partial
// rows of d floats are the backward's scratch.
int rmsnorm_bwd_blocks(long long N);
cudaError_t launch_rmsnorm_fwd(const void* x, const float* w, long long N, int d, float eps, void* H, float* rstd,
                               cudaStream_t s);
cudaError_t launch_rmsnorm_bwd(const void* x, const float* w, const float* rstd, const void* dH, long long N, int d,
                               void* dx, float* dw, float* part, cudaStream_t s);
// In-place x *= *g of n_bf16 bf16 values (a multiple of 8) and n_f32 fp32 values (a multiple of 4).
cudaError_t launch_scale(void* bf16, long long n_bf16, float* f32, long long n_f32, const float* g, int num_sms,
                         cudaStream_t s);
cudaError_t launch_finalize(const float* loss_i, long long N, const DevStatus* st, float* loss, cudaStream_t s);

// GEMM tile geometry (must match the kernels): each CTA of a pair loads 128
// rows of a K-major operand per box and 64 rows of an MN-major one.
constexpr int kBoxRowsK = 128;
constexpr int kBoxRowsMN = 64;
constexpr int kTileN = 256;   // vocabulary tile of the logits GEMM (partials: two per tile)

}  // namespace lce
