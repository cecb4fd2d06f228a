// C ABI of liblce.so (declared in include/lce.h): argument checks, workspace
// carve-up, TMA tensor maps and the stream-ordered launch sequence of the
// chunked LM-head cross-entropy. No device memory is allocated here; every
// launch goes to the caller's stream and nothing synchronises the host unless
// the caller asks for it (opts->sync_check).
//
// Launch sequence of lce_fwd_bwd ("XTuner on Ascend 910C: Qwen3.5-2B training
// optimisation", section 3.1.4; tokens in chunks as in "XTuner V1
// introduction", memory optimisation section):
//   prepare                      label scan -> n, g/n, range-error bit
//   logits GEMM (FWD_REF)        row reference of every row: max over the first 128 words
//   for each chunk of C tokens:
//     logits GEMM (FWD_STATS_P)  exp tile P = bf16(exp(z - ref)), per half tile (ref, sum of
//                                those exps), z_{i,y_i}
//     combine                    lse_i, loss_i, alpha_i = exp(ref_i - lse_i), label entry of P,
//                                Ht = alpha * H_c
//     only if the chunk's guard is set (a 32-column sum of exp(z - ref) above ~e^60):
//       logits GEMM (FWD_STATS)  exact online statistics
//       combine                  again, with alpha = 1
//       logits GEMM (FWD_GRAD)   the exact gradient tile replaces P
//     backward GEMMs (one launch) dH_c = (g/n) alpha (P W) and dW (+)= (g/n) P^T Ht
//   finalize                     loss = sum_i loss_i / n
// lce_forward runs prepare, FWD_STATS + combine per chunk, finalize;
// lce_backward recomputes: FWD_GRAD (from the saved lse), then the backward
// GEMMs. lce_fwd_bwd_sliced issues the last chunk's backward GEMMs as one
// launch per vocabulary slice of dW and records an event after each.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <vector>

#include "../../include/lce.h"
#include "lce_internal.h"

namespace {

using lce::DevStatus;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

constexpr int64_t kDefaultChunk = 4096;
constexpr int64_t kVocabTile = lce::kTileN;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
  int64_t C = 0;       // tokens per chunk
  int64_t T = 0;       // vocabulary tiles per row
  int64_t ldp = 0;     // row stride (elements) of the exp / gradient tile buffer
  int64_t chunks = 0;  // number of chunks
  size_t status = 0, loss_i = 0, lse = 0, ztgt = 0, partials = 0, P = 0;
  size_t ref = 0, alpha = 0, guard = 0, Ht = 0, total = 0;
  size_t dh_cnt = 0, dh_part = 0;  // dH part counters and part sums (backward calls)
  int dh_ncnt = 0;                 // number of dH part counters
};

// The dH part counters and part sums of one chunk's backward launch: a counter
// per (dH tile, CTA, epilogue warp), and, when the vocabulary is cut into more
// than one part, one fp32 [256 x 256] sum per dH tile and part.
void take_dh_parts(Layout& L, int64_t d, int64_t V, const std::function<size_t(size_t)>& take) {
  const int64_t tiles = ceil_div(L.C, 256) * ceil_div(d, 256);
  L.dh_ncnt = static_cast<int>(tiles * 8);
  L.dh_cnt = take(sizeof(int) * static_cast<size_t>(L.dh_ncnt));
  const int parts = lce::dh_parts_for(V);
  if (parts > 1) L.dh_part = take(sizeof(float) * 256 * 256 * static_cast<size_t>(tiles) * static_cast<size_t>(parts));
}

int64_t chunk_of(int64_t N, const lce_opts* o) {
  int64_t C = (o && o->chunk_tokens > 0) ? o->chunk_tokens : kDefaultChunk;
  if (C > N) C = N;
  if (C < 1) C = 1;
  return C;
}

Layout make_layout(int op, int64_t N, int64_t d, int64_t V, const lce_opts* o) {
  Layout L;
  L.C = chunk_of(N, o);
  L.T = ceil_div(V, kVocabTile);
  L.ldp = ceil_div(V, kVocabTile) * kVocabTile;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.status = take(sizeof(DevStatus));
  if (op == LCE_OP_VSHARD_CHUNK) {  // one chunk: its exp tile, statistics, references, alpha and Ht
    L.chunks = 1;
    L.ztgt = take(sizeof(float) * static_cast<size_t>(L.C));
    L.partials = take(sizeof(float) * 2 * static_cast<size_t>(L.C) * static_cast<size_t>(2 * L.T));
    L.ref = take(sizeof(float) * static_cast<size_t>(L.C));
    L.alpha = take(sizeof(float) * static_cast<size_t>(L.C));
    L.guard = take(sizeof(int));
    L.Ht = take(2 * static_cast<size_t>(L.C) * static_cast<size_t>(d));
    L.P = take(2 * static_cast<size_t>(L.C) * static_cast<size_t>(L.ldp));
    take_dh_parts(L, d, V, take);
    L.total = off;
    return L;
  }
  if (op == LCE_OP_VSHARD_COMBINE) {
    L.loss_i = take(sizeof(float) * static_cast<size_t>(N > 0 ? N : 1));
    L.total = off;
    return L;
  }
  const bool fwd = op == LCE_OP_FORWARD || op == LCE_OP_FWD_BWD;
  const bool bwd = op == LCE_OP_BACKWARD || op == LCE_OP_FWD_BWD;
  if (fwd) {
    L.loss_i = take(sizeof(float) * static_cast<size_t>(N > 0 ? N : 1));
    L.ztgt = take(sizeof(float) * static_cast<size_t>(L.C));
    L.partials = take(sizeof(float) * 2 * static_cast<size_t>(L.C) * static_cast<size_t>(2 * L.T));
  }
  L.chunks = N > 0 ? ceil_div(N, L.C) : 0;
  if (op == LCE_OP_FWD_BWD) {
    L.lse = take(sizeof(float) * static_cast<size_t>(N > 0 ? N : 1));
    L.ref = take(sizeof(float) * static_cast<size_t>(N > 0 ? N : 1));
    L.alpha = take(sizeof(float) * static_cast<size_t>(L.C));
    L.guard = take(sizeof(int) * static_cast<size_t>(L.chunks > 0 ? L.chunks : 1));
    L.Ht = take(2 * static_cast<size_t>(L.C) * static_cast<size_t>(d));
  }
  if (bwd) {
    L.P = take(2 * static_cast<size_t>(L.C) * static_cast<size_t>(L.ldp));
    take_dh_parts(L, d, V, take);
  }
  L.total = off;
  return L;
}

// lce_norm_fwd_bwd: the fused linear-CE workspace, then H, rstd, dH and the
// RMSNorm backward's partial rows.
struct NormLayout {
  Layout lce;
  size_t H = 0, rstd = 0, dH = 0, part = 0, total = 0;
};

NormLayout norm_layout(int64_t N, int64_t d, int64_t V, const lce_opts* o) {
  NormLayout L;
  L.lce = make_layout(LCE_OP_FWD_BWD, N, d, V, o);
  size_t off = L.lce.total;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  const size_t nd = static_cast<size_t>(N > 0 ? N : 1) * static_cast<size_t>(d);
  L.H = take(2 * nd);
  L.rstd = take(sizeof(float) * static_cast<size_t>(N > 0 ? N : 1));
  L.dH = take(2 * nd);
  L.part = take(sizeof(float) * static_cast<size_t>(lce::rmsnorm_bwd_blocks(N > 0 ? N : 1)) * static_cast<size_t>(d));
  L.total = off;
  return L;
}

constexpr int64_t kNormMaxD = 32768;  // the norm backward keeps a row of dw partials in shared memory

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_sizes(int64_t N, int64_t d, int64_t V, const lce_opts* o) {
  if (N < 0 || d <= 0 || V <= 0 || (d % 8) != 0) return LCE_ERR_INVALID_ARG;
  if (N > (int64_t{1} << 31) - 1 || V > (int64_t{1} << 31) - 1 || d > (int64_t{1} << 24)) return LCE_ERR_INVALID_ARG;
  if (o) {
    if (o->reduction != LCE_MEAN && o->reduction != LCE_SUM) return LCE_ERR_INVALID_ARG;
    if (o->chunk_tokens < 0 || (o->reserved != 0 && o->reserved != LCE_TEST_FORCE_TIMEOUT))
      return LCE_ERR_INVALID_ARG;
    if (o->accumulate_dW != 0 && o->accumulate_dW != 1) return LCE_ERR_INVALID_ARG;
  }
  return LCE_OK;
}

struct DeviceInfo {
  int num_sms = 0;
};

int device_check(DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LCE_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LCE_ERR_CUDA;
  if (major != 10 || minor != 3) return LCE_ERR_UNSUPPORTED_DEVICE;
  if (encode_fn() == nullptr) return LCE_ERR_CUDA;
  info->num_sms = sms;
  return LCE_OK;
}

// 2-D tensor map over a row-major [rows, cols] matrix with row stride ld
// (elements), 128-byte swizzle, box = {box_cols, box_rows} (box_cols * element
// size = 128 bytes). Loads past rows/cols return zeros; stores there are dropped.
int make_map_t(CUtensorMap* m, CUtensorMapDataType dtype, uint32_t esize, const void* base, int64_t rows,
               int64_t cols, int64_t ld, uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = encode_fn()(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LCE_OK : LCE_ERR_CUDA;
}

// bf16 operand / output map: boxes of 64 columns.
int make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows) {
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, ld, 64u, box_rows);
}

// Rows of output tile one epilogue warp stores at a time.
constexpr uint32_t kStoreRows = 32;

#define LCE_TRY(x)                         \
  do {                                     \
    const int _rc = (x);                   \
    if (_rc != LCE_OK) return _rc;         \
  } while (0)
#define LCE_CUDA(x)                                  \
  do {                                               \
    if ((x) != cudaSuccess) return LCE_ERR_CUDA;     \
  } while (0)

// ---------------------------------------------------------------------------
// Measurement hook: events around each launch while profiling is on.
// ---------------------------------------------------------------------------
enum Kind : int {
  K_PREPARE = 0,
  K_LOGITS_STATS = 1,   // FWD_STATS and FWD_STATS_P
  K_COMBINE = 2,
  K_LOGITS_GRAD = 3,    // unconditional FWD_GRAD (lce_backward)
  K_GEMM_BWD = 4,       // dH and dW GEMMs of a chunk (one launch)
  K_RMSNORM_FWD = 5,
  K_FINALIZE = 6,
  K_OTHER = 7,          // the guard-conditional passes (work counted as 0), gradient scaling
  K_LOGITS_REF = 8,
  K_MEMSET = 9,         // zeroing dW when there are no tokens (a copy-engine memset, not a kernel)
  K_RMSNORM_BWD = 10,   // norm backward and the column sum of its dw partials
};
const char* const kKindNames[LCE_KERNEL_KINDS] = {"prepare",    "logits_stats", "combine",  "logits_grad",
                                                  "gemm_dH_dW", "rmsnorm_fwd",  "finalize", "other",
                                                  "logits_ref", "memset",       "rmsnorm_bwd"};

struct ProfRecord {
  int kind;
  cudaEvent_t start, stop;
  double work;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> pool;
  std::vector<ProfRecord> recs;
};
Profiler g_prof;

cudaEvent_t take_event() {
  if (!g_prof.pool.empty()) {
    cudaEvent_t e = g_prof.pool.back();
    g_prof.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Run one launch; while profiling, bracket it with events on stream s.
template <class F>
int timed(cudaStream_t s, int kind, double work, F&& launch) {
  if (!g_prof.on) return launch();
  std::lock_guard<std::mutex> lock(g_prof.mu);
  cudaEvent_t a = take_event(), b = take_event();
  if (!a || !b) return LCE_ERR_CUDA;
  if (cudaEventRecord(a, s) != cudaSuccess) return LCE_ERR_CUDA;
  const int rc = launch();
  if (cudaEventRecord(b, s) != cudaSuccess) return LCE_ERR_CUDA;
  g_prof.recs.push_back({kind, a, b, work});
  return rc;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? LCE_OK : LCE_ERR_CUDA; }

struct Call {
  const uint16_t* H;
  const uint16_t* W;
  const int64_t* y;
  int64_t N, d, V;
  int64_t V_total = 0;   // label range (V unless W is a vocabulary shard)
  int64_t y_offset = 0;  // first vocabulary row of the shard
  lce_opts o;
  uint8_t* ws;
  Layout L;
  DevStatus* st;
  cudaStream_t s;
  DeviceInfo dev;
};

// Logits GEMM for one chunk, in one of the FwdMode epilogues.
struct LogitsArgs {
  int mode = lce::FWD_STATS;
  const float* lse_rows = nullptr;  // FWD_GRAD
  uint16_t* P = nullptr;            // FWD_STATS_P, FWD_GRAD
  float* ref = nullptr;             // FWD_REF out, FWD_STATS_P in
  int* guard = nullptr;             // FWD_STATS_P
  const int* only_if = nullptr;     // conditional launch
};

int logits_gemm(const Call& c, int64_t c0, int64_t rows, const LogitsArgs& a) {
  CUtensorMap mA, mB, mC;
  LCE_TRY(make_map(&mA, c.H + c0 * c.d, rows, c.d, c.d, lce::kBoxRowsK));
  LCE_TRY(make_map(&mB, c.W, c.V, c.d, c.d, lce::kBoxRowsK));
  if (a.P)  // exp / gradient tile: [rows, V] bf16 with row stride ldp
    LCE_TRY(make_map(&mC, a.P, rows, c.V, c.L.ldp, kStoreRows));
  else
    mC = mB;  // this epilogue stores nothing
  const int64_t ncols = a.mode == lce::FWD_REF ? lce::kTileN : c.V;  // FWD_REF: the first vocabulary tile only
  lce::FwdParams p;
  std::memset(&p, 0, sizeof p);
  p.mode = a.mode;
  p.rows = static_cast<int>(rows);
  p.V = static_cast<int>(c.V);
  p.V_total = static_cast<int>(c.V_total);
  p.y_offset = c.y_offset;
  p.nparts = static_cast<int>(2 * c.L.T);
  p.ignore_index = c.o.ignore_index;
  p.y = c.y + c0;
  p.partials = reinterpret_cast<float2*>(c.ws + c.L.partials);
  p.ztgt = reinterpret_cast<float*>(c.ws + c.L.ztgt);
  p.ref = a.ref;
  p.lse = a.lse_rows;
  p.P = reinterpret_cast<__nv_bfloat16*>(a.P);
  p.ldp = c.L.ldp;
  p.flags = &c.st->flags;
  p.guard = a.guard;
  p.only_if = a.only_if;
  const double flops = 2.0 * static_cast<double>(rows) * static_cast<double>(ncols) * static_cast<double>(c.d);
  int kind = a.only_if ? K_OTHER : K_LOGITS_STATS;
  if (a.mode == lce::FWD_REF) kind = K_LOGITS_REF;
  if (a.mode == lce::FWD_GRAD && !a.only_if) kind = K_LOGITS_GRAD;
  const int no_loads = (c.o.reserved == LCE_TEST_FORCE_TIMEOUT && a.mode == lce::FWD_STATS) ? 1 : 0;
  return timed(c.s, kind, a.only_if ? 0.0 : flops, [&] {
    return cuda_rc(lce::launch_logits(mA, mB, mC, rows, ncols, c.d, p, no_loads, c.dev.num_sms, c.s));
  });
}

int forward_chunk(const Call& c, int64_t c0, int64_t rows, float* lse, float* loss_i) {
  LogitsArgs a;
  a.mode = lce::FWD_STATS;
  LCE_TRY(logits_gemm(c, c0, rows, a));
  const double bytes = static_cast<double>(rows) * (16.0 * static_cast<double>(c.L.T) + 4 + 8 + 4 + 4);
  return timed(c.s, K_COMBINE, bytes, [&] {
    return cuda_rc(lce::launch_combine(reinterpret_cast<const float2*>(c.ws + c.L.partials), static_cast<int>(2 * c.L.T),
                                       static_cast<int>(rows), reinterpret_cast<const float*>(c.ws + c.L.ztgt),
                                       c.y + c0, static_cast<int>(c.V), c.o.ignore_index, lse + c0, loss_i + c0,
                                       c.s));
  });
}

// Which part of the backward one launch computes: the dW rows [v_begin, v_end)
// (v_end < 0: to V) and, if with_dh, the chunk's dH.
struct BwdPart {
  int64_t v_begin = 0, v_end = -1;
  bool with_dh = true;
};

// dH_c = (g/n) [rowscale] (G W) and dW (+)= (g/n) G^T B, with G [rows, V] in
// the chunk's tile buffer and B = H_c or Ht: one launch for both GEMMs.
int dh_dw(const Call& c, int64_t c0, int64_t rows, const float* rowscale, const uint16_t* B, void* dH, float* dW,
          bool accumulate, bool dH_f32 = false, const BwdPart& part = BwdPart()) {
  const uint16_t* P = reinterpret_cast<const uint16_t*>(c.ws + c.L.P);
  CUtensorMap mG, mW, mdH, mGt, mB, mdW;
  LCE_TRY(make_map(&mG, P, rows, c.V, c.L.ldp, lce::kBoxRowsK));      // dH: A, K-major
  LCE_TRY(make_map(&mW, c.W, c.V, c.d, c.d, lce::kBoxRowsMN));        // dH: B, N-major
  if (dH_f32)                                                           // dH store
    LCE_TRY(make_map_t(&mdH, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, static_cast<float*>(dH) + c0 * c.d, rows, c.d, c.d,
                       32u, kStoreRows));
  else
    LCE_TRY(make_map(&mdH, static_cast<uint16_t*>(dH) + c0 * c.d, rows, c.d, c.d, kStoreRows));
  LCE_TRY(make_map(&mGt, P, rows, c.V, c.L.ldp, lce::kBoxRowsMN));    // dW: A, M-major
  LCE_TRY(make_map(&mB, B, rows, c.d, c.d, lce::kBoxRowsMN));          // dW: B, N-major
  LCE_TRY(make_map_t(&mdW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW, c.V, c.d, c.d, 32u, kStoreRows));
  lce::DhParams dp;
  dp.rows = static_cast<int>(rows);
  dp.N = static_cast<int>(c.d);
  dp.f32_out = dH_f32 ? 1 : 0;
  dp.out = nullptr;  // written through the store map
  dp.ld = c.d;
  dp.rowscale = rowscale;
  dp.st = c.st;
  dp.part_buf = c.L.dh_part ? reinterpret_cast<float4*>(c.ws + c.L.dh_part) : nullptr;
  dp.part_cnt = reinterpret_cast<int*>(c.ws + c.L.dh_cnt);
  dp.part_slices = c.L.dh_ncnt;
  lce::DwParams wp;
  wp.rows = static_cast<int>(c.V);
  wp.N = static_cast<int>(c.d);
  wp.out = dW;
  wp.ld = c.d;
  wp.accumulate = accumulate ? 1 : 0;
  wp.st = c.st;
  const int64_t v_end = part.v_end < 0 ? c.V : part.v_end;
  const double dw_rows = static_cast<double>(v_end - part.v_begin);
  const double flops = 2.0 * static_cast<double>(rows) * static_cast<double>(c.d) *
                       ((part.with_dh ? static_cast<double>(c.V) : 0.0) + dw_rows);
  return timed(c.s, K_GEMM_BWD, flops, [&] {
    return cuda_rc(lce::launch_backward(mG, mW, mdH, mGt, mB, mdW, rows, c.V, c.d, dp, wp, &c.st->flags,
                                        c.dev.num_sms, c.s, part.v_begin, v_end, part.with_dh));
  });
}

// dW in vocabulary slices (lce_fwd_bwd_sliced): the last chunk's backward runs
// as one launch per slice, the dH tiles with the last slice, and events[s] is
// recorded once rows [bounds[s], bounds[s+1]) of dW are final.
struct Slices {
  int n = 0;
  const int64_t* bounds = nullptr;
  void* const* events = nullptr;
};

int record_slice_events(const Call& c, const Slices* sl, int first) {
  if (!sl || !sl->events) return LCE_OK;
  for (int k = first; k < sl->n; ++k)
    LCE_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(sl->events[k]), c.s));
  return LCE_OK;
}

int dh_dw_sliced(const Call& c, int64_t c0, int64_t rows, const float* rowscale, const uint16_t* B, void* dH,
                 float* dW, bool accumulate, const Slices& sl) {
  for (int k = 0; k < sl.n; ++k) {
    BwdPart part;
    part.v_begin = sl.bounds[k];
    part.v_end = sl.bounds[k + 1];
    part.with_dh = k == sl.n - 1;
    if (part.with_dh || part.v_end > part.v_begin)
      LCE_TRY(dh_dw(c, c0, rows, rowscale, B, dH, dW, accumulate, false, part));
    if (sl.events) LCE_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(sl.events[k]), c.s));
  }
  return LCE_OK;
}

// Backward of one chunk from a known lse: recompute the logits into the
// exact gradient tile, then the two GEMMs.
int backward_chunk(const Call& c, int64_t c0, int64_t rows, const float* lse, void* dH, float* dW, bool accumulate,
                   bool dH_f32 = false) {
  LogitsArgs a;
  a.mode = lce::FWD_GRAD;
  a.lse_rows = lse + c0;
  a.P = reinterpret_cast<uint16_t*>(c.ws + c.L.P);
  LCE_TRY(logits_gemm(c, c0, rows, a));
  return dh_dw(c, c0, rows, nullptr, c.H + c0 * c.d, dH, dW, accumulate, dH_f32);
}

// Forward and backward of one chunk without recomputing the logits: the
// forward stores the exp tile, the backward rescales it per row.
int fused_chunk(const Call& c, int64_t chunk, int64_t c0, int64_t rows, float* lse, float* loss_i, uint16_t* dH,
                float* dW, bool accumulate, const Slices* sl = nullptr) {
  uint16_t* P = reinterpret_cast<uint16_t*>(c.ws + c.L.P);
  float* ref = reinterpret_cast<float*>(c.ws + c.L.ref) + c0;  // row references of every row, computed up front
  float* alpha = reinterpret_cast<float*>(c.ws + c.L.alpha);
  int* guard = reinterpret_cast<int*>(c.ws + c.L.guard) + chunk;
  uint16_t* Ht = reinterpret_cast<uint16_t*>(c.ws + c.L.Ht);

  LogitsArgs a;
  a.mode = lce::FWD_STATS_P;
  a.ref = ref;
  a.P = P;
  a.guard = guard;
  LCE_TRY(logits_gemm(c, c0, rows, a));

  const double cbytes = static_cast<double>(rows) *
                        (16.0 * static_cast<double>(c.L.T) + 4 + 8 + 4 + 4 + 4 + 4 + 2 + 4.0 * static_cast<double>(c.d));
  auto combine = [&](const int* only_if) {
    return timed(c.s, only_if ? K_OTHER : K_COMBINE, only_if ? 0.0 : cbytes, [&] {
      return cuda_rc(lce::launch_combine_exp(
          reinterpret_cast<const float2*>(c.ws + c.L.partials), static_cast<int>(2 * c.L.T), static_cast<int>(rows),
          reinterpret_cast<const float*>(c.ws + c.L.ztgt), c.y + c0, static_cast<int>(c.V), c.o.ignore_index, ref,
          guard, lse + c0, loss_i + c0, alpha, reinterpret_cast<__nv_bfloat16*>(P), c.L.ldp,
          reinterpret_cast<const __nv_bfloat16*>(c.H + c0 * c.d), static_cast<int>(c.d),
          reinterpret_cast<__nv_bfloat16*>(Ht), only_if, &c.st->flags, c.s));
    });
  };
  LCE_TRY(combine(nullptr));

  // If the guard is set (a logit far above its row reference), the statistics
  // above may have overflowed: recompute them exactly (online max / sum-exp),
  // combine again (alpha = 1), and write the exact gradient tile. All three
  // launches return at once when the guard is clear.
  LogitsArgs x;
  x.mode = lce::FWD_STATS;
  x.only_if = guard;
  LCE_TRY(logits_gemm(c, c0, rows, x));
  LCE_TRY(combine(guard));

  LogitsArgs g;
  g.mode = lce::FWD_GRAD;
  g.lse_rows = lse + c0;
  g.P = P;
  g.only_if = guard;
  LCE_TRY(logits_gemm(c, c0, rows, g));

  if (sl) return dh_dw_sliced(c, c0, rows, alpha, Ht, dH, dW, accumulate, *sl);
  return dh_dw(c, c0, rows, alpha, Ht, dH, dW, accumulate);
}

// Row references m~_i for all N rows in one launch (one round of 256-row tiles
// over the first vocabulary tile), before the chunk loop.
int row_references(const Call& c) {
  LogitsArgs a;
  a.mode = lce::FWD_REF;
  a.ref = reinterpret_cast<float*>(c.ws + c.L.ref);
  return logits_gemm(c, 0, c.N, a);
}

int prepare(const Call& c, const float* grad_loss, bool reset_guards = true) {
  int* guards = c.L.guard ? reinterpret_cast<int*>(c.ws + c.L.guard) : nullptr;
  const int nguards = c.L.guard && reset_guards ? static_cast<int>(c.L.chunks) : 0;
  int* cnt = c.L.dh_cnt ? reinterpret_cast<int*>(c.ws + c.L.dh_cnt) : nullptr;
  const int ncnt = c.L.dh_cnt ? c.L.dh_ncnt : 0;
  return timed(c.s, K_PREPARE, 8.0 * static_cast<double>(c.N), [&] {
    return cuda_rc(lce::launch_prepare(c.y, c.N, static_cast<int>(c.V_total), c.o.ignore_index, c.o.reduction,
                                       c.o.n_valid_override, grad_loss, c.st, guards, nguards, cnt, ncnt, c.s));
  });
}

int finalize(const Call& c, const float* loss_i, float* loss) {
  return timed(c.s, K_FINALIZE, 4.0 * static_cast<double>(c.N),
               [&] { return cuda_rc(lce::launch_finalize(loss_i, c.N, c.st, loss, c.s)); });
}

int finish(const Call& c) {
  if (!c.o.sync_check) return LCE_OK;
  LCE_CUDA(cudaStreamSynchronize(c.s));
  int flags = 0;
  LCE_CUDA(cudaMemcpy(&flags, &c.st->flags, sizeof flags, cudaMemcpyDeviceToHost));
  if (flags & lce::kFlagBounds) return LCE_ERR_BOUNDS;
  if (flags & lce::kFlagTimeout) return LCE_ERR_TIMEOUT;
  if (flags & lce::kFlagLabelRange) return LCE_ERR_LABEL_RANGE;
  return LCE_OK;
}

int begin(Call* c, int op, const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
          const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  lce_opts_init(&c->o);
  if (opts) c->o = *opts;
  LCE_TRY(check_sizes(N, d, V, &c->o));
  if (!W || !ws || (N > 0 && (!H || !y))) return LCE_ERR_INVALID_ARG;
  if (!aligned(W, 16) || (H && !aligned(H, 16)) || (y && !aligned(y, 8)) || !aligned(ws, 256))
    return LCE_ERR_ALIGNMENT;
  c->L = make_layout(op, N, d, V, &c->o);
  if (ws_bytes < c->L.total) return LCE_ERR_WORKSPACE;
  c->H = static_cast<const uint16_t*>(H);
  c->W = static_cast<const uint16_t*>(W);
  c->y = y;
  c->N = N;
  c->d = d;
  c->V = V;
  c->V_total = V;
  c->y_offset = 0;
  c->ws = static_cast<uint8_t*>(ws);
  c->st = reinterpret_cast<DevStatus*>(c->ws + c->L.status);
  c->s = static_cast<cudaStream_t>(stream);
  return LCE_OK;
}

}  // namespace

extern "C" {

void lce_opts_init(lce_opts* o) {
  if (!o) return;
  std::memset(o, 0, sizeof *o);
  o->chunk_tokens = 0;
  o->ignore_index = -100;
  o->n_valid_override = -1;
  o->reduction = LCE_MEAN;
}

size_t lce_workspace_size(int op, int64_t N, int64_t d, int64_t V, const lce_opts* opts) {
  lce_opts o;
  lce_opts_init(&o);
  if (opts) o = *opts;
  if (op < LCE_OP_FORWARD || op > LCE_OP_VSHARD_CHUNK) return 0;
  if (check_sizes(N, d, V, &o) != LCE_OK) return 0;
  if (op == LCE_OP_NORM_FWD_BWD) return norm_layout(N, d, V, &o).total;
  return make_layout(op, N, d, V, &o).total;
}

int64_t lce_auto_chunk(int64_t N, int64_t d, int64_t V, size_t budget_bytes, const lce_opts* opts) {
  lce_opts o;
  lce_opts_init(&o);
  if (opts) o = *opts;
  if (check_sizes(N, d, V, &o) != LCE_OK || N <= 0) return 0;
  const int64_t cap = ((N + 255) / 256) * 256;
  for (int64_t C = 4096 < cap ? 4096 : cap; C >= 256; C -= 256) {
    o.chunk_tokens = C;
    if (make_layout(LCE_OP_FWD_BWD, N, d, V, &o).total <= budget_bytes) return C;
  }
  return 0;
}

int lce_forward(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V, float* loss,
                float* lse, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  Call c;
  LCE_TRY(begin(&c, LCE_OP_FORWARD, H, W, y, N, d, V, opts, ws, ws_bytes, stream));
  if (!loss || (N > 0 && !lse)) return LCE_ERR_INVALID_ARG;
  if (!aligned(loss, 4) || (lse && !aligned(lse, 4))) return LCE_ERR_ALIGNMENT;
  LCE_TRY(device_check(&c.dev));
  LCE_TRY(prepare(c, nullptr));
  float* loss_i = reinterpret_cast<float*>(c.ws + c.L.loss_i);
  for (int64_t c0 = 0; c0 < N; c0 += c.L.C) {
    const int64_t rows = (N - c0) < c.L.C ? (N - c0) : c.L.C;
    LCE_TRY(forward_chunk(c, c0, rows, lse, loss_i));
  }
  LCE_TRY(finalize(c, loss_i, loss));
  return finish(c);
}

int lce_backward(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V, const float* lse,
                 const float* grad_loss, void* dH, float* dW, const lce_opts* opts, void* ws, size_t ws_bytes,
                 void* stream) {
  Call c;
  LCE_TRY(begin(&c, LCE_OP_BACKWARD, H, W, y, N, d, V, opts, ws, ws_bytes, stream));
  if (c.o.reserved != 0) return LCE_ERR_INVALID_ARG;
  if (!dW || (N > 0 && (!lse || !dH))) return LCE_ERR_INVALID_ARG;
  if (!aligned(dW, 16) || (dH && !aligned(dH, 16)) || (lse && !aligned(lse, 4)) ||
      (grad_loss && !aligned(grad_loss, 4)))
    return LCE_ERR_ALIGNMENT;
  LCE_TRY(device_check(&c.dev));
  LCE_TRY(prepare(c, grad_loss));
  if (N == 0 && !c.o.accumulate_dW)
    LCE_TRY(timed(c.s, K_MEMSET, 4.0 * static_cast<double>(V * d),
                  [&] { return cuda_rc(cudaMemsetAsync(dW, 0, sizeof(float) * static_cast<size_t>(V * d), c.s)); }));
  for (int64_t c0 = 0; c0 < N; c0 += c.L.C) {
    const int64_t rows = (N - c0) < c.L.C ? (N - c0) : c.L.C;
    LCE_TRY(backward_chunk(c, c0, rows, lse, static_cast<uint16_t*>(dH), dW, c.o.accumulate_dW || c0 > 0));
  }
  return finish(c);
}

}  // extern "C"

namespace {

int fwd_bwd(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V, const float* grad_loss,
            float* loss, float* lse, void* dH, float* dW, const lce_opts* opts, void* ws, size_t ws_bytes,
            void* stream, const Slices* sl, int sm_limit) {
  Call c;
  LCE_TRY(begin(&c, LCE_OP_FWD_BWD, H, W, y, N, d, V, opts, ws, ws_bytes, stream));
  if (c.o.reserved != 0) return LCE_ERR_INVALID_ARG;
  if (!loss || !dW || (N > 0 && !dH)) return LCE_ERR_INVALID_ARG;
  if (!aligned(loss, 4) || !aligned(dW, 16) || (dH && !aligned(dH, 16)) || (lse && !aligned(lse, 4)) ||
      (grad_loss && !aligned(grad_loss, 4)))
    return LCE_ERR_ALIGNMENT;
  LCE_TRY(device_check(&c.dev));
  if (sm_limit > 0 && sm_limit < c.dev.num_sms) c.dev.num_sms = sm_limit & ~1;
  float* lse_rows = lse ? lse : reinterpret_cast<float*>(c.ws + c.L.lse);
  float* loss_i = reinterpret_cast<float*>(c.ws + c.L.loss_i);
  LCE_TRY(prepare(c, grad_loss));
  if (N == 0 && !c.o.accumulate_dW)
    LCE_TRY(timed(c.s, K_MEMSET, 4.0 * static_cast<double>(V * d),
                  [&] { return cuda_rc(cudaMemsetAsync(dW, 0, sizeof(float) * static_cast<size_t>(V * d), c.s)); }));
  if (N == 0) LCE_TRY(record_slice_events(c, sl, 0));
  if (N > 0) LCE_TRY(row_references(c));
  for (int64_t k = 0, c0 = 0; c0 < N; ++k, c0 += c.L.C) {
    const int64_t rows = (N - c0) < c.L.C ? (N - c0) : c.L.C;
    const bool last = c0 + rows >= N;
    LCE_TRY(fused_chunk(c, k, c0, rows, lse_rows, loss_i, static_cast<uint16_t*>(dH), dW,
                        c.o.accumulate_dW || c0 > 0, last ? sl : nullptr));
  }
  LCE_TRY(finalize(c, loss_i, loss));
  return finish(c);
}

}  // namespace

extern "C" {

int lce_fwd_bwd(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                const float* grad_loss, float* loss, float* lse, void* dH, float* dW, const lce_opts* opts, void* ws,
                size_t ws_bytes, void* stream) {
  return fwd_bwd(H, W, y, N, d, V, grad_loss, loss, lse, dH, dW, opts, ws, ws_bytes, stream, nullptr, 0);
}

int lce_fwd_bwd_sliced(const void* H, const void* W, const int64_t* y, int64_t N, int64_t d, int64_t V,
                       const float* grad_loss, float* loss, float* lse, void* dH, float* dW, int32_t n_slices,
                       const int64_t* slice_bounds, void* const* slice_events, int32_t sm_limit,
                       const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  if (n_slices < 1 || n_slices > LCE_MAX_SLICES || !slice_bounds || sm_limit < 0 || sm_limit == 1)
    return LCE_ERR_INVALID_ARG;
  if (slice_bounds[0] != 0 || slice_bounds[n_slices] != V) return LCE_ERR_INVALID_ARG;
  for (int k = 0; k < n_slices; ++k) {
    if (slice_bounds[k + 1] < slice_bounds[k]) return LCE_ERR_INVALID_ARG;
    if (k > 0 && slice_bounds[k] % LCE_SLICE_ALIGN != 0) return LCE_ERR_INVALID_ARG;
    if (slice_events && !slice_events[k]) return LCE_ERR_INVALID_ARG;
  }
  Slices sl;
  sl.n = n_slices;
  sl.bounds = slice_bounds;
  sl.events = slice_events;
  return fwd_bwd(H, W, y, N, d, V, grad_loss, loss, lse, dH, dW, opts, ws, ws_bytes, stream, &sl, sm_limit);
}

static int shard_args(int64_t V_shard, int64_t vocab_offset, int64_t V_total) {
  if (vocab_offset < 0 || V_shard <= 0 || V_total > (int64_t{1} << 31) - 1 || vocab_offset + V_shard > V_total)
    return LCE_ERR_INVALID_ARG;
  return LCE_OK;
}

int lce_vshard_forward_stats(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d,
                             int64_t V_shard, int64_t vocab_offset, int64_t V_total, float* stats,
                             const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  Call c;
  LCE_TRY(begin(&c, LCE_OP_FORWARD, H, W_shard, y, N, d, V_shard, opts, ws, ws_bytes, stream));
  LCE_TRY(shard_args(V_shard, vocab_offset, V_total));
  if (c.o.reserved != 0 || (N > 0 && !stats)) return LCE_ERR_INVALID_ARG;
  if (stats && !aligned(stats, 16)) return LCE_ERR_ALIGNMENT;
  c.V_total = V_total;
  c.y_offset = vocab_offset;
  LCE_TRY(device_check(&c.dev));
  LCE_TRY(prepare(c, nullptr));
  for (int64_t c0 = 0; c0 < N; c0 += c.L.C) {
    const int64_t rows = (N - c0) < c.L.C ? (N - c0) : c.L.C;
    LogitsArgs a;
    a.mode = lce::FWD_STATS;
    LCE_TRY(logits_gemm(c, c0, rows, a));
    const double bytes = static_cast<double>(rows) * (16.0 * static_cast<double>(c.L.T) + 8 + 4 + 16);
    LCE_TRY(timed(c.s, K_COMBINE, bytes, [&] {
      return cuda_rc(lce::launch_shard_stats(reinterpret_cast<const float2*>(c.ws + c.L.partials),
                                             static_cast<int>(2 * c.L.T), static_cast<int>(rows),
                                             reinterpret_cast<const float*>(c.ws + c.L.ztgt), c.y + c0,
                                             vocab_offset, static_cast<int>(V_shard), static_cast<int>(V_total),
                                             c.o.ignore_index, reinterpret_cast<float4*>(stats) + c0, c.s));
    }));
  }
  return finish(c);
}

int lce_vshard_combine(const float* stats, int64_t R, const int64_t* y, int64_t N, int64_t V_total, float* lse,
                       float* loss, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  Call c;
  lce_opts_init(&c.o);
  if (opts) c.o = *opts;
  LCE_TRY(check_sizes(N, 8, V_total, &c.o));
  if (R <= 0 || R > 4096 || !ws || !loss || (N > 0 && (!stats || !y || !lse)) || c.o.reserved != 0)
    return LCE_ERR_INVALID_ARG;
  if (!aligned(ws, 256) || (stats && !aligned(stats, 16)) || (lse && !aligned(lse, 4)) || !aligned(loss, 4) ||
      (y && !aligned(y, 8)))
    return LCE_ERR_ALIGNMENT;
  c.L = make_layout(LCE_OP_VSHARD_COMBINE, N, 8, V_total, &c.o);
  if (ws_bytes < c.L.total) return LCE_ERR_WORKSPACE;
  c.H = nullptr;
  c.W = nullptr;
  c.y = y;
  c.N = N;
  c.d = 8;
  c.V = V_total;
  c.V_total = V_total;
  c.ws = static_cast<uint8_t*>(ws);
  c.st = reinterpret_cast<DevStatus*>(c.ws + c.L.status);
  c.s = static_cast<cudaStream_t>(stream);
  LCE_TRY(device_check(&c.dev));
  LCE_TRY(prepare(c, nullptr));
  float* loss_i = reinterpret_cast<float*>(c.ws + c.L.loss_i);
  LCE_TRY(timed(c.s, K_COMBINE, static_cast<double>(N) * (16.0 * static_cast<double>(R) + 16), [&] {
    return cuda_rc(lce::launch_shard_merge(reinterpret_cast<const float4*>(stats), static_cast<int>(R), N, y,
                                           static_cast<int>(V_total), c.o.ignore_index, lse, loss_i, c.s));
  }));
  LCE_TRY(finalize(c, loss_i, loss));
  return finish(c);
}

int lce_vshard_backward(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d, int64_t V_shard,
                        int64_t vocab_offset, int64_t V_total, const float* lse, const float* grad_loss,
                        float* dH_partial, float* dW_shard, const lce_opts* opts, void* ws, size_t ws_bytes,
                        void* stream) {
  Call c;
  LCE_TRY(begin(&c, LCE_OP_BACKWARD, H, W_shard, y, N, d, V_shard, opts, ws, ws_bytes, stream));
  LCE_TRY(shard_args(V_shard, vocab_offset, V_total));
  if (c.o.reserved != 0 || !dW_shard || (N > 0 && (!lse || !dH_partial))) return LCE_ERR_INVALID_ARG;
  if (!aligned(dW_shard, 16) || (dH_partial && !aligned(dH_partial, 16)) || (lse && !aligned(lse, 4)) ||
      (grad_loss && !aligned(grad_loss, 4)))
    return LCE_ERR_ALIGNMENT;
  c.V_total = V_total;
  c.y_offset = vocab_offset;
  LCE_TRY(device_check(&c.dev));
  LCE_TRY(prepare(c, grad_loss));
  if (N == 0 && !c.o.accumulate_dW)
    LCE_TRY(timed(c.s, K_MEMSET, 4.0 * static_cast<double>(V_shard * d), [&] {
      return cuda_rc(cudaMemsetAsync(dW_shard, 0, sizeof(float) * static_cast<size_t>(V_shard * d), c.s));
    }));
  for (int64_t c0 = 0; c0 < N; c0 += c.L.C) {
    const int64_t rows = (N - c0) < c.L.C ? (N - c0) : c.L.C;
    LCE_TRY(backward_chunk(c, c0, rows, lse, dH_partial, dW_shard, c.o.accumulate_dW || c0 > 0, true));
  }
  return finish(c);
}

// Checks shared by the two per-chunk shard calls; fills the call record.
static int vshard_chunk_begin(Call* c, const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d,
                              int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t c0, int64_t rows,
                              const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  LCE_TRY(begin(c, LCE_OP_VSHARD_CHUNK, H, W_shard, y, N, d, V_shard, opts, ws, ws_bytes, stream));
  LCE_TRY(shard_args(V_shard, vocab_offset, V_total));
  if (c->o.reserved != 0 || c0 < 0 || rows < 0 || c0 > N - rows || rows > c->L.C) return LCE_ERR_INVALID_ARG;
  c->V_total = V_total;
  c->y_offset = vocab_offset;
  return LCE_OK;
}

int lce_vshard_chunk_stats(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d,
                           int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t c0, int64_t rows,
                           float* stats, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  Call c;
  LCE_TRY(vshard_chunk_begin(&c, H, W_shard, y, N, d, V_shard, vocab_offset, V_total, c0, rows, opts, ws, ws_bytes,
                             stream));
  if (rows > 0 && !stats) return LCE_ERR_INVALID_ARG;
  if (stats && !aligned(stats, 16)) return LCE_ERR_ALIGNMENT;
  if (rows == 0) return LCE_OK;
  LCE_TRY(device_check(&c.dev));
  LCE_TRY(prepare(c, nullptr));  // also clears the chunk's guard word
  float* ref = reinterpret_cast<float*>(c.ws + c.L.ref);
  LogitsArgs r;
  r.mode = lce::FWD_REF;
  r.ref = ref;
  LCE_TRY(logits_gemm(c, c0, rows, r));
  LogitsArgs a;
  a.mode = lce::FWD_STATS_PX;
  a.ref = ref;
  a.P = reinterpret_cast<uint16_t*>(c.ws + c.L.P);
  a.guard = reinterpret_cast<int*>(c.ws + c.L.guard);
  LCE_TRY(logits_gemm(c, c0, rows, a));
  const double bytes = static_cast<double>(rows) * (16.0 * static_cast<double>(c.L.T) + 8 + 4 + 16);
  LCE_TRY(timed(c.s, K_COMBINE, bytes, [&] {
    return cuda_rc(lce::launch_shard_stats(reinterpret_cast<const float2*>(c.ws + c.L.partials),
                                           static_cast<int>(2 * c.L.T), static_cast<int>(rows),
                                           reinterpret_cast<const float*>(c.ws + c.L.ztgt), c.y + c0, vocab_offset,
                                           static_cast<int>(V_shard), static_cast<int>(V_total), c.o.ignore_index,
                                           reinterpret_cast<float4*>(stats), c.s));
  }));
  return finish(c);
}

int lce_vshard_chunk_backward(const void* H, const void* W_shard, const int64_t* y, int64_t N, int64_t d,
                              int64_t V_shard, int64_t vocab_offset, int64_t V_total, int64_t c0, int64_t rows,
                              const float* stats_all, int64_t R, const float* grad_loss, float* lse,
                              float* dH_partial, float* dW_shard, const lce_opts* opts, void* ws, size_t ws_bytes,
                              void* stream) {
  Call c;
  LCE_TRY(vshard_chunk_begin(&c, H, W_shard, y, N, d, V_shard, vocab_offset, V_total, c0, rows, opts, ws, ws_bytes,
                             stream));
  if (R < 1 || R > 4096 || !dW_shard || (rows > 0 && (!stats_all || !lse || !dH_partial))) return LCE_ERR_INVALID_ARG;
  if (!aligned(dW_shard, 16) || (stats_all && !aligned(stats_all, 16)) || (lse && !aligned(lse, 4)) ||
      (dH_partial && !aligned(dH_partial, 16)) || (grad_loss && !aligned(grad_loss, 4)))
    return LCE_ERR_ALIGNMENT;
  if (rows == 0) return LCE_OK;
  LCE_TRY(device_check(&c.dev));
  LCE_TRY(prepare(c, grad_loss, false));  // n and g/n over all N labels; keeps the guard of the stats call
  float* alpha = reinterpret_cast<float*>(c.ws + c.L.alpha);
  int* guard = reinterpret_cast<int*>(c.ws + c.L.guard);
  uint16_t* P = reinterpret_cast<uint16_t*>(c.ws + c.L.P);
  uint16_t* Ht = reinterpret_cast<uint16_t*>(c.ws + c.L.Ht);
  const double sbytes = static_cast<double>(rows) * (16.0 * static_cast<double>(R) + 8 + 4 + 4 + 4 + 2 +
                                                     4.0 * static_cast<double>(d));
  LCE_TRY(timed(c.s, K_COMBINE, sbytes, [&] {
    return cuda_rc(lce::launch_vshard_scale(
        reinterpret_cast<const float4*>(stats_all), static_cast<int>(R), static_cast<int>(rows), c.y + c0,
        vocab_offset, static_cast<int>(V_shard), static_cast<int>(V_total), c.o.ignore_index,
        reinterpret_cast<const float*>(c.ws + c.L.ref), guard, lse + c0, alpha,
        reinterpret_cast<__nv_bfloat16*>(P), c.L.ldp, reinterpret_cast<const __nv_bfloat16*>(c.H + c0 * d),
        static_cast<int>(d), reinterpret_cast<__nv_bfloat16*>(Ht), &c.st->flags, c.s));
  }));
  // The exact gradient tile, only if the stats call found the exp tile out of range.
  LogitsArgs g;
  g.mode = lce::FWD_GRAD;
  g.lse_rows = lse + c0;
  g.P = P;
  g.only_if = guard;
  LCE_TRY(logits_gemm(c, c0, rows, g));
  LCE_TRY(dh_dw(c, c0, rows, alpha, Ht, dH_partial, dW_shard, c.o.accumulate_dW || c0 > 0, true));
  return finish(c);
}

size_t lce_rmsnorm_workspace_size(int64_t N, int64_t d) {
  if (N < 0 || d <= 0 || d % 8 != 0 || d > kNormMaxD) return 0;
  return align256(sizeof(float) * static_cast<size_t>(lce::rmsnorm_bwd_blocks(N > 0 ? N : 1)) *
                  static_cast<size_t>(d));
}

int lce_rmsnorm_forward(const void* x, const float* w, int64_t N, int64_t d, float eps, void* H, float* rstd,
                        void* stream) {
  if (N < 0 || d <= 0 || d % 8 != 0 || d > kNormMaxD || !(eps >= 0.f)) return LCE_ERR_INVALID_ARG;
  if (!w || (N > 0 && (!x || !H || !rstd))) return LCE_ERR_INVALID_ARG;
  if (!aligned(w, 16) || (x && !aligned(x, 16)) || (H && !aligned(H, 16)) || (rstd && !aligned(rstd, 4)))
    return LCE_ERR_ALIGNMENT;
  DeviceInfo dev;
  LCE_TRY(device_check(&dev));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return timed(s, K_RMSNORM_FWD, 4.0 * static_cast<double>(N * d) + 4.0 * static_cast<double>(N + d), [&] {
    return cuda_rc(lce::launch_rmsnorm_fwd(x, w, N, static_cast<int>(d), eps, H, rstd, s));
  });
}

int lce_rmsnorm_backward(const void* x, const float* w, const float* rstd, const void* dH, int64_t N, int64_t d,
                         void* dx, float* dw, void* ws, size_t ws_bytes, void* stream) {
  if (N < 0 || d <= 0 || d % 8 != 0 || d > kNormMaxD) return LCE_ERR_INVALID_ARG;
  if (!w || !dw || !ws || (N > 0 && (!x || !rstd || !dH || !dx))) return LCE_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(ws, 256) || (x && !aligned(x, 16)) || (dH && !aligned(dH, 16)) ||
      (dx && !aligned(dx, 16)) || (rstd && !aligned(rstd, 4)) || !aligned(dw, 4))
    return LCE_ERR_ALIGNMENT;
  if (ws_bytes < lce_rmsnorm_workspace_size(N, d)) return LCE_ERR_WORKSPACE;
  DeviceInfo dev;
  LCE_TRY(device_check(&dev));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return timed(s, K_RMSNORM_BWD, 6.0 * static_cast<double>(N * d) + 4.0 * static_cast<double>(N + 2 * d), [&] {
    return cuda_rc(lce::launch_rmsnorm_bwd(x, w, rstd, dH, N, static_cast<int>(d), dx, dw, static_cast<float*>(ws),
                                           s));
  });
}

int lce_norm_fwd_bwd(const void* x, const float* w_norm, float eps, const void* W, const int64_t* y, int64_t N,
                     int64_t d, int64_t V, const float* grad_loss, float* loss, float* lse, void* dx, float* dw_norm,
                     float* dW, const lce_opts* opts, void* ws, size_t ws_bytes, void* stream) {
  lce_opts o;
  lce_opts_init(&o);
  if (opts) o = *opts;
  LCE_TRY(check_sizes(N, d, V, &o));
  if (d > kNormMaxD || !(eps >= 0.f) || o.reserved != 0) return LCE_ERR_INVALID_ARG;
  if (!w_norm || !dw_norm || !ws || (N > 0 && (!x || !dx))) return LCE_ERR_INVALID_ARG;
  if (!aligned(ws, 256) || !aligned(w_norm, 16) || !aligned(dw_norm, 4) || (x && !aligned(x, 16)) ||
      (dx && !aligned(dx, 16)))
    return LCE_ERR_ALIGNMENT;
  const NormLayout L = norm_layout(N, d, V, &o);
  if (ws_bytes < L.total) return LCE_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* H = base + L.H;
  float* rstd = reinterpret_cast<float*>(base + L.rstd);
  void* dH = base + L.dH;
  LCE_TRY(lce_rmsnorm_forward(x, w_norm, N, d, eps, H, rstd, stream));
  lce_opts inner = o;
  inner.sync_check = 0;
  LCE_TRY(lce_fwd_bwd(H, W, y, N, d, V, grad_loss, loss, lse, dH, dW, &inner, ws, L.lce.total, stream));
  LCE_TRY(lce_rmsnorm_backward(x, w_norm, rstd, dH, N, d, dx, dw_norm, base + L.part, L.total - L.part, stream));
  if (!o.sync_check) return LCE_OK;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LCE_ERR_CUDA;
  int flags = 0;
  if (cudaMemcpy(&flags, base, sizeof flags, cudaMemcpyDeviceToHost) != cudaSuccess) return LCE_ERR_CUDA;
  if (flags & lce::kFlagBounds) return LCE_ERR_BOUNDS;
  if (flags & lce::kFlagTimeout) return LCE_ERR_TIMEOUT;
  if (flags & lce::kFlagLabelRange) return LCE_ERR_LABEL_RANGE;
  return LCE_OK;
}

int lce_scale_grads(void* dH, float* dW, int64_t N, int64_t d, int64_t V, const float* grad_loss, void* stream) {
  if (N < 0 || d <= 0 || d % 8 != 0 || V < 0 || !grad_loss) return LCE_ERR_INVALID_ARG;
  if ((dH && !aligned(dH, 16)) || (dW && !aligned(dW, 16)) || !aligned(grad_loss, 4)) return LCE_ERR_ALIGNMENT;
  DeviceInfo dev;
  LCE_TRY(device_check(&dev));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long nbf = dH ? N * d : 0, nf = dW ? V * d : 0;
  return timed(s, K_OTHER, 4.0 * static_cast<double>(nbf) + 8.0 * static_cast<double>(nf), [&] {
    return cuda_rc(lce::launch_scale(dH, nbf, dW, nf, grad_loss, dev.num_sms, s));
  });
}

int lce_read_device_status(const void* ws, void* stream, int* flags) {
  if (!ws || !flags) return LCE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return LCE_ERR_ALIGNMENT;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LCE_ERR_CUDA;
  int f = 0;
  if (cudaMemcpy(&f, ws, sizeof f, cudaMemcpyDeviceToHost) != cudaSuccess) return LCE_ERR_CUDA;
  *flags = f & (LCE_DEVICE_LABEL_RANGE | LCE_DEVICE_TIMEOUT);
  return LCE_OK;
}

const char* lce_status_string(int status) {
  switch (status) {
    case LCE_OK: return "ok";
    case LCE_ERR_INVALID_ARG: return "invalid argument";
    case LCE_ERR_ALIGNMENT: return "misaligned pointer";
    case LCE_ERR_WORKSPACE: return "workspace too small";
    case LCE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case LCE_ERR_CUDA: return "CUDA error";
    case LCE_ERR_LABEL_RANGE: return "label outside [0, V) and not ignore_index";
    case LCE_ERR_TIMEOUT: return "device wait timed out";
    case LCE_ERR_BOUNDS: return "index outside its buffer (bounds-checked build)";
    default: return "unknown status";
  }
}

int lce_version(void) { return LCE_VERSION; }

int lce_profile_begin(void) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.recs.clear();
  g_prof.on = true;
  return LCE_OK;
}

int lce_profile_end(lce_profile* out) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.on = false;
  lce_profile p;
  std::memset(&p, 0, sizeof p);
  int rc = LCE_OK;
  for (const ProfRecord& r : g_prof.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      rc = LCE_ERR_CUDA;
    p.launches[r.kind] += 1;
    p.ms[r.kind] += ms;
    p.work[r.kind] += r.work;
    g_prof.pool.push_back(r.start);
    g_prof.pool.push_back(r.stop);
  }
  g_prof.recs.clear();
  if (out) *out = p;
  return rc;
}

const char* lce_kernel_name(int kind) {
  return (kind >= 0 && kind < LCE_KERNEL_KINDS) ? kKindNames[kind] : nullptr;
}

}  // extern "C"
