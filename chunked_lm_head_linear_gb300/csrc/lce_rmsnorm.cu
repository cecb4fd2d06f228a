// The final zero-centred RMSNorm in front of the LM head, forward and backward
// ("XTuner on Ascend 910C: Qwen3.5-2B training optimisation", section 3.1.1:
// one pass over the bf16 input, the (1 + w) scale folded into an fp32 gamma,
// a single bf16 rounding of the output):
//
//   r_i   = 1 / sqrt(mean_k x_ik^2 + eps)
//   H_ik  = bf16(x_ik r_i (1 + w_k))
//   dx_ik = r_i ((1 + w_k) dH_ik - x_ik r_i^2 c_i / d),  c_i = sum_k dH_ik (1 + w_k) x_ik
//   dw_k  = sum_i dH_ik x_ik r_i
//
// Both kernels are HBM-bound (a few bytes per element) and read rows with
// 16-byte vector loads. dw is summed in a fixed order: each block owns a fixed
// set of rows and writes one partial row per block, and a second kernel adds
// the block partials in a fixed two-level order, so results do not depend on
// scheduling.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lce_internal.h"

namespace lce {

namespace {

constexpr int kNormThreads = 256;
constexpr int kFwdBlocksPerSm = 2;                    // persistent grid of the forward
constexpr int kFwdRegGroups = 8;                      // 16-byte groups a lane keeps in registers (d <= 2048)
constexpr int kBwdRowsPerBlock = 16;
constexpr int kBwdRowGroup = 4;                       // rows reduced together (one set of block barriers)
constexpr int kColsumWarps = 32;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void gamma8(const float* __restrict__ w, int gI, float (&g)[8]) {
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * gI);
  const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * gI + 1);
  g[0] = 1.f + w0.x; g[1] = 1.f + w0.y; g[2] = 1.f + w0.z; g[3] = 1.f + w0.w;
  g[4] = 1.f + w1.x; g[5] = 1.f + w1.y; g[6] = 1.f + w1.z; g[7] = 1.f + w1.w;
}

__device__ __forceinline__ uint4 norm8(const uint4& xv, const float (&g)[8], float r) {
  float f[8];
  unpack8(xv, f);
  return make_uint4(pack2(f[0] * r * g[0], f[1] * r * g[1]), pack2(f[2] * r * g[2], f[3] * r * g[3]),
                    pack2(f[4] * r * g[4], f[5] * r * g[5]), pack2(f[6] * r * g[6], f[7] * r * g[7]));
}

// Persistent warps: warp u of the grid normalises rows u, u + U, ... (U warps
// in all), loading the next row while it finishes the current one. Lane l
// owns the 16-byte groups l, l + 32, ... of a row; the first kFwdRegGroups of
// them stay in registers between the two passes, the rest (rows longer than
// 2048) are read again.
__device__ __forceinline__ void load_row(const uint4* __restrict__ xr, int groups, int lane, bool on,
                                         uint4 (&v)[kFwdRegGroups]) {
#pragma unroll
  for (int j = 0; j < kFwdRegGroups; ++j) {
    const int gI = lane + 32 * j;
    v[j] = (on && gI < groups) ? xr[gI] : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(kNormThreads, 2) k_rmsnorm_fwd(const uint4* __restrict__ x, const float* __restrict__ w,
                                                                 long long N, int d, float eps, uint4* __restrict__ H,
                                                                 float* __restrict__ rstd) {
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const long long U = static_cast<long long>(gridDim.x) * (kNormThreads / 32);
  long long i = static_cast<long long>(blockIdx.x) * (kNormThreads / 32) + (threadIdx.x >> 5);
  const int groups = d / 8;
  uint4 cur[kFwdRegGroups], nxt[kFwdRegGroups];
  load_row(x + (i < N ? i : 0) * groups, groups, lane, i < N, cur);
  for (; i < N; i += U) {
    const bool more = i + U < N;
    load_row(x + (more ? i + U : i) * groups, groups, lane, more, nxt);
    const uint4* xr = x + i * groups;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kFwdRegGroups; ++j) {
      float f[8];
      unpack8(cur[j], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(f[k], f[k], ss);
    }
    for (int gI = lane + 32 * kFwdRegGroups; gI < groups; gI += 32) {
      float f[8];
      unpack8(xr[gI], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(f[k], f[k], ss);
    }
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = rsqrtf(ss / static_cast<float>(d) + eps);
    if (lane == 0) rstd[i] = r;
    uint4* hr = H + i * groups;
#pragma unroll
    for (int j = 0; j < kFwdRegGroups; ++j) {
      const int gI = lane + 32 * j;
      if (gI < groups) {
        float g[8];
        gamma8(w, gI, g);
        hr[gI] = norm8(cur[j], g, r);
      }
    }
    for (int gI = lane + 32 * kFwdRegGroups; gI < groups; gI += 32) {
      float g[8];
      gamma8(w, gI, g);
      hr[gI] = norm8(xr[gI], g, r);
    }
#pragma unroll
    for (int j = 0; j < kFwdRegGroups; ++j) cur[j] = nxt[j];
  }
}

// Block b owns rows [b*R, b*R + R), taken kBwdRowGroup at a time: thread t
// owns the 16-byte column groups t, t + 256, ... of every row, so its share of
// dw (in shared memory) has no other writer. Per row group: c_i for the group's
// rows (one block reduction for all of them), then dx and the dw terms. A
// thread's first column group of each row stays in registers between the two
// passes (the whole row when d <= 2048); further groups are read again. The
// block's dw partial row goes to part[b].
__global__ void __launch_bounds__(kNormThreads, 3) k_rmsnorm_bwd(const uint4* __restrict__ x, const float* __restrict__ w,
                                                              const float* __restrict__ rstd,
                                                              const uint4* __restrict__ dH, long long N, int d,
                                                              uint4* __restrict__ dx, float* __restrict__ part) {
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ float dw_acc[];  // [d]
  __shared__ float red[kNormThreads / 32][kBwdRowGroup];
  __shared__ float cs_row[kBwdRowGroup];
  const int groups = d / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g0 = threadIdx.x;  // the column group kept in registers
  for (int k = threadIdx.x; k < d; k += blockDim.x) dw_acc[k] = 0.f;
  const long long r0 = static_cast<long long>(blockIdx.x) * kBwdRowsPerBlock;
  for (int rr = 0; rr < kBwdRowsPerBlock; rr += kBwdRowGroup) {
    if (r0 + rr >= N) break;
    const int nq = static_cast<int>((N - r0 - rr) < kBwdRowGroup ? (N - r0 - rr) : kBwdRowGroup);
    uint4 xv[kBwdRowGroup], gv[kBwdRowGroup];
    float c[kBwdRowGroup];
    float r[kBwdRowGroup];
#pragma unroll
    for (int q = 0; q < kBwdRowGroup; ++q) {
      const long long i = r0 + rr + q;
      const bool on = q < nq && g0 < groups;
      xv[q] = on ? x[i * groups + g0] : make_uint4(0u, 0u, 0u, 0u);
      gv[q] = on ? dH[i * groups + g0] : make_uint4(0u, 0u, 0u, 0u);
      r[q] = q < nq ? rstd[i] : 0.f;
      c[q] = 0.f;
    }
    if (g0 < groups) {
      float g[8];
      gamma8(w, g0, g);
#pragma unroll
      for (int q = 0; q < kBwdRowGroup; ++q) {
        float f[8], gd[8];
        unpack8(xv[q], f);
        unpack8(gv[q], gd);
#pragma unroll
        for (int k = 0; k < 8; ++k) c[q] = fmaf(gd[k] * g[k], f[k], c[q]);
      }
    }
    for (int gI = g0 + kNormThreads; gI < groups; gI += kNormThreads) {
      float g[8];
      gamma8(w, gI, g);
#pragma unroll
      for (int q = 0; q < kBwdRowGroup; ++q) {
        if (q < nq) {
          const long long i = r0 + rr + q;
          float f[8], gd[8];
          unpack8(x[i * groups + gI], f);
          unpack8(dH[i * groups + gI], gd);
#pragma unroll
          for (int k = 0; k < 8; ++k) c[q] = fmaf(gd[k] * g[k], f[k], c[q]);
        }
      }
    }
    // block sums of the group's c values, in a fixed order
#pragma unroll
    for (int q = 0; q < kBwdRowGroup; ++q)
      for (int off = 16; off > 0; off >>= 1) c[q] += __shfl_xor_sync(0xffffffffu, c[q], off);
    __syncthreads();  // the previous group's readers of red / cs_row are done
    if (lane == 0)
#pragma unroll
      for (int q = 0; q < kBwdRowGroup; ++q) red[warp][q] = c[q];
    __syncthreads();
    if (threadIdx.x < nq) {
      float t = 0.f;
      for (int k = 0; k < kNormThreads / 32; ++k) t += red[k][threadIdx.x];
      const float rq = rstd[r0 + rr + threadIdx.x];
      cs_row[threadIdx.x] = t * rq * rq / static_cast<float>(d);
    }
    __syncthreads();
    for (int gI = g0; gI < groups; gI += kNormThreads) {
      const bool cached = gI == g0;
      float g[8];
      gamma8(w, gI, g);
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = dw_acc[8 * gI + k];
#pragma unroll
      for (int q = 0; q < kBwdRowGroup; ++q) {
        if (q < nq) {
          const long long i = r0 + rr + q;
          float f[8], gd[8], o[8];
          unpack8(cached ? xv[q] : x[i * groups + gI], f);
          unpack8(cached ? gv[q] : dH[i * groups + gI], gd);
          const float cs = cs_row[q];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            o[k] = r[q] * (g[k] * gd[k] - f[k] * cs);
            acc[k] += gd[k] * f[k] * r[q];
          }
          dx[i * groups + gI] = make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) dw_acc[8 * gI + k] = acc[k];
    }
  }
  __syncthreads();
  float* pb = part + static_cast<long long>(blockIdx.x) * d;
  for (int k = threadIdx.x; k < d; k += blockDim.x) pb[k] = dw_acc[k];
}

// dw_k = sum over blocks b of part[b][k]: a block covers 32 columns with
// kColsumWarps warps; warp s sums the partial rows b = s, s + kColsumWarps, ...
// in order, then the warp sums are added in warp order.
__global__ void __launch_bounds__(32 * kColsumWarps) k_colsum(const float* __restrict__ part, int nblocks, int d,
                                                              float* __restrict__ dw) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float red[kColsumWarps][33];
  const int lane = threadIdx.x & 31, s = threadIdx.x >> 5;
  const int k = blockIdx.x * 32 + lane;
  float t = 0.f;
  if (k < d)
    for (int b = s; b < nblocks; b += kColsumWarps) t += part[static_cast<long long>(b) * d + k];
  red[s][lane] = t;
  __syncthreads();
  if (s == 0 && k < d) {
    float u = 0.f;
    for (int q = 0; q < kColsumWarps; ++q) u += red[q][lane];
    dw[k] = u;
  }
}

}  // namespace

int rmsnorm_bwd_blocks(long long N) { return static_cast<int>((N + kBwdRowsPerBlock - 1) / kBwdRowsPerBlock); }

cudaError_t launch_rmsnorm_fwd(const void* x, const float* w, long long N, int d, float eps, void* H, float* rstd,
                               cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long need = (N + kNormThreads / 32 - 1) / (kNormThreads / 32);
  const long long blocks = need < static_cast<long long>(kFwdBlocksPerSm) * sms ? need : kFwdBlocksPerSm * sms;
  return launch_k(k_rmsnorm_fwd, static_cast<unsigned>(blocks), kNormThreads, 0, s, static_cast<const uint4*>(x), w,
                  N, d, eps, static_cast<uint4*>(H), rstd);
}

cudaError_t launch_rmsnorm_bwd(const void* x, const float* w, const float* rstd, const void* dH, long long N, int d,
                               void* dx, float* dw, float* part, cudaStream_t s) {
  const int nb = rmsnorm_bwd_blocks(N);
  if (N > 0) {
    const size_t smem = sizeof(float) * static_cast<size_t>(d);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(k_rmsnorm_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_k(k_rmsnorm_bwd, nb, kNormThreads, smem, s, static_cast<const uint4*>(x), w, rstd,
                                   static_cast<const uint4*>(dH), N, d, static_cast<uint4*>(dx), part);
    if (e != cudaSuccess) return e;
  }
  return launch_k(k_colsum, (d + 31) / 32, 32 * kColsumWarps, 0, s, part, N > 0 ? nb : 0, d, dw);
}

}  // namespace lce
