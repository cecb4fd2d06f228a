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
// the block partials in block order, so results do not depend on scheduling.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lce_internal.h"

namespace lce {

namespace {

constexpr int kNormThreads = 256;
constexpr int kBwdRowsPerBlock = 32;

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

// Block-wide sum in a fixed order (warp butterflies, then warp 0 over the warp sums).
__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  if (w == 0) {
    t = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.f;
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  return red[0];
}

// One block per row.
__global__ void __launch_bounds__(kNormThreads) k_rmsnorm_fwd(const uint4* __restrict__ x, const float* __restrict__ w,
                                                              long long N, int d, float eps, uint4* __restrict__ H,
                                                              float* __restrict__ rstd) {
  __shared__ float red[32];
  const long long i = blockIdx.x;
  if (i >= N) return;
  const int groups = d / 8;
  const uint4* xr = x + i * groups;
  float ss = 0.f;
  for (int gI = threadIdx.x; gI < groups; gI += blockDim.x) {
    float f[8];
    unpack8(xr[gI], f);
#pragma unroll
    for (int k = 0; k < 8; ++k) ss = fmaf(f[k], f[k], ss);
  }
  const float total = block_sum(ss, red);
  const float r = rsqrtf(total / static_cast<float>(d) + eps);
  if (threadIdx.x == 0) rstd[i] = r;
  uint4* hr = H + i * groups;
  for (int gI = threadIdx.x; gI < groups; gI += blockDim.x) {
    float f[8];
    unpack8(xr[gI], f);
    const float4 w0 = reinterpret_cast<const float4*>(w)[2 * gI];
    const float4 w1 = reinterpret_cast<const float4*>(w)[2 * gI + 1];
    const float g[8] = {1.f + w0.x, 1.f + w0.y, 1.f + w0.z, 1.f + w0.w, 1.f + w1.x, 1.f + w1.y, 1.f + w1.z, 1.f + w1.w};
    uint4 o;
    o.x = pack2(f[0] * r * g[0], f[1] * r * g[1]);
    o.y = pack2(f[2] * r * g[2], f[3] * r * g[3]);
    o.z = pack2(f[4] * r * g[4], f[5] * r * g[5]);
    o.w = pack2(f[6] * r * g[6], f[7] * r * g[7]);
    hr[gI] = o;
  }
}

// Block b owns rows [b*R, b*R + R): dx for those rows, and its partial of dw
// (accumulated in shared memory, one column per thread slot) written to part[b].
__global__ void __launch_bounds__(kNormThreads) k_rmsnorm_bwd(const uint4* __restrict__ x, const float* __restrict__ w,
                                                              const float* __restrict__ rstd,
                                                              const uint4* __restrict__ dH, long long N, int d,
                                                              uint4* __restrict__ dx, float* __restrict__ part) {
  extern __shared__ float dw_acc[];  // [d]
  __shared__ float red[32];
  const int groups = d / 8;
  for (int k = threadIdx.x; k < d; k += blockDim.x) dw_acc[k] = 0.f;
  __syncthreads();
  const long long r0 = static_cast<long long>(blockIdx.x) * kBwdRowsPerBlock;
  for (int rr = 0; rr < kBwdRowsPerBlock; ++rr) {
    const long long i = r0 + rr;
    if (i >= N) break;
    const uint4* xr = x + i * groups;
    const uint4* dr = dH + i * groups;
    const float r = rstd[i];
    float c = 0.f;
    for (int gI = threadIdx.x; gI < groups; gI += blockDim.x) {
      float f[8], gd[8];
      unpack8(xr[gI], f);
      unpack8(dr[gI], gd);
      const float4 w0 = reinterpret_cast<const float4*>(w)[2 * gI];
      const float4 w1 = reinterpret_cast<const float4*>(w)[2 * gI + 1];
      const float g[8] = {1.f + w0.x, 1.f + w0.y, 1.f + w0.z, 1.f + w0.w,
                          1.f + w1.x, 1.f + w1.y, 1.f + w1.z, 1.f + w1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        c = fmaf(gd[k] * g[k], f[k], c);
        dw_acc[8 * gI + k] += gd[k] * f[k] * r;  // this thread owns these columns
      }
    }
    const float cs = block_sum(c, red) * r * r / static_cast<float>(d);
    uint4* xo = dx + i * groups;
    for (int gI = threadIdx.x; gI < groups; gI += blockDim.x) {
      float f[8], gd[8];
      unpack8(xr[gI], f);
      unpack8(dr[gI], gd);
      const float4 w0 = reinterpret_cast<const float4*>(w)[2 * gI];
      const float4 w1 = reinterpret_cast<const float4*>(w)[2 * gI + 1];
      const float g[8] = {1.f + w0.x, 1.f + w0.y, 1.f + w0.z, 1.f + w0.w,
                          1.f + w1.x, 1.f + w1.y, 1.f + w1.z, 1.f + w1.w};
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = r * (g[k] * gd[k] - f[k] * cs);
      xo[gI] = make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
    }
  }
  __syncthreads();
  float* pb = part + static_cast<long long>(blockIdx.x) * d;
  for (int k = threadIdx.x; k < d; k += blockDim.x) pb[k] = dw_acc[k];
}

// dw_k = sum over blocks b (in order) of part[b][k].
__global__ void __launch_bounds__(256) k_colsum(const float* __restrict__ part, int nblocks, int d,
                                                float* __restrict__ dw) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= d) return;
  float s = 0.f;
  for (int b = 0; b < nblocks; ++b) s += part[static_cast<long long>(b) * d + k];
  dw[k] = s;
}

}  // namespace

int rmsnorm_bwd_blocks(long long N) { return static_cast<int>((N + kBwdRowsPerBlock - 1) / kBwdRowsPerBlock); }

cudaError_t launch_rmsnorm_fwd(const void* x, const float* w, long long N, int d, float eps, void* H, float* rstd,
                               cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  k_rmsnorm_fwd<<<static_cast<unsigned>(N), kNormThreads, 0, s>>>(static_cast<const uint4*>(x), w, N, d, eps,
                                                                  static_cast<uint4*>(H), rstd);
  return cudaGetLastError();
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
    k_rmsnorm_bwd<<<nb, kNormThreads, smem, s>>>(static_cast<const uint4*>(x), w, rstd,
                                                  static_cast<const uint4*>(dH), N, d, static_cast<uint4*>(dx),
                                                  part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_colsum<<<(d + 255) / 256, 256, 0, s>>>(part, N > 0 ? nb : 0, d, dw);
  return cudaGetLastError();
}

}  // namespace lce
