// Row-wise kernels of the multi-layer path: the residual stream h (fp32, one
// row per (document, evaluated node)) through RMSNorms, the SwiGLU MLP's
// SiLU(gate) * up, and the residual adds of the k-split GEMM slabs. Every
// activation that feeds a tensor-core GEMM is written as a two-term bf16
// split [x_hi | x_lo] (hi = bf16(x), lo = bf16(x - hi)), as in the
// single-layer path.
#include <cuda_bf16.h>

#include "kernels.h"
#include "quail_internal.h"

namespace quail {

namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float row_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += scratch[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ void write_split(bf16* hi, bf16* lo, float x) {
  const bf16 h = __float2bfloat16(x);
  *hi = h;
  *lo = __float2bfloat16(x - __bfloat162float(h));
}

// h[r] = E[tokens[r]] (fp32).
__global__ void gather_embed_kernel(const bf16* __restrict__ embed, const int* __restrict__ tokens, int d,
                                    float* __restrict__ h) {
  const int r = blockIdx.x;
  const bf16* e = embed + static_cast<size_t>(__ldg(tokens + r)) * d;
  float* out = h + static_cast<size_t>(r) * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) out[i] = __bfloat162float(e[i]);
}

// h[r] += sum of the ks slabs (when ks > 0); then, when out != null,
// out[r] = split(RMSNorm(h[r]) * gain) as [hi (d) | lo (d)].
__global__ void residual_norm_kernel(float* __restrict__ h, const float* __restrict__ part, int ks, size_t slab,
                                     int d, const bf16* __restrict__ gain, float eps, bf16* __restrict__ out) {
  __shared__ float scratch[32];
  const int r = blockIdx.x;
  float* hr = h + static_cast<size_t>(r) * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float x = hr[i];
    for (int s = 0; s < ks; ++s) x += part[s * slab + static_cast<size_t>(r) * d + i];
    if (ks > 0) hr[i] = x;
    ss += x * x;
  }
  if (out == nullptr) return;
  const float inv = rsqrtf(row_sum(ss, scratch) / d + eps);
  bf16* o = out + static_cast<size_t>(r) * 2 * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x)
    write_split(o + i, o + d + i, hr[i] * inv * __bfloat162float(gain[i]));
}

// act[r] = split(SiLU(g) * u), g = sum of slabs [:, 0:I), u = [:, I:2I).
__global__ void silu_mul_split_kernel(const float* __restrict__ part, int ks, size_t slab, int rows, int I,
                                      bf16* __restrict__ act) {
  const size_t n = static_cast<size_t>(rows) * I;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = idx / I, c = idx % I;
    float g = 0.f, u = 0.f;
    for (int s = 0; s < ks; ++s) {
      const float* p = part + s * slab + r * 2 * I;
      g += p[c];
      u += p[I + c];
    }
    const float a = g / (1.f + expf(-g)) * u;
    bf16* o = act + r * 2 * I;
    write_split(o + c, o + I + c, a);
  }
}

// z[r] = RMSNorm(h[r]) * gain as bf16 and (when z_f32) fp32.
__global__ void norm_out_kernel(const float* __restrict__ h, int d, const bf16* __restrict__ gain, float eps,
                                bf16* __restrict__ z, float* __restrict__ z_f32) {
  __shared__ float scratch[32];
  const int r = blockIdx.x;
  const float* hr = h + static_cast<size_t>(r) * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) ss += hr[i] * hr[i];
  const float inv = rsqrtf(row_sum(ss, scratch) / d + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float y = hr[i] * inv * __bfloat162float(gain[i]);
    z[static_cast<size_t>(r) * d + i] = __float2bfloat16(y);
    if (z_f32) z_f32[static_cast<size_t>(r) * d + i] = y;
  }
}

}  // namespace

cudaError_t launch_gather_embed(const bf16* embed, const int* tokens, int rows, int d, float* h, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  gather_embed_kernel<<<rows, kRowThreads, 0, st>>>(embed, tokens, d, h);
  return cudaGetLastError();
}

cudaError_t launch_residual_norm(float* h, const float* part, int ks, size_t slab, int rows, int d, const bf16* gain,
                                 float eps, bf16* out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  residual_norm_kernel<<<rows, kRowThreads, 0, st>>>(h, part, ks, slab, d, gain, eps, out);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_split(const float* part, int ks, size_t slab, int rows, int I, bf16* act,
                                  cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const size_t n = static_cast<size_t>(rows) * I;
  const int blocks = static_cast<int>((n + kRowThreads - 1) / kRowThreads < 4096 ? (n + kRowThreads - 1) / kRowThreads
                                                                                  : 4096);
  count_launch();
  silu_mul_split_kernel<<<blocks, kRowThreads, 0, st>>>(part, ks, slab, rows, I, act);
  return cudaGetLastError();
}

cudaError_t launch_norm_out(const float* h, int rows, int d, const bf16* gain, float eps, bf16* z, float* z_f32,
                            cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  norm_out_kernel<<<rows, kRowThreads, 0, st>>>(h, d, gain, eps, z, z_f32);
  return cudaGetLastError();
}

}  // namespace quail
