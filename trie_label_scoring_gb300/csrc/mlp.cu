// Row-wise kernels of the multi-layer path: the residual stream h (fp32, one
// row per (document, evaluated node)) through RMSNorms, the SwiGLU MLP's
// SiLU(gate) * up, and the residual adds of the k-split GEMM slabs. Every
// activation that feeds a tensor-core GEMM is written as a two-term bf16
// split [x_hi | x_lo] (hi = bf16(x), lo = bf16(x - hi)), as in the
// single-layer path.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "launch.cuh"
#include "quail_internal.h"

namespace quail {

namespace {

constexpr int kRowThreads = 256;
constexpr int kRowMaxVec = 12;  // float4 vectors per thread: d <= 4 * 256 * 12 = 12288

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

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 u) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// The two-term split of 4 values: hi = bf16(y), lo = bf16(y - hi).
__device__ __forceinline__ void split4(float4 y, uint2* hi, uint2* lo) {
  const uint2 h = make_uint2(pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
  const float4 hf = bf16x4_to_f4(h);
  *hi = h;
  *lo = make_uint2(pack_bf16x2(y.x - hf.x, y.y - hf.y), pack_bf16x2(y.z - hf.z, y.w - hf.w));
}

// h[r] = E[tokens[r]] (fp32).
__global__ void gather_embed_kernel(const bf16* __restrict__ embed, const int* __restrict__ tokens, int d,
                                    float* __restrict__ h) {
  grid_dependency_wait();
  const int r = blockIdx.x;
  const uint2* e = reinterpret_cast<const uint2*>(embed + static_cast<size_t>(__ldg(tokens + r)) * d);
  float4* out = reinterpret_cast<float4*>(h + static_cast<size_t>(r) * d);
  for (int c = threadIdx.x; c < (d >> 2); c += blockDim.x) out[c] = bf16x4_to_f4(__ldg(e + c));
}

// Block per row, the row in registers: h[r] += the KS k-split slabs (all
// loaded in one memory round trip); then, when out != null,
// out[r] = split(RMSNorm(h[r]) * gain) as [hi (d) | lo (d)].
template <int KS>
__global__ void __launch_bounds__(kRowThreads) residual_norm_kernel(float* __restrict__ h,
                                                                     const float* __restrict__ part, size_t slab,
                                                                     int d, const bf16* __restrict__ gain, float eps,
                                                                     bf16* __restrict__ out) {
  grid_dependency_wait();
  __shared__ float scratch[32];
  const int r = blockIdx.x;
  float4* hr = reinterpret_cast<float4*>(h + static_cast<size_t>(r) * d);
  const float4* pr = reinterpret_cast<const float4*>(part + static_cast<size_t>(r) * d);
  const size_t slab4 = slab >> 2;
  const int nv = d >> 2;
  float4 v[kRowMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kRowMaxVec; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nv) {
      float4 p[KS > 0 ? KS : 1];
#pragma unroll
      for (int s = 0; s < KS; ++s) p[s] = pr[s * slab4 + c];
      a = hr[c];
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        a.x += p[s].x;
        a.y += p[s].y;
        a.z += p[s].z;
        a.w += p[s].w;
      }
      if (KS > 0) hr[c] = a;
    }
    v[i] = a;
    ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
  }
  if (out == nullptr) return;
  const float inv = rsqrtf(row_sum(ss, scratch) / d + eps);
  const uint2* gv = reinterpret_cast<const uint2*>(gain);
  uint2* o = reinterpret_cast<uint2*>(out + static_cast<size_t>(r) * 2 * d);
#pragma unroll
  for (int i = 0; i < kRowMaxVec; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    if (c >= nv) break;
    const float4 g = bf16x4_to_f4(__ldg(gv + c));
    split4(make_float4(v[i].x * inv * g.x, v[i].y * inv * g.y, v[i].z * inv * g.z, v[i].w * inv * g.w), o + c,
           o + nv + c);
  }
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

// act[r] = split(SiLU(g) * u), g = sum of the KS slabs [:, 0:I), u = [:, I:2I);
// one float4 of g and of u per thread, every slab loaded before the sums.
template <int KS>
__global__ void silu_mul_split_kernel(const float* __restrict__ part, size_t slab, int rows, int I,
                                      bf16* __restrict__ act) {
  grid_dependency_wait();
  const int iv = I >> 2;
  const size_t n = static_cast<size_t>(rows) * iv;
  const size_t slab4 = slab >> 2;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = idx / iv, c = idx % iv;
    const float4* p = reinterpret_cast<const float4*>(part) + r * 2 * iv + c;
    float4 g[KS], u[KS];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      g[s] = p[s * slab4];
      u[s] = p[s * slab4 + iv];
    }
#pragma unroll
    for (int s = 1; s < KS; ++s) {
      g[0].x += g[s].x;
      g[0].y += g[s].y;
      g[0].z += g[s].z;
      g[0].w += g[s].w;
      u[0].x += u[s].x;
      u[0].y += u[s].y;
      u[0].z += u[s].z;
      u[0].w += u[s].w;
    }
    const float4 a = make_float4(silu(g[0].x) * u[0].x, silu(g[0].y) * u[0].y, silu(g[0].z) * u[0].z,
                                 silu(g[0].w) * u[0].w);
    uint2* o = reinterpret_cast<uint2*>(act) + r * 2 * iv;
    split4(a, o + c, o + iv + c);
  }
}

// z[r] = RMSNorm(h[r]) * gain as bf16 and (when z_f32) fp32.
__global__ void __launch_bounds__(kRowThreads) norm_out_kernel(const float* __restrict__ h, int d,
                                                                const bf16* __restrict__ gain, float eps,
                                                                bf16* __restrict__ z, float* __restrict__ z_f32) {
  grid_dependency_wait();
  __shared__ float scratch[32];
  const int r = blockIdx.x;
  const float4* hr = reinterpret_cast<const float4*>(h + static_cast<size_t>(r) * d);
  const int nv = d >> 2;
  float4 v[kRowMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kRowMaxVec; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    v[i] = c < nv ? hr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  }
  const float inv = rsqrtf(row_sum(ss, scratch) / d + eps);
  const uint2* gv = reinterpret_cast<const uint2*>(gain);
  uint2* zb = reinterpret_cast<uint2*>(z + static_cast<size_t>(r) * d);
  float4* zf = z_f32 ? reinterpret_cast<float4*>(z_f32 + static_cast<size_t>(r) * d) : nullptr;
#pragma unroll
  for (int i = 0; i < kRowMaxVec; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    if (c >= nv) break;
    const float4 g = bf16x4_to_f4(__ldg(gv + c));
    const float4 y = make_float4(v[i].x * inv * g.x, v[i].y * inv * g.y, v[i].z * inv * g.z, v[i].w * inv * g.w);
    zb[c] = make_uint2(pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
    if (zf) zf[c] = y;
  }
}

}  // namespace

cudaError_t launch_gather_embed(const bf16* embed, const int* tokens, int rows, int d, float* h, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(gather_embed_kernel, dim3(rows), dim3(kRowThreads), 0, st, embed, tokens, d, h); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_residual_norm(float* h, const float* part, int ks, size_t slab, int rows, int d, const bf16* gain,
                                 float eps, bf16* out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (d % 4 != 0 || d > 4 * kRowThreads * kRowMaxVec || slab % 4 != 0) return cudaErrorInvalidValue;
  switch (ks) {
#define QUAIL_RESIDUAL_NORM(KS)                                                                   \
  case KS:                                                                                        \
    count_launch();                                                                               \
    { const cudaError_t le_ = launch_pdl(residual_norm_kernel<KS>, dim3(rows), dim3(kRowThreads), 0, st, h, part, slab, d, gain, eps, out); if (le_ != cudaSuccess) return le_; }     \
    break;
    QUAIL_RESIDUAL_NORM(0)
    QUAIL_RESIDUAL_NORM(1)
    QUAIL_RESIDUAL_NORM(2)
    QUAIL_RESIDUAL_NORM(3)
    QUAIL_RESIDUAL_NORM(4)
    QUAIL_RESIDUAL_NORM(5)
    QUAIL_RESIDUAL_NORM(6)
    QUAIL_RESIDUAL_NORM(7)
    QUAIL_RESIDUAL_NORM(8)
#undef QUAIL_RESIDUAL_NORM
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_split(const float* part, int ks, size_t slab, int rows, int I, bf16* act,
                                  cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (I % 4 != 0 || slab % 4 != 0) return cudaErrorInvalidValue;
  const size_t n = static_cast<size_t>(rows) * (I / 4);
  const int blocks = static_cast<int>(std::min<size_t>((n + kRowThreads - 1) / kRowThreads, 1u << 16));
  switch (ks) {
#define QUAIL_SILU_MUL(KS)                                                                 \
  case KS:                                                                                 \
    count_launch();                                                                        \
    { const cudaError_t le_ = launch_pdl(silu_mul_split_kernel<KS>, dim3(blocks), dim3(kRowThreads), 0, st, part, slab, rows, I, act); if (le_ != cudaSuccess) return le_; }   \
    break;
    QUAIL_SILU_MUL(1)
    QUAIL_SILU_MUL(2)
    QUAIL_SILU_MUL(3)
    QUAIL_SILU_MUL(4)
    QUAIL_SILU_MUL(5)
    QUAIL_SILU_MUL(6)
    QUAIL_SILU_MUL(7)
    QUAIL_SILU_MUL(8)
#undef QUAIL_SILU_MUL
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_norm_out(const float* h, int rows, int d, const bf16* gain, float eps, bf16* z, float* z_f32,
                            cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(norm_out_kernel, dim3(rows), dim3(kRowThreads), 0, st, h, d, gain, eps, z, z_f32); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

}  // namespace quail
