// Row-wise kernels of the answer-position layer and the label scoring:
// RMSNorms, log-sum-exp reduction, label path sums and softmax
// ("To Classify, Try a Trie Tree", sec. 3.2), the letters head (sec. 3.3) and
// the trie_decode step bookkeeping (sec. 3.1).
#include <cfloat>

#include "kernels.h"
#include "launch.cuh"
#include "quail_internal.h"

namespace quail {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide sum for blockDim.x <= 1024 (multiple of 32).
__device__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float t = (threadIdx.x < nw) ? scratch[threadIdx.x] : 0.f;
  if (w == 0) t = warp_sum(t);
  if (threadIdx.x == 0) scratch[0] = t;
  __syncthreads();
  return scratch[0];
}

constexpr int kNormThreads = 256;
constexpr int kNormMaxVec = 12;  // float4 / 8-bf16 vectors per thread: d <= 4 * 256 * 12 = 12288

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 u) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ uint32_t f2_to_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Block per row; the row stays in registers between the two passes; 8-byte
// vector accesses. Output: [hi | lo] two-term bf16 split of RMSNorm(x) * gain.
__global__ void __launch_bounds__(kNormThreads) embed_rmsnorm_kernel(const bf16* __restrict__ embed,
                                                                     const int* __restrict__ tokens, int d,
                                                                     const bf16* __restrict__ gain, float eps,
                                                                     bf16* __restrict__ out,
                                                                     const int* __restrict__ live) {
  grid_dependency_wait();
  if (live != nullptr && static_cast<int>(blockIdx.x) >= *live) return;
  __shared__ float scratch[32];
  const int r = blockIdx.x;
  const uint2* x = reinterpret_cast<const uint2*>(embed + static_cast<size_t>(__ldg(tokens + r)) * d);
  const int nv = d >> 2;
  float4 v[kNormMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    v[i] = c < nv ? bf16x4_to_float4(__ldg(x + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  }
  const float inv = rsqrtf(block_sum(ss, scratch) / d + eps);
  const uint2* gv = reinterpret_cast<const uint2*>(gain);
  uint2* ohi = reinterpret_cast<uint2*>(out + static_cast<size_t>(r) * 2 * d);
  uint2* olo = reinterpret_cast<uint2*>(out + static_cast<size_t>(r) * 2 * d + d);
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    if (c >= nv) break;
    const float4 g = bf16x4_to_float4(__ldg(gv + c));
    const float y0 = v[i].x * inv * g.x, y1 = v[i].y * inv * g.y, y2 = v[i].z * inv * g.z, y3 = v[i].w * inv * g.w;
    const uint2 hi = make_uint2(f2_to_bf16x2(y0, y1), f2_to_bf16x2(y2, y3));
    const float4 h = bf16x4_to_float4(hi);
    ohi[c] = hi;
    olo[c] = make_uint2(f2_to_bf16x2(y0 - h.x, y1 - h.y), f2_to_bf16x2(y2 - h.z, y3 - h.w));
  }
}

// One warp per (row, head) of 128 values: sum the k-split slabs, then the
// per-head RMSNorm for q and k heads (v heads are only summed).
__global__ void qk_head_norm_kernel(const float* __restrict__ part, int k_splits, size_t slab, float* qkv, int rows,
                                    int ld, int hq, int hkv, const bf16* __restrict__ gq,
                                    const bf16* __restrict__ gk, float eps, const int* __restrict__ live) {
  grid_dependency_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (live != nullptr) rows = min(rows, *live);
  const int lane = threadIdx.x & 31;
  const int heads = hq + 2 * hkv;
  if (warp >= rows * heads) return;
  const int r = warp / heads, h = warp % heads;
  const size_t off = static_cast<size_t>(r) * ld + h * 128 + lane * 4;
  // every slab's load issued before the first add (k_splits <= 8)
  float4 w[8];
#pragma unroll
  for (int s = 0; s < 8; ++s)
    if (s < k_splits) w[s] = *reinterpret_cast<const float4*>(part + s * slab + off);
  float4 v = w[0];
#pragma unroll
  for (int s = 1; s < 8; ++s) {
    if (s < k_splits) {
      v.x += w[s].x;
      v.y += w[s].y;
      v.z += w[s].z;
      v.w += w[s].w;
    }
  }
  if (h < hq + hkv) {
    const float inv = rsqrtf(warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w) / 128.f + eps);
    const bf16* g = (h < hq ? gq : gk) + lane * 4;
    v.x *= inv * __bfloat162float(g[0]);
    v.y *= inv * __bfloat162float(g[1]);
    v.z *= inv * __bfloat162float(g[2]);
    v.w *= inv * __bfloat162float(g[3]);
  }
  *reinterpret_cast<float4*>(qkv + off) = v;
}

// Block per row: h = x + sum of the k-split slabs, kept in registers; z in bf16
// (and fp32 when z_f32 is given). float4 / 8-byte vector accesses.
template <int KS>
__global__ void __launch_bounds__(kNormThreads) final_norm_kernel(const float* __restrict__ h_part, size_t slab,
                                                                  const bf16* __restrict__ embed,
                                                                  const int* __restrict__ node_token, RowMap map,
                                                                  int d, const bf16* __restrict__ gain, float eps,
                                                                  bf16* __restrict__ z_bf16,
                                                                  float* __restrict__ z_f32) {
  grid_dependency_wait();
  __shared__ float scratch[32];
  const int r = blockIdx.x;
  const int slot = r / map.nq;
  if (map.n_slots_dev != nullptr && slot >= *map.n_slots_dev) return;
  const int e = r - slot * map.nq;
  const int node =
      map.slot_node ? map.slot_node[slot] : slot * map.slot_stride + (map.row_nodes ? map.row_nodes[e] : e);
  const uint2* x = reinterpret_cast<const uint2*>(embed + static_cast<size_t>(__ldg(node_token + node)) * d);
  const float4* hp = reinterpret_cast<const float4*>(h_part + static_cast<size_t>(r) * d);
  const size_t slab4 = slab >> 2;
  const int nv = d >> 2;
  // per vector: the residual and the KS k-split slabs are loaded together
  // (one memory round trip), then summed
  float4 v[kNormMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nv) {
      float4 p[KS];
#pragma unroll
      for (int s = 0; s < KS; ++s) p[s] = hp[s * slab4 + c];
      a = bf16x4_to_float4(__ldg(x + c));
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        a.x += p[s].x;
        a.y += p[s].y;
        a.z += p[s].z;
        a.w += p[s].w;
      }
    }
    v[i] = a;
    ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
  }
  const float inv = rsqrtf(block_sum(ss, scratch) / d + eps);
  const uint2* gv = reinterpret_cast<const uint2*>(gain);
  uint2* zb = reinterpret_cast<uint2*>(z_bf16 + static_cast<size_t>(r) * d);
  float4* zf = z_f32 ? reinterpret_cast<float4*>(z_f32 + static_cast<size_t>(r) * d) : nullptr;
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    if (c >= nv) break;
    const float4 g = bf16x4_to_float4(__ldg(gv + c));
    const float4 y = make_float4(v[i].x * inv * g.x, v[i].y * inv * g.y, v[i].z * inv * g.z, v[i].w * inv * g.w);
    zb[c] = make_uint2(f2_to_bf16x2(y.x, y.y), f2_to_bf16x2(y.z, y.w));
    if (zf) zf[c] = y;
  }
}

// One warp per row: max over the tile partials, then the rescaled sum.
__global__ void lse_reduce_kernel(const float2* __restrict__ part, int rows, int n_tiles, float* __restrict__ lse,
                                  const int* __restrict__ live) {
  grid_dependency_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows || (live != nullptr && warp >= *live)) return;
  const float2* p = part + static_cast<size_t>(warp) * n_tiles;
  float m = -INFINITY;
#pragma unroll 4
  for (int j = lane; j < n_tiles; j += 32) m = fmaxf(m, p[j].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
#pragma unroll 4
  for (int j = lane; j < n_tiles; j += 32) {
    const float2 v = p[j];
    s += v.y * exp2f(v.x - m);
  }
  s = warp_sum(s);
  if (lane == 0) lse[warp] = (m + log2f(s)) * 0.69314718055994531f;
}

// One block per document; warp per label.
//   logscore_m = sum_{k <= d_m} (logit(p_{k-1}, x_k) - LSE(p_{k-1}))
//              + [prefix label] log(1 - sum_c exp(logit(end, c) - LSE(end)))
//   prob = softmax over labels; argmax = lowest index of the maximum.
__global__ void label_score_kernel(LabelScoreArgs a) {
  grid_dependency_wait();
  __shared__ float s_max[32];
  __shared__ int s_arg[32];
  __shared__ float s_sum[32];
  const int doc = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float* cl = a.child_logit + static_cast<size_t>(doc) * a.n_child;
  float* lse = a.lse + static_cast<size_t>(doc) * a.a;
  // log-sum-exp of this document's a rows from the head's tile partials (warp per row)
  for (int e = warp; e < a.a; e += nw) {
    const float2* p = a.lse_part + (static_cast<size_t>(doc) * a.a + e) * a.n_tiles;
    float m = -INFINITY;
#pragma unroll 4
    for (int j = lane; j < a.n_tiles; j += 32) m = fmaxf(m, p[j].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sm = 0.f;
#pragma unroll 4
    for (int j = lane; j < a.n_tiles; j += 32) {
      const float2 v = p[j];
      sm += v.y * exp2f(v.x - m);
    }
    sm = warp_sum(sm);
    if (lane == 0) lse[e] = (m + log2f(sm)) * 0.69314718055994531f;
  }
  __syncthreads();
  float* out_ls = a.logscore + static_cast<size_t>(doc) * a.M;
  float best = -INFINITY;
  int best_i = 0x7fffffff;
  for (int m = warp; m < a.M; m += nw) {
    const int t0 = __ldg(a.term_offsets + m), t1 = __ldg(a.term_offsets + m + 1);
    float acc = 0.f;
    for (int t = t0 + lane; t < t1; t += 32) acc += cl[__ldg(a.term_slot + t)] - lse[__ldg(a.term_eval + t)];
    acc = warp_sum(acc);
    const int pe = __ldg(a.prefix_eval + m);
    if (pe >= 0) {  // prefix label: probability of stopping at its end node
      const int c0 = __ldg(a.eval_child_offsets + pe), c1 = __ldg(a.eval_child_offsets + pe + 1);
      double cont = 0.0;
      for (int c = c0 + lane; c < c1; c += 32) cont += exp(static_cast<double>(cl[c]) - static_cast<double>(lse[pe]));
      cont = warp_sum_d(cont);
      acc = (cont < 1.0 - 1e-12) ? acc + static_cast<float>(log1p(-cont)) : -INFINITY;
    }
    if (lane == 0) out_ls[m] = acc;
    if (acc > best) {  // m increases within a warp, so the first max keeps the lowest index
      best = acc;
      best_i = m;
    }
  }
  // block argmax (value desc, index asc)
  if (lane == 0) {
    s_max[warp] = best;
    s_arg[warp] = best_i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = -INFINITY;
    int bi = 0x7fffffff;
    for (int w = 0; w < nw; ++w) {
      if (s_max[w] > b || (s_max[w] == b && s_arg[w] < bi)) {
        b = s_max[w];
        bi = s_arg[w];
      }
    }
    s_max[0] = b;
    s_arg[0] = (bi == 0x7fffffff) ? 0 : bi;
  }
  __syncthreads();
  const float mx = s_max[0];
  if (threadIdx.x == 0) a.argmax[doc] = s_arg[0];
  float part = 0.f;
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) part += expf(out_ls[m] - mx);
  const float total = block_sum(part, s_sum);
  float* out_p = a.prob + static_cast<size_t>(doc) * a.M;
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) out_p[m] = expf(out_ls[m] - mx) / total;
}

// The same scoring split over many CTAs, for calls with few documents whose
// work is large (the fused kernel above runs one CTA per document): the LSE
// rows come from lse_reduce_kernel (warp per row, every document at once);
// then label_logscore_kernel (CTA per (document, 64 labels), warp per label)
// and label_softmax_kernel (CTA per document).
constexpr int kLabelsPerCta = 64;
// A document is small work for one CTA of the fused kernel up to this many
// tile partials (evaluated rows x vocabulary tiles) and labels.
constexpr long kLabelScoreSmallPartials = 16384;
constexpr int kLabelScoreSmallLabels = 1024;
__global__ void label_logscore_kernel(LabelScoreArgs a) {
  grid_dependency_wait();
  const int doc = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float* cl = a.child_logit + static_cast<size_t>(doc) * a.n_child;
  const float* lse = a.lse + static_cast<size_t>(doc) * a.a;
  float* out_ls = a.logscore + static_cast<size_t>(doc) * a.M;
  const int m_end = min(a.M, static_cast<int>(blockIdx.y + 1) * kLabelsPerCta);
  for (int m = blockIdx.y * kLabelsPerCta + warp; m < m_end; m += nw) {
    const int t0 = __ldg(a.term_offsets + m), t1 = __ldg(a.term_offsets + m + 1);
    float acc = 0.f;
    for (int t = t0 + lane; t < t1; t += 32) acc += cl[__ldg(a.term_slot + t)] - lse[__ldg(a.term_eval + t)];
    acc = warp_sum(acc);
    const int pe = __ldg(a.prefix_eval + m);
    if (pe >= 0) {  // prefix label: probability of stopping at its end node
      const int c0 = __ldg(a.eval_child_offsets + pe), c1 = __ldg(a.eval_child_offsets + pe + 1);
      double cont = 0.0;
      for (int c = c0 + lane; c < c1; c += 32) cont += exp(static_cast<double>(cl[c]) - static_cast<double>(lse[pe]));
      cont = warp_sum_d(cont);
      acc = (cont < 1.0 - 1e-12) ? acc + static_cast<float>(log1p(-cont)) : -INFINITY;
    }
    if (lane == 0) out_ls[m] = acc;
  }
}

__global__ void label_softmax_kernel(LabelScoreArgs a) {
  grid_dependency_wait();
  __shared__ float s_max[32];
  __shared__ int s_arg[32];
  __shared__ float s_sum[32];
  const int doc = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float* ls = a.logscore + static_cast<size_t>(doc) * a.M;
  float best = -INFINITY;
  int best_i = 0x7fffffff;
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) {  // m increases per thread: the first max keeps the lowest index
    const float v = ls[m];
    if (v > best) {
      best = v;
      best_i = m;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
    if (ob > best || (ob == best && oi < best_i)) {
      best = ob;
      best_i = oi;
    }
  }
  if (lane == 0) {
    s_max[warp] = best;
    s_arg[warp] = best_i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = -INFINITY;
    int bi = 0x7fffffff;
    for (int w = 0; w < nw; ++w) {
      if (s_max[w] > b || (s_max[w] == b && s_arg[w] < bi)) {
        b = s_max[w];
        bi = s_arg[w];
      }
    }
    s_max[0] = b;
    s_arg[0] = (bi == 0x7fffffff) ? 0 : bi;
  }
  __syncthreads();
  const float mx = s_max[0];
  if (threadIdx.x == 0) a.argmax[doc] = s_arg[0];
  float part = 0.f;
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) part += expf(ls[m] - mx);
  const float total = block_sum(part, s_sum);
  float* out_p = a.prob + static_cast<size_t>(doc) * a.M;
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) out_p[m] = expf(ls[m] - mx) / total;
}

// AI.IF on joined pairs: CTA per (anchor, partner), warp per restricted row.
// logit_r = z_f32[row] . W_lm[token_r] in fp32 for the R answer spellings
// (the first n_true are TRUE's); p_true = sum of the TRUE rows' softmax over
// the R rows.
__global__ void join_head_kernel(const float* __restrict__ z, const bf16* __restrict__ lm_head,
                                 const int* __restrict__ tokens, int n_true, int R, int M, int d,
                                 float* __restrict__ p_true) {
  grid_dependency_wait();
  __shared__ float s_logit[kJoinMaxRows];
  const int row = blockIdx.x;  // anchor * M + partner
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float* zr = z + static_cast<size_t>(row) * d;
  for (int r = warp; r < R; r += nw) {
    const bf16* w = lm_head + static_cast<size_t>(__ldg(tokens + r)) * d;
    float acc = 0.f;
    for (int i = lane * 2; i < d; i += 64) {
      const float2 wv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(w + i));
      acc += zr[i] * wv.x + zr[i + 1] * wv.y;
    }
    acc = warp_sum(acc);
    if (lane == 0) s_logit[r] = acc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float mx = -INFINITY;
    for (int r = 0; r < R; ++r) mx = fmaxf(mx, s_logit[r]);
    float all = 0.f, yes = 0.f;
    for (int r = 0; r < R; ++r) {
      const float e = expf(s_logit[r] - mx);
      all += e;
      if (r < n_true) yes += e;
    }
    p_true[row] = yes / all;
  }
}

// letters: one block per document, warp per letter row.
// Warp per (document, listed token): logit = z32[doc] . W_lm[token] in fp32,
// 16-byte weight loads; 8 tokens per CTA, documents along y.
__global__ void restricted_logits_kernel(const float* __restrict__ z, const bf16* __restrict__ lm_head,
                                         const int* __restrict__ tokens, int M, int d, float* __restrict__ logits) {
  grid_dependency_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int m = blockIdx.x * (blockDim.x >> 5) + warp;
  const int doc = blockIdx.y;
  if (m >= M) return;
  const float4* zr = reinterpret_cast<const float4*>(z + static_cast<size_t>(doc) * d);
  const uint4* w = reinterpret_cast<const uint4*>(lm_head + static_cast<size_t>(__ldg(tokens + m)) * d);
  float acc = 0.f;
#pragma unroll 4
  for (int i = lane; i < (d >> 3); i += 32) {
    const uint4 wv = __ldg(w + i);
    const float4 w0 = bf16x4_to_float4(make_uint2(wv.x, wv.y)), w1 = bf16x4_to_float4(make_uint2(wv.z, wv.w));
    const float4 z0 = zr[2 * i], z1 = zr[2 * i + 1];
    acc = fmaf(z0.x, w0.x, fmaf(z0.y, w0.y, fmaf(z0.z, w0.z, fmaf(z0.w, w0.w, acc))));
    acc = fmaf(z1.x, w1.x, fmaf(z1.y, w1.y, fmaf(z1.z, w1.z, fmaf(z1.w, w1.w, acc))));
  }
  acc = warp_sum(acc);
  if (lane == 0) logits[static_cast<size_t>(doc) * M + m] = acc;
}

// CTA per document: the row of M logits (in logprob) renormalised in place:
// log-softmax and softmax over the M entries, argmax (lowest index of the max).
__global__ void letters_softmax_kernel(int M, float* __restrict__ logprob, float* __restrict__ prob,
                                       int* __restrict__ argmax) {
  grid_dependency_wait();
  extern __shared__ float s_logit[];
  __shared__ float s_red[32];
  const int doc = blockIdx.x;
  float* row = logprob + static_cast<size_t>(doc) * M;
  for (int m = threadIdx.x; m < M; m += blockDim.x) s_logit[m] = row[m];
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = -INFINITY;
    int bi = 0;
    for (int m = 0; m < M; ++m)
      if (s_logit[m] > b) {
        b = s_logit[m];
        bi = m;
      }
    s_red[0] = b;
    argmax[doc] = bi;
  }
  __syncthreads();
  const float mx = s_red[0];
  float part = 0.f;
  for (int m = threadIdx.x; m < M; m += blockDim.x) part += expf(s_logit[m] - mx);
  __syncthreads();
  const float total = block_sum(part, s_red);
  const float lt = logf(total);
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    const float lp = s_logit[m] - mx - lt;
    row[m] = lp;
    prob[static_cast<size_t>(doc) * M + m] = expf(lp);
  }
}

// Descends forced single-child chains; returns the node where a choice is
// needed or where one label is left.
__device__ __forceinline__ int settle(const DecodeTrie& t, int u) {
  for (int guard = 0; guard < t.n_nodes; ++guard) {
    if (t.subtree_labels[u] <= 1) break;
    const int c0 = t.child_offsets[u], c1 = t.child_offsets[u + 1];
    if (c1 - c0 != 1) break;
    u = t.child_nodes[c0];
  }
  return u;
}

// Single block: settles every undecided cursor and compacts the documents
// that still need the model into slots (in document order).
__global__ void decode_prepare_kernel(DecodeTrie t, int num_docs, int* node_cursor, int* label_out, int* slot_doc,
                                      int* slot_node, int* n_slots, int* active_count) {
  grid_dependency_wait();
  __shared__ int s_warp[32];
  __shared__ int s_base;
  if (threadIdx.x == 0) {
    s_base = 0;
    *active_count = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int i0 = 0; i0 < num_docs; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    bool active = false;
    int u = 0;
    if (i < num_docs && label_out[i] < 0) {
      u = node_cursor[i];
      if (u < 0 || u >= t.n_nodes) u = 0;
      u = settle(t, u);
      node_cursor[i] = u;
      if (t.subtree_labels[u] <= 1) {
        label_out[i] = t.unique_label[u];
      } else {
        active = true;
      }
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, active);
    if (lane == 0) s_warp[warp] = __popc(ballot);
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = s_base;
      for (int w = 0; w < nw; ++w) {
        const int c = s_warp[w];
        s_warp[w] = acc;
        acc += c;
      }
      s_base = acc;
    }
    __syncthreads();
    if (active) {
      const int k = s_warp[warp] + __popc(ballot & ((1u << lane) - 1u));
      slot_doc[k] = i;
      slot_node[k] = t.int_index_of_node[u];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_slots = s_base;
}

// One block per slot: logits of the cursor's children (z in fp32), argmax with
// the lowest token id on ties, advance, settle, record the result.
__global__ void decode_select_kernel(DecodeTrie t, const float* __restrict__ z, const bf16* __restrict__ lm_head,
                                     int d, const int* __restrict__ slot_doc, const int* __restrict__ n_slots,
                                     int* node_cursor, int* label_out, int* active_count, uint8_t* touched) {
  grid_dependency_wait();
  __shared__ float scratch[32];
  const int slot = blockIdx.x;
  if (slot >= *n_slots) return;
  const int doc = slot_doc[slot];
  const int u = node_cursor[doc];
  const float* zr = z + static_cast<size_t>(slot) * d;
  const int c0 = t.child_offsets[u], c1 = t.child_offsets[u + 1];
  float best = -INFINITY;
  int best_c = c0;
  for (int c = c0; c < c1; ++c) {
    const bf16* w = lm_head + static_cast<size_t>(t.child_tokens[c]) * d;
    float acc = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) acc += zr[i] * __bfloat162float(w[i]);
    acc = block_sum(acc, scratch);
    if (acc > best) {  // children ascend by token: the first maximum has the lowest token id
      best = acc;
      best_c = c;
    }
  }
  if (threadIdx.x == 0) {
    if (touched) touched[static_cast<size_t>(doc) * t.n_nodes + u] = 1;
    const int v = settle(t, t.child_nodes[best_c]);
    node_cursor[doc] = v;
    if (t.subtree_labels[v] <= 1) {
      label_out[doc] = t.unique_label[v];
    } else {
      atomicAdd(active_count, 1);
    }
  }
}

}  // namespace

cudaError_t launch_embed_rmsnorm(const bf16* embed, const int* tokens, int n, int d, const bf16* gain, float eps,
                                 bf16* out, cudaStream_t st, const int* live) {
  if (n <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(embed_rmsnorm_kernel, dim3(n), dim3(kNormThreads), 0, st, embed, tokens, d, gain, eps, out, live); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_qk_head_norm(const float* part, int k_splits, size_t slab, float* qkv, int rows, int ld, int hq,
                                int hkv, const bf16* gq, const bf16* gk, float eps, cudaStream_t st, const int* live) {
  const long warps = static_cast<long>(rows) * (hq + 2 * hkv);
  if (warps <= 0) return cudaSuccess;
  if (k_splits < 1 || k_splits > 8) return cudaErrorInvalidValue;  // the kernel sums at most 8 slabs
  const int blocks = static_cast<int>((warps * 32 + 255) / 256);
  count_launch();
  { const cudaError_t le_ = launch_pdl(qk_head_norm_kernel, dim3(blocks), dim3(256), 0, st, part, k_splits, slab, qkv, rows, ld, hq, hkv, gq, gk, eps, live); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_final_norm(const float* h_part, int k_splits, size_t slab, const bf16* embed,
                              const int* node_token, RowMap map, int rows, int d, const bf16* gain, float eps,
                              bf16* z_bf16, float* z_f32, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  switch (k_splits) {  // the slab count is a template argument so that every load is issued up front
#define QUAIL_FINAL_NORM(KS)                                                                                    \
  case KS:                                                                                                      \
    count_launch();                                                                                          \
    { const cudaError_t le_ = launch_pdl(final_norm_kernel<KS>, dim3(rows), dim3(kNormThreads), 0, st, h_part, slab, embed, node_token, map, d, gain, eps, \
                                                         z_bf16, z_f32); if (le_ != cudaSuccess) return le_; }                                       \
    break;
    QUAIL_FINAL_NORM(1)
    QUAIL_FINAL_NORM(2)
    QUAIL_FINAL_NORM(3)
    QUAIL_FINAL_NORM(4)
    QUAIL_FINAL_NORM(5)
    QUAIL_FINAL_NORM(6)
    QUAIL_FINAL_NORM(7)
    QUAIL_FINAL_NORM(8)
#undef QUAIL_FINAL_NORM
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_lse_reduce(const float2* lse_part, int rows, int n_tiles, float* lse, cudaStream_t st,
                              const int* live) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(lse_reduce_kernel, dim3((rows * 32 + 255) / 256), dim3(256), 0, st, lse_part, rows, n_tiles, lse, live); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_label_score(const LabelScoreArgs& args, int num_docs, int num_sms, cudaStream_t st) {
  if (num_docs <= 0) return cudaSuccess;
  // One CTA per document when there are enough documents to fill the GPU, or
  // when a document's work is small enough for one CTA (its rows' tile
  // partials and its labels): then one launch costs less than three.
  const bool small_doc = static_cast<long>(args.a) * args.n_tiles <= kLabelScoreSmallPartials &&
                         args.M <= kLabelScoreSmallLabels;
  if (num_docs >= num_sms || small_doc) {
    count_launch();
    { const cudaError_t le_ = launch_pdl(label_score_kernel, dim3(num_docs), dim3(256), 0, st, args); if (le_ != cudaSuccess) return le_; }
    return cudaGetLastError();
  }
  cudaError_t e = launch_lse_reduce(args.lse_part, num_docs * args.a, args.n_tiles, args.lse, st);
  if (e != cudaSuccess) return e;
  count_launch();
  { const cudaError_t le_ = launch_pdl(label_logscore_kernel, dim3(dim3(num_docs, (args.M + kLabelsPerCta - 1) / kLabelsPerCta)), dim3(256), 0, st, args); if (le_ != cudaSuccess) return le_; }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  { const cudaError_t le_ = launch_pdl(label_softmax_kernel, dim3(num_docs), dim3(512), 0, st, args); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_join_head(const float* z, const bf16* lm_head, const int* tokens, int n_true, int R, int rows,
                             int M, int d, float* p_true, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (R < 1 || R > kJoinMaxRows || n_true < 0 || n_true > R) return cudaErrorInvalidValue;
  count_launch();
  { const cudaError_t le_ = launch_pdl(join_head_kernel, dim3(rows), dim3(256), 0, st, z, lm_head, tokens, n_true, R, M, d, p_true); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_restricted_logits(const float* z, const bf16* lm_head, const int* tokens, int M, int num_docs,
                                     int d, float* logits, cudaStream_t st) {
  if (num_docs <= 0 || M <= 0) return cudaSuccess;
  if (d % 8 != 0 || num_docs > 65535) return cudaErrorInvalidValue;
  count_launch();
  { const cudaError_t le_ = launch_pdl(restricted_logits_kernel, dim3(dim3((M + 7) / 8, num_docs)), dim3(256), 0, st, z, lm_head, tokens, M, d, logits); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_letters_head(const float* z, const bf16* lm_head, const int* letter_tokens, int M, int num_docs,
                                int d, float* logprob, float* prob, int* argmax, cudaStream_t st) {
  if (num_docs <= 0) return cudaSuccess;
  cudaError_t e = launch_restricted_logits(z, lm_head, letter_tokens, M, num_docs, d, logprob, st);
  if (e != cudaSuccess) return e;
  count_launch();
  { const cudaError_t le_ = launch_pdl(letters_softmax_kernel, dim3(num_docs), dim3(256), M * sizeof(float), st, M, logprob, prob, argmax); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_decode_prepare(DecodeTrie t, int num_docs, int* node_cursor, int* label_out, int* slot_doc,
                                  int* slot_node, int* n_slots, int* active_count, cudaStream_t st) {
  count_launch();
  { const cudaError_t le_ = launch_pdl(decode_prepare_kernel, dim3(1), dim3(1024), 0, st, t, num_docs, node_cursor, label_out, slot_doc, slot_node, n_slots,
                                            active_count); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_decode_select(DecodeTrie t, const float* z, const bf16* lm_head, int d, int num_docs,
                                 const int* slot_doc, const int* n_slots, int* node_cursor, int* label_out,
                                 int* active_count, uint8_t* touched, cudaStream_t st) {
  if (num_docs <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(decode_select_kernel, dim3(num_docs), dim3(256), 0, st, t, z, lm_head, d, slot_doc, n_slots, node_cursor, label_out,
                                                 active_count, touched); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

}  // namespace quail
