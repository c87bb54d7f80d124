// Kernels of the shortlisted trie_tree for huge label sets ("Trie Automata
// for Constrained Decoding over Large Finite Sets": a top-k shortlist ahead
// of exact trie scoring; hierarchical groups are the special case whose
// prefixes are the group names). The first pass scores every group's prefix
// with the ordinary trie_tree kernels; these kernels pick each document's best
// groups, lay out the second pass's rows, and score the kept labels from the
// second pass's hidden states (label scores as in "To Classify, Try a Trie
// Tree", sec. 3.2).
#include <algorithm>
#include <cfloat>

#include "kernels.h"
#include "launch.cuh"
#include "quail_internal.h"

namespace quail {

namespace {

constexpr int kSelectThreads = 256;
constexpr int kScoreThreads = 512;

// (value, index) order of the shortlist: higher value first, lower index on ties.
__device__ __forceinline__ bool ranks_before(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Block-wide best (value, index) under ranks_before; blockDim.x <= 1024.
__device__ void block_best(float& v, int& i, float* s_v, int* s_i) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ranks_before(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
  __syncthreads();
  if (lane == 0) {
    s_v[warp] = v;
    s_i[warp] = i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < nw; ++w)
      if (ranks_before(s_v[w], s_i[w], s_v[0], s_i[0])) {
        s_v[0] = s_v[w];
        s_i[0] = s_i[w];
      }
  }
  __syncthreads();
  v = s_v[0];
  i = s_i[0];
}

__device__ float block_sum_f(float v, float* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += s[w];
    s[0] = t;
  }
  __syncthreads();
  return s[0];
}

// CTA per document: B rounds, each taking the best group ranked after the
// previous pick (so no group is taken twice and no mark table is needed).
__global__ void __launch_bounds__(kSelectThreads) shortlist_select_kernel(const float* __restrict__ ls, int G, int B,
                                                                          int* __restrict__ sel) {
  grid_dependency_wait();
  __shared__ float s_v[32];
  __shared__ int s_i[32];
  const int doc = blockIdx.x;
  const float* row = ls + static_cast<size_t>(doc) * G;
  float pv = INFINITY;
  int pi = -1;
  for (int b = 0; b < B; ++b) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
      float v = row[g];
      if (v != v) v = -INFINITY;  // a NaN score ranks last
      const bool after = v < pv || (v == pv && g > pi);
      if (after && ranks_before(v, g, bv, bi)) {
        bv = v;
        bi = g;
      }
    }
    block_best(bv, bi, s_v, s_i);
    if (threadIdx.x == 0) sel[doc * B + b] = bi;
    pv = bv;
    pi = bi;
  }
}

// Warp per (block, child slot): the child token's logit from the unrounded
// hidden state in fp32 (z32 . W_lm[tok]), minus the row's log-sum-exp.
__global__ void shortlist_child_logprob_kernel(ShortlistTables T, const int* __restrict__ sel, int n_blocks,
                                               const int* __restrict__ block_base, const float* __restrict__ z32,
                                               const bf16* __restrict__ lm_head, int d, const float* __restrict__ lse,
                                               float* __restrict__ clp) {
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long total = static_cast<long long>(n_blocks) * T.max_children;
  for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total;
       w += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    const int blk = static_cast<int>(w / T.max_children);
    const int t = static_cast<int>(w - static_cast<long long>(blk) * T.max_children);
    const int g = sel[blk];
    const int c0 = T.child_off[g];
    if (t >= T.child_off[g + 1] - c0) continue;
    const int r = block_base[blk] + T.child_row[c0 + t];
    const int tok = T.child_tok[c0 + t];
    const float4* zr = reinterpret_cast<const float4*>(z32 + static_cast<size_t>(r) * d);
    const uint2* wr = reinterpret_cast<const uint2*>(lm_head + static_cast<size_t>(tok) * d);
    float acc = 0.f;
    for (int i = lane; i < (d >> 2); i += 32) {
      const float4 z4 = zr[i];
      const uint2 w4 = __ldg(wr + i);
      const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4.x));
      const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4.y));
      acc = fmaf(z4.x, w01.x, acc);
      acc = fmaf(z4.y, w01.y, acc);
      acc = fmaf(z4.z, w23.x, acc);
      acc = fmaf(z4.w, w23.y, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) clp[w] = acc - lse[r];
  }
}

// One CTA: exclusive scan of the kept groups' row counts in (document, group)
// order, each document's first row and row count, and the total.
__global__ void __launch_bounds__(1024) shortlist_scan_kernel(ShortlistTables T, const int* __restrict__ sel,
                                                              int num_docs, int B, int* __restrict__ block_base,
                                                              int* __restrict__ doc_base, int* __restrict__ doc_rows,
                                                              int* __restrict__ count) {
  grid_dependency_wait();
  __shared__ int s_part[1024];
  __shared__ int s_total;
  const int n_blocks = num_docs * B;
  const int per = (n_blocks + blockDim.x - 1) / blockDim.x;
  const int b0 = min(n_blocks, static_cast<int>(threadIdx.x) * per), b1 = min(n_blocks, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) sum += T.row_off[sel[b] + 1] - T.row_off[sel[b]];
  s_part[threadIdx.x] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {  // exclusive scan of the per-thread sums
    int run = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x); ++i) {
      const int v = s_part[i];
      s_part[i] = run;
      run += v;
    }
    s_total = run;
    *count = run;
  }
  __syncthreads();
  int base = s_part[threadIdx.x];
  for (int b = b0; b < b1; ++b) {
    block_base[b] = base;
    base += T.row_off[sel[b] + 1] - T.row_off[sel[b]];
  }
  __syncthreads();
  for (int d = threadIdx.x; d < num_docs; d += blockDim.x) {
    const int first = block_base[d * B];
    const int end = d + 1 < num_docs ? block_base[(d + 1) * B] : s_total;
    doc_base[d] = first;
    doc_rows[d] = end - first;
  }
}

// Block per (document, kept group): that group's rows at their compact
// numbers; one more block fills rows count..R-1 with root copies.
__global__ void shortlist_expand_kernel(ShortlistTables T, const int* __restrict__ sel, int B, int Bq, int R,
                                        const int* __restrict__ block_base, const int* __restrict__ doc_base,
                                        const int* __restrict__ count, const int* __restrict__ eval_token,
                                        const int* __restrict__ eval_depth, int* __restrict__ row_token,
                                        int* __restrict__ row_depth, int* __restrict__ row_parent,
                                        int* __restrict__ padded_of) {
  grid_dependency_wait();
  const int blk = blockIdx.x;
  if (blk == static_cast<int>(gridDim.x) - 1) {
    for (int c = *count + threadIdx.x; c < R; c += blockDim.x) {
      row_token[c] = eval_token[0];
      row_depth[c] = eval_depth[0];
      row_parent[c] = -1;
    }
    return;
  }
  const int doc = blk / B;
  const int g = sel[blk];
  const int base = block_base[blk];
  const int local0 = base - doc_base[doc];  // first row of this group within its document
  const int off = T.row_off[g];
  const int n = T.row_off[g + 1] - off;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int e = T.row_eval[off + j];
    const int p = T.row_parent[off + j];
    const int c = base + j;
    row_token[c] = eval_token[e];
    row_depth[c] = eval_depth[e];
    row_parent[c] = p >= 0 ? base + p : -1;
    padded_of[c] = doc * Bq + local0 + j;
  }
}

// Block per compact row c < *count: 16-byte copies of row padded_of[c].
__global__ void gather_rows_kernel(const uint4* __restrict__ src, const int* __restrict__ padded_of,
                                   const int* __restrict__ count, int vec_per_row, uint4* __restrict__ dst) {
  grid_dependency_wait();
  const int c = blockIdx.x;
  if (c >= *count) return;
  const uint4* s = src + static_cast<size_t>(padded_of[c]) * vec_per_row;
  uint4* d = dst + static_cast<size_t>(c) * vec_per_row;
  for (int i = threadIdx.x; i < vec_per_row; i += blockDim.x) d[i] = s[i];
}

// Every label's score -inf and probability 0 (the kept ones are overwritten next).
__global__ void shortlist_clear_kernel(float* __restrict__ logscore, float* __restrict__ prob, size_t n) {
  grid_dependency_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    logscore[i] = -INFINITY;
    prob[i] = 0.f;
  }
}

// CTA per (document, kept group): warp per label of that group, its terms
// summed from the child log-probs plus the prefix-label correction.
__global__ void __launch_bounds__(kScoreThreads) shortlist_label_score_kernel(
    ShortlistTables T, const int* __restrict__ sel, int B, int M, const float* __restrict__ clp,
    float* __restrict__ logscore) {
  grid_dependency_wait();
  const int doc = blockIdx.x, b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int blk = doc * B + b;
  const int g = sel[blk];
  const float* cl = clp + static_cast<size_t>(blk) * T.max_children;
  float* ls = logscore + static_cast<size_t>(doc) * M;
  for (int li = T.lab_off[g] + warp; li < T.lab_off[g + 1]; li += nw) {
    float acc = 0.f;
    for (int k = T.term_off[li] + lane; k < T.term_off[li + 1]; k += 32) acc += cl[T.term_t[k]];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int p0 = T.pref_t0[li], p1 = T.pref_t1[li];
    if (p1 > p0) {  // prefix label: probability of stopping at its end node
      double cont = 0.0;
      for (int c = p0 + lane; c < p1; c += 32) cont += exp(static_cast<double>(cl[c]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cont += __shfl_xor_sync(0xffffffffu, cont, o);
      acc = (cont < 1.0 - 1e-12) ? acc + static_cast<float>(log1p(-cont)) : -INFINITY;
    }
    if (lane == 0) ls[T.lab_id[li]] = acc;
  }
}

// CTA per document: softmax and argmax over the kept labels' scores.
__global__ void __launch_bounds__(kScoreThreads) shortlist_softmax_kernel(ShortlistTables T,
                                                                          const int* __restrict__ sel, int B, int M,
                                                                          const float* __restrict__ logscore,
                                                                          float* __restrict__ prob,
                                                                          int* __restrict__ argmax) {
  grid_dependency_wait();
  __shared__ float s_v[32];
  __shared__ int s_i[32];
  const int doc = blockIdx.x;
  const float* ls = logscore + static_cast<size_t>(doc) * M;
  float* pr = prob + static_cast<size_t>(doc) * M;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int b = 0; b < B; ++b) {
    const int g = sel[doc * B + b];
    for (int li = T.lab_off[g] + threadIdx.x; li < T.lab_off[g + 1]; li += blockDim.x) {
      const int m = T.lab_id[li];
      if (ranks_before(ls[m], m, bv, bi)) {
        bv = ls[m];
        bi = m;
      }
    }
  }
  block_best(bv, bi, s_v, s_i);
  float part = 0.f;
  for (int b = 0; b < B; ++b) {
    const int g = sel[doc * B + b];
    for (int li = T.lab_off[g] + threadIdx.x; li < T.lab_off[g + 1]; li += blockDim.x)
      part += expf(ls[T.lab_id[li]] - bv);
  }
  const float sum = block_sum_f(part, s_v);
  const float inv = (bv == -INFINITY) ? __int_as_float(0x7fc00000) : 1.f / sum;
  for (int b = 0; b < B; ++b) {
    const int g = sel[doc * B + b];
    for (int li = T.lab_off[g] + threadIdx.x; li < T.lab_off[g + 1]; li += blockDim.x) {
      const int m = T.lab_id[li];
      pr[m] = (bv == -INFINITY) ? inv : expf(ls[m] - bv) * inv;
    }
  }
  if (threadIdx.x == 0) argmax[doc] = bi == 0x7fffffff ? 0 : bi;
}

}  // namespace

cudaError_t launch_shortlist_select(const float* prefix_logscore, int num_docs, int G, int B, int* sel,
                                    cudaStream_t st) {
  if (num_docs <= 0) return cudaSuccess;
  if (B < 1 || B > G) return cudaErrorInvalidValue;
  count_launch();
  { const cudaError_t le_ = launch_pdl(shortlist_select_kernel, dim3(num_docs), dim3(kSelectThreads), 0, st, prefix_logscore, G, B, sel); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_shortlist_scan(const ShortlistTables& T, const int* sel, int num_docs, int B, int* block_base,
                                  int* doc_base, int* doc_rows, int* count, cudaStream_t st) {
  if (num_docs <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(shortlist_scan_kernel, dim3(1), dim3(1024), 0, st, T, sel, num_docs, B, block_base, doc_base, doc_rows, count); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_shortlist_expand(const ShortlistTables& T, const int* sel, int num_docs, int B, int Bq, int R,
                                    const int* block_base, const int* doc_base, const int* count,
                                    const int* eval_token, const int* eval_depth, int* row_token, int* row_depth,
                                    int* row_parent, int* padded_of, cudaStream_t st) {
  if (num_docs <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(shortlist_expand_kernel, dim3(num_docs * B + 1), dim3(128), 0, st, T, sel, B, Bq, R, block_base, doc_base, count,
                                                            eval_token, eval_depth, row_token, row_depth, row_parent,
                                                            padded_of); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* src, const int* padded_of, const int* count, int max_rows,
                               size_t row_bytes, void* dst, cudaStream_t st) {
  if (max_rows <= 0) return cudaSuccess;
  if (row_bytes % 16 != 0) return cudaErrorInvalidValue;
  count_launch();
  { const cudaError_t le_ = launch_pdl(gather_rows_kernel, dim3(max_rows), dim3(256), 0, st, static_cast<const uint4*>(src), padded_of, count,
                                               static_cast<int>(row_bytes / 16), static_cast<uint4*>(dst)); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_shortlist_child_logprob(const ShortlistTables& T, const int* sel, int num_docs, int B,
                                           const int* block_base, const float* z32, const bf16* lm_head, int d,
                                           const float* lse, float* clp, cudaStream_t st) {
  if (num_docs <= 0 || T.max_children <= 0) return cudaSuccess;
  if (d % 4 != 0) return cudaErrorInvalidValue;
  const long long warps = static_cast<long long>(num_docs) * B * T.max_children;
  const int blocks = static_cast<int>(std::min<long long>((warps + 7) / 8, 1 << 16));
  count_launch();
  { const cudaError_t le_ = launch_pdl(shortlist_child_logprob_kernel, dim3(blocks), dim3(256), 0, st, T, sel, num_docs * B, block_base, z32, lm_head, d, lse,
                                                         clp); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_shortlist_label_score(const ShortlistTables& T, const int* sel, int num_docs, int B, int M,
                                         const float* clp, float* logscore, float* prob, int* argmax,
                                         cudaStream_t st) {
  if (num_docs <= 0) return cudaSuccess;
  if (B > 65535) return cudaErrorInvalidValue;
  const size_t n = static_cast<size_t>(num_docs) * M;
  count_launch();
  { const cudaError_t le_ = launch_pdl(shortlist_clear_kernel, dim3(static_cast<int>(std::min<size_t>((n + 255) / 256, 4096))), dim3(256), 0, st, logscore, prob, n); if (le_ != cudaSuccess) return le_; }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  { const cudaError_t le_ = launch_pdl(shortlist_label_score_kernel, dim3(dim3(num_docs, B)), dim3(kScoreThreads), 0, st, T, sel, B, M, clp, logscore); if (le_ != cudaSuccess) return le_; }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  { const cudaError_t le_ = launch_pdl(shortlist_softmax_kernel, dim3(num_docs), dim3(kScoreThreads), 0, st, T, sel, B, M, logscore, prob, argmax); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

}  // namespace quail
