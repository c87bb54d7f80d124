// tcgen05 GEMM instantiations: plain fp32 store (q/k/v and W_o projections)
// and the output head with the fused log-sum-exp + child-token gather
// ("To Classify, Try a Trie Tree", sec. 4.1 "Output head": the head has one
// row per vocabulary token and a token's score is the dot product of the
// hidden state with that row; probabilities need every row).
#include "kernels.h"
#include "umma_gemm.cuh"

namespace quail {

namespace {

constexpr int kProjBN = 256;
constexpr int kProjStages = 3;  // 64 KB per stage (A_hi, A_lo, B)
constexpr int kHeadStages = 4;  // 48 KB per stage
constexpr float kLog2e = 1.4426950408889634f;

// 2^x, one MUFU op with flush-to-zero: the summands of a log-sum-exp are
// relative to the running maximum, so results below 2^-126 are negligible.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per 128 x 256 accumulator tile and row: the max and the sum of exp over the
// valid columns (base-2 units: m2 = max * log2 e), from the tensor-core
// logits, in two passes over the TMEM accumulator (max, then one FFMA and one
// exp2 per logit on four independent sums).
// The child tokens of the row's node that fall inside the tile are gathered
// here too; their logits are evaluated in fp32 from the unrounded hidden
// state (z_f32 . W_lm[c], warp-cooperative, the tile's W rows being hot in
// L2), because a label's log score sums up to d_m of them while the LSE
// averages the bf16 rounding of z away. Child tokens are sorted, so one
// binary search per tile finds the first candidate and a cursor walks the
// 32-column chunks in order.
struct EpiHead {
  static constexpr uint32_t kScratchBytes = 0;
  HeadEpilogueArgs a;
  int M;
  int V;
  __device__ __forceinline__ void operator()(int m_blk, int n_blk, int /*ks*/, int lane_row, uint32_t taddr,
                                             float* /*warp_scratch*/) const {
    const int row = m_blk * kGemmBM + lane_row;
    const int lane = threadIdx.x & 31;
    const bool valid = row < M;
    const int n0 = n_blk * kHeadBN;
    int cur = 0, cend = 0;
    float* cl_out = nullptr;
    if (valid) {
      const int slot = row / a.nq;
      const int e = row - slot * a.nq;
      int lo = __ldg(a.child_offsets + e), hi = __ldg(a.child_offsets + e + 1);
      cend = hi;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.child_tokens + mid) < n0) lo = mid + 1; else hi = mid;
      }
      cur = lo;
      cl_out = a.child_logit + static_cast<size_t>(slot) * a.n_child;
    }
    const int n_valid = min(kHeadBN, V - n0);  // >= 1: column n0 of every tile is a real token
    // Pass 1: the row's largest logit in the tile, and the child logits that
    // fall in it. Four independent max chains per thread.
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
    for (int c = 0; c < kHeadBN / 32; ++c) {
      if (c * 32 >= n_valid) break;  // warp-uniform
      float v[32];
      tmem_ld_32cols(taddr + c * 32, v);
      const int col_end = n0 + c * 32 + 32;
      int tok = (cur < cend) ? __ldg(a.child_tokens + cur) : 0x7fffffff;
      unsigned hit = __ballot_sync(0xffffffffu, tok < col_end);
      while (hit) {
        const int src = __ffs(hit) - 1;
        const int t_src = __shfl_sync(0xffffffffu, tok, src);
        const int r_src = __shfl_sync(0xffffffffu, row, src);
        const float4* zr = reinterpret_cast<const float4*>(a.z32 + static_cast<size_t>(r_src) * a.d);
        const uint2* wr = reinterpret_cast<const uint2*>(a.lm_head + static_cast<size_t>(t_src) * a.d);
        float acc = 0.f;
        for (int i = lane; i < (a.d >> 2); i += 32) {
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
        if (lane == src) {
          cl_out[cur] = acc;
          ++cur;
          tok = (cur < cend) ? __ldg(a.child_tokens + cur) : 0x7fffffff;
        }
        hit = __ballot_sync(0xffffffffu, tok < col_end);
      }
      if (c * 32 + 32 <= n_valid) {
#pragma unroll
        for (int i = 0; i < 32; ++i) mx[i & 3] = fmaxf(mx[i & 3], v[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c * 32 + i < n_valid) mx[i & 3] = fmaxf(mx[i & 3], v[i]);
      }
    }
    // Pass 2: sum of 2^(logit log2 e - m2) over the tile's tokens, one FFMA
    // and one MUFU op per logit, four independent sums per thread (the TMEM
    // accumulator is read a second time instead of being kept in registers).
    const float m2 = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * kLog2e;
    float sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int c = 0; c < kHeadBN / 32; ++c) {
      if (c * 32 >= n_valid) break;
      float v[32];
      tmem_ld_32cols(taddr + c * 32, v);
      if (c * 32 + 32 <= n_valid) {
#pragma unroll
        for (int i = 0; i < 32; ++i) sa[i & 3] += fast_exp2(fmaf(v[i], kLog2e, -m2));
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c * 32 + i < n_valid) sa[i & 3] += fast_exp2(fmaf(v[i], kLog2e, -m2));
      }
    }
    const float s = (sa[0] + sa[1]) + (sa[2] + sa[3]);
    if (valid) a.lse_part[static_cast<size_t>(row) * a.n_tiles + n_blk] = make_float2(m2, s);
  }
};

template <int BN, int STAGES, bool SPLIT_A, class Epi, int CM = 1>
cudaError_t launch_umma(const CUtensorMap& tmA, const BSet& bset, int M, int N, int nk, int k_splits, const Epi& epi,
                        int num_sms, int* err, cudaStream_t st, const int* m_live = nullptr) {
  using Cfg = GemmCfg<BN, STAGES, SPLIT_A>;
  constexpr size_t smem = Cfg::kSmemBytes + Epi::kScratchBytes;
  static_assert(smem <= 232448, "shared memory per CTA");
  auto kern = umma_gemm_kernel<BN, STAGES, SPLIT_A, Epi, CM>;
  static int configured_device = -1;  // the attribute is set per device
  static int resident = 0;            // CTAs of this kernel that can be resident at once (whole clusters)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    resident = num_sms;
    if (CM > 1) {
      // Clusters are placed within one GPC, so a GPC with an odd number of
      // free SMs leaves one idle: a persistent grid of num_sms CTAs could
      // then hold clusters that only start when others finish.
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(num_sms / CM * CM, 1, 1);
      q.blockDim = dim3(kGemmThreads, 1, 1);
      q.dynamicSmemBytes = smem;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = CM;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &q);
      if (e != cudaSuccess) return e;
      if (clusters > 0 && clusters * CM < resident) resident = clusters * CM;
    }
    configured_device = dev;
  }
  const int m_tiles = (M + kGemmBM - 1) / kGemmBM;
  const int units = ((m_tiles + CM - 1) / CM * CM) * ((N + BN - 1) / BN) * k_splits;
  // Walk M-major when A is the larger operand (a W_o over many rows); the
  // CTAs of a cluster share B bands, so clusters always walk N bands.
  const double a_bytes = static_cast<double>(M) * nk * kGemmBK * 2.0 * (SPLIT_A ? 2 : 1);
  const double b_bytes = static_cast<double>(N) * nk * kGemmBK * 2.0;
  const int m_major = (CM == 1 && a_bytes > b_bytes) ? 1 : 0;
  // Walking N bands, the M tiles go in groups whose A rows (every k-block)
  // fit in kGemmGroupABytes of L2: with thousands of rows (the head of a
  // large label set) A would otherwise stream through L2 once per band.
  const int m_tiles_s = (m_tiles + CM - 1) / CM * CM;
  const double a_tile_bytes = static_cast<double>(kGemmBM) * nk * kGemmBK * 2.0 * (SPLIT_A ? 2 : 1);
  int m_group = static_cast<int>(kGemmGroupABytes / a_tile_bytes) / CM * CM;
  if (m_group < CM) m_group = CM;
  if (m_group > m_tiles_s) m_group = m_tiles_s;
  if (m_major) m_group = 0;
  const int pf_depth = CM > 1 ? kPrefetchKb : 0;
  int grid = units < resident ? units : resident;
  grid = grid / CM * CM;  // whole clusters; units is a multiple of CM
  if (grid <= 0) return cudaSuccess;
  if (CM == 1) {
    count_launch();
    return launch_pdl(kern, dim3(grid), dim3(kGemmThreads), smem, st, tmA, bset, M, N, nk, k_splits, m_group, pf_depth,
                      epi, err, m_live);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CM;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch.cuh
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, tmA, bset, M, N, nk, k_splits, m_group, pf_depth, epi, err, m_live);
}

}  // namespace

int choose_k_splits(int tiles, int nk, int num_sms) {
  // The smallest split count whose units fill the SMs to >= 75% over whole
  // waves (fewer splits = fewer partial slabs); else the best one found. Each
  // unit keeps at least 4 k-blocks. Measured at the W_o shape, more splits
  // add slab traffic without speeding up the operand stream.
  int best = 1;
  double best_eff = 0.0;
  for (int ks = 1; ks <= 8 && nk / ks >= 4; ++ks) {
    const long units = static_cast<long>(tiles) * ks;
    const long waves = (units + num_sms - 1) / num_sms;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * num_sms);
    if (eff >= 0.75) return ks;
    if (eff > best_eff) {
      best_eff = eff;
      best = ks;
    }
  }
  return best;
}

cudaError_t launch_gemm_proj(const CUtensorMap& tmA, const BSet& bset, int M, int N, int K, int k_splits, float* C,
                             size_t slab, int ldc, int num_sms, int* err, cudaStream_t st, const int* m_live) {
  EpiStoreF32<kProjBN> epi;
  if (k_splits < 1 || ldc % 4 != 0 || slab % 4 != 0 ||
      !encode_3d_f32_store(&epi.tm, C, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                           static_cast<uint64_t>(k_splits), static_cast<uint64_t>(ldc), slab, 32, 32))
    return cudaErrorInvalidValue;
  return launch_umma<kProjBN, kProjStages, true>(tmA, bset, M, N, K / kGemmBK, k_splits, epi, num_sms, err, st,
                                                 m_live);
}

// SwiGLU epilogue of a gate|up GEMM in glu mode (one k-split): columns
// [0, BN/2) of the tile are gate, [BN/2, BN) up, for outputs j0 = n_blk BN/2 ..
// act[row][j] = split(SiLU(gate) * up) as [hi (I) | lo (I)] bf16. Each warp
// builds its 32 rows x 32 outputs as two bf16 planes (hi, lo) in shared memory
// and one lane issues a bulk tile store through tm, a [2][M][I] view of act
// (plane stride I elements): 4 stores per warp and unit instead of 2 per
// output. Lane r writes row r's 16-byte chunks in an order rotated by r / 2,
// so the 32 lanes' chunk writes spread over all banks.
template <int BN>
struct EpiSwiGLU {
  static constexpr uint32_t kScratchBytes = 4 * 2 * 4096;
  CUtensorMap tm;
  __device__ __forceinline__ void operator()(int m_blk, int n_blk, int /*ks*/, int lane_row, uint32_t taddr,
                                             float* ws) const {
    const int lane = threadIdx.x & 31;
    const int row0 = m_blk * kGemmBM + lane_row - lane;
    const int j0 = n_blk * (BN / 2);
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      float gv[32], uv[32];
      tmem_ld_32cols(taddr + c * 32, gv);
      tmem_ld_32cols(taddr + BN / 2 + c * 32, uv);
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a0 = gv[2 * i] / (1.f + expf(-gv[2 * i])) * uv[2 * i];
        const float a1 = gv[2 * i + 1] / (1.f + expf(-gv[2 * i + 1])) * uv[2 * i + 1];
        const __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(a0 - hf.x, a1 - hf.y);
        hi[i] = *reinterpret_cast<const uint32_t*>(&h);
        lo[i] = *reinterpret_cast<const uint32_t*>(&l);
      }
      uint4* buf = reinterpret_cast<uint4*>(ws + (c & 1) * 1024);  // 4 KB: planes hi, lo of 32 rows x 64 B
      if (lane == 0) bulk_wait_group_read<1>();  // the store that last read this buffer is done with it
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int qq = (q + (lane >> 1)) & 3;
        uint4 h, l;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (qq == k) {
            h = make_uint4(hi[4 * k], hi[4 * k + 1], hi[4 * k + 2], hi[4 * k + 3]);
            l = make_uint4(lo[4 * k], lo[4 * k + 1], lo[4 * k + 2], lo[4 * k + 3]);
          }
        }
        buf[lane * 4 + qq] = h;
        buf[128 + lane * 4 + qq] = l;
      }
      fence_proxy_async_smem();  // the tile writes, visible to the bulk copy
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm, buf, j0 + c * 32, row0, 0);
        bulk_commit_group();
      }
    }
  }
  // Before the CTA exits: every store of this warp has completed.
  __device__ __forceinline__ void drain() const {
    if ((threadIdx.x & 31) == 0) bulk_wait_group_all();
    __syncwarp();
  }
};

cudaError_t launch_gemm_swiglu(const CUtensorMap& tmA, const BSet& bset, int M, int I, int K, bf16* act,
                               int num_sms, int* err, cudaStream_t st) {
  if (!bset.glu || bset.count != 2 || I % (kProjBN / 2) != 0) return cudaErrorInvalidValue;
  EpiSwiGLU<kProjBN> epi;
  if (!encode_3d_bf16_store(&epi.tm, act, static_cast<uint64_t>(I), static_cast<uint64_t>(M), 2,
                            2 * static_cast<uint64_t>(I), static_cast<uint64_t>(I), 32, 32))
    return cudaErrorInvalidValue;
  return launch_umma<kProjBN, kProjStages, true>(tmA, bset, M, 2 * I, K / kGemmBK, 1, epi, num_sms, err, st);
}

int head_cluster_ctas(int M) {
  const int t = (M + kGemmBM - 1) / kGemmBM;
  return t <= kHeadWideClusterMaxTiles && (t + 3) / 4 * 4 <= (t + 1) / 2 * 2 ? 4 : 2;
}

cudaError_t launch_gemm_head(const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int V, int K,
                             const HeadEpilogueArgs& args, int num_sms, int* err, cudaStream_t st,
                             const int* m_live) {
  EpiHead epi{args, M, V};
  BSet b{};
  b.map[0] = tmB;
  b.n_begin[0] = 0;
  b.n_begin[1] = V;
  b.count = 1;
  if (head_cluster_ctas(M) == 4)
    return launch_umma<kHeadBN, kHeadStages, false, EpiHead, 4>(tmA, b, M, V, K / kGemmBK, 1, epi, num_sms, err, st,
                                                                m_live);
  return launch_umma<kHeadBN, kHeadStages, false, EpiHead, 2>(tmA, b, M, V, K / kGemmBK, 1, epi, num_sms, err, st,
                                                              m_live);
}

// Test hook: this translation unit's copy of the pipeline wait limit.
cudaError_t set_pipeline_wait_limit_gemm(long long cycles) {
  return cudaMemcpyToSymbol(g_pipeline_wait_limit, &cycles, sizeof(cycles));
}

}  // namespace quail
