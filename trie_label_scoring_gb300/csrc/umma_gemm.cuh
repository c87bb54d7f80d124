// Persistent, warp-specialised tcgen05 GEMM for sm_103a:  C = A * B^T
//   A: [M, K] bf16, K contiguous (row-major)      -> TMA box 64 x 128, 128B swizzle
//   B: [N, K] bf16, K contiguous (nn.Linear rows) -> TMA box 64 x BN,  128B swizzle
// The fp32 accumulator for one 128 x BN tile lives in TMEM (two buffers, so the
// epilogue of tile t overlaps the MMAs of tile t+1). The epilogue is a functor,
// which is how the LM head fuses its log-sum-exp and child-token gather without
// ever writing logits to global memory.
//
// Options:
//  * SPLIT_A: A = [X_hi | X_lo] (a two-term bf16 split of an fp32 operand,
//    2K columns). Each pipeline stage holds the k-block of X_hi, of X_lo and of
//    B; both A halves multiply the same B tile into one accumulator, so
//    C = (X_hi + X_lo) B^T to ~16 bits while B is read once.
//  * Up to three B tensors side by side along N (BSet), each starting at a
//    multiple of BN: q, k and v projections in one launch.
//  * Split-K over CTAs: work unit = (tile, k-split); the epilogue receives the
//    split index and writes its partial tile to its own slab (no atomics); the
//    next kernel sums the slabs.
//  * CM = 2 or 4: clusters of CM CTAs along M share each B tile. The CTAs of
//    a cluster always work on M tiles CM i .. CM i + CM - 1 of the same N
//    band; each loads 1/CM of the B band with TMA multicast into all of them,
//    so every byte of B crosses from L2 once per cluster. A stage is refilled
//    only after every CTA's MMAs have released it (a multicast commit to all
//    empty barriers). M tiles are scheduled in whole clusters; the padding
//    tiles read zeros past the end of A and the epilogue skips rows >= M.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA
// issuer, warps 2..5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
// Units are walked N-band-major: consecutive ids share one B band, so the CTAs
// resident at any moment read each band of B from HBM about once and re-read it
// from L2 for the other M tiles.
#pragma once
#include "sm103.cuh"
#include "launch.cuh"
#include "quail_internal.h"

namespace quail {

constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;  // 64 bf16 = one 128-byte swizzle row
constexpr int kGemmThreads = 192;
constexpr int kPrefetchKb = 8;  // k-blocks of B requested into L2 ahead of their loads (clusters)
constexpr double kGemmGroupABytes = 24.0 * 1024 * 1024;  // A rows in use at once, N-band-major walks

// Up to three B operands covering output columns [n_begin[i], n_begin[i+1]).
// glu != 0: two operands of equal shape whose rows pair up (gate and up
// projections). Unit n's B band is rows [n BN/2, (n+1) BN/2) of map[0]
// followed by the same rows of map[1] (boxes of BN/2 rows), so accumulator
// column c < BN/2 and column BN/2 + c hold the two halves of one output.
struct BSet {
  CUtensorMap map[3];
  int n_begin[4];
  int count;
  int glu;
};

template <int BN, int STAGES, bool SPLIT_A>
struct GemmCfg {
  static constexpr uint32_t kABytes = kGemmBM * kGemmBK * 2;
  static constexpr uint32_t kBBytes = BN * kGemmBK * 2;
  static constexpr uint32_t kStageBytes = (SPLIT_A ? 2 : 1) * kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                        : (2 * BN <= 256) ? 256 : 512;
  // 1024 alignment slack + stages + barriers + tmem slot + abort flag
  static constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + (2 * STAGES + 5) * 8 + 16;
};

struct GemmUnit {
  int m_blk, n_blk, ks, kb0, kb1;
};

// unit -> (k-split, tile) with the k-split slowest, so the CTAs resident at
// one time share B bands and A rows in L2; tile -> (n band, m tile):
//  * m_group > 0: N-band-major within groups of m_group M tiles (consecutive
//    units share a B band; a group walks every band before the next group
//    starts), so the A rows in use stay within one group's L2 footprint while
//    each B band is read once per group;
//  * m_group == 0: M-major, when A is the larger operand (consecutive units
//    share an A tile, so A streams from DRAM once while the smaller B stays
//    in L2).
__device__ __forceinline__ GemmUnit gemm_unit(int u, int m_tiles, int n_tiles, int k_splits, int nk, int m_group) {
  GemmUnit g;
  const int tiles = m_tiles * n_tiles;
  g.ks = u / tiles;
  const int tile = u - g.ks * tiles;
  if (m_group <= 0) {
    g.m_blk = tile / n_tiles;
    g.n_blk = tile - g.m_blk * n_tiles;
  } else {
    const int grp = tile / (m_group * n_tiles);
    const int m0 = grp * m_group;
    const int gm = min(m_group, m_tiles - m0);
    const int t = tile - m0 * n_tiles;
    g.n_blk = t / gm;
    g.m_blk = m0 + (t - g.n_blk * gm);
  }
  g.kb0 = g.ks * nk / k_splits;
  g.kb1 = (g.ks + 1) * nk / k_splits;
  return g;
}

// L2 prefetch cursor over one CTA's sequence of (unit, k-block) B loads:
// step() requests the next B tile of that sequence (this CTA's part of the band).
struct BPrefetch {
  int u, kb, kb1, nb;
  const CUtensorMap* map;
  __device__ __forceinline__ void step(const BSet& bs, int bn, int cm, uint32_t crank, int m_tiles_s, int n_tiles,
                                       int k_splits, int nk, int num_units, int m_group) {
    while (kb >= kb1) {  // advance to this CTA's next unit
      u += gridDim.x;
      if (u >= num_units) return;
      const GemmUnit h = gemm_unit(u, m_tiles_s, n_tiles, k_splits, nk, m_group);
      int bi = 0;
      while (bi + 1 < bs.count && h.n_blk * bn >= bs.n_begin[bi + 1]) ++bi;
      map = &bs.map[bi];
      nb = h.n_blk * bn - bs.n_begin[bi] + static_cast<int>(crank) * (bn / cm);
      kb = h.kb0;
      kb1 = h.kb1;
    }
    tma_prefetch_l2_2d(map, kb * kGemmBK, nb);
    ++kb;
  }
};

// Calls epi.drain() where the epilogue functor defines one (stores still in
// flight when its warps are done); nothing otherwise.
template <class E>
__device__ __forceinline__ auto epi_drain(const E& e, int) -> decltype(e.drain()) {
  e.drain();
}
template <class E>
__device__ __forceinline__ void epi_drain(const E&, long) {}
template <class E>
__device__ __forceinline__ void epi_drain(const E& e) {
  epi_drain(e, 0);
}

// Epi must provide:
//   static constexpr uint32_t kScratchBytes;   // shared memory it needs (a multiple of 64; 0 for none)
//   __device__ void operator()(int m_blk, int n_blk, int ks, int lane_row, uint32_t taddr, float* warp_scratch) const;
// called by each of the 128 epilogue threads for every unit; lane_row in [0,128)
// is this thread's accumulator row, taddr the TMEM address of (row, column 0),
// warp_scratch this warp's quarter of the scratch. All 32 lanes of a warp
// must execute the same tcgen05.ld sequence.
// nk = k-blocks of B's K extent (A has nk k-blocks, or 2*nk with SPLIT_A).
// m_live (may be null): the rows actually present, written by an earlier
// kernel; M is then the bound the grid and A's tensor map were sized for, and
// M tiles past m_live are not computed.
template <int BN, int STAGES, bool SPLIT_A, class Epi, int CM = 1>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ BSet bset, int M, int N,
                     int nk, int k_splits, int m_group, int pf_depth, const __grid_constant__ Epi epi, int* err,
                     const int* m_live) {
  static_assert(CM == 1 || ((CM == 2 || CM == 4) && !SPLIT_A && BN % (8 * CM) == 0),
                "clusters: plain A, B band split in CM parts of whole 8-row swizzle atoms");
  using Cfg = GemmCfg<BN, STAGES, SPLIT_A>;
  constexpr uint32_t kBPart = Cfg::kBBytes / CM;  // bytes of B each CTA of a cluster loads
  constexpr uint16_t kClusterMask = static_cast<uint16_t>((1u << CM) - 1u);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // the epilogue's scratch (Epi::kScratchBytes) follows the ring, then the barriers
  uint8_t* epi_scratch = base + STAGES * Cfg::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_scratch + Epi::kScratchBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2]
  uint64_t* tempty = tfull + 2;      // [2]
  uint64_t* drain = tempty + 2;      // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = CM > 1 ? cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CM);  // released by the MMAs of every CTA whose copies land in it
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 128);
    mbar_init(&tempty[1], 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    for (int i = 0; i < bset.count; ++i) tma_prefetch_desc(&bset.map[i]);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (CM > 1) cluster_sync();  // the peers' barriers exist before any multicast reaches them
  // Everything above touched shared memory, TMEM and the kernel parameters
  // only; from here on the previous kernel's outputs are read.
  grid_dependency_wait();
  const int M_eff = m_live != nullptr ? min(M, max(*m_live, 0)) : M;
  const int m_tiles = (M_eff + kGemmBM - 1) / kGemmBM;
  const int m_tiles_s = (m_tiles + CM - 1) / CM * CM;  // scheduled M tiles: whole clusters
  const int n_tiles = (N + BN - 1) / BN;
  const int num_units = m_tiles_s * n_tiles * k_splits;
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int armed_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) armed_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      BPrefetch pf{static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x), 0, 0, 0, nullptr};
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const GemmUnit g = gemm_unit(u, m_tiles_s, n_tiles, k_splits, nk, m_group);
        const int n0 = g.n_blk * BN;
        int bi = 0;
        while (bi + 1 < bset.count && n0 >= bset.n_begin[bi + 1]) ++bi;
        const CUtensorMap* tmB = &bset.map[bi];
        const int nb = n0 - bset.n_begin[bi];
        const int nb_own = nb + static_cast<int>(crank) * (BN / CM);
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          // Clusters stream each B band once from DRAM into L2 and then share
          // it: this CTA's part-band k-blocks are requested kPrefetchKb loads
          // ahead (running on into its next unit), so the first cluster on a
          // band does not wait on DRAM at every k-block.
          if (CM > 1) {
            const int n = (u == static_cast<int>(blockIdx.x) && kb == g.kb0) ? pf_depth + 1 : 1;
            for (int p = 0; p < n; ++p)
              pf.step(bset, BN, CM, crank, m_tiles_s, n_tiles, k_splits, nk, num_units, m_group);
          }
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = base + stage * Cfg::kStageBytes;
          mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
          tma_load_2d(st, &tmA, &full[stage], kb * kGemmBK, g.m_blk * kGemmBM);
          if (SPLIT_A) tma_load_2d(st + Cfg::kABytes, &tmA, &full[stage], (nk + kb) * kGemmBK, g.m_blk * kGemmBM);
          if (CM > 1) {
            tma_load_2d_mcast(st + Cfg::kABytes + crank * kBPart, tmB, &full[stage], kb * kGemmBK, nb_own,
                              kClusterMask);
          } else if (bset.glu) {
            uint8_t* b_st = st + (SPLIT_A ? 2 : 1) * Cfg::kABytes;
            tma_load_2d(b_st, &bset.map[0], &full[stage], kb * kGemmBK, g.n_blk * (BN / 2));
            tma_load_2d(b_st + Cfg::kBBytes / 2, &bset.map[1], &full[stage], kb * kGemmBK, g.n_blk * (BN / 2));
          } else {
            tma_load_2d(st + (SPLIT_A ? 2 : 1) * Cfg::kABytes, tmB, &full[stage], kb * kGemmBK, nb);
          }
          armed_parity[stage] = static_cast<int>(phase);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Never leave with copies in flight: every armed stage must have landed.
      // In a cluster, also wait until the last fill of every stage has been
      // released by all CTAs, so that no commit from a peer is still on its
      // way to this CTA's barriers when the cluster synchronises and exits.
      for (int s = 0; s < STAGES; ++s) {
        if (armed_parity[s] < 0) continue;
        for (int which = 0; which < (CM > 1 ? 2 : 1); ++which) {
          const uint32_t a = smem_u32(which == 0 ? &full[s] : &empty[s]);
          const long long t0 = clock64();
          while (!mbar_try_wait(a, static_cast<uint32_t>(armed_parity[s]))) {
            if ((which == 1 && *abort_flag) || clock64() - t0 > kWaitLimitCycles) {
              *abort_flag = 1;
              break;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = umma_idesc_bf16_f32(kGemmBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const GemmUnit g = gemm_unit(u, m_tiles_s, n_tiles, k_splits, nk, m_group);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(base + stage * Cfg::kStageBytes);
          const uint32_t b_addr = st + (SPLIT_A ? 2 : 1) * Cfg::kABytes;
#pragma unroll
          for (int half = 0; half < (SPLIT_A ? 2 : 1); ++half) {
            const uint32_t a_addr = st + half * Cfg::kABytes;
#pragma unroll
            for (int k = 0; k < kGemmBK / 16; ++k) {
              umma_bf16(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), idesc,
                        (kb > g.kb0 || half > 0 || k > 0) ? 1u : 0u);
            }
          }
          if (CM > 1)
            umma_commit_mcast(&empty[stage], kClusterMask);
          else
            umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Drain: all MMAs issued by this thread complete before TMEM is released.
      umma_commit(drain);
      const uint32_t a = smem_u32(drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(a, 0u)) {
        if (clock64() - t0 > kWaitLimitCycles) {
          *abort_flag = 1;
          break;
        }
      }
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int lane_row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) break;
      tc_fence_after();
      const GemmUnit g = gemm_unit(u, m_tiles_s, n_tiles, k_splits, nk, m_group);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      epi(g.m_blk, g.n_blk, g.ks, lane_row, taddr,
          reinterpret_cast<float*>(epi_scratch) + quarter * (Epi::kScratchBytes / 16));
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    epi_drain(epi);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) raise_device_error(err, QUAIL_ERR_DEVICE_TIMEOUT, 1000 + blockIdx.x);
  // No CTA of a cluster leaves while another may still multicast into its
  // shared memory or arrive on its barriers: every producer has drained its
  // copies and every MMA thread its commits before reaching this point.
  if (CM > 1) cluster_sync();
}

// ------------------------------------------------------------ epilogues

// fp32 store of the partial tile of k-split ks:
//   C[ks * slab + row * ldc + col] = acc   (row < M, col < N)
// Each warp writes its 32 rows x 32 columns to shared memory in the 128-byte
// swizzled layout of the tensor map tm (a [ks][M][N] view of C) and one lane
// issues a bulk tile store, so a warp issues 8 stores per unit instead of
// 256. Two buffers per warp: the next chunk is written while the previous
// store still reads the other. The map clips rows >= M and columns >= N.
template <int BN>
struct EpiStoreF32 {
  static constexpr uint32_t kScratchBytes = 4 * 2 * 4096;
  CUtensorMap tm;
  __device__ __forceinline__ void operator()(int m_blk, int n_blk, int ks, int lane_row, uint32_t taddr,
                                             float* ws) const {
    const int lane = threadIdx.x & 31;
    const int row0 = m_blk * kGemmBM + lane_row - lane;  // this warp's first row
    const int n0 = n_blk * BN;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float* buf = ws + (c & 1) * 1024;  // 4 KB: 32 rows x 128 bytes
      float v[32];
      tmem_ld_32cols(taddr + c * 32, v);
      if (lane == 0) bulk_wait_group_read<1>();  // the store that last read this buffer is done with it
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 8; ++q)  // 16-byte chunk q of row `lane` at chunk position q ^ (lane & 7)
        *reinterpret_cast<float4*>(buf + lane * 32 + ((q ^ (lane & 7)) << 2)) =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      fence_proxy_async_smem();  // the tile writes, visible to the bulk copy
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm, buf, n0 + c * 32, row0, ks);
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

}  // namespace quail
