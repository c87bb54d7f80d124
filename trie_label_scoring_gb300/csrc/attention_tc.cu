// Doc-part attention on tcgen05 for many query rows per KV head (hundreds to
// thousands of evaluated trie nodes x G query heads). Same math as
// attn_doc_kernel in attention.cu ("To Classify, Try a Trie Tree", sec. 3.2:
// every evaluated node attends to the document; the tree part and the merge
// are shared), but a CTA owns a 128-row query tile and the two products run on
// the 5th-generation tensor cores with fp32 accumulators in TMEM:
//   S   = Q_hi K^T + Q_lo K^T          (M 128 rows, N 64 keys, K 128 dims)
//   O  += P_hi V   + P_lo V            (M 128 rows, N 128 dims, K 64 keys)
// per block of 64 keys (4 pages). Q and P are two-term bf16 splits (as in the
// mma.sync path); K comes from the TMA page ring as a K-major operand and V,
// unchanged, as an MN-major one (dims contiguous).
//
// Roles (192 threads): warp 0 loads pages with TMA, warp 1 owns TMEM and issues
// the MMAs, warps 2..5 (one thread per query row) build Q, run the softmax
// (lazy reference max, as in attention.cu), write P, and finish the rows.
#include "attn_common.cuh"
#include "kernels.h"
#include "quail_internal.h"
#include "sm103.cuh"

namespace quail {

namespace {

constexpr int kTcThreads = 192;
constexpr int kTcRows = 128;
constexpr int kTcBlkKeys = 64;                    // keys per block = 4 pages
constexpr int kTcStages = 3;
constexpr int kTcMaxPages = 256;                  // split_tokens <= 4096
constexpr uint32_t kTcQPart = 2 * 128 * 128;      // 32 KB: 2 dim-halves x 128 rows x 128 B
constexpr uint32_t kTcKVHalf = kTcBlkKeys * 128;  // 8 KB: 64 keys x 128 B
constexpr uint32_t kTcStage = 4 * kTcKVHalf;      // K lo|hi, V lo|hi = 32 KB
constexpr uint32_t kTcPPart = 128 * 128;          // 16 KB: 128 rows x 64 keys x 2 B
constexpr uint32_t kOffKV = 2 * kTcQPart;
constexpr uint32_t kOffP = kOffKV + kTcStages * kTcStage;
constexpr uint32_t kOffBar = kOffP + 2 * kTcPPart;
constexpr size_t kTcSmem = 1024 + kOffBar + 256 + kTcMaxPages * 4;
constexpr uint32_t kTmemCols = 256;  // S double buffer (2 x 64) + O (128)
constexpr uint32_t kTmemO = 128;

// 16-byte chunk c of row r in a 128B-swizzled region of 128-byte rows.
__device__ __forceinline__ uint32_t sw_off(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_doc_tc_kernel(AttnArgs a, RopeTable rt, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(base + kOffBar);
  uint64_t* kv_empty = kv_full + kTcStages;
  uint64_t* s_full = kv_empty + kTcStages;  // [2]
  uint64_t* s_empty = s_full + 2;           // [2]
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 1;
  uint64_t* q_full = p_empty + 1;
  uint64_t* drain = q_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_pages = reinterpret_cast<int*>(base + kOffBar + 256);

  const int slot = blockIdx.z;
  if (a.map.n_slots_dev != nullptr && slot >= *a.map.n_slots_dev) return;
  const int split = blockIdx.x;
  const int row_tiles = a.rows_pad / kTcRows;
  const int g = blockIdx.y / row_tiles;
  const int rt_idx = blockIdx.y % row_tiles;
  const int doc = row_doc(a.map, slot);
  const int L = a.doc_len[doc];
  if (L < 1 || L > a.max_doc_len) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) raise_device_error(a.err, QUAIL_ERR_DEVICE_BOUNDS, doc);
    return;
  }
  const int k_lo = split * a.split_tokens;
  if (k_lo >= L) return;
  const int k_hi = min(L, k_lo + a.split_tokens);
  const int p0 = k_lo / 16;
  const int n_pages = (k_hi - k_lo + 15) / 16;
  const int n_blocks = (n_pages + 3) / 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(p_empty, 1);
    mbar_init(q_full, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ page loader
    const int* pt = a.page_table + static_cast<size_t>(doc) * a.max_pages;
    for (int j = lane; j < n_pages; j += 32) s_pages[j] = pt[p0 + j];
    __syncwarp();
    if (lane == 0) {
      int armed[kTcStages];
#pragma unroll
      for (int s = 0; s < kTcStages; ++s) armed[s] = -1;
      for (int blk = 0; blk < n_blocks; ++blk) {
        const int s = blk % kTcStages;
        const int use = blk / kTcStages;
        if (use > 0 && !mbar_wait(&kv_empty[s], static_cast<uint32_t>((use - 1) & 1), abort_flag)) break;
        const int np = min(4, n_pages - blk * 4);
        int good = 0;
        for (int q = 0; q < np; ++q) {
          const int phys = s_pages[blk * 4 + q];
          good += (phys >= 0 && phys < a.num_pages) ? 1 : 0;
        }
        if (good < np) raise_device_error(a.err, QUAIL_ERR_DEVICE_BOUNDS, doc);
        armed[s] = -1;
        if (good == 0) {
          mbar_arrive(&kv_full[s]);  // release the consumer on stale data; results of this doc are void
          continue;
        }
        uint8_t* st = base + kOffKV + s * kTcStage;
        mbar_arrive_expect_tx(&kv_full[s], good * 4 * 2048);
        for (int q = 0; q < np; ++q) {
          const int phys = s_pages[blk * 4 + q];
          if (phys < 0 || phys >= a.num_pages) continue;
          const int y = (phys * a.hkv + g) * 16;
          tma_load_2d(st + q * 2048, &tmK, &kv_full[s], 0, y);
          tma_load_2d(st + kTcKVHalf + q * 2048, &tmK, &kv_full[s], 64, y);
          tma_load_2d(st + 2 * kTcKVHalf + q * 2048, &tmV, &kv_full[s], 0, y);
          tma_load_2d(st + 3 * kTcKVHalf + q * 2048, &tmV, &kv_full[s], 64, y);
        }
        armed[s] = use & 1;
      }
      for (int s = 0; s < kTcStages; ++s) {  // no copy may still be landing when the CTA exits
        if (armed[s] < 0) continue;
        const uint32_t ad = smem_u32(&kv_full[s]);
        const long long t0 = clock64();
        while (!mbar_try_wait(ad, static_cast<uint32_t>(armed[s]))) {
          if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16_f32(kTcRows, kTcBlkKeys);
      constexpr uint32_t idesc_pv = umma_idesc_bf16_f32_bmn(kTcRows, 128);
      const uint32_t q_addr = smem_u32(base);
      const uint32_t p_addr = smem_u32(base + kOffP);
      // O += (P_hi + P_lo) V for block j, once the softmax has written P_j.
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait(p_full, static_cast<uint32_t>(j & 1), abort_flag)) return false;
        tc_fence_after();
        const int s = j % kTcStages;
        const uint32_t v_addr = smem_u32(base + kOffKV + s * kTcStage + 2 * kTcKVHalf);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 16 keys = one page per instruction
            umma_bf16(tmem_base + kTmemO, smem_desc_sw128(p_addr + part * kTcPPart + kk * 32),
                      smem_desc_sw128_mn(v_addr + kk * 2048, kTcKVHalf, 1024), idesc_pv,
                      (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(p_empty);
        umma_commit(&kv_empty[s]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0u, abort_flag);
      if (ok) tc_fence_after();
      for (int blk = 0; blk < n_blocks && ok; ++blk) {
        const int s = blk % kTcStages;
        const int sb = blk & 1;
        if (!mbar_wait(&kv_full[s], static_cast<uint32_t>((blk / kTcStages) & 1), abort_flag) ||
            (blk >= 2 && !mbar_wait(&s_empty[sb], static_cast<uint32_t>(((blk >> 1) - 1) & 1), abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(base + kOffKV + s * kTcStage);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {  // 16 dims per instruction; dims 0..63 in half 0
            umma_bf16(tmem_base + sb * kTcBlkKeys,
                      smem_desc_sw128(q_addr + part * kTcQPart + (ks >> 2) * 16384 + (ks & 3) * 32),
                      smem_desc_sw128(k_addr + (ks >> 2) * kTcKVHalf + (ks & 3) * 32), idesc_s,
                      (part | ks) != 0 ? 1u : 0u);
          }
        }
        umma_commit(&s_full[sb]);
        if (blk >= 1 && !issue_pv(blk - 1)) ok = false;
      }
      if (ok && n_blocks >= 1) issue_pv(n_blocks - 1);
      // Drain: all MMAs issued by this thread complete before TMEM is released.
      umma_commit(drain);
      const uint32_t ad = smem_u32(drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(ad, 0u)) {
        if (clock64() - t0 > kWaitLimitCycles) {
          *abort_flag = 1;
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------ softmax warps: one thread per query row
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // TMEM lane of this row
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const int G = a.hq / a.hkv;
    const int rows_per_kv = (a.map.slot_node ? 1 : a.map.nq) * G;
    const int rr = rt_idx * kTcRows + row;
    const bool row_ok = rr < rows_per_kv;
    int node = 0, h = 0, e = 0;
    if (row_ok) {
      e = rr / G;
      h = g * G + rr % G;
      node = row_node(a.map, slot, e);
    }
    // Q row: RoPE at l_i + depth, two-term bf16 split, K-major 128B-swizzled.
    {
      const float* q = row_ok ? a.qkv + static_cast<size_t>(node) * a.ldq + h * 128 : nullptr;
      const int pos = row_ok ? L + a.node_depth[node] : 0;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {  // dims 8c..8c+7 (half 0) and 64+8c.. (half 1)
        uint32_t h0[4], l0[4], h1[4], l1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float y[4] = {0.f, 0.f, 0.f, 0.f};  // dims j, j+1 and j+64, j+65
          if (row_ok) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = c * 8 + 2 * i + u;
              float cs, sn;
              rope_cs(pos, rt.w[j], cs, sn);
              const float x1 = q[j], x2 = q[j + 64];
              y[u] = x1 * cs - x2 * sn;
              y[2 + u] = x2 * cs + x1 * sn;
            }
          }
          split_bf16(y[0], y[1], h0[i], l0[i]);
          split_bf16(y[2], y[3], h1[i], l1[i]);
        }
        const uint32_t off = sw_off(row, c);
        *reinterpret_cast<uint4*>(base + off) = make_uint4(h0[0], h0[1], h0[2], h0[3]);
        *reinterpret_cast<uint4*>(base + 16384 + off) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
        *reinterpret_cast<uint4*>(base + kTcQPart + off) = make_uint4(l0[0], l0[1], l0[2], l0[3]);
        *reinterpret_cast<uint4*>(base + kTcQPart + 16384 + off) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    const float scale = kAttnLog2e * 0.08838834764831845f;  // log2(e) / sqrt(128)
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int blk = 0; blk < n_blocks; ++blk) {
      const int sb = blk & 1;
      const int s = blk % kTcStages;
      // waits are made warp-uniform: the warp-collective tcgen05.ld / __any_sync
      // below must never run with lanes that left the loop
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], static_cast<uint32_t>((blk >> 1) & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s0[32], s1[32];
      tmem_ld_32cols(lane_addr + sb * kTcBlkKeys, s0);
      tmem_ld_32cols(lane_addr + sb * kTcBlkKeys + 32, s1);
      tc_fence_before();
      mbar_arrive(&s_empty[sb]);
      const int valid = min(kTcBlkKeys, k_hi - (k_lo + blk * kTcBlkKeys));
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s0[i] = i < valid ? s0[i] * scale : -INFINITY;
        s1[i] = i + 32 < valid ? s1[i] * scale : -INFINITY;
        mx = fmaxf(mx, fmaxf(s0[i], s1[i]));
      }
      // PV of the previous block must be done before P is overwritten (and O rescaled).
      if (blk >= 1 &&
          !__all_sync(0xffffffffu, mbar_wait(p_empty, static_cast<uint32_t>((blk - 1) & 1), abort_flag))) {
        ok = false;
        break;
      }
      // Lazy reference max (see attention.cu): moves only past +8 in base 2.
      const bool need = mx > m_ref + 8.f;
      float alpha = 1.f;
      if (need) {
        const float nm = fmaxf(m_ref, mx);
        alpha = exp2f(m_ref - nm);
        m_ref = nm;
        l_sum *= alpha;
      }
      if (blk >= 1 && __any_sync(0xffffffffu, need)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld_32cols(lane_addr + kTmemO + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st_32cols(lane_addr + kTmemO + c * 32, o);
        }
      }
      // P = exp2(s - m_ref) as a two-term bf16 split, K-major 128B-swizzled rows.
      float psum = 0.f;
      uint8_t* prow = base + kOffP;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = c < 4 ? s0[c * 8 + 2 * i] : s1[(c - 4) * 8 + 2 * i];
          const float x1 = c < 4 ? s0[c * 8 + 2 * i + 1] : s1[(c - 4) * 8 + 2 * i + 1];
          const float e0 = exp2f(x0 - m_ref), e1 = exp2f(x1 - m_ref);
          psum += e0 + e1;
          split_bf16(e0, e1, ph[i], pl[i]);
        }
        const uint32_t off = sw_off(row, c);
        *reinterpret_cast<uint4*>(prow + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        *reinterpret_cast<uint4*>(prow + kTcPPart + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
      }
      l_sum += psum;
      // Keys past the document end (tail of the last page, pages not loaded):
      // zero their V rows so stale contents cannot reach O through P = 0.
      if (valid < kTcBlkKeys) {
        uint8_t* vst = base + kOffKV + s * kTcStage + 2 * kTcKVHalf;
        const int t = threadIdx.x - 64;  // 0..127
        for (int idx = t; idx < (kTcBlkKeys - valid) * 16; idx += 128) {
          const int r = valid + idx / 16, hc = idx % 16;
          *reinterpret_cast<uint4*>(vst + (hc / 8) * kTcKVHalf + r * 128 + (hc % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // Row epilogue once the last PV has landed in TMEM.
    if (ok && n_blocks > 0 &&
        __all_sync(0xffffffffu, mbar_wait(p_empty, static_cast<uint32_t>((n_blocks - 1) & 1), abort_flag))) {
      tc_fence_after();
      const bool fused = a.n_splits == 1;
      float f1 = 1.f, f2 = 0.f, inv = 1.f;
      const float* to = nullptr;
      bf16* dst = nullptr;
      float* pdst = nullptr;
      if (row_ok && fused) {
        const float2 tml = a.tree_ml[static_cast<size_t>(node) * a.hq + h];
        const float M = fmaxf(m_ref, tml.x);
        f1 = exp2f(m_ref - M);
        f2 = exp2f(tml.x - M);
        inv = 1.f / (f1 * l_sum + f2 * tml.y);
        to = a.tree_o + (static_cast<size_t>(node) * a.hq + h) * 128;
        dst = a.out + (static_cast<size_t>(slot) * a.map.nq + e) * 2 * a.hq * 128 + h * 128;
      } else if (row_ok) {
        const size_t pr =
            ((static_cast<size_t>(slot) * a.hkv + g) * a.n_splits + split) * static_cast<size_t>(a.rows_pad) + rr;
        pdst = a.part_o + pr * 128;
        a.part_ml[pr] = make_float2(m_ref, l_sum);
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld_32cols(lane_addr + kTmemO + c * 32, o);
        if (dst != nullptr) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int col = c * 32 + i + 2 * u;
              split_bf16((f1 * o[i + 2 * u] + f2 * to[col]) * inv, (f1 * o[i + 2 * u + 1] + f2 * to[col + 1]) * inv,
                         hv[u], lv[u]);
            }
            *reinterpret_cast<uint4*>(dst + c * 32 + i) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4*>(dst + a.hq * 128 + c * 32 + i) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
          }
        } else if (pdst != nullptr) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(pdst + c * 32 + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) raise_device_error(a.err, QUAIL_ERR_DEVICE_TIMEOUT, 3000 + slot);
}

}  // namespace

}  // namespace quail

namespace quail {

size_t attn_tc_smem_bytes() { return kTcSmem; }

cudaError_t launch_attn_doc_tc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV, cudaStream_t st) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(attn_doc_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kTcSmem));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(a.n_splits, a.hkv * (a.rows_pad / kTcRows), a.n_slots);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  attn_doc_tc_kernel<<<grid, kTcThreads, kTcSmem, st>>>(a, make_rope_table(a.theta), tmK, tmV);
  return cudaGetLastError();
}

}  // namespace quail
