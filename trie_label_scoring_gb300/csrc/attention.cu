// Tree-masked GQA attention for trie nodes ("To Classify, Try a Trie Tree",
// sec. 3.2 "Custom attention kernel": all evaluated nodes of a document in one
// request, each attending to the prompt and to the nodes on its own path).
//
// The attention of node v in document i splits into two disjoint key sets,
// merged with the log-sum-exp / online-softmax rule ("Building an Ultra-High
// Throughput AI-SQL Engine", sec. 3.2.4, join attention in two parts):
//   doc part  -- the l_i cached document keys, read once per (document, KV head)
//                for ALL of that document's nodes and query heads;
//   tree part -- v's ancestors and v itself. Keys sit at positions l_i + depth,
//                so q(l_i+dv).k(l_i+du) = q . R(du - dv) k: the tree part does
//                not depend on the document and is computed once per call.
#include <cfloat>

#include "kernels.h"
#include "launch.cuh"
#include "quail_internal.h"
#include "sm103.cuh"
#include "attn_common.cuh"

namespace quail {

namespace {

constexpr int kPage = 16;
constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = 160;  // warps 0..3 consume, warp 4 loads pages
constexpr uint32_t kHalfBytes = kPage * 64 * 2;   // 16 keys x 64 bf16, 128B-swizzled
constexpr uint32_t kPageBytes = 4 * kHalfBytes;   // K[0:64) K[64:128) V[0:64) V[64:128)

// Byte offset of 16-byte chunk `c` (0..7) of key row `r` in a 128B-swizzled half tile.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ tree part
// Warp per (node, KV head, group of up to kTreeHeads query heads): online
// softmax over the node's ancestors and itself with relative RoPE; fp32 q, k,
// v straight from the projection. Each ancestor's k and v row and its
// rotation are loaded and computed once for the query heads that share them.
constexpr int kTreeHeads = 4;

__global__ void tree_part_kernel(AttnArgs a, RopeTable rt) {
  grid_dependency_wait();
  // Everything before this kernel is complete now, so the doc-part kernel may
  // launch: it streams its KV pages and builds its Q tiles meanwhile, and
  // waits for this kernel only before it reads the tree part.
  grid_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.hq / a.hkv;
  const int chunks = (G + kTreeHeads - 1) / kTreeHeads;
  const int per_node = a.hkv * chunks;
  if (warp >= a.n_nodes * per_node) return;
  const int node = warp / per_node, rem = warp - node * per_node;
  const int g = rem / chunks, ch = rem - g * chunks;
  if (a.nodes_live != nullptr && node >= *a.nodes_live) return;
  const int h0 = g * G + ch * kTreeHeads;
  const int nh = min(kTreeHeads, G - ch * kTreeHeads);
  float q[kTreeHeads][4];
#pragma unroll
  for (int i = 0; i < kTreeHeads; ++i) {
    if (i < nh) {
      const float* qr = a.qkv + static_cast<size_t>(node) * a.ldq + (h0 + i) * 128;
      q[i][0] = qr[lane];
      q[i][1] = qr[lane + 32];
      q[i][2] = qr[lane + 64];
      q[i][3] = qr[lane + 96];
    }
  }
  const float2 w0 = rt.w[lane], w1 = rt.w[lane + 32];
  const float scale = kAttnLog2e * 0.08838834764831845f;  // log2(e) / sqrt(128)
  const int dnode = a.node_depth[node];
  float m[kTreeHeads], l[kTreeHeads], o[kTreeHeads][4];
#pragma unroll
  for (int i = 0; i < kTreeHeads; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
    o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }
  int anc = node;
  for (int guard = 0; anc >= 0 && guard < 4096; ++guard) {
    const float* kr = a.qkv + static_cast<size_t>(anc) * a.ldq + (a.hq + g) * 128;
    const float* vr = a.qkv + static_cast<size_t>(anc) * a.ldq + (a.hq + a.hkv + g) * 128;
    const float delta = static_cast<float>(a.node_depth[anc] - dnode);
    float c0, s0, c1, s1;
    sincosf(delta * w0.x, &s0, &c0);
    sincosf(delta * w1.x, &s1, &c1);
    const float k0 = kr[lane], k1 = kr[lane + 32], k2 = kr[lane + 64], k3 = kr[lane + 96];
    const float v0 = vr[lane], v1 = vr[lane + 32], v2 = vr[lane + 64], v3 = vr[lane + 96];
    const float r0 = k0 * c0 - k2 * s0, r2 = k2 * c0 + k0 * s0, r1 = k1 * c1 - k3 * s1, r3 = k3 * c1 + k1 * s1;
#pragma unroll
    for (int i = 0; i < kTreeHeads; ++i) {
      if (i < nh) {
        float dot = q[i][0] * r0 + q[i][2] * r2 + q[i][1] * r1 + q[i][3] * r3;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float sc = dot * scale;
        const float nm = fmaxf(m[i], sc);
        const float alpha = exp2f(m[i] - nm), p = exp2f(sc - nm);
        l[i] = l[i] * alpha + p;
        o[i][0] = o[i][0] * alpha + p * v0;
        o[i][1] = o[i][1] * alpha + p * v1;
        o[i][2] = o[i][2] * alpha + p * v2;
        o[i][3] = o[i][3] * alpha + p * v3;
        m[i] = nm;
      }
    }
    anc = a.node_parent[anc];
  }
#pragma unroll
  for (int i = 0; i < kTreeHeads; ++i) {
    if (i < nh) {
      const int h = h0 + i;
      float* to = a.tree_o + (static_cast<size_t>(node) * a.hq + h) * 128;
      to[lane] = o[i][0];
      to[lane + 32] = o[i][1];
      to[lane + 64] = o[i][2];
      to[lane + 96] = o[i][3];
      if (lane == 0) a.tree_ml[static_cast<size_t>(node) * a.hq + h] = make_float2(m[i], l[i]);
    }
  }
}

// ------------------------------------------------------------------ slot order
// One block: a counting sort of the slots by document pages, longest first.
// Slots whose document length is out of range sort as empty documents; slots
// past the live count go last. The order of equal keys is whatever the
// shared-memory atomics give: it changes only which CTA runs when, never a
// result.
constexpr int kOrderBins = 1024;
constexpr int kOrderThreads = 1024;

__global__ void __launch_bounds__(kOrderThreads) slot_order_kernel(AttnArgs a) {
  __shared__ int hist[kOrderBins];
  __shared__ int warp_tot[kOrderThreads / 32];
  grid_dependency_wait();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  hist[t] = 0;  // kOrderBins == kOrderThreads
  __syncthreads();
  const int live = a.map.n_slots_dev != nullptr ? min(*a.map.n_slots_dev, a.n_slots) : a.n_slots;
  auto bin_of = [&](int s) {
    if (s >= live) return kOrderBins - 1;
    const int L = a.doc_len[row_doc(a.map, s)];
    const int pages = (L >= 1 && L <= a.max_doc_len) ? (L + 15) / 16 : 0;
    return (kOrderBins - 2) - min(pages, kOrderBins - 2);
  };
  for (int s = t; s < a.n_slots; s += kOrderThreads) atomicAdd(&hist[bin_of(s)], 1);
  __syncthreads();
  // exclusive scan of hist (bin t) across the block
  const int v = hist[t];
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w - warp_tot[lane];  // exclusive prefix of the warp totals
  }
  __syncthreads();
  hist[t] = warp_tot[warp] + x - v;  // first position of bin t
  __syncthreads();
  for (int s = t; s < a.n_slots; s += kOrderThreads) a.slot_order[atomicAdd(&hist[bin_of(s)], 1)] = s;
}

// ------------------------------------------------------------------ doc part
// CTA = (split, kv head x row group, slot). Warp 4 streams the split's KV pages
// (K and V of one KV head: 8 KB per page) into an 8-stage ring with TMA; warps
// 0..3 run bf16 mma.sync on one 16-row query tile with an online softmax:
// the four warps share the 16 rows, take pages round-robin, then merge.
// The q fragments (RoPE at l_i + depth, two-term bf16 split) are built once
// per CTA in shared memory in mma fragment order. With one split per
// document the epilogue merges the tree part and writes O itself; otherwise
// it writes (O, max, sum) partials for attn_combine_kernel.
constexpr uint32_t kQTileBytes = 8 * 2 * 32 * 16;  // ks x {hi, lo} x lane x uint4
constexpr int kMaxSplitPagesV2 = 256;              // split_tokens <= 4096

// The four consumer warps merge their softmax states through the page ring
// once every page has been consumed (16 rows x 128 dims + 32 floats each);
// the ring region is sized to hold that merge too.
constexpr uint32_t kMergeBytes = kConsumerWarps * (16 * 128 + 32) * 4;

// The page ring: STAGES pages (a multiple of kConsumerWarps, so stage s is
// always read by warp s % 4). Short splits run 8 stages at three CTAs per SM,
// so one CTA's fixed work (Q build, merge, epilogue) overlaps two others'
// pages; long splits run 12 stages at two CTAs per SM, so the loader keeps
// streaming through the Q build of its own CTA.
template <int STAGES>
struct AttnRing {
  static_assert(STAGES % kConsumerWarps == 0, "each stage must belong to one consumer warp");
  static constexpr uint32_t kRingBytes = STAGES * kPageBytes > kMergeBytes ? STAGES * kPageBytes : kMergeBytes;
  static constexpr size_t kSmemBytes = 1024 + kRingBytes + kQTileBytes + 2 * STAGES * 8 + 16 + kMaxSplitPagesV2 * 4;
  static constexpr int kCtasPerSm = STAGES <= 8 ? 3 : 2;
};
constexpr int kLongSplitPages = 65;  // splits longer than 1,024 tokens take the 12-stage ring

__device__ __forceinline__ void mma_pair(float (&d0)[4], float (&d1)[4], const uint4& a, uint32_t b0, uint32_t b1,
                                         uint32_t b2, uint32_t b3) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  mma_bf16(d0, av, b0, b1);
  mma_bf16(d1, av, b2, b3);
}

template <int kAttnStages>
__global__ void __launch_bounds__(kAttnThreads, AttnRing<kAttnStages>::kCtasPerSm)
    attn_doc_kernel(AttnArgs a, RopeTable rt, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
  // No grid_dependency_wait here: tree_part_kernel, the kernel before this
  // one, lets it launch only after its own wait, so the document KV, page
  // table and lengths (inputs) and q and the row maps (written before
  // tree_part) are complete. Only the tree part itself is waited for, below.
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kRingBytes = AttnRing<kAttnStages>::kRingBytes;
  uint8_t* s_q = base + kRingBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_q + kQTileBytes);
  uint64_t* empty = full + kAttnStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kAttnStages);
  int* s_pages = reinterpret_cast<int*>(empty + kAttnStages) + 4;  // physical page of each split page

  // Slots run longest document first (slot_order_kernel, complete before
  // tree_part_kernel passed its wait), so the last wave holds short CTAs.
  const int slot = a.slot_order != nullptr ? a.slot_order[blockIdx.z] : static_cast<int>(blockIdx.z);
  if (a.map.n_slots_dev != nullptr && slot >= *a.map.n_slots_dev) return grid_dependency_wait();
  const int split = blockIdx.x;
  const int n_row_groups = a.rows_pad / a.row_tile;
  const int g = blockIdx.y / n_row_groups;
  const int rg = blockIdx.y % n_row_groups;
  if (rows_past_end(a.map, slot, rg * a.row_tile / (a.hq / a.hkv)))  // a row group of padding only
    return grid_dependency_wait();
  const int doc = row_doc(a.map, slot);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.hq / a.hkv;
  const int nq_rows = (a.map.slot_node ? 1 : a.map.nq);
  const int rows_per_kv = nq_rows * G;
  const int t = threadIdx.x;
  const int k_lo = split * a.split_tokens;
  const int p0 = k_lo / kPage;

  // Every load the CTA needs before its first copy goes out at once: the
  // document length, the split's page ids (loader warp; up to a full split,
  // trimmed to the document below) and the q items with their node depths
  // (consumers). item = (row r, pair j) -> dims j and j + 64 (j = t % 64
  // for every item, since 128 threads step 128 items).
  const int L = a.doc_len[doc];
  constexpr int kIdRegs = kMaxSplitPagesV2 / 32;
  int ids[kIdRegs];
  if (warp == kConsumerWarps) {
    const int* pt = a.page_table + static_cast<size_t>(doc) * a.max_pages + p0;
    const int avail = min(a.split_tokens / kPage, a.max_pages - p0);
#pragma unroll
    for (int k = 0; k < kIdRegs; ++k) ids[k] = (lane + 32 * k < avail) ? pt[lane + 32 * k] : 0;
  }
  constexpr int kPer = 16 * 64 / (kConsumerWarps * 32);  // items per thread
  float x1[kPer], x2[kPer];
  int dep[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    x1[k] = x2[k] = 0.f;
    dep[k] = -1;
  }
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int it = t + k * kConsumerWarps * 32;
      const int r = it / 64, j = it % 64;
      const int rr = rg * a.row_tile + r;  // row within (slot, kv head)
      if (rr < rows_per_kv) {
        const int e = rr / G, hl = rr % G;
        const int node = row_node(a.map, slot, e);
        const float* q = a.qkv + static_cast<size_t>(node) * a.ldq + (g * G + hl) * 128;
        x1[k] = q[j];
        x2[k] = q[j + 64];
        dep[k] = a.node_depth[node];
      }
    }
  }
  if (L < 1 || L > a.max_doc_len) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) raise_device_error(a.err, QUAIL_ERR_DEVICE_BOUNDS, doc);
    return grid_dependency_wait();  // every exit waits, so this grid ends after the ones before it
  }
  if (k_lo >= L) return grid_dependency_wait();
  const int k_hi = min(L, k_lo + a.split_tokens);
  const int n_pages = (k_hi - k_lo + kPage - 1) / kPage;
  int pos[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) pos[k] = dep[k] >= 0 ? L + dep[k] : -1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------ page loader
#pragma unroll
    for (int k = 0; k < kIdRegs; ++k)
      if (lane + 32 * k < n_pages) s_pages[lane + 32 * k] = ids[k];
    __syncwarp();
    if (lane == 0) {
      int armed[kAttnStages];
#pragma unroll
      for (int s = 0; s < kAttnStages; ++s) armed[s] = -1;
      for (int j = 0; j < n_pages; ++j) {
        const int s = j % kAttnStages;
        const int use = j / kAttnStages;
        if (use > 0 && !mbar_wait(&empty[s], static_cast<uint32_t>((use - 1) & 1), abort_flag)) break;
        const int phys = s_pages[j];
        if (phys < 0 || phys >= a.num_pages) {
          raise_device_error(a.err, QUAIL_ERR_DEVICE_BOUNDS, doc);
          mbar_arrive(&full[s]);  // release the consumer on stale data; results of this doc are void
          armed[s] = -1;
          continue;
        }
        uint8_t* dst = base + s * kPageBytes;
        const int y = (phys * a.hkv + g) * kPage;
        mbar_arrive_expect_tx(&full[s], kPageBytes);
        tma_load_2d(dst, &tmK, &full[s], 0, y);
        tma_load_2d(dst + kHalfBytes, &tmK, &full[s], 64, y);
        tma_load_2d(dst + 2 * kHalfBytes, &tmV, &full[s], 0, y);
        tma_load_2d(dst + 3 * kHalfBytes, &tmV, &full[s], 64, y);
        armed[s] = use & 1;
      }
      for (int s = 0; s < kAttnStages; ++s) {  // no copy may still be landing when the CTA exits
        if (armed[s] < 0) continue;
        const uint32_t ad = smem_u32(&full[s]);
        const long long t0 = clock64();
        while (!mbar_try_wait(ad, static_cast<uint32_t>(armed[s]))) {
          if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            break;
          }
        }
      }
    }
    grid_dependency_wait();
    return;  // the loader warp takes no part in the consumers' named barrier
  }

  // -------------------------------------------------- consumers
  const int gq = lane >> 2, tq = lane & 3;

  // q fragments: item = (row, pair j) -> rotated dims j and j + 64, split
  // into hi/lo bf16 and scattered to their (ks, lane, register, half) slots.
  {
    uint16_t* sq16 = reinterpret_cast<uint16_t*>(s_q);
    const float2 wj = rt.w[t & 63];  // the one frequency this thread needs
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int it = t + k * kConsumerWarps * 32;
      const int r = it / 64, j = it % 64;
      float y0 = 0.f, y1 = 0.f;
      if (pos[k] >= 0) {
        float c, sn;
        rope_cs(pos[k], wj, c, sn);
        y0 = x1[k] * c - x2[k] * sn;
        y1 = x2[k] * c + x1[k] * sn;
      }
      const int col = j % 16;
      const int reg = (r >= 8 ? 1 : 0) + (col >= 8 ? 2 : 0);
      const int ln = (r % 8) * 4 + (col % 8) / 2;
      const int half = col & 1;
#pragma unroll
      for (int w = 0; w < 2; ++w) {  // dims j (ks = j / 16) and j + 64 (ks + 4)
        const float y = w ? y1 : y0;
        const int ks = j / 16 + 4 * w;
        const __nv_bfloat16 hb = __float2bfloat16(y);
        const __nv_bfloat16 lb = __float2bfloat16(y - __bfloat162float(hb));
        const int idx = ((ks * 2 + 0) * 32 + ln) * 8 + reg * 2 + half;  // in bf16 units
        sq16[idx] = *reinterpret_cast<const uint16_t*>(&hb);
        sq16[idx + 32 * 8] = *reinterpret_cast<const uint16_t*>(&lb);
      }
    }
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  const uint4* qf = reinterpret_cast<const uint4*>(s_q) + lane;  // [ks][hi/lo][lane]

  const float scale = kAttnLog2e * 0.08838834764831845f;
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  for (int j = warp; j < n_pages; j += kConsumerWarps) {  // pages round-robin over the warps
    const int s = j % kAttnStages;
    // warp-uniform wait: the shuffles and __any_sync below need every lane
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>((j / kAttnStages) & 1), abort_flag)))
      break;
    const uint32_t kb = smem_u32(base + s * kPageBytes);
    const uint32_t vb = kb + 2 * kHalfBytes;
    const int key0 = (p0 + j) * kPage;
    const int valid = min(kPage, L - key0);  // >= 1

    // S = (q_hi + q_lo) K^T for 16 keys; four independent accumulator chains
    float sh[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float sl[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int mi = lane >> 3, ri = lane & 7;
      const uint32_t key = (mi >> 1) * 8 + ri;
      const uint32_t chunk = (ks & 3) * 2 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb + (ks >> 2) * kHalfBytes + swz(key, chunk), b0, b1, b2, b3);
      const uint4 qh = qf[(ks * 2 + 0) * 32];
      const uint4 ql = qf[(ks * 2 + 1) * 32];
      mma_pair(sh[0], sh[1], qh, b0, b1, b2, b3);
      mma_pair(sl[0], sl[1], ql, b0, b1, b2, b3);
    }
    // online softmax (base 2); rows gq (c0, c1) and gq + 8 (c2, c3)
    float sc[2][4];
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = nt * 8 + tq * 2 + (c & 1);
        sc[nt][c] = key < valid ? (sh[nt][c] + sl[nt][c]) * scale : -INFINITY;
        mx[c >> 1] = fmaxf(mx[c >> 1], sc[nt][c]);
      }
    }
    // Lazy rescale: the reference max m_r only moves when a row max exceeds it
    // by more than 8 (base 2), so p <= 256 stays far from fp32 overflow and the
    // O rescale (64 multiplies) is skipped on almost every page. Exact: O, l
    // and m_r always describe sum_j exp2(s_j - m_r) (v_j, 1).
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
    }
    if (__any_sync(0xffffffffu, mx[0] > m_r[0] + 8.f || mx[1] > m_r[1] + 8.f)) {
      float alpha[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const float nm = fmaxf(m_r[hr], mx[hr]);
        alpha[hr] = exp2f(m_r[hr] - nm);
        m_r[hr] = nm;
        l_r[hr] *= alpha[hr];
      }
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
    }
    // P as a two-term bf16 split (pa + pl = p to ~16 bits)
    uint32_t pa[4], pl[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const float e0 = exp2f(sc[nt][hr * 2] - m_r[hr]);
        const float e1 = exp2f(sc[nt][hr * 2 + 1] - m_r[hr]);
        l_r[hr] += e0 + e1;
        split_bf16(e0, e1, pa[nt * 2 + hr], pl[nt * 2 + hr]);
      }
    }
    // O += P V; V fragments via transposed ldmatrix. Keys past the document
    // end are zeroed in registers so stale slot contents never reach O.
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      const int mi = lane >> 3, ri = lane & 7;
      const uint32_t key = (mi & 1) * 8 + ri;
      const uint32_t chunk = (np & 3) * 2 + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vb + (np >> 2) * kHalfBytes + swz(key, chunk), b0, b1, b2, b3);
      if (valid < kPage) {
        const int k0 = tq * 2, k1 = tq * 2 + 8;
        const uint32_t m0 = (k0 < valid ? 0x0000ffffu : 0u) | (k0 + 1 < valid ? 0xffff0000u : 0u);
        const uint32_t m1 = (k1 < valid ? 0x0000ffffu : 0u) | (k1 + 1 < valid ? 0xffff0000u : 0u);
        b0 &= m0;
        b2 &= m0;
        b1 &= m1;
        b3 &= m1;
      }
      mma_bf16(o[np * 2], pa, b0, b1);
      mma_bf16(o[np * 2 + 1], pa, b2, b3);
      mma_bf16(o[np * 2], pl, b0, b1);
      mma_bf16(o[np * 2 + 1], pl, b2, b3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // full row sums
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 1);
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 2);
  }

  const bool fused = a.n_splits == 1;
  const size_t part_row0 =
      ((static_cast<size_t>(slot) * a.hkv + g) * a.n_splits + split) * static_cast<size_t>(a.rows_pad);
  // Thread t of the epilogue: row r = t / 8 and dims 8k .. 8k + 7, 64 + 8k ..
  // 64 + 8k + 7 (k = t % 8), so the 8 threads of a row write each 128-byte
  // half of a bf16 output row (or read each 256-byte run of a tree_o row)
  // together. Its tree-part values are requested before the merge, so their
  // latency overlaps it.
  const int r = t >> 3, k8 = t & 7;
  auto dim = [&](int i) { return (i < 8 ? 8 * k8 : 64 + 8 * k8 - 8) + i; };  // dim of acc[i]
  const bool out_row = fused && r < rows_per_kv;
  grid_dependency_wait();  // tree_part_kernel's outputs (and, by this wait, everything before this kernel)
  float tv[16];
  float2 tml = make_float2(-INFINITY, 0.f);
  int e_out = 0, h_out = 0;
  if (out_row) {
    e_out = r / G;
    h_out = g * G + r % G;
    const int node = row_node(a.map, slot, e_out);
    tml = a.tree_ml[static_cast<size_t>(node) * a.hq + h_out];
    const float* to = a.tree_o + (static_cast<size_t>(node) * a.hq + h_out) * 128;
#pragma unroll
    for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4*>(tv + i) = *reinterpret_cast<const float4*>(to + dim(i));
  }
  {
    // Merge the four warps' partial softmax states through the (now idle) page ring.
    asm volatile("bar.sync 1, 128;" ::: "memory");
    float* so = reinterpret_cast<float*>(base) + warp * (16 * 128 + 32);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = gq + hr * 8;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        *reinterpret_cast<float2*>(so + r * 128 + n * 8 + tq * 2) = make_float2(o[n][hr * 2], o[n][hr * 2 + 1]);
      if (tq == 0) {
        so[16 * 128 + r] = m_r[hr];
        so[16 * 128 + 16 + r] = l_r[hr];
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const float* s0 = reinterpret_cast<const float*>(base);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s0[w * (16 * 128 + 32) + 16 * 128 + r]);
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float* sw = s0 + w * (16 * 128 + 32);
      const float mw = sw[16 * 128 + r];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      lsum += f * sw[16 * 128 + 16 + r];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(sw + r * 128 + dim(i));
        acc[i] += f * v.x;
        acc[i + 1] += f * v.y;
        acc[i + 2] += f * v.z;
        acc[i + 3] += f * v.w;
      }
    }
    if (!fused) {
      float* dst = a.part_o + (part_row0 + r) * 128;
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(dst + dim(i)) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
      if (k8 == 0) a.part_ml[part_row0 + r] = make_float2(M, lsum);
    } else if (out_row) {
      const int e = e_out, h = h_out;
      const float M2 = fmaxf(M, tml.x);
      const float f1 = exp2f(M - M2), f2 = exp2f(tml.x - M2);
      const float inv = 1.f / (f1 * lsum + f2 * tml.y);
      bf16* orow = a.out + (static_cast<size_t>(slot) * a.map.nq + e) * 2 * a.hq * 128 + h * 128;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {  // dims 8k.. and 64 + 8k..: one 16-byte hi and lo store each
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = hf * 8 + 2 * u;
          split_bf16((f1 * acc[i] + f2 * tv[i]) * inv, (f1 * acc[i + 1] + f2 * tv[i + 1]) * inv, hv[u], lv[u]);
        }
        *reinterpret_cast<uint4*>(orow + dim(hf * 8)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(orow + a.hq * 128 + dim(hf * 8)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
      }
    }
  }
  if (threadIdx.x == 0 && *abort_flag) raise_device_error(a.err, QUAIL_ERR_DEVICE_TIMEOUT, 2000 + slot);
}

// ------------------------------------------------------------------ combine
// Block per output row (slot, node); warp per q head: merge the document
// splits with the tree part, normalise, write bf16 O.
__global__ void attn_combine_kernel(AttnArgs a) {
  grid_dependency_wait();
  const int row = blockIdx.x;
  const int nq = a.map.nq;
  const int slot = row / nq, e = row % nq;
  if (a.map.n_slots_dev != nullptr && slot >= *a.map.n_slots_dev) return;
  if (rows_past_end(a.map, slot, e)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.hq / a.hkv;
  const int doc = row_doc(a.map, slot);
  const int L = a.doc_len[doc];
  const int node = row_node(a.map, slot, e);
  const int rl_base = (a.map.slot_node ? 0 : e) * G;
  for (int h = warp; h < a.hq; h += blockDim.x >> 5) {
    const int g = h / G;
    const int rl = rl_base + h % G;
    const float2 tml = a.tree_ml[static_cast<size_t>(node) * a.hq + h];
    float M = tml.x;
    const bool doc_ok = L >= 1 && L <= a.max_doc_len;
    const int ns = doc_ok ? (L + a.split_tokens - 1) / a.split_tokens : 0;
    const size_t base = (static_cast<size_t>(slot) * a.hkv + g) * a.n_splits;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, a.part_ml[(base + s) * a.rows_pad + rl].x);
    float f = exp2f(tml.x - M);
    float l = f * tml.y;
    float4 acc = *reinterpret_cast<const float4*>(a.tree_o + (static_cast<size_t>(node) * a.hq + h) * 128 + lane * 4);
    acc.x *= f;
    acc.y *= f;
    acc.z *= f;
    acc.w *= f;
    for (int s = 0; s < ns; ++s) {
      const size_t pr = (base + s) * a.rows_pad + rl;
      const float2 ml = a.part_ml[pr];
      f = exp2f(ml.x - M);
      l += f * ml.y;
      const float4 v = *reinterpret_cast<const float4*>(a.part_o + pr * 128 + lane * 4);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    const float inv = 1.f / l;
    const float o0 = acc.x * inv, o1 = acc.y * inv, o2 = acc.z * inv, o3 = acc.w * inv;
    bf16* dst = a.out + static_cast<size_t>(row) * 2 * a.hq * 128 + h * 128 + lane * 4;
    uint32_t h01, l01, h23, l23;
    split_bf16(o0, o1, h01, l01);
    split_bf16(o2, o3, h23, l23);
    *reinterpret_cast<uint2*>(dst) = make_uint2(h01, h23);                 // O_hi
    *reinterpret_cast<uint2*>(dst + a.hq * 128) = make_uint2(l01, l23);    // O_lo

  }
}


}  // namespace

cudaError_t launch_tree_part(const AttnArgs& a, cudaStream_t st) {
  const int G = a.hq / a.hkv;
  const long warps = static_cast<long>(a.n_nodes) * a.hkv * ((G + kTreeHeads - 1) / kTreeHeads);
  if (warps <= 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(tree_part_kernel, dim3(static_cast<int>((warps * 32 + 255) / 256)), dim3(256), 0, st, a, make_rope_table(a.theta)); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

cudaError_t launch_slot_order(const AttnArgs& a, cudaStream_t st) {
  if (a.n_slots <= 0 || a.slot_order == nullptr) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(slot_order_kernel, dim3(1), dim3(kOrderThreads), 0, st, a); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

template <int STAGES>
cudaError_t launch_attn_doc_ring(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV, cudaStream_t st) {
  auto kern = attn_doc_kernel<STAGES>;
  constexpr size_t smem = AttnRing<STAGES>::kSmemBytes;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(a.n_splits, a.hkv * (a.rows_pad / a.row_tile), a.n_slots);
  if (grid.x == 0 || grid.z == 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(kern, dim3(grid), dim3(kAttnThreads), smem, st, a, make_rope_table(a.theta), tmK, tmV); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

bool attn_doc_wants_slot_order(const AttnArgs& a, int num_sms) {
  // Few waves: the last partial wave decides the kernel's end, and starting
  // the long documents first leaves short CTAs for it. Over many waves the
  // order is left alone: CTAs of equal length started together reach their
  // setup and merge phases together, and an SM then streams less. Within one
  // wave every CTA is resident at once and the order cannot matter.
  const int per_sm = a.split_tokens / kPage >= kLongSplitPages ? AttnRing<12>::kCtasPerSm : AttnRing<8>::kCtasPerSm;
  const long ctas = static_cast<long>(a.n_slots) * a.hkv * a.n_splits;
  return ctas > static_cast<long>(per_sm) * num_sms && 2 * ctas <= 3L * per_sm * num_sms;
}

cudaError_t launch_attn_doc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV, cudaStream_t st) {
  if (a.row_tile != 16 || a.rows_pad != 16) return cudaErrorInvalidValue;  // one shared 16-row tile
  if (a.split_tokens / kPage >= kLongSplitPages) return launch_attn_doc_ring<12>(a, tmK, tmV, st);
  return launch_attn_doc_ring<8>(a, tmK, tmV, st);
}

cudaError_t launch_attn_combine(const AttnArgs& a, cudaStream_t st) {
  const int rows = a.n_slots * a.map.nq;
  if (rows <= 0) return cudaSuccess;
  const int threads = (a.hq < 32 ? a.hq : 32) * 32;
  count_launch();
  { const cudaError_t le_ = launch_pdl(attn_combine_kernel, dim3(rows), dim3(threads), 0, st, a); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

// Test hook: this translation unit's copy of the pipeline wait limit.
cudaError_t set_pipeline_wait_limit_attention(long long cycles) {
  return cudaMemcpyToSymbol(g_pipeline_wait_limit, &cycles, sizeof(cycles));
}

}  // namespace quail
