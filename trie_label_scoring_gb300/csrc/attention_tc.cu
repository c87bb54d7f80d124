// Doc-part attention on tcgen05 for many query rows per KV head (hundreds to
// thousands of evaluated trie nodes x G query heads). Same math as
// attn_doc_kernel in attention.cu ("To Classify, Try a Trie Tree", sec. 3.2:
// every evaluated node attends to the document; the tree part and the merge
// are shared), but a CTA owns a 128-row query tile and both products run on
// the 5th-generation tensor cores with fp32 accumulators in TMEM:
//   S_b  = Q_hi K^T + Q_lo K^T      (M 128 rows, N 128 keys, K 128 dims)
//   O   += P_hi V   + P_lo V        (M 128 rows, N 128 dims, K 128 keys)
// per block of 128 keys (8 pages). Q and P are two-term bf16 splits (as in
// the mma.sync path) and both live in TMEM as the A operand: Q once per CTA,
// P written by the softmax over the S block it was computed from. K and V come
// from two TMA page rings (K-major K, MN-major V), so while the blocks run
// shared memory holds nothing but keys and values; the epilogue then stages
// the tile's tree-part rows in and output rows out through the idle rings.
//
// An M=128, K=16 MMA costs max(64, N/2) cycles on this part, so both products
// use N = 128; per 128-key block the tensor pipe is busy 2 x 16 x 64 cycles.
// MMAs are issued in pairs S(j) S(j+1) PV(j) PV(j+1): the softmax of block j
// runs under S(j+1) and that of j+1 under PV(j), and S(j+2) (which reuses the
// TMEM columns of P(j)) waits for PV(j) while PV(j+1) keeps the pipe busy.
//
// Roles (352 threads): warp 0 loads K pages, warp 1 owns TMEM and issues the
// MMAs, warp 2 loads V pages, warps 3..10 (two warpgroups; each thread one
// query row and half of every key block / of O's columns) build Q (each
// warpgroup half of the rotate-half pairs), run the softmax (lazy reference
// max, as in attention.cu), write P and finish rows.
#include "attn_common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "quail_internal.h"
#include "sm103.cuh"

namespace quail {

namespace {

constexpr int kTcSoftmaxWarps = 8;
constexpr int kTcThreads = 32 * (3 + kTcSoftmaxWarps);
constexpr int kTcRows = 128;
constexpr int kTcBlkKeys = 128;                // keys per block = 8 pages
constexpr int kTcBlkPages = kTcBlkKeys / 16;
constexpr int kTcStages = 3;                   // per ring
constexpr int kTcMaxPages = 512;               // split_tokens <= 8192
constexpr uint32_t kTcHalf = kTcBlkKeys * 128;  // 16 KB: 128 keys x 64 dims (128 B rows, 128B swizzle)
constexpr uint32_t kTcStage = 2 * kTcHalf;      // dims 0..63 | dims 64..127
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kTcStages * kTcStage;
constexpr uint32_t kOffBar = kOffV + kTcStages * kTcStage;
constexpr uint32_t kOffPages = kOffBar + 256;
constexpr uint32_t kOffX = kOffPages + kTcMaxPages * 4;  // softmax exchange: 3 KB
constexpr size_t kTcSmem = 1024 + kOffX + 3 * 1024;
constexpr uint32_t kStageRow = 528;  // bytes per row of the epilogue's shared-memory staging
static_assert(128 * kStageRow <= kTcStages * kTcStage, "a ring holds a 128-row staging block");
constexpr uint32_t kTmemCols = 512;  // S/P buffers 0..127, 128..255 | O 256..383 | Q hi 384..447, lo 448..511
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemQ = 384;  // column c of lane r: (q[r][2c], q[r][2c+1]) as bf16x2

struct TcBars {
  uint64_t k_full[kTcStages], k_empty[kTcStages], v_full[kTcStages], v_empty[kTcStages];
  uint64_t s_full[2];   // S_b complete (MMA commit)
  uint64_t p_full[2];   // P_b written over S_b (256 softmax threads)
  uint64_t pv_done[2];  // O += P_b V complete (MMA commit): P_b's columns and V's stage are free
  uint64_t q_full, drain, xbar[2], lbar;
  uint64_t ebar[3];  // row epilogue steps (256 softmax threads each)
  uint32_t tmem_slot;
  int abort_flag;
};
static_assert(sizeof(TcBars) <= 256, "barrier block");
static_assert(kTcSmem <= 227 * 1024, "shared memory");

// Stores 16 consecutive fp32 columns of this thread's TMEM lane without
// waiting; tmem_st_wait() completes every store issued before it.
__device__ __forceinline__ void tmem_st_16cols_nowait(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (+)= A * B^T with A in TMEM (M rows = lanes, K packed two bf16 per column)
// and the B shared-memory descriptor given as its two 32-bit words.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One TMA page ring (K or V): block j's 8 pages into stage j % kTcStages, both
// 64-dim halves, once the stage's previous block has been consumed.
__device__ __forceinline__ void load_ring(uint8_t* ring, uint64_t* full, uint64_t* empty, const CUtensorMap* tm,
                                          const int* s_pages, int n_pages, int n_blocks, const AttnArgs& a, int g,
                                          int doc, volatile int* abort_flag) {
  int armed[kTcStages];
#pragma unroll
  for (int s = 0; s < kTcStages; ++s) armed[s] = -1;
  for (int blk = 0; blk < n_blocks; ++blk) {
    const int s = blk % kTcStages;
    const int use = blk / kTcStages;
    if (use > 0 && !mbar_wait(&empty[s], static_cast<uint32_t>((use - 1) & 1), abort_flag)) break;
    const int np = min(kTcBlkPages, n_pages - blk * kTcBlkPages);
    int good = 0;
    for (int q = 0; q < np; ++q) {
      const int phys = s_pages[blk * kTcBlkPages + q];
      good += (phys >= 0 && phys < a.num_pages) ? 1 : 0;
    }
    if (good < np) raise_device_error(a.err, QUAIL_ERR_DEVICE_BOUNDS, doc);
    armed[s] = -1;
    if (good == 0) {
      mbar_arrive(&full[s]);  // release the consumer on stale data; results of this doc are void
      continue;
    }
    uint8_t* st = ring + s * kTcStage;
    mbar_arrive_expect_tx(&full[s], good * 2 * 2048);
    for (int q = 0; q < np; ++q) {
      const int phys = s_pages[blk * kTcBlkPages + q];
      if (phys < 0 || phys >= a.num_pages) continue;
      const int y = (phys * a.hkv + g) * 16;
      tma_load_2d(st + q * 2048, tm, &full[s], 0, y);
      tma_load_2d(st + kTcHalf + q * 2048, tm, &full[s], 64, y);
    }
    armed[s] = use & 1;
  }
  for (int s = 0; s < kTcStages; ++s) {  // no copy may still be landing when the CTA exits
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

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_doc_tc_kernel(AttnArgs a, RopeTable rt, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
  grid_dependency_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(base + kOffBar);
  volatile int* abort_flag = &bars->abort_flag;
  int* s_pages = reinterpret_cast<int*>(base + kOffPages);

  // grid: x = row tile (fastest, so the tiles that share a document's KV run
  // together and re-read it from L2), y = slot, z = split + n_splits * kv
  // head: the documents of one KV head come next, so their tiles re-read the
  // same q and tree-part rows from L2 as well
  const int slot = blockIdx.y;
  if (a.map.n_slots_dev != nullptr && slot >= *a.map.n_slots_dev) return;
  if (rows_past_end(a.map, slot, static_cast<int>(blockIdx.x) * kTcRows / (a.hq / a.hkv))) return;  // padding tile
  const int rt_idx = blockIdx.x;
  const int split = blockIdx.z % a.n_splits;
  const int g = blockIdx.z / a.n_splits;
  const int doc = row_doc(a.map, slot);
  const int L = a.doc_len[doc];
  if (L < 1 || L > a.max_doc_len) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.x == 0 && g == 0) raise_device_error(a.err, QUAIL_ERR_DEVICE_BOUNDS, doc);
    return;
  }
  const int k_lo = split * a.split_tokens;
  if (k_lo >= L) return;
  const int k_hi = min(L, k_lo + a.split_tokens);
  const int p0 = k_lo / 16;
  const int n_pages = (k_hi - k_lo + 15) / 16;
  const int n_blocks = (n_pages + kTcBlkPages - 1) / kTcBlkPages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  {
    const int* pt = a.page_table + static_cast<size_t>(doc) * a.max_pages;
    for (int j = threadIdx.x; j < n_pages; j += kTcThreads) s_pages[j] = pt[p0 + j];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 256);
      mbar_init(&bars->pv_done[b], 1);
      mbar_init(&bars->xbar[b], 256);
    }
    mbar_init(&bars->q_full, 256);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->lbar, 256);
    for (int i = 0; i < 3; ++i) mbar_init(&bars->ebar[i], 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_slot;

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------ page loaders (K: warp 0, V: warp 2)
    if (lane == 0) {
      if (warp == 0)
        load_ring(base + kOffK, bars->k_full, bars->k_empty, &tmK, s_pages, n_pages, n_blocks, a, g, doc, abort_flag);
      else
        load_ring(base + kOffV, bars->v_full, bars->v_empty, &tmV, s_pages, n_pages, n_blocks, a, g, doc, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // Issues S(j) as soon as K_j has landed and buffer j % 2 is free (PV(j - 2)
    // done), and PV(j) as soon as the softmax has written P_j: whichever is
    // ready first, so the tensor pipe never idles behind a fixed order while
    // the softmax of the other buffer is still running.
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16_f32(kTcRows, kTcBlkKeys);
      constexpr uint32_t idesc_pv = umma_idesc_bf16_f32_bmn(kTcRows, 128);
      // descriptors as two 32-bit words; stepping the start address (bits
      // 0..13, in 16-byte units, addresses < 256 KB) is a 32-bit add
      const uint64_t dk = smem_desc_sw128(smem_u32(base + kOffK));
      const uint64_t dv = smem_desc_sw128_mn(smem_u32(base + kOffV), kTcHalf, 1024);
      const uint32_t dk_lo = static_cast<uint32_t>(dk), dk_hi = static_cast<uint32_t>(dk >> 32);
      const uint32_t dv_lo = static_cast<uint32_t>(dv), dv_hi = static_cast<uint32_t>(dv >> 32);
      auto issue_s = [&](int j) {
        const int s = j % kTcStages, b = j & 1;
        const uint32_t k_lo = dk_lo + ((s * kTcStage) >> 4);
        const uint32_t d = tmem_base + b * kTcBlkKeys, aq = tmem_base + kTmemQ;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // 16 dims per instruction; dims 0..63 in half 0
            umma_ts(d, aq + part * 64 + ks * 8, k_lo + (((ks >> 2) * kTcHalf + (ks & 3) * 32) >> 4), dk_hi, idesc_s,
                    (part | ks) != 0 ? 1u : 0u);
        }
        umma_commit(&bars->s_full[b]);
        umma_commit(&bars->k_empty[s]);
      };
      // O += (P_hi + P_lo) V_j with P_j read from the columns of S_b: keys
      // 64w..64w+63 were written by softmax warpgroup w, hi at +64w, lo at +64w+32.
      auto issue_pv = [&](int j) {
        const int s = j % kTcStages, b = j & 1;
        const uint32_t v_lo = dv_lo + ((s * kTcStage) >> 4);
        const uint32_t ap = tmem_base + b * kTcBlkKeys, d = tmem_base + kTmemO;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // 16 keys = one page per instruction
            umma_ts(d, ap + (kk >> 2) * 64 + part * 32 + (kk & 3) * 8, v_lo + ((kk * 2048) >> 4), dv_hi, idesc_pv,
                    (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars->pv_done[b]);
        umma_commit(&bars->v_empty[s]);
      };
      bool ok = mbar_wait(&bars->q_full, 0u, abort_flag);
      if (ok) tc_fence_after();
      int js = 0, jp = 0;  // next S, next PV
      long long t_idle = clock64();
      while (ok && jp < n_blocks) {
        bool progressed = false;
        if (jp < js && mbar_try_wait(smem_u32(&bars->p_full[jp & 1]), static_cast<uint32_t>((jp >> 1) & 1)) &&
            mbar_try_wait(smem_u32(&bars->v_full[jp % kTcStages]), static_cast<uint32_t>((jp / kTcStages) & 1))) {
          tc_fence_after();
          issue_pv(jp++);
          progressed = true;
        }
        if (js < n_blocks && js < jp + 2 &&
            mbar_try_wait(smem_u32(&bars->k_full[js % kTcStages]), static_cast<uint32_t>((js / kTcStages) & 1)) &&
            (js < 2 ||
             mbar_try_wait(smem_u32(&bars->pv_done[js & 1]), static_cast<uint32_t>(((js - 2) >> 1) & 1)))) {
          tc_fence_after();
          issue_s(js++);
          progressed = true;
        }
        if (progressed) {
          t_idle = clock64();
        } else if (*abort_flag) {
          ok = false;
        } else if (clock64() - t_idle > kWaitLimitCycles) {
          *abort_flag = 1;
          ok = false;
        }
      }
      // Drain: all MMAs issued by this thread complete before TMEM is released.
      umma_commit(&bars->drain);
      const uint32_t ad = smem_u32(&bars->drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(ad, 0u)) {
        if (clock64() - t0 > kWaitLimitCycles) {
          *abort_flag = 1;
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------ softmax warps
    // Two warpgroups: wg 0 takes keys 0..63 of every block and O columns
    // 0..63, wg 1 keys 64..127 and columns 64..127. Warp w reaches TMEM lanes
    // 32 (w % 4) .. +31, so thread (wg, row) <-> TMEM lane row.
    const int wg = (warp - 3) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int sthr = wg * 128 + row;  // 0..255
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    float* xmax = reinterpret_cast<float*>(base + kOffX);  // [2 buffers][2 halves][128 rows]
    float* xl = xmax + 512;                                // [2 halves][128 rows]
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
    if (row_ok && a.n_splits == 1) {
      // the epilogue's tree-part inputs: start them towards L2 now, so the
      // reads after the last block do not wait on HBM (this warpgroup's two
      // 128-byte lines of the row, and the row's max / sum)
      const float* to = a.tree_o + (static_cast<size_t>(node) * a.hq + h) * 128 + wg * 64;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(to));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(to + 32));
      if (wg == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.tree_ml + static_cast<size_t>(node) * a.hq + h));
    }
    // Q row into TMEM: RoPE at l_i + depth, two-term bf16 split. Warpgroup w
    // takes the rotate-half pairs (j, j + 64) for j = 32w .. 32w + 31 and
    // writes both outputs of each pair, so it reads only those 64 dims (one
    // round of 16-byte loads) and evaluates each angle once. TMEM column c
    // holds dims (2c, 2c + 1): this thread fills columns 16w .. 16w + 15 and
    // 32 + 16w .. 32 + 16w + 15 of the hi and of the lo half.
    {
      const float4* q4 =
          row_ok ? reinterpret_cast<const float4*>(a.qkv + static_cast<size_t>(node) * a.ldq + h * 128) : nullptr;
      const int pos = row_ok ? L + a.node_depth[node] : 0;
      float4 x1[8], x2[8];  // dims 32w .. 32w + 31 and 64 + 32w .. 64 + 32w + 31
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x1[i] = row_ok ? q4[wg * 8 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
        x2[i] = row_ok ? q4[16 + wg * 8 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float hi1[16], lo1[16], hi2[16], lo2[16];  // first outputs (dims j), second outputs (dims j + 64)
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float* p1 = reinterpret_cast<const float*>(x1) + 2 * c;
        const float* p2 = reinterpret_cast<const float*>(x2) + 2 * c;
        float y1[2], y2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float cs, sn;
          rope_cs(pos, rt.w[wg * 32 + 2 * c + u], cs, sn);
          y1[u] = p1[u] * cs - p2[u] * sn;
          y2[u] = p2[u] * cs + p1[u] * sn;
        }
        uint32_t hv, lv;
        split_bf16(y1[0], y1[1], hv, lv);
        hi1[c] = __uint_as_float(hv);
        lo1[c] = __uint_as_float(lv);
        split_bf16(y2[0], y2[1], hv, lv);
        hi2[c] = __uint_as_float(hv);
        lo2[c] = __uint_as_float(lv);
      }
      tmem_st_16cols_nowait(lane_addr + kTmemQ + wg * 16, hi1);
      tmem_st_16cols_nowait(lane_addr + kTmemQ + 32 + wg * 16, hi2);
      tmem_st_16cols_nowait(lane_addr + kTmemQ + 64 + wg * 16, lo1);
      tmem_st_16cols_nowait(lane_addr + kTmemQ + 96 + wg * 16, lo2);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->q_full);
    }
    const float scale = kAttnLog2e * 0.08838834764831845f;  // log2(e) / sqrt(128)
    float m_ref = -INFINITY, l_part = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < n_blocks; ++j) {
      const int b = j & 1;
      const uint32_t sp_col = b * kTcBlkKeys + wg * 64;  // this half's S columns, then its P columns
      // waits are made warp-uniform: the warp-collective tcgen05.ld/st and
      // __any_sync below must never run with lanes that left the loop
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[b], static_cast<uint32_t>((j >> 1) & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s0[32], s1[32];
      tmem_ld_32cols(lane_addr + sp_col, s0);
      tmem_ld_32cols(lane_addr + sp_col + 32, s1);
      const int valid = min(kTcBlkKeys, k_hi - (k_lo + j * kTcBlkKeys)) - wg * 64;  // keys of this half
      if (valid < 64) {  // last block only: keys past the document end
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s0[i] = i < valid ? s0[i] : -INFINITY;
          s1[i] = i + 32 < valid ? s1[i] : -INFINITY;
        }
      }
      float mraw = -INFINITY;  // max of the raw scores; the scale is positive
#pragma unroll
      for (int i = 0; i < 32; ++i) mraw = fmaxf(mraw, fmaxf(s0[i], s1[i]));
      // row max over both halves (double-buffered exchange; bounded waits only,
      // so an aborted peer cannot hang this CTA)
      xmax[(b * 2 + wg) * 128 + row] = mraw;
      mbar_arrive(&bars->xbar[b]);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->xbar[b], static_cast<uint32_t>((j >> 1) & 1), abort_flag))) {
        ok = false;
        break;
      }
      mraw = fmaxf(mraw, xmax[(b * 2 + (wg ^ 1)) * 128 + row]);
      const float mx = mraw * scale;
      // Lazy reference max (see attention.cu): moves only past +8 in base 2.
      // Both halves of a row see the same maxima, so they move it together.
      const bool need = mx > m_ref + 8.f;
      float alpha = 1.f;
      if (need) {
        const float nm = fmaxf(m_ref, mx);
        alpha = exp2f(m_ref - nm);
        m_ref = nm;
        l_part *= alpha;
      }
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        // O must hold every PV up to block j - 1 before it is rescaled
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[(j - 1) & 1],
                                               static_cast<uint32_t>(((j - 1) >> 1) & 1), abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {  // this warpgroup's 64 columns of O
          float o[32];
          const uint32_t col = kTmemO + wg * 64 + c * 32;
          tmem_ld_32cols(lane_addr + col, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st_32cols(lane_addr + col, o);
        }
      }
      // P = exp2(s * scale - m_ref) as a two-term bf16 split, written over this
      // half's S columns: hi in the first 32, lo in the last 32 (keys 2c, 2c+1
      // in column c), the A operand layout of the PV product.
      float psum = 0.f;
      {
        float ph[32], pl[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float x0 = c < 16 ? s0[2 * c] : s1[2 * c - 32];
          const float x1 = c < 16 ? s0[2 * c + 1] : s1[2 * c - 31];
          const float e0 = fast_exp2(fmaf(x0, scale, -m_ref));
          const float e1 = fast_exp2(fmaf(x1, scale, -m_ref));
          psum += e0 + e1;
          uint32_t hv, lv;
          split_bf16(e0, e1, hv, lv);
          ph[c] = __uint_as_float(hv);
          pl[c] = __uint_as_float(lv);
        }
        tmem_st_32cols(lane_addr + sp_col, ph);
        tmem_st_32cols(lane_addr + sp_col + 32, pl);
      }
      l_part += psum;
      // Keys past the document end (tail of the last page, pages not loaded):
      // zero their V rows so stale contents cannot reach O through P = 0.
      const int vblk = min(kTcBlkKeys, k_hi - (k_lo + j * kTcBlkKeys));
      if (vblk < kTcBlkKeys) {
        const int s = j % kTcStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[s], static_cast<uint32_t>((j / kTcStages) & 1),
                                               abort_flag))) {
          ok = false;
          break;
        }
        uint8_t* vst = base + kOffV + s * kTcStage;
        for (int idx = sthr; idx < (kTcBlkKeys - vblk) * 16; idx += 256) {
          const int r = vblk + idx / 16, hc = idx % 16;
          *reinterpret_cast<uint4*>(vst + (hc / 8) * kTcHalf + r * 128 + (hc % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&bars->p_full[b]);
    }
    // Row epilogue once the last PV has landed in TMEM.
    if (ok && __all_sync(0xffffffffu, mbar_wait(&bars->pv_done[(n_blocks - 1) & 1],
                                                static_cast<uint32_t>(((n_blocks - 1) >> 1) & 1), abort_flag))) {
      tc_fence_after();
      xl[wg * 128 + row] = l_part;
      mbar_arrive(&bars->lbar);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->lbar, 0u, abort_flag));
    } else {
      ok = false;
    }
    // Rows out through shared memory. Every page has been consumed, so the K
    // ring stages tree_o rows in and the V ring stages output rows out: both
    // cross global memory as whole rows, one row per warp instruction, while
    // each thread works on its own row in shared memory. Rows are 528 bytes
    // apart, so 8 consecutive rows fall in 8 different 16-byte bank groups.
    uint8_t* tstage = base + kOffK;
    uint8_t* ostage = base + kOffV;
    long long* tab = reinterpret_cast<long long*>(xmax);  // [128 rows][tree_o row offset, output offset] (-1: none)
    const bool fused = a.n_splits == 1;
    const int cw = warp - 3;  // copy warp 0..7: rows 16 cw .. 16 cw + 15
    if (ok) {
      // the exchange buffer is free: the last block's maxima were read before lbar
      if (wg == 0) {
        long long src = -1, dstoff = -1;
        if (row_ok && fused) {
          src = (static_cast<long long>(node) * a.hq + h) * 128;
          dstoff = (static_cast<long long>(slot) * a.map.nq + e) * 2 * a.hq * 128 + h * 128;
        } else if (row_ok) {
          dstoff = (((static_cast<long long>(slot) * a.hkv + g) * a.n_splits + split) * a.rows_pad + rr) * 128;
        }
        tab[2 * row] = src;
        tab[2 * row + 1] = dstoff;
      }
      mbar_arrive(&bars->ebar[0]);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->ebar[0], 0u, abort_flag));
    }
    if (ok && fused) {  // tree_o rows in (all loads first)
      float4 tv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const long long src = tab[2 * (cw * 16 + i)];
        tv[i] = src >= 0 ? reinterpret_cast<const float4*>(a.tree_o + src)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) reinterpret_cast<float4*>(tstage + (cw * 16 + i) * kStageRow)[lane] = tv[i];
    }
    if (ok) {
      mbar_arrive(&bars->ebar[1]);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->ebar[1], 0u, abort_flag));
    }
    if (ok) {
      const float l_sum = l_part + xl[(wg ^ 1) * 128 + row];
      float f1 = 1.f, f2 = 0.f, inv = 1.f;
      if (row_ok && fused) {
        const float2 tml = a.tree_ml[static_cast<size_t>(node) * a.hq + h];
        const float M = fmaxf(m_ref, tml.x);
        f1 = exp2f(m_ref - M);
        f2 = exp2f(tml.x - M);
        inv = 1.f / (f1 * l_sum + f2 * tml.y);
      } else if (row_ok && wg == 0) {
        a.part_ml[tab[2 * row + 1] / 128] = make_float2(m_ref, l_sum);
      }
      uint8_t* orow = ostage + row * kStageRow;
      const float* trow = reinterpret_cast<const float*>(tstage + row * kStageRow);
#pragma unroll 1
      for (int c = wg * 2; c < wg * 2 + 2; ++c) {  // this warpgroup's 64 columns of O, 32 at a time
        float o[32];
        tmem_ld_32cols(lane_addr + kTmemO + c * 32, o);
        if (fused) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            const float4 ta = reinterpret_cast<const float4*>(trow + c * 32 + i)[0];
            const float4 tb = reinterpret_cast<const float4*>(trow + c * 32 + i)[1];
            const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
            uint32_t hv[4], lv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k = i + 2 * u;
              split_bf16((f1 * o[k] + f2 * tv[2 * u]) * inv, (f1 * o[k + 1] + f2 * tv[2 * u + 1]) * inv, hv[u], lv[u]);
            }
            *reinterpret_cast<uint4*>(orow + (c * 32 + i) * 2) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4*>(orow + 256 + (c * 32 + i) * 2) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(orow + (c * 32 + i) * 4) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
        }
      }
      mbar_arrive(&bars->ebar[2]);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->ebar[2], 0u, abort_flag));
    }
    if (ok) {  // output rows out: [hi | lo] bf16 halves to their two places, or fp32 partials
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int r = cw * 16 + i;
        const long long dstoff = tab[2 * r + 1];
        if (dstoff < 0) continue;
        const uint4 v = reinterpret_cast<const uint4*>(ostage + r * kStageRow)[lane];
        if (fused) {
          bf16* dst = a.out + dstoff + (lane < 16 ? lane * 8 : a.hq * 128 + (lane - 16) * 8);
          *reinterpret_cast<uint4*>(dst) = v;
        } else {
          reinterpret_cast<uint4*>(a.part_o + dstoff)[lane] = v;
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
  if (a.row_tile != kTcRows || a.rows_pad % kTcRows != 0 || a.split_tokens > 16 * kTcMaxPages ||
      a.split_tokens % 16 != 0)
    return cudaErrorInvalidValue;
  dim3 grid(a.rows_pad / kTcRows, a.n_slots, a.n_splits * a.hkv);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  count_launch();
  { const cudaError_t le_ = launch_pdl(attn_doc_tc_kernel, dim3(grid), dim3(kTcThreads), kTcSmem, st, a, make_rope_table(a.theta), tmK, tmV); if (le_ != cudaSuccess) return le_; }
  return cudaGetLastError();
}

// Test hook: this translation unit's copy of the pipeline wait limit.
cudaError_t set_pipeline_wait_limit_attention_tc(long long cycles) {
  return cudaMemcpyToSymbol(g_pipeline_wait_limit, &cycles, sizeof(cycles));
}

}  // namespace quail
