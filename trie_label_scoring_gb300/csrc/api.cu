// C ABI of libquail (see include/quail.h): argument validation, workspace
// planning, TMA descriptors and the launch sequence of each call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"
#include "umma_gemm.cuh"
#include "quail_internal.h"
#include "trie.h"
#include "shortlist.h"

using namespace quail;

// ------------------------------------------------------------------ errors
namespace {

thread_local std::string g_last_error;
thread_local int32_t g_launches = 0;

quail_status fail(quail_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                         \
  do {                                                                                         \
    cudaError_t _e = (expr);                                                                   \
    if (_e != cudaSuccess) return fail(QUAIL_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(_e)); \
  } while (0)

// First device error (code, detail); kernels set it with atomicCAS, never trap.
__device__ int g_quail_err[2];

struct DeviceState {
  bool ready = false;
  int* err = nullptr;
  int num_sms = 0;
};
std::mutex g_dev_mu;
DeviceState g_dev[64];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

quail_status device_state(DeviceState** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(QUAIL_ERR_CUDA, "device id %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    CUDA_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_quail_err));
    CUDA_TRY(cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev));
    int major = 0, minor = 0;
    CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    if (major != 10 || minor != 3)
      return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "libquail is built for sm_103a; device %d is sm_%d%d", dev, major,
                  minor);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
      if (fn == nullptr || q != cudaDriverEntryPointSuccess)
        return fail(QUAIL_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return QUAIL_OK;
}

// 2D bf16 tensor [rows, cols] (cols contiguous, row stride ld elements), box
// box_cols x box_rows, 128-byte swizzle (box_cols * 2 must be 128).
quail_status encode_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                            uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QUAIL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return QUAIL_OK;
}

// ------------------------------------------------------------------ profiling hook
std::mutex g_ev_mu;
std::vector<cudaEvent_t> g_events;

void stage_mark(int stage, bool end, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_ev_mu);
  const size_t i = 2 * static_cast<size_t>(stage) + (end ? 1 : 0);
  if (i < g_events.size() && g_events[i] != nullptr) cudaEventRecord(g_events[i], st);
}

// ------------------------------------------------------------------ validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

quail_status check_model(const quail_model_desc* m) {
  if (m == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "model is null");
  if (m->head_dim != 128) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "head_dim must be 128 (got %d)", m->head_dim);
  if (m->hidden <= 0 || m->hidden % 64 != 0)
    return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "hidden must be a positive multiple of 64 (got %d)", m->hidden);
  if (m->n_kv_heads <= 0 || m->n_q_heads <= 0 || m->n_q_heads % m->n_kv_heads != 0)
    return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "n_q_heads must be a positive multiple of n_kv_heads");
  if (m->n_q_heads > 128) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 128 query heads");
  if (m->vocab < 256) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "vocab must be >= 256");
  if (m->hidden > 12288) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "hidden must be <= 12288");
  if (!(m->rms_eps > 0.f) || !(m->rope_theta > 1.f)) return fail(QUAIL_ERR_INVALID_ARG, "bad rms_eps / rope_theta");
  const void* ptrs[] = {m->embed, m->w_q, m->w_k, m->w_v, m->q_norm, m->k_norm,
                        m->w_o, m->in_norm, m->final_norm, m->lm_head};
  for (const void* p : ptrs) {
    if (p == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "a model weight pointer is null");
    if (!aligned16(p)) return fail(QUAIL_ERR_INVALID_ARG, "model weights must be 16-byte aligned");
  }
  return QUAIL_OK;
}

quail_status check_kv(const quail_paged_kv* kv, const quail_model_desc* m) {
  if (kv == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "kv is null");
  if (kv->page_size != 16) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "page_size must be 16 (got %d)", kv->page_size);
  if (kv->k_pool == nullptr || kv->v_pool == nullptr || kv->page_table == nullptr || kv->doc_len == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "a kv pointer is null");
  if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool)) return fail(QUAIL_ERR_INVALID_ARG, "kv pools must be 16-byte aligned");
  if (kv->num_pages <= 0 || kv->max_doc_len <= 0 || kv->max_pages < (kv->max_doc_len + 15) / 16)
    return fail(QUAIL_ERR_INVALID_ARG, "num_pages, max_doc_len or max_pages inconsistent");
  if (static_cast<int64_t>(kv->num_pages) * m->n_kv_heads * 16 > (int64_t(1) << 31) - 1)
    return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "KV pool too large for 32-bit row coordinates");
  return QUAIL_OK;
}

quail_status check_workspace(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(QUAIL_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  if (ws_bytes < need) return fail(QUAIL_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  return QUAIL_OK;
}

// ------------------------------------------------------------------ workspace plan
struct Carver {
  uint8_t* base;
  size_t off = 0;
  template <class T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

struct AttnShape {
  int rows_per_kv, row_tile, rows_pad, split_tokens, n_splits;
  bool tc;  // tcgen05 kernel (128-row tiles) instead of the mma.sync one
};

AttnShape attn_shape(const quail_model_desc* m, int nq, int slots, int max_doc_len, int sms) {
  AttnShape s;
  const int G = m->n_q_heads / m->n_kv_heads;
  s.rows_per_kv = nq * G;
  const int whole = static_cast<int>(round_up(max_doc_len, 16));
  if (s.rows_per_kv <= 16) {
    // A few query rows per KV head (the support-topic shape): mma.sync kernel,
    // four warps share 16 rows. One split per document when the (document,
    // KV head) items already fill the GPU several times over (the epilogue then
    // merges the tree part); else 512-token splits and the combine kernel.
    s.tc = false;
    s.row_tile = 16;
    s.rows_pad = 16;
    const long items = static_cast<long>(slots) * m->n_kv_heads;
    s.split_tokens = (items >= 3L * sms) ? std::min(whole, 4096) : std::min(whole, 512);
  } else {
    // Many rows: tcgen05 kernel on 128-row tiles, one CTA per SM. Besides
    // its 128-key blocks a tile carries fixed work (pipeline fill, Q build,
    // the epilogue) measured at about ten blocks' time, so the key split (in
    // whole blocks, at most 8192 keys) minimises waves x (blocks per tile +
    // 10): long documents on few (document, KV head) items are split only
    // when that fills the SMs better than it costs in tiles.
    s.tc = true;
    s.row_tile = 128;
    s.rows_pad = static_cast<int>(round_up(s.rows_per_kv, 128));
    const long items = static_cast<long>(slots) * m->n_kv_heads * (s.rows_pad / 128);
    const int nb = (max_doc_len + 127) / 128;
    long best = -1;
    int split = 128;
    for (int p = 1; p <= nb; ++p) {
      const int blocks = (nb + p - 1) / p;
      if (blocks * 128 > 8192) continue;
      const long splits = (nb + blocks - 1) / blocks;
      const long waves = (items * splits + sms - 1) / sms;
      const long cost = waves * (blocks + 10);
      if (best < 0 || cost < best) {
        best = cost;
        split = blocks * 128;
      }
      if (blocks == 1) break;
    }
    s.split_tokens = split;
  }
  s.n_splits = (max_doc_len + s.split_tokens - 1) / s.split_tokens;
  return s;
}

// SM count used to balance split-K; the workspace size and the call use the
// same device, so they agree.
int planning_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
    return n;
  cudaGetLastError();
  return 152;
}

struct GemmPlan {
  int ks_qkv, ks_wo;
};

GemmPlan gemm_plan(const quail_model_desc* m, int nodes, size_t rows, int sms) {
  const int ldq = (m->n_q_heads + 2 * m->n_kv_heads) * 128;
  GemmPlan g;
  g.ks_qkv = choose_k_splits(static_cast<int>(round_up(nodes, 128) / 128 * round_up(ldq, 256) / 256),
                             m->hidden / 64, sms);
  g.ks_wo = choose_k_splits(static_cast<int>(round_up(rows, 128) / 128 * round_up(m->hidden, 256) / 256),
                            m->n_q_heads * 128 / 64, sms);
  return g;
}

struct Buffers {
  GemmPlan gp;
  bf16* xhat;
  float* qkv_part;
  float* qkv;
  float* tree_o;
  float2* tree_ml;
  float* part_o;
  float2* part_ml;
  bf16* attn_out;
  float* h_part;
  bf16* z;
  float* z_f32;
  float2* lse_part;
  float* lse;
  float* child_logit;
  int* slot_order;  // the doc attention's slot order
  int* small;       // node tables / slot lists
};

// Carves (or sizes, when base is null) the workspace of one call.
// nodes: rows of the node prologue; slots x nq: output rows.
size_t plan(uint8_t* base, const quail_model_desc* m, int nodes, int slots, int nq, int max_doc_len, bool head,
            int n_child, bool need_zf32, int small_ints, Buffers* b) {
  const int d = m->hidden, hq = m->n_q_heads, hkv = m->n_kv_heads;
  const int ldq = (hq + 2 * hkv) * 128;
  const AttnShape as = attn_shape(m, nq, slots, max_doc_len, planning_sms());
  const size_t rows = static_cast<size_t>(slots) * nq;
  const size_t rows_p = round_up(rows, 128);
  const int n_tiles = (m->vocab + kHeadBN - 1) / kHeadBN;
  Carver c{base};
  Buffers t{};
  t.gp = gemm_plan(m, nodes, rows, planning_sms());
  t.xhat = c.take<bf16>(round_up(nodes, 128) * 2 * d);
  t.qkv_part = c.take<float>(static_cast<size_t>(t.gp.ks_qkv) * nodes * ldq);
  t.qkv = c.take<float>(static_cast<size_t>(nodes) * ldq);
  t.tree_o = c.take<float>(static_cast<size_t>(nodes) * hq * 128);
  t.tree_ml = c.take<float2>(static_cast<size_t>(nodes) * hq);
  const size_t prow = as.n_splits > 1 ? static_cast<size_t>(slots) * hkv * as.n_splits * as.rows_pad : 0;
  t.part_o = c.take<float>(prow * 128);
  t.part_ml = c.take<float2>(prow);
  t.attn_out = c.take<bf16>(rows_p * 2 * hq * 128);
  t.h_part = c.take<float>(static_cast<size_t>(t.gp.ks_wo) * rows * d);
  t.z = c.take<bf16>(rows_p * d);
  t.z_f32 = (need_zf32 || head) ? c.take<float>(rows * d) : nullptr;
  t.lse_part = head ? c.take<float2>(rows * n_tiles) : nullptr;
  t.lse = head ? c.take<float>(rows) : nullptr;
  t.child_logit = head ? c.take<float>(static_cast<size_t>(slots) * n_child) : nullptr;
  t.slot_order = c.take<int>(slots);
  t.small = c.take<int>(small_ints);
  if (b) *b = t;
  return c.off + 256;
}

// ------------------------------------------------------------------ shared layer steps
struct NodeTables {
  const int* token;   // [nodes]
  const int* depth;   // [nodes]
  const int* parent;  // [nodes]
  int nodes;
};

// Node prologue: x^ = RMSNorm(E[tok]) g_in (two-term bf16 split);
// q|k|v = x^ W^T in one launch when the three weight blocks align to 256 rows;
// per-head q/k RMSNorm while summing the k-split slabs.
quail_status run_qkv(const quail_model_desc* m, const NodeTables& nt, const Buffers& b, DeviceState* ds,
                     cudaStream_t st, const int* m_live = nullptr);

quail_status run_prologue(const quail_model_desc* m, const NodeTables& nt, const Buffers& b, DeviceState* ds,
                          cudaStream_t st, const int* m_live = nullptr) {
  CUDA_TRY(launch_embed_rmsnorm(static_cast<const bf16*>(m->embed), nt.token, nt.nodes, m->hidden,
                                static_cast<const bf16*>(m->in_norm), m->rms_eps, b.xhat, st, m_live));
  return run_qkv(m, nt, b, ds, st, m_live);
}

// q|k|v = x^ W^T from the split rows already in b.xhat; per-head q/k RMSNorm.
// m_live (optional): device count of the node rows present; the GEMM skips the rest.
quail_status run_qkv(const quail_model_desc* m, const NodeTables& nt, const Buffers& b, DeviceState* ds,
                     cudaStream_t st, const int* m_live) {
  const int d = m->hidden, hq = m->n_q_heads, hkv = m->n_kv_heads;
  const int ldq = (hq + 2 * hkv) * 128;
  CUtensorMap tA;
  quail_status s = encode_2d_bf16(&tA, b.xhat, round_up(nt.nodes, 128), 2 * d, 2 * d, 64, 128);
  if (s != QUAIL_OK) return s;
  const void* w[3] = {m->w_q, m->w_k, m->w_v};
  const int nrows[3] = {hq * 128, hkv * 128, hkv * 128};
  const size_t slab = static_cast<size_t>(nt.nodes) * ldq;
  const bool aligned = (hq * 128) % 256 == 0 && (hkv * 128) % 256 == 0;
  BSet bs{};
  int col = 0;
  for (int i = 0; i < 3; ++i) {
    const int slot = aligned ? i : 0;
    s = encode_2d_bf16(&bs.map[slot], w[i], nrows[i], d, d, 64, 256);
    if (s != QUAIL_OK) return s;
    bs.n_begin[slot] = aligned ? col : 0;
    bs.n_begin[slot + 1] = aligned ? col + nrows[i] : nrows[i];
    if (!aligned) {
      bs.count = 1;
      CUDA_TRY(launch_gemm_proj(tA, bs, nt.nodes, nrows[i], d, b.gp.ks_qkv, b.qkv_part + col, slab, ldq, ds->num_sms,
                                ds->err, st, m_live));
    }
    col += nrows[i];
  }
  if (aligned) {
    bs.count = 3;
    CUDA_TRY(launch_gemm_proj(tA, bs, nt.nodes, ldq, d, b.gp.ks_qkv, b.qkv_part, slab, ldq, ds->num_sms, ds->err,
                              st, m_live));
  }
  CUDA_TRY(launch_qk_head_norm(b.qkv_part, b.gp.ks_qkv, slab, b.qkv, nt.nodes, ldq, hq, hkv,
                               static_cast<const bf16*>(m->q_norm), static_cast<const bf16*>(m->k_norm), m->rms_eps,
                               st, m_live));
  return QUAIL_OK;
}

// Attention (tree part, paged doc part, combine) for rows = slots x nq.
// order_ready: b.slot_order already holds the slot order of these documents
// (an earlier layer of the same call computed it), so it is not recomputed.
quail_status run_attention(const quail_model_desc* m, const quail_paged_kv* kv, const NodeTables& nt, RowMap map,
                           int slots, const Buffers& b, DeviceState* ds, cudaStream_t st,
                           const int* nodes_live = nullptr, bool order_ready = false) {
  const int hq = m->n_q_heads, hkv = m->n_kv_heads;
  const AttnShape as = attn_shape(m, map.nq, slots, kv->max_doc_len, ds->num_sms);
  AttnArgs a{};
  a.num_pages = kv->num_pages;
  a.max_pages = kv->max_pages;
  a.max_doc_len = kv->max_doc_len;
  a.page_table = kv->page_table;
  a.doc_len = kv->doc_len;
  a.hq = hq;
  a.hkv = hkv;
  a.theta = m->rope_theta;
  a.qkv = b.qkv;
  a.ldq = (hq + 2 * hkv) * 128;
  a.node_depth = nt.depth;
  a.node_parent = nt.parent;
  a.n_nodes = nt.nodes;
  a.nodes_live = nodes_live;
  a.map = map;
  a.n_slots = slots;
  a.split_tokens = as.split_tokens;
  a.n_splits = as.n_splits;
  a.rows_pad = as.rows_pad;
  a.row_tile = as.row_tile;
  a.part_o = b.part_o;
  a.part_ml = b.part_ml;
  a.tree_o = b.tree_o;
  a.tree_ml = b.tree_ml;
  a.out = b.attn_out;
  a.err = ds->err;
  a.slot_order = nullptr;
  if (!as.tc && attn_doc_wants_slot_order(a, ds->num_sms)) a.slot_order = b.slot_order;
  CUtensorMap tK, tV;
  const uint64_t pool_rows = static_cast<uint64_t>(kv->num_pages) * hkv * 16;
  quail_status s = encode_2d_bf16(&tK, kv->k_pool, pool_rows, 128, 128, 64, 16);
  if (s != QUAIL_OK) return s;
  s = encode_2d_bf16(&tV, kv->v_pool, pool_rows, 128, 128, 64, 16);
  if (s != QUAIL_OK) return s;
  if (a.slot_order != nullptr && !order_ready) CUDA_TRY(launch_slot_order(a, st));
  CUDA_TRY(launch_tree_part(a, st));
  if (as.tc) {
    CUDA_TRY(launch_attn_doc_tc(a, tK, tV, st));
  } else {
    CUDA_TRY(launch_attn_doc(a, tK, tV, st));
  }
  if (as.n_splits > 1) CUDA_TRY(launch_attn_combine(a, st));
  return QUAIL_OK;
}

// h = x + O W_o^T (O as a two-term bf16 split); z = RMSNorm(h) g_f.
quail_status run_wo_gemm(const quail_model_desc* m, int rows, const Buffers& b, DeviceState* ds, cudaStream_t st);

quail_status run_wo_norm(const quail_model_desc* m, const NodeTables& nt, RowMap map, int rows, const Buffers& b,
                         DeviceState* ds, cudaStream_t st) {
  quail_status s = run_wo_gemm(m, rows, b, ds, st);
  if (s != QUAIL_OK) return s;
  const size_t slab = static_cast<size_t>(rows) * m->hidden;
  CUDA_TRY(launch_final_norm(b.h_part, b.gp.ks_wo, slab, static_cast<const bf16*>(m->embed), nt.token, map, rows,
                             m->hidden, static_cast<const bf16*>(m->final_norm), m->rms_eps, b.z, b.z_f32, st));
  return QUAIL_OK;
}

// W_o projection of the split O rows into b.h_part (ks_wo fp32 slabs).
quail_status run_wo_gemm(const quail_model_desc* m, int rows, const Buffers& b, DeviceState* ds, cudaStream_t st) {
  const int d = m->hidden, hq = m->n_q_heads;
  CUtensorMap tA;
  quail_status s = encode_2d_bf16(&tA, b.attn_out, round_up(rows, 128), 2 * hq * 128, 2 * hq * 128, 64, 128);
  if (s != QUAIL_OK) return s;
  BSet bs{};
  s = encode_2d_bf16(&bs.map[0], m->w_o, d, hq * 128, hq * 128, 64, 256);
  if (s != QUAIL_OK) return s;
  bs.n_begin[0] = 0;
  bs.n_begin[1] = d;
  bs.count = 1;
  const size_t slab = static_cast<size_t>(rows) * d;
  CUDA_TRY(launch_gemm_proj(tA, bs, rows, d, hq * 128, b.gp.ks_wo, b.h_part, slab, d, ds->num_sms, ds->err, st));
  return QUAIL_OK;
}

// ------------------------------------------------------------------ trie device image
quail_status upload_trie(quail_trie* t, cudaStream_t st, const quail_trie::DeviceImage** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(t->mu);
  auto it = t->images.find(dev);
  if (it != t->images.end()) {
    *out = &it->second;
    return QUAIL_OK;
  }
  const std::vector<int32_t>* arrays[] = {
      &t->eval_token,        &t->eval_depth,      &t->eval_parent,     &t->eval_child_offsets,
      &t->eval_child_tokens, &t->label_term_offsets, &t->label_term_eval, &t->label_term_slot,
      &t->label_prefix_eval, &t->int_token,       &t->int_depth,       &t->int_parent,
      &t->int_index_of_node, &t->child_offsets,   &t->child_nodes,     &t->child_tokens,
      &t->subtree_labels,    &t->unique_label};
  const int na = sizeof(arrays) / sizeof(arrays[0]);
  std::vector<size_t> offs(na);
  size_t total = 0;
  for (int i = 0; i < na; ++i) {
    offs[i] = total;
    total += round_up(std::max<size_t>(arrays[i]->size(), 1) * 4, 256);
  }
  std::vector<uint8_t> host(total, 0);
  for (int i = 0; i < na; ++i)
    if (!arrays[i]->empty()) std::memcpy(host.data() + offs[i], arrays[i]->data(), arrays[i]->size() * 4);
  void* dptr = nullptr;
  CUDA_TRY(cudaMalloc(&dptr, total));
  cudaError_t e = cudaMemcpyAsync(dptr, host.data(), total, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaFree(dptr);
    return fail(QUAIL_ERR_CUDA, "trie upload: %s", cudaGetErrorString(e));
  }
  quail_trie::DeviceImage img;
  img.base = dptr;
  img.bytes = total;
  const int32_t** fields[] = {&img.eval_token,        &img.eval_depth,         &img.eval_parent,
                              &img.eval_child_offsets, &img.eval_child_tokens,  &img.label_term_offsets,
                              &img.label_term_eval,   &img.label_term_slot,    &img.label_prefix_eval,
                              &img.int_token,         &img.int_depth,          &img.int_parent,
                              &img.int_index_of_node, &img.child_offsets,      &img.child_nodes,
                              &img.child_tokens,      &img.subtree_labels,     &img.unique_label};
  for (int i = 0; i < na; ++i)
    *fields[i] = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(dptr) + offs[i]);
  auto res = t->images.emplace(dev, img);
  *out = &res.first->second;
  return QUAIL_OK;
}

// ------------------------------------------------------------------ fixed scratch
// Scratch for quail_classify_trie_tree_noalloc: one fixed device array that the
// library holds on every device it is loaded on, so that entry point never
// allocates. Host code only uses its address from cudaGetSymbolAddress.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(QUAIL_NOALLOC_SCRATCH_BYTES);
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
uint8_t* g_noalloc_ptr[64] = {};

// Device address of the fixed scratch on the current device (looked up once per device).
quail_status noalloc_scratch(uint8_t** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(QUAIL_ERR_CUDA, "device id %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(QUAIL_ERR_CUDA, "cudaGetSymbolAddress(fixed scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return QUAIL_OK;
}

// The trie tables the trie_tree kernels read, in one block of `bytes` bytes.
size_t trie_tree_image_bytes(const quail_trie* t) {
  const std::vector<int32_t>* arrays[] = {&t->eval_token,         &t->eval_depth,         &t->eval_parent,
                                          &t->eval_child_offsets, &t->eval_child_tokens,  &t->label_term_offsets,
                                          &t->label_term_eval,    &t->label_term_slot,    &t->label_prefix_eval};
  size_t total = 0;
  for (const auto* a : arrays) total += round_up(std::max<size_t>(a->size(), 1) * 4, 256);
  return total;
}

// Copies those tables into dst (device) on `st` and points img at them.
quail_status copy_trie_tree_image(const quail_trie* t, uint8_t* dst, cudaStream_t st, quail_trie::DeviceImage* img) {
  const std::vector<int32_t>* arrays[] = {&t->eval_token,         &t->eval_depth,         &t->eval_parent,
                                          &t->eval_child_offsets, &t->eval_child_tokens,  &t->label_term_offsets,
                                          &t->label_term_eval,    &t->label_term_slot,    &t->label_prefix_eval};
  const int32_t** fields[] = {&img->eval_token,         &img->eval_depth,        &img->eval_parent,
                              &img->eval_child_offsets, &img->eval_child_tokens, &img->label_term_offsets,
                              &img->label_term_eval,    &img->label_term_slot,   &img->label_prefix_eval};
  size_t off = 0;
  for (int i = 0; i < 9; ++i) {
    if (!arrays[i]->empty())
      CUDA_TRY(cudaMemcpyAsync(dst + off, arrays[i]->data(), arrays[i]->size() * 4, cudaMemcpyHostToDevice, st));
    *fields[i] = reinterpret_cast<const int32_t*>(dst + off);
    off += round_up(std::max<size_t>(arrays[i]->size(), 1) * 4, 256);
  }
  return QUAIL_OK;
}


// ------------------------------------------------------------------ multi-layer path
// One layer of the stack as a single-layer descriptor (the shared steps take it).
quail_model_desc layer_desc(const quail_model_ml_desc* m, int l) {
  quail_model_desc d{};
  d.hidden = m->hidden;
  d.n_q_heads = m->n_q_heads;
  d.n_kv_heads = m->n_kv_heads;
  d.head_dim = m->head_dim;
  d.vocab = m->vocab;
  d.rms_eps = m->rms_eps;
  d.rope_theta = m->rope_theta;
  d.embed = m->embed;
  d.final_norm = m->final_norm;
  d.lm_head = m->lm_head;
  const quail_layer_weights& w = m->layers[l];
  d.w_q = w.w_q;
  d.w_k = w.w_k;
  d.w_v = w.w_v;
  d.q_norm = w.q_norm;
  d.k_norm = w.k_norm;
  d.w_o = w.w_o;
  d.in_norm = w.in_norm;
  return d;
}

quail_status check_model_ml(const quail_model_ml_desc* m) {
  if (m == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "model is null");
  if (m->n_layers < 1 || m->n_layers > QUAIL_MAX_LAYERS || m->layers == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "need n_layers in [1, %d] and layers", QUAIL_MAX_LAYERS);
  if (m->intermediate < 256 || m->intermediate % 256 != 0 || m->intermediate > 65536)
    return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "intermediate must be a multiple of 256 in [256, 65536] (got %d)",
                m->intermediate);
  for (int l = 0; l < m->n_layers; ++l) {
    const quail_model_desc d = layer_desc(m, l);
    const quail_status s = check_model(&d);
    if (s != QUAIL_OK) return s;
    const quail_layer_weights& w = m->layers[l];
    for (const void* p : {w.post_norm, w.w_gate, w.w_up, w.w_down}) {
      if (p == nullptr || !aligned16(p)) return fail(QUAIL_ERR_INVALID_ARG, "layer %d: MLP weight null or misaligned", l);
    }
  }
  return QUAIL_OK;
}

quail_paged_kv layer_kv(const quail_paged_kv_ml* kv, int l) {
  quail_paged_kv k{};
  k.k_pool = kv->k_pools[l];
  k.v_pool = kv->v_pools[l];
  k.num_pages = kv->num_pages;
  k.page_size = kv->page_size;
  k.page_table = kv->page_table;
  k.max_pages = kv->max_pages;
  k.doc_len = kv->doc_len;
  k.max_doc_len = kv->max_doc_len;
  return k;
}

struct MLBuffers {
  Buffers b;        // rows of the shared steps = (document, evaluated node)
  float* h;         // [rows, d] residual stream
  bf16* act;        // [rows_p, 2I] SiLU(gate) * up, split
  float* gu_part;   // [ks_gu, rows, 2I]
  float* dn_part;   // [ks_dn, rows, d]
  int ks_gu, ks_dn;
};

size_t plan_ml(uint8_t* base, const quail_model_ml_desc* m, const quail_trie* t, int N, int max_doc_len,
               MLBuffers* out) {
  const quail_model_desc d0 = layer_desc(m, 0);
  const int a = t->n_eval();
  const int rows = N * a;
  MLBuffers x{};
  const size_t base_bytes = round_up(plan(base, &d0, rows, N, a, max_doc_len, true, t->eval_child_offsets.back(),
                                           false, 3 * rows, base ? &x.b : nullptr),
                                      256);  // the extras start 256-byte aligned like every carved buffer
  const int sms = planning_sms();
  const int I = m->intermediate, d = m->hidden;
  const int m_tiles = static_cast<int>(round_up(rows, 128) / 128);
  x.ks_gu = choose_k_splits(m_tiles * (2 * I / 256), d / 64, sms);
  x.ks_dn = choose_k_splits(m_tiles * static_cast<int>(round_up(d, 256) / 256), I / 64, sms);
  Carver c{base ? base + base_bytes : nullptr};
  x.h = c.take<float>(static_cast<size_t>(rows) * d);
  x.act = c.take<bf16>(round_up(rows, 128) * 2 * I);
  x.gu_part = c.take<float>(static_cast<size_t>(x.ks_gu) * rows * 2 * I);
  x.dn_part = c.take<float>(static_cast<size_t>(x.ks_dn) * rows * d);
  if (out) *out = x;
  return base_bytes + c.off + 256;
}

// C[ks] = A W^T over the split A rows (A [rows_p, 2K] bf16, W [n, K] bf16 blocks).
quail_status run_split_gemm(const bf16* A, int rows, int K, const void* const* w, const int* nrows, int count,
                            int ks, float* C, int ldc, DeviceState* ds, cudaStream_t st) {
  CUtensorMap tA;
  quail_status s = encode_2d_bf16(&tA, A, round_up(rows, 128), 2 * K, 2 * K, 64, 128);
  if (s != QUAIL_OK) return s;
  BSet bs{};
  int col = 0;
  for (int i = 0; i < count; ++i) {
    s = encode_2d_bf16(&bs.map[i], w[i], nrows[i], K, K, 64, 256);
    if (s != QUAIL_OK) return s;
    bs.n_begin[i] = col;
    col += nrows[i];
    bs.n_begin[i + 1] = col;
  }
  bs.count = count;
  const size_t slab = static_cast<size_t>(rows) * ldc;
  CUDA_TRY(launch_gemm_proj(tA, bs, rows, col, K, ks, C, slab, ldc, ds->num_sms, ds->err, st));
  return QUAIL_OK;
}

// The trie_tree pass over num_docs documents with the trie's device image
// and the buffers of plan(..., a, N, a, ..., head = true, n_child, ...);
// stage events when `marks`.
quail_status trie_tree_pass(const quail_model_desc* model, const quail_paged_kv* kv, const quail_trie* trie,
                            const quail_trie::DeviceImage* img, int num_docs, const Buffers& b, DeviceState* ds,
                            cudaStream_t st, float* label_logscore, float* label_prob, int32_t* label_argmax,
                            bool marks) {
  const int a = trie->n_eval();
  const int n_child = trie->eval_child_offsets.back();
  const NodeTables nt{img->eval_token, img->eval_depth, img->eval_parent, a};
  const RowMap map{a, nullptr, nullptr, nullptr};
  const int rows = num_docs * a;
  auto mark = [&](int stage, bool end) {
    if (marks) stage_mark(stage, end, st);
  };

  mark(QUAIL_STAGE_PROLOGUE, false);
  quail_status s = run_prologue(model, nt, b, ds, st);
  if (s != QUAIL_OK) return s;
  mark(QUAIL_STAGE_PROLOGUE, true);

  mark(QUAIL_STAGE_ATTENTION, false);
  s = run_attention(model, kv, nt, map, num_docs, b, ds, st);
  if (s != QUAIL_OK) return s;
  mark(QUAIL_STAGE_ATTENTION, true);

  mark(QUAIL_STAGE_WO_NORM, false);
  s = run_wo_norm(model, nt, map, rows, b, ds, st);
  if (s != QUAIL_OK) return s;
  mark(QUAIL_STAGE_WO_NORM, true);

  mark(QUAIL_STAGE_HEAD, false);
  {
    const int d = model->hidden;
    const int n_tiles = (model->vocab + kHeadBN - 1) / kHeadBN;
    CUtensorMap tA, tB;
    s = encode_2d_bf16(&tA, b.z, round_up(rows, 128), d, d, 64, 128);
    if (s != QUAIL_OK) return s;
    s = encode_2d_bf16(&tB, model->lm_head, model->vocab, d, d, 64, head_b_box_rows(rows));
    if (s != QUAIL_OK) return s;
    HeadEpilogueArgs ha{b.lse_part, b.child_logit, img->eval_child_offsets, img->eval_child_tokens, b.z_f32,
                        static_cast<const bf16*>(model->lm_head), d, a, n_child, n_tiles};
    CUDA_TRY(launch_gemm_head(tA, tB, rows, model->vocab, d, ha, ds->num_sms, ds->err, st));
    mark(QUAIL_STAGE_HEAD, true);
  }
  mark(QUAIL_STAGE_SCORING, false);
  LabelScoreArgs la{b.child_logit,
                    b.lse_part,
                    (model->vocab + kHeadBN - 1) / kHeadBN,
                    b.lse,
                    img->label_term_offsets,
                    img->label_term_eval,
                    img->label_term_slot,
                    img->label_prefix_eval,
                    img->eval_child_offsets,
                    a,
                    n_child,
                    trie->num_labels,
                    label_logscore,
                    label_prob,
                    label_argmax};
  CUDA_TRY(launch_label_score(la, num_docs, ds->num_sms, st));
  mark(QUAIL_STAGE_SCORING, true);
  return QUAIL_OK;
}

// ------------------------------------------------------------------ shortlist
quail_status upload_shortlist(quail_shortlist* sl, cudaStream_t st, const quail_shortlist::DeviceImage** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(sl->mu);
  auto it = sl->images.find(dev);
  if (it != sl->images.end()) {
    *out = &it->second;
    return QUAIL_OK;
  }
  const std::vector<int32_t>* arrays[] = {&sl->row_off, &sl->row_eval, &sl->row_parent, &sl->child_off,
                                          &sl->child_row, &sl->child_tok, &sl->lab_off, &sl->lab_id,
                                          &sl->term_off, &sl->term_t, &sl->pref_t0, &sl->pref_t1};
  const int na = sizeof(arrays) / sizeof(arrays[0]);
  std::vector<size_t> offs(na);
  size_t total = 0;
  for (int i = 0; i < na; ++i) {
    offs[i] = total;
    total += round_up(std::max<size_t>(arrays[i]->size(), 1) * 4, 256);
  }
  std::vector<uint8_t> host(total, 0);
  for (int i = 0; i < na; ++i)
    if (!arrays[i]->empty()) std::memcpy(host.data() + offs[i], arrays[i]->data(), arrays[i]->size() * 4);
  void* dptr = nullptr;
  CUDA_TRY(cudaMalloc(&dptr, total));
  cudaError_t e = cudaMemcpyAsync(dptr, host.data(), total, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaFree(dptr);
    return fail(QUAIL_ERR_CUDA, "shortlist upload: %s", cudaGetErrorString(e));
  }
  quail_shortlist::DeviceImage img;
  img.base = dptr;
  const int32_t** fields[] = {&img.row_off,   &img.row_eval, &img.row_parent, &img.child_off,
                              &img.child_row, &img.child_tok, &img.lab_off,   &img.lab_id,
                              &img.term_off,  &img.term_t,   &img.pref_t0,    &img.pref_t1};
  for (int i = 0; i < na; ++i)
    *fields[i] = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(dptr) + offs[i]);
  auto res = sl->images.emplace(dev, img);
  *out = &res.first->second;
  return QUAIL_OK;
}

// A plan made from this trie (the counts it was built from agree).
bool shortlist_matches(const quail_shortlist* sl, const quail_trie* t) {
  return sl->num_labels == t->num_labels && sl->trie_nodes == t->n_nodes() && sl->trie_eval == t->n_eval() &&
         sl->prefix_trie != nullptr && sl->prefix_trie->vocab == t->vocab;
}

// Workspace of the shortlisted call: the prefix pass and the second pass
// share one region (the second starts after the first has finished on the
// stream); the selection, child log-probs and prefix scores follow it.
struct ShortlistBuffers {
  Buffers b1, b2;
  int* sel;       // [N, B]
  float* clp;     // [N * B, max_children]
  bf16* attn_c;   // [round_up(R, 128), 2 hq 128] attention output of the real rows, compacted
  float* ls1;     // [N, G] prefix log scores
  float* prob1;   // [N, G]
  int* am1;       // [N]
  int B, Bq;      // kept groups per document; rows per document (B * max_rows)
  int R;          // second-pass rows (N * Bq)
};

size_t plan_shortlist(uint8_t* base, const quail_model_desc* m, const quail_shortlist* sl, int beam, int N,
                      int max_doc_len, ShortlistBuffers* out) {
  const quail_trie* pt = sl->prefix_trie;
  ShortlistBuffers x{};
  x.B = std::min(beam, sl->num_groups);
  x.Bq = x.B * sl->max_rows;
  x.R = N * x.Bq;
  const int a1 = pt->n_eval();
  const size_t p1 = plan(base, m, a1, N, a1, max_doc_len, true, pt->eval_child_offsets.back(), false, 0,
                         base ? &x.b1 : nullptr);
  // small ints: token, depth, parent, padded row of every row; 2 zeros; count; block bases; document bases
  // and row counts
  const size_t p2 = plan(base, m, x.R, N, x.Bq, max_doc_len, true, 0, true, 4 * x.R + 3 + N * x.B + 2 * N,
                         base ? &x.b2 : nullptr);
  const size_t shared = round_up(std::max(p1, p2), 256);
  Carver c{base ? base + shared : nullptr};
  x.sel = c.take<int>(static_cast<size_t>(N) * x.B);
  x.clp = c.take<float>(static_cast<size_t>(N) * x.B * std::max(sl->max_children, 1));
  x.attn_c = c.take<bf16>(round_up(x.R, 128) * 2 * m->n_q_heads * 128);
  x.ls1 = c.take<float>(static_cast<size_t>(N) * sl->num_groups);
  x.prob1 = c.take<float>(static_cast<size_t>(N) * sl->num_groups);
  x.am1 = c.take<int>(N);
  if (out) *out = x;
  return shared + c.off + 256;
}

}  // namespace

// ================================================================== C ABI
void quail::count_launch() { ++g_launches; }

namespace quail {

bool encode_3d_f32_store(void* tm, void* ptr, uint64_t cols, uint64_t rows, uint64_t planes, uint64_t ld,
                         uint64_t plane_ld, uint32_t box_cols, uint32_t box_rows) {
  if (g_encode == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {ld * 4, plane_ld * 4};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(static_cast<CUtensorMap*>(tm), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d_bf16_store(void* tm, void* ptr, uint64_t cols, uint64_t rows, uint64_t planes, uint64_t ld,
                          uint64_t plane_ld, uint32_t box_cols, uint32_t box_rows) {
  if (g_encode == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {ld * 2, plane_ld * 2};
  cuuint32_t box[3] = {box_cols, box_rows, static_cast<cuuint32_t>(planes)};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(static_cast<CUtensorMap*>(tm), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

quail_status estimate_methods_host(const quail_cost_model* md, const quail_cost_workload* w, const quail_trie* t,
                                   quail_method_cost* costs, int32_t* best, std::string* msg);
}

extern "C" {

const char* quail_last_error(void) { return g_last_error.c_str(); }

int32_t quail_launch_count(void) { return g_launches; }

quail_status quail_estimate_methods(const quail_cost_model* model, const quail_cost_workload* work,
                                    const quail_trie* trie, quail_method_cost* costs, int32_t* best) {
  std::string msg;
  const quail_status s = estimate_methods_host(model, work, trie, costs, best, &msg);
  if (s != QUAIL_OK) return fail(s, "%s", msg.c_str());
  return QUAIL_OK;
}

quail_status quail_trie_build(const int32_t* tokens, const int64_t* label_offsets, int32_t num_labels,
                              int32_t root_token, int32_t vocab, const uint8_t* word_continuation_bitmap,
                              int32_t flags, quail_trie** out) {
  if (out == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  quail_trie* t = new quail_trie();
  std::string msg;
  quail_status s = quail_build_trie_host(tokens, label_offsets, num_labels, root_token, vocab,
                                         word_continuation_bitmap, flags, t, &msg);
  if (s != QUAIL_OK) {
    delete t;
    return fail(s, "%s", msg.c_str());
  }
  *out = t;
  return QUAIL_OK;
}

quail_status quail_trie_view(const quail_trie* t, quail_trie_csr* v) {
  if (t == nullptr || v == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "null argument");
  v->n_nodes = t->n_nodes();
  v->num_labels = t->num_labels;
  v->n_eval = t->n_eval();
  v->n_eval_children = t->eval_child_offsets.back();
  v->max_depth = t->max_depth;
  v->has_prefix_labels = t->has_prefix_labels;
  v->parent = t->parent.data();
  v->depth = t->depth.data();
  v->token = t->token.data();
  v->subtree_size = t->subtree_size.data();
  v->child_offsets = t->child_offsets.data();
  v->child_nodes = t->child_nodes.data();
  v->child_tokens = t->child_tokens.data();
  v->is_branching = t->is_branching.data();
  v->subtree_labels = t->subtree_labels.data();
  v->node_label = t->node_label.data();
  v->label_end_node = t->label_end_node.data();
  v->label_length = t->label_length.data();
  v->label_decide_depth = t->label_decide_depth.data();
  v->eval_nodes = t->eval_nodes.data();
  v->eval_index_of_node = t->eval_index_of_node.data();
  v->eval_child_offsets = t->eval_child_offsets.data();
  return QUAIL_OK;
}

void quail_trie_free(quail_trie* t) {
  if (t == nullptr) return;
  int cur = -1;
  cudaGetDevice(&cur);
  for (auto& kv : t->images) {
    if (kv.second.base == nullptr) continue;
    if (cudaSetDevice(kv.first) == cudaSuccess) cudaFree(kv.second.base);
  }
  if (cur >= 0 && !t->images.empty()) cudaSetDevice(cur);
  delete t;
}

quail_status quail_trie_upload(quail_trie* t, quail_stream_t stream) {
  if (t == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "trie is null");
  const quail_trie::DeviceImage* img = nullptr;
  return upload_trie(t, reinterpret_cast<cudaStream_t>(stream), &img);
}

size_t quail_workspace_size(const quail_model_desc* model, const quail_trie* trie, int32_t num_letters,
                            int32_t num_docs, int32_t max_doc_len, quail_mode mode) {
  if (model == nullptr || num_docs < 0 || max_doc_len <= 0) return 0;
  if (model->n_kv_heads <= 0 || model->n_q_heads <= 0 || model->hidden <= 0 || model->vocab <= 0) return 0;
  switch (mode) {
    case QUAIL_MODE_TRIE_TREE:
      if (trie == nullptr) return 0;
      return plan(nullptr, model, trie->n_eval(), num_docs, trie->n_eval(), max_doc_len, true,
                  trie->eval_child_offsets.back(), false, 0, nullptr);
    case QUAIL_MODE_LETTERS:
      if (num_letters < 2) return 0;
      return plan(nullptr, model, 1, num_docs, 1, max_doc_len, false, 0, true, num_letters + 4, nullptr);
    case QUAIL_MODE_TRIE_DECODE:
      if (trie == nullptr) return 0;
      return plan(nullptr, model, trie->n_int(), num_docs, 1, max_doc_len, false, 0, true, 2 * num_docs + 4,
                  nullptr);
    case QUAIL_MODE_JOIN_IF:
      if (trie == nullptr || num_letters < 1) return 0;
      return plan(nullptr, model, trie->n_eval(), num_docs, trie->num_labels, max_doc_len, false, 0, true,
                  trie->num_labels + num_letters, nullptr);
  }
  return 0;
}

quail_status quail_classify_trie_tree(const quail_model_desc* model, const quail_paged_kv* kv, quail_trie* trie,
                                      int32_t num_docs, void* workspace, size_t workspace_bytes,
                                      float* label_logscore, float* label_prob, int32_t* label_argmax,
                                      quail_stream_t stream) {
  g_launches = 0;
  quail_status s = check_model(model);
  if (s != QUAIL_OK) return s;
  s = check_kv(kv, model);
  if (s != QUAIL_OK) return s;
  if (trie == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "trie is null");
  if (trie->vocab != model->vocab) return fail(QUAIL_ERR_INVALID_ARG, "trie vocab %d != model vocab %d", trie->vocab, model->vocab);
  if (num_docs < 0) return fail(QUAIL_ERR_INVALID_ARG, "num_docs < 0");
  if (num_docs == 0) return QUAIL_OK;
  if (num_docs > 65535) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 65535 documents per call");
  if (label_logscore == nullptr || label_prob == nullptr || label_argmax == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "an output pointer is null");
  const int a = trie->n_eval();
  const int n_child = trie->eval_child_offsets.back();
  const size_t need = plan(nullptr, model, a, num_docs, a, kv->max_doc_len, true, n_child, false, 0, nullptr);
  s = check_workspace(workspace, workspace_bytes, need);
  if (s != QUAIL_OK) return s;
  DeviceState* ds = nullptr;
  s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const quail_trie::DeviceImage* img = nullptr;
  s = upload_trie(trie, st, &img);
  if (s != QUAIL_OK) return s;
  Buffers b;
  plan(static_cast<uint8_t*>(workspace), model, a, num_docs, a, kv->max_doc_len, true, n_child, false, 0, &b);
  return trie_tree_pass(model, kv, trie, img, num_docs, b, ds, st, label_logscore, label_prob, label_argmax, true);
}

quail_status quail_classify_letters(const quail_model_desc* model, const quail_paged_kv* kv,
                                    const int32_t* letter_tokens, int32_t num_letters, int32_t root_token,
                                    int32_t num_docs, void* workspace, size_t workspace_bytes,
                                    float* letter_logprob, float* letter_prob, int32_t* letter_argmax,
                                    quail_stream_t stream) {
  g_launches = 0;
  quail_status s = check_model(model);
  if (s != QUAIL_OK) return s;
  s = check_kv(kv, model);
  if (s != QUAIL_OK) return s;
  if (letter_tokens == nullptr || num_letters < 2) return fail(QUAIL_ERR_INVALID_ARG, "need at least 2 letters");
  if (num_letters > 8192) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 8192 letters");
  if (root_token < 0 || root_token >= model->vocab) return fail(QUAIL_ERR_TOKEN_RANGE, "root token out of range");
  for (int i = 0; i < num_letters; ++i) {
    if (letter_tokens[i] < 0 || letter_tokens[i] >= model->vocab)
      return fail(QUAIL_ERR_TOKEN_RANGE, "letter %d has token %d outside [0, vocab)", i, letter_tokens[i]);
  }
  {
    std::vector<int32_t> sorted(letter_tokens, letter_tokens + num_letters);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
      return fail(QUAIL_ERR_DUPLICATE_LABEL, "letter tokens must be distinct");
  }
  if (num_docs < 0) return fail(QUAIL_ERR_INVALID_ARG, "num_docs < 0");
  if (num_docs == 0) return QUAIL_OK;
  if (num_docs > 65535) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 65535 documents per call");
  if (letter_logprob == nullptr || letter_prob == nullptr || letter_argmax == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "an output pointer is null");
  const size_t need = plan(nullptr, model, 1, num_docs, 1, kv->max_doc_len, false, 0, true, num_letters + 4, nullptr);
  s = check_workspace(workspace, workspace_bytes, need);
  if (s != QUAIL_OK) return s;
  DeviceState* ds = nullptr;
  s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Buffers b;
  plan(static_cast<uint8_t*>(workspace), model, 1, num_docs, 1, kv->max_doc_len, false, 0, true, num_letters + 4, &b);
  // small ints: [0] root token, [1] depth 0, [2] parent -1, [4..] letters
  std::vector<int32_t> host(num_letters + 4);
  host[0] = root_token;
  host[1] = 0;
  host[2] = -1;
  host[3] = 0;
  std::memcpy(host.data() + 4, letter_tokens, num_letters * sizeof(int32_t));
  CUDA_TRY(cudaMemcpyAsync(b.small, host.data(), host.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st));
  const NodeTables nt{b.small, b.small + 1, b.small + 2, 1};
  const RowMap map{1, nullptr, nullptr, nullptr};

  stage_mark(QUAIL_STAGE_PROLOGUE, false, st);
  s = run_prologue(model, nt, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_PROLOGUE, true, st);
  stage_mark(QUAIL_STAGE_ATTENTION, false, st);
  s = run_attention(model, kv, nt, map, num_docs, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_ATTENTION, true, st);
  stage_mark(QUAIL_STAGE_WO_NORM, false, st);
  s = run_wo_norm(model, nt, map, num_docs, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_WO_NORM, true, st);
  stage_mark(QUAIL_STAGE_HEAD, false, st);
  CUDA_TRY(launch_letters_head(b.z_f32, static_cast<const bf16*>(model->lm_head), b.small + 4, num_letters,
                               num_docs, model->hidden, letter_logprob, letter_prob, letter_argmax, st));
  stage_mark(QUAIL_STAGE_HEAD, true, st);
  return QUAIL_OK;
}

size_t quail_workspace_size_ml(const quail_model_ml_desc* model, const quail_trie* trie, int32_t num_docs,
                               int32_t max_doc_len) {
  if (model == nullptr || trie == nullptr || num_docs < 0 || max_doc_len <= 0 || model->n_layers < 1 ||
      model->layers == nullptr || model->intermediate < 256 || model->intermediate % 256 != 0)
    return 0;
  if (model->n_kv_heads <= 0 || model->n_q_heads <= 0 || model->hidden <= 0 || model->vocab <= 0) return 0;
  return plan_ml(nullptr, model, trie, num_docs, max_doc_len, nullptr);
}

quail_status quail_classify_trie_tree_ml(const quail_model_ml_desc* model, const quail_paged_kv_ml* kv,
                                         quail_trie* trie, int32_t num_docs, void* workspace, size_t workspace_bytes,
                                         float* label_logscore, float* label_prob, int32_t* label_argmax,
                                         quail_stream_t stream) {
  g_launches = 0;
  quail_status s = check_model_ml(model);
  if (s != QUAIL_OK) return s;
  if (kv == nullptr || kv->k_pools == nullptr || kv->v_pools == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "kv is null");
  const quail_model_desc d0 = layer_desc(model, 0);
  for (int l = 0; l < model->n_layers; ++l) {
    const quail_paged_kv kl = layer_kv(kv, l);
    s = check_kv(&kl, &d0);
    if (s != QUAIL_OK) return s;
  }
  if (trie == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "trie is null");
  if (trie->vocab != model->vocab)
    return fail(QUAIL_ERR_INVALID_ARG, "trie vocab %d != model vocab %d", trie->vocab, model->vocab);
  if (num_docs < 0) return fail(QUAIL_ERR_INVALID_ARG, "num_docs < 0");
  if (num_docs == 0) return QUAIL_OK;
  if (num_docs > 65535) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 65535 documents per call");
  if (label_logscore == nullptr || label_prob == nullptr || label_argmax == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "an output pointer is null");
  const int a = trie->n_eval();
  const int rows = num_docs * a;
  const int n_child = trie->eval_child_offsets.back();
  const size_t need = plan_ml(nullptr, model, trie, num_docs, kv->max_doc_len, nullptr);
  s = check_workspace(workspace, workspace_bytes, need);
  if (s != QUAIL_OK) return s;
  DeviceState* ds = nullptr;
  s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const quail_trie::DeviceImage* img = nullptr;
  s = upload_trie(trie, st, &img);
  if (s != QUAIL_OK) return s;
  MLBuffers x;
  plan_ml(static_cast<uint8_t*>(workspace), model, trie, num_docs, kv->max_doc_len, &x);
  const Buffers& b = x.b;
  // node tables of the (document, evaluated node) rows: N disjoint copies of P
  std::vector<int32_t> host(3 * static_cast<size_t>(rows));
  for (int i = 0; i < num_docs; ++i) {
    for (int e = 0; e < a; ++e) {
      const size_t r = static_cast<size_t>(i) * a + e;
      host[r] = trie->eval_token[e];
      host[rows + r] = trie->eval_depth[e];
      host[2 * static_cast<size_t>(rows) + r] = trie->eval_parent[e] < 0 ? -1 : i * a + trie->eval_parent[e];
    }
  }
  CUDA_TRY(cudaMemcpyAsync(b.small, host.data(), host.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st));
  const NodeTables nt{b.small, b.small + rows, b.small + 2 * static_cast<size_t>(rows), rows};
  const RowMap map{a, nullptr, nullptr, nullptr, nullptr, a};
  const int d = model->hidden, I = model->intermediate;

  stage_mark(QUAIL_STAGE_PROLOGUE, false, st);
  CUDA_TRY(launch_gather_embed(static_cast<const bf16*>(model->embed), nt.token, rows, d, x.h, st));
  for (int l = 0; l < model->n_layers; ++l) {
    const quail_model_desc ml = layer_desc(model, l);
    const quail_paged_kv kl = layer_kv(kv, l);
    const quail_layer_weights& w = model->layers[l];
    auto span = [&](int j, bool end) { stage_mark(QUAIL_NUM_STAGES + l * QUAIL_LAYER_SPANS + j, end, st); };
    // h += previous layer's MLP output (none before layer 0); x^ = split(RMSNorm(h) g_in)
    span(QUAIL_SPAN_QKV, false);
    CUDA_TRY(launch_residual_norm(x.h, x.dn_part, l == 0 ? 0 : x.ks_dn, static_cast<size_t>(rows) * d, rows, d,
                                  static_cast<const bf16*>(w.in_norm), model->rms_eps, b.xhat, st));
    s = run_qkv(&ml, nt, b, ds, st);
    if (s != QUAIL_OK) return s;
    span(QUAIL_SPAN_QKV, true);
    span(QUAIL_SPAN_ATTENTION, false);
    // every layer sees the same documents: the slot order is computed once
    s = run_attention(&ml, &kl, nt, map, num_docs, b, ds, st, nullptr, l > 0);
    if (s != QUAIL_OK) return s;
    span(QUAIL_SPAN_ATTENTION, true);
    span(QUAIL_SPAN_WO_NORM, false);
    s = run_wo_gemm(&ml, rows, b, ds, st);
    if (s != QUAIL_OK) return s;
    // h += O W_o^T; y = split(RMSNorm(h) g_post)
    CUDA_TRY(launch_residual_norm(x.h, b.h_part, b.gp.ks_wo, static_cast<size_t>(rows) * d, rows, d,
                                  static_cast<const bf16*>(w.post_norm), model->rms_eps, b.xhat, st));
    span(QUAIL_SPAN_WO_NORM, true);
    span(QUAIL_SPAN_GATE_UP, false);
    if (x.ks_gu == 1) {
      // one k-split: SiLU(gate) * up fused into the projection's epilogue
      CUtensorMap tA;
      s = encode_2d_bf16(&tA, b.xhat, round_up(rows, 128), 2 * d, 2 * d, 64, 128);
      if (s != QUAIL_OK) return s;
      BSet bs{};
      s = encode_2d_bf16(&bs.map[0], w.w_gate, I, d, d, 64, 128);
      if (s != QUAIL_OK) return s;
      s = encode_2d_bf16(&bs.map[1], w.w_up, I, d, d, 64, 128);
      if (s != QUAIL_OK) return s;
      bs.count = 2;
      bs.glu = 1;
      bs.n_begin[1] = bs.n_begin[2] = 2 * I;
      CUDA_TRY(launch_gemm_swiglu(tA, bs, rows, I, d, x.act, ds->num_sms, ds->err, st));
      span(QUAIL_SPAN_GATE_UP, true);
      span(QUAIL_SPAN_SILU_MUL, false);
      span(QUAIL_SPAN_SILU_MUL, true);
    } else {
      const void* gu[2] = {w.w_gate, w.w_up};
      const int gu_rows[2] = {I, I};
      s = run_split_gemm(b.xhat, rows, d, gu, gu_rows, 2, x.ks_gu, x.gu_part, 2 * I, ds, st);
      if (s != QUAIL_OK) return s;
      span(QUAIL_SPAN_GATE_UP, true);
      span(QUAIL_SPAN_SILU_MUL, false);
      CUDA_TRY(launch_silu_mul_split(x.gu_part, x.ks_gu, static_cast<size_t>(rows) * 2 * I, rows, I, x.act, st));
      span(QUAIL_SPAN_SILU_MUL, true);
    }
    const void* dn[1] = {w.w_down};
    const int dn_rows[1] = {d};
    span(QUAIL_SPAN_DOWN, false);
    s = run_split_gemm(x.act, rows, I, dn, dn_rows, 1, x.ks_dn, x.dn_part, d, ds, st);
    if (s != QUAIL_OK) return s;
    span(QUAIL_SPAN_DOWN, true);
  }
  CUDA_TRY(launch_residual_norm(x.h, x.dn_part, x.ks_dn, static_cast<size_t>(rows) * d, rows, d, nullptr,
                                model->rms_eps, nullptr, st));
  CUDA_TRY(launch_norm_out(x.h, rows, d, static_cast<const bf16*>(model->final_norm), model->rms_eps, b.z, b.z_f32,
                           st));
  stage_mark(QUAIL_STAGE_PROLOGUE, true, st);

  stage_mark(QUAIL_STAGE_HEAD, false, st);
  {
    const int n_tiles = (model->vocab + kHeadBN - 1) / kHeadBN;
    CUtensorMap tA, tB;
    s = encode_2d_bf16(&tA, b.z, round_up(rows, 128), d, d, 64, 128);
    if (s != QUAIL_OK) return s;
    s = encode_2d_bf16(&tB, model->lm_head, model->vocab, d, d, 64, head_b_box_rows(rows));
    if (s != QUAIL_OK) return s;
    HeadEpilogueArgs ha{b.lse_part, b.child_logit, img->eval_child_offsets, img->eval_child_tokens, b.z_f32,
                        static_cast<const bf16*>(model->lm_head), d, a, n_child, n_tiles};
    CUDA_TRY(launch_gemm_head(tA, tB, rows, model->vocab, d, ha, ds->num_sms, ds->err, st));
  }
  stage_mark(QUAIL_STAGE_HEAD, true, st);
  stage_mark(QUAIL_STAGE_SCORING, false, st);
  LabelScoreArgs la{b.child_logit,          b.lse_part,           (model->vocab + kHeadBN - 1) / kHeadBN,
                    b.lse,                  img->label_term_offsets, img->label_term_eval,
                    img->label_term_slot,   img->label_prefix_eval,  img->eval_child_offsets,
                    a,                      n_child,              trie->num_labels,
                    label_logscore,         label_prob,           label_argmax};
  CUDA_TRY(launch_label_score(la, num_docs, ds->num_sms, st));
  stage_mark(QUAIL_STAGE_SCORING, true, st);
  return QUAIL_OK;
}

quail_status quail_join_if(const quail_model_desc* model, const quail_paged_kv* kv, quail_trie* partners,
                           int32_t num_anchors, const int32_t* answer_tokens, int32_t n_true, int32_t n_false,
                           void* workspace, size_t workspace_bytes, float* p_true, quail_stream_t stream) {
  g_launches = 0;
  quail_status s = check_model(model);
  if (s != QUAIL_OK) return s;
  s = check_kv(kv, model);
  if (s != QUAIL_OK) return s;
  if (partners == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "partner trie is null");
  if (partners->vocab != model->vocab)
    return fail(QUAIL_ERR_INVALID_ARG, "trie vocab %d != model vocab %d", partners->vocab, model->vocab);
  if (partners->n_eval() != partners->n_nodes())
    return fail(QUAIL_ERR_INVALID_ARG, "the partner trie must be built with QUAIL_TRIE_ALL_NODES");
  const int R = n_true + n_false;
  if (answer_tokens == nullptr || n_true < 0 || n_false < 0 || R < 1 || R > kJoinMaxRows)
    return fail(QUAIL_ERR_INVALID_ARG, "need 1..%d answer tokens (n_true, n_false >= 0)", kJoinMaxRows);
  for (int i = 0; i < R; ++i) {
    if (answer_tokens[i] < 0 || answer_tokens[i] >= model->vocab)
      return fail(QUAIL_ERR_TOKEN_RANGE, "answer token %d is %d, outside [0, vocab)", i, answer_tokens[i]);
  }
  {
    std::vector<int32_t> sorted(answer_tokens, answer_tokens + R);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
      return fail(QUAIL_ERR_DUPLICATE_LABEL, "answer tokens must be distinct");
  }
  if (num_anchors < 0) return fail(QUAIL_ERR_INVALID_ARG, "num_anchors < 0");
  if (num_anchors == 0) return QUAIL_OK;
  if (num_anchors > 65535) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 65535 anchors per call");
  if (p_true == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "p_true is null");
  const int nodes = partners->n_eval();
  const int M = partners->num_labels;
  const size_t need = plan(nullptr, model, nodes, num_anchors, M, kv->max_doc_len, false, 0, true, M + R, nullptr);
  s = check_workspace(workspace, workspace_bytes, need);
  if (s != QUAIL_OK) return s;
  DeviceState* ds = nullptr;
  s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const quail_trie::DeviceImage* img = nullptr;
  s = upload_trie(partners, st, &img);
  if (s != QUAIL_OK) return s;
  Buffers b;
  plan(static_cast<uint8_t*>(workspace), model, nodes, num_anchors, M, kv->max_doc_len, false, 0, true, M + R, &b);
  // small ints: [0, M) the node row of each partner's last token, [M, M + R) the answer tokens
  std::vector<int32_t> host(M + R);
  for (int m = 0; m < M; ++m) host[m] = partners->eval_index_of_node[partners->label_end_node[m]];
  std::memcpy(host.data() + M, answer_tokens, R * sizeof(int32_t));
  CUDA_TRY(cudaMemcpyAsync(b.small, host.data(), host.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st));
  const NodeTables nt{img->eval_token, img->eval_depth, img->eval_parent, nodes};
  const RowMap map{M, nullptr, nullptr, nullptr, b.small};
  const int rows = num_anchors * M;

  stage_mark(QUAIL_STAGE_PROLOGUE, false, st);
  s = run_prologue(model, nt, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_PROLOGUE, true, st);
  stage_mark(QUAIL_STAGE_ATTENTION, false, st);
  s = run_attention(model, kv, nt, map, num_anchors, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_ATTENTION, true, st);
  stage_mark(QUAIL_STAGE_WO_NORM, false, st);
  s = run_wo_norm(model, nt, map, rows, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_WO_NORM, true, st);
  stage_mark(QUAIL_STAGE_HEAD, false, st);
  CUDA_TRY(launch_join_head(b.z_f32, static_cast<const bf16*>(model->lm_head), b.small + M, n_true, R, rows, M,
                            model->hidden, p_true, st));
  stage_mark(QUAIL_STAGE_HEAD, true, st);
  return QUAIL_OK;
}

quail_status quail_classify_trie_decode_step(const quail_model_desc* model, const quail_paged_kv* kv,
                                             quail_trie* trie, int32_t num_docs, int32_t* node_cursor,
                                             int32_t* label_out, int32_t* active_count, uint8_t* touched_nodes,
                                             void* workspace, size_t workspace_bytes, quail_stream_t stream) {
  g_launches = 0;
  quail_status s = check_model(model);
  if (s != QUAIL_OK) return s;
  s = check_kv(kv, model);
  if (s != QUAIL_OK) return s;
  if (trie == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "trie is null");
  if (trie->vocab != model->vocab) return fail(QUAIL_ERR_INVALID_ARG, "trie vocab %d != model vocab %d", trie->vocab, model->vocab);
  if (trie->has_prefix_labels)
    return fail(QUAIL_ERR_PREFIX_LABEL_UNSUPPORTED,
                "greedy decoding cannot stop at a label that is a prefix of another label");
  if (num_docs < 0) return fail(QUAIL_ERR_INVALID_ARG, "num_docs < 0");
  if (node_cursor == nullptr || label_out == nullptr || active_count == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "cursor, label or count pointer is null");
  if (num_docs == 0) {
    CUDA_TRY(cudaMemsetAsync(active_count, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)));
    return QUAIL_OK;
  }
  if (num_docs > 65535) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 65535 documents per call");
  const int ni = trie->n_int();
  const size_t need = plan(nullptr, model, ni, num_docs, 1, kv->max_doc_len, false, 0, true, 2 * num_docs + 4, nullptr);
  s = check_workspace(workspace, workspace_bytes, need);
  if (s != QUAIL_OK) return s;
  DeviceState* ds = nullptr;
  s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const quail_trie::DeviceImage* img = nullptr;
  s = upload_trie(trie, st, &img);
  if (s != QUAIL_OK) return s;
  Buffers b;
  plan(static_cast<uint8_t*>(workspace), model, ni, num_docs, 1, kv->max_doc_len, false, 0, true, 2 * num_docs + 4, &b);
  int* slot_doc = b.small;
  int* slot_node = b.small + num_docs;
  int* n_slots = b.small + 2 * num_docs;
  const DecodeTrie dt{img->child_offsets, img->child_nodes, img->child_tokens, img->subtree_labels,
                      img->unique_label,  img->int_index_of_node, trie->n_nodes()};
  const NodeTables nt{img->int_token, img->int_depth, img->int_parent, ni};
  const RowMap map{1, slot_node, slot_doc, n_slots};

  CUDA_TRY(launch_decode_prepare(dt, num_docs, node_cursor, label_out, slot_doc, slot_node, n_slots, active_count, st));
  stage_mark(QUAIL_STAGE_PROLOGUE, false, st);
  s = run_prologue(model, nt, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_PROLOGUE, true, st);
  stage_mark(QUAIL_STAGE_ATTENTION, false, st);
  s = run_attention(model, kv, nt, map, num_docs, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_ATTENTION, true, st);
  stage_mark(QUAIL_STAGE_WO_NORM, false, st);
  s = run_wo_norm(model, nt, map, num_docs, b, ds, st);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_WO_NORM, true, st);
  stage_mark(QUAIL_STAGE_HEAD, false, st);
  CUDA_TRY(launch_decode_select(dt, b.z_f32, static_cast<const bf16*>(model->lm_head), model->hidden, num_docs,
                                slot_doc, n_slots, node_cursor, label_out, active_count, touched_nodes, st));
  stage_mark(QUAIL_STAGE_HEAD, true, st);
  return QUAIL_OK;
}

// Test hook, not part of the public header: shortens the limit of every
// pipeline wait (cycles > 0), or restores the default (cycles <= 0), so that a
// test can make a wait run out and check that QUAIL_ERR_DEVICE_TIMEOUT comes
// back through quail_device_status with the context still usable. Waits that
// drain in-flight copies and MMAs before a block exits keep the long limit.
// Synchronises the device.
quail_status quail_test_set_pipeline_wait_limit(long long cycles) {
  DeviceState* ds = nullptr;
  quail_status s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  const long long v = cycles > 0 ? cycles : quail::kWaitLimitCycles;
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(set_pipeline_wait_limit_gemm(v));
  CUDA_TRY(set_pipeline_wait_limit_attention(v));
  CUDA_TRY(set_pipeline_wait_limit_attention_tc(v));
  CUDA_TRY(cudaDeviceSynchronize());
  return QUAIL_OK;
}

quail_status quail_device_status(quail_stream_t stream) {
  DeviceState* ds = nullptr;
  quail_status s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int h[2] = {0, 0};
  CUDA_TRY(cudaMemcpy(h, ds->err, sizeof(h), cudaMemcpyDeviceToHost));
  if (h[0] == 0) return QUAIL_OK;
  const int zero[2] = {0, 0};
  CUDA_TRY(cudaMemcpy(ds->err, zero, sizeof(zero), cudaMemcpyHostToDevice));
  if (h[0] == QUAIL_ERR_DEVICE_BOUNDS)
    return fail(QUAIL_ERR_DEVICE_BOUNDS, "document %d: doc_len or a page id out of range", h[1]);
  if (h[0] == QUAIL_ERR_DEVICE_TIMEOUT)
    return fail(QUAIL_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (block tag %d)", h[1]);
  return fail(static_cast<quail_status>(h[0]), "device error %d (detail %d)", h[0], h[1]);
}

quail_status quail_set_stage_events(quail_event_t* events, int32_t num_stages) {
  std::lock_guard<std::mutex> lk(g_ev_mu);
  g_events.clear();
  if (events == nullptr || num_stages <= 0) return QUAIL_OK;
  if (num_stages > QUAIL_NUM_STAGES + QUAIL_LAYER_SPANS * QUAIL_MAX_LAYERS)
    return fail(QUAIL_ERR_INVALID_ARG, "at most %d stages", QUAIL_NUM_STAGES + QUAIL_LAYER_SPANS * QUAIL_MAX_LAYERS);
  for (int i = 0; i < 2 * num_stages; ++i) g_events.push_back(reinterpret_cast<cudaEvent_t>(events[i]));
  return QUAIL_OK;
}


// trie_tree without any device allocation: the same kernels as
// quail_classify_trie_tree, with the trie tables and every intermediate placed
// in the library's fixed scratch array instead of a caller workspace and a
// library-allocated trie image. For callers that must not allocate device
// memory (see quail.h).
quail_status quail_classify_trie_tree_noalloc(const quail_model_desc* model, const quail_paged_kv* kv,
                                              const quail_trie* trie, int32_t num_docs, float* label_logscore,
                                              float* label_prob, int32_t* label_argmax, quail_stream_t stream) {
  g_launches = 0;
  quail_status s = check_model(model);
  if (s != QUAIL_OK) return s;
  s = check_kv(kv, model);
  if (s != QUAIL_OK) return s;
  if (trie == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "trie is null");
  if (trie->vocab != model->vocab) return fail(QUAIL_ERR_INVALID_ARG, "trie vocab %d != model vocab %d", trie->vocab, model->vocab);
  if (num_docs < 0) return fail(QUAIL_ERR_INVALID_ARG, "num_docs < 0");
  if (num_docs == 0) return QUAIL_OK;
  if (num_docs > 65535) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 65535 documents per call");
  if (label_logscore == nullptr || label_prob == nullptr || label_argmax == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "an output pointer is null");
  const int a = trie->n_eval();
  const int n_child = trie->eval_child_offsets.back();
  const size_t image = trie_tree_image_bytes(trie);
  const size_t need = image + plan(nullptr, model, a, num_docs, a, kv->max_doc_len, true, n_child, false, 0, nullptr);
  if (need > kNoAllocScratchBytes)
    return fail(QUAIL_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch but the fixed scratch holds %zu: pass fewer documents "
                "or use quail_classify_trie_tree with a caller-allocated workspace",
                need, kNoAllocScratchBytes);
  DeviceState* ds = nullptr;
  s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  uint8_t* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != QUAIL_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  quail_trie::DeviceImage img{};
  s = copy_trie_tree_image(trie, scratch, st, &img);
  if (s != QUAIL_OK) return s;
  Buffers b;
  plan(scratch + image, model, a, num_docs, a, kv->max_doc_len, true, n_child, false, 0, &b);
  return trie_tree_pass(model, kv, trie, &img, num_docs, b, ds, st, label_logscore, label_prob, label_argmax, false);
}


// ------------------------------------------------------------------ huge label sets
quail_status quail_trie_build_grouped(const int32_t* tokens, const int64_t* label_offsets, int32_t num_labels,
                                      int32_t root_token, int32_t vocab, const uint8_t* word_continuation_bitmap,
                                      int32_t flags, int32_t num_groups, const int32_t* group_names,
                                      int32_t name_len, quail_trie** out, int32_t* group_of_label) {
  if (out == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  if (tokens == nullptr || label_offsets == nullptr || group_names == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "null argument");
  if (num_labels < 2) return fail(QUAIL_ERR_INVALID_ARG, "need at least 2 labels");
  if (name_len < 1) return fail(QUAIL_ERR_INVALID_ARG, "name_len must be >= 1");
  if (label_offsets[0] != 0) return fail(QUAIL_ERR_INVALID_ARG, "label_offsets[0] must be 0");
  for (int32_t m = 0; m < num_labels; ++m)
    if (label_offsets[m + 1] < label_offsets[m]) return fail(QUAIL_ERR_INVALID_ARG, "label_offsets decrease at %d", m);
  int32_t G = num_groups;
  if (G <= 0) {  // ceil(sqrt(K))
    G = static_cast<int32_t>(std::sqrt(static_cast<double>(num_labels)));
    while (static_cast<int64_t>(G) * G < num_labels) ++G;
    while (G > 1 && static_cast<int64_t>(G - 1) * (G - 1) >= num_labels) --G;
  }
  if (G > num_labels) return fail(QUAIL_ERR_INVALID_ARG, "num_groups %d > num_labels %d", G, num_labels);
  for (int64_t i = 0; i < static_cast<int64_t>(G) * name_len; ++i)
    if (group_names[i] < 0 || group_names[i] >= vocab)
      return fail(QUAIL_ERR_TOKEN_RANGE, "group name token %d outside [0, vocab)", group_names[i]);
  {
    std::vector<int32_t> order(G);
    for (int32_t g = 0; g < G; ++g) order[g] = g;
    auto name = [&](int32_t g) { return group_names + static_cast<int64_t>(g) * name_len; };
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      return std::lexicographical_compare(name(a), name(a) + name_len, name(b), name(b) + name_len);
    });
    for (int32_t i = 1; i < G; ++i)
      if (std::equal(name(order[i]), name(order[i]) + name_len, name(order[i - 1])))
        return fail(QUAIL_ERR_DUPLICATE_LABEL, "group names %d and %d are equal", order[i - 1], order[i]);
  }
  std::vector<int32_t> gol(num_labels);
  quail_group_labels_host(tokens, label_offsets, num_labels, G, gol.data());
  std::vector<int32_t> toks;
  std::vector<int64_t> offs(num_labels + 1, 0);
  toks.reserve(static_cast<size_t>(label_offsets[num_labels]) + static_cast<size_t>(num_labels) * name_len);
  for (int32_t m = 0; m < num_labels; ++m) {
    const int32_t* nm = group_names + static_cast<int64_t>(gol[m]) * name_len;
    toks.insert(toks.end(), nm, nm + name_len);
    toks.insert(toks.end(), tokens + label_offsets[m], tokens + label_offsets[m + 1]);
    offs[m + 1] = static_cast<int64_t>(toks.size());
  }
  quail_trie* t = new quail_trie();
  std::string msg;
  const quail_status s = quail_build_trie_host(toks.data(), offs.data(), num_labels, root_token, vocab,
                                               word_continuation_bitmap, flags, t, &msg);
  if (s != QUAIL_OK) {
    delete t;
    return fail(s, "%s", msg.c_str());
  }
  if (group_of_label != nullptr) std::copy(gol.begin(), gol.end(), group_of_label);
  *out = t;
  return QUAIL_OK;
}

quail_status quail_shortlist_create(const quail_trie* trie, int32_t cut_depth, quail_shortlist** out) {
  if (out == nullptr || trie == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  quail_shortlist* sl = new quail_shortlist();
  std::string msg;
  const quail_status s = quail_build_shortlist_host(trie, cut_depth, sl, &msg);
  if (s != QUAIL_OK) {
    quail_trie_free(sl->prefix_trie);
    delete sl;
    return fail(s, "%s", msg.c_str());
  }
  *out = sl;
  return QUAIL_OK;
}

void quail_shortlist_free(quail_shortlist* sl) {
  if (sl == nullptr) return;
  int cur = -1;
  cudaGetDevice(&cur);
  for (auto& kv : sl->images) {
    if (kv.second.base == nullptr) continue;
    if (cudaSetDevice(kv.first) == cudaSuccess) cudaFree(kv.second.base);
  }
  if (cur >= 0 && !sl->images.empty()) cudaSetDevice(cur);
  quail_trie_free(sl->prefix_trie);
  delete sl;
}

int32_t quail_shortlist_groups(const quail_shortlist* sl, int32_t* group_of_label) {
  if (sl == nullptr) return 0;
  if (group_of_label != nullptr) std::copy(sl->group_of_label.begin(), sl->group_of_label.end(), group_of_label);
  return sl->num_groups;
}

size_t quail_workspace_size_shortlist(const quail_model_desc* model, const quail_trie* trie,
                                      const quail_shortlist* sl, int32_t beam, int32_t num_docs,
                                      int32_t max_doc_len) {
  if (model == nullptr || trie == nullptr || sl == nullptr || beam < 1 || num_docs < 0 || max_doc_len <= 0) return 0;
  if (!shortlist_matches(sl, trie)) return 0;
  if (model->n_kv_heads <= 0 || model->n_q_heads <= 0 || model->hidden <= 0 || model->vocab <= 0) return 0;
  return plan_shortlist(nullptr, model, sl, beam, num_docs, max_doc_len, nullptr);
}

quail_status quail_classify_trie_tree_shortlist(const quail_model_desc* model, const quail_paged_kv* kv,
                                                quail_trie* trie, quail_shortlist* sl, int32_t beam,
                                                int32_t num_docs, void* workspace, size_t workspace_bytes,
                                                float* label_logscore, float* label_prob, int32_t* label_argmax,
                                                int32_t* group_selected, quail_stream_t stream) {
  g_launches = 0;
  quail_status s = check_model(model);
  if (s != QUAIL_OK) return s;
  s = check_kv(kv, model);
  if (s != QUAIL_OK) return s;
  if (trie == nullptr || sl == nullptr) return fail(QUAIL_ERR_INVALID_ARG, "trie or shortlist is null");
  if (trie->vocab != model->vocab)
    return fail(QUAIL_ERR_INVALID_ARG, "trie vocab %d != model vocab %d", trie->vocab, model->vocab);
  if (!shortlist_matches(sl, trie)) return fail(QUAIL_ERR_INVALID_ARG, "the shortlist was made from another trie");
  if (beam < 1) return fail(QUAIL_ERR_INVALID_ARG, "beam must be >= 1");
  if (num_docs < 0) return fail(QUAIL_ERR_INVALID_ARG, "num_docs < 0");
  if (num_docs == 0) return QUAIL_OK;
  if (num_docs > 65535) return fail(QUAIL_ERR_UNSUPPORTED_SHAPE, "at most 65535 documents per call");
  if (label_logscore == nullptr || label_prob == nullptr || label_argmax == nullptr)
    return fail(QUAIL_ERR_INVALID_ARG, "an output pointer is null");
  const size_t need = plan_shortlist(nullptr, model, sl, beam, num_docs, kv->max_doc_len, nullptr);
  s = check_workspace(workspace, workspace_bytes, need);
  if (s != QUAIL_OK) return s;
  DeviceState* ds = nullptr;
  s = device_state(&ds);
  if (s != QUAIL_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const quail_trie::DeviceImage* img = nullptr;
  s = upload_trie(trie, st, &img);
  if (s != QUAIL_OK) return s;
  const quail_trie::DeviceImage* img1 = nullptr;
  s = upload_trie(sl->prefix_trie, st, &img1);
  if (s != QUAIL_OK) return s;
  const quail_shortlist::DeviceImage* simg = nullptr;
  s = upload_shortlist(sl, st, &simg);
  if (s != QUAIL_OK) return s;
  ShortlistBuffers x;
  plan_shortlist(static_cast<uint8_t*>(workspace), model, sl, beam, num_docs, kv->max_doc_len, &x);
  const ShortlistTables T{simg->row_off, simg->row_eval, simg->row_parent, simg->child_off, simg->child_row,
                          simg->child_tok, simg->lab_off, simg->lab_id, simg->term_off, simg->term_t,
                          simg->pref_t0, simg->pref_t1, sl->num_groups, sl->max_rows, sl->max_children};
  const int G = sl->num_groups, B = x.B, R = x.R;
  const int d = model->hidden;

  // prefix pass (every group's prefix, every document), selection, row layout
  stage_mark(QUAIL_STAGE_PROLOGUE, false, st);
  const int a1 = sl->prefix_trie->n_eval();
  if (sl->cut_depth == 1 && a1 == 1) {
    // One-token prefixes: S(p) = logit(p) - LSE with one LSE per document, so
    // the ranking is that of the G logits; the prefix pass is the root row and
    // the G prefix tokens' logits (the root's children, in group order).
    const NodeTables nt1{img1->eval_token, img1->eval_depth, img1->eval_parent, a1};
    const RowMap map1{a1, nullptr, nullptr, nullptr};
    s = run_prologue(model, nt1, x.b1, ds, st);
    if (s != QUAIL_OK) return s;
    s = run_attention(model, kv, nt1, map1, num_docs, x.b1, ds, st);
    if (s != QUAIL_OK) return s;
    s = run_wo_norm(model, nt1, map1, num_docs, x.b1, ds, st);
    if (s != QUAIL_OK) return s;
    CUDA_TRY(launch_restricted_logits(x.b1.z_f32, static_cast<const bf16*>(model->lm_head), img1->eval_child_tokens,
                                      G, num_docs, d, x.ls1, st));
  } else {
    s = trie_tree_pass(model, kv, sl->prefix_trie, img1, num_docs, x.b1, ds, st, x.ls1, x.prob1, x.am1, false);
    if (s != QUAIL_OK) return s;
  }
  CUDA_TRY(launch_shortlist_select(x.ls1, num_docs, G, B, x.sel, st));
  const Buffers& b = x.b2;
  int* row_token = b.small;
  int* row_depth = b.small + R;
  int* row_parent = b.small + 2 * static_cast<size_t>(R);
  int* padded_of = b.small + 3 * static_cast<size_t>(R);
  int* zeros = b.small + 4 * static_cast<size_t>(R);  // [2]
  int* count = zeros + 2;
  int* block_base = count + 1;
  int* doc_base = block_base + static_cast<size_t>(num_docs) * B;
  int* doc_rows = doc_base + num_docs;
  CUDA_TRY(cudaMemsetAsync(zeros, 0, 2 * sizeof(int), st));
  CUDA_TRY(launch_shortlist_scan(T, x.sel, num_docs, B, block_base, doc_base, doc_rows, count, st));
  CUDA_TRY(launch_shortlist_expand(T, x.sel, num_docs, B, x.Bq, R, block_base, doc_base, count, img->eval_token,
                                   img->eval_depth, row_token, row_depth, row_parent, padded_of, st));
  stage_mark(QUAIL_STAGE_PROLOGUE, true, st);

  // second pass over the kept groups' rows, numbered compactly document by
  // document (count real rows, then root copies up to the bound R): the
  // GEMMs skip the M tiles past count; the attention sees Bq padded rows per
  // document (row e of document i is node doc_base[i] + e, padding reads its
  // last row) and skips row tiles of padding only; its padded output rows are
  // gathered back into the compact order before W_o.
  const NodeTables nt{row_token, row_depth, row_parent, R};
  RowMap map{x.Bq, nullptr, nullptr, nullptr, nullptr, 0};
  map.slot_base = doc_base;
  map.slot_rows = doc_rows;
  const int hq = model->n_q_heads;
  stage_mark(QUAIL_STAGE_ATTENTION, false, st);
  s = run_prologue(model, nt, b, ds, st, count);
  if (s != QUAIL_OK) return s;
  s = run_attention(model, kv, nt, map, num_docs, b, ds, st, count);
  if (s != QUAIL_OK) return s;
  stage_mark(QUAIL_STAGE_ATTENTION, true, st);
  stage_mark(QUAIL_STAGE_WO_NORM, false, st);
  CUDA_TRY(launch_gather_rows(b.attn_out, padded_of, count, R, static_cast<size_t>(2) * hq * 128 * sizeof(bf16),
                              x.attn_c, st));
  {
    CUtensorMap tA;
    s = encode_2d_bf16(&tA, x.attn_c, round_up(R, 128), 2 * hq * 128, 2 * hq * 128, 64, 128);
    if (s != QUAIL_OK) return s;
    BSet bs{};
    s = encode_2d_bf16(&bs.map[0], model->w_o, d, hq * 128, hq * 128, 64, 256);
    if (s != QUAIL_OK) return s;
    bs.n_begin[0] = 0;
    bs.n_begin[1] = d;
    bs.count = 1;
    const size_t slab = static_cast<size_t>(R) * d;
    CUDA_TRY(launch_gemm_proj(tA, bs, R, d, hq * 128, b.gp.ks_wo, b.h_part, slab, d, ds->num_sms, ds->err, st,
                              count));
    const RowMap cmap{1, nullptr, nullptr, count, nullptr, 1};  // row r is node r; rows past count skipped
    CUDA_TRY(launch_final_norm(b.h_part, b.gp.ks_wo, slab, static_cast<const bf16*>(model->embed), nt.token, cmap, R,
                               d, static_cast<const bf16*>(model->final_norm), model->rms_eps, b.z, b.z_f32, st));
  }
  stage_mark(QUAIL_STAGE_WO_NORM, true, st);
  const int n_tiles = (model->vocab + kHeadBN - 1) / kHeadBN;
  stage_mark(QUAIL_STAGE_HEAD, false, st);
  {
    CUtensorMap tA, tB;
    s = encode_2d_bf16(&tA, b.z, round_up(R, 128), d, d, 64, 128);
    if (s != QUAIL_OK) return s;
    s = encode_2d_bf16(&tB, model->lm_head, model->vocab, d, d, 64, head_b_box_rows(R));
    if (s != QUAIL_OK) return s;
    // log-sum-exp partials only: one row per slot and an empty child list
    HeadEpilogueArgs ha{b.lse_part, reinterpret_cast<float*>(zeros), zeros, zeros, b.z_f32,
                        static_cast<const bf16*>(model->lm_head), d, 1, 0, n_tiles};
    CUDA_TRY(launch_gemm_head(tA, tB, R, model->vocab, d, ha, ds->num_sms, ds->err, st, count));
  }
  stage_mark(QUAIL_STAGE_HEAD, true, st);
  stage_mark(QUAIL_STAGE_SCORING, false, st);
  CUDA_TRY(launch_lse_reduce(b.lse_part, R, n_tiles, b.lse, st, count));
  CUDA_TRY(launch_shortlist_child_logprob(T, x.sel, num_docs, B, block_base, b.z_f32,
                                          static_cast<const bf16*>(model->lm_head), d, b.lse, x.clp, st));
  CUDA_TRY(launch_shortlist_label_score(T, x.sel, num_docs, B, trie->num_labels, x.clp, label_logscore, label_prob,
                                        label_argmax, st));
  stage_mark(QUAIL_STAGE_SCORING, true, st);
  if (group_selected != nullptr)
    CUDA_TRY(cudaMemcpyAsync(group_selected, x.sel, static_cast<size_t>(num_docs) * B * sizeof(int),
                             cudaMemcpyDeviceToDevice, st));
  return QUAIL_OK;
}

}  // extern "C"
