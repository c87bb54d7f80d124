// Launch wrappers for the sm_103a kernels (one translation unit each group).
// All pointers are device pointers; every launch goes to `st` and returns the
// launch status (cudaGetLastError).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace quail {

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------ GEMM (gemm.cu)
// Tensor maps are built by the caller (encode_2d_bf16 in api.cu).
// Projection GEMM with a two-term bf16 split A = [X_hi | X_lo] ([M, 2K]) and up
// to three B tensors side by side along N (BSet, each [N_i, K], segment starts
// multiples of 256): partial tiles of k-split s go to C + s * slab
// ([M, ldc] fp32 each); the consumer sums the k_splits slabs.
struct BSet;
// m_live (optional): device count of the rows present (<= M); M tiles past it are skipped.
cudaError_t launch_gemm_proj(const CUtensorMap& tmA, const BSet& bset, int M, int N, int K, int k_splits, float* C,
                             size_t slab, int ldc, int num_sms, int* err, cudaStream_t st,
                             const int* m_live = nullptr);
// Fused SwiGLU input projection: A = split y [M, 2K]; bset in glu mode (map[0]
// = W_gate, map[1] = W_up, boxes of kProjBN/2 rows); writes
// act = split(SiLU(y W_gate^T) * (y W_up^T)) [round_up(M,128), 2I] bf16 directly
// (no k-split). I must be a multiple of 128.
cudaError_t launch_gemm_swiglu(const CUtensorMap& tmA, const BSet& bset, int M, int I, int K, bf16* act,
                               int num_sms, int* err, cudaStream_t st);
// k-splits that balance `tiles` work tiles of nk k-blocks over num_sms SMs.
int choose_k_splits(int tiles, int nk, int num_sms);

// Output head: for every row r < M and vocabulary tile j (256 tokens):
//   lse_part[r * n_tiles + j] = (max2, sum exp2(logit*log2e - max2)) over the tile,
// and for every child token c of row r's node that falls in the tile:
//   child_logit[(r / nq) * n_child + eval_child_offsets[e] + i] = z32[r] . lm_head[c]
// (fp32), with e = r % nq. Logits never leave the chip.
struct HeadEpilogueArgs {
  float2* lse_part;
  float* child_logit;
  const int* child_offsets;  // [nq + 1]
  const int* child_tokens;   // ascending within each node
  const float* z32;          // [M, d] unrounded hidden states
  const bf16* lm_head;       // [V, d]
  int d;
  int nq;
  int n_child;
  int n_tiles;
};
constexpr int kHeadBN = 256;
// The head runs on clusters of CTAs along M that share each 256-row band of
// W_lm: every CTA loads 1/C of the band (tmB's box: 64 columns x 256/C rows)
// and multicasts it to the others. The M tiles are scheduled in whole
// clusters, so a padding tile costs a full tile of MMAs. C = 4 when the rows
// span at most kHeadWideClusterMaxTiles 128-row tiles (A is small and B's L2
// reads dominate: four CTAs share each band) and clusters of four schedule no
// more tiles than pairs do (3, 4, 7 or 8 tiles); else C = 2 (A's re-reads
// dominate, and four CTAs in lockstep cost more than the B they share).
constexpr int kHeadWideClusterMaxTiles = 8;
int head_cluster_ctas(int M);
inline int head_b_box_rows(int M) { return kHeadBN / head_cluster_ctas(M); }
cudaError_t launch_gemm_head(const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int V, int K,
                             const HeadEpilogueArgs& args, int num_sms, int* err, cudaStream_t st,
                             const int* m_live = nullptr);

// ------------------------------------------------------------ layer kernels (layer.cu)
// y = RMSNorm(E[tokens[r]]) * gain as a two-term bf16 split:
// out[r, 0:d] = bf16(y), out[r, d:2d] = bf16(y - bf16(y)); rows = n
// live (optional): device count of the rows present; rows past it are skipped.
cudaError_t launch_embed_rmsnorm(const bf16* embed, const int* tokens, int n, int d, const bf16* gain, float eps,
                                 bf16* out, cudaStream_t st, const int* live = nullptr);
// qkv[r] = sum over the k_splits slabs of part (slab stride `slab`), then
// per-head RMSNorm of the q heads [0, hq) with gq and k heads [hq, hq + hkv)
// with gk; v heads copied. qkv and each slab are [rows, ld].
cudaError_t launch_qk_head_norm(const float* part, int k_splits, size_t slab, float* qkv, int rows, int ld, int hq,
                                int hkv, const bf16* gq, const bf16* gk, float eps, cudaStream_t st,
                                const int* live = nullptr);

// Maps an attention/output row to its trie node: slot = row / nq, e = row % nq,
// node = slot_node ? slot_node[slot] : e.
struct RowMap {
  int nq;
  const int* slot_node;   // nullable
  const int* slot_doc;    // nullable: slot -> document (identity when null)
  const int* n_slots_dev; // nullable: rows of slots >= *n_slots_dev are skipped
  const int* row_nodes;   // nullable: query row e of every slot -> node row (identity when null)
  int slot_stride;        // node rows of slot s start at s * slot_stride (0: shared by all slots)
  const int* slot_base;   // nullable: slot s's rows are nodes slot_base[s] + e for e < slot_rows[s]
  const int* slot_rows;   //   (rows past slot_rows[s] are padding: they read its last row and are skipped
                          //   where whole row tiles are padding)
};

// z = RMSNorm(sum_s h_part[s][r] + E[node_token[node(r)]]) * g_f over the
// k_splits slabs of h_part; writes bf16 (and fp32 if z_f32).
cudaError_t launch_final_norm(const float* h_part, int k_splits, size_t slab, const bf16* embed,
                              const int* node_token, RowMap map, int rows, int d, const bf16* gain, float eps,
                              bf16* z_bf16, float* z_f32, cudaStream_t st);
// lse[r] = log-sum-exp over the n_tiles partials of row r.
cudaError_t launch_lse_reduce(const float2* lse_part, int rows, int n_tiles, float* lse, cudaStream_t st,
                              const int* live = nullptr);

// Label path sums, prefix correction, softmax over labels and argmax, one block
// per document; the block first reduces its a rows' log-sum-exp from the
// head's tile partials (and stores them in lse).
struct LabelScoreArgs {
  const float* child_logit;  // [N, n_child]
  const float2* lse_part;    // [N * a, n_tiles]
  int n_tiles;
  float* lse;                // [N * a], written
  const int* term_offsets;   // [M + 1]
  const int* term_eval;
  const int* term_slot;
  const int* prefix_eval;    // [M]
  const int* eval_child_offsets;  // [a + 1]
  int a;
  int n_child;
  int M;
  float* logscore;  // [N, M]
  float* prob;      // [N, M]
  int* argmax;      // [N]
};
// One CTA per document when there are at least num_sms documents; else
// the LSE reduce, per-label scores and per-document softmax as three kernels
// spread over many CTAs.
cudaError_t launch_label_score(const LabelScoreArgs& args, int num_docs, int num_sms, cudaStream_t st);

// Multi-layer path (mlp.cu): the fp32 residual stream h [rows, d].
// h[r] = E[tokens[r]].
cudaError_t launch_gather_embed(const bf16* embed, const int* tokens, int rows, int d, float* h, cudaStream_t st);
// h += sum of ks slabs of part (ks may be 0); out (nullable) = split(RMSNorm(h) * gain) [rows, 2d].
cudaError_t launch_residual_norm(float* h, const float* part, int ks, size_t slab, int rows, int d, const bf16* gain,
                                 float eps, bf16* out, cudaStream_t st);
// act [rows, 2I] = split(SiLU(gate) * up) from ks slabs of [rows, 2I] (gate | up).
cudaError_t launch_silu_mul_split(const float* part, int ks, size_t slab, int rows, int I, bf16* act,
                                  cudaStream_t st);
// z = RMSNorm(h) * gain as bf16 [rows, d] and fp32 (nullable).
cudaError_t launch_norm_out(const float* h, int rows, int d, const bf16* gain, float eps, bf16* z, float* z_f32,
                            cudaStream_t st);

// AI.IF on joined pairs: for every row of z_f32 [rows, d] (anchor * M +
// partner), the softmax over the R answer-spelling rows of W_lm (tokens[0,
// n_true) spell TRUE) and p_true[row] = the TRUE rows' share.
constexpr int kJoinMaxRows = 64;
cudaError_t launch_join_head(const float* z, const bf16* lm_head, const int* tokens, int n_true, int R, int rows,
                             int M, int d, float* p_true, cudaStream_t st);

// logits[doc * M + m] = z_f32[doc] . W_lm[tokens[m]] in fp32 (d a multiple of 8).
cudaError_t launch_restricted_logits(const float* z, const bf16* lm_head, const int* tokens, int M, int num_docs,
                                     int d, float* logits, cudaStream_t st);
// letters: logits of the M letter rows from z_f32 [N, d], renormalised softmax, argmax.
cudaError_t launch_letters_head(const float* z, const bf16* lm_head, const int* letter_tokens, int M, int num_docs,
                                int d, float* logprob, float* prob, int* argmax, cudaStream_t st);

// trie_decode bookkeeping.
struct DecodeTrie {
  const int* child_offsets;
  const int* child_nodes;
  const int* child_tokens;
  const int* subtree_labels;
  const int* unique_label;
  const int* int_index_of_node;
  int n_nodes;
};
// Normalises every undecided document's cursor (forced chains, decided
// subtrees) and compacts the still-undecided ones into slots.
cudaError_t launch_decode_prepare(DecodeTrie t, int num_docs, int* node_cursor, int* label_out, int* slot_doc,
                                  int* slot_node, int* n_slots, int* active_count, cudaStream_t st);
// Picks the most likely child for every active slot and advances.
cudaError_t launch_decode_select(DecodeTrie t, const float* z, const bf16* lm_head, int d, int num_docs,
                                 const int* slot_doc, const int* n_slots, int* node_cursor, int* label_out,
                                 int* active_count, uint8_t* touched, cudaStream_t st);

// ------------------------------------------------------------ attention (attention.cu)
// ------------------------------------------------------------ shortlist (shortlist.cu)
// Device view of a shortlist plan (see shortlist.h for the table layout).
struct ShortlistTables {
  const int *row_off, *row_eval, *row_parent, *child_off, *child_row, *child_tok;
  const int *lab_off, *lab_id, *term_off, *term_t, *pref_t0, *pref_t1;
  int num_groups;
  int max_rows;      // rows per (document, kept group) block
  int max_children;  // child log-prob slots per block
};
// sel[doc * B + b]: the B groups of highest prefix log score (ties: lower group).
cudaError_t launch_shortlist_select(const float* prefix_logscore, int num_docs, int G, int B, int* sel,
                                    cudaStream_t st);
// Node tables of the second pass in that compact numbering (rows count..R-1
// are root copies with no parent), and padded_of[c] = doc * Bq + the row's
// index within its document (the attention's padded output row).
cudaError_t launch_shortlist_expand(const ShortlistTables& T, const int* sel, int num_docs, int B, int Bq, int R,
                                    const int* block_base, const int* doc_base, const int* count,
                                    const int* eval_token, const int* eval_depth, int* row_token, int* row_depth,
                                    int* row_parent, int* padded_of, cudaStream_t st);
// The kept groups' rows numbered compactly, document by document and group by
// group: block_base[doc * B + b] (first row of that group's block), count,
// doc_base / doc_rows (each document's first row and row count).
cudaError_t launch_shortlist_scan(const ShortlistTables& T, const int* sel, int num_docs, int B, int* block_base,
                                  int* doc_base, int* doc_rows, int* count, cudaStream_t st);
// dst[c] = src[padded_of[c]] for c < *count (rows of row_bytes, a multiple of 16).
cudaError_t launch_gather_rows(const void* src, const int* padded_of, const int* count, int max_rows,
                               size_t row_bytes, void* dst, cudaStream_t st);
// clp[blk * max_children + t] = z32[row] . W_lm[tok] - lse[row] (fp32) for
// every child t of the block's group; row = block_base[blk] + the child's row.
cudaError_t launch_shortlist_child_logprob(const ShortlistTables& T, const int* sel, int num_docs, int B,
                                           const int* block_base, const float* z32, const bf16* lm_head, int d,
                                           const float* lse, float* clp, cudaStream_t st);
// Label scores of the kept groups' labels (-inf / 0 elsewhere), softmax over
// the kept labels, argmax (lowest label index of the maximum).
cudaError_t launch_shortlist_label_score(const ShortlistTables& T, const int* sel, int num_docs, int B, int M,
                                         const float* clp, float* logscore, float* prob, int* argmax,
                                         cudaStream_t st);

struct AttnArgs {
  // paged document KV
  int num_pages, max_pages, max_doc_len;
  const int* page_table;
  const int* doc_len;
  // layer
  int hq, hkv;
  float theta;
  // query nodes (rows of qkv: normalised, not rotated q | k | v in fp32)
  const float* qkv;
  int ldq;
  const int* node_depth;
  const int* node_parent;  // tree part
  int n_nodes;             // rows of qkv
  const int* nodes_live;   // nullable: device count of the nodes present (tree part skips the rest)
  RowMap map;
  int n_slots;             // host bound on slots (documents)
  // split-KV decomposition
  int split_tokens;
  int n_splits;
  int rows_pad;            // rows per (slot, kv head), padded to the row tile
  int row_tile;            // 16 (mma.sync kernel: one tile shared by its 4 warps) or 128 (tcgen05 kernel)
  float* part_o;           // [n_slots, hkv, n_splits, rows_pad, 128]
  float2* part_ml;         // [n_slots, hkv, n_splits, rows_pad]
  float* tree_o;           // [n_nodes, hq, 128]
  float2* tree_ml;         // [n_nodes, hq]
  bf16* out;               // [n_slots * nq, 2 * hq * 128]: O as a two-term bf16 split [O_hi | O_lo]
  int* err;
  int* slot_order;         // nullable: [n_slots] the mma.sync doc attention's slot order (longest document first)
};
cudaError_t launch_tree_part(const AttnArgs& a, cudaStream_t st);
// slot_order = the slots sorted by document length, longest first (slots past
// *map.n_slots_dev last), so the doc attention's long CTAs start in the first
// waves and the last wave holds short ones.
cudaError_t launch_slot_order(const AttnArgs& a, cudaStream_t st);
// True when the mma.sync doc attention's grid spans more than one and at
// most 1.5 waves of resident CTAs: there it runs its slots in slot_order.
bool attn_doc_wants_slot_order(const AttnArgs& a, int num_sms);
cudaError_t launch_attn_doc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV, cudaStream_t st);
cudaError_t launch_attn_combine(const AttnArgs& a, cudaStream_t st);
// tcgen05 doc attention for 128-row query tiles (attention_tc.cu); row_tile must be 128.
cudaError_t launch_attn_doc_tc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV, cudaStream_t st);

// Test hooks: set the pipeline wait limit (cycles) of the GEMM, mma.sync
// attention and tcgen05 attention translation units.
cudaError_t set_pipeline_wait_limit_gemm(long long cycles);
cudaError_t set_pipeline_wait_limit_attention(long long cycles);
cudaError_t set_pipeline_wait_limit_attention_tc(long long cycles);

}  // namespace quail
