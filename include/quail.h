/*
 * quail.h -- C ABI of libquail: trie-constrained label scoring on one GB300.
 *
 * The operation (from "To Classify, Try a Trie Tree", sections 3.1-3.3, and the
 * Quail "Execution" page, section "Label scoring"): a document whose KV is
 * already cached is followed by the answer position (the ANSWER: token, the
 * trie root). The label token sequences form a prefix trie hanging off that
 * position. trie_tree scores every label in one request: each evaluated trie
 * node attends to the document KV and to its own trie ancestors only, the node
 * outputs go through W_o, RMSNorm and the vocabulary output head, and
 *     score(m) = prod_{k <= d_m} P(x_k | prompt, x_1..x_{k-1})          (sec. 3.2)
 *     P^(m)    = score(m) / sum_m' score(m')                            (sec. 3.2)
 * with the prefix-label correction score(m) *= (1 - P(continue | m)).  (sec. 3.2)
 * letters scores one answer position against M letter tokens and rescales
 * them to sum to 1 (sec. 3.3). trie_decode walks the trie greedily, running
 * the model only at branching nodes, and stops once one label is left
 * (sec. 3.1).
 *
 * Conventions for every call:
 *  - Every function returns a quail_status; no exception crosses the ABI.
 *    quail_last_error() gives a thread-local message for the last failure.
 *  - Argument errors are detected on the host before any launch. Index errors
 *    that only the device can see (page ids, doc lengths) set a per-device
 *    error word that quail_device_status() reads; kernels never trap.
 *  - Classify calls are asynchronous on the given stream (a cudaStream_t; NULL
 *    is the legacy default stream). The caller owns every device buffer passed
 *    in (weights, KV pool, outputs, workspace). The library owns quail_trie
 *    objects, including their device image.
 *  - All device pointers must be 16-byte aligned; bf16 tensors are row-major
 *    with the innermost dimension contiguous.
 */
#ifndef QUAIL_H_
#define QUAIL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* quail_stream_t; /* same type as cudaStream_t */
typedef struct CUevent_st* quail_event_t;   /* same type as cudaEvent_t  */

typedef enum {
  QUAIL_OK = 0,
  QUAIL_ERR_INVALID_ARG = -1,                /* null pointer, bad size, bad flag */
  QUAIL_ERR_EMPTY_LABEL = -2,                /* a label with zero tokens */
  QUAIL_ERR_DUPLICATE_LABEL = -3,            /* two labels (or letters) with the same tokens */
  QUAIL_ERR_TOKEN_RANGE = -4,                /* a token id outside [0, vocab) */
  QUAIL_ERR_PREFIX_LABEL_UNSUPPORTED = -5,   /* trie_decode on a set where one label prefixes another */
  QUAIL_ERR_WORKSPACE = -6,                  /* workspace null, misaligned or too small */
  QUAIL_ERR_CUDA = -7,                       /* a CUDA runtime/driver call failed */
  QUAIL_ERR_DEVICE_BOUNDS = -8,              /* device saw a page id / doc length out of range */
  QUAIL_ERR_DEVICE_TIMEOUT = -9,             /* a bounded device-side wait gave up */
  QUAIL_ERR_UNSUPPORTED_SHAPE = -10          /* a model shape these kernels do not handle */
} quail_status;

/* Thread-local, NUL-terminated description of the last non-OK status. */
const char* quail_last_error(void);

/* ------------------------------------------------------------------ trie
 * Label trie over token ids ("To Classify, Try a Trie Tree", sec. 3.1, Fig. 2;
 * sec. 3.2 for d_m and the evaluated positions).
 *
 * Canonical form (bit-exact and unique, so two builders agree): node 0 is the
 * root (token = root_token, depth 0); nodes are numbered in DFS preorder with
 * children visited in ascending token id, so the subtree of u is the id range
 * [u, u + subtree_size). Labels keep their input order 0..M-1.
 *
 * Decision depth d_m: k0 = the smallest k such that label m is the only label
 * with prefix x_1..x_k (a label that is a prefix of another never reaches 1,
 * so k0 = t_m for it); then d_m = the smallest k >= k0 with k = t_m or
 * x_{k+1} not a word-continuation token (sec. 3.2: score up to the end of the
 * word where the label branches away). With no bitmap every token starts a
 * word and d_m = k0. Flag QUAIL_TRIE_FULL_DEPTH sets d_m = t_m (the "simple
 * approach", full label probability, sec. 3.2).
 * Evaluated set P: the root plus the parent of every scored token
 * (x_k, k <= d_m), plus the end node of every prefix label, in ascending node
 * id. P is closed under ancestors.
 */
typedef struct quail_trie quail_trie;

enum { QUAIL_TRIE_FULL_DEPTH = 1, QUAIL_TRIE_ALL_NODES = 2 };

/*
 * tokens:        host, concatenated label token ids (label m = tokens[label_offsets[m] .. label_offsets[m+1]))
 * label_offsets: host, num_labels + 1 entries, non-decreasing, label_offsets[0] = 0
 * num_labels:    >= 2
 * root_token:    token id of the answer position (the ANSWER: token), in [0, vocab)
 * vocab:         vocabulary size V
 * word_continuation_bitmap: host, nullable; ceil(V/8) bytes, bit t (byte t>>3, bit t&7) set
 *                when token t continues the previous word instead of starting one
 * flags:         0, QUAIL_TRIE_FULL_DEPTH, and/or QUAIL_TRIE_ALL_NODES (every node
 *                is an evaluated position: the partner tries of quail_join_if)
 * out:           receives a library-owned trie; free with quail_trie_free
 * Errors: INVALID_ARG, EMPTY_LABEL, DUPLICATE_LABEL, TOKEN_RANGE. Host only; no GPU needed.
 */
quail_status quail_trie_build(const int32_t* tokens, const int64_t* label_offsets, int32_t num_labels,
                              int32_t root_token, int32_t vocab, const uint8_t* word_continuation_bitmap,
                              int32_t flags, quail_trie** out);

/* Read-only host view of a built trie. Pointers stay valid until quail_trie_free. */
typedef struct {
  int32_t n_nodes;        /* including the root */
  int32_t num_labels;     /* M */
  int32_t n_eval;         /* a = |P| */
  int32_t n_eval_children;/* sum over P of the child count */
  int32_t max_depth;      /* deepest node depth (= longest label) */
  int32_t has_prefix_labels; /* 1 if some label ends at a node with children */
  const int32_t* parent;          /* [n_nodes], -1 for the root */
  const int32_t* depth;           /* [n_nodes] */
  const int32_t* token;           /* [n_nodes], token[0] = root_token */
  const int32_t* subtree_size;    /* [n_nodes] */
  const int32_t* child_offsets;   /* [n_nodes + 1], CSR into child_nodes */
  const int32_t* child_nodes;     /* [n_nodes - 1], ascending token within a node */
  const int32_t* child_tokens;    /* [n_nodes - 1], token of child_nodes[j] */
  const uint8_t* is_branching;    /* [n_nodes], 1 if the node has more than one child */
  const int32_t* subtree_labels;  /* [n_nodes], labels ending in the subtree (node included) */
  const int32_t* node_label;      /* [n_nodes], label ending at the node, -1 if none */
  const int32_t* label_end_node;  /* [M] */
  const int32_t* label_length;    /* [M] t_m */
  const int32_t* label_decide_depth; /* [M] d_m */
  const int32_t* eval_nodes;      /* [n_eval], ascending node id */
  const int32_t* eval_index_of_node; /* [n_nodes], position in eval_nodes or -1 */
  const int32_t* eval_child_offsets; /* [n_eval + 1], children of eval node e occupy
                                        [eval_child_offsets[e], eval_child_offsets[e+1]) in the
                                        per-row child-logit arrays, in CSR child order */
} quail_trie_csr;

quail_status quail_trie_view(const quail_trie* trie, quail_trie_csr* out);
void quail_trie_free(quail_trie* trie);

/* Uploads the trie's device image to the current device (synchronously on
 * `stream`). Classify calls do this on first use; calling it ahead keeps the
 * allocation and copy out of a later call. */
quail_status quail_trie_upload(quail_trie* trie, quail_stream_t stream);

/* ------------------------------------------------------------------ model
 * One decoder layer's attention block plus the output head, as used at the
 * answer positions: x = E[tok]; x^ = RMSNorm(x)*in_norm; q,k,v = x^ W^T;
 * per-head RMSNorm on q and k; rotate-half RoPE at absolute position
 * (doc_len + depth); GQA attention (q head h uses KV head h / (Hq/Hkv));
 * h = x + O W_o^T; z = RMSNorm(h)*final_norm; logits = z lm_head^T.
 * All weights are device bf16, row-major [out_features, in_features]
 * (nn.Linear layout), caller-owned. head_dim must be 128, hidden a multiple
 * of 64, vocab >= 256.
 */
typedef struct {
  int32_t hidden;      /* d_model */
  int32_t n_q_heads;   /* H_q */
  int32_t n_kv_heads;  /* H_kv, divides H_q */
  int32_t head_dim;    /* 128 */
  int32_t vocab;       /* V */
  float rms_eps;       /* RMSNorm epsilon */
  float rope_theta;    /* RoPE base */
  const void* embed;      /* [V, hidden] */
  const void* w_q;        /* [H_q*128, hidden] */
  const void* w_k;        /* [H_kv*128, hidden] */
  const void* w_v;        /* [H_kv*128, hidden] */
  const void* q_norm;     /* [128] */
  const void* k_norm;     /* [128] */
  const void* w_o;        /* [hidden, H_q*128] */
  const void* in_norm;    /* [hidden] */
  const void* final_norm; /* [hidden] */
  const void* lm_head;    /* [V, hidden] */
} quail_model_desc;

/* Paged document KV ("a fixed pool of KV pages in HBM", Quail intro, sec. 3.2.3).
 * k_pool, v_pool: device bf16 [num_pages, n_kv_heads, page_size, 128]; keys are
 *                 already normalised and rotated at their absolute positions.
 * page_table:     device int32 [num_docs, max_pages]; entry (i, p) = physical page
 *                 holding tokens [16p, 16p+16) of document i.
 * doc_len:        device int32 [num_docs], 1 <= doc_len[i] <= max_doc_len.
 * max_doc_len:    host-side bound used to size the launch; a device doc_len
 *                 above it, or a page id outside [0, num_pages), sets
 *                 QUAIL_ERR_DEVICE_BOUNDS and that document's work is skipped. */
typedef struct {
  const void* k_pool;
  const void* v_pool;
  int32_t num_pages;
  int32_t page_size; /* must be 16 */
  const int32_t* page_table;
  int32_t max_pages;
  const int32_t* doc_len;
  int32_t max_doc_len;
} quail_paged_kv;

typedef enum { QUAIL_MODE_TRIE_TREE = 0, QUAIL_MODE_LETTERS = 1, QUAIL_MODE_TRIE_DECODE = 2, QUAIL_MODE_JOIN_IF = 3 } quail_mode;

/* Bytes of device workspace one classify call of `mode` needs (256-byte aligned
 * base required). trie may be NULL for QUAIL_MODE_LETTERS; num_letters is used
 * only by that mode. Returns 0 on invalid arguments. */
size_t quail_workspace_size(const quail_model_desc* model, const quail_trie* trie, int32_t num_letters,
                            int32_t num_docs, int32_t max_doc_len, quail_mode mode);

/* trie_tree ("To Classify, Try a Trie Tree", sec. 3.2; Quail "Execution",
 * "Label scoring"): all labels of all documents scored in one pass.
 * Outputs (device, caller-owned):
 *   label_logscore [num_docs, M] f32: log score(m), -inf for a prefix label whose
 *                  continuation probability reaches 1
 *   label_prob     [num_docs, M] f32: P^(m), sums to 1 per document
 *   label_argmax   [num_docs] i32:    argmax of P^, lowest label index on ties
 * Asynchronous on `stream`. */
quail_status quail_classify_trie_tree(const quail_model_desc* model, const quail_paged_kv* kv, quail_trie* trie,
                                      int32_t num_docs, void* workspace, size_t workspace_bytes,
                                      float* label_logscore, float* label_prob, int32_t* label_argmax,
                                      quail_stream_t stream);

/* letters (sec. 3.3): one answer position (root_token at position doc_len),
 * logits of the M letter rows only (V_out = M, sec. 4.1), renormalised.
 * letter_tokens: host, M distinct ids in [0, vocab), M >= 2.
 * Outputs (device): letter_logprob [num_docs, M] = log P^ (renormalised),
 * letter_prob [num_docs, M], letter_argmax [num_docs] (lowest index on ties). */
quail_status quail_classify_letters(const quail_model_desc* model, const quail_paged_kv* kv,
                                    const int32_t* letter_tokens, int32_t num_letters, int32_t root_token,
                                    int32_t num_docs, void* workspace, size_t workspace_bytes,
                                    float* letter_logprob, float* letter_prob, int32_t* letter_argmax,
                                    quail_stream_t stream);

/* One batched greedy trie_decode step (sec. 3.1): for every document whose
 * label is still undecided, run the model at its current branching node,
 * pick the most likely child (lowest token id on ties), follow forced
 * single-child chains, and stop once the subtree holds one label.
 *   node_cursor  [num_docs] i32 device, in/out; initialise to 0 (root)
 *   label_out    [num_docs] i32 device, in/out; initialise to -1; set once decided
 *   active_count i32 device scalar, out: documents still undecided after the step
 *   touched_nodes nullable u8 device [num_docs, n_nodes]; set to 1 at every node
 *                where this step computed logits (for tests)
 * Requires a trie with no prefix labels (else QUAIL_ERR_PREFIX_LABEL_UNSUPPORTED:
 * greedy decoding has no stop token, sec. 3.1 note 2). Call until active_count
 * reads 0; documents already decided cost no attention work. */
quail_status quail_classify_trie_decode_step(const quail_model_desc* model, const quail_paged_kv* kv,
                                             quail_trie* trie, int32_t num_docs, int32_t* node_cursor,
                                             int32_t* label_out, int32_t* active_count, uint8_t* touched_nodes,
                                             void* workspace, size_t workspace_bytes, quail_stream_t stream);

/* trie_tree for callers that cannot allocate device memory: an engine that has
 * already claimed nearly all of the GPU's memory for its own pools (a KV-cache
 * manager that reserves HBM at start-up), or a code path where cudaMalloc is
 * not allowed because it would synchronise the device in the middle of
 * latency-critical work. The pages this library follows have no counterpart of
 * this call; it exists for such integrations only.
 *
 * Same arguments, kernels and outputs as quail_classify_trie_tree, without the
 * workspace: the trie tables and every intermediate live in one fixed device
 * array of QUAIL_NOALLOC_SCRATCH_BYTES (64 MiB) that the library holds on every
 * GPU it is loaded on, until the process exits. The call allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library routine) and does not
 * need quail_trie_upload. If the call would need more scratch than the array
 * holds (about 230 documents of up to 1,024 tokens at the Qwen3-4B shape with
 * the 10-label trie), it returns QUAIL_ERR_WORKSPACE before launching anything.
 * Its first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. Every call shares the array: calls whose work overlaps on the GPU
 * (two streams, or two threads) race and corrupt each other's results, so
 * serialise them. The array keeps the previous call's contents; nothing in it
 * needs to start at zero. */
#define QUAIL_NOALLOC_SCRATCH_BYTES (64ull << 20)
quail_status quail_classify_trie_tree_noalloc(const quail_model_desc* model, const quail_paged_kv* kv,
                                              const quail_trie* trie, int32_t num_docs, float* label_logscore,
                                              float* label_prob, int32_t* label_argmax, quail_stream_t stream);

/* ------------------------------------------------------------ multi-layer
 * trie_tree through a whole decoder stack ("To Classify, Try a Trie Tree",
 * sec. 3.2 and 4.2: every answer position "goes through the whole LLM").
 * Per layer (Qwen3-style): x = RMSNorm(h) g_in; q, k, v projections; per-head
 * q/k RMSNorm; RoPE at l_i + depth; attention over the document's cached KV
 * of that layer and the node's own path (ancestors and itself) at that layer;
 * h += O W_o^T; h += W_down (SiLU(W_gate y) * W_up y), y = RMSNorm(h) g_post.
 * Then z = RMSNorm(h) g_f and the output head, LSE and label scoring as in
 * quail_classify_trie_tree. From layer 1 on a node's state depends on the
 * document, so the rows are (document, evaluated node) pairs; the path part
 * is computed per document. */
typedef struct {
  const void *w_q, *w_k, *w_v;      /* [H_q*128, d], [H_kv*128, d], [H_kv*128, d] */
  const void *q_norm, *k_norm;      /* [128] */
  const void *w_o;                  /* [d, H_q*128] */
  const void *in_norm, *post_norm;  /* [d] */
  const void *w_gate, *w_up;        /* [I, d] */
  const void *w_down;               /* [d, I] */
} quail_layer_weights;              /* device bf16, caller-owned */

typedef struct {
  int32_t hidden, n_q_heads, n_kv_heads, head_dim, vocab, intermediate, n_layers;
  float rms_eps, rope_theta;
  const void *embed, *final_norm, *lm_head;  /* device bf16 */
  const quail_layer_weights* layers;         /* host array [n_layers] */
} quail_model_ml_desc;

typedef struct {
  const void* const* k_pools;  /* host array [n_layers] of device pools [num_pages, n_kv_heads, 16, 128] */
  const void* const* v_pools;
  int32_t num_pages, page_size; /* page_size 16 */
  const int32_t* page_table;    /* device [N, max_pages], shared by the layers */
  int32_t max_pages;
  const int32_t* doc_len;       /* device [N] */
  int32_t max_doc_len;
} quail_paged_kv_ml;

/* Workspace bytes of quail_classify_trie_tree_ml; 0 on invalid arguments.
 * intermediate must be a multiple of 256 (SwiGLU width). */
size_t quail_workspace_size_ml(const quail_model_ml_desc* model, const quail_trie* trie, int32_t num_docs,
                               int32_t max_doc_len);
/* trie_tree through the whole decoder stack ("To Classify, Try a Trie
 * Tree", sec. 3.2 and 4.2: every evaluated answer position goes through every
 * layer and attends, at each layer, to the document and to its own path).
 * Each layer is Qwen3-style: h += W_o attn(q, k, v of RMSNorm(h) g_in, per-head
 * q/k RMSNorm, RoPE at doc_len + depth); h += W_down (SiLU(W_gate y) * W_up y),
 * y = RMSNorm(h) g_post. Then z = RMSNorm(h) final_norm and the output head
 * and label scoring as in quail_classify_trie_tree. kv holds every layer's
 * document K and V (one shared page table). Rows are (document, evaluated
 * node), so the workspace grows with num_docs x evaluated nodes. Outputs,
 * ownership and errors as quail_classify_trie_tree; n_layers must be in
 * [1, QUAIL_MAX_LAYERS]. */
quail_status quail_classify_trie_tree_ml(const quail_model_ml_desc* model, const quail_paged_kv_ml* kv,
                                         quail_trie* trie, int32_t num_docs, void* workspace, size_t workspace_bytes,
                                         float* label_logscore, float* label_prob, int32_t* label_argmax,
                                         quail_stream_t stream);

/* AI.IF over joined pairs ("Building an Ultra-High Throughput AI-SQL Engine",
 * sec. 3.2.4 "specialize attention for joins"; Quail docs "Execution",
 * Joins): every anchor document, whose KV is cached, is paired with every
 * partner. A partner is a token sequence that follows the anchor's prompt
 * (its text, the join question, the answer token) and attends to the anchor
 * and to its own earlier tokens only; partners share no tokens with one
 * another. The partners are the labels of a trie built with
 * QUAIL_TRIE_ALL_NODES, whose root token is the first token every partner
 * starts with; shared leading tokens (the join instructions) are one path.
 * The anchor KV is read once per KV head for all partners (as in
 * trie_tree); the partner-internal attention is computed once per call; the
 * two parts merge by log-sum-exp. At each partner's last token the output
 * head is restricted to the R answer spellings (sec. 3.2.4: "8 rows instead
 * of 151,936"): p_true = softmax over those R logits, summed over the first
 * n_true (the TRUE spellings).
 *   kv:          anchors' paged KV (doc = anchor)
 *   partners:    trie built with QUAIL_TRIE_ALL_NODES (else QUAIL_ERR_INVALID_ARG)
 *   answer_tokens: host, R = n_true + n_false distinct ids, TRUE spellings first,
 *                1 <= R <= 64
 *   p_true:      device [num_anchors, num_partners] fp32, row-major
 * Errors as quail_classify_trie_tree; QUAIL_ERR_DUPLICATE_LABEL for repeated
 * answer tokens. Workspace: quail_workspace_size(..., num_letters = R, ..., QUAIL_MODE_JOIN_IF). */
quail_status quail_join_if(const quail_model_desc* model, const quail_paged_kv* kv, quail_trie* partners,
                           int32_t num_anchors, const int32_t* answer_tokens, int32_t n_true, int32_t n_false,
                           void* workspace, size_t workspace_bytes, float* p_true, quail_stream_t stream);

/* ------------------------------------------------------------ huge label sets
 * Two ways to keep a very large label set cheap ("Trie Automata for
 * Constrained Decoding over Large Finite Sets", the extensions for
 * K > 50,000 labels):
 *  - hierarchical schema rewriting: the K labels split into G ~ sqrt(K)
 *    groups, each label spelled as its group's name followed by the label
 *    (no step then chooses among more than max(G, ceil(K / G)) tokens,
 *    smallest at G = ceil(sqrt K): Proposition 2);
 *  - a shortlist: a cheap score keeps the best candidates and exact trie
 *    scoring runs on those only.
 * Here the cheap score of the labels that share their first D tokens p is
 * the exact log-probability that the answer starts with p, sum over k <= D of
 * log P(p_k | context, p_1 .. p_{k-1}) (one trie_tree pass over the trie of
 * the distinct D-prefixes, to full depth). Each document keeps its B best
 * prefixes (ties: the lower prefix index, prefixes numbered in lexicographic
 * token order); its labels under them get their exact trie_tree log scores
 * ("To Classify, Try a Trie Tree", sec. 3.2), every other label -inf and
 * probability 0, and the probabilities are renormalised over the kept labels.
 * With B >= the number of prefixes the result is quail_classify_trie_tree's.
 * Hierarchical grouping is the case D = the group-name length. */

/* Trie of the grouped labels: the labels sorted by token sequence and cut
 * into num_groups contiguous runs whose sizes differ by at most one
 * (num_groups <= 0: ceil(sqrt(num_labels))); label m becomes
 * group_names[g * name_len .. + name_len) followed by label m (g its run).
 * Label indices are kept. group_names: host, num_groups * name_len ids, the
 * names distinct; group_of_label: host [num_labels] or NULL. Other arguments
 * and errors as quail_trie_build; QUAIL_ERR_DUPLICATE_LABEL for repeated
 * names. */
quail_status quail_trie_build_grouped(const int32_t* tokens, const int64_t* label_offsets, int32_t num_labels,
                                      int32_t root_token, int32_t vocab, const uint8_t* word_continuation_bitmap,
                                      int32_t flags, int32_t num_groups, const int32_t* group_names,
                                      int32_t name_len, quail_trie** out, int32_t* group_of_label);

/* Shortlist plan of `trie` at cut depth D >= 1 (host only): its groups (the
 * distinct D-prefixes, every label at least D tokens long, at least two
 * groups; else QUAIL_ERR_INVALID_ARG), the prefix trie and the per-group
 * tables of the second pass. Valid for that trie only; free it with
 * quail_shortlist_free before the trie. */
typedef struct quail_shortlist quail_shortlist;
quail_status quail_shortlist_create(const quail_trie* trie, int32_t cut_depth, quail_shortlist** out);
void quail_shortlist_free(quail_shortlist* sl);
/* Number of groups; group_of_label[m] for m < num_labels when the pointer is
 * not NULL (host). */
int32_t quail_shortlist_groups(const quail_shortlist* sl, int32_t* group_of_label);

/* Workspace bytes of quail_classify_trie_tree_shortlist; 0 on invalid
 * arguments. */
size_t quail_workspace_size_shortlist(const quail_model_desc* model, const quail_trie* trie,
                                      const quail_shortlist* sl, int32_t beam, int32_t num_docs,
                                      int32_t max_doc_len);
/* The shortlisted trie_tree: the prefix pass, each document's best
 * min(beam, groups) prefixes, then one pass over the rows of the kept groups
 * (document by document, padded to the largest group) and the kept labels'
 * scores.
 *   label_logscore, label_prob: device [num_docs, num_labels] fp32
 *   label_argmax:   device [num_docs] int32 (lowest index of the maximum)
 *   group_selected: device [num_docs, min(beam, groups)] int32, best first,
 *                   or NULL
 * Errors as quail_classify_trie_tree; QUAIL_ERR_INVALID_ARG when sl was made
 * from another trie or beam < 1. Stage events: 0 prefix pass + selection +
 * row layout, 1 second pass prologue + attention, 2 W_o + RMSNorm, 3 the
 * second pass's output-head GEMM alone, 4 log-sum-exp + child log-probs +
 * label scores. */
quail_status quail_classify_trie_tree_shortlist(const quail_model_desc* model, const quail_paged_kv* kv,
                                                quail_trie* trie, quail_shortlist* sl, int32_t beam,
                                                int32_t num_docs, void* workspace, size_t workspace_bytes,
                                                float* label_logscore, float* label_prob, int32_t* label_argmax,
                                                int32_t* group_selected, quail_stream_t stream);

/* ------------------------------------------------------------ cost model
 * Speed-of-light estimates of the three ways to classify and the choice
 * among them ("To Classify, Try a Trie Tree", sec. 4): for each method the
 * total tokens n_tok = L1 + N (q_pre + q_tail + a) and forward passes
 * K = ceil(n_tok / C) (sec. 4.1), the cached-KV tokens read R (prompt once;
 * trie_decode (b - 1) times), the attention bytes B_kv (W + R) with W = n_tok,
 * the output head F = 2 d V_out N a, B = 2 d V_out K, T_head = max(F/Pi, B/beta),
 * projections and MLP in the same roofline form over their weights, attention
 * as B_attn / beta, and T_classify = T_proj + T_attn + T_mlp + T_head.
 * Per method: trie_tree a = |P| and V_out = vocab; letters q_tail + 2M + 3
 * instruction tokens, a = 1, V_out = M (sec. 4.2); trie_decode b requests
 * (mean branching nodes per label path, sec. 4.3) over E[1 + depth of the
 * deciding node] tokens, V_out = vocab, not runnable when probabilities are
 * requested or a label prefixes another. The pick is the runnable method with
 * the lowest T_classify (sec. 4.4; ties in the order decode, tree, letters).
 * Host only; no device work. */
typedef enum {
  QUAIL_METHOD_TRIE_DECODE = 0,
  QUAIL_METHOD_TRIE_TREE = 1,
  QUAIL_METHOD_LETTERS = 2,
  QUAIL_NUM_METHODS = 3
} quail_method;

typedef struct {
  int32_t d_model, vocab;
  double proj_params;        /* q, k, v and output-projection weights summed over layers (elements) */
  double mlp_params;         /* MLP weights summed over layers (elements) */
  double kv_bytes_per_token; /* B_kv: one token's K and V over all layers (bytes) */
  double peak_flops;         /* Pi: bf16 FLOP/s, > 0 */
  double hbm_bytes_per_s;    /* beta: bytes/s, > 0 */
} quail_cost_model;

typedef struct {
  int32_t num_docs;           /* N >= 0 */
  double doc_tokens;          /* L1 = sum of the documents' token counts, >= 0 */
  int32_t q_pre;              /* preamble tokens per request, >= 0 */
  int32_t q_tail;             /* instruction tokens of the trie methods, >= 0 */
  int32_t max_pass_tokens;    /* C: tokens per forward pass, >= 1 */
  int32_t need_probabilities; /* 1: the query asks for label probabilities */
} quail_cost_workload;

typedef struct {
  int32_t runnable;                          /* 0: the other fields are zero */
  double q_tail, a, v_out, requests;         /* the method's shape */
  double n_tok, passes, kv_read_tokens, attn_bytes;
  double head_flops, head_bytes;
  double t_head, t_proj, t_attn, t_mlp, t_classify; /* seconds */
} quail_method_cost;

/* Fills costs[QUAIL_NUM_METHODS] (indexed by quail_method) for the labels of
 * `trie` and writes the chosen method to *best. QUAIL_ERR_INVALID_ARG on a
 * null pointer or a value outside the ranges above. */
quail_status quail_estimate_methods(const quail_cost_model* model, const quail_cost_workload* work,
                                    const quail_trie* trie, quail_method_cost* costs, int32_t* best);

/* Synchronises `stream`, then reads and clears the current device's error
 * word. Returns QUAIL_OK, QUAIL_ERR_DEVICE_BOUNDS or QUAIL_ERR_DEVICE_TIMEOUT
 * (the message names the first failing item), or QUAIL_ERR_CUDA. */
quail_status quail_device_status(quail_stream_t stream);

/* Number of kernels the last classify call made on this thread launched
 * (including calls that failed part-way: the launches made before the
 * failure). Host-side bookkeeping only; no device synchronisation. */
int32_t quail_launch_count(void);

/* Profiling hook: when events != NULL, each classify call records
 * events[2s] before and events[2s+1] after stage s on its stream, for
 * s < num_stages (stages: 0 node prologue, 1 attention, 2 W_o + RMSNorm,
 * 3 output-head GEMM alone, 4 log-sum-exp reduction + label scoring). NULL
 * entries are skipped; events == NULL switches the hook off. Process-wide.
 *
 * quail_classify_trie_tree_ml marks stage 0 around the whole layer stack and
 * in addition, for layer l, span j at stage QUAIL_NUM_STAGES +
 * l * QUAIL_LAYER_SPANS + j (spans: 0 residual + RMSNorm + q|k|v GEMM + q/k
 * norms, 1 attention, 2 W_o GEMM + residual + post-norm, 3 gate|up GEMM,
 * with SiLU(gate) * up fused into its epilogue when the projection
 * runs without a k-split, 4 SiLU(gate) * up when it runs as its own kernel,
 * 5 down GEMM alone); num_stages may then reach
 * QUAIL_NUM_STAGES + QUAIL_LAYER_SPANS * QUAIL_MAX_LAYERS. */
enum { QUAIL_STAGE_PROLOGUE = 0, QUAIL_STAGE_ATTENTION = 1, QUAIL_STAGE_WO_NORM = 2, QUAIL_STAGE_HEAD = 3,
       QUAIL_STAGE_SCORING = 4, QUAIL_NUM_STAGES = 5 };
enum { QUAIL_SPAN_QKV = 0, QUAIL_SPAN_ATTENTION = 1, QUAIL_SPAN_WO_NORM = 2, QUAIL_SPAN_GATE_UP = 3,
       QUAIL_SPAN_SILU_MUL = 4, QUAIL_SPAN_DOWN = 5, QUAIL_LAYER_SPANS = 6, QUAIL_MAX_LAYERS = 1024 };
quail_status quail_set_stage_events(quail_event_t* events, int32_t num_stages);

#ifdef __cplusplus
}
#endif
#endif /* QUAIL_H_ */
