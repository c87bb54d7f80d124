// Host-side label trie construction ("To Classify, Try a Trie Tree", sec. 3.1
// Figure 2; sec. 3.2 for the decision depth d_m and the evaluated positions).
//
// Construction: sort the labels lexicographically by token sequence, then scan
// them in that order keeping the path of the previous label. A label creates
// nodes only past its longest common prefix with the previous label. Nodes are
// thereby created in lexicographic order of their prefixes, which is DFS
// preorder with children in ascending token id: the canonical numbering, in
// which the subtree of u is the id range [u, u + subtree_size[u]).
#include "trie.h"

#include <algorithm>
#include <cstring>
#include <numeric>

namespace {

bool continues_word(const uint8_t* bitmap, int32_t tok) {
  return bitmap != nullptr && ((bitmap[tok >> 3] >> (tok & 7)) & 1) != 0;
}

}  // namespace

quail_status quail_build_trie_host(const int32_t* tokens, const int64_t* label_offsets, int32_t num_labels,
                                   int32_t root_token, int32_t vocab, const uint8_t* continuation, int32_t flags,
                                   quail_trie* t, std::string* msg) {
  if (tokens == nullptr || label_offsets == nullptr || t == nullptr) {
    *msg = "null argument";
    return QUAIL_ERR_INVALID_ARG;
  }
  if (num_labels < 2) {
    *msg = "need at least 2 labels";
    return QUAIL_ERR_INVALID_ARG;
  }
  if (vocab <= 0 || (flags & ~(QUAIL_TRIE_FULL_DEPTH | QUAIL_TRIE_ALL_NODES)) != 0) {
    *msg = "bad vocab or flags";
    return QUAIL_ERR_INVALID_ARG;
  }
  if (root_token < 0 || root_token >= vocab) {
    *msg = "root token " + std::to_string(root_token) + " outside [0, vocab)";
    return QUAIL_ERR_TOKEN_RANGE;
  }
  if (label_offsets[0] != 0) {
    *msg = "label_offsets[0] must be 0";
    return QUAIL_ERR_INVALID_ARG;
  }
  const int32_t M = num_labels;
  for (int32_t m = 0; m < M; ++m) {
    const int64_t lo = label_offsets[m], hi = label_offsets[m + 1];
    if (hi < lo) {
      *msg = "label_offsets decrease at label " + std::to_string(m);
      return QUAIL_ERR_INVALID_ARG;
    }
    if (hi == lo) {
      *msg = "label " + std::to_string(m) + " is empty";
      return QUAIL_ERR_EMPTY_LABEL;
    }
    if (hi - lo > (1 << 20)) {
      *msg = "label " + std::to_string(m) + " is too long";
      return QUAIL_ERR_INVALID_ARG;
    }
    for (int64_t j = lo; j < hi; ++j) {
      if (tokens[j] < 0 || tokens[j] >= vocab) {
        *msg = "label " + std::to_string(m) + " has token " + std::to_string(tokens[j]) + " outside [0, vocab)";
        return QUAIL_ERR_TOKEN_RANGE;
      }
    }
  }
  auto seq_begin = [&](int32_t m) { return tokens + label_offsets[m]; };
  auto seq_len = [&](int32_t m) { return static_cast<int32_t>(label_offsets[m + 1] - label_offsets[m]); };

  std::vector<int32_t> order(M);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return std::lexicographical_compare(seq_begin(a), seq_begin(a) + seq_len(a), seq_begin(b),
                                        seq_begin(b) + seq_len(b));
  });
  for (int32_t i = 1; i < M; ++i) {
    const int32_t a = order[i - 1], b = order[i];
    if (seq_len(a) == seq_len(b) && std::equal(seq_begin(a), seq_begin(a) + seq_len(a), seq_begin(b))) {
      *msg = "labels " + std::to_string(std::min(a, b)) + " and " + std::to_string(std::max(a, b)) +
             " have the same tokens";
      return QUAIL_ERR_DUPLICATE_LABEL;
    }
  }

  // ---- nodes in creation (= canonical) order
  t->num_labels = M;
  t->vocab = vocab;
  t->root_token = root_token;
  t->parent.assign(1, -1);
  t->depth.assign(1, 0);
  t->token.assign(1, root_token);
  t->label_end_node.assign(M, 0);
  t->label_length.assign(M, 0);
  std::vector<int32_t> path(1, 0);  // node id at each depth of the previous label
  int32_t prev = -1;
  for (int32_t i = 0; i < M; ++i) {
    const int32_t m = order[i];
    const int32_t L = seq_len(m);
    const int32_t* s = seq_begin(m);
    int32_t lcp = 0;
    if (prev >= 0) {
      const int32_t* ps = seq_begin(prev);
      const int32_t pl = seq_len(prev);
      while (lcp < L && lcp < pl && ps[lcp] == s[lcp]) ++lcp;
    }
    path.resize(lcp + 1);
    for (int32_t k = lcp; k < L; ++k) {
      const int32_t id = static_cast<int32_t>(t->parent.size());
      t->parent.push_back(path[k]);
      t->depth.push_back(k + 1);
      t->token.push_back(s[k]);
      path.push_back(id);
    }
    t->label_end_node[m] = path[L];
    t->label_length[m] = L;
    prev = m;
  }
  const int32_t n = t->n_nodes();

  // ---- CSR children (creation order = ascending token within a parent)
  t->child_offsets.assign(n + 1, 0);
  for (int32_t u = 1; u < n; ++u) t->child_offsets[t->parent[u] + 1]++;
  for (int32_t u = 0; u < n; ++u) t->child_offsets[u + 1] += t->child_offsets[u];
  t->child_nodes.assign(n - 1, 0);
  t->child_tokens.assign(n - 1, 0);
  std::vector<int32_t> fill(t->child_offsets.begin(), t->child_offsets.end() - 1);
  std::vector<int32_t> child_pos(n, 0);  // position of u within its parent's child list
  for (int32_t u = 1; u < n; ++u) {
    const int32_t p = t->parent[u];
    child_pos[u] = fill[p] - t->child_offsets[p];
    t->child_nodes[fill[p]] = u;
    t->child_tokens[fill[p]] = t->token[u];
    fill[p]++;
  }
  t->is_branching.assign(n, 0);
  for (int32_t u = 0; u < n; ++u) t->is_branching[u] = (t->child_offsets[u + 1] - t->child_offsets[u] > 1) ? 1 : 0;

  // ---- subtree sizes and label counts (children have larger ids than parents)
  t->subtree_size.assign(n, 1);
  t->subtree_labels.assign(n, 0);
  t->node_label.assign(n, -1);
  for (int32_t m = 0; m < M; ++m) {
    t->subtree_labels[t->label_end_node[m]] += 1;
    t->node_label[t->label_end_node[m]] = m;
  }
  for (int32_t u = n - 1; u >= 1; --u) {
    t->subtree_size[t->parent[u]] += t->subtree_size[u];
    t->subtree_labels[t->parent[u]] += t->subtree_labels[u];
  }
  t->unique_label.assign(n, -1);
  for (int32_t m = 0; m < M; ++m) {
    for (int32_t u = t->label_end_node[m]; u >= 0 && t->subtree_labels[u] == 1; u = t->parent[u])
      t->unique_label[u] = m;
  }
  t->max_depth = *std::max_element(t->depth.begin(), t->depth.end());

  // ---- decision depth d_m and the evaluated set P
  t->label_decide_depth.assign(M, 0);
  std::vector<uint8_t> in_eval(n, 0);
  in_eval[0] = 1;
  t->has_prefix_labels = 0;
  std::vector<std::vector<int32_t>> label_paths(M);
  for (int32_t m = 0; m < M; ++m) {
    std::vector<int32_t>& p = label_paths[m];
    const int32_t L = t->label_length[m];
    p.assign(L + 1, 0);
    for (int32_t u = t->label_end_node[m], k = L; k >= 0; u = t->parent[u], --k) p[k] = u;
    int32_t d = L;
    if (!(flags & QUAIL_TRIE_FULL_DEPTH)) {
      int32_t k0 = L;
      for (int32_t k = 1; k <= L; ++k) {
        if (t->subtree_labels[p[k]] == 1) {
          k0 = k;
          break;
        }
      }
      d = k0;
      const int32_t* s = seq_begin(m);
      while (d < L && continues_word(continuation, s[d])) ++d;  // s[d] is token x_{d+1}
    }
    t->label_decide_depth[m] = d;
    for (int32_t k = 1; k <= d; ++k) in_eval[p[k - 1]] = 1;
    const int32_t end = p[L];
    if (t->child_offsets[end + 1] > t->child_offsets[end]) {
      t->has_prefix_labels = 1;
      in_eval[end] = 1;
    }
  }
  if (flags & QUAIL_TRIE_ALL_NODES) std::fill(in_eval.begin(), in_eval.end(), 1);  // every node evaluated
  t->eval_nodes.clear();
  t->eval_index_of_node.assign(n, -1);
  for (int32_t u = 0; u < n; ++u) {
    if (in_eval[u]) {
      t->eval_index_of_node[u] = static_cast<int32_t>(t->eval_nodes.size());
      t->eval_nodes.push_back(u);
    }
  }
  const int32_t a = t->n_eval();
  t->eval_child_offsets.assign(a + 1, 0);
  t->eval_token.resize(a);
  t->eval_depth.resize(a);
  t->eval_parent.resize(a);
  t->eval_child_tokens.clear();
  for (int32_t e = 0; e < a; ++e) {
    const int32_t u = t->eval_nodes[e];
    t->eval_token[e] = t->token[u];
    t->eval_depth[e] = t->depth[u];
    t->eval_parent[e] = u == 0 ? -1 : t->eval_index_of_node[t->parent[u]];
    for (int32_t j = t->child_offsets[u]; j < t->child_offsets[u + 1]; ++j)
      t->eval_child_tokens.push_back(t->child_tokens[j]);
    t->eval_child_offsets[e + 1] = static_cast<int32_t>(t->eval_child_tokens.size());
  }

  // ---- per-label (evaluated row, child slot) terms of the path sum
  t->label_term_offsets.assign(M + 1, 0);
  t->label_term_eval.clear();
  t->label_term_slot.clear();
  t->label_prefix_eval.assign(M, -1);
  for (int32_t m = 0; m < M; ++m) {
    const std::vector<int32_t>& p = label_paths[m];
    for (int32_t k = 1; k <= t->label_decide_depth[m]; ++k) {
      const int32_t e = t->eval_index_of_node[p[k - 1]];
      t->label_term_eval.push_back(e);
      t->label_term_slot.push_back(t->eval_child_offsets[e] + child_pos[p[k]]);
    }
    t->label_term_offsets[m + 1] = static_cast<int32_t>(t->label_term_eval.size());
    const int32_t end = p[t->label_length[m]];
    if (t->child_offsets[end + 1] > t->child_offsets[end]) t->label_prefix_eval[m] = t->eval_index_of_node[end];
  }

  // ---- internal nodes (with children), for trie_decode
  t->int_nodes.clear();
  t->int_index_of_node.assign(n, -1);
  for (int32_t u = 0; u < n; ++u) {
    if (t->child_offsets[u + 1] > t->child_offsets[u]) {
      t->int_index_of_node[u] = static_cast<int32_t>(t->int_nodes.size());
      t->int_nodes.push_back(u);
    }
  }
  const int32_t ni = t->n_int();
  t->int_token.resize(ni);
  t->int_depth.resize(ni);
  t->int_parent.resize(ni);
  for (int32_t i = 0; i < ni; ++i) {
    const int32_t u = t->int_nodes[i];
    t->int_token[i] = t->token[u];
    t->int_depth[i] = t->depth[u];
    t->int_parent[i] = u == 0 ? -1 : t->int_index_of_node[t->parent[u]];
  }
  return QUAIL_OK;
}
