// Host construction of the shortlist plan and of the hierarchical grouping
// ("Trie Automata for Constrained Decoding over Large Finite Sets", the
// extensions for K > 50,000: hierarchical schema rewriting into ~sqrt(K)
// balanced groups, and a top-k shortlist ahead of exact trie scoring).
//
// The groups of a trie at cut depth D are its depth-D nodes: in the canonical
// numbering (DFS preorder, children by ascending token) they come in
// lexicographic order of their D-token prefixes, and each group's subtree is
// one contiguous id range.
#include "shortlist.h"

#include <algorithm>
#include <numeric>

#include "trie.h"

void quail_group_labels_host(const int32_t* tokens, const int64_t* label_offsets, int32_t K, int32_t G,
                             int32_t* group_of_label) {
  std::vector<int32_t> order(K);
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return std::lexicographical_compare(tokens + label_offsets[a], tokens + label_offsets[a + 1],
                                        tokens + label_offsets[b], tokens + label_offsets[b + 1]);
  });
  // Run g holds the sorted positions j with floor(g K / G) <= j < floor((g+1) K / G),
  // i.e. g = ceil((j + 1) G / K) - 1.
  for (int64_t j = 0; j < K; ++j) {
    const int64_t g = ((j + 1) * G + K - 1) / K - 1;
    group_of_label[order[j]] = static_cast<int32_t>(g);
  }
}

quail_status quail_build_shortlist_host(const quail_trie* t, int32_t D, quail_shortlist* sl, std::string* msg) {
  const int32_t M = t->num_labels;
  if (D < 1) {
    *msg = "cut depth must be >= 1";
    return QUAIL_ERR_INVALID_ARG;
  }
  for (int32_t m = 0; m < M; ++m) {
    if (t->label_length[m] < D) {
      *msg = "label " + std::to_string(m) + " is shorter than the cut depth " + std::to_string(D);
      return QUAIL_ERR_INVALID_ARG;
    }
  }
  const int32_t n = t->n_nodes();
  // groups = depth-D nodes in node order
  std::vector<int32_t> group_of_node(n, -1), group_node;
  for (int32_t u = 0; u < n; ++u) {
    if (t->depth[u] == D) {
      group_of_node[u] = static_cast<int32_t>(group_node.size());
      group_node.push_back(u);
    }
  }
  const int32_t G = static_cast<int32_t>(group_node.size());
  if (G < 2) {
    *msg = "the cut depth leaves fewer than two groups";
    return QUAIL_ERR_INVALID_ARG;
  }
  sl->cut_depth = D;
  sl->num_groups = G;
  sl->num_labels = M;
  sl->trie_nodes = n;
  sl->trie_eval = t->n_eval();

  // each label's group: the depth-D ancestor of its end node
  sl->group_of_label.assign(M, -1);
  std::vector<std::vector<int32_t>> labels_of(G);
  for (int32_t m = 0; m < M; ++m) {
    int32_t u = t->label_end_node[m];
    while (t->depth[u] > D) u = t->parent[u];
    sl->group_of_label[m] = group_of_node[u];
    labels_of[group_of_node[u]].push_back(m);
  }

  // the prefix trie: one D-token label per group, scored to full depth
  {
    std::vector<int32_t> toks(static_cast<size_t>(G) * D);
    std::vector<int64_t> offs(G + 1);
    for (int32_t g = 0; g < G; ++g) {
      offs[g] = static_cast<int64_t>(g) * D;
      for (int32_t u = group_node[g]; u != 0; u = t->parent[u]) toks[static_cast<size_t>(g) * D + t->depth[u] - 1] = t->token[u];
    }
    offs[G] = static_cast<int64_t>(G) * D;
    sl->prefix_trie = new quail_trie();
    const quail_status s = quail_build_trie_host(toks.data(), offs.data(), G, t->root_token, t->vocab, nullptr,
                                                 QUAIL_TRIE_FULL_DEPTH, sl->prefix_trie, msg);
    if (s != QUAIL_OK) return s;
  }

  sl->row_off.assign(1, 0);
  sl->child_off.assign(1, 0);
  sl->lab_off.assign(1, 0);
  sl->term_off.assign(1, 0);
  sl->row_eval.clear();
  sl->row_parent.clear();
  sl->child_row.clear();
  sl->child_tok.clear();
  sl->lab_id.clear();
  sl->term_t.clear();
  sl->pref_t0.clear();
  sl->pref_t1.clear();
  sl->max_rows = 0;
  sl->max_children = 0;
  std::vector<int32_t> local(n, -1);  // node -> row of the group being built
  for (int32_t g = 0; g < G; ++g) {
    const int32_t c = group_node[g];
    std::vector<int32_t> nodes;
    for (int32_t u = t->parent[c]; u >= 0; u = t->parent[u])
      if (t->eval_index_of_node[u] >= 0) nodes.push_back(u);
    std::reverse(nodes.begin(), nodes.end());  // root first
    for (int32_t u = c; u < c + t->subtree_size[c]; ++u)
      if (t->eval_index_of_node[u] >= 0) nodes.push_back(u);
    const int32_t rows = static_cast<int32_t>(nodes.size());
    for (int32_t j = 0; j < rows; ++j) local[nodes[j]] = j;
    // every child of every row, numbered row by row ...
    std::vector<int32_t> full_base(rows + 1, 0);
    for (int32_t j = 0; j < rows; ++j) {
      const int32_t e = t->eval_index_of_node[nodes[j]];
      full_base[j + 1] = full_base[j] + (t->eval_child_offsets[e + 1] - t->eval_child_offsets[e]);
    }
    // ... of which the group keeps those its labels read: the scored child of
    // each term, and all children of a prefix label's end row
    std::vector<int32_t> keep(full_base[rows], -1);
    for (const int32_t m : labels_of[g]) {
      for (int32_t k = t->label_term_offsets[m]; k < t->label_term_offsets[m + 1]; ++k) {
        const int32_t e = t->label_term_eval[k];
        keep[full_base[local[t->eval_nodes[e]]] + (t->label_term_slot[k] - t->eval_child_offsets[e])] = 0;
      }
      const int32_t pe = t->label_prefix_eval[m];
      if (pe >= 0) {
        const int32_t j = local[t->eval_nodes[pe]];
        for (int32_t i = full_base[j]; i < full_base[j + 1]; ++i) keep[i] = 0;
      }
    }
    for (int32_t j = 0; j < rows; ++j) {
      const int32_t u = nodes[j];
      const int32_t e = t->eval_index_of_node[u];
      const int32_t p = t->parent[u];
      if (p >= 0 && local[p] < 0) {
        *msg = "evaluated set is not ancestor-closed";
        return QUAIL_ERR_INVALID_ARG;
      }
      sl->row_eval.push_back(e);
      sl->row_parent.push_back(p >= 0 ? local[p] : -1);
      for (int32_t i = full_base[j]; i < full_base[j + 1]; ++i) {
        if (keep[i] < 0) continue;
        keep[i] = static_cast<int32_t>(sl->child_tok.size()) - sl->child_off.back();  // index in the group's list
        sl->child_row.push_back(j);
        sl->child_tok.push_back(t->eval_child_tokens[t->eval_child_offsets[e] + (i - full_base[j])]);
      }
    }
    for (const int32_t m : labels_of[g]) {
      sl->lab_id.push_back(m);
      for (int32_t k = t->label_term_offsets[m]; k < t->label_term_offsets[m + 1]; ++k) {
        const int32_t e = t->label_term_eval[k];
        sl->term_t.push_back(keep[full_base[local[t->eval_nodes[e]]] + (t->label_term_slot[k] - t->eval_child_offsets[e])]);
      }
      sl->term_off.push_back(static_cast<int32_t>(sl->term_t.size()));
      const int32_t pe = t->label_prefix_eval[m];
      if (pe >= 0) {  // all of the end row's children are kept, in order
        const int32_t j = local[t->eval_nodes[pe]];
        sl->pref_t0.push_back(keep[full_base[j]]);
        sl->pref_t1.push_back(keep[full_base[j + 1] - 1] + 1);
      } else {
        sl->pref_t0.push_back(0);
        sl->pref_t1.push_back(0);
      }
    }
    for (const int32_t u : nodes) local[u] = -1;
    sl->row_off.push_back(static_cast<int32_t>(sl->row_eval.size()));
    sl->child_off.push_back(static_cast<int32_t>(sl->child_tok.size()));
    sl->lab_off.push_back(static_cast<int32_t>(sl->lab_id.size()));
    sl->max_rows = std::max(sl->max_rows, rows);
    sl->max_children = std::max(sl->max_children, sl->child_off[g + 1] - sl->child_off[g]);
  }
  return QUAIL_OK;
}
