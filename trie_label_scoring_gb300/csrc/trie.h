// Library-owned label trie: host arrays (canonical CSR form exposed through
// quail_trie_view) plus the derived index arrays the kernels read, and one
// device image per CUDA device.
#pragma once
#include <cstdint>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "quail_internal.h"

struct quail_trie {
  int32_t num_labels = 0;
  int32_t vocab = 0;
  int32_t root_token = 0;
  int32_t max_depth = 0;
  int32_t has_prefix_labels = 0;

  // canonical node arrays (DFS preorder, children ascending by token)
  std::vector<int32_t> parent, depth, token, subtree_size, child_offsets, child_nodes, child_tokens;
  std::vector<uint8_t> is_branching;
  std::vector<int32_t> subtree_labels, node_label, unique_label;
  std::vector<int32_t> label_end_node, label_length, label_decide_depth;
  std::vector<int32_t> eval_nodes, eval_index_of_node, eval_child_offsets;

  // derived arrays for the kernels (trie_tree)
  std::vector<int32_t> eval_token, eval_depth, eval_parent, eval_child_tokens;
  std::vector<int32_t> label_term_offsets, label_term_eval, label_term_slot, label_prefix_eval;
  // derived arrays for trie_decode: internal nodes (nodes with children)
  std::vector<int32_t> int_nodes, int_index_of_node, int_token, int_depth, int_parent;

  int32_t n_nodes() const { return static_cast<int32_t>(parent.size()); }
  int32_t n_eval() const { return static_cast<int32_t>(eval_nodes.size()); }
  int32_t n_int() const { return static_cast<int32_t>(int_nodes.size()); }

  // Device image: one allocation per device holding every array above that a
  // kernel reads, at the offsets recorded in DeviceImage.
  struct DeviceImage {
    void* base = nullptr;
    size_t bytes = 0;
    const int32_t *eval_token, *eval_depth, *eval_parent, *eval_child_offsets, *eval_child_tokens;
    const int32_t *label_term_offsets, *label_term_eval, *label_term_slot, *label_prefix_eval;
    const int32_t *int_token, *int_depth, *int_parent, *int_index_of_node;
    const int32_t *child_offsets, *child_nodes, *child_tokens, *subtree_labels, *unique_label;
  };
  std::map<int, DeviceImage> images;
  std::mutex mu;
};

// Builds *t from the label lists; returns QUAIL_OK or an error status with the
// message in `msg`. Host only.
quail_status quail_build_trie_host(const int32_t* tokens, const int64_t* label_offsets, int32_t num_labels,
                                   int32_t root_token, int32_t vocab, const uint8_t* continuation, int32_t flags,
                                   quail_trie* t, std::string* msg);
