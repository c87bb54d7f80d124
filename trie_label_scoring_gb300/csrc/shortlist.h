// Shortlist plan of a trie for huge label sets: the groups of labels that
// share their first D tokens, the trie of those prefixes (scored first, for
// every document), and per group the tables a document's second pass needs
// ("Trie Automata for Constrained Decoding over Large Finite Sets":
// hierarchical rewriting and a top-k shortlist ahead of exact scoring).
#pragma once
#include <cstdint>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "quail_internal.h"

struct quail_trie;

struct quail_shortlist {
  int32_t cut_depth = 0;
  int32_t num_groups = 0;
  int32_t num_labels = 0;
  int32_t trie_nodes = 0;  // of the trie the plan was made from (a consistency check)
  int32_t trie_eval = 0;
  int32_t max_rows = 0;      // most rows of any group
  int32_t max_children = 0;  // most child tokens of any group's rows
  quail_trie* prefix_trie = nullptr;  // owned; labels = the groups' prefixes, full depth

  std::vector<int32_t> group_of_label;
  // Group g's rows: the evaluated ancestors of its depth-D node (depth order),
  // then the evaluated nodes of its subtree (node order). Row entries hold the
  // trie's evaluated-node index and the row index of the parent (-1: root).
  std::vector<int32_t> row_off, row_eval, row_parent;
  // Group g's child tokens that its labels read (each term's scored child, and
  // every child of a prefix label's end row), row by row: [child_off[g], child_off[g+1]).
  std::vector<int32_t> child_off, child_row, child_tok;
  // Group g's labels (ascending label index); each label's terms as indices
  // into its group's child list (CSR term_off over all groups' labels in
  // order), and for a prefix label the child range [pref_t0, pref_t1) of its
  // end row (empty otherwise).
  std::vector<int32_t> lab_off, lab_id, term_off, term_t, pref_t0, pref_t1;

  struct DeviceImage {
    void* base = nullptr;
    const int32_t *row_off, *row_eval, *row_parent, *child_off, *child_row, *child_tok;
    const int32_t *lab_off, *lab_id, *term_off, *term_t, *pref_t0, *pref_t1;
  };
  std::map<int, DeviceImage> images;  // freed with the prefix trie by quail_shortlist_free
  std::mutex mu;
};

// Builds the plan of trie t at cut depth D (host only).
quail_status quail_build_shortlist_host(const quail_trie* t, int32_t D, quail_shortlist* sl, std::string* msg);

// Labels of K token lists sorted by their token sequences and cut into G
// contiguous runs whose sizes differ by at most one: group_of_label[m].
void quail_group_labels_host(const int32_t* tokens, const int64_t* label_offsets, int32_t K, int32_t G,
                             int32_t* group_of_label);
