"""Label trie, decision depth d_m and evaluated positions -- oracle (test infrastructure).

"To Classify, Try a Trie Tree", sec. 3.1 (Figure 2): the labels form a
prefix tree over token ids whose root is the ANSWER: token; labels that start
with the same tokens share the start of their path. sec. 3.2: each label is
scored up to the end of the word where it branches away from every other
label (its last scored position is d_m), and the model runs only at the
positions whose next token is scored (4 positions in the running example).

Canonical numbering (the pages are silent; this reading makes the trie unique,
as a minimal DFA is): root = node 0; DFS preorder; children in ascending
token id. Labels keep their input order.

Pinned by: the running example's counts (18 nodes, 3 branching nodes, 8 nodes
with children, 4 evaluated positions, b = 1.5; sec. 3.1, 3.2, 4.3) and brute
force on tiny label sets (the nodes are exactly the distinct label prefixes).
"""
from __future__ import annotations

import numpy as np


class TrieError(ValueError):
    """kind is one of: invalid_arg, empty_label, duplicate_label, token_range."""

    def __init__(self, kind: str, msg: str):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind


def _is_continuation(bitmap, t: int) -> bool:
    if bitmap is None:
        return False
    return bool((int(bitmap[t >> 3]) >> (t & 7)) & 1)


def build_trie(labels, root_token: int, vocab: int, continuation=None, full_depth: bool = False,
               all_nodes: bool = False) -> dict:
    """Builds the trie of `labels` (lists of token ids) and its derived sets.

    Returns a dict of numpy arrays named like the fields of the library's
    trie view: parent, depth, token, subtree_size, child_offsets, child_nodes,
    child_tokens, is_branching, subtree_labels, node_label, label_end_node,
    label_length, label_decide_depth, eval_nodes, eval_index_of_node,
    eval_child_offsets, plus scalars n_nodes, num_labels, n_eval,
    n_eval_children, max_depth, has_prefix_labels.
    """
    M = len(labels)
    if M < 2:
        raise TrieError("invalid_arg", "need at least 2 labels")
    if vocab <= 0 or not (0 <= root_token < vocab):
        raise TrieError("token_range" if vocab > 0 else "invalid_arg", "root token out of range")
    seqs = [tuple(int(t) for t in lab) for lab in labels]
    for m, s in enumerate(seqs):
        if len(s) == 0:
            raise TrieError("empty_label", f"label {m} is empty")
        for t in s:
            if not (0 <= t < vocab):
                raise TrieError("token_range", f"label {m} has token {t}")
    seen = {}
    for m, s in enumerate(seqs):
        if s in seen:
            raise TrieError("duplicate_label", f"labels {seen[s]} and {m}")
        seen[s] = m

    # Nested dictionaries: one dict per node, keyed by child token.
    root: dict = {}
    for s in seqs:
        node = root
        for t in s:
            node = node.setdefault(t, {})

    # Number the nodes: DFS preorder, children by ascending token.
    prefixes: list = []

    def visit(prefix: tuple, node: dict) -> None:
        prefixes.append(prefix)
        for t in sorted(node):
            visit(prefix + (t,), node[t])

    visit((), root)
    n = len(prefixes)
    node_id = {p: i for i, p in enumerate(prefixes)}

    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int32)
    token = np.zeros(n, dtype=np.int32)
    token[0] = root_token
    children: list = [[] for _ in range(n)]
    for i, p in enumerate(prefixes):
        depth[i] = len(p)
        if p:
            token[i] = p[-1]
            parent[i] = node_id[p[:-1]]
            children[parent[i]].append(i)
    for c in children:  # already ascending by token because of the visit order
        assert all(token[c[j]] < token[c[j + 1]] for j in range(len(c) - 1))

    subtree_size = np.ones(n, dtype=np.int32)
    for i in range(n - 1, 0, -1):
        subtree_size[parent[i]] += subtree_size[i]

    child_offsets = np.zeros(n + 1, dtype=np.int32)
    child_offsets[1:] = np.cumsum([len(c) for c in children])
    child_nodes = np.array([j for c in children for j in c], dtype=np.int32)
    child_tokens = token[child_nodes] if len(child_nodes) else np.zeros(0, dtype=np.int32)
    is_branching = np.array([1 if len(c) > 1 else 0 for c in children], dtype=np.uint8)

    # How many labels have each prefix (a label counts for its own sequence too).
    prefix_count: dict = {}
    for s in seqs:
        for k in range(0, len(s) + 1):
            prefix_count[s[:k]] = prefix_count.get(s[:k], 0) + 1
    subtree_labels = np.array([prefix_count[p] for p in prefixes], dtype=np.int32)
    node_label = np.full(n, -1, dtype=np.int32)
    label_end_node = np.zeros(M, dtype=np.int32)
    label_length = np.zeros(M, dtype=np.int32)
    for m, s in enumerate(seqs):
        e = node_id[s]
        node_label[e] = m
        label_end_node[m] = e
        label_length[m] = len(s)

    # Decision depth d_m (sec. 3.2): first k at which label m is the only label
    # with prefix x_1..x_k, then extended to the end of that word.
    decide = np.zeros(M, dtype=np.int32)
    for m, s in enumerate(seqs):
        t = len(s)
        if full_depth:
            decide[m] = t
            continue
        k0 = t
        for k in range(1, t + 1):
            if prefix_count[s[:k]] == 1:
                k0 = k
                break
        d = k0
        while d < t and _is_continuation(continuation, s[d]):  # s[d] is x_{d+1}
            d += 1
        decide[m] = d

    # Evaluated positions P: root, every parent of a scored token, every
    # prefix label's end node.
    evalset = {0}
    has_prefix = 0
    for m, s in enumerate(seqs):
        for k in range(1, int(decide[m]) + 1):
            evalset.add(node_id[s[: k - 1]])
        end = node_id[s]
        if children[end]:
            has_prefix = 1
            evalset.add(end)
    if all_nodes:  # every node evaluated (partner tries of a join)
        evalset = set(range(n))
    eval_nodes = np.array(sorted(evalset), dtype=np.int32)
    eval_index_of_node = np.full(n, -1, dtype=np.int32)
    eval_index_of_node[eval_nodes] = np.arange(len(eval_nodes), dtype=np.int32)
    eval_child_offsets = np.zeros(len(eval_nodes) + 1, dtype=np.int32)
    eval_child_offsets[1:] = np.cumsum([len(children[e]) for e in eval_nodes])

    return {
        "n_nodes": n,
        "num_labels": M,
        "n_eval": len(eval_nodes),
        "n_eval_children": int(eval_child_offsets[-1]),
        "max_depth": int(depth.max()),
        "has_prefix_labels": has_prefix,
        "parent": parent,
        "depth": depth,
        "token": token,
        "subtree_size": subtree_size,
        "child_offsets": child_offsets,
        "child_nodes": child_nodes,
        "child_tokens": child_tokens.astype(np.int32),
        "is_branching": is_branching,
        "subtree_labels": subtree_labels,
        "node_label": node_label,
        "label_end_node": label_end_node,
        "label_length": label_length,
        "label_decide_depth": decide,
        "eval_nodes": eval_nodes,
        "eval_index_of_node": eval_index_of_node,
        "eval_child_offsets": eval_child_offsets,
    }


def label_path(trie: dict, m: int) -> list:
    """Node ids root..end of label m (length t_m + 1)."""
    path = [int(trie["label_end_node"][m])]
    while path[-1] != 0:
        path.append(int(trie["parent"][path[-1]]))
    return path[::-1]


def children_of(trie: dict, u: int) -> np.ndarray:
    return trie["child_nodes"][trie["child_offsets"][u]: trie["child_offsets"][u + 1]]


def expected_decode_requests(trie: dict) -> float:
    """b = (1/M) sum_m c_m, c_m = branching nodes on label m's path up to and
    including the one that decides it ("To Classify, Try a Trie Tree", sec. 4.3).
    A label decided at node u means subtree_labels of u's chosen child is 1."""
    M = trie["num_labels"]
    total = 0
    for m in range(M):
        path = label_path(trie, m)
        c = 0
        for k in range(len(path) - 1):
            u = path[k]
            if trie["subtree_labels"][u] <= 1:
                break
            if trie["is_branching"][u]:
                c += 1
        total += c
    return total / M
