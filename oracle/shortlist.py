"""Huge label sets: hierarchical grouping and a top-B shortlist ahead of exact
trie scoring -- oracle (test infrastructure), float64.

"Trie Automata for Constrained Decoding over Large Finite Sets", the two
extensions sketched for K > 50,000 labels:
  * hierarchical schema rewriting: the K labels are split into G ~ sqrt(K)
    groups and the answer becomes a group name followed by the label, so no
    step chooses among more than max(G, ceil(K / G)) continuations
    (Proposition 2: for balanced groups this is smallest, ceil(sqrt K), at
    G = ceil(sqrt K));
  * speculative short-circuiting: a cheap score keeps a top-k shortlist and
    exact trie-constrained scoring runs on the shortlist only.
Scores of the shortlisted labels are those of "To Classify, Try a Trie Tree",
sec. 3.2 (oracle.scoring).

Readings (the pages say no more than the above):
  * groups: the labels sorted by their token sequences, cut into G contiguous
    runs whose sizes differ by at most one; group g's name is a caller-given
    token sequence, every name of the same length D;
  * cheap score of the labels sharing their first D tokens p: the exact
    log-probability that the answer starts with p,
    S(p) = sum_{k=1..D} log P(p_k | context, p_1..p_{k-1});
  * shortlist: the B prefixes of highest S (ties: the lower prefix index,
    prefixes numbered in lexicographic token order); every label under them
    gets its exact trie_tree log score, every other label -inf, and P^ is
    renormalised over the shortlist (argmax: the lowest label index of the
    maximum, as for trie_tree). Labels shorter than D are not allowed.
With B at least the number of distinct prefixes this is trie_tree itself.
"""
from __future__ import annotations

import math

import numpy as np

from . import scoring as OS
from .trie import children_of, label_path


class ShortlistError(ValueError):
    pass


def effective_cardinality(K: int, G: int) -> int:
    """Most continuations any step chooses among after splitting K labels
    into G balanced groups: G at the group step, ceil(K / G) inside a group."""
    if K < 1 or G < 1:
        raise ShortlistError("K and G must be positive")
    return max(G, -(-K // G))


def default_groups(K: int) -> int:
    """G = ceil(sqrt K) (Proposition 2)."""
    return math.isqrt(K - 1) + 1 if K > 1 else 1


def group_labels(labels, G: int) -> np.ndarray:
    """group_of_label[m]: labels sorted by token sequence, cut into G runs;
    sorted position j falls in group g when floor(g K / G) <= j < floor((g+1) K / G)."""
    K = len(labels)
    if not (1 <= G <= K):
        raise ShortlistError(f"need 1 <= G <= K (G = {G}, K = {K})")
    order = sorted(range(K), key=lambda m: tuple(int(t) for t in labels[m]))
    out = np.empty(K, dtype=np.int32)
    for j, m in enumerate(order):
        g = (j * G) // K
        # the smallest g with j < floor((g+1) K / G)
        while j >= ((g + 1) * K) // G:
            g += 1
        while g > 0 and j < (g * K) // G:
            g -= 1
        out[m] = g
    return out


def rewrite_grouped(labels, group_names, group_of_label) -> list:
    """Label m becomes group_names[group_of_label[m]] followed by label m."""
    names = [list(int(t) for t in nm) for nm in group_names]
    if len({len(nm) for nm in names}) != 1 or len(names[0]) == 0:
        raise ShortlistError("group names must share one positive length")
    if len({tuple(nm) for nm in names}) != len(names):
        raise ShortlistError("group names must be distinct")
    return [names[int(g)] + [int(t) for t in lab] for lab, g in zip(labels, group_of_label)]


def prefix_groups(trie: dict, D: int) -> tuple:
    """(prefixes, group_of_label): the distinct first-D-token prefixes of the
    trie's labels in lexicographic order, and each label's prefix index."""
    if D < 1:
        raise ShortlistError("cut depth must be >= 1")
    tok = trie["token"]
    pref = []
    for m in range(trie["num_labels"]):
        path = label_path(trie, m)
        if len(path) - 1 < D:
            raise ShortlistError(f"label {m} is shorter than the cut depth {D}")
        pref.append(tuple(int(tok[u]) for u in path[1: D + 1]))
    prefixes = sorted(set(pref))
    index = {p: i for i, p in enumerate(prefixes)}
    return prefixes, np.array([index[p] for p in pref], dtype=np.int32)


class _Rows:
    """Next-token log-probs of trie nodes, computed on first use."""

    def __init__(self, L, doc_k, doc_v, trie):
        self.L, self.dk, self.dv, self.trie = L, doc_k, doc_v, trie
        self.rows = {}

    def logp(self, u: int, t: int) -> float:
        if u not in self.rows:
            self.rows.update(OS.eval_logprob_rows(self.L, self.dk, self.dv, self.trie, nodes=[u]))
        return self.rows[u][t]


def prefix_logscores(rows: _Rows, trie: dict, D: int, prefixes) -> np.ndarray:
    """S(p) for every prefix: the log-probs of its D tokens along the trie path."""
    tok = trie["token"]
    out = np.empty(len(prefixes), dtype=np.float64)
    for i, p in enumerate(prefixes):
        u, s = 0, 0.0
        for t in p:
            s += rows.logp(u, int(t))
            u = next(int(c) for c in children_of(trie, u) if int(tok[c]) == int(t))
        out[i] = s
    return out


def select_top(scores: np.ndarray, B: int) -> list:
    """Indices of the B highest scores, highest first, ties to the lower index."""
    return sorted(range(len(scores)), key=lambda i: (-scores[i], i))[: max(0, min(B, len(scores)))]


def _restricted(rows: _Rows, trie: dict, gol: np.ndarray, groups) -> tuple:
    """Exact log scores of the labels in `groups`, -inf elsewhere; P^ over them."""
    keep = np.isin(gol, np.array(list(groups), dtype=np.int32))
    ls = np.full(trie["num_labels"], -np.inf)
    for m in np.nonzero(keep)[0]:
        ls[m] = OS.label_logscore(trie, int(m), rows.logp)
    prob, am = OS.normalise(ls)
    return ls, np.where(keep, prob, 0.0), am


def scores_for_groups(L, doc_k, doc_v, trie: dict, D: int, groups) -> dict:
    """The prefix scores S of every group, and the label scores of the
    shortlist made of `groups` (any set of prefix indices)."""
    prefixes, gol = prefix_groups(trie, D)
    rows = _Rows(L, doc_k, doc_v, trie)
    S = prefix_logscores(rows, trie, D, prefixes)
    ls, prob, am = _restricted(rows, trie, gol, groups)
    return {"logscore": ls, "prob": prob, "argmax": am, "prefix_logscore": S, "group_of_label": gol,
            "prefixes": prefixes}


def shortlist(L, doc_k, doc_v, trie: dict, D: int, B: int) -> dict:
    """Shortlisted trie_tree for one document: the B prefixes of highest S,
    exact log scores for the labels under them, -inf for the rest."""
    prefixes, gol = prefix_groups(trie, D)
    rows = _Rows(L, doc_k, doc_v, trie)
    S = prefix_logscores(rows, trie, D, prefixes)
    sel = select_top(S, B)
    ls, prob, am = _restricted(rows, trie, gol, sel)
    return {"logscore": ls, "prob": prob, "argmax": am, "selected": sel, "prefix_logscore": S,
            "group_of_label": gol, "prefixes": prefixes}
