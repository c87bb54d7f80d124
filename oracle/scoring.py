"""Label scores, probabilities and the three label-scoring methods -- oracle
(test infrastructure), float64.

"To Classify, Try a Trie Tree":
  sec. 3.2  score(m) = prod_{k=1}^{d_m} P(x_k | prompt, x_1..x_{k-1})
            P^(m)    = score(m) / sum_{m'} score(m')
            prefix label: score(refund) = P(refund) * (1 - P(request | refund));
            read for several continuations as (1 - sum over all children c of
            P(c | label)), and -inf (probability 0) once that sum reaches 1.
  sec. 3.3  letters: the M letter probabilities at ANSWER:, rescaled to sum to 1.
  sec. 3.1  trie_decode: at a branching node pick the most likely child,
            follow forced tokens, stop once one label is left.
Ties (a reading; the pages are silent): argmax takes the lowest label index,
trie_decode the lowest child token id.
"""
from __future__ import annotations

import numpy as np

from . import model as M
from .trie import children_of, label_path

NEG_INF = -np.inf
PREFIX_SATURATION = 1.0 - 1e-12


def label_logscore(trie: dict, m: int, logp) -> float:
    """log score(m) given logp(node, child_token) = log P(child token | context
    ending at node): the first d_m token log-probs of the label's path, plus
    log(1 - sum over the end node's children) for a prefix label."""
    tok = trie["token"]
    path = label_path(trie, m)
    d = int(trie["label_decide_depth"][m])
    s = 0.0
    for k in range(1, d + 1):
        s += logp(path[k - 1], int(tok[path[k]]))
    end = path[-1]
    ch = children_of(trie, end)
    if len(ch):
        cont = sum(np.exp(logp(end, int(tok[c]))) for c in ch)
        s = s + np.log1p(-cont) if cont < PREFIX_SATURATION else NEG_INF
    return s


def logscores_from_table(trie: dict, logp) -> np.ndarray:
    """log score(m) for every label (model-free: planted tables use it too)."""
    return np.array([label_logscore(trie, m, logp) for m in range(trie["num_labels"])], dtype=np.float64)


def label_nodes(trie: dict, m: int) -> list:
    """Nodes whose next-token distribution label m's score reads."""
    path = label_path(trie, m)
    nodes = path[: int(trie["label_decide_depth"][m])]
    if len(children_of(trie, path[-1])):
        nodes.append(path[-1])
    return nodes


def normalise(logscore: np.ndarray) -> tuple:
    """(P^, argmax): P^(m) = score(m) / sum score; argmax = lowest index of the max."""
    finite = logscore[np.isfinite(logscore)]
    if len(finite) == 0:
        return np.full(len(logscore), np.nan), 0
    mx = finite.max()
    w = np.where(np.isfinite(logscore), np.exp(logscore - mx), 0.0)
    prob = w / w.sum()
    return prob, int(np.argmax(logscore))


def eval_logprob_rows(L: M.Layer, doc_k: np.ndarray, doc_v: np.ndarray, trie: dict, nodes=None,
                      head_rows: int = 128) -> dict:
    """log-prob of every child token at each node (default: the evaluated set
    P), each node attending to the document and to its own path. The nodes'
    states go through the output head head_rows at a time (one product per
    block, each row's log-sum-exp on its own)."""
    tok = trie["token"]
    nodes = [int(e) for e in (trie["eval_nodes"] if nodes is None else nodes)]
    Z = []
    for e in nodes:
        path = [e]
        while path[-1] != 0:
            path.append(int(trie["parent"][path[-1]]))
        path = path[::-1]
        Z.append(M.path_state(L, doc_k, doc_v, [int(tok[u]) for u in path]))
    rows = {}
    for lo in range(0, len(nodes), head_rows):
        lp = M.head_logprobs_rows(L, np.stack(Z[lo: lo + head_rows]))
        for r, e in enumerate(nodes[lo: lo + head_rows]):
            rows[e] = {int(tok[c]): float(lp[r, tok[c]]) for c in children_of(trie, e)}
    return rows


def trie_tree(L: M.Layer, doc_k: np.ndarray, doc_v: np.ndarray, trie: dict) -> dict:
    """trie_tree for one document (doc_k, doc_v float64 [l, H_kv, 128])."""
    rows = eval_logprob_rows(L, doc_k, doc_v, trie)
    ls = logscores_from_table(trie, lambda u, t: rows[u][t])
    prob, am = normalise(ls)
    return {"logscore": ls, "prob": prob, "argmax": am, "rows": rows}


def label_logscore_flat(L: M.Layer, doc_k, doc_v, root_token: int, label: list, decide_depth: int,
                        continuation_children: list | None = None) -> float:
    """Scores one label as its own flat causal sequence [root, x_1 .. x_t]
    (the "simple" per-label request of sec. 3.2), summing its first
    decide_depth token log-probs; continuation_children (prefix labels) adds
    log(1 - sum_c P(c | label))."""
    seq = [int(root_token)] + [int(t) for t in label]
    lp = M.sequence_logprobs(L, doc_k, doc_v, seq)
    s = sum(lp[k - 1, seq[k]] for k in range(1, decide_depth + 1))
    if continuation_children:
        cont = sum(np.exp(lp[len(label), c]) for c in continuation_children)
        s = s + np.log1p(-cont) if cont < PREFIX_SATURATION else NEG_INF
    return float(s)


def letters(L: M.Layer, doc_k, doc_v, letter_tokens: list, root_token: int) -> dict:
    """letters (sec. 3.3): logits of the M letter rows at ANSWER:, softmax over them."""
    z = M.path_state(L, doc_k, doc_v, [int(root_token)])
    W = M.bf16_to_f64(L.lm_bits[np.asarray(letter_tokens)])
    logits = W @ z
    lp = logits - M.logsumexp(logits)
    prob = np.exp(lp)
    return {"logprob": lp, "prob": prob, "argmax": int(np.argmax(lp)), "logits": logits}


def _unique_label(trie: dict, u: int) -> int:
    lo, hi = u, u + int(trie["subtree_size"][u])
    for m, e in enumerate(trie["label_end_node"]):
        if lo <= e < hi:
            return m
    raise AssertionError("subtree holds no label")


def trie_decode(L: M.Layer, doc_k, doc_v, trie: dict, child_logits=None) -> dict:
    """Greedy trie_decode (sec. 3.1) for one document. child_logits(u) may
    supply {child_token: logit} at node u (planted tables); by default the
    layer computes them. Returns the label and the nodes where logits were
    computed, in order."""
    tok = trie["token"]
    u = 0
    touched = []
    while True:
        while trie["subtree_labels"][u] > 1 and len(children_of(trie, u)) == 1:
            u = int(children_of(trie, u)[0])
        if trie["subtree_labels"][u] == 1:
            return {"label": _unique_label(trie, u), "touched": touched}
        if child_logits is None:
            path = [u]
            while path[-1] != 0:
                path.append(int(trie["parent"][path[-1]]))
            z = M.path_state(L, doc_k, doc_v, [int(tok[p]) for p in path[::-1]])
            W = L.lm_head()
            cl = {int(tok[c]): float(W[tok[c]].astype(np.float64) @ z) for c in children_of(trie, u)}
        else:
            cl = child_logits(u)
        touched.append(u)
        best = None
        for c in children_of(trie, u):  # ascending token id: first max wins ties
            if best is None or cl[int(tok[c])] > cl[int(tok[best])]:
                best = int(c)
        u = best
