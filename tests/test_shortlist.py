"""Huge label sets: hierarchical grouping and the top-B shortlist. The oracle
(oracle.shortlist) against Proposition 2, closed forms and the trie_tree
oracle; the library's grouped trie and shortlist tables against the oracle;
the CUDA path (quail_classify_trie_tree_shortlist) against the oracle."""
import math

import numpy as np
import pytest

import synthetic as S
from tests import gpu_cases as C


def _tiny_tree(seed=0, M=40, lens=(2, 5)):
    w = S.Workload("tiny-tree", S.TINY, 3, (64, 200), "tree", M, lens)
    return w, S.make_labels(w, seed)


# ----------------------------------------------------------------- oracle pins
def test_proposition2_sqrt_groups_minimise_the_step_cardinality():
    """Balanced groups: min over G of max(G, ceil(K/G)) is ceil(sqrt K), reached at G = ceil(sqrt K)."""
    from oracle import shortlist as SL
    for K in range(1, 2501):
        best = min(SL.effective_cardinality(K, G) for G in range(1, K + 1))
        r = math.ceil(math.sqrt(K))
        assert best == r, K
        assert SL.default_groups(K) == r, K
        assert SL.effective_cardinality(K, SL.default_groups(K)) == r, K


def test_groups_are_balanced_runs_in_token_order():
    from oracle import shortlist as SL
    rng = np.random.default_rng(5)
    labels = [list(rng.integers(0, 50, size=int(rng.integers(1, 5)))) for _ in range(137)]
    labels = [list(x) for x in {tuple(l) for l in labels}]
    K = len(labels)
    for G in (1, 2, 7, SL.default_groups(K), K):
        g = SL.group_labels(labels, G)
        sizes = np.bincount(g, minlength=G)
        assert sizes.sum() == K and sizes.max() - sizes.min() <= 1 and sizes.min() >= 1
        order = sorted(range(K), key=lambda m: tuple(labels[m]))
        assert np.all(np.diff(g[order]) >= 0)  # contiguous runs in sorted order


def test_rewrite_prepends_the_group_name():
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    labels = [[5, 6], [5, 7], [9], [3, 3, 3], [8, 1]]
    g = SL.group_labels(labels, 2)
    names = [[100, 101], [102, 103]]
    rw = SL.rewrite_grouped(labels, names, g)
    for lab, r, gg in zip(labels, rw, g):
        assert r == names[gg] + lab
    t = build_trie(rw, 0, 200)
    pref, gol = SL.prefix_groups(t, 2)
    assert pref == [tuple(n) for n in names] and list(gol) == list(g)
    with pytest.raises(SL.ShortlistError):
        SL.rewrite_grouped(labels, [[1], [1]], g)
    with pytest.raises(SL.ShortlistError):
        SL.prefix_groups(build_trie(labels, 0, 200), 2)  # [9] is shorter than 2


@pytest.mark.parametrize("D", [1, 2])
def test_full_beam_is_trie_tree(D):
    from oracle import scoring as OS
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    w, ls = _tiny_tree(1)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab)
    L = C.oracle_layer(w.shape, 0)
    docs = S.make_docs(w, 0)
    dk, dv = C.oracle_doc_kv(docs, 0)
    full = OS.trie_tree(L, dk, dv, t)
    r = SL.shortlist(L, dk, dv, t, D, 10 ** 6)
    np.testing.assert_allclose(r["logscore"], full["logscore"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["prob"], full["prob"], rtol=0, atol=1e-12)
    assert r["argmax"] == full["argmax"]


def test_prefix_score_is_the_flat_prefix_probability():
    """S(p) through the trie's rows equals the log-probability of p from a
    flat causal pass over [root, p] (oracle.model.sequence_logprobs)."""
    import oracle.model as OM
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    w, ls = _tiny_tree(2)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab)
    L = C.oracle_layer(w.shape, 0)
    dk, dv = C.oracle_doc_kv(S.make_docs(w, 0), 1)
    r = SL.shortlist(L, dk, dv, t, 2, 3)
    for i in (0, len(r["prefixes"]) // 2, len(r["prefixes"]) - 1):
        p = list(r["prefixes"][i])
        lp = OM.sequence_logprobs(L, dk, dv, [ls.root_token] + p)
        flat = lp[0, p[0]] + lp[1, p[1]]
        assert r["prefix_logscore"][i] == pytest.approx(flat, abs=1e-10)
    assert np.exp(r["prefix_logscore"]).sum() <= 1.0 + 1e-12  # disjoint prefixes


@pytest.mark.parametrize("D,B", [(1, 1), (1, 3), (2, 4)])
def test_shortlist_is_the_renormalised_restriction(D, B):
    from oracle import scoring as OS
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    w, ls = _tiny_tree(3)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab)
    L = C.oracle_layer(w.shape, 0)
    dk, dv = C.oracle_doc_kv(S.make_docs(w, 0), 2)
    full = OS.trie_tree(L, dk, dv, t)
    B = min(B, len(SL.prefix_groups(t, D)[0]) - 1)  # a proper shortlist
    r = SL.shortlist(L, dk, dv, t, D, B)
    S_ = r["prefix_logscore"]
    assert r["selected"] == sorted(range(len(S_)), key=lambda i: (-S_[i], i))[:B]
    keep = np.isin(r["group_of_label"], r["selected"])
    assert keep.any() and not keep.all()
    np.testing.assert_allclose(r["logscore"][keep], full["logscore"][keep], rtol=0, atol=1e-12)
    assert np.all(np.isneginf(r["logscore"][~keep])) and np.all(r["prob"][~keep] == 0)
    pk = full["prob"][keep]
    np.testing.assert_allclose(r["prob"][keep], pk / pk.sum(), rtol=1e-12, atol=0)
    assert keep[r["argmax"]]
