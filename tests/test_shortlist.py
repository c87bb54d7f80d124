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


# ------------------------------------------------------- library host tables
def _view_equal(view, ref):
    for k in ("parent", "depth", "token", "subtree_size", "child_offsets", "child_tokens", "label_end_node",
              "label_decide_depth", "eval_nodes", "eval_child_offsets"):
        np.testing.assert_array_equal(view[k], ref[k], err_msg=k)


@pytest.mark.parametrize("G", [0, 5, 40])
def test_grouped_trie_is_the_oracle_rewrite(G):
    import trie_label_scoring_gb300 as Q
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    w, ls = _tiny_tree(4, M=40)
    K = len(ls.labels)
    Gr = G or SL.default_groups(K)
    names = S.make_group_names(0, Gr, 2, w.shape.vocab)
    t, gol = Q.Trie.grouped(ls.labels, ls.root_token, w.shape.vocab, names, num_groups=G)
    ref_g = SL.group_labels(ls.labels, Gr)
    np.testing.assert_array_equal(gol, ref_g)
    rw = SL.rewrite_grouped(ls.labels, names, ref_g)
    _view_equal(t.view(), build_trie(rw, ls.root_token, w.shape.vocab))


def test_shortlist_plan_groups_are_the_oracle_prefixes():
    import trie_label_scoring_gb300 as Q
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    w, ls = _tiny_tree(5, M=60, lens=(2, 6))
    t = Q.Trie(ls.labels, ls.root_token, w.shape.vocab)
    ref = build_trie(ls.labels, ls.root_token, w.shape.vocab)
    for D in (1, 2):
        sl = Q.Shortlist(t, D)
        pref, gol = SL.prefix_groups(ref, D)
        assert sl.num_groups == len(pref)
        np.testing.assert_array_equal(sl.group_of_label(), gol)
        sl.close()


def test_shortlist_and_grouping_reject_bad_arguments():
    import trie_label_scoring_gb300 as Q
    labels = [[5, 6], [5, 7], [9], [3, 3, 3]]
    t = Q.Trie(labels, 0, 100)
    with pytest.raises(Q.QuailError):
        Q.Shortlist(t, 2)  # [9] is shorter than the cut
    with pytest.raises(Q.QuailError):
        Q.Shortlist(Q.Trie([[5, 6], [5, 7]], 0, 100), 1)  # a single group
    with pytest.raises(Q.QuailError):
        Q.Trie.grouped(labels, 0, 100, [[1], [1]], num_groups=2)  # equal names
    with pytest.raises(Q.QuailError):
        Q.Trie.grouped(labels, 0, 100, [[1], [2], [3], [4], [5]], num_groups=5)  # more groups than labels


def test_scores_for_the_selected_groups_are_the_shortlist():
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    w, ls = _tiny_tree(6)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab)
    L = C.oracle_layer(w.shape, 0)
    dk, dv = C.oracle_doc_kv(S.make_docs(w, 0), 0)
    r = SL.shortlist(L, dk, dv, t, 2, 3)
    q = SL.scores_for_groups(L, dk, dv, t, 2, r["selected"])
    np.testing.assert_array_equal(q["logscore"], r["logscore"])
    np.testing.assert_array_equal(q["prob"], r["prob"])


# ------------------------------------------------------------------ GPU parity
def _run_shortlist(w, docs, trie, sl, beam, seed=0):
    import torch
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    model = C.device_model(w.shape, seed)
    kv = kv_from_docs(docs)
    N, M = len(docs.doc_len), trie.num_labels
    B = min(beam, sl.num_groups)
    ws = torch.empty(Q.workspace_size_shortlist(model, trie, sl, beam, N, docs.max_doc_len), dtype=torch.uint8,
                     device="cuda")
    lsc = torch.full((N, M), float("nan"), device="cuda")
    prob = torch.full((N, M), float("nan"), device="cuda")
    am = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    sel = torch.full((N, B), -1, dtype=torch.int32, device="cuda")
    Q.classify_trie_tree_shortlist(model, kv, trie, sl, beam, N, ws, lsc, prob, am, sel)
    Q.device_status()
    return lsc.cpu().numpy(), prob.cpu().numpy(), am.cpu().numpy(), sel.cpu().numpy()


def _check_shortlist(w, docs, ref_trie, D, beam, docs_idx, out, seed=0):
    """Per document: the GPU's kept groups are a valid top-B set of the
    oracle's prefix scores (equal to the oracle's set where its B-th and
    next scores differ by more than twice the log-score tolerance), and the
    scores equal the oracle's for that kept set."""
    from oracle import shortlist as SL
    lsc, prob, am, sel = out
    L = C.oracle_layer(w.shape, seed)
    for i in docs_idx:
        dk, dv = C.oracle_doc_kv(docs, i)
        g_sel = [int(g) for g in sel[i]]
        r = SL.scores_for_groups(L, dk, dv, ref_trie, D, g_sel)
        S_ = r["prefix_logscore"]
        top = SL.select_top(S_, beam)
        B = len(top)
        assert len(g_sel) == B and len(set(g_sel)) == B, f"doc {i}: selection {g_sel}"
        kth = S_[top[-1]]
        assert all(S_[g] >= kth - C.TOL_LOGSCORE for g in g_sel), f"doc {i}: {g_sel} vs {top}"
        rest = [S_[g] for g in range(len(S_)) if g not in top]
        if not rest or kth - max(rest) > 2 * C.TOL_LOGSCORE:
            assert set(g_sel) == set(top), f"doc {i}: {g_sel} vs {top}"
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


@pytest.mark.gpu
def test_shortlist_full_beam_is_trie_tree_gpu():
    import trie_label_scoring_gb300 as Q
    from oracle import scoring as OS
    from oracle.trie import build_trie
    w, ls = _tiny_tree(7, M=40)
    w = S.with_docs(w, 5, (1, 600))
    docs = S.make_docs(w, 7)
    t = Q.Trie(ls.labels, ls.root_token, w.shape.vocab)
    sl = Q.Shortlist(t, 1)
    lsc, prob, am, sel = _run_shortlist(w, docs, t, sl, 10 ** 4)
    ref_t = build_trie(ls.labels, ls.root_token, w.shape.vocab)
    L = C.oracle_layer(w.shape, 0)
    for i in range(5):
        dk, dv = C.oracle_doc_kv(docs, i)
        r = OS.trie_tree(L, dk, dv, ref_t)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")
        assert sorted(sel[i]) == list(range(sl.num_groups))


@pytest.mark.gpu
@pytest.mark.parametrize("D,beam", [(1, 1), (1, 2), (2, 3)])
def test_shortlist_tiny_gpu(D, beam):
    import trie_label_scoring_gb300 as Q
    from oracle.trie import build_trie
    w, ls = _tiny_tree(8, M=60, lens=(2, 6))
    w = S.with_docs(w, 6, (1, 500))
    docs = S.make_docs(w, 8)
    t = Q.Trie(ls.labels, ls.root_token, w.shape.vocab)
    sl = Q.Shortlist(t, D)
    out = _run_shortlist(w, docs, t, sl, beam)
    _check_shortlist(w, docs, build_trie(ls.labels, ls.root_token, w.shape.vocab), D, beam, range(6), out)


@pytest.mark.gpu
def test_grouped_labels_tiny_gpu():
    """Hierarchical grouping: ceil(sqrt K) one-token group names, the two most
    likely groups kept; more than 128 query rows per KV head per document."""
    import trie_label_scoring_gb300 as Q
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    w, ls = _tiny_tree(9, M=400, lens=(2, 6))
    w = S.with_docs(w, 4, (100, 700))
    docs = S.make_docs(w, 9)
    G = SL.default_groups(len(ls.labels))
    names = S.make_group_names(9, G, 1, w.shape.vocab)
    t, gol = Q.Trie.grouped(ls.labels, ls.root_token, w.shape.vocab, names)
    sl = Q.Shortlist(t, 1)
    assert sl.num_groups == G
    out = _run_shortlist(w, docs, t, sl, 2)
    rw = SL.rewrite_grouped(ls.labels, names, SL.group_labels(ls.labels, G))
    _check_shortlist(w, docs, build_trie(rw, ls.root_token, w.shape.vocab), 1, 2, range(4), out)


@pytest.mark.gpu
def test_grouped_labels_qwen_shape_sampled():
    import trie_label_scoring_gb300 as Q
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    base = S.SHORTLIST_WORKLOADS["qwen3-4b-grouped60k-16x1024"].base
    w = S.dataclasses.replace(S.with_docs(base, 4, (256, 1024)), num_labels=2000)
    ls = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    G = SL.default_groups(len(ls.labels))
    names = S.make_group_names(0, G, 1, w.shape.vocab)
    t, _ = Q.Trie.grouped(ls.labels, ls.root_token, w.shape.vocab, names)
    sl = Q.Shortlist(t, 1)
    out = _run_shortlist(w, docs, t, sl, 2)
    rw = SL.rewrite_grouped(ls.labels, names, SL.group_labels(ls.labels, G))
    _check_shortlist(w, docs, build_trie(rw, ls.root_token, w.shape.vocab), 1, 2, [0, 3], out)


@pytest.mark.gpu
def test_grouped_labels_full_size_sampled():
    """The bench workload itself: 60,000 labels in ceil(sqrt K) one-token
    groups, 16 documents of 1,024 tokens, beam 4; two documents checked."""
    import trie_label_scoring_gb300 as Q
    from oracle import shortlist as SL
    from oracle.trie import build_trie
    sw = S.SHORTLIST_WORKLOADS["qwen3-4b-grouped60k-16x1024"]
    w = sw.base
    ls = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    G = SL.default_groups(len(ls.labels))
    names = S.make_group_names(0, G, 1, w.shape.vocab)
    t, _ = Q.Trie.grouped(ls.labels, ls.root_token, w.shape.vocab, names, num_groups=G)
    sl = Q.Shortlist(t, 1)
    out = _run_shortlist(w, docs, t, sl, sw.beam)
    rw = SL.rewrite_grouped(ls.labels, names, SL.group_labels(ls.labels, G))
    _check_shortlist(w, docs, build_trie(rw, ls.root_token, w.shape.vocab), 1, sw.beam, [0, 15], out)
