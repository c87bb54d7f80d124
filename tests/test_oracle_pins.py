"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test compares the oracle with something other than itself: numbers the
pages print (tests/golden/*.json, each with its citation), closed forms,
brute force on tiny inputs, library routines for special cases, and an
independent flat causal evaluation. No GPU.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import synthetic as S
from oracle import model as OM
from oracle import scoring as OS
from oracle.trie import TrieError, build_trie, children_of, expected_decode_requests, label_path

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ trie
def _support(vocab=8192, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    return S.support_labels(vocab, rng)


def test_support_shape_counts():
    g = golden("support_shape.json")
    ls = _support()
    t = build_trie(ls.labels, ls.root_token, 8192, ls.continuation)
    assert t["n_nodes"] == g["n_nodes_including_root"]
    assert int(t["is_branching"].sum()) == g["branching_nodes"]
    assert int((np.diff(t["child_offsets"]) > 0).sum()) == g["nodes_with_children"]
    assert t["n_eval"] == g["evaluated_positions"]
    assert expected_decode_requests(t) == pytest.approx(g["expected_decode_requests_b"], abs=1e-12)
    # evaluated nodes are ANSWER:, refund, shipping, two = root and the first
    # tokens of labels 1, 3 and 7 of the running example
    names = g["labels"]
    first_tok = {names[m]: ls.labels[m][0] for m in range(len(names))}
    want = {0} | {int(t["child_nodes"][j]) for j in range(t["child_offsets"][0], t["child_offsets"][1])
                  if int(t["child_tokens"][j]) in (first_tok["refund request"], first_tok["shipping delay"],
                                                   first_tok["two-factor authentication issue"])}
    assert set(t["eval_nodes"].tolist()) == want
    # 5 labels are decided right at ANSWER: (sec. 4.3)
    decided_at_root = sum(1 for m in range(10) if t["subtree_labels"][label_path(t, m)[1]] == 1)
    assert decided_at_root == g["labels_decided_at_root"]


def test_support_score_table():
    g = golden("support_shape.json")
    ls = _support()
    t = build_trie(ls.labels, ls.root_token, 8192, ls.continuation)
    for name, d in g["score_table"].items():
        if name.startswith("_"):
            continue
        m = g["labels"].index(name)
        assert t["label_decide_depth"][m] == d, name


def _random_label_set(rng, vocab, M, maxlen, allow_prefix):
    labels = set()
    while len(labels) < M:
        L = int(rng.integers(1, maxlen + 1))
        labels.add(tuple(int(x) for x in rng.integers(0, vocab, size=L)))
    labels = [list(l) for l in labels]
    if not allow_prefix:
        labels = [l for l in labels if not any(o != l and o[: len(l)] == l for o in labels)]
    rng.shuffle(labels)
    return labels


@pytest.mark.parametrize("seed", range(20))
def test_trie_is_sorted_distinct_prefixes(seed):
    """Brute force: the nodes are exactly the distinct label prefixes, and
    preorder with ascending children is the lexicographic order of those
    prefixes (the trie is the minimal DFA of the finite set, unique up to
    isomorphism; "Trie Automata for Constrained Decoding over Large Finite
    Sets", Proposition 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    labels = _random_label_set(rng, 5, int(rng.integers(2, 12)), 4, allow_prefix=True)
    if len(labels) < 2:
        labels = [[0], [1, 2]]
    t = build_trie(labels, 3, 5)
    prefixes = sorted({tuple(l[:k]) for l in labels for k in range(len(l) + 1)})
    assert t["n_nodes"] == len(prefixes)
    for i, p in enumerate(prefixes):
        assert t["depth"][i] == len(p)
        if p:
            assert t["token"][i] == p[-1]
            assert t["parent"][i] == prefixes.index(p[:-1])
        # subtree = contiguous id range of the prefixes extending p
        ext = [j for j, q in enumerate(prefixes) if q[: len(p)] == p]
        assert ext == list(range(i, i + int(t["subtree_size"][i])))
        assert t["subtree_labels"][i] == sum(1 for l in labels if tuple(l[: len(p)]) == p)
    for m, l in enumerate(labels):
        assert t["label_end_node"][m] == prefixes.index(tuple(l))
        # d_m: tokens before it are shared with another label, the prefix up to it is not
        d = int(t["label_decide_depth"][m])
        assert 1 <= d <= len(l)
        assert sum(1 for o in labels if o[:d] == l[:d]) == 1 or d == len(l)
        if d > 1:
            assert sum(1 for o in labels if o[: d - 1] == l[: d - 1]) > 1
    # P is closed under ancestors and holds every parent of a scored token
    ev = set(t["eval_nodes"].tolist())
    for e in ev:
        if e:
            assert int(t["parent"][e]) in ev
    for m, l in enumerate(labels):
        path = label_path(t, m)
        for k in range(1, int(t["label_decide_depth"][m]) + 1):
            assert path[k - 1] in ev


def test_trie_errors():
    with pytest.raises(TrieError) as e:
        build_trie([[1], []], 0, 10)
    assert e.value.kind == "empty_label"
    with pytest.raises(TrieError) as e:
        build_trie([[1, 2], [3], [1, 2]], 0, 10)
    assert e.value.kind == "duplicate_label"
    with pytest.raises(TrieError) as e:
        build_trie([[1, 10], [3]], 0, 10)
    assert e.value.kind == "token_range"
    with pytest.raises(TrieError) as e:
        build_trie([[1]], 0, 10)
    assert e.value.kind == "invalid_arg"


def test_prefix_label_structure():
    t = build_trie([[5], [5, 7], [9]], 1, 10)  # refund, refund request, praise
    refund = label_path(t, 0)[-1]
    assert t["node_label"][refund] == 0 and len(children_of(t, refund)) == 1
    assert t["has_prefix_labels"] == 1
    assert refund in set(t["eval_nodes"].tolist())
    assert t["label_decide_depth"].tolist() == [1, 2, 1]


def test_continuation_extends_to_word_end():
    # two-factor authentication issue: x_2 continues the word "two" -> d = 2
    bitmap = np.zeros(2, dtype=np.uint8)
    bitmap[7 >> 3] |= 1 << (7 & 7)
    t = build_trie([[3, 7, 8, 9], [4]], 0, 16, bitmap)
    assert t["label_decide_depth"].tolist() == [2, 1]
    t = build_trie([[3, 7, 8, 9], [4]], 0, 16, None)
    assert t["label_decide_depth"].tolist() == [1, 1]
    t = build_trie([[3, 7, 8, 9], [4]], 0, 16, None, full_depth=True)
    assert t["label_decide_depth"].tolist() == [4, 1]


# ------------------------------------------------------------------ scoring math (model-free)
def _planted(trie, table):
    """table: {(node path as token tuple, next token): prob}"""
    tok = trie["token"]

    def path_tokens(u):
        p = []
        while u:
            p.append(int(tok[u]))
            u = int(trie["parent"][u])
        return tuple(p[::-1])

    return lambda u, t: math.log(table[(path_tokens(u), t)])


def test_refund_vs_praise_worked_example():
    g = golden("label_scoring_examples.json")["refund_vs_praise"]
    r1, r2, p = 11, 12, 13
    bitmap = np.zeros(4, dtype=np.uint8)
    bitmap[r2 >> 3] |= 1 << (r2 & 7)  # refund is one word of two tokens
    t = build_trie([[r1, r2], [p]], 1, 32, bitmap)
    table = {((), r1): g["p_refund_tok1"], ((r1,), r2): g["p_refund_tok2_given_tok1"], ((), p): g["p_praise"]}
    ls = OS.logscores_from_table(t, _planted(t, table))
    assert math.exp(ls[0]) == pytest.approx(g["sequence_probability_refund"], abs=1e-12)
    prob, am = OS.normalise(ls)
    assert am == 0
    assert prob[0] == pytest.approx(g["normalised_probability_refund"], abs=1e-12)
    assert prob.sum() == pytest.approx(1.0, abs=1e-15)


def test_prefix_label_worked_numbers():
    g = golden("label_scoring_examples.json")["prefix_label"]
    r, q, pr = 5, 7, 9
    t = build_trie([[r], [r, q], [pr]], 1, 10)
    table = {((), r): g["p_refund"], ((r,), q): g["p_request_given_refund"], ((), pr): 0.1}
    ls = OS.logscores_from_table(t, _planted(t, table))
    assert math.exp(ls[0]) == pytest.approx(g["score_refund"], abs=1e-12)
    assert math.exp(ls[1]) == pytest.approx(g["score_refund_request"], abs=1e-12)


def test_prefix_label_saturates_to_zero():
    t = build_trie([[5], [5, 7]], 1, 10)
    table = {((), 5): 0.9, ((5,), 7): 1.0}
    ls = OS.logscores_from_table(t, _planted(t, table))
    assert ls[0] == -np.inf
    prob, am = OS.normalise(ls)
    assert prob.tolist() == [0.0, 1.0] and am == 1


def test_greedy_can_disagree_with_tree():
    g = golden("label_scoring_examples.json")["greedy_disagrees"]
    r1, r2, p = 11, 12, 13
    bitmap = np.zeros(4, dtype=np.uint8)
    bitmap[r2 >> 3] |= 1 << (r2 & 7)
    t = build_trie([[r1, r2], [p]], 1, 32, bitmap)
    table = {((), r1): g["p_refund_tok1"], ((r1,), r2): g["p_refund_tok2_given_tok1"], ((), p): g["p_praise"]}
    lp = _planted(t, table)
    ls = OS.logscores_from_table(t, lp)
    assert ["refund", "praise"][OS.normalise(ls)[1]] == g["trie_tree_choice"]
    dec = OS.trie_decode(None, None, None, t, child_logits=lambda u: {
        int(t["token"][c]): lp(u, int(t["token"][c])) for c in children_of(t, u)})
    assert ["refund", "praise"][dec["label"]] == g["trie_decode_choice"]
    assert dec["touched"] == [0]


# ------------------------------------------------------------------ layer math
def test_rms_norm_closed_form():
    y = OM.rms_norm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    assert y.tolist() == pytest.approx([3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], abs=1e-15)
    y = OM.rms_norm(np.array([1.0, 1.0, 1.0, 1.0]), np.array([1.0, 2.0, 3.0, 4.0]), 0.0)
    assert y.tolist() == pytest.approx([1.0, 2.0, 3.0, 4.0], abs=1e-15)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(128)
    theta = 1e6
    for pos in (0, 1, 17, 1000, 8200):
        y = OM.rope(x, pos, theta)
        w = theta ** (-np.arange(64) * 2.0 / 128)
        zc = (x[:64] + 1j * x[64:]) * np.exp(1j * pos * w)
        assert np.allclose(y[:64], zc.real, atol=1e-12) and np.allclose(y[64:], zc.imag, atol=1e-12)
    assert np.allclose(OM.rope(x, 0, theta), x)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    a = OM.rope(q, 1030, theta) @ OM.rope(k, 1027, theta)
    b = OM.rope(q, 3, theta) @ OM.rope(k, 0, theta)
    assert a == pytest.approx(b, abs=1e-9)


def test_attention_matches_double_loop():
    rng = np.random.default_rng(1)
    hq, hkv, D, n = 4, 2, 8, 7
    q = rng.standard_normal((hq, D))
    K = rng.standard_normal((n, hkv, D))
    V = rng.standard_normal((n, hkv, D))
    out = OM.gqa_attention(q, K, V).reshape(hq, D)
    for h in range(hq):
        g = h // (hq // hkv)
        num = np.zeros(D)
        den = 0.0
        for j in range(n):
            s = sum(q[h, i] * K[j, g, i] for i in range(D)) / math.sqrt(D)
            num += math.exp(s) * V[j, g]
            den += math.exp(s)
        assert np.allclose(out[h], num / den, atol=1e-12)


def _tiny_setup(shape=S.TINY, ndocs=2, doc_len=(20, 37), seed=0):
    w = S.Workload("pin", shape, ndocs, doc_len, "support")
    L = OM.Layer(S.make_model(shape, seed), shape)
    docs = S.make_docs(w, seed)
    kv = []
    for i in range(ndocs):
        k, v = docs.doc_kv(i)
        kv.append((OM.bf16_to_f64(k), OM.bf16_to_f64(v)))
    return L, kv


def test_head_logprobs_match_scipy():
    L, kv = _tiny_setup()
    z = OM.path_state(L, kv[0][0], kv[0][1], [5, 6])
    lp = OM.head_logprobs(L, z)
    logits = OM.bf16_to_f64(L.lm_bits) @ z
    assert np.allclose(lp, scipy.special.log_softmax(logits), atol=1e-12)
    assert np.exp(lp).sum() == pytest.approx(1.0, abs=1e-12)
    # several states through the head at once: each row is its own log-softmax
    Z = np.stack([OM.path_state(L, kv[0][0], kv[0][1], p) for p in ([5], [5, 6], [9, 1, 2])])
    rows = OM.head_logprobs_rows(L, Z)
    assert np.allclose(rows, scipy.special.log_softmax(Z @ OM.bf16_to_f64(L.lm_bits).T, axis=1), atol=1e-12)


def test_flat_sequence_equals_tree_masked():
    """Scoring each label as its own flat causal sequence equals the
    tree-masked result ("Building an Ultra-High Throughput AI-SQL Engine",
    sec. 3.2.4: the tree evaluation produces the same output as attention
    over each full sequence; "To Classify, Try a Trie Tree", sec. 3.2: each
    node attends only to the prompt and its own path)."""
    L, kv = _tiny_setup()
    ls = _support(S.TINY.vocab, 3)
    for full in (False, True):
        t = build_trie(ls.labels, ls.root_token, S.TINY.vocab, ls.continuation, full_depth=full)
        for dk, dv in kv:
            tree = OS.trie_tree(L, dk, dv, t)
            for m, lab in enumerate(ls.labels):
                flat = OS.label_logscore_flat(L, dk, dv, ls.root_token, lab, int(t["label_decide_depth"][m]))
                assert tree["logscore"][m] == pytest.approx(flat, abs=1e-10)
            assert tree["prob"].sum() == pytest.approx(1.0, abs=1e-12)


def test_flat_sequence_equals_tree_masked_many_rows():
    """The same equivalence on a shared-prefix label set with more evaluated
    nodes than one block of the oracle's batched output head (128 rows), so
    several blocks and a partial one are checked."""
    L, kv = _tiny_setup()
    rng = np.random.Generator(np.random.PCG64(12))
    ls = S.shared_prefix_labels(1200, 2, 6, S.TINY.vocab, rng, 4.0)
    t = build_trie(ls.labels, ls.root_token, S.TINY.vocab)
    assert t["n_eval"] > 2 * 128 and t["n_eval"] % 128 != 0
    dk, dv = kv[0]
    tree = OS.trie_tree(L, dk, dv, t)
    assert tree["prob"].sum() == pytest.approx(1.0, abs=1e-12)
    for m in range(0, 1200, 67):
        flat = OS.label_logscore_flat(L, dk, dv, ls.root_token, ls.labels[m], int(t["label_decide_depth"][m]))
        assert tree["logscore"][m] == pytest.approx(flat, abs=1e-10)


def test_shared_prefix_generator_shape():
    """The generator of the 5,000-label workload: lengths on [lmin, lmax], no
    label a prefix of another, and about 20,000 trie nodes of depth at most 10
    at the workload's sharing (the workload names 5,000 labels of 2-10 tokens,
    ~20k nodes, maximum depth 10)."""
    w = S.WORKLOADS["qwen3-4b-tree5000-16x1024"]
    ls = S.make_labels(w, 0)
    lens = [len(l) for l in ls.labels]
    assert len(ls.labels) == 5000 and min(lens) == 2 and max(lens) == 10
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab)
    assert not t["has_prefix_labels"]
    assert 16000 <= t["n_nodes"] <= 24000 and t["max_depth"] == 10


SMALL_V = S.LayerShape(hidden=64, n_q_heads=2, n_kv_heads=1, vocab=4, weight_std=0.5, kv_std=1.0)


def test_complete_vocabulary_trie_sums_to_one():
    """Every length-2 sequence over a 4-token vocabulary: the label scores are
    the probabilities of all outcomes of two steps, so they sum to 1."""
    L, kv = _tiny_setup(SMALL_V, 1, (9, 9))
    labels = [list(p) for p in itertools.product(range(4), repeat=2)]
    for full in (False, True):
        t = build_trie(labels, 2, 4, None, full_depth=full)
        r = OS.trie_tree(L, kv[0][0], kv[0][1], t)
        assert np.exp(r["logscore"]).sum() == pytest.approx(1.0, abs=1e-12)


def test_prefix_labels_complete_the_distribution():
    """Labels [0], [0,1], [0,2], [1], [2], [3] over a 4-token vocabulary: with
    the prefix correction score([0]) = P(0)(1 - P(1|0) - P(2|0)), the scores
    still account for all of P(0), so they sum to 1."""
    L, kv = _tiny_setup(SMALL_V, 1, (9, 9))
    labels = [[0], [0, 1], [0, 2], [1], [2], [3]]
    t = build_trie(labels, 2, 4)
    r = OS.trie_tree(L, kv[0][0], kv[0][1], t)
    assert np.exp(r["logscore"]).sum() == pytest.approx(1.0, abs=1e-12)
    # and each prefix-label score equals the flat evaluation with its continuation term
    dk, dv = kv[0]
    flat0 = OS.label_logscore_flat(L, dk, dv, 2, [0], 1, continuation_children=[1, 2])
    assert r["logscore"][0] == pytest.approx(flat0, abs=1e-10)


def test_letters_equals_full_vocabulary_route():
    """letters rescales the letter probabilities to sum to 1 (sec. 3.3): the
    same numbers come out of the full log-softmax restricted to the letters."""
    L, kv = _tiny_setup()
    letters = [5, 900, 33, 7000, 12]
    r = OS.letters(L, kv[1][0], kv[1][1], letters, 77)
    z = OM.path_state(L, kv[1][0], kv[1][1], [77])
    full = OM.head_logprobs(L, z)[letters]
    ref = np.exp(full) / np.exp(full).sum()
    assert np.allclose(r["prob"], ref, atol=1e-12)
    assert r["argmax"] == int(np.argmax(ref))


def test_trie_decode_matches_argmax_walk():
    """Greedy decode = walk the argmax child at every branching node (brute
    force from the tree evaluation at all internal nodes); it touches only
    branching nodes (3 on the support shape) and stops at one label."""
    L, kv = _tiny_setup(ndocs=4)
    ls = _support(S.TINY.vocab, 5)
    t = build_trie(ls.labels, ls.root_token, S.TINY.vocab, ls.continuation)
    internal = [u for u in range(t["n_nodes"]) if len(children_of(t, u))]
    branching = {u for u in range(t["n_nodes"]) if t["is_branching"][u]}
    assert len(branching) == 3
    for dk, dv in kv:
        rows = OS.eval_logprob_rows(L, dk, dv, t, nodes=internal)
        u = 0
        while t["subtree_labels"][u] > 1:
            ch = children_of(t, u)
            u = int(max(ch, key=lambda c: (rows[u][int(t["token"][c])], -int(t["token"][c]))))
        want = [m for m in range(10) if u <= t["label_end_node"][m] < u + t["subtree_size"][u]]
        dec = OS.trie_decode(L, dk, dv, t)
        assert dec["label"] == want[0]
        assert set(dec["touched"]) <= branching
        assert len(dec["touched"]) <= 2
