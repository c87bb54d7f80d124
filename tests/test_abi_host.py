"""C ABI checks that need no GPU: the library loads and exports every function
include/quail.h declares; the host trie builder agrees bit-exactly with the
oracle's independent builder; host-side argument errors map to the declared
statuses."""
import ctypes
import os
import re

import numpy as np
import pytest

import synthetic as S
import trie_label_scoring_gb300 as Q
from oracle.trie import TrieError, build_trie

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "quail.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    Q.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(quail_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 10
    L = ctypes.CDLL(Q.LIB)
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(Q._SIGNATURES), "binding and header disagree"
    for n in Q._TEST_SIGNATURES:  # test hooks: exported, deliberately not in the public header
        assert hasattr(L, n) and n not in names, n


FIELDS = ["parent", "depth", "token", "subtree_size", "child_offsets", "child_nodes", "child_tokens",
          "is_branching", "subtree_labels", "node_label", "label_end_node", "label_length", "label_decide_depth",
          "eval_nodes", "eval_index_of_node", "eval_child_offsets"]
SCALARS = ["n_nodes", "num_labels", "n_eval", "n_eval_children", "max_depth", "has_prefix_labels"]


def assert_same_trie(lib_view, oracle):
    for k in SCALARS:
        assert lib_view[k] == oracle[k], k
    for k in FIELDS:
        np.testing.assert_array_equal(lib_view[k], oracle[k].astype(lib_view[k].dtype), err_msg=k)


@pytest.mark.parametrize("name", list(S.WORKLOADS))
@pytest.mark.parametrize("full", [False, True])
def test_trie_bit_exact_on_workloads(name, full):
    w = S.WORKLOADS[name]
    ls = S.make_labels(w, 0)
    t = Q.Trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation, full_depth=full)
    o = build_trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation, full_depth=full)
    assert_same_trie(t.view(), o)


@pytest.mark.parametrize("seed", range(8))
def test_trie_all_nodes_flag_bit_exact(seed):
    """QUAIL_TRIE_ALL_NODES: every node is an evaluated position (join partner tries)."""
    rng = np.random.default_rng(100 + seed)
    labels = set()
    while len(labels) < 12:
        labels.add(tuple(int(x) for x in rng.integers(0, 9, size=int(rng.integers(1, 6)))))
    labels = [list(l) for l in labels]
    t = Q.Trie(labels, 20, 64, all_nodes=True)
    o = build_trie(labels, 20, 64, all_nodes=True)
    assert o["n_eval"] == o["n_nodes"]
    assert_same_trie(t.view(), o)


@pytest.mark.parametrize("seed", range(40))
def test_trie_bit_exact_random_with_prefix_labels(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(3, 9))
    M = int(rng.integers(2, 25))
    labels = set()
    while len(labels) < M:
        labels.add(tuple(int(x) for x in rng.integers(0, V, size=int(rng.integers(1, 6)))))
    labels = [list(l) for l in labels]
    rng.shuffle(labels)
    cont = np.zeros((V + 7) // 8, dtype=np.uint8)
    for t in rng.choice(V, size=int(rng.integers(0, V)), replace=False):
        cont[t >> 3] |= 1 << (t & 7)
    root = int(rng.integers(0, V))
    t = Q.Trie(labels, root, V, cont)
    assert_same_trie(t.view(), build_trie(labels, root, V, cont))


@pytest.mark.parametrize("labels,vocab,kind,status", [
    ([[1], []], 10, "empty_label", "QUAIL_ERR_EMPTY_LABEL"),
    ([[1, 2], [3], [1, 2]], 10, "duplicate_label", "QUAIL_ERR_DUPLICATE_LABEL"),
    ([[1, 10], [3]], 10, "token_range", "QUAIL_ERR_TOKEN_RANGE"),
    ([[1, -1], [3]], 10, "token_range", "QUAIL_ERR_TOKEN_RANGE"),
    ([[1]], 10, "invalid_arg", "QUAIL_ERR_INVALID_ARG"),
])
def test_trie_errors_match_oracle(labels, vocab, kind, status):
    with pytest.raises(TrieError) as e:
        build_trie(labels, 0, vocab)
    assert e.value.kind == kind
    with pytest.raises(Q.QuailError) as e2:
        Q.Trie(labels, 0, vocab)
    assert e2.value.name == status


def test_root_token_range():
    with pytest.raises(Q.QuailError) as e:
        Q.Trie([[1], [2]], 10, 10)
    assert e.value.name == "QUAIL_ERR_TOKEN_RANGE"


def test_workspace_size_positive_and_monotone():
    sh = S.QWEN3_4B
    bits = {k: np.zeros(1, np.uint16) for k in ("embed", "w_q", "w_k", "w_v", "q_norm", "k_norm", "w_o",
                                                 "in_norm", "final_norm", "lm_head")}
    desc = Q.ModelDesc(sh.hidden, sh.n_q_heads, sh.n_kv_heads, 128, sh.vocab, 1e-6, 1e6)
    m = type("M", (), {"desc": desc})()
    ls = S.make_labels(S.WORKLOADS["qwen3-4b-support10-256docs"], 0)
    t = Q.Trie(ls.labels, ls.root_token, sh.vocab, ls.continuation)
    a = Q.workspace_size(m, t, 0, 16, 1024, Q.MODE_TRIE_TREE)
    b = Q.workspace_size(m, t, 0, 256, 1024, Q.MODE_TRIE_TREE)
    assert 0 < a < b
    assert Q.workspace_size(m, None, 255, 64, 2048, Q.MODE_LETTERS) > 0
    assert Q.workspace_size(m, t, 0, 32, 8192, Q.MODE_TRIE_DECODE) > 0
    with pytest.raises(Q.QuailError):
        Q.workspace_size(m, None, 0, 16, 1024, Q.MODE_TRIE_TREE)


def _desc_only_model(sh):
    desc = Q.ModelDesc(sh.hidden, sh.n_q_heads, sh.n_kv_heads, 128, sh.vocab, 1e-6, 1e6)
    return type("M", (), {"desc": desc})()


def test_shortlist_workspace_and_argument_errors():
    """Host-side checks of the shortlist calls: workspace sizes grow with the
    beam and the documents; a plan from another trie or a beam below 1 is
    rejected before any device work."""
    sh = S.QWEN3_4B
    m = _desc_only_model(sh)
    w = S.Workload("t", sh, 4, (64, 64), "tree", 300, (2, 6))
    ls = S.make_labels(w, 0)
    t = Q.Trie(ls.labels, ls.root_token, sh.vocab)
    sl = Q.Shortlist(t, 1)
    a = Q.workspace_size_shortlist(m, t, sl, 1, 16, 1024)
    b = Q.workspace_size_shortlist(m, t, sl, 2, 16, 1024)
    c = Q.workspace_size_shortlist(m, t, sl, 2, 64, 1024)
    assert 0 < a < b < c
    with pytest.raises(Q.QuailError):
        Q.workspace_size_shortlist(m, t, sl, 0, 16, 1024)
    other = Q.Trie(ls.labels[:-1], ls.root_token, sh.vocab)
    with pytest.raises(Q.QuailError):
        Q.workspace_size_shortlist(m, other, sl, 2, 16, 1024)
    assert sl.num_groups == len(set(l[0] for l in ls.labels))


def test_multilayer_workspace_grows_with_documents_and_layers():
    sh = S.QWEN3_4B
    ls = S.make_labels(S.WORKLOADS["qwen3-4b-support10-256docs"], 0)
    t = Q.Trie(ls.labels, ls.root_token, sh.vocab, ls.continuation)

    def model(n_layers):
        lw = (Q.LayerWeights * n_layers)()
        desc = Q.ModelMLDesc(sh.hidden, sh.n_q_heads, sh.n_kv_heads, 128, sh.vocab, 9728, n_layers, 1e-6, 1e6,
                             None, None, None, lw)
        return type("M", (), {"desc": desc})()

    a = Q.workspace_size_ml(model(2), t, 16, 1024)
    b = Q.workspace_size_ml(model(2), t, 64, 1024)
    assert 0 < a < b
    assert Q.workspace_size_ml(model(36), t, 64, 1024) == b  # activations are reused layer to layer
