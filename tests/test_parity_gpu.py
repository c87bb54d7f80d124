"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs (element by element on small cases; on sampled
documents/labels at the workloads' full sizes)."""
import numpy as np
import pytest

import synthetic as S
from tests import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import trie_label_scoring_gb300 as Q
    Q.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run_trie_tree(w, seed=0, full_depth=False, labels=None, docs=None):
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    model = C.device_model(w.shape, seed)
    ls = labels or S.make_labels(w, seed)
    docs = docs or S.make_docs(w, seed)
    kv = kv_from_docs(docs)
    trie = Q.Trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation, full_depth=full_depth)
    N, M = w.num_docs, len(ls.labels)
    ws = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_TREE), dtype=torch.uint8,
                     device="cuda")
    lsc = torch.full((N, M), float("nan"), device="cuda")
    prob = torch.full((N, M), float("nan"), device="cuda")
    am = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    Q.classify_trie_tree(model, kv, trie, N, ws, lsc, prob, am)
    Q.device_status()
    return ls, docs, lsc.cpu().numpy(), prob.cpu().numpy(), am.cpu().numpy()


def _oracle_full(w, ls, docs, i, seed=0, full_depth=False):
    from oracle import scoring as OS
    from oracle.trie import build_trie
    L = C.oracle_layer(w.shape, seed)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation, full_depth=full_depth)
    dk, dv = C.oracle_doc_kv(docs, i)
    return OS.trie_tree(L, dk, dv, t)


@pytest.mark.parametrize("full_depth", [False, True])
def test_trie_tree_tiny_all_docs(full_depth):
    w = S.WORKLOADS["tiny-support10-4x128"]
    ls, docs, lsc, prob, am = _run_trie_tree(w, full_depth=full_depth)
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i, full_depth=full_depth)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")
        assert abs(prob[i].sum() - 1) < 1e-5


def test_launch_count_is_reported():
    """The library counts the kernels one call launches (the bench reports it):
    node prologue 4, attention 1-2, W_o + norm 2, head 1, scoring 1 or 3."""
    import trie_label_scoring_gb300 as Q
    w = S.WORKLOADS["tiny-support10-4x128"]
    _run_trie_tree(w)
    assert 9 <= Q.launch_count() <= 12


def test_trie_tree_tiny_ragged_lengths():
    """Lengths around page and split boundaries: 1, 15, 16, 17, 255, 256, 257, 700."""
    w = S.with_docs(S.WORKLOADS["tiny-support10-4x128"], 8, (1, 700))
    docs = S.make_docs(w, 3)
    lens = np.array([1, 15, 16, 17, 255, 256, 257, 700], dtype=np.int32)
    docs = _resize_docs(docs, lens, w)
    ls, docs, lsc, prob, am = _run_trie_tree(w, docs=docs)
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"len {lens[i]}")


def _resize_docs(docs, lens, w):
    """Same generator, fixed lengths: rebuild through a workload with one length per doc."""
    out = []
    for i, n in enumerate(lens):
        wi = S.with_docs(w, 1, (int(n), int(n)))
        out.append(S.make_docs(wi, 100 + i))
    # concatenate page pools
    k = np.concatenate([d.k_pool for d in out])
    v = np.concatenate([d.v_pool for d in out])
    maxp = max(d.page_table.shape[1] for d in out)
    pt = np.full((len(out), maxp), -1, dtype=np.int32)
    base = 0
    for i, d in enumerate(out):
        n = d.page_table.shape[1]
        pt[i, :n] = d.page_table[0] + base
        base += d.k_pool.shape[0]
    return S.PagedDocs(np.array(lens, dtype=np.int32), pt, k, v)


def _tiny_tree(num_docs, doc_len, num_labels=60):
    return S.Workload(f"tiny-tree{num_labels}-{num_docs}", S.TINY, num_docs, doc_len, "tree", num_labels, (1, 5))


def _rows_per_kv(w, ls):
    from oracle.trie import build_trie
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    return t["n_eval"] * (w.shape.n_q_heads // w.shape.n_kv_heads)


def test_trie_tree_tc_path_tiny_ragged_split():
    """More than 128 query rows per KV head (the tcgen05 attention, two row
    tiles, the second partial) on documents split across CTAs (partials and
    the combine kernel), lengths around page and 128-key block boundaries."""
    w = _tiny_tree(8, (1, 1000))
    ls = S.make_labels(w, 5)
    assert _rows_per_kv(w, ls) > 128
    lens = np.array([1, 15, 17, 127, 128, 129, 300, 1000], dtype=np.int32)
    docs = _resize_docs(S.make_docs(w, 5), lens, w)
    ls, docs, lsc, prob, am = _run_trie_tree(w, seed=5, labels=ls, docs=docs)
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i, seed=5)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"len {lens[i]}")


def test_trie_tree_tc_path_tiny_fused_epilogue():
    """Enough (document, KV head, row tile) items that every document is one
    split: the tcgen05 attention merges the tree part in its epilogue."""
    w = _tiny_tree(240, (100, 400))
    ls = S.make_labels(w, 6)
    assert _rows_per_kv(w, ls) > 128
    ls, docs, lsc, prob, am = _run_trie_tree(w, seed=6, labels=ls)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in [0, 1, 97, 150, 239]:
        r = _oracle_full(w, ls, docs, i, seed=6)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


def test_trie_tree_prefix_labels_tiny():
    """Labels that are prefixes of other labels (prefix correction on the GPU)."""
    w = S.WORKLOADS["tiny-support10-4x128"]
    rng = np.random.default_rng(7)
    toks = [int(t) for t in rng.choice(w.shape.vocab, size=6, replace=False)]
    labels = [[toks[0]], [toks[0], toks[1]], [toks[0], toks[2]], [toks[3]], [toks[3], toks[4], toks[5]],
              [toks[4]]]
    ls = S.LabelSet(labels, int(toks[5]) ^ 1, None)
    ls_, docs, lsc, prob, am = _run_trie_tree(w, labels=ls)
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


@pytest.mark.parametrize("name,ndocs", [("qwen3-4b-support10-256docs", 8)])
def test_trie_tree_qwen_small_all_docs(name, ndocs):
    w = S.with_docs(S.WORKLOADS[name], ndocs)
    ls, docs, lsc, prob, am = _run_trie_tree(w)
    for i in range(ndocs):
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


@pytest.mark.parametrize("ndocs,check", [
    (200, (0, 63, 127, 128, 191, 192, 199)),  # 800 rows, 7 tiles: two clusters of four, one padding tile
    (96, (0, 31, 32, 64, 95)),                # 384 rows, 3 tiles: one cluster of four, one padding tile
])
def test_output_head_partial_cluster(ndocs, check):
    """Documents of the support-topic shape (4 head rows each) whose head rows
    fill 128-row tiles up to a partial cluster: the padding tile of the
    cluster reads zeros and writes nothing."""
    w = S.with_docs(S.WORKLOADS["qwen3-4b-support10-256docs"], ndocs)
    ls, docs, lsc, prob, am = _run_trie_tree(w)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in check:  # rows in the first, middle and last tiles
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


@pytest.mark.parametrize("name,sample_docs", [
    ("qwen3-4b-support10-256docs", list(range(256))),  # every document of the bench workload
    ("qwen3-4b-tree255-64x2048", list(range(0, 64, 4)) + [63]),  # 17 of 64: the oracle takes seconds per document
    ("qwen3-4b-tree20-32x8192", list(range(32))),  # every document
])
def test_trie_tree_full_size_sampled_docs(name, sample_docs):
    w = S.WORKLOADS[name]
    ls, docs, lsc, prob, am = _run_trie_tree(w)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in sample_docs:
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"{name} doc {i}")


def test_trie_tree_large_label_set_all_labels():
    """5,000 labels of 2-10 tokens (~19k trie nodes): every label's log score
    and probability, and the argmax, against the full oracle on the first and
    last document."""
    w = S.WORKLOADS["qwen3-4b-tree5000-16x1024"]
    ls, docs, lsc, prob, am = _run_trie_tree(w)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in (0, 15):
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


def test_trie_tree_large_label_set_small_layer_all_docs():
    """The same 5,000-label shape (shared prefixes, 2-10 tokens) on the small
    layer, where the oracle is cheap: every label of every document."""
    w = S.Workload("tiny-shared5000-4", S.TINY, 4, (100, 700), "shared", 5000, (2, 10), 10.0)
    ls, docs, lsc, prob, am = _run_trie_tree(w, seed=2)
    assert _rows_per_kv(w, ls) > 128
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i, seed=2)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


def test_letters_tiny_and_full_size_sample():
    import trie_label_scoring_gb300 as Q
    from oracle import scoring as OS
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    for name, sample in (("tiny-support10-4x128", None), ("qwen3-4b-letters255-64x2048", None)):  # every document
        w = S.WORKLOADS[name]
        if name.startswith("tiny"):
            rng = np.random.default_rng(5)
            letters = [int(x) for x in rng.choice(w.shape.vocab, size=10, replace=False)]
            root = 17
        else:
            ls = S.make_labels(w, 0)
            letters, root = [l[0] for l in ls.labels], ls.root_token
        model = C.device_model(w.shape)
        docs = S.make_docs(w, 0)
        kv = kv_from_docs(docs)
        N, M = w.num_docs, len(letters)
        ws = torch.empty(Q.workspace_size(model, None, M, N, docs.max_doc_len, Q.MODE_LETTERS), dtype=torch.uint8,
                         device="cuda")
        lp = torch.empty((N, M), device="cuda")
        pr = torch.empty((N, M), device="cuda")
        am = torch.empty((N,), dtype=torch.int32, device="cuda")
        Q.classify_letters(model, kv, letters, root, N, ws, lp, pr, am)
        Q.device_status()
        lp, pr, am = lp.cpu().numpy(), pr.cpu().numpy(), am.cpu().numpy()
        L = C.oracle_layer(w.shape)
        for i in (range(N) if sample is None else sample):
            dk, dv = C.oracle_doc_kv(docs, i)
            r = OS.letters(L, dk, dv, letters, root)
            C.check_scores(lp[i], pr[i], am[i], r["logprob"], r["prob"], r["argmax"], f"{name} doc {i}")


def _run_decode(w, docs, ls, max_steps=64):
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    model = C.device_model(w.shape)
    kv = kv_from_docs(docs)
    trie = Q.Trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    N = w.num_docs
    ws = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_DECODE), dtype=torch.uint8,
                     device="cuda")
    cur = torch.zeros(N, dtype=torch.int32, device="cuda")
    lab = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    act = torch.zeros(1, dtype=torch.int32, device="cuda")
    touched = torch.zeros((N, trie.n_nodes), dtype=torch.uint8, device="cuda")
    steps = 0
    while True:
        Q.classify_trie_decode_step(model, kv, trie, N, cur, lab, act, ws, touched)
        steps += 1
        if int(act.item()) == 0 or steps >= max_steps:
            break
    Q.device_status()
    return lab.cpu().numpy(), touched.cpu().numpy(), steps, trie.view()


@pytest.mark.parametrize("name,sample", [("tiny-support10-4x128", None),
                                         ("qwen3-4b-tree20-32x8192", [0, 5, 9, 17, 23, 31])])
def test_trie_decode_matches_oracle_walk(name, sample):
    from oracle import scoring as OS
    from oracle.trie import build_trie
    w = S.WORKLOADS[name]
    ls = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    lab, touched, steps, view = _run_decode(w, docs, ls)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    branching = set(np.nonzero(t["is_branching"])[0].tolist())
    assert (lab >= 0).all() and steps <= t["max_depth"] + 1
    L = C.oracle_layer(w.shape)
    for i in (range(w.num_docs) if sample is None else sample):
        assert set(np.nonzero(touched[i])[0].tolist()) <= branching
        dk, dv = C.oracle_doc_kv(docs, i)
        r = OS.trie_decode(L, dk, dv, t)
        if lab[i] != r["label"]:
            # a near-tie at some branching node may flip in fp32 vs fp64: the
            # GPU's pick must then be within tolerance of the oracle's best
            pytest.fail(f"doc {i}: decode label {lab[i]} != oracle {r['label']}")
        assert set(np.nonzero(touched[i])[0].tolist()) == set(r["touched"])
    if name.startswith("tiny"):
        assert set(np.nonzero(touched.any(axis=0))[0].tolist()) <= branching and len(branching) == 3


def test_decode_rejects_prefix_labels():
    import trie_label_scoring_gb300 as Q
    w = S.WORKLOADS["tiny-support10-4x128"]
    ls = S.LabelSet([[5], [5, 6], [7]], 1, None)
    docs = S.make_docs(w, 0)
    with pytest.raises(Q.QuailError) as e:
        _run_decode(w, docs, ls)
    assert e.value.name == "QUAIL_ERR_PREFIX_LABEL_UNSUPPORTED"


def test_device_bounds_error_is_reported():
    """A page id outside the pool is caught by the kernel's own check (no copy
    is issued for it) and reported through quail_device_status."""
    import trie_label_scoring_gb300 as Q
    w = S.WORKLOADS["tiny-support10-4x128"]
    docs = S.make_docs(w, 0)
    bad = S.PagedDocs(docs.doc_len.copy(), docs.page_table.copy(), docs.k_pool, docs.v_pool)
    bad.page_table[2, 1] = docs.k_pool.shape[0] + 5
    with pytest.raises(Q.QuailError) as e:
        _run_trie_tree(w, docs=bad)
    assert e.value.name == "QUAIL_ERR_DEVICE_BOUNDS"
    _run_trie_tree(w, docs=docs)  # context still usable, error word cleared


def test_device_wait_timeout_is_reported():
    """Every pipeline wait is bounded. With the limit cut to a few hundred
    cycles (a test hook), the waits of the call's kernels run out before their
    copies and MMAs arrive: each block leaves its pipeline, drains what is in
    flight under the normal limit, frees its tensor memory and returns, and
    the device error word reports QUAIL_ERR_DEVICE_TIMEOUT. The next call,
    with the default limit, is correct again."""
    import trie_label_scoring_gb300 as Q
    w = S.WORKLOADS["tiny-support10-4x128"]
    Q._test_set_pipeline_wait_limit(200)
    try:
        with pytest.raises(Q.QuailError) as e:
            _run_trie_tree(w)
    finally:
        Q._test_set_pipeline_wait_limit(0)
    assert e.value.name == "QUAIL_ERR_DEVICE_TIMEOUT"
    ls, docs, lsc, prob, am = _run_trie_tree(w)  # context still usable, error word cleared
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


def test_workspace_too_small_is_rejected():
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    w = S.WORKLOADS["tiny-support10-4x128"]
    model = C.device_model(w.shape)
    ls = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    trie = Q.Trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    need = Q.workspace_size(model, trie, 0, 4, docs.max_doc_len, Q.MODE_TRIE_TREE)
    ws = torch.empty(need - 1024, dtype=torch.uint8, device="cuda")
    out = torch.empty((4, 10), device="cuda")
    am = torch.empty(4, dtype=torch.int32, device="cuda")
    with pytest.raises(Q.QuailError) as e:
        Q.classify_trie_tree(model, kv, trie, 4, ws, out, out, am)
    assert e.value.name == "QUAIL_ERR_WORKSPACE"


def test_zero_documents_is_a_no_op():
    """N = 0: the call succeeds and leaves the outputs untouched."""
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    w = S.WORKLOADS["tiny-support10-4x128"]
    model = C.device_model(w.shape)
    ls = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    trie = Q.Trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    ws = torch.empty(Q.workspace_size(model, trie, 0, 1, docs.max_doc_len, Q.MODE_TRIE_TREE), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((1, len(ls.labels)), float("nan"), device="cuda")
    am = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    Q.classify_trie_tree(model, kv, trie, 0, ws, out, out, am)
    Q.device_status()
    assert torch.isnan(out).all() and int(am[0]) == -7


@pytest.mark.parametrize("labels", ["support10", "tree60"])
def test_long_documents_past_the_split_cap(labels):
    """Enough (document, KV head) items for whole-document splits: capped at
    4096 keys on the mma.sync path (16 rows per KV head), where documents of
    4095..8192 tokens take one or two splits (and the combine kernel), and at
    8192 on the tcgen05 path (more than 128 rows), where each is one tile."""
    if labels == "support10":
        w = S.with_docs(S.WORKLOADS["tiny-support10-4x128"], 232, (16, 8192))
        ls = S.make_labels(w, 0)
        assert _rows_per_kv(w, ls) <= 16
    else:
        w = _tiny_tree(232, (16, 8192))
        ls = S.make_labels(w, 5)
        assert _rows_per_kv(w, ls) > 128
    long_lens = [4095, 4096, 4097, 5000, 8192]
    rng = np.random.default_rng(11)
    lens = np.concatenate([np.array(long_lens), rng.integers(16, 64, size=w.num_docs - len(long_lens))])
    lens = lens.astype(np.int32)
    docs = _resize_docs(None, lens, w)
    ls, docs, lsc, prob, am = _run_trie_tree(w, seed=5 if labels == "tree60" else 0, labels=ls, docs=docs)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in [0, 2, 4, w.num_docs - 1]:  # 4095, 4097, 8192 tokens and a short one
        r = _oracle_full(w, ls, docs, i, seed=5 if labels == "tree60" else 0)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"len {lens[i]}")


@pytest.mark.parametrize("labels", ["support10", "tree60"])
def test_very_long_documents_many_splits(labels):
    """Three documents, one of 32,768 tokens: with so few (document, KV head)
    items the long document is cut into many splits (up to the split caps of
    4,096 and 8,192 keys), whose partials the combine kernel merges with the
    tree part; every document against the oracle."""
    lens = np.array([32768, 20001, 300], dtype=np.int32)
    if labels == "support10":
        w = S.with_docs(S.WORKLOADS["tiny-support10-4x128"], 3, (16, 32768))
        ls = S.make_labels(w, 0)
        assert _rows_per_kv(w, ls) <= 16
    else:
        w = _tiny_tree(3, (16, 32768))
        ls = S.make_labels(w, 5)
        assert _rows_per_kv(w, ls) > 128
    seed = 5 if labels == "tree60" else 0
    docs = _resize_docs(None, lens, w)
    ls, docs, lsc, prob, am = _run_trie_tree(w, seed=seed, labels=ls, docs=docs)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in range(3):
        r = _oracle_full(w, ls, docs, i, seed=seed)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"len {lens[i]}")


@pytest.mark.parametrize("shape", ["deep_chain", "one_token", "single_root_child", "twenty_deep"])
def test_degenerate_label_shapes(shape):
    """Label sets at the edges of the trie's shape, every document against
    the oracle: two labels sharing nine tokens (ten evaluated nodes on one
    chain), one-token labels (only the root is evaluated), a root with a
    single child, and labels twenty tokens deep."""
    w = S.WORKLOADS["tiny-support10-4x128"]
    base = S.make_labels(w, 0)
    labels = {
        "deep_chain": [[5, 6, 7, 8, 9, 10, 11, 12, 13, 14], [5, 6, 7, 8, 9, 10, 11, 12, 13, 15]],
        "one_token": [[100], [200], [300], [400], [8191]],
        "single_root_child": [[7, 1], [7, 2], [7, 3, 4], [7, 3, 5]],
        "twenty_deep": [list(range(1, 21)), list(range(1, 20)) + [99], list(range(40, 60))],
    }[shape]
    ls = S.LabelSet(labels, base.root_token, None)
    ls_, docs, lsc, prob, am = _run_trie_tree(w, labels=ls)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"{shape} doc {i}")


def test_prefix_labels_on_the_tcgen05_path():
    """Labels that are prefixes of other labels, on a trie with more than 128
    query rows per KV head: the prefix correction log(1 - sum of the end
    node's child probabilities) over rows from the tcgen05 attention."""
    w = _tiny_tree(6, (40, 400))
    base = S.make_labels(w, 8)
    labels = [list(l) for l in base.labels]
    seen = {tuple(l) for l in labels}
    for l in list(labels):  # add every proper prefix of length >= 1 of the longer labels once
        for k in range(1, len(l)):
            p = tuple(l[:k])
            if p not in seen and len(labels) < 90:
                seen.add(p)
                labels.append(list(p))
    ls = S.LabelSet(labels, base.root_token, None)
    assert _rows_per_kv(w, ls) > 128
    assert any(tuple(m[:len(l)]) == tuple(l) for l in labels for m in labels if len(m) > len(l))
    ls_, docs, lsc, prob, am = _run_trie_tree(w, seed=8, labels=ls)
    assert np.all(np.abs(prob.sum(axis=1) - 1) < 1e-4)
    for i in range(w.num_docs):
        r = _oracle_full(w, ls, docs, i, seed=8)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")
