"""AI.IF over joined pairs (quail_join_if): the oracle against closed forms,
and the CUDA path against the oracle on every (anchor, partner) pair."""
import numpy as np
import pytest

import synthetic as S
from tests import gpu_cases as C

TOL_P = 1e-3


def _partners(rng, vocab, n=12):
    """Partner token lists after the root token: a shared 3-token instruction,
    then a distinct 1..4-token tail (one tail a prefix of another)."""
    shared = [int(t) for t in rng.choice(vocab, size=3, replace=False)]
    tails = set()
    while len(tails) < n - 1:
        tails.add(tuple(int(t) for t in rng.integers(0, vocab, size=int(rng.integers(1, 5)))))
    tails = [list(t) for t in tails]
    tails.append(tails[0][:1] if len(tails[0]) > 1 else tails[0] + [int(rng.integers(0, vocab))])
    return [shared + t for t in tails]


def _answers(rng, vocab):
    t = [int(x) for x in rng.choice(vocab, size=6, replace=False)]
    return t[:3], t[3:]


# ----------------------------------------------------------------- oracle pins
def test_restricted_softmax_is_the_renormalised_full_distribution():
    import oracle.model as OM
    from oracle import join as J
    w = S.WORKLOADS["tiny-support10-4x128"]
    L = C.oracle_layer(w.shape, 0)
    docs = S.make_docs(w, 0)
    dk, dv = C.oracle_doc_kv(docs, 1)
    rng = np.random.default_rng(1)
    yes, no = _answers(rng, w.shape.vocab)
    z = OM.path_state(L, dk, dv, [5, 17, 42])
    lp = OM.head_logprobs(L, z)
    full = np.exp(lp[yes]).sum() / np.exp(lp[yes + no]).sum()
    assert J.restricted_p_true(z, L, yes, no) == pytest.approx(full, rel=1e-12)
    assert J.restricted_p_true(z, L, yes, []) == pytest.approx(1.0, abs=1e-15)
    assert J.restricted_p_true(z, L, yes[:1], no) + J.restricted_p_true(z, L, no, yes[:1]) == pytest.approx(1.0)


# ------------------------------------------------------------------ GPU parity
def _run_join(w, docs, partners, root, yes, no, seed=0):
    import torch
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    model = C.device_model(w.shape, seed)
    kv = kv_from_docs(docs)
    t = Q.Trie(partners, root, w.shape.vocab, all_nodes=True)
    N, M = len(docs.doc_len), len(partners)
    ws = torch.empty(Q.workspace_size(model, t, len(yes) + len(no), N, docs.max_doc_len, Q.MODE_JOIN_IF),
                     dtype=torch.uint8, device="cuda")
    p = torch.full((N, M), float("nan"), device="cuda")
    Q.join_if(model, kv, t, N, yes, no, ws, p)
    Q.device_status()
    return p.cpu().numpy()


def _check(w, docs, partners, root, yes, no, anchors, p_gpu, seed=0):
    from oracle import join as J
    L = C.oracle_layer(w.shape, seed)
    for i in anchors:
        dk, dv = C.oracle_doc_kv(docs, i)
        ref = J.join_if(L, dk, dv, root, partners, yes, no)
        d = np.abs(p_gpu[i] - ref)
        assert d.max() <= TOL_P, f"anchor {i}: max |d p_true| = {d.max():.2e}"


@pytest.mark.gpu
def test_join_if_tiny_ragged_anchors():
    w = S.with_docs(S.WORKLOADS["tiny-support10-4x128"], 6, (1, 600))
    rng = np.random.default_rng(2)
    docs = S.make_docs(w, 2)
    partners = _partners(rng, w.shape.vocab)
    yes, no = _answers(rng, w.shape.vocab)
    root = int(rng.integers(0, w.shape.vocab))
    p = _run_join(w, docs, partners, root, yes, no)
    assert np.all(np.isfinite(p)) and np.all((p >= 0) & (p <= 1))
    _check(w, docs, partners, root, yes, no, range(6), p)


@pytest.mark.gpu
def test_join_if_many_anchors_single_split():
    """Enough anchors that each is one split: the attention epilogue merges
    the partner part itself."""
    w = S.with_docs(S.WORKLOADS["tiny-support10-4x128"], 240, (64, 256))
    rng = np.random.default_rng(3)
    docs = S.make_docs(w, 3)
    partners = _partners(rng, w.shape.vocab, n=40)
    yes, no = _answers(rng, w.shape.vocab)
    root = int(rng.integers(0, w.shape.vocab))
    p = _run_join(w, docs, partners, root, yes, no)
    _check(w, docs, partners, root, yes, no, [0, 101, 239], p)


@pytest.mark.gpu
def test_join_if_qwen_shape_sampled():
    w = S.with_docs(S.WORKLOADS["qwen3-4b-support10-256docs"], 16)
    rng = np.random.default_rng(4)
    docs = S.make_docs(w, 0)
    partners = _partners(rng, w.shape.vocab, n=20)
    yes, no = _answers(rng, w.shape.vocab)
    root = int(rng.integers(0, w.shape.vocab))
    p = _run_join(w, docs, partners, root, yes, no)
    _check(w, docs, partners, root, yes, no, [0, 15], p)


@pytest.mark.gpu
def test_join_if_rejects_tries_without_all_nodes():
    import torch
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    w = S.WORKLOADS["tiny-support10-4x128"]
    docs = S.make_docs(w, 0)
    model = C.device_model(w.shape, 0)
    t = Q.Trie([[1, 2], [1, 3]], 0, w.shape.vocab)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    p = torch.empty((4, 2), device="cuda")
    with pytest.raises(Q.QuailError):
        Q.join_if(model, kv_from_docs(docs), t, 4, [5], [6], ws, p)
